// Expansion of selected pools to token indices plus the causal tail
// (Megatron-LM PR "GLM5.3 Flash (KDA + mHC + KPool DSA) support + FP8",
// Changes section 3: top-k pools are expanded back to token indices;
// always_select_tail appends each query's incomplete causal pool; packed THD
// restarts pools at document boundaries).
//
// HBM-write-bound: one warp per query row, lanes stride over the
// Kp*kpool + kpool - 1 outputs of the row (128-byte coalesced stores); for a
// few rows (decode) one block per row.
#include "kpool_internal.h"

namespace kpool {
namespace {

constexpr int kThreads = 256;
constexpr int kRowsPerBlock = kThreads / 32;

// Document of row t: the largest d < n_docs with cu[d] <= t, found by one warp
// probing 32 evenly spaced offsets per round (two rounds up to 1024 documents)
// instead of a chain of dependent binary-search loads.  All lanes get the
// answer.  Invariant: cu[lo] <= t (cu[0] = 0).
__device__ __forceinline__ int doc_of_row_warp(const int32_t *cu, int n_docs, int64_t t, int lane)
{
    int lo = 0, hi = n_docs;   // answer in [lo, hi)
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int idx = lo + lane * step;
        const bool le = idx < hi && cu[idx] <= t;
        const unsigned m = __ballot_sync(0xFFFFFFFFu, le);   // bit 0 set: idx = lo
        const int nlo = lo + (31 - __clz(m)) * step;
        hi = min(hi, nlo + step);
        lo = nlo;
    }
    return lo;
}

constexpr int kStageInts = 512;   // per-warp staging of a row's pool list (larger Kp read directly)

template <int KP>   // KP > 0: compile-time kpool; 0: runtime kp
__global__ void __launch_bounds__(kThreads) expand_kernel(
    const int32_t *__restrict__ pool_idx, const int32_t *__restrict__ cu_seqlens,
    const int32_t *__restrict__ q_pos, const int32_t *__restrict__ cu_k,
    const int32_t *__restrict__ cu_pools, int n_docs, int64_t T, int kp_rt, int Kp, int tail,
    int32_t *__restrict__ out)
{
    __shared__ int32_t stage[kRowsPerBlock][kStageInts];
    const int kp = KP > 0 ? KP : kp_rt;
    const int wib = threadIdx.x >> 5;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kRowsPerBlock + wib;
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    // query row t: document d, position tau, keys starting at token key0
    int64_t doc_start = 0, key0 = 0, pos0 = 0, pool_lo = 0, pool_hi = T / kp;
    if (cu_seqlens != nullptr) {
        const int d = doc_of_row_warp(cu_seqlens, n_docs, t, lane);
        doc_start = cu_seqlens[d];
        key0 = cu_k != nullptr ? cu_k[d] : doc_start;
        pos0 = q_pos != nullptr ? q_pos[d] : 0;
        pool_lo = cu_pools[d];
        pool_hi = cu_pools[d + 1];
    }
    const int64_t tau = pos0 + (t - doc_start);
    const int64_t nc = min((tau + 1) / kp, pool_hi - pool_lo);
    const int n_sel = static_cast<int>(nc < Kp ? nc : Kp);
    const int n_pool_tok = n_sel * kp;
    const int n_tail = tail ? static_cast<int>((tau + 1) % kp) : 0;   // own incomplete pool
    const int W = Kp * kp + kp - 1;
    const int32_t *row_in = pool_idx + t * Kp;
    int32_t *row_out = out + t * W;
    // the row's selected pools, staged with coalesced loads
    const bool staged = n_sel <= kStageInts;
    int32_t *st = stage[wib];
    if (staged) {
        for (int e = lane; e < n_sel; e += 32) st[e] = __ldg(row_in + e);
        __syncwarp();
    }
    for (int c = lane; c < W; c += 32) {
        int32_t v = -1;
        if (c < n_pool_tok) {
            const int e = c / kp;
            const int s = c - e * kp;
            const int32_t g = staged ? st[e] : row_in[e];
            if (g >= pool_lo && g < pool_hi)
                v = static_cast<int32_t>(key0 + (g - pool_lo) * kp + s);
        } else if (c < n_pool_tok + n_tail) {
            v = static_cast<int32_t>(key0 + tau - n_tail + 1 + (c - n_pool_tok));
        }
        __stcs(row_out + c, v);   // streaming store: the table is not re-read here
    }
}

// Few rows (decode): one block of kThreads per row, so that the rows spread
// over the SMs and each row's outputs are written by 256 threads.
template <int KP>
__global__ void __launch_bounds__(kThreads) expand_row_kernel(
    const int32_t *__restrict__ pool_idx, const int32_t *__restrict__ cu_seqlens,
    const int32_t *__restrict__ q_pos, const int32_t *__restrict__ cu_k,
    const int32_t *__restrict__ cu_pools, int n_docs, int64_t T, int kp_rt, int Kp, int tail,
    int32_t *__restrict__ out)
{
    __shared__ int32_t stage[kStageInts];
    __shared__ int64_t rowinfo[5];   // key0, tau, pool_lo, pool_hi, n_sel
    const int kp = KP > 0 ? KP : kp_rt;
    const int64_t t = blockIdx.x;
    const int lane = threadIdx.x & 31;
    if (threadIdx.x < 32) {
        int64_t doc_start = 0, key0 = 0, pos0 = 0, pool_lo = 0, pool_hi = T / kp;
        if (cu_seqlens != nullptr) {
            const int d = doc_of_row_warp(cu_seqlens, n_docs, t, lane);
            doc_start = cu_seqlens[d];
            key0 = cu_k != nullptr ? cu_k[d] : doc_start;
            pos0 = q_pos != nullptr ? q_pos[d] : 0;
            pool_lo = cu_pools[d];
            pool_hi = cu_pools[d + 1];
        }
        if (lane == 0) {
            const int64_t tau = pos0 + (t - doc_start);
            const int64_t nc = min((tau + 1) / kp, pool_hi - pool_lo);
            rowinfo[0] = key0;
            rowinfo[1] = tau;
            rowinfo[2] = pool_lo;
            rowinfo[3] = pool_hi;
            rowinfo[4] = nc < Kp ? nc : Kp;
        }
    }
    __syncthreads();
    const int64_t key0 = rowinfo[0], tau = rowinfo[1], pool_lo = rowinfo[2],
                  pool_hi = rowinfo[3];
    const int n_sel = static_cast<int>(rowinfo[4]);
    const int n_pool_tok = n_sel * kp;
    const int n_tail = tail ? static_cast<int>((tau + 1) % kp) : 0;
    const int W = Kp * kp + kp - 1;
    const int32_t *row_in = pool_idx + t * Kp;
    int32_t *row_out = out + t * W;
    const bool staged = n_sel <= kStageInts;
    if (staged) {
        for (int e = threadIdx.x; e < n_sel; e += kThreads) stage[e] = __ldg(row_in + e);
        __syncthreads();
    }
    for (int c = threadIdx.x; c < W; c += kThreads) {
        int32_t v = -1;
        if (c < n_pool_tok) {
            const int e = c / kp;
            const int s = c - e * kp;
            const int32_t g = staged ? stage[e] : row_in[e];
            if (g >= pool_lo && g < pool_hi)
                v = static_cast<int32_t>(key0 + (g - pool_lo) * kp + s);
        } else if (c < n_pool_tok + n_tail) {
            v = static_cast<int32_t>(key0 + tau - n_tail + 1 + (c - n_pool_tok));
        }
        __stcs(row_out + c, v);
    }
}

}  // namespace

cudaError_t launch_expand(const int32_t *pool_idx, const int32_t *cu_seqlens,
                          const int32_t *q_pos, const int32_t *cu_k, const int32_t *cu_pools,
                          int n_docs, int64_t T, int kpool, int Kp, int tail, int32_t *tok_idx,
                          cudaStream_t s)
{
    if (T == 0) return cudaSuccess;
    if (T <= 4 * num_sms()) {
        const unsigned rblocks = static_cast<unsigned>(T);
        switch (kpool) {
        case 1: expand_row_kernel<1><<<rblocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
        case 2: expand_row_kernel<2><<<rblocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
        case 4: expand_row_kernel<4><<<rblocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
        case 8: expand_row_kernel<8><<<rblocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
        default: expand_row_kernel<0><<<rblocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
        }
        return cudaGetLastError();
    }
    const unsigned blocks = static_cast<unsigned>((T + kRowsPerBlock - 1) / kRowsPerBlock);
    switch (kpool) {
    case 1: expand_kernel<1><<<blocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
    case 2: expand_kernel<2><<<blocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
    case 4: expand_kernel<4><<<blocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
    case 8: expand_kernel<8><<<blocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
    default: expand_kernel<0><<<blocks, kThreads, 0, s>>>(pool_idx, cu_seqlens, q_pos, cu_k, cu_pools, n_docs, T, kpool, Kp, tail, tok_idx); break;
    }
    return cudaGetLastError();
}

}  // namespace kpool
