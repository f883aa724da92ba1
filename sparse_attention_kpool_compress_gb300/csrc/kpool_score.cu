// Causal pool scoring fused with a streaming per-query top-k.
//
//   score[t, p] = sum_h w[t, h] * relu( q[t, h, :] . pk[p, :] )
//
// over the complete causal pools p of t's document, then the best
// Kp = index_topk / kpool pools per query (Megatron-LM PR "GLM5.3 Flash (KDA +
// mHC + KPool DSA) support + FP8", Changes section 3; xtuner PR
// "GLM-5.3-Flash F5: NoPE DSA + KPool indexer": relu homogeneity lets any
// head_dim^-0.5 factor live in w; DeepSelect-style radix selection).
//
// Design (one persistent CTA per SM, 12 warps):
//   warp 0      TMA producer + tile scheduler (atomic counter over a
//               longest-first query-tile table built by schedule_kernel)
//   warp 1      tcgen05.mma issuer (one thread)
//   warp 2      TMEM allocator
//   warps 4-11  epilogue: tcgen05.ld of the accumulator, relu * w head
//               reduction, threshold filter, ordered append into per-query
//               candidate buffers in shared memory, radix-select compaction.
// MMA tile: M = 128 pools (TMEM lanes, one epilogue thread per pool),
// N = 256 (query, head) columns = 256 / H queries, K = D (bf16: 16 per
// instruction, E4M3: 32).  q of the query tile stays resident in shared
// memory; pooled-key tiles stream through a ring of `stages` buffers; two
// 256-column TMEM accumulators let the epilogue of tile i overlap the MMAs of
// tile i+1.  Candidates are kept in ascending pool order, so ties resolve to
// the lower pool index by position and no final sort is needed.
#include <cuda.h>

#include <cstring>
#include <mutex>
#include <vector>

#include "kpool_internal.h"
#include "kpool_ptx.cuh"

namespace kpool {
namespace {

constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;           // 256
constexpr int kThreads = 128 + kEpiThreads;           // 384
constexpr int kBM = 128;                              // pools per tile
constexpr int kBN = 256;                              // (query, head) columns per tile
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;
constexpr int kSmemLimit = 232448;                    // 227 KiB per block (opt-in max)
constexpr int kMaxC = 4096;
constexpr int kMaxR = kMaxC / kEpiThreads;            // 16 entries per thread in a compaction
constexpr int kMaxStages = 6;
constexpr uint64_t kTimeoutNs = 2000000000ull;        // 2 s per wait
constexpr uint32_t kFull = 0xFFFFFFFFu;

// barrier indices
constexpr int BQ_FULL = 0, BQ_EMPTY = 1, BTM_FULL = 2, BTM_EMPTY = 4, BTI_FULL = 6,
              BTI_EMPTY = 8, BDRAIN = 10, BPK_FULL = 11;   // then pk_full[S], pk_empty[S]

// workspace header (ints)
constexpr int WS_COUNTER = 0, WS_STATUS = 1, WS_NTILES = 2, WS_TABLE_INTS = 64;

struct Layout {
    int n_kchunks;      // 128-byte K chunks per operand row
    int stages;
    int C;              // candidate capacity per query
    uint32_t q_off, q_chunk;
    uint32_t pk_off, pk_chunk, pk_stage;
    uint32_t ws_off, hist_off, cnt_off, scr_off, thr_off, bar_off, ti_off, misc_off;
    uint32_t cs_off, ci_off;
    uint32_t total;
};

__host__ __device__ inline int qt_of(int H) { return kBN / H; }

Layout make_layout(int H, int D, int fp8)
{
    Layout L{};
    const int esize = fp8 ? 1 : 2;
    L.n_kchunks = (D * esize + 127) / 128;
    L.stages = fp8 ? 4 : 3;
    const int QT = qt_of(H);
    L.q_chunk = kBN * 128;
    L.pk_chunk = kBM * 128;
    L.q_off = 0;
    L.pk_off = L.q_off + L.n_kchunks * L.q_chunk;
    L.pk_stage = L.n_kchunks * L.pk_chunk;
    uint32_t off = L.pk_off + L.stages * L.pk_stage;
    L.ws_off = off;   off += kEpiWarps * 128 * 4;
    L.hist_off = off; off += 256 * 4;
    L.cnt_off = off;  off += 2 * QT * 4 * 4;
    L.scr_off = off;  off += 64 * 4;
    L.thr_off = off;  off += ((QT * 4 + 15) / 16) * 16;
    L.bar_off = off;  off += 256;
    L.ti_off = off;   off += 2 * 16;
    L.misc_off = off; off += 16;
    const int avail = kSmemLimit - 1024 - static_cast<int>(off);
    int C = avail / (8 * QT);
    C &= ~31;
    if (C > kMaxC) C = kMaxC;
    L.C = C > 0 ? C : 0;
    L.cs_off = off;
    L.ci_off = off + QT * L.C * 4;
    L.total = L.ci_off + QT * L.C * 4;
    return L;
}

struct Params {
    const float *w;
    const float *q_scale;
    const float *pk_scale;
    const int32_t *cu_seqlens;
    const int32_t *cu_pools;
    int n_docs, T, P_total, kp, Kp, fp8, mode;
    int32_t *pool_idx;
    float *pool_score;
    float *scores;
    int *ws;
    uint32_t q_tx, pk_tx, idesc;
    Layout L;
};

// Orderable key of a score: larger float -> larger key; -0 folded into +0.
__device__ __forceinline__ uint32_t fkey(float f)
{
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

struct Sync {
    volatile uint32_t *abort_flag;
    int *status;
};

// Bounded mbarrier wait: completion first, then the CTA abort flag, then a
// 2 s timer (sets KPOOL_STATUS_TIMEOUT and the abort flag).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Sync &sy)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*sy.abort_flag) return false;
        if (ptx::globaltimer() - t0 > kTimeoutNs) {
            *sy.abort_flag = 1u;
            atomicOr(sy.status, KPOOL_STATUS_TIMEOUT);
            return false;
        }
    }
}

// Warp-uniform version for the epilogue warps.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Sync &sy)
{
    bool ok = wait_bar(bar, parity, sy);
    return __all_sync(kFull, ok);
}

struct TileInfo {
    int t0, doc_start, doc_end, pool_base;
};

__device__ __forceinline__ int pool_tiles_of(const TileInfo &ti, int QT, int kp)
{
    const int tau0 = ti.t0 - ti.doc_start;
    const int nq = min(QT, ti.doc_end - ti.t0);
    const int nc_last = (tau0 + nq) / kp;       // (tau_last + 1) / kp
    return (nc_last + kBM - 1) / kBM;
}

// Keep the k best entries (score desc; earlier position wins ties) of
// cs/ci[0..n), n > k, in place and in order.  All 256 epilogue threads.
// Writes the threshold key to *thr_out.
__device__ void select_topk(float *cs, int *ci, int n, int k, int etid, int *hist, int *scr,
                            uint32_t *thr_out)
{
    const int lane = etid & 31, ew = etid >> 5;
    uint32_t prefix = 0;
    int kr = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        hist[etid] = 0;
        ptx::named_bar_sync(1, kEpiThreads);
        for (int base = 0; base < n; base += kEpiThreads) {
            const int e = base + etid;
            uint32_t key = 0;
            bool ok = false;
            if (e < n) {
                key = fkey(cs[e]);
                ok = (pass == 0) || ((key >> (shift + 8)) == (prefix >> (shift + 8)));
            }
            const uint32_t digit = (key >> shift) & 255u;
            const unsigned m = __ballot_sync(kFull, ok);
            if (ok) {
                const unsigned peers = __match_any_sync(m, digit);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[digit], __popc(peers));
            }
        }
        ptx::named_bar_sync(1, kEpiThreads);
        if (ew == 0) {
            int b[8];
            int local = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                b[i] = hist[lane * 8 + i];
                local += b[i];
            }
            int suf = local;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int o = __shfl_down_sync(kFull, suf, off);
                if (lane + off < 32) suf += o;
            }
            int cum = suf - local;   // entries in higher bins of higher lanes
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                if (cum < kr && cum + b[i] >= kr) {
                    scr[2 * pass] = lane * 8 + i;
                    scr[2 * pass + 1] = cum;
                }
                cum += b[i];
            }
        }
        ptx::named_bar_sync(1, kEpiThreads);
        prefix |= static_cast<uint32_t>(scr[2 * pass]) << shift;
        kr -= scr[2 * pass + 1];
    }
    const uint32_t kstar = prefix;
    const int need = kr;   // entries equal to kstar to keep (the earliest ones)
    const int R = (n + kEpiThreads - 1) / kEpiThreads;
    const unsigned lt = (1u << lane) - 1u;
    float sv[kMaxR];
    int iv[kMaxR];
    unsigned tb[kMaxR];
    int nt = 0;
#pragma unroll
    for (int r = 0; r < kMaxR; ++r) {
        tb[r] = 0;
        sv[r] = 0.f;
        iv[r] = 0;
        if (r < R) {
            const int e = ew * 32 * R + r * 32 + lane;
            bool tie = false;
            if (e < n) {
                sv[r] = cs[e];
                iv[r] = ci[e];
                tie = fkey(sv[r]) == kstar;
            }
            tb[r] = __ballot_sync(kFull, tie);
            nt += __popc(tb[r]);
        }
    }
    if (lane == 0) scr[8 + ew] = nt;
    ptx::named_bar_sync(1, kEpiThreads);
    int run = 0;
    for (int w2 = 0; w2 < ew; ++w2) run += scr[8 + w2];
    unsigned kb[kMaxR];
    int nk = 0;
#pragma unroll
    for (int r = 0; r < kMaxR; ++r) {
        kb[r] = 0;
        if (r < R) {
            const int e = ew * 32 * R + r * 32 + lane;
            const uint32_t key = fkey(sv[r]);
            const bool tie = (tb[r] >> lane) & 1u;
            const int trank = run + __popc(tb[r] & lt);
            const bool keep = (e < n) && (key > kstar || (tie && trank < need));
            run += __popc(tb[r]);
            kb[r] = __ballot_sync(kFull, keep);
            nk += __popc(kb[r]);
        }
    }
    if (lane == 0) scr[16 + ew] = nk;
    ptx::named_bar_sync(1, kEpiThreads);
    int pos = 0;
    for (int w2 = 0; w2 < ew; ++w2) pos += scr[16 + w2];
#pragma unroll
    for (int r = 0; r < kMaxR; ++r) {
        if (r < R) {
            if ((kb[r] >> lane) & 1u) {
                const int d = pos + __popc(kb[r] & lt);
                cs[d] = sv[r];
                ci[d] = iv[r];
            }
            pos += __popc(kb[r]);
        }
    }
    if (etid == 0) *thr_out = kstar;
    ptx::named_bar_sync(1, kEpiThreads);
}

template <int H>
__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_pk,
                 const __grid_constant__ Params p)
{
    constexpr int QT = kBN / H;   // queries per tile
    constexpr int QW = QT / 2;    // queries per epilogue warp
    constexpr int NSL = QT > 32 ? 2 : 1;

    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const Layout &L = p.L;
    const uint32_t sbase = ptx::smem_u32(smem);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    const int S = L.stages;
    TileInfo *ti_slots = reinterpret_cast<TileInfo *>(smem + L.ti_off);
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + L.misc_off);   // [0] tmem, [1] abort
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(BQ_FULL), 1);
        ptx::mbar_init(bar(BQ_EMPTY), 1);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(BTM_FULL + i), 1);
            ptx::mbar_init(bar(BTM_EMPTY + i), kEpiWarps);
            ptx::mbar_init(bar(BTI_FULL + i), 1);
            ptx::mbar_init(bar(BTI_EMPTY + i), 1 + kEpiWarps);
        }
        ptx::mbar_init(bar(BDRAIN), 1);
        for (int s = 0; s < S; ++s) {
            ptx::mbar_init(bar(BPK_FULL + s), 1);
            ptx::mbar_init(bar(BPK_FULL + S + s), 1);
        }
        misc[1] = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_u32(&misc[0]), kTmemCols);
        ptx::tmem_relinquish();
        ptx::tc_fence_before();
    }
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = misc[0];
    Sync sy{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.ws + WS_STATUS};

    auto tile_info = [&](int tile) {
        TileInfo t;
        const int2 e = reinterpret_cast<const int2 *>(p.ws + WS_TABLE_INTS)[tile];
        t.t0 = e.x;
        if (p.cu_seqlens != nullptr) {
            t.doc_start = p.cu_seqlens[e.y];
            t.doc_end = p.cu_seqlens[e.y + 1];
            t.pool_base = p.cu_pools[e.y];
        } else {
            t.doc_start = 0;
            t.doc_end = p.T;
            t.pool_base = 0;
        }
        return t;
    };

    if (warp == 0) {
        // ---------------- TMA producer + scheduler ----------------
        if (lane == 0) {
            ptx::tma_prefetch_desc(&tm_q);
            ptx::tma_prefetch_desc(&tm_pk);
            const int ntiles = *reinterpret_cast<volatile int *>(p.ws + WS_NTILES);
            const int celem = p.fp8 ? 128 : 64;   // elements per 128-byte chunk
            int stage = 0;
            uint32_t ph = 0, qe_ph = 0;
            uint32_t issued_mask = 0, issued_ph = 0;   // last issued phase per stage
            bool q_issued = false;
            uint32_t q_issued_ph = 0;
            for (int it = 0;; ++it) {
                const int slot = it & 1;
                const uint32_t tph = (it >> 1) & 1;
                if (!wait_bar(bar(BTI_EMPTY + slot), tph ^ 1, sy)) break;
                const int tile = atomicAdd(p.ws + WS_COUNTER, 1);
                TileInfo t;
                if (tile >= ntiles) {
                    t.t0 = -1;
                    t.doc_start = t.doc_end = t.pool_base = 0;
                } else {
                    t = tile_info(tile);
                }
                ti_slots[slot] = t;   // published by the mbarrier arrive (release)
                ptx::mbar_arrive(bar(BTI_FULL + slot));
                if (t.t0 < 0) break;
                const int npt = pool_tiles_of(t, QT, p.kp);
                if (npt == 0) continue;
                if (!wait_bar(bar(BQ_EMPTY), qe_ph ^ 1, sy)) break;
                qe_ph ^= 1;
                ptx::mbar_arrive_expect_tx(bar(BQ_FULL), p.q_tx);
                for (int c = 0; c < L.n_kchunks; ++c)
                    ptx::tma_load_2d(sbase + L.q_off + c * L.q_chunk, &tm_q, bar(BQ_FULL),
                                     c * celem, t.t0 * H);
                q_issued = true;
                q_issued_ph = qe_ph ^ 1;
                bool ok = true;
                for (int i = 0; i < npt; ++i) {
                    if (!wait_bar(bar(BPK_FULL + S + stage), ph ^ 1, sy)) { ok = false; break; }
                    ptx::mbar_arrive_expect_tx(bar(BPK_FULL + stage), p.pk_tx);
                    const uint32_t dst = sbase + L.pk_off + stage * L.pk_stage;
                    for (int c = 0; c < L.n_kchunks; ++c)
                        ptx::tma_load_2d(dst + c * L.pk_chunk, &tm_pk, bar(BPK_FULL + stage),
                                         c * celem, t.pool_base + i * kBM);
                    issued_mask |= 1u << stage;
                    issued_ph = (issued_ph & ~(1u << stage)) | (ph << stage);
                    if (++stage == S) { stage = 0; ph ^= 1; }
                }
                if (!ok) break;
            }
            // let our own copies land before the CTA can exit (bounded)
            const uint64_t t0 = ptx::globaltimer();
            for (int s = 0; s < S; ++s) {
                if (!(issued_mask & (1u << s))) continue;
                while (!ptx::mbar_try_wait(bar(BPK_FULL + s), (issued_ph >> s) & 1u))
                    if (ptx::globaltimer() - t0 > kTimeoutNs) break;
            }
            if (q_issued) {
                // q_full completes once per issue; parity of the last issue
                while (!ptx::mbar_try_wait(bar(BQ_FULL), q_issued_ph))
                    if (ptx::globaltimer() - t0 > kTimeoutNs) break;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t ph = 0, qf_ph = 0, acc_ph = 0;
            bool any = false;
            for (int it = 0;; ++it) {
                const int slot = it & 1;
                const uint32_t tph = (it >> 1) & 1;
                if (!wait_bar(bar(BTI_FULL + slot), tph, sy)) break;
                const TileInfo t = ti_slots[slot];   // after the acquiring wait
                ptx::mbar_arrive(bar(BTI_EMPTY + slot));
                if (t.t0 < 0) break;
                const int npt = pool_tiles_of(t, QT, p.kp);
                if (npt == 0) continue;
                if (!wait_bar(bar(BQ_FULL), qf_ph, sy)) break;
                qf_ph ^= 1;
                bool ok = true;
                for (int i = 0; i < npt; ++i) {
                    if (!wait_bar(bar(BTM_EMPTY + acc), acc_ph ^ 1, sy)) { ok = false; break; }
                    if (!wait_bar(bar(BPK_FULL + stage), ph, sy)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * kAccCols;
                    const uint32_t a0 = sbase + L.pk_off + stage * L.pk_stage;
                    const uint32_t b0 = sbase + L.q_off;
                    for (int c = 0; c < L.n_kchunks; ++c) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = ptx::smem_desc_sw128(a0 + c * L.pk_chunk + kk * 32);
                            const uint64_t bd = ptx::smem_desc_sw128(b0 + c * L.q_chunk + kk * 32);
                            const uint32_t accum = (c | kk) != 0;
                            if (p.fp8) ptx::mma_fp8(d_tmem, ad, bd, p.idesc, accum);
                            else ptx::mma_bf16(d_tmem, ad, bd, p.idesc, accum);
                        }
                    }
                    ptx::mma_commit(bar(BPK_FULL + S + stage));
                    ptx::mma_commit(bar(BTM_FULL + acc));
                    any = true;
                    if (++stage == S) { stage = 0; ph ^= 1; }
                    if (++acc == 2) { acc = 0; acc_ph ^= 1; }
                }
                ptx::mma_commit(bar(BQ_EMPTY));
                if (!ok) break;
            }
            if (any) {
                // every MMA issued by this thread has completed before teardown
                ptx::mma_commit(bar(BDRAIN));
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(bar(BDRAIN), 0))
                    if (ptx::globaltimer() - t0 > kTimeoutNs) break;
            }
        }
    } else if (warp >= 4) {
        // ---------------- epilogue ----------------
        const int ew = warp - 4;
        const int qr = warp & 3;            // TMEM lane quarter
        const int hf = ew >> 2;             // which half of the 256 columns
        const int etid = threadIdx.x - 128;
        float *ws = reinterpret_cast<float *>(smem + L.ws_off) + ew * 128;
        int *hist = reinterpret_cast<int *>(smem + L.hist_off);
        int *cnts = reinterpret_cast<int *>(smem + L.cnt_off);
        int *scr = reinterpret_cast<int *>(smem + L.scr_off);
        uint32_t *thr_s = reinterpret_cast<uint32_t *>(smem + L.thr_off);
        float *cs = reinterpret_cast<float *>(smem + L.cs_off);
        int *ci = reinterpret_cast<int *>(smem + L.ci_off);
        const int C = L.C;
        const int Kp = p.Kp;
        const unsigned lt = (1u << lane) - 1u;
        int acc = 0, tile_seq = 0;
        uint32_t acc_ph = 0;
        for (int it = 0;; ++it) {
            const int slot = it & 1;
            const uint32_t tph = (it >> 1) & 1;
            if (!wait_bar_warp(bar(BTI_FULL + slot), tph, sy)) break;
            const TileInfo t = ti_slots[slot];
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(BTI_EMPTY + slot));
            if (t.t0 < 0) break;
            const int tau0 = t.t0 - t.doc_start;
            const int nq = min(QT, t.doc_end - t.t0);
            const int npt = pool_tiles_of(t, QT, p.kp);

            // this warp's head weights (128 contiguous floats), w * q_scale in FP8 mode
            __syncwarp();
            {
                const int c0 = lane * 4;
                const int qi = hf * QW + c0 / H;
                float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
                if (qi < nq) {
                    const int64_t off = static_cast<int64_t>(t.t0 + hf * QW) * H + c0;
                    v = *reinterpret_cast<const float4 *>(p.w + off);
                    if (p.fp8) {
                        const float4 s4 = *reinterpret_cast<const float4 *>(p.q_scale + off);
                        v.x *= s4.x; v.y *= s4.y; v.z *= s4.z; v.w *= s4.w;
                    }
                }
                *reinterpret_cast<float4 *>(ws + c0) = v;
            }
            __syncwarp();
            const float4 *ws4 = reinterpret_cast<const float4 *>(ws);

            uint32_t thr[QW];
            int nc[QW];
#pragma unroll
            for (int j = 0; j < QW; ++j) {
                thr[j] = 0u;
                nc[j] = (tau0 + hf * QW + j + 1) / p.kp;
            }
            int tot[NSL];
#pragma unroll
            for (int sl = 0; sl < NSL; ++sl) tot[sl] = 0;
            if (etid < QT) thr_s[etid] = 0u;
            bool aborted = false;

            for (int i = 0; i < npt; ++i) {
                if (!wait_bar_warp(bar(BTM_FULL + acc), acc_ph, sy)) { aborted = true; break; }
                ptx::tc_fence_after();
                const uint32_t tb = tmem_base + (static_cast<uint32_t>(qr * 32) << 16) +
                                    acc * kAccCols + hf * 128;
                float a0[QW], a1[QW];
#pragma unroll
                for (int j = 0; j < QW; ++j) { a0[j] = 0.f; a1[j] = 0.f; }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v0[32], v1[32];
                    ptx::tmem_ld32(tb + half * 64, v0);
                    ptx::tmem_ld32(tb + half * 64 + 32, v1);
                    ptx::tmem_ld_wait();
                    if (half == 1) {
                        ptx::tc_fence_before();
                        __syncwarp();
                        if (lane == 0) ptx::mbar_arrive(bar(BTM_EMPTY + acc));
                    }
#pragma unroll
                    for (int cc = 0; cc < 2; ++cc) {
                        const uint32_t *v = cc ? v1 : v0;
#pragma unroll
                        for (int x = 0; x < 32; x += 4) {
                            const int col = half * 64 + cc * 32 + x;
                            const int j = col / H;
                            const float4 w4 = ws4[col >> 2];
                            a0[j] = fmaf(fmaxf(__uint_as_float(v[x + 0]), 0.f), w4.x, a0[j]);
                            a1[j] = fmaf(fmaxf(__uint_as_float(v[x + 1]), 0.f), w4.y, a1[j]);
                            a0[j] = fmaf(fmaxf(__uint_as_float(v[x + 2]), 0.f), w4.z, a0[j]);
                            a1[j] = fmaf(fmaxf(__uint_as_float(v[x + 3]), 0.f), w4.w, a1[j]);
                        }
                    }
                }
                if (++acc == 2) { acc = 0; acc_ph ^= 1; }

                const int pool_local = i * kBM + qr * 32 + lane;
                const int pool_g = t.pool_base + pool_local;
                float sk = 1.f;
                if (p.fp8 && pool_g < p.P_total) sk = p.pk_scale[pool_g];
                float s[QW];
#pragma unroll
                for (int j = 0; j < QW; ++j) {
                    float v = a0[j] + a1[j];
                    if (p.fp8) v *= sk;
                    s[j] = (v == 0.f) ? 0.f : v;   // fold -0 into +0
                }

                if (p.mode == 1) {   // dense scores (test/debug)
#pragma unroll
                    for (int j = 0; j < QW; ++j) {
                        const int qi = hf * QW + j;
                        if (qi < nq && pool_local < nc[j])
                            p.scores[static_cast<int64_t>(t.t0 + qi) * p.P_total + pool_g] = s[j];
                    }
                    continue;
                }

                // ordered append of survivors of the threshold filter
                const int par = (tile_seq & 1) * QT * 4;
                ++tile_seq;
                unsigned bal[QW];
#pragma unroll
                for (int j = 0; j < QW; ++j) {
                    const int qi = hf * QW + j;
                    const bool ps = (qi < nq) && (pool_local < nc[j]) && (fkey(s[j]) > thr[j]);
                    bal[j] = __ballot_sync(kFull, ps);
                    if (lane == 0) cnts[par + qi * 4 + qr] = __popc(bal[j]);
                }
                ptx::named_bar_sync(1, kEpiThreads);
#pragma unroll
                for (int j = 0; j < QW; ++j) {
                    const int qi = hf * QW + j;
                    const int4 c4 = *reinterpret_cast<const int4 *>(&cnts[par + qi * 4]);
                    const int tq = __shfl_sync(kFull, (NSL > 1 && qi >= 32) ? tot[NSL - 1] : tot[0],
                                               qi & 31);
                    const int pre = (qr > 0 ? c4.x : 0) + (qr > 1 ? c4.y : 0) + (qr > 2 ? c4.z : 0);
                    if ((bal[j] >> lane) & 1u) {
                        const int d = qi * C + tq + pre + __popc(bal[j] & lt);
                        cs[d] = s[j];
                        ci[d] = pool_g;
                    }
                }
                bool over = false;
#pragma unroll
                for (int sl = 0; sl < NSL; ++sl) {
                    const int qi = lane + 32 * sl;
                    if (qi < QT) {
                        const int4 c4 = *reinterpret_cast<const int4 *>(&cnts[par + qi * 4]);
                        tot[sl] += c4.x + c4.y + c4.z + c4.w;
                        over |= tot[sl] > C - kBM;
                    }
                }
                if (__any_sync(kFull, over)) {
                    ptx::named_bar_sync(1, kEpiThreads);
                    for (int qi = 0; qi < QT; ++qi) {
                        const int sl = qi >> 5;
                        const int tq = __shfl_sync(kFull, sl ? tot[NSL - 1] : tot[0], qi & 31);
                        if (tq > C - kBM) {
                            select_topk(cs + qi * C, ci + qi * C, tq, Kp, etid, hist, scr,
                                        &thr_s[qi]);
                            if (lane == (qi & 31)) {
                                if (sl) tot[NSL - 1] = Kp;
                                else tot[0] = Kp;
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < QW; ++j) thr[j] = thr_s[hf * QW + j];
                }
            }
            if (aborted) break;
            if (p.mode == 1) continue;

            // final selection and output, one query at a time
            ptx::named_bar_sync(1, kEpiThreads);
            for (int qi = 0; qi < nq; ++qi) {
                const int sl = qi >> 5;
                int tq = __shfl_sync(kFull, sl ? tot[NSL - 1] : tot[0], qi & 31);
                if (tq > Kp) {
                    select_topk(cs + qi * C, ci + qi * C, tq, Kp, etid, hist, scr, &thr_s[qi]);
                    tq = Kp;
                }
                const int64_t row = static_cast<int64_t>(t.t0 + qi) * Kp;
                for (int e = etid; e < Kp; e += kEpiThreads) {
                    const bool v = e < tq;
                    p.pool_idx[row + e] = v ? ci[qi * C + e] : -1;
                    p.pool_score[row + e] = v ? cs[qi * C + e] : -INFINITY;
                }
            }
            ptx::named_bar_sync(1, kEpiThreads);
        }
    }

    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// Longest-first query-tile table.  Tile (d, i) covers document-local queries
// [i*QT, min((i+1)*QT, L_d)); its rank orders tiles by descending i (more
// causal pools first), ties by document.  Also validates cu_seqlens and
// resets the tile counter and the status word.
__global__ void schedule_kernel(const int32_t *cu, int n_docs, int T, int QT, int max_tiles,
                                int *ws)
{
    __shared__ int s_ok, s_ntiles;
    if (threadIdx.x == 0) {
        int ok = 1, nt = 0;
        if (cu != nullptr) {
            if (cu[0] != 0 || cu[n_docs] != T) ok = 0;
            for (int d = 0; d < n_docs && ok; ++d) {
                const int L = cu[d + 1] - cu[d];
                if (L < 0) ok = 0;
                else nt += (L + QT - 1) / QT;
            }
        } else {
            nt = (T + QT - 1) / QT;
        }
        if (nt > max_tiles) ok = 0;
        s_ok = ok;
        s_ntiles = ok ? nt : 0;
        ws[WS_COUNTER] = 0;
        ws[WS_STATUS] = ok ? 0 : KPOOL_STATUS_BAD_SEQLENS;
        ws[WS_NTILES] = s_ntiles;
    }
    __syncthreads();
    const int nt = s_ntiles;
    int2 *table = reinterpret_cast<int2 *>(ws + WS_TABLE_INTS);
    for (int g = threadIdx.x; g < nt; g += blockDim.x) {
        if (cu == nullptr) {
            const int ntl = nt;
            table[ntl - 1 - g] = make_int2(g * QT, 0);
            continue;
        }
        int d = 0, acc = 0;
        for (; d < n_docs; ++d) {
            const int n = (cu[d + 1] - cu[d] + QT - 1) / QT;
            if (g < acc + n) break;
            acc += n;
        }
        const int i = g - acc;
        int rank = 0;
        for (int d2 = 0; d2 < n_docs; ++d2) {
            const int n = (cu[d2 + 1] - cu[d2] + QT - 1) / QT;
            rank += max(0, n - i - 1);
            if (d2 < d && n > i) ++rank;
        }
        table[rank] = make_int2(cu[d] + i * QT, d);
    }
}

__global__ void fill_kernel(uint32_t *a, int64_t n, uint32_t va, uint32_t *b, uint32_t vb)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        a[i] = va;
        if (b) b[i] = vb;
    }
}

// ---- host side -------------------------------------------------------------

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    });
    return fn;
}

int encode_2d(CUtensorMap *m, const void *base, int fp8, uint64_t cols, uint64_t rows,
              uint32_t box_rows)
{
    EncodeTiledFn enc = get_encode();
    if (!enc) return fail(KPOOL_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    const uint32_t esize = fp8 ? 1 : 2;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {cols * esize};
    cuuint32_t box[2] = {128 / esize, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                     const_cast<void *>(base), gdim, gstride, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KPOOL_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return KPOOL_OK;
}

template <int H>
int launch_h(const ScoreArgs &a, const Layout &L, const CUtensorMap &mq, const CUtensorMap &mpk,
             const Params &prm, int grid, cudaStream_t s)
{
    const int smem = static_cast<int>(L.total) + 1024;
    KPOOL_CUDA_CHECK(cudaFuncSetAttribute(score_kernel<H>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    score_kernel<H><<<grid, kThreads, smem, s>>>(mq, mpk, prm);
    KPOOL_CUDA_CHECK(cudaGetLastError());
    (void)a;
    return KPOOL_OK;
}

// Scratch of the allocation-free entry point (kpool_score_topk_noalloc): the
// workspace header and the query-tile table for up to kNoAllocMaxTiles tiles,
// 1 MiB + 256 B, held by every device that loads the library.  The schedule
// kernel rewrites the counter, status word, tile count and table on every
// call, so no state from an earlier call is read.
constexpr size_t kNoAllocWords = WS_TABLE_INTS + 2 * static_cast<size_t>(kNoAllocMaxTiles);
static __device__ __align__(256) int g_noalloc_scratch[kNoAllocWords];

}  // namespace

int noalloc_scratch(int **ptr, size_t *bytes, int64_t *max_tiles)
{
    static std::mutex mu;
    static std::vector<int *> addr;   // device address of the scratch, per device
    int dev = 0;
    KPOOL_CUDA_CHECK(cudaGetDevice(&dev));
    std::lock_guard<std::mutex> lk(mu);
    if (static_cast<int>(addr.size()) <= dev) addr.resize(dev + 1, nullptr);
    if (addr[dev] == nullptr) {
        // The array's name is a host-side stand-in; the kernel needs the device
        // address, looked up once per device with that device current.
        void *p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || p == nullptr)
            return fail(KPOOL_ERR_CUDA, "cudaGetSymbolAddress(no-alloc scratch) failed: %s",
                        cudaGetErrorString(e));
        addr[dev] = static_cast<int *>(p);
    }
    *ptr = addr[dev];
    *bytes = kNoAllocWords * sizeof(int);
    *max_tiles = kNoAllocMaxTiles;
    return KPOOL_OK;
}

size_t score_workspace_bytes(int64_t T, int H, int n_docs)
{
    const int64_t QT = qt_of(H);
    const int64_t max_tiles = (T + QT - 1) / QT + n_docs;
    size_t b = WS_TABLE_INTS * 4 + static_cast<size_t>(max_tiles) * 8;
    return (b + 255) & ~static_cast<size_t>(255);
}

int score_capacity(int H, int D, int fp8)
{
    const Layout L = make_layout(H, D, fp8);
    return L.C;
}

int run_score(const ScoreArgs &a, cudaStream_t s)
{
    const int QT = qt_of(a.H);
    const int64_t max_tiles = (a.T + QT - 1) / QT + a.n_docs;
    if (a.T == 0) return KPOOL_OK;
    if (a.mode == 1) {
        const int64_t n = a.T * a.P_total;
        if (n > 0) {
            fill_kernel<<<1024, 256, 0, s>>>(reinterpret_cast<uint32_t *>(a.scores), n,
                                             0xFF800000u, nullptr, 0u);
            KPOOL_CUDA_CHECK(cudaGetLastError());
        }
    }
    if (a.P_total == 0) {
        // no complete pool anywhere: every row selects nothing
        if (a.mode == 0) {
            fill_kernel<<<1024, 256, 0, s>>>(reinterpret_cast<uint32_t *>(a.pool_idx),
                                             a.T * a.Kp, 0xFFFFFFFFu,
                                             reinterpret_cast<uint32_t *>(a.pool_score),
                                             0xFF800000u);
            KPOOL_CUDA_CHECK(cudaGetLastError());
        }
        // still validate the layout / reset the status word
        schedule_kernel<<<1, 1024, 0, s>>>(a.cu_seqlens, a.n_docs, static_cast<int>(a.T), QT,
                                           static_cast<int>(max_tiles), a.ws);
        KPOOL_CUDA_CHECK(cudaGetLastError());
        return KPOOL_OK;
    }
    const Layout L = make_layout(a.H, a.D, a.fp8);
    CUtensorMap mq, mpk;
    int rc = encode_2d(&mq, a.q, a.fp8, static_cast<uint64_t>(a.D),
                       static_cast<uint64_t>(a.T) * a.H, kBN);
    if (rc) return rc;
    rc = encode_2d(&mpk, a.pk, a.fp8, static_cast<uint64_t>(a.D), static_cast<uint64_t>(a.P_total),
                   kBM);
    if (rc) return rc;

    Params prm{};
    prm.w = a.w;
    prm.q_scale = a.q_scale;
    prm.pk_scale = a.pk_scale;
    prm.cu_seqlens = a.cu_seqlens;
    prm.cu_pools = a.cu_pools;
    prm.n_docs = a.n_docs;
    prm.T = static_cast<int>(a.T);
    prm.P_total = static_cast<int>(a.P_total);
    prm.kp = a.kpool;
    prm.Kp = a.Kp;
    prm.fp8 = a.fp8;
    prm.mode = a.mode;
    prm.pool_idx = a.pool_idx;
    prm.pool_score = a.pool_score;
    prm.scores = a.scores;
    prm.ws = a.ws;
    prm.q_tx = L.n_kchunks * L.q_chunk;
    prm.pk_tx = L.n_kchunks * L.pk_chunk;
    prm.idesc = ptx::make_idesc(a.fp8 ? 0u : 1u, kBM, kBN);
    prm.L = L;

    schedule_kernel<<<1, 1024, 0, s>>>(a.cu_seqlens, a.n_docs, static_cast<int>(a.T), QT,
                                       static_cast<int>(max_tiles), a.ws);
    KPOOL_CUDA_CHECK(cudaGetLastError());
    const int grid = static_cast<int>(std::min<int64_t>(num_sms(), max_tiles));
    switch (a.H) {
    case 4: return launch_h<4>(a, L, mq, mpk, prm, grid, s);
    case 8: return launch_h<8>(a, L, mq, mpk, prm, grid, s);
    case 16: return launch_h<16>(a, L, mq, mpk, prm, grid, s);
    case 32: return launch_h<32>(a, L, mq, mpk, prm, grid, s);
    case 64: return launch_h<64>(a, L, mq, mpk, prm, grid, s);
    case 128: return launch_h<128>(a, L, mq, mpk, prm, grid, s);
    default: return fail(KPOOL_ERR_UNSUPPORTED, "H=%d not built", a.H);
    }
}

}  // namespace kpool
