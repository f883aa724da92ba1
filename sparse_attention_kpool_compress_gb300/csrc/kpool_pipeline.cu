// The whole indexer pass from host buffers, with the copies overlapped
// (Megatron-LM PR "GLM5.3 Flash (KDA + mHC + KPool DSA) support + FP8",
// Changes section 3: compression, pool top-k, expansion with the causal tail,
// packed THD; the FP8 input path of the same section).
//
// Keys (k, gate, ape) are copied and compressed first.  The query rows are then
// processed in chunks on three streams: copy-in of chunk c+1, scoring and
// expansion of chunk c, and copy-out of chunk c-1 run at the same time, with
// two device buffers for the copied q/w rows and two for the token indices.
// Chunks ramp up in size at the start and down at the end (chunk_bounds).  (A
// second compute stream, letting consecutive chunks' scoring kernels overlap,
// was measured slower on long sequences and is not used.)
// A chunk is scored as positioned queries over the global pooled keys (each
// document's rows of the chunk start at their own position), so every query
// gets exactly the result of the unchunked pass: scores and selections are per
// query and do not depend on how queries share a tile.
#include <algorithm>
#include <vector>

#include "kpool_internal.h"

namespace kpool {
namespace {

constexpr int64_t kDefaultChunkRows = 16384;

// Chunk [r0, r1) of the query rows: document d's rows in it are
// [cu_q[d], cu_q[d+1]) (chunk-local), the first at document position q_pos[d].
__global__ void chunk_layout_kernel(const int32_t *__restrict__ cu, int n_docs, int64_t r0,
                                    int64_t r1, int32_t *__restrict__ cu_q,
                                    int32_t *__restrict__ q_pos)
{
    for (int d = blockIdx.x * blockDim.x + threadIdx.x; d <= n_docs;
         d += gridDim.x * blockDim.x) {
        const int64_t s = cu[d];
        const int64_t c = s < r0 ? r0 : (s > r1 ? r1 : s);
        cu_q[d] = static_cast<int32_t>(c - r0);
        if (d < n_docs) q_pos[d] = static_cast<int32_t>((s < r0 ? r0 : s) - s);
    }
}

// Document offsets {0, T} of a single sequence.
__global__ void one_sequence_kernel(int32_t *cu, int32_t T)
{
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        cu[0] = 0;
        cu[1] = T;
    }
}

// Sticky status of the whole pass: the per-chunk status word ORed in.
__global__ void status_accum_kernel(const int *__restrict__ ws_status, int *__restrict__ sticky)
{
    if (blockIdx.x == 0 && threadIdx.x == 0) *sticky |= *ws_status;
}

struct PipeStreams {
    cudaStream_t in = nullptr, cmp = nullptr, out = nullptr;
    cudaEvent_t start = nullptr, keys = nullptr, ev_in[2] = {}, ev_cmp[2] = {}, ev_out[2] = {};
    bool ok = false;
};

// Streams and events of the calling host thread on the current device, created
// on first use and kept for the life of the thread (one host thread drives one
// pipeline at a time; separate threads get separate streams).
int pipe_streams(PipeStreams **out)
{
    thread_local std::vector<PipeStreams> per_device;
    int dev = 0;
    KPOOL_CUDA_CHECK(cudaGetDevice(&dev));
    if (static_cast<int>(per_device.size()) <= dev) per_device.resize(dev + 1);
    PipeStreams &p = per_device[dev];
    if (!p.ok) {
        KPOOL_CUDA_CHECK(cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking));
        KPOOL_CUDA_CHECK(cudaStreamCreateWithFlags(&p.cmp, cudaStreamNonBlocking));
        KPOOL_CUDA_CHECK(cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking));
        cudaEvent_t *evs[] = {&p.start, &p.keys, &p.ev_in[0], &p.ev_in[1], &p.ev_cmp[0],
                              &p.ev_cmp[1], &p.ev_out[0], &p.ev_out[1]};
        for (cudaEvent_t *e : evs) KPOOL_CUDA_CHECK(cudaEventCreateWithFlags(e, cudaEventDisableTiming));
        p.ok = true;
    }
    *out = &p;
    return KPOOL_OK;
}

size_t align256(size_t b) { return (b + 255) & ~static_cast<size_t>(255); }

// Chunk boundaries over [0, T): sizes ramp up R/8, R/4, R/2 at the start and
// down R/2, R/4, R/8 at the end, R in between, so that the first copy-in and
// the last copy-out (which nothing overlaps) are short.
std::vector<int64_t> chunk_bounds(int64_t T, int64_t R)
{
    std::vector<int64_t> head, tail;
    int64_t lo = 0, hi = T;
    for (int64_t s = std::max<int64_t>(R / 8, 1); s < R && hi - lo >= 2 * s; s *= 2) {
        head.push_back(s);
        tail.push_back(s);
        lo += s;
        hi -= s;
    }
    std::vector<int64_t> b{0};
    for (int64_t s : head) b.push_back(b.back() + s);
    while (hi - b.back() > 0) b.push_back(std::min(hi, b.back() + R));
    for (auto it = tail.rbegin(); it != tail.rend(); ++it) b.push_back(b.back() + *it);
    return b;
}

// Scratch layout (byte offsets, each 256-aligned).  The first 256 bytes are a
// header whose int 1 is the sticky status (read by kpool_read_status).
struct PipeLayout {
    size_t ws, cu, cu_pools, cu_q, q_pos, k, gate, ape, pk, pk8, pks;
    size_t qbuf[2], wbuf[2], tok[2], q8, qs, idx, score;
    size_t ws_bytes, total;
};

PipeLayout pipe_layout(int64_t T, int H, int D, int n_docs, int kpool, int Kp, int fp8,
                       int64_t R, int64_t P)
{
    PipeLayout L{};
    const int64_t W = static_cast<int64_t>(Kp) * kpool + kpool - 1;
    size_t off = 256;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off += align256(bytes);
        return at;
    };
    L.ws_bytes = score_workspace_split_bytes(R, H, n_docs, Kp);
    L.ws = take(L.ws_bytes);
    L.cu = take(static_cast<size_t>(n_docs + 1) * 4);
    L.cu_pools = take(static_cast<size_t>(n_docs + 1) * 4);
    L.cu_q = take(static_cast<size_t>(n_docs + 1) * 4);
    L.q_pos = take(static_cast<size_t>(n_docs) * 4);
    L.k = take(static_cast<size_t>(T) * D * 2);
    L.gate = take(static_cast<size_t>(T) * D * 2);
    L.ape = take(static_cast<size_t>(kpool) * D * 4);
    L.pk = take(static_cast<size_t>(P) * D * 2);
    L.pk8 = fp8 ? take(static_cast<size_t>(P) * D) : 0;
    L.pks = fp8 ? take(static_cast<size_t>(P) * 4) : 0;
    for (int b = 0; b < 2; ++b) {
        L.qbuf[b] = take(static_cast<size_t>(R) * H * D * 2);
        L.wbuf[b] = take(static_cast<size_t>(R) * H * 4);
        L.tok[b] = take(static_cast<size_t>(R) * W * 4);
    }
    L.q8 = fp8 ? take(static_cast<size_t>(R) * H * D) : 0;
    L.qs = fp8 ? take(static_cast<size_t>(R) * H * 4) : 0;
    L.idx = take(static_cast<size_t>(R) * Kp * 4);
    L.score = take(static_cast<size_t>(R) * Kp * 4);
    L.total = off;
    return L;
}

}  // namespace

size_t pipeline_scratch_bytes(int64_t T, int H, int D, int n_docs, int kpool, int index_topk,
                              int fp8, int64_t chunk_rows, int64_t P_total)
{
    const int64_t R = chunk_rows > 0 ? std::min<int64_t>(chunk_rows, std::max<int64_t>(T, 1))
                                     : std::min<int64_t>(kDefaultChunkRows, std::max<int64_t>(T, 1));
    return pipe_layout(T, H, D, n_docs, kpool, index_topk / kpool, fp8, R, P_total).total;
}

int run_pipeline(const PipelineArgs &a, cudaStream_t stream)
{
    const int64_t T = a.T;
    const int Kp = a.index_topk / a.kpool;
    const int64_t W = static_cast<int64_t>(Kp) * a.kpool + a.kpool - 1;
    const int64_t R = a.chunk_rows > 0 ? std::min<int64_t>(a.chunk_rows, std::max<int64_t>(T, 1))
                                       : std::min<int64_t>(kDefaultChunkRows,
                                                           std::max<int64_t>(T, 1));
    const PipeLayout L = pipe_layout(T, a.H, a.D, a.n_docs, a.kpool, Kp, a.fp8, R, a.P_total);
    if (a.scratch_bytes < L.total)
        return fail(KPOOL_ERR_WORKSPACE, "scratch needs %zu bytes (got %zu)", L.total,
                    a.scratch_bytes);
    uint8_t *base = static_cast<uint8_t *>(a.scratch);
    auto at = [&](size_t off) { return static_cast<void *>(base + off); };
    int *sticky = reinterpret_cast<int *>(base);
    int *ws = static_cast<int *>(at(L.ws));
    int32_t *cu = static_cast<int32_t *>(at(L.cu));
    int32_t *cu_pools = static_cast<int32_t *>(at(L.cu_pools));
    int32_t *cu_q = static_cast<int32_t *>(at(L.cu_q));
    int32_t *q_pos = static_cast<int32_t *>(at(L.q_pos));

    PipeStreams *ps = nullptr;
    int rc = pipe_streams(&ps);
    if (rc) return rc;
    cudaStream_t s_in = ps->in, s_cmp = ps->cmp, s_out = ps->out;
    KPOOL_CUDA_CHECK(cudaEventRecord(ps->start, stream));
    KPOOL_CUDA_CHECK(cudaStreamWaitEvent(s_in, ps->start, 0));
    KPOOL_CUDA_CHECK(cudaStreamWaitEvent(s_cmp, ps->start, 0));
    KPOOL_CUDA_CHECK(cudaStreamWaitEvent(s_out, ps->start, 0));

    // keys: copy, pool counts, compression (and the FP8 pooled keys)
    KPOOL_CUDA_CHECK(cudaMemsetAsync(sticky, 0, 256, s_cmp));
    if (a.cu_seqlens_host != nullptr) {
        KPOOL_CUDA_CHECK(cudaMemcpyAsync(cu, a.cu_seqlens_host,
                                         (a.n_docs + 1) * sizeof(int32_t),
                                         cudaMemcpyHostToDevice, s_in));
    } else {
        one_sequence_kernel<<<1, 32, 0, s_in>>>(cu, static_cast<int32_t>(T));
        KPOOL_CUDA_CHECK(cudaGetLastError());
    }
    KPOOL_CUDA_CHECK(cudaMemcpyAsync(at(L.k), a.k, static_cast<size_t>(T) * a.D * 2,
                                     cudaMemcpyHostToDevice, s_in));
    KPOOL_CUDA_CHECK(cudaMemcpyAsync(at(L.gate), a.gate, static_cast<size_t>(T) * a.D * 2,
                                     cudaMemcpyHostToDevice, s_in));
    KPOOL_CUDA_CHECK(cudaMemcpyAsync(at(L.ape), a.ape, static_cast<size_t>(a.kpool) * a.D * 4,
                                     cudaMemcpyHostToDevice, s_in));
    KPOOL_CUDA_CHECK(cudaEventRecord(ps->keys, s_in));
    KPOOL_CUDA_CHECK(cudaStreamWaitEvent(s_cmp, ps->keys, 0));
    KPOOL_CUDA_CHECK(launch_cu_pools(cu, a.n_docs, a.kpool, cu_pools, s_cmp));
    KPOOL_CUDA_CHECK(launch_compress(at(L.k), at(L.gate), static_cast<const float *>(at(L.ape)),
                                     cu, cu_pools, a.n_docs, T, a.D, a.kpool, a.P_total,
                                     at(L.pk), a.fp8 ? static_cast<uint8_t *>(at(L.pk8)) : nullptr,
                                     a.fp8 ? static_cast<float *>(at(L.pks)) : nullptr, s_cmp));

    const std::vector<int64_t> bounds = chunk_bounds(T, R);
    const int64_t n_chunks = static_cast<int64_t>(bounds.size()) - 1;
    for (int64_t c = 0; c < n_chunks; ++c) {
        const int b = static_cast<int>(c & 1);
        const int64_t r0 = bounds[c], r1 = bounds[c + 1], rows = r1 - r0;
        // copy-in of the chunk's q and w rows once buffer b is free again
        if (c >= 2) KPOOL_CUDA_CHECK(cudaStreamWaitEvent(s_in, ps->ev_cmp[b], 0));
        KPOOL_CUDA_CHECK(cudaMemcpyAsync(
            at(L.qbuf[b]), static_cast<const uint8_t *>(a.q) + static_cast<size_t>(r0) * a.H * a.D * 2,
            static_cast<size_t>(rows) * a.H * a.D * 2, cudaMemcpyHostToDevice, s_in));
        KPOOL_CUDA_CHECK(cudaMemcpyAsync(at(L.wbuf[b]), a.w + static_cast<size_t>(r0) * a.H,
                                         static_cast<size_t>(rows) * a.H * 4,
                                         cudaMemcpyHostToDevice, s_in));
        KPOOL_CUDA_CHECK(cudaEventRecord(ps->ev_in[b], s_in));

        // scoring and expansion of the chunk as positioned queries
        KPOOL_CUDA_CHECK(cudaStreamWaitEvent(s_cmp, ps->ev_in[b], 0));
        if (c >= 2) KPOOL_CUDA_CHECK(cudaStreamWaitEvent(s_cmp, ps->ev_out[b], 0));
        chunk_layout_kernel<<<1, 256, 0, s_cmp>>>(cu, a.n_docs, r0, r1, cu_q, q_pos);
        KPOOL_CUDA_CHECK(cudaGetLastError());
        ScoreArgs sa{};
        sa.q = at(L.qbuf[b]);
        sa.w = static_cast<const float *>(at(L.wbuf[b]));
        sa.pk = at(L.pk);
        if (a.fp8) {
            KPOOL_CUDA_CHECK(launch_quantize_fp8(at(L.qbuf[b]), rows * a.H,
                                                 static_cast<uint8_t *>(at(L.q8)),
                                                 static_cast<float *>(at(L.qs)), s_cmp));
            sa.q = at(L.q8);
            sa.q_scale = static_cast<const float *>(at(L.qs));
            sa.pk = at(L.pk8);
            sa.pk_scale = static_cast<const float *>(at(L.pks));
        }
        sa.cu_seqlens = cu_q;
        sa.cu_pools = cu_pools;
        sa.q_pos = q_pos;
        sa.n_docs = a.n_docs;
        sa.T = rows;
        sa.P_total = a.P_total;
        sa.H = a.H;
        sa.D = a.D;
        sa.kpool = a.kpool;
        sa.Kp = Kp;
        sa.fp8 = a.fp8;
        sa.mode = 0;
        sa.pool_idx = static_cast<int32_t *>(at(L.idx));
        sa.pool_score = static_cast<float *>(at(L.score));
        sa.ws = ws;
        sa.ws_bytes = L.ws_bytes;
        if ((rc = run_score(sa, s_cmp))) return rc;
        status_accum_kernel<<<1, 32, 0, s_cmp>>>(ws + 1, sticky + 1);
        KPOOL_CUDA_CHECK(cudaGetLastError());
        KPOOL_CUDA_CHECK(launch_expand(static_cast<const int32_t *>(at(L.idx)), cu_q, q_pos, cu,
                                       cu_pools, a.n_docs, rows, a.kpool, Kp, a.tail,
                                       static_cast<int32_t *>(at(L.tok[b])), s_cmp));
        KPOOL_CUDA_CHECK(cudaEventRecord(ps->ev_cmp[b], s_cmp));

        // copy-out of the chunk's token indices
        KPOOL_CUDA_CHECK(cudaStreamWaitEvent(s_out, ps->ev_cmp[b], 0));
        KPOOL_CUDA_CHECK(cudaMemcpyAsync(a.tok_out + static_cast<size_t>(r0) * W, at(L.tok[b]),
                                         static_cast<size_t>(rows) * W * 4,
                                         cudaMemcpyDeviceToHost, s_out));
        KPOOL_CUDA_CHECK(cudaEventRecord(ps->ev_out[b], s_out));
    }
    // the caller's stream resumes after the last copy-out (the copy-out stream
    // runs in order, after every compute and copy-in it waited for)
    if (n_chunks > 0) {
        KPOOL_CUDA_CHECK(cudaStreamWaitEvent(stream, ps->ev_out[(n_chunks - 1) & 1], 0));
    } else {
        KPOOL_CUDA_CHECK(cudaEventRecord(ps->ev_cmp[0], s_cmp));
        KPOOL_CUDA_CHECK(cudaStreamWaitEvent(stream, ps->ev_cmp[0], 0));
    }
    return KPOOL_OK;
}

}  // namespace kpool
