// C ABI of libkpool.so: host-side argument checks, then one or two kernel
// launches per call on the caller's stream.  See include/kpool.h for the
// contract of every entry point.
#include <cstdarg>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include <cmath>

#include "kpool_internal.h"

namespace kpool {

namespace {
thread_local std::string g_last_error;
}

void set_error(const std::string &msg) { g_last_error = msg; }
void clear_error() { g_last_error.clear(); }
const char *last_error_cstr() { return g_last_error.c_str(); }

int fail(int code, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    set_error(buf);
    return code;
}

int num_sms()
{
    static std::mutex mu;
    static std::vector<int> cache;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    std::lock_guard<std::mutex> lk(mu);
    if (static_cast<int>(cache.size()) <= dev) cache.resize(dev + 1, 0);
    if (cache[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cache[dev] = n > 0 ? n : 1;
    }
    return cache[dev];
}

int check_docs(const int32_t *cu_seqlens, const int32_t *cu_pools, int n_docs, int64_t T,
               int kpool, int64_t P_total)
{
    if (n_docs < 1) return fail(KPOOL_ERR_INVALID_ARG, "n_docs must be >= 1 (got %d)", n_docs);
    if ((cu_seqlens == nullptr) != (cu_pools == nullptr))
        return fail(KPOOL_ERR_INVALID_ARG, "cu_seqlens and cu_pools must both be NULL or both set");
    if (cu_seqlens == nullptr) {
        if (n_docs != 1)
            return fail(KPOOL_ERR_INVALID_ARG, "n_docs must be 1 when cu_seqlens is NULL");
        if (P_total >= 0 && P_total != T / kpool)
            return fail(KPOOL_ERR_INVALID_ARG, "P_total must be T / kpool for one sequence");
    } else {
        if (!aligned(cu_seqlens, 4) || !aligned(cu_pools, 4))
            return fail(KPOOL_ERR_INVALID_ARG, "cu_seqlens / cu_pools must be 4-byte aligned");
    }
    if (P_total > T) return fail(KPOOL_ERR_INVALID_ARG, "P_total exceeds T");
    return KPOOL_OK;
}

}  // namespace kpool

using namespace kpool;

namespace {

int check_common(int64_t T, int kpool)
{
    if (T < 0 || T > 0x7FFFFFFFLL) return fail(KPOOL_ERR_INVALID_ARG, "T out of range");
    if (kpool < 1 || kpool > 64)
        return fail(KPOOL_ERR_UNSUPPORTED, "kpool must be in [1, 64] (got %d)", kpool);
    return KPOOL_OK;
}

// Shared checks of the sparse-attention entry points.
int check_mla_args(const void *q, const void *kv, int64_t T, int64_t Tk, int H, int Dc,
                   float scale, const void *o_out, const float *lse_out, const void *workspace,
                   size_t workspace_bytes)
{
    if (T < 0 || T > 0x7FFFFFFFLL) return fail(KPOOL_ERR_INVALID_ARG, "T out of range");
    if (Tk < 0 || Tk > 0x7FFFFFFFLL) return fail(KPOOL_ERR_INVALID_ARG, "Tk out of range");
    if (H != 64 || Dc != 512)
        return fail(KPOOL_ERR_UNSUPPORTED, "the sparse attention is built for H = 64, Dc = 512 "
                    "(got H = %d, Dc = %d)", H, Dc);
    if (!(scale > 0.f) || !std::isfinite(scale))
        return fail(KPOOL_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
    if (T > 0 && (!q || !o_out || !lse_out))
        return fail(KPOOL_ERR_INVALID_ARG, "q, o_out and lse_out are required");
    if (T > 0 && !kv) return fail(KPOOL_ERR_INVALID_ARG, "kv is required");
    if (!aligned(q, 16) || !aligned(kv, 16) || !aligned(o_out, 16) || !aligned(lse_out, 4))
        return fail(KPOOL_ERR_INVALID_ARG, "q, kv and o_out must be 16-byte aligned");
    if (!workspace || workspace_bytes < sparse_mla_workspace_bytes() || !aligned(workspace, 256))
        return fail(KPOOL_ERR_WORKSPACE, "workspace of at least %zu bytes, 256-byte aligned, needed",
                    sparse_mla_workspace_bytes());
    return KPOOL_OK;
}

int check_h(int H)
{
    if (H != 4 && H != 8 && H != 16 && H != 32 && H != 64 && H != 128)
        return fail(KPOOL_ERR_UNSUPPORTED, "H must be one of 4, 8, 16, 32, 64, 128 (got %d)", H);
    return KPOOL_OK;
}

int check_score_args(const void *q, const float *q_scale, const float *w, const void *pk,
                     const float *pk_scale, const int32_t *cu_seqlens, const int32_t *cu_pools,
                     int n_docs, int64_t T, int64_t P_total, int H, int D, int kpool, int fp8,
                     void *workspace, size_t workspace_bytes)
{
    int rc = check_common(T, kpool);
    if (rc) return rc;
    if ((rc = check_h(H))) return rc;
    if (fp8) {
        if (D != 128) return fail(KPOOL_ERR_UNSUPPORTED, "FP8 mode needs D = 128 (got %d)", D);
        if (!q_scale || !pk_scale)
            return fail(KPOOL_ERR_INVALID_ARG, "FP8 mode needs q_scale and pk_scale");
        if (!aligned(q_scale, 16) || !aligned(pk_scale, 4))
            return fail(KPOOL_ERR_INVALID_ARG, "q_scale must be 16-byte aligned");
    } else {
        if (D != 32 && D != 64 && D != 128)
            return fail(KPOOL_ERR_UNSUPPORTED, "D must be 32, 64 or 128 (got %d)", D);
        if (q_scale || pk_scale)
            return fail(KPOOL_ERR_INVALID_ARG, "q_scale / pk_scale must be NULL in bf16 mode");
    }
    if (T > 0 && (!q || !w)) return fail(KPOOL_ERR_INVALID_ARG, "q and w must be non-NULL");
    if (P_total > 0 && !pk) return fail(KPOOL_ERR_INVALID_ARG, "pk must be non-NULL");
    if (!aligned(q, 16) || !aligned(pk, 16) || !aligned(w, 16))
        return fail(KPOOL_ERR_INVALID_ARG, "q, pk and w must be 16-byte aligned");
    if (P_total < 0) return fail(KPOOL_ERR_INVALID_ARG, "P_total < 0");
    if (static_cast<int64_t>(T) * H > 0x7FFFFFFFLL)
        return fail(KPOOL_ERR_UNSUPPORTED, "T * H exceeds 2^31 - 1");
    if ((rc = check_docs(cu_seqlens, cu_pools, n_docs, T, kpool, P_total))) return rc;
    const size_t need = score_workspace_bytes(T, H, n_docs);
    if (!workspace || workspace_bytes < need)
        return fail(KPOOL_ERR_WORKSPACE, "workspace needs %zu bytes (got %zu)", need,
                    workspace ? workspace_bytes : static_cast<size_t>(0));
    if (!aligned(workspace, 256))
        return fail(KPOOL_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    return KPOOL_OK;
}

}  // namespace

extern "C" {

const char *kpool_last_error(void) { return last_error_cstr(); }

int kpool_version(void) { return 10000; }

int kpool_num_pools(const int32_t *cu_seqlens_host, int n_docs, int64_t T, int kpool,
                    int32_t *cu_pools_host_out, int64_t *total_pools_out)
{
    clear_error();
    int rc = check_common(T, kpool);
    if (rc) return rc;
    if (!cu_seqlens_host || !cu_pools_host_out || !total_pools_out)
        return fail(KPOOL_ERR_INVALID_ARG, "NULL pointer");
    if (n_docs < 1) return fail(KPOOL_ERR_INVALID_ARG, "n_docs must be >= 1");
    if (cu_seqlens_host[0] != 0)
        return fail(KPOOL_ERR_INVALID_ARG, "cu_seqlens[0] must be 0 (got %d)", cu_seqlens_host[0]);
    if (cu_seqlens_host[n_docs] != T)
        return fail(KPOOL_ERR_INVALID_ARG, "cu_seqlens[n_docs] must equal T");
    int64_t acc = 0;
    cu_pools_host_out[0] = 0;
    for (int d = 0; d < n_docs; ++d) {
        const int64_t L = static_cast<int64_t>(cu_seqlens_host[d + 1]) - cu_seqlens_host[d];
        if (L < 0) return fail(KPOOL_ERR_INVALID_ARG, "cu_seqlens decreases at document %d", d);
        acc += L / kpool;
        cu_pools_host_out[d + 1] = static_cast<int32_t>(acc);
    }
    *total_pools_out = acc;
    return KPOOL_OK;
}

int kpool_cu_pools(const int32_t *cu_seqlens, int n_docs, int kpool, int32_t *cu_pools_out,
                   kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_cu_pools");
    if (kpool < 1 || kpool > 64) return fail(KPOOL_ERR_UNSUPPORTED, "kpool must be in [1, 64]");
    if (n_docs < 1) return fail(KPOOL_ERR_INVALID_ARG, "n_docs must be >= 1");
    if (!cu_seqlens || !cu_pools_out) return fail(KPOOL_ERR_INVALID_ARG, "NULL pointer");
    KPOOL_CUDA_CHECK(launch_cu_pools(cu_seqlens, n_docs, kpool, cu_pools_out,
                                     reinterpret_cast<cudaStream_t>(stream)));
    return KPOOL_OK;
}

int kpool_compress(const void *k, const void *gate, const float *ape,
                   const int32_t *cu_seqlens, const int32_t *cu_pools, int n_docs,
                   int64_t T, int D, int kpool, int64_t P_total, void *pk_out,
                   uint8_t *pk_fp8_out, float *pk_scale_out, kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_compress");
    int rc = check_common(T, kpool);
    if (rc) return rc;
    if (D != 32 && D != 64 && D != 128)
        return fail(KPOOL_ERR_UNSUPPORTED, "D must be 32, 64 or 128 (got %d)", D);
    if (P_total < 0) return fail(KPOOL_ERR_INVALID_ARG, "P_total < 0");
    if ((rc = check_docs(cu_seqlens, cu_pools, n_docs, T, kpool, P_total))) return rc;
    if (P_total > 0 && (!k || !gate || !ape || !pk_out))
        return fail(KPOOL_ERR_INVALID_ARG, "k, gate, ape and pk_out must be non-NULL");
    if (!aligned(k, 16) || !aligned(gate, 16) || !aligned(pk_out, 16) || !aligned(ape, 16))
        return fail(KPOOL_ERR_INVALID_ARG, "k, gate, ape and pk_out must be 16-byte aligned");
    if ((pk_fp8_out == nullptr) != (pk_scale_out == nullptr))
        return fail(KPOOL_ERR_INVALID_ARG, "pk_fp8_out and pk_scale_out go together");
    if (pk_fp8_out) {
        if (D != 128) return fail(KPOOL_ERR_UNSUPPORTED, "FP8 pooled keys need D = 128");
        if (!aligned(pk_fp8_out, 16) || !aligned(pk_scale_out, 4))
            return fail(KPOOL_ERR_INVALID_ARG, "pk_fp8_out must be 16-byte aligned");
    }
    KPOOL_CUDA_CHECK(launch_compress(k, gate, ape, cu_seqlens, cu_pools, n_docs, T, D, kpool,
                                     P_total, pk_out, pk_fp8_out, pk_scale_out,
                                     reinterpret_cast<cudaStream_t>(stream)));
    return KPOOL_OK;
}

int kpool_quantize_fp8(const void *x, int64_t rows, int D, uint8_t *x_fp8_out, float *scale_out,
                       kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_quantize_fp8");
    if (D != 128) return fail(KPOOL_ERR_UNSUPPORTED, "FP8 rows need D = 128 (got %d)", D);
    if (rows < 0) return fail(KPOOL_ERR_INVALID_ARG, "rows < 0");
    if (rows > 0 && (!x || !x_fp8_out || !scale_out))
        return fail(KPOOL_ERR_INVALID_ARG, "NULL pointer");
    if (!aligned(x, 16) || !aligned(x_fp8_out, 16) || !aligned(scale_out, 4))
        return fail(KPOOL_ERR_INVALID_ARG, "x and x_fp8_out must be 16-byte aligned");
    KPOOL_CUDA_CHECK(launch_quantize_fp8(x, rows, x_fp8_out, scale_out,
                                         reinterpret_cast<cudaStream_t>(stream)));
    return KPOOL_OK;
}

size_t kpool_score_topk_workspace_size(int64_t T, int H, int n_docs)
{
    if (T < 0 || n_docs < 1 || check_h(H) != KPOOL_OK) return 0;
    return score_workspace_bytes(T, H, n_docs);
}

size_t kpool_score_topk_workspace_size_split(int64_t T, int H, int n_docs, int kpool,
                                             int index_topk)
{
    if (T < 0 || n_docs < 1 || check_h(H) != KPOOL_OK) return 0;
    if (kpool < 1 || index_topk < 1 || index_topk % kpool != 0) return 0;
    return score_workspace_split_bytes(T, H, n_docs, index_topk / kpool);
}

int kpool_score_topk(const void *q, const float *q_scale, const float *w, const void *pk,
                     const float *pk_scale, const int32_t *cu_seqlens, const int32_t *cu_pools,
                     int n_docs, int64_t T, int64_t P_total, int H, int D, int kpool,
                     int index_topk, int fp8, int32_t *pool_idx_out, float *pool_score_out,
                     void *workspace, size_t workspace_bytes, kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_score_topk");
    int rc = check_score_args(q, q_scale, w, pk, pk_scale, cu_seqlens, cu_pools, n_docs, T,
                              P_total, H, D, kpool, fp8, workspace, workspace_bytes);
    if (rc) return rc;
    if (index_topk < 1 || index_topk % kpool != 0)
        return fail(KPOOL_ERR_INVALID_ARG, "index_topk must be a positive multiple of kpool");
    const int Kp = index_topk / kpool;
    const int cap = score_capacity(H, D, fp8);
    int kp2 = 1;
    while (kp2 < Kp) kp2 <<= 1;
    if (Kp + 128 > cap || kp2 > cap)
        return fail(KPOOL_ERR_UNSUPPORTED,
                    "index_topk / kpool = %d exceeds the per-query candidate capacity %d for H=%d "
                    "(needs Kp + 128 and the next power of two of Kp to fit)",
                    Kp, cap, H);
    if (T > 0 && (!pool_idx_out || !pool_score_out))
        return fail(KPOOL_ERR_INVALID_ARG, "pool_idx_out and pool_score_out must be non-NULL");
    ScoreArgs a{};
    a.q = q; a.q_scale = q_scale; a.w = w; a.pk = pk; a.pk_scale = pk_scale;
    a.cu_seqlens = cu_seqlens; a.cu_pools = cu_pools; a.n_docs = n_docs;
    a.T = T; a.P_total = P_total; a.H = H; a.D = D; a.kpool = kpool; a.Kp = Kp;
    a.fp8 = fp8 ? 1 : 0; a.mode = 0;
    a.pool_idx = pool_idx_out; a.pool_score = pool_score_out; a.scores = nullptr;
    a.ws = static_cast<int *>(workspace); a.ws_bytes = workspace_bytes;
    return run_score(a, reinterpret_cast<cudaStream_t>(stream));
}

int kpool_score_topk_noalloc(const void *q, const float *q_scale, const float *w, const void *pk,
                             const float *pk_scale, const int32_t *cu_seqlens,
                             const int32_t *cu_pools, int n_docs, int64_t T, int64_t P_total,
                             int H, int D, int kpool, int index_topk, int fp8,
                             int32_t *pool_idx_out, float *pool_score_out, kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_score_topk_noalloc");
    int rc = check_common(T, kpool);
    if (rc) return rc;
    if ((rc = check_h(H))) return rc;
    if (n_docs < 1) return fail(KPOOL_ERR_INVALID_ARG, "n_docs must be >= 1 (got %d)", n_docs);
    int *scratch = nullptr;
    size_t scratch_bytes = 0;
    int64_t max_tiles = 0;
    const int64_t QT = 256 / H;
    const int64_t need_tiles = (T + QT - 1) / QT + n_docs;
    // the capacity is a compile-time constant: reject before touching the device
    if (need_tiles > kNoAllocMaxTiles)
        return fail(KPOOL_ERR_UNSUPPORTED,
                    "kpool_score_topk_noalloc: T=%lld with H=%d and %d documents needs %lld "
                    "query tiles; its fixed scratch holds at most %d (use kpool_score_topk "
                    "with a caller-provided workspace)",
                    static_cast<long long>(T), H, n_docs, static_cast<long long>(need_tiles),
                    kNoAllocMaxTiles);
    if ((rc = noalloc_scratch(&scratch, &scratch_bytes, &max_tiles))) return rc;
    if (need_tiles > max_tiles)
        return fail(KPOOL_ERR_UNSUPPORTED, "no-alloc scratch too small (%lld tiles needed)",
                    static_cast<long long>(need_tiles));
    return kpool_score_topk(q, q_scale, w, pk, pk_scale, cu_seqlens, cu_pools, n_docs, T, P_total,
                            H, D, kpool, index_topk, fp8, pool_idx_out, pool_score_out, scratch,
                            scratch_bytes, stream);
}

int kpool_score_topk_at(const void *q, const float *q_scale, const float *w, const void *pk,
                        const float *pk_scale, const int32_t *cu_seqlens_q,
                        const int32_t *q_start_pos, const int32_t *cu_pools, int n_docs,
                        int64_t Tq, int64_t P_total, int H, int D, int kpool, int index_topk,
                        int fp8, int32_t *pool_idx_out, float *pool_score_out, void *workspace,
                        size_t workspace_bytes, kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_score_topk_at");
    if (!cu_seqlens_q || !q_start_pos || !cu_pools)
        return fail(KPOOL_ERR_INVALID_ARG, "cu_seqlens_q, q_start_pos and cu_pools are required");
    if (!aligned(q_start_pos, 4)) return fail(KPOOL_ERR_INVALID_ARG, "q_start_pos misaligned");
    // the key-side pool count is independent of the number of query rows
    int rc = check_score_args(q, q_scale, w, pk, pk_scale, cu_seqlens_q, cu_pools, n_docs, Tq, 0,
                              H, D, kpool, fp8, workspace, workspace_bytes);
    if (rc) return rc;
    if (P_total < 0) return fail(KPOOL_ERR_INVALID_ARG, "P_total < 0");
    if (P_total > 0 && !pk) return fail(KPOOL_ERR_INVALID_ARG, "pk must be non-NULL");
    if (index_topk < 1 || index_topk % kpool != 0)
        return fail(KPOOL_ERR_INVALID_ARG, "index_topk must be a positive multiple of kpool");
    const int Kp = index_topk / kpool;
    const int cap = score_capacity(H, D, fp8);
    int kp2 = 1;
    while (kp2 < Kp) kp2 <<= 1;
    if (Kp + 128 > cap || kp2 > cap)
        return fail(KPOOL_ERR_UNSUPPORTED,
                    "index_topk / kpool = %d exceeds the per-query candidate capacity %d for H=%d",
                    Kp, cap, H);
    if (Tq > 0 && (!pool_idx_out || !pool_score_out))
        return fail(KPOOL_ERR_INVALID_ARG, "pool_idx_out and pool_score_out must be non-NULL");
    ScoreArgs a{};
    a.q = q; a.q_scale = q_scale; a.w = w; a.pk = pk; a.pk_scale = pk_scale;
    a.cu_seqlens = cu_seqlens_q; a.cu_pools = cu_pools; a.q_pos = q_start_pos; a.n_docs = n_docs;
    a.T = Tq; a.P_total = P_total; a.H = H; a.D = D; a.kpool = kpool; a.Kp = Kp;
    a.fp8 = fp8 ? 1 : 0; a.mode = 0;
    a.pool_idx = pool_idx_out; a.pool_score = pool_score_out; a.scores = nullptr;
    a.ws = static_cast<int *>(workspace); a.ws_bytes = workspace_bytes;
    return run_score(a, reinterpret_cast<cudaStream_t>(stream));
}

int kpool_expand_indices_at(const int32_t *pool_idx, const int32_t *cu_seqlens_q,
                            const int32_t *q_start_pos, const int32_t *cu_seqlens_k,
                            const int32_t *cu_pools, int n_docs, int64_t Tq, int kpool,
                            int index_topk, int always_select_tail, int32_t *tok_idx_out,
                            kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_expand_indices_at");
    int rc = check_common(Tq, kpool);
    if (rc) return rc;
    if (!cu_seqlens_q || !q_start_pos || !cu_seqlens_k || !cu_pools)
        return fail(KPOOL_ERR_INVALID_ARG,
                    "cu_seqlens_q, q_start_pos, cu_seqlens_k and cu_pools are required");
    if (n_docs < 1) return fail(KPOOL_ERR_INVALID_ARG, "n_docs must be >= 1");
    if (!aligned(cu_seqlens_q, 4) || !aligned(q_start_pos, 4) || !aligned(cu_seqlens_k, 4) ||
        !aligned(cu_pools, 4))
        return fail(KPOOL_ERR_INVALID_ARG, "index arrays must be 4-byte aligned");
    if (index_topk < 1 || index_topk % kpool != 0)
        return fail(KPOOL_ERR_INVALID_ARG, "index_topk must be a positive multiple of kpool");
    if (Tq > 0 && (!pool_idx || !tok_idx_out))
        return fail(KPOOL_ERR_INVALID_ARG, "pool_idx and tok_idx_out must be non-NULL");
    if (!aligned(pool_idx, 4) || !aligned(tok_idx_out, 4))
        return fail(KPOOL_ERR_INVALID_ARG, "pool_idx and tok_idx_out must be 4-byte aligned");
    const int Kp = index_topk / kpool;
    KPOOL_CUDA_CHECK(launch_expand(pool_idx, cu_seqlens_q, q_start_pos, cu_seqlens_k, cu_pools,
                                   n_docs, Tq, kpool, Kp, always_select_tail ? 1 : 0, tok_idx_out,
                                   reinterpret_cast<cudaStream_t>(stream)));
    return KPOOL_OK;
}

int kpool_score_dense(const void *q, const float *q_scale, const float *w, const void *pk,
                      const float *pk_scale, const int32_t *cu_seqlens, const int32_t *cu_pools,
                      int n_docs, int64_t T, int64_t P_total, int H, int D, int kpool, int fp8,
                      float *scores_out, void *workspace, size_t workspace_bytes,
                      kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_score_dense");
    int rc = check_score_args(q, q_scale, w, pk, pk_scale, cu_seqlens, cu_pools, n_docs, T,
                              P_total, H, D, kpool, fp8, workspace, workspace_bytes);
    if (rc) return rc;
    if (T > 0 && P_total > 0 && !scores_out)
        return fail(KPOOL_ERR_INVALID_ARG, "scores_out must be non-NULL");
    if (static_cast<double>(T) * static_cast<double>(P_total) > 4.0e9)
        return fail(KPOOL_ERR_UNSUPPORTED, "dense scores are meant for small T");
    ScoreArgs a{};
    a.q = q; a.q_scale = q_scale; a.w = w; a.pk = pk; a.pk_scale = pk_scale;
    a.cu_seqlens = cu_seqlens; a.cu_pools = cu_pools; a.n_docs = n_docs;
    a.T = T; a.P_total = P_total; a.H = H; a.D = D; a.kpool = kpool; a.Kp = 1;
    a.fp8 = fp8 ? 1 : 0; a.mode = 1;
    a.pool_idx = nullptr; a.pool_score = nullptr; a.scores = scores_out;
    a.ws = static_cast<int *>(workspace); a.ws_bytes = workspace_bytes;
    return run_score(a, reinterpret_cast<cudaStream_t>(stream));
}

int kpool_expand_indices(const int32_t *pool_idx, const int32_t *cu_seqlens,
                         const int32_t *cu_pools, int n_docs, int64_t T, int kpool,
                         int index_topk, int always_select_tail, int32_t *tok_idx_out,
                         kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_expand_indices");
    int rc = check_common(T, kpool);
    if (rc) return rc;
    if (index_topk < 1 || index_topk % kpool != 0)
        return fail(KPOOL_ERR_INVALID_ARG, "index_topk must be a positive multiple of kpool");
    if ((rc = check_docs(cu_seqlens, cu_pools, n_docs, T, kpool, -1))) return rc;
    if (T > 0 && (!pool_idx || !tok_idx_out))
        return fail(KPOOL_ERR_INVALID_ARG, "pool_idx and tok_idx_out must be non-NULL");
    if (!aligned(pool_idx, 4) || !aligned(tok_idx_out, 4))
        return fail(KPOOL_ERR_INVALID_ARG, "pool_idx and tok_idx_out must be 4-byte aligned");
    const int Kp = index_topk / kpool;
    if (static_cast<int64_t>(Kp) * kpool + kpool > 0x7FFFFFFF)
        return fail(KPOOL_ERR_UNSUPPORTED, "row width overflows");
    KPOOL_CUDA_CHECK(launch_expand(pool_idx, cu_seqlens, nullptr, nullptr, cu_pools, n_docs, T,
                                   kpool, Kp, always_select_tail ? 1 : 0, tok_idx_out,
                                   reinterpret_cast<cudaStream_t>(stream)));
    return KPOOL_OK;
}

}  // extern "C"

namespace {

// Host-side layout check of a host cu_seqlens; fills *P_total.
int host_layout(const int32_t *cu_host, int n_docs, int64_t T, int kpool, int64_t *P_total)
{
    if (!cu_host) {
        *P_total = T / kpool;
        return KPOOL_OK;
    }
    if (n_docs < 1) return fail(KPOOL_ERR_INVALID_ARG, "n_docs must be >= 1 (got %d)", n_docs);
    if (cu_host[0] != 0 || cu_host[n_docs] != T)
        return fail(KPOOL_ERR_INVALID_ARG, "cu_seqlens must run from 0 to T");
    int64_t P = 0;
    for (int d = 0; d < n_docs; ++d) {
        const int64_t L = static_cast<int64_t>(cu_host[d + 1]) - cu_host[d];
        if (L < 0) return fail(KPOOL_ERR_INVALID_ARG, "cu_seqlens must be non-decreasing");
        P += L / kpool;
    }
    *P_total = P;
    return KPOOL_OK;
}

int check_forward_shapes(int64_t T, int H, int D, int kpool, int index_topk, int fp8)
{
    int rc = check_common(T, kpool);
    if (rc) return rc;
    if ((rc = check_h(H))) return rc;
    if (fp8 ? D != 128 : (D != 32 && D != 64 && D != 128))
        return fail(KPOOL_ERR_UNSUPPORTED, "D must be 32, 64 or 128 (128 in FP8 mode)");
    if (index_topk < 1 || index_topk % kpool != 0)
        return fail(KPOOL_ERR_INVALID_ARG, "index_topk must be a positive multiple of kpool");
    const int Kp = index_topk / kpool;
    const int cap = score_capacity(H, D, fp8);
    int kp2 = 1;
    while (kp2 < Kp) kp2 <<= 1;
    if (Kp + 128 > cap || kp2 > cap)
        return fail(KPOOL_ERR_UNSUPPORTED,
                    "index_topk / kpool = %d exceeds the per-query candidate capacity %d", Kp,
                    cap);
    if (T * H > 0x7FFFFFFFLL) return fail(KPOOL_ERR_UNSUPPORTED, "T * H exceeds 2^31 - 1");
    return KPOOL_OK;
}

}  // namespace

extern "C" {

size_t kpool_indexer_forward_host_scratch_size(const int32_t *cu_seqlens_host, int n_docs,
                                               int64_t T, int H, int D, int kpool,
                                               int index_topk, int fp8, int64_t chunk_rows)
{
    if (chunk_rows < 0 || check_forward_shapes(T, H, D, kpool, index_topk, fp8)) return 0;
    int64_t P = 0;
    if (host_layout(cu_seqlens_host, cu_seqlens_host ? n_docs : 1, T, kpool, &P)) return 0;
    return pipeline_scratch_bytes(T, H, D, cu_seqlens_host ? n_docs : 1, kpool, index_topk, fp8,
                                  chunk_rows, P);
}

int kpool_indexer_forward_host(const void *q, const void *k, const void *gate, const float *ape,
                               const float *w, const int32_t *cu_seqlens_host, int n_docs,
                               int64_t T, int H, int D, int kpool, int index_topk,
                               int always_select_tail, int fp8, int64_t chunk_rows,
                               int32_t *tok_idx_out, void *scratch, size_t scratch_bytes,
                               kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_indexer_forward_host");
    int rc = check_forward_shapes(T, H, D, kpool, index_topk, fp8);
    if (rc) return rc;
    if (chunk_rows < 0) return fail(KPOOL_ERR_INVALID_ARG, "chunk_rows < 0");
    if (!cu_seqlens_host) n_docs = 1;
    int64_t P = 0;
    if ((rc = host_layout(cu_seqlens_host, n_docs, T, kpool, &P))) return rc;
    if (T == 0) return KPOOL_OK;
    if (!q || !k || !gate || !ape || !w || !tok_idx_out)
        return fail(KPOOL_ERR_INVALID_ARG, "NULL host pointer");
    if (!scratch) return fail(KPOOL_ERR_WORKSPACE, "scratch is NULL");
    if (!aligned(scratch, 256))
        return fail(KPOOL_ERR_INVALID_ARG, "scratch must be 256-byte aligned");
    PipelineArgs a{};
    a.q = q;
    a.k = k;
    a.gate = gate;
    a.ape = ape;
    a.w = w;
    a.cu_seqlens_host = cu_seqlens_host;   // NULL: one sequence
    a.n_docs = n_docs;
    a.T = T;
    a.P_total = P;
    a.chunk_rows = chunk_rows;
    a.H = H;
    a.D = D;
    a.kpool = kpool;
    a.index_topk = index_topk;
    a.tail = always_select_tail ? 1 : 0;
    a.fp8 = fp8 ? 1 : 0;
    a.tok_out = tok_idx_out;
    a.scratch = scratch;
    a.scratch_bytes = scratch_bytes;
    return run_pipeline(a, reinterpret_cast<cudaStream_t>(stream));
}

int kpool_read_status(const void *workspace, int *status_out)
{
    clear_error();
    if (!workspace || !status_out) return fail(KPOOL_ERR_INVALID_ARG, "NULL pointer");
    KPOOL_CUDA_CHECK(cudaDeviceSynchronize());
    int v = 0;
    KPOOL_CUDA_CHECK(cudaMemcpy(&v, static_cast<const int *>(workspace) + 1, sizeof(int),
                                cudaMemcpyDeviceToHost));
    *status_out = v;
    return KPOOL_OK;
}

int kpool_project_compress(const void *x, const void *w_kg, const float *k_norm_weight,
                           const float *k_norm_bias, float k_norm_eps, const float *ape,
                           const int32_t *cu_seqlens, const int32_t *cu_pools, int n_docs,
                           int64_t T, int hidden, int D, int kpool, int64_t P_total, void *pk_out,
                           void *k_out, void *gate_out, void *workspace, size_t workspace_bytes,
                           kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_project_compress");
    int rc = check_common(T, kpool);
    if (rc) return rc;
    if (D != 128) return fail(KPOOL_ERR_UNSUPPORTED, "the fused projection needs D = 128 (got %d)", D);
    if (32 % kpool != 0)
        return fail(KPOOL_ERR_UNSUPPORTED, "the fused projection needs kpool dividing 32 (got %d)",
                    kpool);
    if (hidden < 64 || hidden % 64 != 0 || hidden > 65536)
        return fail(KPOOL_ERR_UNSUPPORTED, "hidden must be a multiple of 64 in [64, 65536] (got %d)",
                    hidden);
    if (T * static_cast<int64_t>(hidden) > (int64_t(1) << 40))
        return fail(KPOOL_ERR_UNSUPPORTED, "T * hidden too large");
    if (P_total < 0) return fail(KPOOL_ERR_INVALID_ARG, "P_total < 0");
    if ((rc = check_docs(cu_seqlens, cu_pools, n_docs, T, kpool, P_total))) return rc;
    if (T > 0 && (!x || !w_kg || !k_norm_weight || !k_norm_bias || !ape))
        return fail(KPOOL_ERR_INVALID_ARG, "x, w_kg, k_norm_weight, k_norm_bias and ape are required");
    if (P_total > 0 && !pk_out) return fail(KPOOL_ERR_INVALID_ARG, "pk_out is required");
    if (!aligned(x, 16) || !aligned(w_kg, 16) || !aligned(pk_out, 16) || !aligned(k_out, 16) ||
        !aligned(gate_out, 16) || !aligned(ape, 4) || !aligned(k_norm_weight, 4) ||
        !aligned(k_norm_bias, 4))
        return fail(KPOOL_ERR_INVALID_ARG, "x, w_kg, pk_out, k_out and gate_out must be 16-byte aligned");
    if (!(k_norm_eps >= 0.f)) return fail(KPOOL_ERR_INVALID_ARG, "k_norm_eps must be >= 0");
    if (!workspace || workspace_bytes < 256 || !aligned(workspace, 256))
        return fail(KPOOL_ERR_WORKSPACE, "workspace of at least 256 bytes, 256-byte aligned, needed");
    ProjectArgs a{};
    a.x = x; a.w = w_kg; a.gamma = k_norm_weight; a.beta = k_norm_bias; a.ape = ape;
    a.eps = k_norm_eps; a.cu_seqlens = cu_seqlens; a.cu_pools = cu_pools; a.n_docs = n_docs;
    a.T = T; a.P_total = P_total; a.hidden = hidden; a.kpool = kpool;
    a.pk_out = pk_out; a.k_out = k_out; a.gate_out = gate_out;
    a.status = static_cast<int *>(workspace) + 1;
    return run_project_compress(a, reinterpret_cast<cudaStream_t>(stream));
}

int kpool_score_topk_noalloc_status(int *status_out)
{
    clear_error();
    if (!status_out) return fail(KPOOL_ERR_INVALID_ARG, "NULL pointer");
    int *scratch = nullptr;
    size_t scratch_bytes = 0;
    int64_t max_tiles = 0;
    const int rc = noalloc_scratch(&scratch, &scratch_bytes, &max_tiles);
    if (rc) return rc;
    return kpool_read_status(scratch, status_out);
}

uint64_t kpool_debug_set_wait_limit_ns(uint64_t ns) { return set_wait_limit_ns(ns); }

size_t kpool_sparse_mla_workspace_size(void) { return sparse_mla_workspace_bytes(); }

int kpool_sparse_mla_fwd(const void *q, const void *kv, const int32_t *tok_idx, int64_t T,
                         int64_t Tk, int W, int H, int Dc, float softmax_scale, void *o_out,
                         float *lse_out, void *workspace, size_t workspace_bytes,
                         kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_sparse_mla_fwd");
    int rc = check_mla_args(q, kv, T, Tk, H, Dc, softmax_scale, o_out, lse_out, workspace,
                            workspace_bytes);
    if (rc) return rc;
    if (W < 0 || W > (1 << 20)) return fail(KPOOL_ERR_INVALID_ARG, "W out of range");
    if (T > 0 && W > 0 && !tok_idx) return fail(KPOOL_ERR_INVALID_ARG, "tok_idx is required");
    if (!aligned(tok_idx, 4)) return fail(KPOOL_ERR_INVALID_ARG, "tok_idx must be 4-byte aligned");
    SparseMlaArgs a{};
    a.q = q; a.kv = kv; a.tok_idx = tok_idx; a.T = T; a.Tk = Tk; a.W = W; a.n_docs = 1;
    a.kpool = 1; a.scale = softmax_scale; a.o = o_out; a.lse = lse_out; a.workspace = workspace;
    // a zero-width list still runs the kernel (every row gets o = 0 and
    // lse = -inf); the kernel never reads a row of width 0
    if (W == 0) a.tok_idx = static_cast<const int32_t *>(workspace);
    return run_sparse_mla(a, reinterpret_cast<cudaStream_t>(stream));
}

int kpool_sparse_mla_fwd_pools(const void *q, const void *kv, const int32_t *pool_idx,
                               const int32_t *cu_seqlens, const int32_t *cu_pools, int n_docs,
                               int64_t T, int H, int Dc, int kpool, int index_topk,
                               int always_select_tail, float softmax_scale, void *o_out,
                               float *lse_out, void *workspace, size_t workspace_bytes,
                               kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_sparse_mla_fwd_pools");
    int rc = check_mla_args(q, kv, T, T, H, Dc, softmax_scale, o_out, lse_out, workspace,
                            workspace_bytes);
    if (rc) return rc;
    if ((rc = check_common(T, kpool))) return rc;
    if (index_topk < 1 || index_topk % kpool != 0)
        return fail(KPOOL_ERR_INVALID_ARG, "index_topk must be a positive multiple of kpool");
    if ((rc = check_docs(cu_seqlens, cu_pools, n_docs, T, kpool, -1))) return rc;
    if (T > 0 && !pool_idx) return fail(KPOOL_ERR_INVALID_ARG, "pool_idx is required");
    if (!aligned(pool_idx, 4)) return fail(KPOOL_ERR_INVALID_ARG, "pool_idx must be 4-byte aligned");
    SparseMlaArgs a{};
    a.q = q; a.kv = kv; a.pool_idx = pool_idx; a.cu_seqlens = cu_seqlens; a.cu_pools = cu_pools;
    a.n_docs = n_docs; a.T = T; a.Tk = T; a.kpool = kpool; a.Kp = index_topk / kpool;
    a.tail = always_select_tail ? 1 : 0; a.scale = softmax_scale; a.o = o_out; a.lse = lse_out;
    a.workspace = workspace;
    return run_sparse_mla(a, reinterpret_cast<cudaStream_t>(stream));
}

int kpool_sparse_mla_fwd_pools_at(const void *q, const void *kv, const int32_t *pool_idx,
                                  const int32_t *cu_seqlens_q, const int32_t *q_start_pos,
                                  const int32_t *cu_seqlens_k, const int32_t *cu_pools, int n_docs,
                                  int64_t Tq, int64_t Tk, int H, int Dc, int kpool, int index_topk,
                                  int always_select_tail, float softmax_scale, void *o_out,
                                  float *lse_out, void *workspace, size_t workspace_bytes,
                                  kpool_stream_t stream)
{
    clear_error();
    KPOOL_NVTX_RANGE("kpool_sparse_mla_fwd_pools_at");
    int rc = check_mla_args(q, kv, Tq, Tk, H, Dc, softmax_scale, o_out, lse_out, workspace,
                            workspace_bytes);
    if (rc) return rc;
    if ((rc = check_common(Tq, kpool))) return rc;
    if (!cu_seqlens_q || !q_start_pos || !cu_seqlens_k || !cu_pools)
        return fail(KPOOL_ERR_INVALID_ARG,
                    "cu_seqlens_q, q_start_pos, cu_seqlens_k and cu_pools are required");
    if (n_docs < 1) return fail(KPOOL_ERR_INVALID_ARG, "n_docs must be >= 1");
    if (!aligned(cu_seqlens_q, 4) || !aligned(q_start_pos, 4) || !aligned(cu_seqlens_k, 4) ||
        !aligned(cu_pools, 4) || !aligned(pool_idx, 4))
        return fail(KPOOL_ERR_INVALID_ARG, "index arrays must be 4-byte aligned");
    if (index_topk < 1 || index_topk % kpool != 0)
        return fail(KPOOL_ERR_INVALID_ARG, "index_topk must be a positive multiple of kpool");
    if (Tq > 0 && !pool_idx) return fail(KPOOL_ERR_INVALID_ARG, "pool_idx is required");
    SparseMlaArgs a{};
    a.q = q; a.kv = kv; a.pool_idx = pool_idx; a.cu_seqlens = cu_seqlens_q; a.q_pos = q_start_pos;
    a.cu_k = cu_seqlens_k; a.cu_pools = cu_pools; a.n_docs = n_docs; a.T = Tq; a.Tk = Tk;
    a.kpool = kpool; a.Kp = index_topk / kpool; a.tail = always_select_tail ? 1 : 0;
    a.scale = softmax_scale; a.o = o_out; a.lse = lse_out; a.workspace = workspace;
    return run_sparse_mla(a, reinterpret_cast<cudaStream_t>(stream));
}

}  // extern "C"
