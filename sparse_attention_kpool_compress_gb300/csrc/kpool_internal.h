// Host-side helpers shared by the library's translation units.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdint>
#include <cstdio>
#include <string>

#include "../../include/kpool.h"

namespace kpool {

// Thread-local message of the last failing call (kpool_last_error).
void set_error(const std::string &msg);
void clear_error();
const char *last_error_cstr();

int fail(int code, const char *fmt, ...);

// NVTX range around one C ABI call (a no-op unless a profiler or tracer
// injects an NVTX handler): nsys / ncu timelines show each entry point.
struct NvtxRange {
    explicit NvtxRange(const char *name) { nvtxRangePushA(name); }
    ~NvtxRange() { nvtxRangePop(); }
    NvtxRange(const NvtxRange &) = delete;
    NvtxRange &operator=(const NvtxRange &) = delete;
};
#define KPOOL_NVTX_RANGE(name) ::kpool::NvtxRange kpool_nvtx_range_(name)

// Number of SMs of the current device (cached per device).
int num_sms();

inline bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

#define KPOOL_CUDA_CHECK(expr)                                                            \
    do {                                                                                  \
        cudaError_t e_ = (expr);                                                          \
        if (e_ != cudaSuccess)                                                            \
            return ::kpool::fail(KPOOL_ERR_CUDA, "%s failed: %s", #expr, cudaGetErrorString(e_)); \
    } while (0)

// Validation of the document layout arguments shared by several entry points.
int check_docs(const int32_t *cu_seqlens, const int32_t *cu_pools, int n_docs, int64_t T,
               int kpool, int64_t P_total);

// ---- launchers implemented in the .cu files ----------------------------
cudaError_t launch_cu_pools(const int32_t *cu_seqlens, int n_docs, int kpool, int32_t *cu_pools,
                            cudaStream_t s);
cudaError_t launch_compress(const void *k, const void *gate, const float *ape,
                            const int32_t *cu_seqlens, const int32_t *cu_pools, int n_docs,
                            int64_t T, int D, int kpool, int64_t P_total, void *pk_out,
                            uint8_t *pk_fp8, float *pk_scale, cudaStream_t s);
cudaError_t launch_quantize_fp8(const void *x, int64_t rows, uint8_t *out, float *scale,
                                cudaStream_t s);
cudaError_t launch_expand(const int32_t *pool_idx, const int32_t *cu_seqlens,
                          const int32_t *q_pos, const int32_t *cu_k, const int32_t *cu_pools,
                          int n_docs, int64_t T, int kpool, int Kp, int tail, int32_t *tok_idx,
                          cudaStream_t s);

// Scoring (kpool_score.cu).  mode 0 = top-k, 1 = dense scores.
struct ScoreArgs {
    const void *q;
    const float *q_scale;
    const float *w;
    const void *pk;
    const float *pk_scale;
    const int32_t *cu_seqlens;
    const int32_t *cu_pools;
    const int32_t *q_pos;    // per-document position of the first query row (NULL = 0)
    int n_docs;
    int64_t T;
    int64_t P_total;
    int H, D, kpool, Kp, fp8, mode;
    int32_t *pool_idx;
    float *pool_score;
    float *scores;
    int *ws;              // workspace header + schedule table
    size_t ws_bytes;
};
size_t score_workspace_bytes(int64_t T, int H, int n_docs);
// Bytes that also hold the split-pool schedule's tables and partial lists
// (equal to score_workspace_bytes when the call cannot use it).
size_t score_workspace_split_bytes(int64_t T, int H, int n_docs, int Kp);
int score_capacity(int H, int D, int fp8);   // candidate slots per query (0 = unsupported)
// Limit of one scoring-pipeline wait for later launches (0 = the 2 s
// default); returns the previous limit.
uint64_t set_wait_limit_ns(uint64_t ns);
uint64_t get_wait_limit_ns();

// The key path fused with compression (kpool_project.cu).
struct ProjectArgs {
    const void *x, *w;             // bf16 [T, hidden], bf16 [2D, hidden]
    const float *gamma, *beta, *ape;
    float eps;
    const int32_t *cu_seqlens, *cu_pools;
    int n_docs;
    int64_t T, P_total;
    int hidden, kpool;
    void *pk_out, *k_out, *gate_out;
    int *status;
};
int run_project_compress(const ProjectArgs &a, cudaStream_t s);
int run_score(const ScoreArgs &a, cudaStream_t s);
// Host-buffer pass with copies overlapped (kpool_pipeline.cu).  All input
// pointers are host memory; cu_seqlens_host NULL means one sequence (n_docs =
// 1); arguments are validated by the caller.
struct PipelineArgs {
    const void *q, *k, *gate;
    const float *ape, *w;
    const int32_t *cu_seqlens_host;
    int n_docs;
    int64_t T, P_total, chunk_rows;
    int H, D, kpool, index_topk, tail, fp8;
    int32_t *tok_out;
    void *scratch;
    size_t scratch_bytes;
};
size_t pipeline_scratch_bytes(int64_t T, int H, int D, int n_docs, int kpool, int index_topk,
                              int fp8, int64_t chunk_rows, int64_t P_total);
int run_pipeline(const PipelineArgs &a, cudaStream_t stream);

// TMA descriptor of a row-major bf16 [rows, cols] tensor: boxes of 64
// columns (128 bytes, 128-byte swizzle) x box_rows rows (kpool_project.cu).
int encode_bf16_tmap(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                     uint32_t box_rows);

// Sparse attention over the selection (kpool_mla.cu): tok_idx mode when
// tok_idx is given, else pool mode (the expansion of pool_idx fused in).
struct SparseMlaArgs {
    const void *q, *kv;                 // bf16 [T, 64, 512], bf16 [Tk, 512]
    const int32_t *tok_idx;             // [T, W] or NULL
    const int32_t *pool_idx;            // [T, Kp] (pool mode)
    const int32_t *cu_seqlens, *q_pos, *cu_k, *cu_pools;
    int n_docs;
    int64_t T, Tk;
    int W, kpool, Kp, tail;
    float scale;
    void *o;                            // bf16 [T, 64, 512]
    float *lse;                         // [T, 64]
    void *workspace;                    // >= sparse_mla_workspace_bytes(), 256-byte aligned
};
size_t sparse_mla_workspace_bytes();
int run_sparse_mla(const SparseMlaArgs &a, cudaStream_t s);

// Query tiles the fixed scratch of kpool_score_topk_noalloc can schedule.
constexpr int kNoAllocMaxTiles = 131072;
// Device address, size and tile capacity of the no-alloc scratch array of
// the current device (looked up on first use per device).
int noalloc_scratch(int **ptr, size_t *bytes, int64_t *max_tiles);

}  // namespace kpool
