/*
 * kpool.h -- C ABI of the GB300 (sm_103a) KPool DSA indexer library
 * (libkpool.so).
 *
 * The KPool indexer picks, for every query token, the key tokens a sparse
 * attention layer attends to.  Keys are first compressed kpool tokens at a
 * time into pooled keys; each query scores the complete pools of its causal
 * prefix, keeps the best index_topk / kpool pools, and expands them back to
 * token indices, appending its own incomplete pool (the "tail").  Source:
 * Megatron-LM PR "GLM5.3 Flash (KDA + mHC + KPool DSA) support + FP8",
 * Changes section 3 "KPool DSA indexer + NoPE"; SkyRL PR "GLM-5.3-Flash
 * (glm5_next) Megatron support", commit "k-pool indexer"; xtuner PR
 * "GLM-5.3-Flash F5: NoPE DSA + KPool indexer", Summary and commit notes.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer argument is a DEVICE pointer owned by the caller unless
 *    its name, or the function's, ends in _host (kpool_indexer_forward_host
 *    takes host buffers and a device scratch).  The library never allocates
 *    device memory and never frees what it is given; the host-buffer pass
 *    creates its streams and events once per host thread and device.
 *  - Each call enqueues its kernels on `stream` (NULL = legacy default
 *    stream) and returns without synchronising.  Results are valid once the
 *    stream has reached that point.
 *  - Return value: KPOOL_OK (0) or a negative KPOOL_ERR_* code.  All
 *    argument checks run on the host before anything is enqueued, so a
 *    rejected call leaves the device untouched.  kpool_last_error() returns
 *    a message for the last failing call of the calling thread.
 *  - Layouts are dense row-major.  bf16 tensors are passed as `const void*`
 *    (raw IEEE bfloat16 bits).  Indices are int32.
 *  - Document layout ("packed THD"): cu_seqlens[n_docs + 1] holds document
 *    start offsets into the token axis (cu_seqlens[0] = 0,
 *    cu_seqlens[n_docs] = T, non-decreasing).  cu_pools[n_docs + 1] holds
 *    the pool offsets, cu_pools[d+1] - cu_pools[d] = floor(L_d / kpool)
 *    (kpool_num_pools / kpool_cu_pools compute it).  Pools and causality
 *    restart at every document start.  Passing cu_seqlens = cu_pools = NULL
 *    with n_docs = 1 means one sequence of T tokens.
 *  - Pool p of document d covers tokens cu_seqlens[d] + j*kpool + s,
 *    s = 0..kpool-1, with j = p - cu_pools[d].  A trailing partial pool of a
 *    document is not compressed.  A query at document-local position tau
 *    may select the complete pools j < floor((tau + 1) / kpool).
 *  - Pool and token indices in outputs are global (packed) indices.
 */
#ifndef KPOOL_H_
#define KPOOL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KPOOL_API __attribute__((visibility("default")))
#else
#define KPOOL_API
#endif

struct CUstream_st;                 /* = cudaStream_t */
typedef struct CUstream_st *kpool_stream_t;

#define KPOOL_OK 0
#define KPOOL_ERR_INVALID_ARG (-1)  /* bad pointer, size, alignment or layout */
#define KPOOL_ERR_UNSUPPORTED (-2)  /* valid but outside the built shapes */
#define KPOOL_ERR_CUDA (-3)         /* a CUDA runtime/driver call failed */
#define KPOOL_ERR_WORKSPACE (-4)    /* workspace missing or too small */

/* Device status word bits (kpool_read_status). */
#define KPOOL_STATUS_TIMEOUT 1      /* a pipeline wait gave up; results invalid */
#define KPOOL_STATUS_BAD_SEQLENS 2  /* cu_seqlens not 0..T non-decreasing */

/* Message for the last failing call on this host thread ("" if none). */
KPOOL_API const char *kpool_last_error(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
KPOOL_API int kpool_version(void);

/*
 * kpool_num_pools -- host helper: validate a HOST copy of cu_seqlens and
 * fill cu_pools_host_out[n_docs + 1] (pool offsets, floor(L_d / kpool) pools
 * per document; Megatron-LM PR section 3: packed THD restarts pools at
 * document boundaries).  *total_pools_out receives cu_pools[n_docs].
 * Errors: KPOOL_ERR_INVALID_ARG if cu_seqlens is not 0..T non-decreasing,
 * kpool < 1, or a pointer is NULL.  Touches no device state.
 */
KPOOL_API int kpool_num_pools(const int32_t *cu_seqlens_host, int n_docs, int64_t T, int kpool,
                    int32_t *cu_pools_host_out, int64_t *total_pools_out);

/*
 * kpool_cu_pools -- device version of kpool_num_pools: cu_pools_out[n_docs+1]
 * from device cu_seqlens[n_docs+1].  One small kernel.  No validation of
 * the device values (see kpool_read_status for the scoring-time check).
 */
KPOOL_API int kpool_cu_pools(const int32_t *cu_seqlens, int n_docs, int kpool, int32_t *cu_pools_out,
                   kpool_stream_t stream);

/*
 * kpool_compress -- pool compression (Megatron-LM PR section 3; SkyRL
 * commit "k-pool indexer").  For every complete pool p and dimension d:
 *     a_s = float(gate[i_s, d]) + ape[s, d]        s = 0..kpool-1
 *     alpha = softmax_s(a)                          (FP32, max-subtracted)
 *     pk[p, d] = bf16_rne( sum_s alpha_s * float(k[i_s, d]) )   (FP32 sum)
 * with i_s the pool's s-th token.
 *   k, gate      bf16 [T, D], 16-byte aligned
 *   ape          fp32 [kpool, D]
 *   cu_seqlens, cu_pools   int32 [n_docs + 1] or both NULL (n_docs = 1)
 *   P_total      number of pools = cu_pools[n_docs] (T / kpool for one
 *                sequence); the host must know it to size pk_out
 *   pk_out       bf16 [P_total, D], 16-byte aligned
 *   pk_fp8_out, pk_scale_out   NULL, or E4M3 [P_total, D] and fp32
 *                [P_total]: the FP8 indexer input of the pooled key
 *                (see kpool_quantize_fp8; requires D = 128)
 * Supported: D in {32, 64, 128}; 1 <= kpool <= 64.
 * Errors: INVALID_ARG (NULL/misaligned pointers, bad sizes), UNSUPPORTED.
 */
KPOOL_API int kpool_compress(const void *k, const void *gate, const float *ape,
                   const int32_t *cu_seqlens, const int32_t *cu_pools, int n_docs,
                   int64_t T, int D, int kpool, int64_t P_total, void *pk_out,
                   uint8_t *pk_fp8_out, float *pk_scale_out, kpool_stream_t stream);

/*
 * kpool_project_compress -- the key path in front of compression fused with
 * it (Megatron-LM PR section 4: linear_wk and k_norm run unquantized in BF16;
 * section 3 and SkyRL commit "k-pool indexer": the BF16 per-token compression
 * gate, then the pooling of kpool_compress).  For every token t:
 *     kproj[t, :] = bf16_rne( x[t, :] . w_kg[0:D, :]^T )      (FP32 accumulation)
 *     gate[t, :]  = bf16_rne( x[t, :] . w_kg[D:2D, :]^T )
 *     k[t, :]     = bf16_rne( (kproj - mean) / sqrt(var + eps) * k_norm_weight
 *                             + k_norm_bias )                  (LayerNorm, FP32,
 *                                                               biased variance)
 * and pk is kpool_compress(k, gate, ape) -- bit for bit the same pooled keys.
 * The projected keys and gate are written only if k_out / gate_out are given.
 *   x            bf16 [T, hidden] hidden states, 16-byte aligned
 *   w_kg         bf16 [2D, hidden]: rows 0..D-1 the key projection, rows
 *                D..2D-1 the gate projection (a linear layer's weight layout)
 *   k_norm_weight, k_norm_bias   fp32 [D]
 *   ape, cu_seqlens, cu_pools, n_docs, T, P_total, pk_out   as kpool_compress
 *   k_out, gate_out   NULL or bf16 [T, D]
 *   workspace    >= 256 bytes, 256-byte aligned: its status word
 *                (kpool_read_status) reports a pipeline timeout
 * Supported: D = 128; hidden a multiple of 64; kpool in {1, 2, 4, 8, 16, 32}.
 * For FP8 pooled keys pass pk_out through kpool_quantize_fp8 (the same codes
 * kpool_compress's FP8 outputs hold).  The head-weight projection (FP32) and
 * the query projection are not part of this call.
 * Errors: INVALID_ARG, UNSUPPORTED, WORKSPACE.
 */
KPOOL_API int kpool_project_compress(const void *x, const void *w_kg, const float *k_norm_weight,
                                     const float *k_norm_bias, float k_norm_eps, const float *ape,
                                     const int32_t *cu_seqlens, const int32_t *cu_pools,
                                     int n_docs, int64_t T, int hidden, int D, int kpool,
                                     int64_t P_total, void *pk_out, void *k_out, void *gate_out,
                                     void *workspace, size_t workspace_bytes,
                                     kpool_stream_t stream);

/*
 * kpool_quantize_fp8 -- FP8 indexer input emulation (Megatron-LM PR
 * section 3: FP32 Hadamard -> BF16 -> E4M3 with a power-of-two row scale).
 * For each row r of x (bf16 [rows, 128]):
 *     y = H128 x / sqrt(128)         FP32, Sylvester-order Hadamard
 *     b = bf16_rne(y)
 *     s = smallest power of two with max|b| <= 448 s   (1 for a zero row)
 *     x_fp8_out[r] = e4m3_rne_satfinite(b / s),  scale_out[r] = s
 * so that x ~= x_fp8 * s after the rotation.  For q [T, H, 128] pass
 * rows = T * H.
 *   x            bf16 [rows, D], 16-byte aligned; D must be 128
 *   x_fp8_out    uint8 (E4M3) [rows, D]; scale_out fp32 [rows]
 */
KPOOL_API int kpool_quantize_fp8(const void *x, int64_t rows, int D, uint8_t *x_fp8_out,
                       float *scale_out, kpool_stream_t stream);

/*
 * kpool_score_topk_workspace_size -- bytes of device workspace that
 * kpool_score_topk / kpool_score_dense need for T tokens, H heads and n_docs
 * documents (a tile counter, a status word and the query-tile schedule).
 */
KPOOL_API size_t kpool_score_topk_workspace_size(int64_t T, int H, int n_docs);

/*
 * kpool_score_topk_workspace_size_split -- bytes of a workspace that also
 * lets kpool_score_topk / kpool_score_topk_at split long pool lists over
 * several CTAs when a call has few query tiles (decode batches, short
 * chunks: at most 1024 tiles of 256 / H rows).  Each query tile's pools are
 * then scored in units (of at least 32 pool tiles) on different SMs, provided
 * 2 * Kp fits the per-query candidate capacity; every unit keeps its own best Kp
 * (the same scores, the same order: score descending, ties to the lower
 * pool index) and the last unit to finish merges them, so the outputs are
 * identical to the unsplit schedule's.  Equal to
 * kpool_score_topk_workspace_size(T, H, n_docs) when the call is not
 * eligible; 0 for unsupported arguments.  A workspace at least this large
 * enables the split schedule; a smaller valid one runs unsplit.
 */
KPOOL_API size_t kpool_score_topk_workspace_size_split(int64_t T, int H, int n_docs, int kpool,
                                                       int index_topk);

/*
 * kpool_score_topk -- causal pool scoring fused with top-k selection
 * (Megatron-LM PR section 3: top-k over index_topk // kpool pools; xtuner
 * PR: relu homogeneity lets any head_dim^-0.5 factor live in w).
 *     score[t, p] = sum_h w[t, h] * relu( sum_d q[t, h, d] * pk[p, d] )
 * over the complete causal pools p of t's document (local index
 * j < floor((tau+1)/kpool)).  Each row t keeps the Kp = index_topk / kpool
 * pools of largest score (ties to the lower pool index; every visible pool
 * when there are at most Kp), written in ascending pool order:
 *     pool_idx_out[t, 0..Kp)    int32 global pool index, -1 padding
 *     pool_score_out[t, 0..Kp)  fp32 score, -inf padding
 * The T x P score matrix is never written to memory.
 * FP8 mode (fp8 = 1): q and pk are E4M3 codes [T, H, 128] / [P, 128] with
 * fp32 scales q_scale [T, H] and pk_scale [P] (kpool_quantize_fp8 /
 * kpool_compress), and
 *     score = pk_scale[p] * sum_h w[t,h] q_scale[t,h] relu(q_fp8 . pk_fp8)
 * In bf16 mode q_scale and pk_scale must be NULL.
 *   q            bf16 [T, H, D] (or E4M3), 16-byte aligned
 *   w            fp32 [T, H]
 *   pk           bf16 [P_total, D] (or E4M3), 16-byte aligned
 *   workspace    >= kpool_score_topk_workspace_size(T, H, n_docs) bytes
 *                (kpool_score_topk_workspace_size_split for the split-pool
 *                schedule), 256-byte aligned; its contents are overwritten.
 *                Calls that share one workspace must not overlap on the
 *                device.
 * Supported: H in {4, 8, 16, 32, 64, 128}; D in {32, 64, 128} (128 in FP8
 * mode); Kp <= a per-H capacity (UNSUPPORTED beyond it).
 * Device-side: cu_seqlens is validated by the schedule kernel; on failure
 * or on an internal pipeline timeout the status word (kpool_read_status)
 * is set and the outputs are not written.
 */
KPOOL_API int kpool_score_topk(const void *q, const float *q_scale, const float *w, const void *pk,
                     const float *pk_scale, const int32_t *cu_seqlens, const int32_t *cu_pools,
                     int n_docs, int64_t T, int64_t P_total, int H, int D, int kpool,
                     int index_topk, int fp8, int32_t *pool_idx_out, float *pool_score_out,
                     void *workspace, size_t workspace_bytes, kpool_stream_t stream);

/*
 * kpool_score_topk_at -- kpool_score_topk for query rows at given positions
 * of their documents (decode and chunked prefill: the queries are fewer than
 * the keys).  Document d's query rows are [cu_seqlens_q[d], cu_seqlens_q[d+1])
 * of q and w; its i-th query row sits at document-local position
 * q_start_pos[d] + i of the key sequence whose pooled keys are
 * pk[cu_pools[d] .. cu_pools[d+1]) (from kpool_compress on the keys).  A query
 * at position tau scores the complete pools j < floor((tau+1)/kpool), clamped
 * to the document's pools.  With q_start_pos = 0 and the keys' cu_seqlens as
 * cu_seqlens_q this is kpool_score_topk.  The caller keeps every position
 * inside its document (q_start_pos[d] + rows_d <= the document's key count);
 * the device does not check it (pools clamp to the document's, but the tail
 * tokens kpool_expand_indices_at writes for a position past the keys would
 * point past them).  All three index arrays are device
 * int32 and required; Tq = cu_seqlens_q[n_docs]; the workspace is sized by
 * kpool_score_topk_workspace_size(Tq, H, n_docs), or by
 * kpool_score_topk_workspace_size_split(Tq, H, n_docs, kpool, index_topk)
 * to let a decode batch spread each document's pools over the SMs.  Outputs as in
 * kpool_score_topk (global pool indices, ascending).
 */
KPOOL_API int kpool_score_topk_at(const void *q, const float *q_scale, const float *w,
                                  const void *pk, const float *pk_scale,
                                  const int32_t *cu_seqlens_q, const int32_t *q_start_pos,
                                  const int32_t *cu_pools, int n_docs, int64_t Tq, int64_t P_total,
                                  int H, int D, int kpool, int index_topk, int fp8,
                                  int32_t *pool_idx_out, float *pool_score_out, void *workspace,
                                  size_t workspace_bytes, kpool_stream_t stream);

/*
 * kpool_expand_indices_at -- kpool_expand_indices for positioned queries:
 * pool p of document d expands to key tokens cu_seqlens_k[d] + j*kpool + s,
 * and the tail of a query at position tau is the key tokens
 * cu_seqlens_k[d] + tau - r + 1 .. cu_seqlens_k[d] + tau, r = (tau+1) mod
 * kpool (the query's own token must lie in its key sequence).
 */
KPOOL_API int kpool_expand_indices_at(const int32_t *pool_idx, const int32_t *cu_seqlens_q,
                                      const int32_t *q_start_pos, const int32_t *cu_seqlens_k,
                                      const int32_t *cu_pools, int n_docs, int64_t Tq, int kpool,
                                      int index_topk, int always_select_tail,
                                      int32_t *tok_idx_out, kpool_stream_t stream);

/*
 * kpool_score_topk_noalloc -- the same computation, arguments and outputs as
 * kpool_score_topk, for callers that cannot allocate device memory: code
 * running where cudaMalloc is not allowed or not wanted, such as inside a
 * framework's custom-op or plugin hook that only hands out its input and
 * output buffers, or an inference runtime that reserves all device memory
 * up front and forbids allocation afterwards.  (The pages have no
 * counterpart of this entry point.)
 *   - No workspace argument: the scratch (tile counter, status word and
 *     query-tile schedule) lives in a fixed array inside the library, about
 *     1 MiB, held on every device that loads the library until the process
 *     exits.  This call itself allocates nothing.
 *   - Capacity: ceil(T / (256 / H)) + n_docs <= 131072 query tiles (e.g.
 *     T up to 524288 - 4 * n_docs tokens at H = 64).  Larger inputs are
 *     rejected with KPOOL_ERR_UNSUPPORTED before anything is enqueued.
 *   - The first call on a device looks up the array's device address (once
 *     per device, with that device current); make that first call before
 *     any stream capture.
 *   - Every call on a device shares the one array.  Each call rewrites
 *     everything it reads from it before use, but calls that overlap on the
 *     GPU (different streams, or host threads) race on it and must be
 *     serialised by the caller.
 *   - Its status word (malformed cu_seqlens, an expired pipeline wait) is
 *     read with kpool_score_topk_noalloc_status.
 *   - It always runs the unsplit schedule (one unit per query tile): the
 *     fixed array has no room for the split-pool tables, so decode-sized
 *     calls (few query tiles over long documents) run on fewer SMs and more
 *     slowly than kpool_score_topk given a split-sized workspace.  Results
 *     are the same.
 */
KPOOL_API int kpool_score_topk_noalloc(const void *q, const float *q_scale, const float *w,
                                       const void *pk, const float *pk_scale,
                                       const int32_t *cu_seqlens, const int32_t *cu_pools,
                                       int n_docs, int64_t T, int64_t P_total, int H, int D,
                                       int kpool, int index_topk, int fp8, int32_t *pool_idx_out,
                                       float *pool_score_out, kpool_stream_t stream);

/*
 * kpool_score_topk_noalloc_status -- the status word (KPOOL_STATUS_* bits, 0 =
 * clean) that the last kpool_score_topk_noalloc on the current device left in
 * the library's fixed scratch: KPOOL_STATUS_BAD_SEQLENS when the device
 * cu_seqlens were malformed (nothing was written to the outputs),
 * KPOOL_STATUS_TIMEOUT when a pipeline wait gave up (outputs invalid).
 * Synchronises the whole device, like kpool_read_status.  Allocates nothing.
 * (The pages have no counterpart: it belongs to the allocation-free entry
 * point.)
 */
KPOOL_API int kpool_score_topk_noalloc_status(int *status_out);

/*
 * kpool_score_dense -- test/debug entry: the same scoring as
 * kpool_score_topk (same kernel pipeline, no selection) written out in full:
 * scores_out[t, p] (fp32 [T, P_total]) for every complete causal pool p of
 * t's document, -inf elsewhere.  Meant for small T only.
 */
KPOOL_API int kpool_score_dense(const void *q, const float *q_scale, const float *w, const void *pk,
                      const float *pk_scale, const int32_t *cu_seqlens, const int32_t *cu_pools,
                      int n_docs, int64_t T, int64_t P_total, int H, int D, int kpool, int fp8,
                      float *scores_out, void *workspace, size_t workspace_bytes,
                      kpool_stream_t stream);

/*
 * kpool_expand_indices -- expansion of selected pools to token indices plus
 * the causal tail (Megatron-LM PR section 3: fused_qk_topk_kpool expands
 * pools back to tokens; always_select_tail appends each query's incomplete
 * causal pool so short prefixes stay fully visible).  Row t of
 * tok_idx_out [T, W], W = Kp*kpool + kpool - 1:
 *   for each of the first min(n_c, Kp) entries of pool_idx[t] (ascending
 *   pools as written by kpool_score_topk) its kpool tokens; then, if
 *   always_select_tail and r = (tau+1) mod kpool != 0, the r tokens
 *   t-r+1 .. t; then -1 padding.  Rows are strictly ascending.
 * An entry of pool_idx outside t's document expands to -1s.
 */
KPOOL_API int kpool_expand_indices(const int32_t *pool_idx, const int32_t *cu_seqlens,
                         const int32_t *cu_pools, int n_docs, int64_t T, int kpool,
                         int index_topk, int always_select_tail, int32_t *tok_idx_out,
                         kpool_stream_t stream);

/*
 * kpool_indexer_forward_host -- the whole indexer pass from HOST buffers to
 * HOST token indices (Megatron-LM PR section 3: compression, pool top-k,
 * expansion with the causal tail, packed THD; the FP8 input path), with the
 * host<->device copies overlapped with the kernels.  Keys are copied and
 * compressed first; the query rows then go in chunks of up to chunk_rows
 * (0 = 16384; the first and last chunks ramp from chunk_rows / 8) over three
 * internal streams: the copy-in of chunk c+1, the scoring and expansion of
 * chunk c and the copy-out of chunk c-1 run concurrently.
 * Each chunk is scored as positioned queries over the global pooled keys, so
 * tok_idx_out equals what kpool_compress -> [kpool_quantize_fp8] ->
 * kpool_score_topk -> kpool_expand_indices give on the same inputs.
 *   q      bf16 [T, H, D]      k, gate  bf16 [T, D]     ape  fp32 [kpool, D]
 *   w      fp32 [T, H]         tok_idx_out  int32 [T, Kp*kpool + kpool - 1]
 *   cu_seqlens_host  int32 [n_docs + 1] host array (NULL = one sequence,
 *                    n_docs = 1), validated on the host
 * All of these are host memory; page-locked (cudaHostAlloc / pinned)
 * buffers are needed for the copies to overlap, pageable ones work but
 * serialise.  fp8 = 1 runs the FP8 mode (D = 128).
 *   scratch  device memory of at least kpool_indexer_forward_host_scratch_size
 *            bytes, 256-byte aligned, owned by the caller; its first 256 bytes
 *            carry the pass's status word (kpool_read_status(scratch, ...)).
 * Asynchronous on `stream`: the call returns once the work is enqueued, and
 * `stream` waits for the last copy-out; synchronise it before reading
 * tok_idx_out or reusing the host inputs.  The internal streams and events
 * belong to the calling host thread (created on its first call per device).
 * Errors: as kpool_score_topk, plus KPOOL_ERR_WORKSPACE for a short scratch.
 */
KPOOL_API size_t kpool_indexer_forward_host_scratch_size(const int32_t *cu_seqlens_host,
                                                         int n_docs, int64_t T, int H, int D,
                                                         int kpool, int index_topk, int fp8,
                                                         int64_t chunk_rows);
KPOOL_API int kpool_indexer_forward_host(const void *q, const void *k, const void *gate,
                                         const float *ape, const float *w,
                                         const int32_t *cu_seqlens_host, int n_docs, int64_t T,
                                         int H, int D, int kpool, int index_topk,
                                         int always_select_tail, int fp8, int64_t chunk_rows,
                                         int32_t *tok_idx_out, void *scratch,
                                         size_t scratch_bytes, kpool_stream_t stream);

/*
 * Sparse attention over the selection: the absorbed NoPE MLA forward that
 * consumes the indexer's output (xtuner PR "GLM-5.3-Flash F5: NoPE DSA +
 * KPool indexer + clamped SwiGLU", Summary: a FlashMLA-style SparseMLA
 * forward over the selected token indices, 64 heads in the production
 * config, head and value width 512 once the rotary slice is gone; Megatron-LM
 * PR section 3, "NoPE": the absorbed query has no positional slice).  Keys and
 * values are the same latent rows kv[j].  For query row t and head h, over the
 * row's token list J(t):
 *     s_j        = softmax_scale * sum_d q[t, h, d] * kv[j, d]     (FP32)
 *     o[t, h, :] = sum_j softmax_j(s) kv[j, :]                      (BF16 out)
 *     lse[t, h]  = ln sum_j exp(s_j)                                (FP32 out)
 * A listed index counts once per listing; -1 entries (and indices outside
 * [0, Tk)) are skipped; a row with no token gets o = 0 and lse = -inf.
 * Arithmetic: tcgen05 MMAs with FP32 accumulation; the softmax weights are
 * rounded to BF16 before they multiply kv (the sums use the FP32 weights).
 *   q            bf16 [T, H, Dc] absorbed queries, 16-byte aligned
 *   kv           bf16 [Tk, Dc] latent rows, 16-byte aligned
 *   o_out        bf16 [T, H, Dc], 16-byte aligned;  lse_out fp32 [T, H]
 *   workspace    >= kpool_sparse_mla_workspace_size() bytes, 256-byte
 *                aligned; its status word (kpool_read_status) reports a
 *                pipeline timeout (KPOOL_STATUS_TIMEOUT: outputs invalid)
 * Supported: H = 64, Dc = 512 (UNSUPPORTED otherwise); softmax_scale finite
 * and > 0.
 *
 * kpool_sparse_mla_fwd -- J(t) is row t of tok_idx (int32 [T, W], as written
 * by kpool_expand_indices, or any list with -1 padding).
 */
KPOOL_API size_t kpool_sparse_mla_workspace_size(void);
KPOOL_API int kpool_sparse_mla_fwd(const void *q, const void *kv, const int32_t *tok_idx,
                                   int64_t T, int64_t Tk, int W, int H, int Dc,
                                   float softmax_scale, void *o_out, float *lse_out,
                                   void *workspace, size_t workspace_bytes, kpool_stream_t stream);

/*
 * kpool_sparse_mla_fwd_pools -- the same attention fused with the expansion:
 * J(t) is what kpool_expand_indices would write for row t of pool_idx (the
 * selected pools' kpool tokens in order, then the causal tail when
 * always_select_tail), built on the fly so that the token table never
 * reaches memory.  Keys are the query tokens themselves (Tk = T).
 * pool_idx int32 [T, index_topk / kpool] as written by kpool_score_topk
 * (a row's first min(n_c, Kp) entries are its pools); cu_seqlens, cu_pools,
 * n_docs as kpool_expand_indices.
 */
KPOOL_API int kpool_sparse_mla_fwd_pools(const void *q, const void *kv, const int32_t *pool_idx,
                                         const int32_t *cu_seqlens, const int32_t *cu_pools,
                                         int n_docs, int64_t T, int H, int Dc, int kpool,
                                         int index_topk, int always_select_tail,
                                         float softmax_scale, void *o_out, float *lse_out,
                                         void *workspace, size_t workspace_bytes,
                                         kpool_stream_t stream);

/*
 * kpool_sparse_mla_fwd_pools_at -- kpool_sparse_mla_fwd_pools for positioned
 * queries (decode, chunked prefill): J(t) is what kpool_expand_indices_at
 * would write; kv holds the Tk key tokens indexed by cu_seqlens_k.
 */
KPOOL_API int kpool_sparse_mla_fwd_pools_at(const void *q, const void *kv, const int32_t *pool_idx,
                                            const int32_t *cu_seqlens_q, const int32_t *q_start_pos,
                                            const int32_t *cu_seqlens_k, const int32_t *cu_pools,
                                            int n_docs, int64_t Tq, int64_t Tk, int H, int Dc,
                                            int kpool, int index_topk, int always_select_tail,
                                            float softmax_scale, void *o_out, float *lse_out,
                                            void *workspace, size_t workspace_bytes,
                                            kpool_stream_t stream);

/*
 * kpool_read_status -- debug helper: synchronously copy the device status
 * word of a workspace (KPOOL_STATUS_* bits, 0 = clean) to *status_out.
 * Synchronises the whole device.
 */
KPOOL_API int kpool_read_status(const void *workspace, int *status_out);

/*
 * kpool_debug_set_wait_limit_ns -- test entry: the time limit of each wait
 * inside the scoring kernel (kpool_score_topk, _at, _noalloc, _dense and the
 * host-buffer pass) and the sparse attention (kpool_sparse_mla_*) for
 * launches made after this call, process-wide; ns = 0
 * restores the default of 2 s.  Returns the previous limit.  A wait that
 * runs out sets KPOOL_STATUS_TIMEOUT in the call's status word and raises an
 * abort flag in its CTA: the CTA's roles stop waiting, let their in-flight
 * copies and MMAs land (bounded by 2 s whatever this limit), free their
 * tensor memory and exit, and the outputs of that call are invalid.  Meant
 * for tests of that path; production code leaves the default.  (The pages
 * have no counterpart.)
 */
KPOOL_API uint64_t kpool_debug_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* KPOOL_H_ */
