// The key path in front of compression, fused into one tcgen05 kernel:
//
//   [k_proj | g] = x . [W_k ; W_g]^T          (BF16 operands, FP32 accumulation,
//                                             each output rounded to BF16)
//   k   = bf16( LayerNorm(k_proj) * gamma + beta )   (k_norm, FP32)
//   pk  = kpool compression of (k, g)                (as kpool_compress)
//
// Megatron-LM PR "GLM5.3 Flash (KDA + mHC + KPool DSA) support + FP8", Changes
// section 4 (linear_wk and k_norm run unquantized, in BF16) and section 3
// (the BF16 per-token compression gate, per-dimension softmax over the slots,
// FP32 accumulation, BF16 pooled key); SkyRL PR "GLM-5.3-Flash (glm5_next)
// Megatron support", commit "k-pool indexer" (softmax of gate_score + ape).
// The projected keys and gate never reach memory unless the caller asks for
// them.
//
// One persistent CTA per SM, 8 warps:
//   warp 0     TMA producer: x tile [128 tokens x 64] and W tile [256 x 64] per
//              K step through a ring of stages
//   warp 1     tcgen05.mma issuer (one thread): M = 128 tokens, N = 256
//              (D key features, then D gate features), K = hidden
//   warp 2     TMEM allocator (two 256-column accumulators)
//   warps 4-7  epilogue: one thread per token row (its TMEM lane); LayerNorm
//              in-thread; the kpool rows of a pool are kpool consecutive lanes
//              of one warp, so the softmax over slots runs on warp shuffles,
//              in the same operation order as kpool_compress (so the pooled
//              keys equal kpool_compress on the rounded k and g, bit for bit)
// A tile is 128 consecutive tokens of one document (tiles restart at
// document starts, so pools never straddle tiles: kpool divides 32).
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <mutex>

#include "kpool_internal.h"
#include "kpool_ptx.cuh"

namespace kpool {
namespace {

constexpr int kPThreads = 256;
constexpr int kPRows = 128;          // tokens per tile (TMEM lanes)
constexpr int kPCols = 256;          // accumulator columns: D = 128 keys + 128 gate
constexpr int kPD = 128;
constexpr int kPKChunk = 64;         // bf16 elements per 128-byte K step
constexpr int kPStages = 4;
constexpr uint32_t kPStageA = kPRows * 128;        // 16 KB
constexpr uint32_t kPStageB = kPCols * 128;        // 32 KB
constexpr uint64_t kPDrainNs = 2000000000ull;

// barrier indices: full[S], empty[S], acc_full[2], acc_empty[2], drain
constexpr int PB_FULL = 0, PB_EMPTY = kPStages, PB_ACC_FULL = 2 * kPStages,
              PB_ACC_EMPTY = 2 * kPStages + 2, PB_DRAIN = 2 * kPStages + 4, PB_COUNT = PB_DRAIN + 1;

struct ProjParams {
    const int32_t *cu_seqlens;   // NULL: one sequence
    const int32_t *cu_pools;
    int n_docs, T, hidden, kp, P_total;
    const float *gamma, *beta, *ape;
    float eps;
    uint16_t *pk, *k_out, *gate_out;
    int *status;
    uint64_t limit_ns;
};

struct PSync {
    volatile uint32_t *abort_flag;
    int *status;
    uint64_t limit_ns;
};

__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, const PSync &sy)
{
    if (ptx::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = ptx::globaltimer();
    while (true) {
        if (ptx::mbar_try_wait(bar, parity)) return true;
        if (*sy.abort_flag) return false;
        if (ptx::globaltimer() - t0 > sy.limit_ns) {
            *sy.abort_flag = 1u;
            atomicOr(sy.status, KPOOL_STATUS_TIMEOUT);
            return false;
        }
    }
}

// Walks the tiles of the call in a fixed order (document by document, 128
// rows at a time) and stops at the ones of this CTA (every grid-th).
struct TileWalk {
    int d = 0, i = 0, g = 0;   // document, tile within it, global tile index
    int doc_start = 0, doc_end = 0, pool_base = 0;

    __device__ void load_doc(const ProjParams &p)
    {
        if (p.cu_seqlens != nullptr) {
            doc_start = p.cu_seqlens[d];
            doc_end = p.cu_seqlens[d + 1];
            pool_base = p.cu_pools[d];
        } else {
            doc_start = 0;
            doc_end = p.T;
            pool_base = 0;
        }
    }
    // advance to global tile `target` (>= g); false once past the last tile
    __device__ bool seek(const ProjParams &p, int target)
    {
        while (d < p.n_docs) {
            load_doc(p);
            const int nt = (doc_end - doc_start + kPRows - 1) / kPRows;
            if (target < g + nt) {
                i = target - g;
                return true;
            }
            g += nt;
            ++d;
        }
        return false;
    }
    __device__ int row0() const { return doc_start + i * kPRows; }
};

__device__ __forceinline__ float bf16r(float x)
{
    return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t bf16_pair(float lo, float hi)
{
    const __nv_bfloat16 a = __float2bfloat16_rn(lo), b = __float2bfloat16_rn(hi);
    return static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(&a)) |
           (static_cast<uint32_t>(*reinterpret_cast<const uint16_t *>(&b)) << 16);
}

// Store 32 consecutive bf16 values (64 bytes) from registers.
__device__ __forceinline__ void store_bf16x32(uint16_t *dst, const float (&v)[32])
{
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q)
        d4[q] = make_uint4(bf16_pair(v[8 * q], v[8 * q + 1]), bf16_pair(v[8 * q + 2], v[8 * q + 3]),
                           bf16_pair(v[8 * q + 4], v[8 * q + 5]),
                           bf16_pair(v[8 * q + 6], v[8 * q + 7]));
}

template <int KP>
__global__ void __launch_bounds__(kPThreads, 1)
    project_compress_kernel(const __grid_constant__ CUtensorMap tm_x,
                            const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ ProjParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t sA = sbase, sB = sbase + kPStages * kPStageA;
    float *s_gamma = reinterpret_cast<float *>(smem + kPStages * (kPStageA + kPStageB));
    float *s_beta = s_gamma + kPD;
    float *s_ape = s_beta + kPD;                                       // [KP][128]
    uint64_t *bars = reinterpret_cast<uint64_t *>(s_ape + KP * kPD);
    uint32_t *misc = reinterpret_cast<uint32_t *>(bars + PB_COUNT);    // [0] tmem, [1] abort
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ksteps = p.hidden / kPKChunk;

    for (int j = threadIdx.x; j < kPD; j += kPThreads) {
        s_gamma[j] = p.gamma[j];
        s_beta[j] = p.beta[j];
    }
    for (int j = threadIdx.x; j < KP * kPD; j += kPThreads) s_ape[j] = p.ape[j];
    if (threadIdx.x == 0) {
        for (int s = 0; s < kPStages; ++s) {
            ptx::mbar_init(bar(PB_FULL + s), 1);
            ptx::mbar_init(bar(PB_EMPTY + s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            ptx::mbar_init(bar(PB_ACC_FULL + a), 1);
            ptx::mbar_init(bar(PB_ACC_EMPTY + a), 4);   // the four epilogue warps
        }
        ptx::mbar_init(bar(PB_DRAIN), 1);
        misc[1] = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 2) {
        ptx::tmem_alloc(ptx::smem_u32(&misc[0]), 512);
        ptx::tmem_relinquish();
        ptx::tc_fence_before();
    }
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    PSync sy{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.status, p.limit_ns};

    if (warp == 0) {
        // ---------------- TMA producer ----------------
        if (lane == 0) {
            ptx::tma_prefetch_desc(&tm_x);
            ptx::tma_prefetch_desc(&tm_w);
            TileWalk tw;
            uint32_t kc = 0, issued = 0;
            bool ok = true;
            for (int n = 0; ok && tw.seek(p, blockIdx.x + n * gridDim.x); ++n) {
                const int row0 = tw.row0();
                for (int ks = 0; ks < ksteps; ++ks, ++kc) {
                    const int st = kc % kPStages;
                    const uint32_t ph = (kc / kPStages) & 1u;
                    if (!pwait(bar(PB_EMPTY + st), ph ^ 1u, sy)) { ok = false; break; }
                    ptx::mbar_arrive_expect_tx(bar(PB_FULL + st), kPStageA + kPStageB);
                    ptx::tma_load_2d(sA + st * kPStageA, &tm_x, bar(PB_FULL + st), ks * kPKChunk, row0);
                    ptx::tma_load_2d(sB + st * kPStageB, &tm_w, bar(PB_FULL + st), ks * kPKChunk, 0);
                    issued = kc + 1;
                }
            }
            // let this thread's copies land before the CTA can exit (bounded)
            const uint64_t t0 = ptx::globaltimer();
            for (uint32_t c = issued > kPStages ? issued - kPStages : 0; c < issued; ++c) {
                const uint32_t st = c % kPStages, ph = (c / kPStages) & 1u;
                while (!ptx::mbar_try_wait(bar(PB_FULL + st), ph))
                    if (ptx::globaltimer() - t0 > kPDrainNs) break;
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            const uint32_t idesc = ptx::make_idesc(1u, kPRows, kPCols);
            TileWalk tw;
            uint32_t kc = 0, acc = 0, acc_ph = 0;
            bool ok = true, any = false;
            for (int n = 0; ok && tw.seek(p, blockIdx.x + n * gridDim.x); ++n) {
                if (!pwait(bar(PB_ACC_EMPTY + acc), acc_ph ^ 1u, sy)) break;
                ptx::tc_fence_after();
                const uint32_t d_tmem = tmem + acc * kPCols;
                for (int ks = 0; ks < ksteps; ++ks, ++kc) {
                    const int st = kc % kPStages;
                    const uint32_t ph = (kc / kPStages) & 1u;
                    if (!pwait(bar(PB_FULL + st), ph, sy)) { ok = false; break; }
                    ptx::tc_fence_after();
                    const uint64_t ad = ptx::smem_desc_sw128(sA + st * kPStageA);
                    const uint64_t bd = ptx::smem_desc_sw128(sB + st * kPStageB);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        ptx::mma_bf16(d_tmem, ad + kk * 2, bd + kk * 2, idesc, (ks | kk) != 0);
                    ptx::mma_commit(bar(PB_EMPTY + st));
                    any = true;
                }
                if (!ok) break;
                ptx::mma_commit(bar(PB_ACC_FULL + acc));
                if (++acc == 2) { acc = 0; acc_ph ^= 1u; }
            }
            if (any) {
                ptx::mma_commit(bar(PB_DRAIN));
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(bar(PB_DRAIN), 0))
                    if (ptx::globaltimer() - t0 > kPDrainNs) break;
            }
        }
    } else if (warp >= 4) {
        // ---------------- epilogue: one token row per thread ----------------
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;                    // row in the tile = TMEM lane
        const int s = r % KP;                                 // slot of this row in its pool
        const int base_lane = lane & ~(KP - 1);
        const float *ape_s = s_ape + s * kPD;
        TileWalk tw;
        uint32_t acc = 0, acc_ph = 0;
        for (int n = 0; tw.seek(p, blockIdx.x + n * gridDim.x); ++n) {
            const bool ok = __all_sync(0xFFFFFFFFu, pwait(bar(PB_ACC_FULL + acc), acc_ph, sy));
            if (!ok) break;
            ptx::tc_fence_after();
            const uint32_t taddr = tmem + (static_cast<uint32_t>(quarter * 32) << 16) + acc * kPCols;
            const int row = tw.row0() + r;                    // token
            const bool valid = row < tw.doc_end;
            const int local = tw.i * kPRows + r;              // position in the document
            // k_proj rounded to BF16; LayerNorm statistics in FP32, two passes
            float sum = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                ptx::tmem_ld32(taddr + c * 32, v);
                ptx::tmem_ld_wait(v);
#pragma unroll
                for (int j = 0; j < 32; ++j) sum += bf16r(__uint_as_float(v[j]));
            }
            const float mean = __fdiv_rn(sum, static_cast<float>(kPD));
            float sq = 0.f;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t v[32];
                ptx::tmem_ld32(taddr + c * 32, v);
                ptx::tmem_ld_wait(v);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const float dv = bf16r(__uint_as_float(v[j])) - mean;
                    sq = fmaf(dv, dv, sq);
                }
            }
            const float rs = __frcp_rn(__fsqrt_rn(__fadd_rn(__fdiv_rn(sq, static_cast<float>(kPD)), p.eps)));
            const bool pool_ok = s == 0 && tw.doc_start + local + KP <= tw.doc_end;
            const int64_t pool_g = static_cast<int64_t>(tw.pool_base) + local / KP;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t kvr[32], gvr[32];
                ptx::tmem_ld32(taddr + c * 32, kvr);
                ptx::tmem_ld32(taddr + kPD + c * 32, gvr);
                ptx::tmem_ld_wait2(kvr, gvr);
                if (c == 3) {
                    // every TMEM read of this accumulator is done: release it
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(PB_ACC_EMPTY + acc));
                }
                float kn[32], gv[32], pooled[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    const int dim = c * 32 + j;
                    const float t = (bf16r(__uint_as_float(kvr[j])) - mean) * rs;
                    kn[j] = bf16r(fmaf(t, s_gamma[dim], s_beta[dim]));
                    gv[j] = bf16r(__uint_as_float(gvr[j]));
                }
                if (valid && p.k_out != nullptr) store_bf16x32(p.k_out + static_cast<int64_t>(row) * kPD + c * 32, kn);
                if (valid && p.gate_out != nullptr) store_bf16x32(p.gate_out + static_cast<int64_t>(row) * kPD + c * 32, gv);
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    // softmax over the pool's slots (lanes base_lane .. +KP-1) in the
                    // order kpool_compress uses: max, then the exponentials summed
                    // slot by slot, then weight * key accumulated slot by slot
                    const float a = gv[j] + ape_s[c * 32 + j];
                    float m = a;
#pragma unroll
                    for (int o = 1; o < KP; o <<= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
                    const float e = expf(a - m);
                    float z = 0.f;
#pragma unroll
                    for (int q = 0; q < KP; ++q) z += __shfl_sync(0xFFFFFFFFu, e, base_lane + q);
                    const float alpha = __fdiv_rn(e, z);
                    float accv = 0.f;
#pragma unroll
                    for (int q = 0; q < KP; ++q)
                        accv = fmaf(__shfl_sync(0xFFFFFFFFu, alpha, base_lane + q),
                                    __shfl_sync(0xFFFFFFFFu, kn[j], base_lane + q), accv);
                    pooled[j] = accv;
                }
                if (pool_ok) store_bf16x32(p.pk + pool_g * kPD + c * 32, pooled);
            }
            if (++acc == 2) { acc = 0; acc_ph ^= 1u; }
        }
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 2) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, 512);
    }
}

typedef CUresult (*EncodeTiledFnP)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFnP get_encode_p()
{
    static EncodeTiledFnP fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFnP>(ptr);
    });
    return fn;
}

// bf16 [rows, cols] row-major, boxes of 64 columns (128 bytes, swizzled) x box_rows
int encode_bf16_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows, uint32_t box_rows)
{
    EncodeTiledFnP enc = get_encode_p();
    if (!enc) return fail(KPOOL_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), gdim,
                           gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KPOOL_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return KPOOL_OK;
}

template <int KP>
int launch_project_kp(const CUtensorMap &mx, const CUtensorMap &mw, const ProjParams &prm,
                      int grid, cudaStream_t s)
{
    const size_t smem = 1024 + kPStages * (kPStageA + kPStageB) + (2 + KP) * kPD * sizeof(float) +
                        PB_COUNT * 8 + 16;
    KPOOL_CUDA_CHECK(cudaFuncSetAttribute(project_compress_kernel<KP>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize,
                                          static_cast<int>(smem)));
    project_compress_kernel<KP><<<grid, kPThreads, smem, s>>>(mx, mw, prm);
    KPOOL_CUDA_CHECK(cudaGetLastError());
    return KPOOL_OK;
}

}  // namespace

int encode_bf16_tmap(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                     uint32_t box_rows)
{
    return encode_bf16_2d(m, base, cols, rows, box_rows);
}

int run_project_compress(const ProjectArgs &a, cudaStream_t s)
{
    KPOOL_CUDA_CHECK(cudaMemsetAsync(a.status, 0, sizeof(int), s));
    if (a.T == 0) return KPOOL_OK;
    CUtensorMap mx, mw;
    int rc = encode_bf16_2d(&mx, a.x, static_cast<uint64_t>(a.hidden), static_cast<uint64_t>(a.T),
                            kPRows);
    if (rc) return rc;
    rc = encode_bf16_2d(&mw, a.w, static_cast<uint64_t>(a.hidden), 2u * kPD, kPCols);
    if (rc) return rc;
    ProjParams prm{};
    prm.cu_seqlens = a.cu_seqlens;
    prm.cu_pools = a.cu_pools;
    prm.n_docs = a.n_docs;
    prm.T = static_cast<int>(a.T);
    prm.hidden = a.hidden;
    prm.kp = a.kpool;
    prm.P_total = static_cast<int>(a.P_total);
    prm.gamma = a.gamma;
    prm.beta = a.beta;
    prm.ape = a.ape;
    prm.eps = a.eps;
    prm.pk = static_cast<uint16_t *>(a.pk_out);
    prm.k_out = static_cast<uint16_t *>(a.k_out);
    prm.gate_out = static_cast<uint16_t *>(a.gate_out);
    prm.status = a.status;
    prm.limit_ns = get_wait_limit_ns();
    // tiles: one sequence ceil(T / 128); packed documents at most that plus one per document
    const int64_t tiles = (a.T + kPRows - 1) / kPRows + (a.cu_seqlens ? a.n_docs : 0);
    const int grid = static_cast<int>(std::min<int64_t>(num_sms(), tiles));
    switch (a.kpool) {
    case 1: return launch_project_kp<1>(mx, mw, prm, grid, s);
    case 2: return launch_project_kp<2>(mx, mw, prm, grid, s);
    case 4: return launch_project_kp<4>(mx, mw, prm, grid, s);
    case 8: return launch_project_kp<8>(mx, mw, prm, grid, s);
    case 16: return launch_project_kp<16>(mx, mw, prm, grid, s);
    case 32: return launch_project_kp<32>(mx, mw, prm, grid, s);
    default: return fail(KPOOL_ERR_UNSUPPORTED, "kpool must divide 32 for the fused projection");
    }
}

}  // namespace kpool
