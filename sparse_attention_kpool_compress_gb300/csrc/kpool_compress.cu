// Pool compression and the FP8 indexer-input emulation.
//
// Compression (Megatron-LM PR "GLM5.3 Flash (KDA + mHC + KPool DSA) support +
// FP8", Changes section 3; SkyRL PR "GLM-5.3-Flash (glm5_next) Megatron
// support", commit "k-pool indexer"): every dimension of a pool takes a
// softmax over the pool's kpool slots of gate + ape, the weighted keys are
// summed in FP32 and rounded once to BF16.
//
// FP8 emulation (same Megatron-LM section): FP32 Hadamard rotation -> BF16 ->
// E4M3 with a power-of-two scale per 128-element row.
//
// Both are HBM streams.  One thread owns 8 consecutive dimensions (one 16-byte
// vector) of one pool or row; a 128-dim row is 16 lanes of one warp, so the
// 128-point Walsh-Hadamard transform runs as 3 in-thread butterfly stages and
// 4 xor-shuffle stages.
#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "kpool_internal.h"

namespace kpool {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ void bf16x8_to_f32(const uint4 &u, float (&f)[8])
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
}

__device__ __forceinline__ uint32_t bf16_bits_rn(float x)
{
    __nv_bfloat16 b = __float2bfloat16_rn(x);
    return static_cast<uint32_t>(*reinterpret_cast<uint16_t *>(&b));
}

// Last document whose pool range starts at or before pool g (skips empty
// documents that share the same start).
__device__ __forceinline__ int find_doc(const int32_t *cu, int n_docs, int64_t g)
{
    int lo = 0, hi = n_docs;   // answer in [0, n_docs)
    while (hi - lo > 1) {
        int mid = (lo + hi) >> 1;
        if (cu[mid] <= g) lo = mid;
        else hi = mid;
    }
    return lo;
}

// FP8 emulation of one 128-element row held by a 16-lane group (8 values per
// lane, lane v owns elements 8v..8v+7).  Writes this lane's 8 E4M3 codes and,
// from lane v == 0, the row scale.
__device__ __forceinline__ void fp8_row(float (&x)[8], int v, uint8_t *codes8, float *scale_out,
                                        bool active)
{
    // Walsh-Hadamard butterflies in natural (Sylvester) order, FP32.
#pragma unroll
    for (int h = 1; h < 8; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if ((i & h) == 0) {
                float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float o = __shfl_xor_sync(0xFFFFFFFFu, x[i], m);
            x[i] = (v & m) ? (o - x[i]) : (x[i] + o);
        }
    }
    const float norm = 0.08838834764831845f;   // 128^-1/2
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        x[i] = __uint_as_float(bf16_bits_rn(x[i] * norm) << 16);
        amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int m = 1; m < 16; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
    // smallest power of two s with amax <= 448 s: amax = f * 2^E, f in [0.5, 1),
    // 448 = 0.875 * 2^9  ->  s = 2^(E - 9 + (f > 0.875)).
    int e = 0;
    if (amax > 0.f) {
        int E;
        const float f = frexpf(amax, &E);
        e = E - 9 + (f > 0.875f ? 1 : 0);
    }
    const float s = ldexpf(1.f, e);
    if (!active) return;
    // x / s exactly: a multiply by the power of two 2^-e when that is a normal
    // float, otherwise an exact exponent shift
    const bool mul_ok = e > -126 && e < 126;
    const float inv = mul_ok ? ldexpf(1.f, -e) : 1.f;
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const float y = mul_ok ? x[i] * inv : ldexpf(x[i], -e);
        uint32_t c = static_cast<uint32_t>(__nv_cvt_float_to_fp8(y, __NV_SATFINITE, __NV_E4M3));
        if (i < 4) lo |= c << (8 * i);
        else hi |= c << (8 * (i - 4));
    }
    *reinterpret_cast<uint2 *>(codes8) = make_uint2(lo, hi);
    if (v == 0) *scale_out = s;
}

// KP > 0: kpool known at compile time -- every slot's 16-byte gate and key
// vectors are loaded up front and the softmax weights stay in registers.
// KP == 0: any kpool, slots re-read from L1 in three passes.
template <int KP>
__global__ void __launch_bounds__(kThreads) compress_kernel(
    const uint16_t *__restrict__ k, const uint16_t *__restrict__ gate,
    const float *__restrict__ ape, const int32_t *__restrict__ cu_seqlens,
    const int32_t *__restrict__ cu_pools, int n_docs, int D, int kp_rt, int64_t P_total,
    uint16_t *__restrict__ pk, uint8_t *__restrict__ pk_fp8, float *__restrict__ pk_scale)
{
    const int kp = KP > 0 ? KP : kp_rt;
    const int vpr = D >> 3;
    const int64_t gid = static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x;
    const int64_t g = gid / vpr;
    const int v = static_cast<int>(gid - g * vpr);
    const bool active = g < P_total;

    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;

    if (active) {
        int64_t tok0;
        if (cu_pools != nullptr) {
            int d = find_doc(cu_pools, n_docs, g);
            tok0 = static_cast<int64_t>(cu_seqlens[d]) + (g - cu_pools[d]) * kp;
        } else {
            tok0 = g * kp;
        }
        const int col = v * 8;
        if constexpr (KP > 0) {
            uint4 gq[KP], kq[KP];
#pragma unroll
            for (int s = 0; s < KP; ++s) {
                gq[s] = __ldg(reinterpret_cast<const uint4 *>(gate + (tok0 + s) * D + col));
                kq[s] = __ldg(reinterpret_cast<const uint4 *>(k + (tok0 + s) * D + col));
            }
            float a[KP][8], m[8], z[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) { m[i] = -INFINITY; z[i] = 0.f; }
#pragma unroll
            for (int s = 0; s < KP; ++s) {
                float gv[8];
                bf16x8_to_f32(gq[s], gv);
                const float4 a0 = __ldg(reinterpret_cast<const float4 *>(ape + s * D + col));
                const float4 a1 = __ldg(reinterpret_cast<const float4 *>(ape + s * D + col + 4));
                const float ap[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    a[s][i] = gv[i] + ap[i];
                    m[i] = fmaxf(m[i], a[s][i]);
                }
            }
#pragma unroll
            for (int s = 0; s < KP; ++s)
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    a[s][i] = expf(a[s][i] - m[i]);
                    z[i] += a[s][i];
                }
#pragma unroll
            for (int s = 0; s < KP; ++s) {
                float kv[8];
                bf16x8_to_f32(kq[s], kv);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = fmaf(__fdiv_rn(a[s][i], z[i]), kv[i], acc[i]);
            }
        } else {
        float m[8], z[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) { m[i] = -INFINITY; z[i] = 0.f; }
        // softmax over slots of a_s = gate + ape, per dimension
        for (int s = 0; s < kp; ++s) {
            float gv[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(gate + (tok0 + s) * D + col), gv);
            const float4 a0 = *reinterpret_cast<const float4 *>(ape + s * D + col);
            const float4 a1 = *reinterpret_cast<const float4 *>(ape + s * D + col + 4);
            const float ap[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) m[i] = fmaxf(m[i], gv[i] + ap[i]);
        }
        for (int s = 0; s < kp; ++s) {
            float gv[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(gate + (tok0 + s) * D + col), gv);
            const float4 a0 = *reinterpret_cast<const float4 *>(ape + s * D + col);
            const float4 a1 = *reinterpret_cast<const float4 *>(ape + s * D + col + 4);
            const float ap[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) z[i] += expf((gv[i] + ap[i]) - m[i]);
        }
        for (int s = 0; s < kp; ++s) {
            float gv[8], kv[8];
            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(gate + (tok0 + s) * D + col), gv);
            bf16x8_to_f32(*reinterpret_cast<const uint4 *>(k + (tok0 + s) * D + col), kv);
            const float4 a0 = *reinterpret_cast<const float4 *>(ape + s * D + col);
            const float4 a1 = *reinterpret_cast<const float4 *>(ape + s * D + col + 4);
            const float ap[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float alpha = __fdiv_rn(expf((gv[i] + ap[i]) - m[i]), z[i]);
                acc[i] = fmaf(alpha, kv[i], acc[i]);
            }
        }
        }
        uint32_t o[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            o[i] = bf16_bits_rn(acc[2 * i]) | (bf16_bits_rn(acc[2 * i + 1]) << 16);
        *reinterpret_cast<uint4 *>(pk + g * D + col) = make_uint4(o[0], o[1], o[2], o[3]);
    }

    if (pk_fp8 != nullptr) {   // D == 128: a row is 16 lanes of this warp
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(bf16_bits_rn(acc[i]) << 16);
        fp8_row(x, v, pk_fp8 + (active ? g : 0) * 128 + v * 8, pk_scale + (active ? g : 0),
                active);
    }
}

// The same chain for rows handled by 8 threads of 16 elements (slice v of the
// row): butterflies over element-index bits 0-3 in the thread, bits 4-6 across
// threads, in the same stage order as fp8_row, so the results are identical.
__device__ __forceinline__ void fp8_row16(float (&x)[16], int v, uint8_t *codes16,
                                          float *scale_out, bool active)
{
#pragma unroll
    for (int h = 1; h < 16; h <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            if ((i & h) == 0) {
                float a = x[i], b = x[i + h];
                x[i] = a + b;
                x[i + h] = a - b;
            }
        }
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            float o = __shfl_xor_sync(0xFFFFFFFFu, x[i], m);
            x[i] = (v & m) ? (o - x[i]) : (x[i] + o);
        }
    }
    const float norm = 0.08838834764831845f;   // 128^-1/2
    float amax = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        x[i] = __uint_as_float(bf16_bits_rn(x[i] * norm) << 16);
        amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int m = 1; m < 8; m <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, m));
    int e = 0;
    if (amax > 0.f) {
        int E;
        const float f = frexpf(amax, &E);
        e = E - 9 + (f > 0.875f ? 1 : 0);
    }
    const float s = ldexpf(1.f, e);
    if (!active) return;
    const bool mul_ok = e > -126 && e < 126;
    const float inv = mul_ok ? ldexpf(1.f, -e) : 1.f;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
    for (int i = 0; i < 16; i += 2) {
        const float y0 = mul_ok ? x[i] * inv : ldexpf(x[i], -e);
        const float y1 = mul_ok ? x[i + 1] * inv : ldexpf(x[i + 1], -e);
        // element i in the low byte, i + 1 in the high byte
        const uint32_t c2 = static_cast<uint32_t>(
            __nv_cvt_float2_to_fp8x2(make_float2(y0, y1), __NV_SATFINITE, __NV_E4M3));
        w[i >> 2] |= c2 << (8 * (i & 3));
    }
    *reinterpret_cast<uint4 *>(codes16) = make_uint4(w[0], w[1], w[2], w[3]);
    if (v == 0) *scale_out = s;
}

// q rows: 8 threads per row; a warp covers 8 consecutive rows, each thread two
// of them (rows 4 apart), with all four 16-byte loads issued before any math.
constexpr int kQuantRowsPerWarp = 8;

__global__ void __launch_bounds__(kThreads) quantize_fp8_kernel(
    const uint16_t *__restrict__ x, int64_t rows, uint8_t *__restrict__ out,
    float *__restrict__ scale)
{
    const int lane = threadIdx.x & 31;
    const int64_t warp = (static_cast<int64_t>(blockIdx.x) * kThreads + threadIdx.x) >> 5;
    const int v = lane & 7;
    int64_t r[2];
    bool act[2];
    uint4 raw[2][2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        r[k] = warp * kQuantRowsPerWarp + 4 * k + (lane >> 3);
        act[k] = r[k] < rows;
        const uint4 *src = reinterpret_cast<const uint4 *>(x + (act[k] ? r[k] : 0) * 128 + v * 16);
        raw[k][0] = act[k] ? src[0] : make_uint4(0u, 0u, 0u, 0u);
        raw[k][1] = act[k] ? src[1] : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int k = 0; k < 2; ++k) {
        float f[16];
        float lo[8], hi[8];
        bf16x8_to_f32(raw[k][0], lo);
        bf16x8_to_f32(raw[k][1], hi);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            f[i] = lo[i];
            f[8 + i] = hi[i];
        }
        fp8_row16(f, v, out + (act[k] ? r[k] : 0) * 128 + v * 16, scale + (act[k] ? r[k] : 0),
                  act[k]);
    }
}

__global__ void cu_pools_kernel(const int32_t *cu_seqlens, int n_docs, int kp, int32_t *cu_pools)
{
    if (blockIdx.x != 0 || threadIdx.x != 0) return;
    int32_t acc = 0;
    cu_pools[0] = 0;
    for (int d = 0; d < n_docs; ++d) {
        acc += (cu_seqlens[d + 1] - cu_seqlens[d]) / kp;
        cu_pools[d + 1] = acc;
    }
}

}  // namespace

cudaError_t launch_cu_pools(const int32_t *cu_seqlens, int n_docs, int kpool, int32_t *cu_pools,
                            cudaStream_t s)
{
    cu_pools_kernel<<<1, 32, 0, s>>>(cu_seqlens, n_docs, kpool, cu_pools);
    return cudaGetLastError();
}

cudaError_t launch_compress(const void *k, const void *gate, const float *ape,
                            const int32_t *cu_seqlens, const int32_t *cu_pools, int n_docs,
                            int64_t T, int D, int kpool, int64_t P_total, void *pk_out,
                            uint8_t *pk_fp8, float *pk_scale, cudaStream_t s)
{
    (void)T;
    if (P_total == 0) return cudaSuccess;
    const int64_t threads = P_total * (D / 8);
    const int64_t blocks = (threads + kThreads - 1) / kThreads;
#define KPOOL_COMPRESS_LAUNCH(KP)                                                              \
    compress_kernel<KP><<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(                     \
        static_cast<const uint16_t *>(k), static_cast<const uint16_t *>(gate), ape, cu_seqlens, \
        cu_pools, n_docs, D, kpool, P_total, static_cast<uint16_t *>(pk_out), pk_fp8, pk_scale)
    switch (kpool) {
    case 1: KPOOL_COMPRESS_LAUNCH(1); break;
    case 2: KPOOL_COMPRESS_LAUNCH(2); break;
    case 4: KPOOL_COMPRESS_LAUNCH(4); break;
    case 8: KPOOL_COMPRESS_LAUNCH(8); break;
    default: KPOOL_COMPRESS_LAUNCH(0); break;
    }
#undef KPOOL_COMPRESS_LAUNCH
    return cudaGetLastError();
}

cudaError_t launch_quantize_fp8(const void *x, int64_t rows, uint8_t *out, float *scale,
                                cudaStream_t s)
{
    if (rows == 0) return cudaSuccess;
    const int64_t warps = (rows + kQuantRowsPerWarp - 1) / kQuantRowsPerWarp;
    const int64_t blocks = (warps * 32 + kThreads - 1) / kThreads;
    quantize_fp8_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        static_cast<const uint16_t *>(x), rows, out, scale);
    return cudaGetLastError();
}

}  // namespace kpool
