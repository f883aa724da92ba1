// Sparse attention over the indexer's selection: the absorbed NoPE MLA
// forward (xtuner PR "GLM-5.3-Flash F5: NoPE DSA + KPool indexer + clamped
// SwiGLU", Summary: a FlashMLA-style SparseMLA forward over the selected token
// indices, with 64 heads in the production config; Megatron-LM PR "GLM5.3
// Flash (KDA + mHC + KPool DSA) support + FP8", Changes section 3, "NoPE": the
// absorbed query has no positional slice, so scores and values both use the
// 512-wide latent rows).  For query row t and head h, over the row's token
// list J(t):
//
//   s_j = scale * q[t, h, :] . c[j, :]
//   o[t, h, :] = sum_j softmax_j(s) c[j, :],   lse[t, h] = ln sum_j exp(s_j)
//
// J(t) is an explicit tok_idx row (-1 = none) or, fused with the expansion,
// the row's selected pools (kpool consecutive tokens each) plus its causal
// tail, computed on the fly so that the token table never reaches memory.
//
// Design (one persistent CTA per SM, 20 warps, rows handed out by an atomic
// counter):
//   warp 0      control: the row's 64 x 512 query block (TMA tiled loads) and,
//               per block of 128 listed tokens, a record (row, block, validity
//               mask) with the block's token ids in shared memory
//   warp 1      TMEM allocation and the tcgen05.mma issuer (one thread)
//   warps 4-11  online softmax and output, two warps per TMEM lane quarter
//               (one TMEM lane per thread: a listed token for the scores, a
//               latent column for the output; each warp of a pair takes half of
//               the heads and half of the output parts)
//   warps 12-19 loaders: the listed tokens' latent rows, gathered with 16-byte
//               cp.async into 128-byte-swizzled tiles (a gather of 128-byte
//               rows moves about 3x more bytes per cycle this way than with
//               one tile::gather4 TMA load per 4 rows)
// Both contractions run transposed, so every MMA has M = 128 and the 64
// heads are its N dimension:
//   S^T [128 tokens x 64 heads]   = C_blk [128 x 512] . Q^T          (A, B K-major)
//   O^T [512 latent x 64 heads]  += C_blk^T [512 x 128] . P          (A, B MN-major)
// A block's latent rows are gathered once into four slots of 128 latent
// columns (slot p always holds columns 128p..128p+127 of the current block);
// the block's output MMAs free the slots in order and the next block's rows
// refill them while the remaining output MMAs run.  (Gathering every row twice,
// into separate score and output rings so that the next block's scores could
// overlap this block's softmax, measured slower: the second gather costs more
// than the overlap gains.)  With one block in flight, a block's scores, softmax
// and output follow one another.  S^T is double-buffered in TMEM (2 x 64 columns)
// and O^T takes 4 x 64.  The online softmax keeps one reference maximum m per
// head and rescales O^T in TMEM only when a block's score exceeds m by more
// than 8 in the base-2 exponent; P = 2^(s*scale*log2(e) - m) <= 256 goes to
// shared memory in BF16, one 128-byte row of 64 heads per listed token.  Each
// softmax thread exponentiates its row against the current maxima before the
// warps agree on whether a rescale is due, so the common block needs one pass.
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>

#include "kpool_internal.h"
#include "kpool_ptx.cuh"

namespace kpool {
namespace {

constexpr int kH = 64;                  // heads = MMA N
constexpr int kDc = 512;                // latent width
constexpr int kBT = 128;                // listed tokens per block = MMA M of S^T
constexpr int kThreads = 640;
constexpr int kSmWarps = 8;             // warps 4..11: two per TMEM lane quarter
constexpr int kSmThreads = 32 * kSmWarps;
constexpr int kHh = 32;                 // heads per softmax thread (half of them)
constexpr int kLoaderWarp0 = 4 + kSmWarps;
constexpr int kLoaders = 256;           // warps 12..19
constexpr int kLoaderWarps = kLoaders / 32;
// register split (setmaxnreg): 640 threads x 96 at launch; the control / MMA
// and loader warpgroups give up part of theirs to the two softmax warpgroups
// (16 loader warps measured no faster than 8: the gather is bound by the
// memory path, not by issue)
constexpr int kRegsSoftmax = 136, kRegsOther = 64;
static_assert(128 * kRegsOther + kSmThreads * kRegsSoftmax + kLoaders * kRegsOther <=
                  (65536 / kThreads) / 8 * 8 * kThreads,
              "register split above the launch's register budget");
constexpr int kChunk = kBT * 128;       // 64 latent columns of a block: 16 KiB
constexpr int kPair = 2 * kChunk;       // 128 latent columns of a block: 32 KiB
constexpr int kCSlots = 4;              // 128-column slots of one block
static_assert(kLoaders == 64 * kCSlots, "two loader warps per slot");
constexpr int kInfoSlots = 4;
constexpr int kOParts = kDc / 128;      // O^T in 128-row (latent) parts of 64 columns
constexpr int kQChunk = kH * 128;       // 64 latent columns of the query block: 8 KiB
constexpr float kRescale = 8.f;         // headroom of the reference maximum (log2)
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kTmemCols = 512;          // S^T: 0..127, O^T: 128..383

// shared memory (from a 1024-byte aligned base)
constexpr int kOffQ = 0;
constexpr int kOffC = kOffQ + 8 * kQChunk;           // 65536
constexpr int kOffP = kOffC + kCSlots * kPair;       // 196608
constexpr int kOffRed = kOffP + 2 * kQChunk;         // 212992: [4][64] floats
constexpr int kOffM = kOffRed + 4 * kH * 4;          // reference maxima [64]
constexpr int kOffL = kOffM + kH * 4;                // per-head scratch [64]
constexpr int kOffFlag = kOffL + kH * 4;             // agreement words [2][kSmWarps]
constexpr int kOffInfo = kOffFlag + 2 * kSmWarps * 4; // BInfo [kInfoSlots]
constexpr int kOffTok = kOffInfo + kInfoSlots * 32;   // token ids [kInfoSlots][128]
constexpr int kOffBar = kOffTok + kInfoSlots * kBT * 4;
enum {
    BQ_FULL = 0, BQ_EMPTY, BC_FULL, BC_EMPTY = BC_FULL + kCSlots, BS_FULL = BC_EMPTY + kCSlots,
    BS_EMPTY = BS_FULL + 2,
    BP_FULL = BS_EMPTY + 2, BO_FULL, BO_EMPTY, BI_FULL,
    BI_EMPTY = BI_FULL + kInfoSlots, BDRAIN = BI_EMPTY + kInfoSlots, NBARS
};
constexpr int kOffMisc = kOffBar + NBARS * 8;        // [0] tmem base, [1] abort flag
constexpr int kSmemUsed = kOffMisc + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;         // alignment slack
static_assert(kSmemBytes <= 232448, "shared memory over the per-block limit");

struct Params {
    const uint16_t *q;          // bf16 [T, 64, 512]
    const uint16_t *kv;         // bf16 [Tk, 512]
    const int32_t *tok;         // [T, W] or NULL (pool mode)
    const int32_t *pool_idx;    // [T, Kp] (pool mode)
    const int32_t *cu_seqlens, *q_pos, *cu_k, *cu_pools;
    int n_docs;
    int T, Tk, W, kp, Kp, tail;
    float c_scale;              // softmax scale * log2(e)
    uint16_t *o;                // bf16 [T, 64, 512]
    float *lse;                 // [T, 64]
    int *ws;                    // [0] row counter, [1] status
    uint64_t wait_limit_ns;
};

// What the loaders need to list the tokens of one row.
struct RowMsg {
    int64_t key0;               // first key token of the row's document
    int t, n_slots, tau, pool_lo, pool_hi, n_sel, n_tail, pad;
};
static_assert(sizeof(RowMsg) <= 48, "RowMsg slot");

// One block of a row, for the MMA issuer and the softmax warps.
struct BInfo {
    int t, b, nb, ksteps;
    uint32_t mask[4];           // bit r of mask[r / 32]: listed token r is valid
};
static_assert(sizeof(BInfo) == 32, "BInfo slot");

struct Sync {
    volatile uint32_t *abort_flag;
    int *status;
    uint64_t limit_ns;
};

// Bounded mbarrier wait (completion, then the CTA abort flag, then a timer
// that raises the flag and KPOOL_STATUS_TIMEOUT).
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Sync &sy)
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

__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Sync &sy)
{
    const bool ok = wait_bar(bar, parity, sy);
    return __all_sync(kFull, ok);
}

// Document of row t (largest d with cu[d] <= t), one warp probing 32 evenly
// spaced offsets per round.  Every lane gets the answer.
__device__ __forceinline__ int doc_of_row(const int32_t *cu, int n_docs, int t, int lane)
{
    int lo = 0, hi = n_docs;
    while (hi - lo > 1) {
        const int step = (hi - lo + 31) / 32;
        const int idx = lo + lane * step;
        const bool le = idx < hi && cu[idx] <= t;
        const unsigned m = __ballot_sync(kFull, le);
        const int nlo = lo + (31 - __clz(m)) * step;
        hi = min(hi, nlo + step);
        lo = nlo;
    }
    return lo;
}

// Key token of slot j of the row (-1: none).  Pool mode lists the selected
// pools' tokens in order, then the tail (the expansion of the selection).
__device__ __forceinline__ int token_of(const Params &p, const RowMsg &m, int j)
{
    if (j >= m.n_slots) return -1;
    if (p.tok != nullptr) {
        const int v = __ldg(p.tok + static_cast<int64_t>(m.t) * p.W + j);
        return (v >= 0 && v < p.Tk) ? v : -1;
    }
    const int npt = m.n_sel * p.kp;
    int64_t v = -1;
    if (j < npt) {
        const int e = j / p.kp;
        const int g = __ldg(p.pool_idx + static_cast<int64_t>(m.t) * p.Kp + e);
        if (g >= m.pool_lo && g < m.pool_hi)
            v = m.key0 + static_cast<int64_t>(g - m.pool_lo) * p.kp + (j - e * p.kp);
    } else {
        v = m.key0 + m.tau - m.n_tail + 1 + (j - npt);
    }
    return (v >= 0 && v < p.Tk) ? static_cast<int>(v) : -1;
}

// Warp 0: the next row's message (t = -1 when there is none or on abort).
__device__ RowMsg next_row(const Params &p, int lane, bool go)
{
    RowMsg m{};
    int t = -1;
    if (lane == 0 && go) t = atomicAdd(p.ws, 1);
    t = __shfl_sync(kFull, t, 0);
    m.t = (t >= 0 && t < p.T) ? t : -1;
    if (m.t < 0) return m;
    if (p.tok != nullptr) {
        // extent of the listed tokens: one past the last valid entry
        int last = -1;
        const int32_t *row = p.tok + static_cast<int64_t>(m.t) * p.W;
        for (int j = lane; j < p.W; j += 32) {
            const int v = __ldg(row + j);
            if (v >= 0 && v < p.Tk) last = j;
        }
        m.n_slots = __reduce_max_sync(kFull, last + 1);
        return m;
    }
    int64_t doc_start = 0;
    m.key0 = 0;
    int pos0 = 0;
    m.pool_lo = 0;
    m.pool_hi = p.Tk / p.kp;
    if (p.cu_seqlens != nullptr) {
        const int d = doc_of_row(p.cu_seqlens, p.n_docs, m.t, lane);
        doc_start = p.cu_seqlens[d];
        m.key0 = p.cu_k != nullptr ? p.cu_k[d] : doc_start;
        pos0 = p.q_pos != nullptr ? p.q_pos[d] : 0;
        m.pool_lo = p.cu_pools[d];
        m.pool_hi = p.cu_pools[d + 1];
    }
    m.tau = pos0 + static_cast<int>(m.t - doc_start);
    const int nc = min((m.tau + 1) / p.kp, m.pool_hi - m.pool_lo);
    m.n_sel = max(0, min(nc, p.Kp));
    m.n_tail = p.tail ? (m.tau + 1) % p.kp : 0;
    m.n_slots = m.n_sel * p.kp + m.n_tail;
    return m;
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ Params p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
    const uint32_t sbase = ptx::smem_u32(smem);
    const uint32_t sQ = sbase + kOffQ, sC = sbase + kOffC, sP = sbase + kOffP;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + kOffBar);
    auto bar = [&](int i) { return ptx::smem_u32(&bars[i]); };
    uint32_t *misc = reinterpret_cast<uint32_t *>(smem + kOffMisc);
    BInfo *info = reinterpret_cast<BInfo *>(smem + kOffInfo);
    int *toks = reinterpret_cast<int *>(smem + kOffTok);
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        ptx::mbar_init(bar(BQ_FULL), 1);
        ptx::mbar_init(bar(BQ_EMPTY), 1);
        for (int i = 0; i < kCSlots; ++i) {
            ptx::mbar_init(bar(BC_FULL + i), 64);   // the slot's two loader warps
            ptx::mbar_init(bar(BC_EMPTY + i), 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(bar(BS_FULL + i), 1);
            ptx::mbar_init(bar(BS_EMPTY + i), kSmWarps);
        }
        for (int i = 0; i < kInfoSlots; ++i) {
            ptx::mbar_init(bar(BI_FULL + i), 1);
            ptx::mbar_init(bar(BI_EMPTY + i), 1 + kSmWarps + kLoaderWarps);
        }
        ptx::mbar_init(bar(BP_FULL), kSmWarps);
        ptx::mbar_init(bar(BO_FULL), 1);
        ptx::mbar_init(bar(BO_EMPTY), kSmWarps);
        ptx::mbar_init(bar(BDRAIN), 1);
        misc[1] = 0u;
        ptx::fence_mbar_init();
    }
    if (warp == 1) {
        ptx::tmem_alloc(ptx::smem_u32(&misc[0]), kTmemCols);
        ptx::tmem_relinquish();
        ptx::tc_fence_before();
    }
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem = misc[0];
    const Sync sy{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.ws + 1, p.wait_limit_ns};

    if (warp < 4) {
    ptx::setmaxnreg_dec<kRegsOther>();
    if (warp == 0) {
        // ---------------- control: rows, records, query blocks ----------------
        if (lane == 0) ptx::tma_prefetch_desc(&tm_q);
        bool ok = true;
        int g = 0;                      // blocks published
        uint32_t q_ph = 0;
        bool q_issued = false;          // a query block was requested (lane 0)
        uint32_t q_par = 0;             // the BQ_FULL phase of the last one
        for (;;) {
            const RowMsg m = next_row(p, lane, ok && !*sy.abort_flag);
            if (m.t < 0) break;
            const int nb = max(1, (m.n_slots + kBT - 1) / kBT);
            // the query block: 8 tiles of 64 heads x 64 latent columns
            ok = ok && wait_bar_warp(bar(BQ_EMPTY), q_ph ^ 1, sy);
            q_ph ^= 1;
            if (ok && lane == 0) {
                ptx::mbar_arrive_expect_tx(bar(BQ_FULL), 8 * kQChunk);
                for (int c = 0; c < 8; ++c)
                    ptx::tma_load_2d(sQ + c * kQChunk, &tm_q, bar(BQ_FULL), 64 * c, m.t * kH);
                q_issued = true;
                q_par = q_ph ^ 1;
            }
            for (int b = 0; b < nb && ok; ++b, ++g) {
                int tk[4];
                uint32_t my4 = 0;
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    tk[k] = token_of(p, m, b * kBT + 4 * lane + k);
                    my4 |= (tk[k] >= 0 ? 1u : 0u) << k;
                }
                // validity word w (tokens 32w..32w+31) from lanes 8w..8w+7
                uint32_t mw = my4 << (4 * (lane & 7));
                mw |= __shfl_xor_sync(kFull, mw, 1);
                mw |= __shfl_xor_sync(kFull, mw, 2);
                mw |= __shfl_xor_sync(kFull, mw, 4);
                const int is = g % kInfoSlots;
                ok = ok && wait_bar_warp(bar(BI_EMPTY + is), ((g / kInfoSlots) & 1) ^ 1, sy);
                if (!ok) break;
                *reinterpret_cast<int4 *>(toks + is * kBT + 4 * lane) = make_int4(tk[0], tk[1], tk[2], tk[3]);
                if ((lane & 7) == 0) info[is].mask[lane >> 3] = mw;
                if (lane == 0) {
                    const int n_in = max(0, min(kBT, m.n_slots - b * kBT));
                    info[is].t = m.t;
                    info[is].b = b;
                    info[is].nb = nb;
                    info[is].ksteps = max(1, (n_in + 15) / 16);
                }
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BI_FULL + is));
            }
        }
        // end of the block stream for every consumer
        const int is = g % kInfoSlots;
        if (ok && wait_bar_warp(bar(BI_EMPTY + is), ((g / kInfoSlots) & 1) ^ 1, sy) && lane == 0) {
            info[is].t = -1;
            ptx::mbar_arrive(bar(BI_FULL + is));
        }
        // no query-block load may still be in flight when the CTA ends (after an
        // expired wait the MMA thread may not have taken the last one): a wait
        // of its own, bounded by the default limit and blind to the abort flag
        if (lane == 0 && q_issued) {
            const uint64_t t0 = ptx::globaltimer();
            while (!ptx::mbar_try_wait(bar(BQ_FULL), q_par))
                if (ptx::globaltimer() - t0 > kTimeoutNs) break;
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            constexpr uint32_t idesc_qk = ptx::make_idesc(1u, kBT, kH);
            constexpr uint32_t idesc_pv = idesc_qk | ptx::kIdescAMajorMN | ptx::kIdescBMajorMN;
            int g = 0;
            uint32_t c_ph = 0, q_ph = 0, p_ph = 0, o_ph = 0;
            bool any = false;
            for (;;) {
                const int is = g % kInfoSlots;
                if (!wait_bar(bar(BI_FULL + is), (g / kInfoSlots) & 1, sy)) break;
                const BInfo in = info[is];
                ptx::mbar_arrive(bar(BI_EMPTY + is));
                if (in.t < 0) break;
                if (in.b == 0) {
                    if (!wait_bar(bar(BQ_FULL), q_ph, sy)) break;
                    q_ph ^= 1;
                }
                const int sb = g & 1;
                if (!wait_bar(bar(BS_EMPTY + sb), ((g >> 1) & 1) ^ 1, sy)) break;
                ptx::tc_fence_after();
                bool ok = true;
                // S^T = C_blk . Q^T over the 512 latent columns
                for (int sl = 0; sl < kCSlots; ++sl) {
                    if (!wait_bar(bar(BC_FULL + sl), c_ph, sy)) {
                        ok = false;
                        break;
                    }
                    ptx::tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint64_t ad = ptx::smem_desc_sw128(sC + sl * kPair + h * kChunk);
                        const uint64_t bd = ptx::smem_desc_sw128(sQ + (2 * sl + h) * kQChunk);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            ptx::mma_bf16(tmem + sb * kH, ad + kk * 2, bd + kk * 2, idesc_qk,
                                          (sl | h | kk) != 0);
                    }
                    any = true;
                }
                if (!ok) break;
                ptx::mma_commit(bar(BS_FULL + sb));
                if (in.b == in.nb - 1) ptx::mma_commit(bar(BQ_EMPTY));
                // O^T += C_blk^T . P^T once P is complete; each slot is freed as
                // soon as its MMAs are done
                if (!wait_bar(bar(BP_FULL), p_ph, sy)) break;
                p_ph ^= 1;
                if (in.b == 0 && !wait_bar(bar(BO_EMPTY), o_ph ^ 1, sy)) break;
                ptx::tc_fence_after();
                for (int sl = 0; sl < kCSlots; ++sl) {
                    const uint32_t a0 = sC + sl * kPair;
                    for (int kk = 0; kk < in.ksteps; ++kk) {
                        const uint64_t ad = ptx::smem_desc_mn_sw128(a0 + kk * 2048, kChunk);
                        const uint64_t bd = ptx::smem_desc_mn_sw128(sP + kk * 2048, 2 * kQChunk);
                        ptx::mma_bf16(tmem + 128 + sl * kH, ad, bd, idesc_pv, (in.b > 0 || kk > 0));
                    }
                    ptx::mma_commit(bar(BC_EMPTY + sl));
                }
                if (in.b == in.nb - 1) {
                    ptx::mma_commit(bar(BO_FULL));
                    o_ph ^= 1;
                }
                c_ph ^= 1;
                ++g;
            }
            if (any) {
                ptx::mma_commit(bar(BDRAIN));
                const uint64_t t0 = ptx::globaltimer();
                while (!ptx::mbar_try_wait(bar(BDRAIN), 0))
                    if (ptx::globaltimer() - t0 > kTimeoutNs) break;
            }
        }
    }
    } else if (warp < kLoaderWarp0) {
        ptx::setmaxnreg_inc<kRegsSoftmax>();
        // ---------------- softmax and output ----------------
        // Two warps per TMEM lane quarter: warp set `hset` takes heads
        // 32*hset..32*hset+31 of the scores and latent parts 2*hset, 2*hset+1 of
        // the output.
        const int sw = warp - 4;                   // 0..7
        const int sub = warp & 3;                  // TMEM lane quarter
        const int hset = sw >> 2;                  // head half
        const int h0 = kHh * hset;
        const int r = 32 * sub + lane;             // listed token / latent column
        const uint32_t lane_base = tmem + (static_cast<uint32_t>(32 * sub) << 16);
        float *m_s = reinterpret_cast<float *>(smem + kOffM);
        float *red = reinterpret_cast<float *>(smem + kOffRed);
        float *hs = reinterpret_cast<float *>(smem + kOffL);
        volatile uint32_t *flags = reinterpret_cast<volatile uint32_t *>(smem + kOffFlag);
        const float c = p.c_scale;
        float l[kHh];                              // this thread's partial sums per head
        int blk = 0, agr = 0;
        uint32_t o_ph = 0;
        // every softmax warp passes each agreement barrier once per round and
        // leaves the loop on the same round; `word` is uniform in a warp.  A
        // barrier reduction first says whether any warp has a nonzero word (the
        // common round ends there); only then are the words exchanged.
        auto agree = [&](uint32_t word) {
            if (!ptx::named_bar_or(4, kSmThreads, word != 0u)) return 0u;
            volatile uint32_t *f = flags + (agr & 1) * kSmWarps;
            if (lane == 0) f[sw] = word;
            ptx::named_bar_sync(3, kSmThreads);
            uint32_t all = 0;
#pragma unroll
            for (int i = 0; i < kSmWarps; ++i) all |= f[i];
            ++agr;
            return all;
        };
        // transpose-reduce of 32 per-head values over the warp: lane ends with
        // head h0 + lane
        auto warp_reduce = [&](float (&v)[kHh], bool is_max) {
#pragma unroll
            for (int w = 16, n = 16; w >= 1; w >>= 1, n >>= 1) {
                const bool up = (lane & w) != 0;
#pragma unroll
                for (int i = 0; i < n; ++i) {
                    const float send = up ? v[i] : v[i + n];
                    const float keep = up ? v[i + n] : v[i];
                    const float got = __shfl_xor_sync(kFull, send, w);
                    v[i] = is_max ? fmaxf(keep, got) : keep + got;
                }
            }
        };
        // v = 2^(v * c - m) in place against the reference maxima (shared, read
        // as broadcasts), 0 for a token that is not listed; true when some
        // exponent exceeds the rescale headroom
        auto exponentiate = [&](float (&v)[kHh], bool valid_row) {
            bool over = false;
            const float4 *m4 = reinterpret_cast<const float4 *>(m_s + h0);
#pragma unroll
            for (int i = 0; i < kHh / 4; ++i) {
                const float4 x = m4[i];
                const float mq[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float a = fmaf(v[4 * i + e], c, -mq[e]);
                    over |= a > kRescale;
                    v[4 * i + e] = valid_row ? ptx::ex2_approx(a) : 0.f;
                }
            }
            return over;
        };
        auto load_s = [&](int bs, float (&v)[kHh]) {
            uint32_t a[32];
            ptx::tmem_ld32(lane_base + bs * kH + h0, a);
            ptx::tmem_ld_wait(a);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(a[i]);
        };
        // this thread's half row of P (32 heads, BF16) in a 128-byte-swizzled tile
        const uint32_t prow = sP + r * 128;
        for (;;) {
            const int bs = blk & 1;
            const uint32_t bph = (blk >> 1) & 1;
            const int is = blk % kInfoSlots;
            bool ok = wait_bar_warp(bar(BI_FULL + is), (blk / kInfoSlots) & 1, sy);
            BInfo in{};
            in.t = -1;
            if (ok) in = info[is];
            __syncwarp();
            if (ok && lane == 0) ptx::mbar_arrive(bar(BI_EMPTY + is));
            const bool end = ok && in.t < 0;
            const bool valid = ok && !end && ((in.mask[sub] >> lane) & 1u);
            bool need = false;
            // the block's probabilities, taken against the current reference
            // maxima before the warps agree (kept unless a rescale is needed);
            // defined on every path, so that none stays live across rounds
            float pv[kHh];
#pragma unroll
            for (int h = 0; h < kHh; ++h) pv[h] = 0.f;
            if (ok && !end) {
                ok = wait_bar_warp(bar(BS_FULL + bs), bph, sy);
                if (ok) {
                    ptx::tc_fence_after();
                    if (in.b == 0) {
                        need = true;   // a new row: the reference maxima start over
#pragma unroll
                        for (int h = 0; h < kHh; ++h) l[h] = 0.f;
                    } else {
                        load_s(bs, pv);
                        need = exponentiate(pv, valid) && valid;
                    }
                }
            }
            const uint32_t all = agree((ok ? 0u : 1u) | (end ? 2u : 0u) |
                                       (__any_sync(kFull, need) ? 4u : 0u));
            if (all & 3u) break;
            if (all & 4u) {
                // exact block maximum per head, new reference maxima, rescale
                load_s(bs, pv);
#pragma unroll
                for (int h = 0; h < kHh; ++h) pv[h] = valid ? pv[h] * c : -INFINITY;
                warp_reduce(pv, true);
                red[sub * kH + h0 + lane] = pv[0];
                ptx::named_bar_sync(3, kSmThreads);
                if (sub == 0) {
                    const int h = h0 + lane;
                    const float bm = fmaxf(fmaxf(red[h], red[kH + h]),
                                           fmaxf(red[2 * kH + h], red[3 * kH + h]));
                    const float mo = in.b == 0 ? -INFINITY : m_s[h];
                    const float mn = fmaxf(mo, bm);
                    hs[h] = (mn == -INFINITY) ? 1.f : ptx::ex2_approx(mo - mn);
                    m_s[h] = mn;
                }
                ptx::named_bar_sync(3, kSmThreads);
                if (in.b > 0) {
                    bool scale_o = false;
#pragma unroll
                    for (int h = 0; h < kHh; ++h) {
                        const float a = hs[h0 + h];
                        l[h] *= a;
                    }
#pragma unroll
                    for (int h = 0; h < kH; ++h) scale_o |= hs[h] != 1.f;
                    if (scale_o) {
                        // the factors are re-read per part rather than held in
                        // registers
                        const volatile float *hsv = hs;
#pragma unroll 1
                        for (int op = 2 * hset; op < 2 * hset + 2; ++op) {
#pragma unroll
                            for (int half = 0; half < 2; ++half) {
                                const uint32_t ta = lane_base + 128 + op * kH + half * 32;
                                uint32_t ov[32];
                                ptx::tmem_ld32(ta, ov);
                                ptx::tmem_ld_wait(ov);
#pragma unroll
                                for (int i = 0; i < 32; ++i)
                                    ov[i] = __float_as_uint(__uint_as_float(ov[i]) * hsv[half * 32 + i]);
                                ptx::tmem_st32(ta, ov);
                            }
                        }
                        ptx::tmem_st_wait();
                    }
                }
                // (unconditional, so that no earlier value of pv stays live
                // across the rescale)
                load_s(bs, pv);
                exponentiate(pv, valid);
            }
            // P[r][h] (BF16, eight heads per 16-byte piece), then the partial sums.
            // This block's scores have landed, so every earlier MMA has completed
            // (a commit's arrival covers all earlier MMAs of the issuing thread):
            // the previous block's output MMAs no longer read P, and O^T above
            // was final when rescaled.
            {
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BS_EMPTY + bs));
#pragma unroll
                for (int j = 0; j < kHh / 8; ++j) {
                    uint32_t w[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const __nv_bfloat162 b2 = __floats2bfloat162_rn(pv[8 * j + 2 * i], pv[8 * j + 2 * i + 1]);
                        w[i] = *reinterpret_cast<const uint32_t *>(&b2);
                    }
                    const int piece = 4 * hset + j;
                    ptx::st_shared_v4(prow + ((piece ^ (r & 7)) << 4), w[0], w[1], w[2], w[3]);
                }
                ptx::fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BP_FULL));
#pragma unroll
                for (int h = 0; h < kHh; ++h) l[h] += pv[h];
            }
            if (in.b == in.nb - 1) {
                // the row's output once its last PV MMAs have landed
                const bool ok2 = wait_bar_warp(bar(BO_FULL), o_ph, sy);
                o_ph ^= 1;
                if (agree(ok2 ? 0u : 1u) & 1u) break;
                ptx::tc_fence_after();
                float v[kHh];
#pragma unroll
                for (int h = 0; h < kHh; ++h) v[h] = l[h];
                warp_reduce(v, false);
                red[sub * kH + h0 + lane] = v[0];
                ptx::named_bar_sync(3, kSmThreads);
                if (sub == 0) {
                    const int h = h0 + lane;
                    const float L = (red[h] + red[kH + h]) + (red[2 * kH + h] + red[3 * kH + h]);
                    hs[h] = L > 0.f ? 1.f / L : 0.f;
                    p.lse[static_cast<int64_t>(in.t) * kH + h] =
                        L > 0.f ? (m_s[h] + log2f(L)) * 0.69314718055994531f : -INFINITY;
                }
                ptx::named_bar_sync(3, kSmThreads);
                uint16_t *orow = p.o + static_cast<int64_t>(in.t) * kH * kDc + r;
#pragma unroll 1
                for (int op = 2 * hset; op < 2 * hset + 2; ++op) {
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        uint32_t ov[32];
                        ptx::tmem_ld32(lane_base + 128 + op * kH + half * 32, ov);
                        ptx::tmem_ld_wait(ov);
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int h = half * 32 + i;
                            const __nv_bfloat16 bv = __float2bfloat16_rn(__uint_as_float(ov[i]) * hs[h]);
                            orow[static_cast<int64_t>(h) * kDc + op * 128] =
                                *reinterpret_cast<const uint16_t *>(&bv);
                        }
                    }
                }
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BO_EMPTY));
            }
            ++blk;
        }
    } else {
        ptx::setmaxnreg_dec<kRegsOther>();
        // ---------------- loaders ----------------
        // Each slot has its own pair of warps, so the four slots of a block
        // refill independently as the output MMAs free them: a pair waits only
        // for its own copies (then a proxy fence and its arrival on the slot).
        const int sl = (warp - kLoaderWarp0) >> 1;                 // the slot of this pair
        const int t64 = ((warp - kLoaderWarp0) & 1) * 32 + lane;   // 0..63 within the pair
        const int k = t64 & 15;                           // 16-byte piece of the slot's 256 bytes
        const char *kvb = reinterpret_cast<const char *>(p.kv) + sl * 256 + k * 16;
        const uint32_t dst_slot = sC + sl * kPair + (k >> 3) * kChunk;
        bool ok = true;
        int g = 0;
        uint32_t c_ph = 0;
        for (;;) {
            const int is = g % kInfoSlots;
            ok = ok && wait_bar_warp(bar(BI_FULL + is), (g / kInfoSlots) & 1, sy);
            if (!ok || info[is].t < 0) break;
            ok = wait_bar_warp(bar(BC_EMPTY + sl), c_ph ^ 1, sy);
            if (!ok) break;
            const int *tk = toks + is * kBT;
#pragma unroll 8
            for (int i = 0; i < kBT / 4; ++i) {           // rows t64 / 16 + 4 i
                const int r = (t64 >> 4) + 4 * i;
                const int tok = tk[r];
                ptx::cp_async16(dst_slot + r * 128 + (((k & 7) ^ (r & 7)) << 4),
                                kvb + (tok >= 0 ? static_cast<int64_t>(tok) * (kDc * 2) : 0),
                                tok >= 0 ? 16u : 0u);
            }
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(bar(BI_EMPTY + is));   // token ids read
            ptx::cp_async_commit();
            ptx::cp_async_wait_all();
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(bar(BC_FULL + sl));
            c_ph ^= 1;
            ++g;
        }
        ptx::cp_async_wait_all();
    }

    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

size_t sparse_mla_workspace_bytes() { return 256; }

namespace {
// No key at all: every row gets o = 0 and lse = -inf.
__global__ void no_keys_kernel(float *lse, int64_t n)
{
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < n;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x)
        lse[i] = -INFINITY;
}
}  // namespace

int run_sparse_mla(const SparseMlaArgs &a, cudaStream_t s)
{
    KPOOL_CUDA_CHECK(cudaMemsetAsync(a.workspace, 0, 8, s));
    if (a.T == 0) return KPOOL_OK;
    if (a.Tk == 0) {
        KPOOL_CUDA_CHECK(cudaMemsetAsync(a.o, 0, static_cast<size_t>(a.T) * kH * kDc * 2, s));
        no_keys_kernel<<<256, 256, 0, s>>>(a.lse, a.T * kH);
        KPOOL_CUDA_CHECK(cudaGetLastError());
        return KPOOL_OK;
    }
    CUtensorMap mq;
    const int rc = encode_bf16_tmap(&mq, a.q, kDc, static_cast<uint64_t>(a.T) * kH, kH);
    if (rc) return rc;
    Params p{};
    p.q = static_cast<const uint16_t *>(a.q);
    p.kv = static_cast<const uint16_t *>(a.kv);
    p.tok = a.tok_idx;
    p.pool_idx = a.pool_idx;
    p.cu_seqlens = a.cu_seqlens;
    p.q_pos = a.q_pos;
    p.cu_k = a.cu_k;
    p.cu_pools = a.cu_pools;
    p.n_docs = a.n_docs;
    p.T = static_cast<int>(a.T);
    p.Tk = static_cast<int>(a.Tk);
    p.W = a.W;
    p.kp = a.kpool;
    p.Kp = a.Kp;
    p.tail = a.tail;
    p.c_scale = static_cast<float>(static_cast<double>(a.scale) * 1.4426950408889634);
    p.o = static_cast<uint16_t *>(a.o);
    p.lse = a.lse;
    p.ws = static_cast<int *>(a.workspace);
    p.wait_limit_ns = get_wait_limit_ns();
    KPOOL_CUDA_CHECK(cudaFuncSetAttribute(sparse_mla_kernel,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes));
    const int grid = static_cast<int>(std::min<int64_t>(num_sms(), a.T));
    sparse_mla_kernel<<<grid, kThreads, kSmemBytes, s>>>(mq, p);
    KPOOL_CUDA_CHECK(cudaGetLastError());
    return KPOOL_OK;
}

}  // namespace kpool
