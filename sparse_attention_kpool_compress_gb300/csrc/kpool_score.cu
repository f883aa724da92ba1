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
// Design (one persistent CTA per SM, 20 warps):
//   warp 0      TMA producer + tile scheduler (atomic counter over a
//               longest-first unit table built by schedule_kernel, or by
//               split_schedule_kernel for calls with few query tiles)
//   warp 1      tcgen05.mma issuer (one thread)
//   warp 2      TMEM allocator
//   warps 4-19  epilogue: tcgen05.ld of the accumulator, relu * w head
//               reduction, threshold filter, unordered appends into per-query
//               candidate areas in shared memory, radix-select compaction,
//               final selection ranked into ascending pool order.
// MMA tile: M = 128 pools (TMEM lanes, one epilogue thread per pool and
// 64-column slice), N = 256 (query, head) columns = 256 / H queries, K = D
// (bf16: 16 per instruction, E4M3: 32).  q of the query tile stays resident in
// shared memory; pooled-key tiles stream through a ring of `stages` buffers;
// two 256-column TMEM accumulators let the epilogue of tile i overlap the MMAs
// of tile i+1.  Ties resolve to the lower pool index inside the selection.
#include <cuda.h>

#include <algorithm>
#include <atomic>
#include <type_traits>
#include <cstring>
#include <mutex>
#include <vector>

#include "kpool_internal.h"
#include "kpool_ptx.cuh"

namespace kpool {
namespace {

constexpr int kEpiWarps = 16;                         // 4 per SM sub-partition
constexpr int kEpiThreads = 32 * kEpiWarps;           // 512
constexpr int kThreads = 128 + kEpiThreads;           // 640
constexpr int kBM = 128;                              // pools per tile
constexpr int kBN = 256;                              // (query, head) columns per tile
constexpr int kAccCols = 256;
constexpr int kTmemCols = 512;
constexpr int kSmemLimit = 232448;                    // 227 KiB per block (opt-in max)
constexpr int kMaxC = 4096;
constexpr uint64_t kTimeoutNs = 2000000000ull;        // 2 s: default wait limit, drain bound
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kGroups = 4;                            // selection groups of the epilogue
constexpr int kGroupWarps = kEpiWarps / kGroups;      // 4 warps per group
constexpr int kGroupThreads = 32 * kGroupWarps;       // 128
constexpr int kSlack = 64;                            // extra entries a mid-stream prune may keep
// register split (setmaxnreg): 128 threads x 32 + 512 x 112 = 640 x 96 (launch budget)
constexpr int kRegsOther = 32, kRegsEpi = 112;
// split-pool schedule (few query tiles with long pool lists: decode, short
// chunks): a query tile's pool tiles are cut into units scored by different
// CTAs, whose best-Kp lists the last unit to finish merges
constexpr int kSplitMaxQT = 1024;                     // query tiles it schedules, at most
constexpr int64_t kSplitEntries = int64_t(1) << 21;   // (index, score) entries of partial lists
constexpr int kSplitMaxSplits = 16;                   // units per query tile, at most
constexpr int kSplitMinTiles = 32;                    // pool tiles per unit, at least

// Optional phase timers (build with -DKPOOL_PHASE_TIMERS): per-role cycle
// counts of waits and work, summed over all CTAs into g_phase_timers and read
// back with kpool_debug_phase_timers.  Compiled out by default.
#ifdef KPOOL_PHASE_TIMERS
__device__ unsigned long long g_phase_timers[32];
#define PT_DECL                                \
    unsigned long long pt_[8] = {};            \
    unsigned long long pt_t = clock64();
#define PT_MARK(i)                             \
    do {                                       \
        const unsigned long long n_ = clock64(); \
        pt_[i] += n_ - pt_t;                   \
        pt_t = n_;                             \
    } while (0)
#define PT_FLUSH(base)                                                       \
    do {                                                                     \
        for (int i_ = 0; i_ < 8; ++i_) atomicAdd(&g_phase_timers[(base) + i_], pt_[i_]); \
    } while (0)
#else
#define PT_DECL
#define PT_MARK(i) do {} while (0)
#define PT_FLUSH(base) do {} while (0)
#endif

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

Layout make_layout(int H, int D, int fp8, int stages = 0)
{
    Layout L{};
    const int esize = fp8 ? 1 : 2;
    L.n_kchunks = (D * esize + 127) / 128;
    L.stages = fp8 ? 4 : 2;   // bf16: two stages leave room for ~1000 more candidates per query
    if (stages > 0) L.stages = stages;
    const int QT = qt_of(H);
    L.q_chunk = kBN * 128;
    L.pk_chunk = kBM * 128;
    L.q_off = 0;
    L.pk_off = L.q_off + L.n_kchunks * L.q_chunk;
    L.pk_stage = L.n_kchunks * L.pk_chunk;
    uint32_t off = L.pk_off + L.stages * L.pk_stage;
    L.ws_off = off;   off += (kBN + 2 * 4 * kBM) * 4;   // head weights + half-query partials
    L.hist_off = off; off += kGroups * 256 * 4;
    L.cnt_off = off;  off += 2 * QT * 4 * 4;
    L.scr_off = off;  off += kGroups * 32 * 4 + ((QT * 4 + 15) / 16) * 16;
    L.thr_off = off;  off += ((QT * 4 + 15) / 16) * 16;
    L.bar_off = off;  off += 256;
    L.ti_off = off;   off += 3 * 64;   // two producer slots + the epilogue's current unit
    L.misc_off = off; off += 32;   // tmem, abort, split flag, -, epilogue agreement [4]
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
    const int32_t *q_pos;     // per-document position of the first query row, or NULL
    int n_docs, T, P_total, kp, Kp, fp8, mode;
    int32_t *pool_idx;
    float *pool_score;
    float *scores;
    int *ws;
    // split-pool schedule (units == NULL: one unit per query tile)
    int *units;          // [n_units][8]: t0, doc, i0, i1, slot_base, splits, tile, k
    int *tile_ctr;       // per query tile: units finished
    int *part_cnt;       // [slot][QT] entries in each partial list
    int32_t *part_idx;   // [slot][QT][Kp]
    float *part_score;   // [slot][QT][Kp]
    uint32_t q_tx, pk_tx, idesc;
    uint64_t wait_limit_ns;   // limit of one pipeline wait (kTimeoutNs unless a test lowers it)
    Layout L;
};

// 2 relu(x), exactly (x + |x| is 2x or +0), as one add with an absolute-value
// operand on the FMA pipe rather than a max on the ALU pipe; the head weights are
// staged halved to match.  (Only an accumulator of -inf, which needs inputs whose
// products overflow FP32, would differ: NaN here, 0 from a max.)
__device__ __forceinline__ float twice_relu(float x) { return __fadd_rn(x, fabsf(x)); }

// Orderable key of a score: larger float -> larger key; -0 folded into +0.
__device__ __forceinline__ uint32_t fkey(float f)
{
    uint32_t u = __float_as_uint(f);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The score of an orderable key (fkey's inverse; -0 comes back as +0).
__device__ __forceinline__ float unkey(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// The smallest score whose key exceeds k, so that fkey(s) > k exactly when
// s >= pass_floor(k) for every score s (never NaN; -0 folded into +0): -inf
// when every score passes, NaN when none does.  One float compare per pool
// then replaces the key computation.
__device__ __forceinline__ float pass_floor(uint32_t k)
{
    if (k < 0x007FFFFFu) return -INFINITY;                    // below the key of -inf
    if (k >= 0xFF800000u) return __uint_as_float(0x7FC00000u);  // at or above +inf's key
    const uint32_t e = k + 1u;
    return __uint_as_float((e & 0x80000000u) ? (e & 0x7FFFFFFFu) : ~e);
}

struct Sync {
    volatile uint32_t *abort_flag;
    int *status;
    uint64_t limit_ns;
};

// Bounded mbarrier wait: completion first, then the CTA abort flag, then a
// timer of limit_ns (sets KPOOL_STATUS_TIMEOUT and the abort flag).  Once the
// abort flag is up every later wait returns after one probe.
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

// Warp-uniform version for the epilogue warps.
__device__ __forceinline__ bool wait_bar_warp(uint32_t bar, uint32_t parity, const Sync &sy)
{
    bool ok = wait_bar(bar, parity, sy);
    return __all_sync(kFull, ok);
}

// A unit of work: pool tiles [i0, i1) of the query tile of rows
// [t0, min(t0 + QT, doc_end)) of the document starting at query row
// doc_start; row t sits at document-local position pos_base + (t - doc_start)
// and may see the document's complete pools
// j < min(floor((pos + 1) / kpool), pool_count), global index pool_base + j.
// A query tile split into `splits` > 1 units has them at table positions
// slot_base .. slot_base + splits - 1 (also their partial-list slots); this
// is unit k; `tile` indexes its arrival counter.
struct TileInfo {
    int t0, doc_start, doc_end, pool_base, pos_base, pool_count;
    int i0, i1, slot_base, splits, tile, k;
    int pad[4];
};

__device__ __forceinline__ int pool_tiles_of(const TileInfo &ti, int QT, int kp)
{
    const int tau0 = ti.pos_base + (ti.t0 - ti.doc_start);
    const int nq = min(QT, ti.doc_end - ti.t0);
    const int nc_last = min((tau0 + nq) / kp, ti.pool_count);   // (tau_last + 1) / kp
    return (nc_last + kBM - 1) / kBM;
}

__device__ __forceinline__ void group_bar(int g) { ptx::named_bar_sync(2 + g, kGroupThreads); }

// A selection group of NW warps: one of the four groups of four warps, or all
// sixteen epilogue warps at once (a lone query).  Its barrier and the slots of
// its scratch words gs (per-warp arrays and scalars; with NW = 16 the scratch
// spans all four groups' areas).
template <int NW>
__device__ __forceinline__ void sel_bar(int g)
{
    if constexpr (NW == kGroupWarps) group_bar(g);
    else ptx::named_bar_sync(1, kEpiThreads);
}
template <int NW>
struct Gs {
    static constexpr int kMin = 0, kMax = NW, kCnt = 2 * NW, kScal = 3 * NW;
    static constexpr int kA = 3 * NW + 4, kB = 4 * NW + 4, kCtr = 5 * NW + 4;
};
static_assert(Gs<kEpiWarps>::kCtr < kGroups * 32, "wide selection scratch");

// Radix search (DeepSelect-style, 8-bit digits) for the k-th largest of
// keyf(e) over the entries e < n with partf(e), by one selection group
// (32 NW threads).
// Digits start at the highest bit where the smallest and largest
// participating key differ, so the first histogram is spread.  Results:
//   kth    the k-th largest key, or (edge) the lower edge of the digit bin
//          holding it when that bin is needed whole or, with allow_edge, when
//          keeping everything at or above the edge keeps <= k + slack entries;
//   above  participants with key above the bin / above kth;
//   inbin  participants in that bin / equal to kth.
template <int NW, class KeyFn, class PartFn>
__device__ void radix_kth(int n, int k, const KeyFn &keyf, const PartFn &partf, bool allow_edge,
                          int slack, int g, int gtid, int *hist, int *gs, uint32_t &kth,
                          int &above, int &inbin, bool &edge)
{
    const int lane = gtid & 31, gw = gtid >> 5;
    uint32_t kmin = 0xFFFFFFFFu, kmax = 0u;
    int cnt = 0;
    for (int e = gtid; e < n; e += (32 * NW)) {
        if (partf(e)) {
            const uint32_t key = keyf(e);
            kmin = min(kmin, key);
            kmax = max(kmax, key);
            ++cnt;
        }
    }
    kmin = __reduce_min_sync(kFull, kmin);
    kmax = __reduce_max_sync(kFull, kmax);
    cnt = __reduce_add_sync(kFull, cnt);
    if (lane == 0) {
        gs[Gs<NW>::kMin + gw] = static_cast<int>(kmin);
        gs[Gs<NW>::kMax + gw] = static_cast<int>(kmax);
        gs[Gs<NW>::kCnt + gw] = cnt;
    }
    sel_bar<NW>(g);
    kmin = 0xFFFFFFFFu;
    kmax = 0u;
    cnt = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        kmin = min(kmin, static_cast<uint32_t>(gs[Gs<NW>::kMin + w]));
        kmax = max(kmax, static_cast<uint32_t>(gs[Gs<NW>::kMax + w]));
        cnt += gs[Gs<NW>::kCnt + w];
    }
    above = 0;
    if (kmin == kmax) {
        kth = kmax;
        inbin = cnt;
        edge = false;
        return;
    }
    int hi = 31 - __clz(kmin ^ kmax);
    uint32_t prefix = hi == 31 ? 0u : (kmax & ~((2u << hi) - 1u));
    int kr = k;
    while (true) {
        const int lo = max(hi - 7, 0);
        const uint32_t dmask = (2u << (hi - lo)) - 1u;
        for (int i = gtid; i < 256; i += (32 * NW)) hist[i] = 0;
        sel_bar<NW>(g);
        for (int e = gtid; e < n; e += (32 * NW)) {
            if (!partf(e)) continue;
            const uint32_t key = keyf(e);
            if (hi == 31 || (key >> (hi + 1)) == (prefix >> (hi + 1)))
                atomicAdd(&hist[(key >> lo) & dmask], 1);
        }
        sel_bar<NW>(g);
        if (gw == 0) {
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
            int cum = suf - local;
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                if (cum < kr && cum + b[i] >= kr) {
                    gs[Gs<NW>::kScal] = lane * 8 + i;
                    gs[Gs<NW>::kScal + 1] = cum;
                    gs[Gs<NW>::kScal + 2] = b[i];
                }
                cum += b[i];
            }
        }
        sel_bar<NW>(g);
        const int d = gs[Gs<NW>::kScal], cum = gs[Gs<NW>::kScal + 1], hb = gs[Gs<NW>::kScal + 2];
        prefix |= static_cast<uint32_t>(d) << lo;
        kr -= cum;
        above += cum;
        if (hb == kr || (allow_edge && above + hb <= k + slack)) {
            kth = prefix;
            inbin = hb;
            edge = true;
            return;
        }
        if (lo == 0) {
            kth = prefix;
            inbin = hb;
            edge = false;
            return;
        }
        hi = lo - 1;
    }
}

// Keep the k best of cs/ci[0..n), n > k (score descending, equal scores by
// lower pool index), in place, by one selection group.  In prune
// mode (exact = false) it may keep up to k + slack entries: all those at or
// above a digit-bin edge.  Returns the number kept and writes to *thr_out the
// key a later candidate (higher pool index) must exceed to possibly enter.
template <int NW = kGroupWarps>
__device__ int group_select(float *cs, int *ci, int n, int k, bool exact, int slack, int g,
                            int gtid, int *hist, int *gs, uint32_t *thr_out)
{
    const int lane = gtid & 31, gw = gtid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    // the scores become their orderable keys in place for the passes below, and
    // the kept ones scores again at the end
    uint32_t *ck = reinterpret_cast<uint32_t *>(cs);
    for (int e = gtid; e < n; e += (32 * NW)) ck[e] = fkey(cs[e]);
    sel_bar<NW>(g);
    uint32_t kth;
    int above, inbin;
    bool edge;
    radix_kth<NW>(n, k, [&](int e) { return ck[e]; }, [](int) { return true; }, !exact, slack, g,
              gtid, hist, gs, kth, above, inbin, edge);
    // ties at the k-th score: keep the lowest pool indices among them
    uint32_t ithr = 0xFFFFFFFFu;   // keep tied entries with ci <= ithr
    const bool ties = !edge && above + inbin > k;
    if (ties) {
        const int need = k - above;
        uint32_t ik;
        int iab, iin;
        bool ied;
        sel_bar<NW>(g);   // gs reuse
        radix_kth<NW>(n, need, [&](int e) { return ~static_cast<uint32_t>(ci[e]); },
                  [&](int e) { return ck[e] == kth; }, false, 0, g, gtid, hist, gs, ik, iab,
                  iin, ied);
        ithr = ~ik;
    }
    sel_bar<NW>(g);   // gs reused below
    const int chunks = (n + 31) / 32;
    const int per = ((chunks + NW - 1) / NW) * 32;
    const int r0 = gw * per, r1 = min(n, r0 + per);
    int cnt = 0;
    for (int c = r0; c < r1; c += 32) {
        const int e = c + lane;
        uint32_t key = 0u;
        int iv = 0;
        bool keep = false;
        if (e < r1) {
            key = ck[e];
            iv = ci[e];
            keep = edge ? key >= kth
                        : (key > kth || (key == kth && static_cast<uint32_t>(iv) <= ithr));
        }
        const unsigned kb = __ballot_sync(kFull, keep);
        if (keep) {
            const int dst = r0 + cnt + __popc(kb & lt);
            ck[dst] = key;
            ci[dst] = iv;
        }
        cnt += __popc(kb);
    }
    if (lane == 0) gs[Gs<NW>::kA + gw] = cnt;
    sel_bar<NW>(g);
    int total = 0, mybase = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        if (w == gw) mybase = total;
        total += gs[Gs<NW>::kA + w];
    }
    // move each later warp's kept block down behind the earlier ones, in order
    for (int w = 1; w < NW; ++w) {
        if (gw == w) {
            for (int c = 0; c < cnt; c += 32) {
                const int i = c + lane;
                uint32_t kv = 0u;
                int iv = 0;
                if (i < cnt) {
                    kv = ck[r0 + i];
                    iv = ci[r0 + i];
                }
                __syncwarp();
                if (i < cnt) {
                    ck[mybase + i] = kv;
                    ci[mybase + i] = iv;
                }
            }
        }
        sel_bar<NW>(g);
    }
    for (int e = gtid; e < total; e += (32 * NW)) cs[e] = unkey(ck[e]);
    if (gtid == 0) *thr_out = edge ? (kth > 0 ? kth - 1u : 0u) : kth;
    sel_bar<NW>(g);
    return total;
}

// Write the n kept entries of cs/ci to out_idx/out_score in ascending pool
// order by ranking them through a bitmap of the query's visible pools (local
// index ci - pool_base < 32 * words).  The bitmap lives in ci[n .. n+words)
// and the per-word prefix counts in cs[n .. n+words) (the free tail of the
// query's candidate area; words <= capacity - n).  One group.
template <int NW = kGroupWarps>
__device__ void group_rank_store(float *cs, int *ci, int n, int pool_base, int words, int g,
                                 int gtid, int *gs, int32_t *out_idx, float *out_score)
{
    const int lane = gtid & 31, gw = gtid >> 5;
    uint32_t *bm = reinterpret_cast<uint32_t *>(ci + n);
    int *pf = reinterpret_cast<int *>(cs + n);
    for (int w = gtid; w < words; w += (32 * NW)) bm[w] = 0u;
    sel_bar<NW>(g);
    for (int e = gtid; e < n; e += (32 * NW)) {
        const int j = ci[e] - pool_base;
        atomicOr(&bm[j >> 5], 1u << (j & 31));
    }
    sel_bar<NW>(g);
    // exclusive prefix of popcounts over words: each thread a contiguous run
    const int per = (words + (32 * NW) - 1) / (32 * NW);
    const int w0 = gtid * per, w1 = min(words, w0 + per);
    int local = 0;
    for (int w = w0; w < w1; ++w) local += __popc(bm[w]);
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) gs[Gs<NW>::kB + gw] = incl;
    sel_bar<NW>(g);
    int run = incl - local;
    for (int w = 0; w < gw; ++w) run += gs[Gs<NW>::kB + w];
    for (int w = w0; w < w1; ++w) {
        pf[w] = run;
        run += __popc(bm[w]);
    }
    sel_bar<NW>(g);
    for (int e = gtid; e < n; e += (32 * NW)) {
        const int j = ci[e] - pool_base;
        const int r = pf[j >> 5] + __popc(bm[j >> 5] & ((1u << (j & 31)) - 1u));
        out_idx[r] = ci[e];
        out_score[r] = cs[e];
    }
}

// Direct mode: the n scores of one query at their local pool positions
// dq[0..n).  Writes the best k (ties to the lower pool index), or all n when
// n <= k, to out_idx/out_score in ascending pool order and returns how many
// it wrote.  One selection group: the scores are turned into their orderable
// keys in place once (dq is scratch afterwards), then a radix search for the
// k-th key and two ordered passes (counts per warp, then ballot-ranked writes)
// read the keys.
template <int NW = kGroupWarps>
__device__ int group_select_direct(float *dq, int n, int k, int pool_base, int g, int gtid,
                                   int *hist, int *gs, int32_t *out_idx, float *out_score)
{
    const int lane = gtid & 31, gw = gtid >> 5;
    const unsigned lt = (1u << lane) - 1u;
    if (n <= k) {
        for (int e = gtid; e < n; e += (32 * NW)) {
            out_idx[e] = pool_base + e;
            out_score[e] = dq[e];
        }
        return n;
    }
    uint32_t *dk = reinterpret_cast<uint32_t *>(dq);
    for (int e = gtid; e < n; e += (32 * NW)) dk[e] = fkey(dq[e]);
    sel_bar<NW>(g);
    uint32_t kth;
    int above, inbin;
    bool edge;
    radix_kth<NW>(n, k, [&](int e) { return dk[e]; }, [](int) { return true; }, false, 0, g,
              gtid, hist, gs, kth, above, inbin, edge);
    // edge: the bin holds exactly the entries still needed -> keep key >= kth;
    // otherwise keep key > kth and the first `need` entries equal to it
    const int need = edge ? 0 : k - above;
    sel_bar<NW>(g);   // gs reuse
    const int per_w = ((n + (32 * NW) - 1) / (32 * NW)) * 32;
    const int r0 = gw * per_w, r1 = min(n, r0 + per_w);
    int cgt = 0, ceq = 0;
    for (int c = r0; c < r1; c += 32) {
        const int e = c + lane;
        const uint32_t key = e < r1 ? dk[e] : 0u;
        cgt += __popc(__ballot_sync(kFull, e < r1 && (edge ? key >= kth : key > kth)));
        ceq += __popc(__ballot_sync(kFull, e < r1 && !edge && key == kth));
    }
    if (lane == 0) {
        gs[Gs<NW>::kA + gw] = cgt;
        gs[Gs<NW>::kB + gw] = ceq;
    }
    sel_bar<NW>(g);
    int base_gt = 0, base_eq = 0;
    for (int w = 0; w < gw; ++w) {
        base_gt += gs[Gs<NW>::kA + w];
        base_eq += gs[Gs<NW>::kB + w];
    }
    int pos = base_gt + min(base_eq, need);
    int eq_seen = base_eq;
    for (int c = r0; c < r1; c += 32) {
        const int e = c + lane;
        const uint32_t key = e < r1 ? dk[e] : 0u;
        const bool gt = e < r1 && (edge ? key >= kth : key > kth);
        const bool eq = e < r1 && !edge && key == kth;
        const unsigned beq = __ballot_sync(kFull, eq);
        const bool keep = gt || (eq && eq_seen + __popc(beq & lt) < need);
        const unsigned bk = __ballot_sync(kFull, keep);
        if (keep) {
            const int d = pos + __popc(bk & lt);
            out_idx[d] = pool_base + e;
            out_score[d] = unkey(key);
        }
        pos += __popc(bk);
        eq_seen += __popc(beq);
    }
    sel_bar<NW>(g);   // gs reuse by the caller
    return k;
}

// Ascending sort of cs/ci[0..n) by pool index (ci), bitonic over the next
// power of two (pad entries carry INT_MAX), by one group.  n2 <= capacity.
template <int NW = kGroupWarps>
__device__ void group_sort_by_pool(float *cs, int *ci, int n, int g, int gtid)
{
    int n2 = 1;
    while (n2 < n) n2 <<= 1;
    for (int i = n + gtid; i < n2; i += (32 * NW)) {
        ci[i] = 0x7FFFFFFF;
        cs[i] = -INFINITY;
    }
    sel_bar<NW>(g);
    for (int kk = 2; kk <= n2; kk <<= 1) {
        for (int j = kk >> 1; j > 0; j >>= 1) {
            for (int i = gtid; i < n2; i += (32 * NW)) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const int a = ci[i], b = ci[ixj];
                    const bool up = (i & kk) == 0;
                    if ((a > b) == up) {
                        ci[i] = b;
                        ci[ixj] = a;
                        const float t = cs[i];
                        cs[i] = cs[ixj];
                        cs[ixj] = t;
                    }
                }
            }
            sel_bar<NW>(g);
        }
    }
}

// Best k (score descending, ties to the lower pool index) of the n entries
// of sc/ix in global memory (read through L2; padding entries carry index
// INT_MAX and score -inf), written to cs/ci[0..) in any order; all real
// entries when at most k of the n_real are real.  One group.  Returns the
// number written (min(k, n_real)).
template <int NW = kGroupWarps>
__device__ int group_select_into(const float *sc, const int32_t *ix, int n, int k, int n_real,
                                 float *cs, int *ci, int g, int gtid, int *hist, int *gs)
{
    const int lane = gtid & 31;
    const bool all = n_real <= k;
    uint32_t kth = 0u, ithr = 0xFFFFFFFFu;
    bool edge = false;
    if (!all) {
        int above, inbin;
        radix_kth<NW>(n, k, [&](int e) { return fkey(__ldcg(sc + e)); }, [](int) { return true; },
                  false, 0, g, gtid, hist, gs, kth, above, inbin, edge);
        if (!edge && above + inbin > k) {
            uint32_t ik;
            int iab, iin;
            bool ied;
            sel_bar<NW>(g);   // gs reuse
            radix_kth<NW>(n, k - above, [&](int e) { return ~static_cast<uint32_t>(__ldcg(ix + e)); },
                      [&](int e) { return fkey(__ldcg(sc + e)) == kth; }, false, 0, g, gtid, hist,
                      gs, ik, iab, iin, ied);
            ithr = ~ik;
        }
    }
    sel_bar<NW>(g);
    if (gtid == 0) gs[Gs<NW>::kCtr] = 0;
    sel_bar<NW>(g);
    for (int c = 0; c < n; c += (32 * NW)) {
        const int e = c + gtid;
        bool keep = false;
        float sv = 0.f;
        int iv = 0;
        if (e < n) {
            sv = __ldcg(sc + e);
            iv = __ldcg(ix + e);
            const uint32_t key = fkey(sv);
            keep = all ? iv != 0x7FFFFFFF
                       : (edge ? key >= kth
                               : (key > kth || (key == kth && static_cast<uint32_t>(iv) <= ithr)));
        }
        const unsigned kb = __ballot_sync(kFull, keep);
        int base = 0;
        if (lane == 0 && kb != 0u) base = atomicAdd(&gs[Gs<NW>::kCtr], __popc(kb));
        base = __shfl_sync(kFull, base, 0);
        if (keep) {
            const int d = base + __popc(kb & ((1u << lane) - 1u));
            cs[d] = sv;
            ci[d] = iv;
        }
    }
    sel_bar<NW>(g);
    const int total = gs[Gs<NW>::kCtr];
    sel_bar<NW>(g);   // gs reuse
    return total;
}

// End of one unit of a split query tile (epilogue threads): its best Kp per
// query (padded to Kp) go to the tile's partial lists, [query][unit][Kp]; the
// unit that finishes the tile last selects the best Kp of their union (each
// of the tile's best Kp lies among the best Kp of its own unit) into its
// candidate areas and returns true.  Kept out of line: the main loop's code
// is faster without it.
__device__ __noinline__ bool split_unit_end(const TileInfo *tu, int nq, int QT, int Kp, int C,
                                            float *cs, int *ci, int *qcnt, uint32_t *thr_s,
                                            int *hist, int *gs, int g, int gtid, int etid,
                                            uint32_t *flag, int32_t *part_idx, float *part_score,
                                            int *part_cnt, int *tile_ctr)
{
    const int splits = tu->splits;
    const int uk = tu->k;
    const int64_t tbase = static_cast<int64_t>(tu->slot_base) * QT;
    // a lone query takes all sixteen warps (one wide group), else each group
    // takes its own queries
    const bool wide = nq == 1;
    int *hist0 = hist - g * 256, *gs0 = gs - g * 32;
    auto unit_out = [&](auto nw, int q, int gg, int tid, int *hh, int *gss) {
        constexpr int NW = decltype(nw)::value;
        int n = qcnt[q];
        float *csq = cs + q * C;
        int *ciq = ci + q * C;
        if (n > Kp) {
            group_select<NW>(csq, ciq, n, Kp, true, 0, gg, tid, hh, gss, &thr_s[q]);
            n = Kp;
        }
        const int64_t li = tbase + q * splits + uk;
        for (int e = tid; e < Kp; e += 32 * NW) {
            const bool real = e < n;
            part_idx[li * Kp + e] = real ? ciq[e] : 0x7FFFFFFF;
            part_score[li * Kp + e] = real ? csq[e] : -INFINITY;
        }
        if (tid == 0) part_cnt[li] = n;
    };
    if (wide) unit_out(std::integral_constant<int, kEpiWarps>{}, 0, 0, etid, hist0, gs0);
    else
        for (int q = g; q < nq; q += kGroups)
            unit_out(std::integral_constant<int, kGroupWarps>{}, q, g, gtid, hist, gs);
    __threadfence();
    ptx::named_bar_sync(1, kEpiThreads);
    if (etid == 0) *flag = atomicAdd(tile_ctr + tu->tile, 1) == splits - 1 ? 1u : 0u;
    ptx::named_bar_sync(1, kEpiThreads);
    const bool last = *flag != 0u;
    if (last) {
        __threadfence();
        auto merge = [&](auto nw, int q, int gg, int tid, int *hh, int *gss) {
            constexpr int NW = decltype(nw)::value;
            const int64_t l0 = tbase + q * splits;
            int n_real = 0;
            for (int u = 0; u < splits; ++u) n_real += __ldcg(part_cnt + l0 + u);
            const int n = group_select_into<NW>(part_score + l0 * Kp, part_idx + l0 * Kp,
                                                splits * Kp, Kp, n_real, cs + q * C, ci + q * C,
                                                gg, tid, hh, gss);
            if (tid == 0) qcnt[q] = n;
            sel_bar<NW>(gg);
        };
        if (wide) merge(std::integral_constant<int, kEpiWarps>{}, 0, 0, etid, hist0, gs0);
        else
            for (int q = g; q < nq; q += kGroups)
                merge(std::integral_constant<int, kGroupWarps>{}, q, g, gtid, hist, gs);
    }
    return last;
}

// kFew: the instantiation for calls with few query tiles (split-pool schedule,
// lone-query tiles); the other one carries none of that code, which keeps the
// main loop of long prefills as fast as it can be compiled.
template <int H, bool kFew, bool kDirect>
__global__ void __launch_bounds__(kThreads, 1)
    score_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_pk,
                 const __grid_constant__ Params p)
{
    constexpr int QT = kBN / H;   // queries per tile
    // lone-query tiles (decode) pack QT pool tiles per accumulator (H >= 64)
    constexpr bool kQuad = kFew && H >= 64;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    // 1024-byte aligned base, derived by pointer arithmetic so that every pointer
    // below stays a shared-memory pointer (LDS/STS/ATOMS, not generic accesses)
    uint8_t *smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
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
        for (int i = 4; i < 8; ++i) misc[i] = 0u;
        int *qcnt0 = reinterpret_cast<int *>(smem + L.cnt_off);
        uint32_t *thr0 = reinterpret_cast<uint32_t *>(smem + L.thr_off);
        for (int q = 0; q < QT; ++q) {
            qcnt0[q] = 0;
            thr0[q] = 0u;
        }
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
    Sync sy{reinterpret_cast<volatile uint32_t *>(&misc[1]), p.ws + WS_STATUS, p.wait_limit_ns};

    auto tile_info = [&](int tile) {
        TileInfo t{};
        int d;
        if (p.units != nullptr) {
            const int4 *u = reinterpret_cast<const int4 *>(p.units) + 2 * tile;
            const int4 a = u[0], b = u[1];
            t.t0 = a.x;
            d = a.y;
            t.i0 = a.z;
            t.i1 = a.w;
            t.slot_base = b.x;
            t.splits = b.y;
            t.tile = b.z;
            t.k = b.w;
        } else {
            const int2 e = reinterpret_cast<const int2 *>(p.ws + WS_TABLE_INTS)[tile];
            t.t0 = e.x;
            d = e.y;
            t.i0 = 0;
            t.i1 = -1;
            t.slot_base = -1;
            t.splits = 1;
            t.tile = tile;
        }
        t.pos_base = p.q_pos != nullptr ? p.q_pos[d] : 0;
        if (p.cu_seqlens != nullptr) {
            t.doc_start = p.cu_seqlens[d];
            t.doc_end = p.cu_seqlens[d + 1];
            t.pool_base = p.cu_pools[d];
            t.pool_count = p.cu_pools[d + 1] - p.cu_pools[d];
        } else {
            t.doc_start = 0;
            t.doc_end = p.T;
            t.pool_base = 0;
            t.pool_count = p.P_total;
        }
        if (t.i1 < 0) t.i1 = pool_tiles_of(t, QT, p.kp);
        return t;
    };

    // registers: the producer/MMA/allocator warpgroup gives up most of its share
    // to the two epilogue warpgroups (head weights stay in registers)
    if (warp < 4) {
    ptx::setmaxnreg_dec<kRegsOther>();
    if (warp == 0) {
        // ---------------- TMA producer + scheduler ----------------
        if (lane == 0) {
            PT_DECL
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
                PT_MARK(4);
                if (!wait_bar(bar(BTI_EMPTY + slot), tph ^ 1, sy)) break;
                PT_MARK(0);
                const int tile = atomicAdd(p.ws + WS_COUNTER, 1);
                TileInfo t{};
                if (tile >= ntiles) {
                    t.t0 = -1;
                } else {
                    t = tile_info(tile);
                }
                ti_slots[slot] = t;   // published by the mbarrier arrive (release)
                ptx::mbar_arrive(bar(BTI_FULL + slot));
                if (t.t0 < 0) break;
                if (t.i1 <= t.i0) continue;
                PT_MARK(4);
                if (!wait_bar(bar(BQ_EMPTY), qe_ph ^ 1, sy)) break;
                PT_MARK(1);
                qe_ph ^= 1;
                ptx::mbar_arrive_expect_tx(bar(BQ_FULL), p.q_tx);
                for (int c = 0; c < L.n_kchunks; ++c)
                    ptx::tma_load_2d(sbase + L.q_off + c * L.q_chunk, &tm_q, bar(BQ_FULL),
                                     c * celem, t.t0 * H);
                q_issued = true;
                q_issued_ph = qe_ph ^ 1;
                bool ok = true;
                for (int i = t.i0; i < t.i1; ++i) {
                    PT_MARK(3);
                    if (!wait_bar(bar(BPK_FULL + S + stage), ph ^ 1, sy)) { ok = false; break; }
                    PT_MARK(2);
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
            PT_MARK(4);
            PT_FLUSH(16);
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer ----------------
        if (lane == 0) {
            PT_DECL
            int stage = 0, acc = 0;
            uint32_t ph = 0, qf_ph = 0, acc_ph = 0;
            bool any = false;
            for (int it = 0;; ++it) {
                const int slot = it & 1;
                const uint32_t tph = (it >> 1) & 1;
                PT_MARK(5);
                if (!wait_bar(bar(BTI_FULL + slot), tph, sy)) break;
                PT_MARK(0);
                const TileInfo t = ti_slots[slot];   // after the acquiring wait
                ptx::mbar_arrive(bar(BTI_EMPTY + slot));
                if (t.t0 < 0) break;
                const int npt = t.i1 - t.i0;
                if (npt <= 0) continue;
                // N = the tile's (query, head) columns, rounded up to 16; a lone
                // query (decode) packs QT pool tiles into one accumulator, N = H each
                uint32_t idesc = p.idesc;
                bool quad = false;
                if constexpr (kFew) {
                    const int nqm = min(QT, t.doc_end - t.t0);
                    quad = kQuad && nqm == 1;
                    const int ncols = min(kBN, ((nqm * H + 15) / 16) * 16);
                    idesc = (p.idesc & ~(0x3Fu << 17)) | (static_cast<uint32_t>(ncols >> 3) << 17);
                }
                PT_MARK(5);
                if (!wait_bar(bar(BQ_FULL), qf_ph, sy)) break;
                PT_MARK(1);
                qf_ph ^= 1;
                bool ok = true;
                for (int i = 0; i < npt; ++i) {
                    const int sub = quad ? i % QT : 0;   // pool tile's column block
                    PT_MARK(4);
                    if (sub == 0 && !wait_bar(bar(BTM_EMPTY + acc), acc_ph ^ 1, sy)) {
                        ok = false;
                        break;
                    }
                    PT_MARK(2);
                    if (!wait_bar(bar(BPK_FULL + stage), ph, sy)) { ok = false; break; }
                    PT_MARK(3);
                    ptx::tc_fence_after();
                    const uint32_t d_tmem = tmem_base + acc * kAccCols + sub * H;
                    // descriptors of the K slices: the start-address field advances by
                    // 32 bytes per MMA inside a 128-byte swizzled row, by a chunk
                    // between 128-byte K chunks
                    const uint64_t ad0 = ptx::smem_desc_sw128(sbase + L.pk_off + stage * L.pk_stage);
                    const uint64_t bd0 = ptx::smem_desc_sw128(sbase + L.q_off);
                    if (p.fp8) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)
                            ptx::mma_fp8(d_tmem, ad0 + kk * 2, bd0 + kk * 2, idesc, kk != 0);
                    } else {
                        for (int c = 0; c < L.n_kchunks; ++c) {
                            const uint64_t ad = ad0 + ((c * L.pk_chunk) >> 4);
                            const uint64_t bd = bd0 + ((c * L.q_chunk) >> 4);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                ptx::mma_bf16(d_tmem, ad + kk * 2, bd + kk * 2, idesc,
                                              (c | kk) != 0);
                        }
                    }
                    ptx::mma_commit(bar(BPK_FULL + S + stage));
                    any = true;
                    if (++stage == S) { stage = 0; ph ^= 1; }
                    if (!quad || sub == QT - 1 || i == npt - 1) {
                        ptx::mma_commit(bar(BTM_FULL + acc));
                        if (++acc == 2) { acc = 0; acc_ph ^= 1; }
                    }
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
            PT_MARK(5);
            PT_FLUSH(8);
        }
    }
    } else {
        ptx::setmaxnreg_inc<kRegsEpi>();
        // ---------------- epilogue ----------------
        // 16 warps: warp (slice, quarter) reads TMEM lanes 32*quarter.. (its 32
        // pools) and columns 64*slice.. of the 256 (query, head) columns.
        constexpr int SLICE = 64;                                  // columns per warp
        constexpr bool kHalfQ = H > SLICE;                         // a query spans two slices
        constexpr int QS = kHalfQ ? 1 : SLICE / H;                 // queries per warp
        constexpr int NACC = H >= 32 ? 4 : (H >= 16 ? 2 : 1);     // FFMA2 chains per query
        const int ew = warp - 4;
        const int qr = warp & 3;            // TMEM lane quarter
        const int sl = ew >> 2;             // column slice
        const int qbase = kHalfQ ? (sl >> 1) : sl * QS;   // first query of this warp
        const bool owner = !kHalfQ || (sl & 1) == 0;      // appends the query's score
        const int etid = threadIdx.x - 128;
        const int g = ew / kGroupWarps;     // selection group
        const int gtid = etid - g * kGroupThreads;
        int *hist = reinterpret_cast<int *>(smem + L.hist_off) + g * 256;
        int *gs = reinterpret_cast<int *>(smem + L.scr_off) + g * 32;
        // the wide group (all sixteen warps, a lone query) uses group 0's histogram
        // and every group's scratch words
        int *hist0 = reinterpret_cast<int *>(smem + L.hist_off);
        int *gs0 = reinterpret_cast<int *>(smem + L.scr_off);
        int *qcnt = reinterpret_cast<int *>(smem + L.cnt_off);   // candidates per query
        uint32_t *thr_s = reinterpret_cast<uint32_t *>(smem + L.thr_off);
        float *cs = reinterpret_cast<float *>(smem + L.cs_off);
        int *ci = reinterpret_cast<int *>(smem + L.ci_off);
        float *cd = cs;                  // direct mode: query q's scores at cd[q * CD + pool]
        const int CD = L.C;
        float *wsm = reinterpret_cast<float *>(smem + L.ws_off);  // 256 head weights
        float *part = wsm + kBN;                                   // [2][4][128] partial scores
        const ulonglong2 *w4 = reinterpret_cast<const ulonglong2 *>(wsm + sl * SLICE);
        // H >= 32: the accumulator is read with the 16x256b shape, so a thread holds 4
        // pools x 16 head columns (columns 8j + 2kq, +1) and keeps its 16 head weights
        // in registers for the whole query tile; the 4 threads of a quad (same rq)
        // finish each pool's head sum with a 2-step transpose-reduce, after which
        // thread (rq, kq) owns pool lane rq + 8 * (2 * (kq & 1) + (kq >> 1)).
        constexpr bool kQL = H >= 32;
        const int kq = lane & 3, rq = lane >> 2;
        const int own = kQL ? rq + 8 * (2 * (kq & 1) + (kq >> 1)) : lane;
        uint64_t wq[kQL ? 8 : 1];
        const int C = L.C;
        const int Kp = p.Kp;
        const int slack = max(0, min(kSlack, C - kBM - Kp));
        // tiles between capacity checks; a query above `room` candidates at a
        // check is compacted, so the next G tiles (<= 128 each) always fit.  G
        // takes at most half of the space above the kept Kp + slack.
        const int G = max(1, min(8, (C - Kp - slack) / (2 * kBM)));
        const int room = C - G * kBM;
        const unsigned lt = (1u << lane) - 1u;
        int acc = 0, tile_seq = 0;
        uint32_t acc_ph = 0;
        PT_DECL
        // The 16 epilogue warps meet at named barriers, so they leave the tile
        // loop only together: a warp whose wait fails (timeout or CTA abort)
        // raises a per-iteration agreement word and keeps to the common control
        // flow; every warp reads the word after the next barrier they all pass
        // (the weight-staging barrier for the tile-info wait, the barrier before
        // the final selection for the accumulator waits) and they all leave
        // there.  Words alternate by iteration parity: a word is written only
        // before its barrier and read only after it, and its next use is two
        // iterations (several barriers) later.
        for (int it = 0;; ++it) {
            const int slot = it & 1;
            const uint32_t tph = (it >> 1) & 1;
            volatile uint32_t *agree_ti = misc + 4 + slot;   // a tile-info wait failed
            volatile uint32_t *agree_tm = misc + 6 + slot;   // an accumulator wait failed
            PT_MARK(7);
            const bool ti_ok = wait_bar_warp(bar(BTI_FULL + slot), tph, sy);
            PT_MARK(0);
            TileInfo t{};
            t.t0 = -1;
            if (ti_ok) t = ti_slots[slot];
            if (kFew && etid == 0 && ti_ok) ti_slots[2] = t;   // for the unit's end (visible after the w barrier)
            __syncwarp();
            if (lane == 0) {
                if (ti_ok) ptx::mbar_arrive(bar(BTI_EMPTY + slot));
                else *agree_ti = 1u;
            }
            const int tau0 = t.pos_base + (t.t0 - t.doc_start);
            const int nq = min(QT, t.doc_end - t.t0);

            // the tile's 256 head weights (w, times q_scale in FP8 mode), staged in
            // shared memory once per query tile and read back as broadcasts
            const bool lone = kQuad && nq == 1;   // its weights fill every query's columns
            if (etid < kBN) {
                const int qi = lone ? 0 : etid / H;
                float v = 0.f;
                if (t.t0 >= 0 && qi < nq) {
                    const int64_t off = static_cast<int64_t>(t.t0) * H + (lone ? etid % H : etid);
                    v = __ldg(p.w + off);
                    if (p.fp8) v *= __ldg(p.q_scale + off);
                }
                wsm[etid] = 0.5f * v;   // halved: the head sums take 2 relu(x) = x + |x|
            }
            ptx::named_bar_sync(1, kEpiThreads);
            if (*agree_ti != 0u || t.t0 < 0) break;   // the same outcome in every warp
            if constexpr (kQL) {
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const float2 wv2 = *reinterpret_cast<const float2 *>(wsm + sl * SLICE + 8 * j + 2 * kq);
                    wq[j] = ptx::pack_f32x2(wv2.x, wv2.y);
                }
            }

            float thf[QS];   // pass_floor of each query's threshold key
            int nc[QS];
#pragma unroll
            for (int j = 0; j < QS; ++j) {
                thf[j] = -INFINITY;
                nc[j] = min((tau0 + qbase + j + 1) / p.kp, t.pool_count);
            }
            bool aborted = false;
            // Direct mode: when every visible pool of the tile's queries fits a
            // query's candidate capacity C, scores are stored at their pool
            // position and the final selection reads them in pool order (no
            // appends, no compaction, no bitmap ranking).  Longer rows keep the
            // threshold filter, whose compactions leave the final selection
            // fewer entries than a row's full pool count.  Not for split units
            // or a lone decode query.
            const int nc_tile = min((tau0 + nq) / p.kp, t.pool_count);
            const bool direct = kDirect && p.mode == 0 && nc_tile <= C;

            // Head sums of accumulator `acc_sel` for this thread's pool(s) (H >= 32):
            // relu(x) * w over the warp's 64 columns, then the quad transpose-reduce.
            // Releases the accumulator once its TMEM reads are done.
            auto head_sums_ql = [&](uint32_t acc_sel, float (&s_out)[QS]) {
                const uint32_t tb = tmem_base + (static_cast<uint32_t>(qr * 32) << 16) +
                                    acc_sel * kAccCols + sl * SLICE;
                uint32_t va[32], vb[32];
                ptx::tmem_ld16x256_x8(tb, va);
                ptx::tmem_ld16x256_x8(tb + (16u << 16), vb);
                ptx::tmem_ld_wait2(va, vb);
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive(bar(BTM_EMPTY + acc_sel));
                uint64_t a[QS][4];
#pragma unroll
                for (int j = 0; j < QS; ++j)
#pragma unroll
                    for (int l = 0; l < 4; ++l) a[j][l] = 0ull;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    const int qj = kHalfQ ? 0 : (8 * j) / H;
                    a[qj][0] = ptx::ffma2(ptx::pack_f32x2(twice_relu(__uint_as_float(va[4 * j])),
                                                          twice_relu(__uint_as_float(va[4 * j + 1]))),
                                          wq[j], a[qj][0]);
                    a[qj][1] = ptx::ffma2(ptx::pack_f32x2(twice_relu(__uint_as_float(va[4 * j + 2])),
                                                          twice_relu(__uint_as_float(va[4 * j + 3]))),
                                          wq[j], a[qj][1]);
                    a[qj][2] = ptx::ffma2(ptx::pack_f32x2(twice_relu(__uint_as_float(vb[4 * j])),
                                                          twice_relu(__uint_as_float(vb[4 * j + 1]))),
                                          wq[j], a[qj][2]);
                    a[qj][3] = ptx::ffma2(ptx::pack_f32x2(twice_relu(__uint_as_float(vb[4 * j + 2])),
                                                          twice_relu(__uint_as_float(vb[4 * j + 3]))),
                                          wq[j], a[qj][3]);
                }
                const bool b0 = (kq & 1) != 0, b1 = (kq & 2) != 0;
#pragma unroll
                for (int j = 0; j < QS; ++j) {
                    const float s0 = ptx::sum_f32x2(a[j][0]), s1 = ptx::sum_f32x2(a[j][1]);
                    const float s2 = ptx::sum_f32x2(a[j][2]), s3 = ptx::sum_f32x2(a[j][3]);
                    // step 1 (partner kq ^ 1): keep lanes {0, 8} or {16, 24}
                    const float r0 = __shfl_xor_sync(kFull, b0 ? s0 : s2, 1);
                    const float r1 = __shfl_xor_sync(kFull, b0 ? s1 : s3, 1);
                    const float t0 = (b0 ? s2 : s0) + r0;
                    const float t1 = (b0 ? s3 : s1) + r1;
                    // step 2 (partner kq ^ 2): keep one of the two
                    const float r2 = __shfl_xor_sync(kFull, b1 ? t0 : t1, 2);
                    s_out[j] = (b1 ? t1 : t0) + r2;
                }
            };

            // The pool-tile loop.  (Counted from 0: a loop over [i0, i1), or one
            // with a per-warp branch, compiles to a slower body.)
            const int npt = t.i1 - t.i0;
            auto tiles = [&](auto direct_tag) {
            constexpr bool kDirect = decltype(direct_tag)::value;
            int gleft = G;   // tiles to the next capacity check (a countdown, not i % G)
            for (int i = 0; i < npt; ++i) {
                PT_MARK(1);
                aborted |= !wait_bar_warp(bar(BTM_FULL + acc), acc_ph, sy);
                PT_MARK(2);
                ptx::tc_fence_after();
                float s[QS];
                if constexpr (kQL) {
                    head_sums_ql(acc, s);
                    if (++acc == 2) { acc = 0; acc_ph ^= 1; }
                } else {
                // relu(x) * w summed per query over this warp's 64 columns
                uint64_t a4[QS][NACC];
#pragma unroll
                for (int j = 0; j < QS; ++j)
#pragma unroll
                    for (int k = 0; k < NACC; ++k) a4[j][k] = 0ull;
                auto accum = [&](const uint32_t(&v)[32], const int c0) {
#pragma unroll
                    for (int x = 0; x < 32; x += 4) {
                        const int col = c0 + x;
                        const int j = kHalfQ ? 0 : col / H;
                        const int k = (col / 4) % NACC;
                        const ulonglong2 wv = w4[col / 4];
                        const uint64_t r0 = ptx::pack_f32x2(twice_relu(__uint_as_float(v[x])),
                                                            twice_relu(__uint_as_float(v[x + 1])));
                        const uint64_t r1 = ptx::pack_f32x2(twice_relu(__uint_as_float(v[x + 2])),
                                                            twice_relu(__uint_as_float(v[x + 3])));
                        a4[j][k] = ptx::ffma2(r0, wv.x, a4[j][k]);
                        a4[j][k] = ptx::ffma2(r1, wv.y, a4[j][k]);
                    }
                };
                {
                    const uint32_t tb = tmem_base + (static_cast<uint32_t>(qr * 32) << 16) +
                                        acc * kAccCols + sl * SLICE;
                    uint32_t v0[32], v1[32];
                    ptx::tmem_ld32(tb, v0);
                    ptx::tmem_ld32(tb + 32, v1);
                    ptx::tmem_ld_wait2(v0, v1);
                    ptx::tc_fence_before();
                    __syncwarp();
                    if (lane == 0) ptx::mbar_arrive(bar(BTM_EMPTY + acc));
                    accum(v0, 0);
                    accum(v1, 32);
                }
                if (++acc == 2) { acc = 0; acc_ph ^= 1; }
#pragma unroll
                for (int j = 0; j < QS; ++j) {
                    float v = ptx::sum_f32x2(a4[j][0]);
#pragma unroll
                    for (int k = 1; k < NACC; ++k) v += ptx::sum_f32x2(a4[j][k]);
                    s[j] = v;
                }
                }

                const int pool_local = (i + t.i0) * kBM + qr * 32 + own;
                const int pool_g = t.pool_base + pool_local;
                if (kHalfQ) {
                    // the two 64-head halves of a query meet in shared memory
                    float *pt = part + (tile_seq & 1) * (4 * kBM);
                    pt[sl * kBM + qr * 32 + own] = s[0];
                    ptx::named_bar_sync(1, kEpiThreads);
                    if (owner) s[0] += pt[(sl + 1) * kBM + qr * 32 + own];
                }
                ++tile_seq;
                float sk = 1.f;
                if (p.fp8 && pool_g < p.P_total) sk = p.pk_scale[pool_g];
#pragma unroll
                for (int j = 0; j < QS; ++j) {
                    float v = s[j];
                    if (p.fp8) v *= sk;
                    s[j] = __fadd_rn(v, 0.f);   // folds -0 into +0
                }
                PT_MARK(3);

                if (p.mode == 1) {   // dense scores (test/debug)
                    if (owner) {
#pragma unroll
                        for (int j = 0; j < QS; ++j) {
                            const int qi = qbase + j;
                            if (qi < nq && pool_local < nc[j])
                                p.scores[static_cast<int64_t>(t.t0 + qi) * p.P_total + pool_g] =
                                    s[j];
                        }
                    }
                    continue;
                }

                if constexpr (kDirect) {
                    // every visible pool's score at its pool position
                    if (owner) {
#pragma unroll
                        for (int j = 0; j < QS; ++j) {
                            const int qi = qbase + j;
                            if (qi < nq && pool_local < nc[j]) cd[qi * CD + pool_local] = s[j];
                        }
                    }
                    continue;
                }
                // survivors of the threshold filter, appended (unordered) with one
                // shared-memory atomic per warp and query that has any
                if (owner) {
#pragma unroll
                    for (int j = 0; j < QS; ++j) {
                        const int qi = qbase + j;
                        const bool ps = (qi < nq) && (pool_local < nc[j]) && s[j] >= thf[j];
                        const unsigned bal = __ballot_sync(kFull, ps);
                        if (bal != 0u) {
                            int base = 0;
                            if (lane == 0) base = atomicAdd(&qcnt[qi], __popc(bal));
                            base = __shfl_sync(kFull, base, 0);
                            if (ps) {
                                const int d = qi * C + base + __popc(bal & lt);
                                cs[d] = s[j];
                                ci[d] = pool_g;
                            }
                        }
                    }
                }
                PT_MARK(4);
                const bool check = --gleft == 0;
                if (check) gleft = G;
                if (check && i != npt - 1) {
                    // capacity check: compact queries past the room, plus those past
                    // half of it, each group on its own queries in parallel
                    ptx::named_bar_sync(1, kEpiThreads);
                    bool over = false;
                    for (int q = lane; q < QT; q += 32) over |= qcnt[q] > room;
                    if (__any_sync(kFull, over)) {
                        for (int q = g; q < QT; q += kGroups) {
                            const int n = qcnt[q];
                            if (n > (room + Kp) / 2) {
                                const int nn = group_select(cs + q * C, ci + q * C, n, Kp, false,
                                                            slack, g, gtid, hist, gs, &thr_s[q]);
                                if (gtid == 0) qcnt[q] = nn;
                            }
                        }
                        ptx::named_bar_sync(1, kEpiThreads);
#pragma unroll
                        for (int j = 0; j < QS; ++j) thf[j] = pass_floor(thr_s[qbase + j]);
                    }
                    PT_MARK(5);
                }
            }
            };
            if constexpr (kQuad) {
                if (nq == 1) {
                    // A lone query (decode): pool tile m*QT + j sits in the columns of
                    // query j of accumulator m, so every warp works on the query; its
                    // candidates may use every query's area (capacity QT * C)
                    const int nquad = (npt + QT - 1) / QT;
                    const int nc0 = min((tau0 + 1) / p.kp, t.pool_count);
                    const int Gq = max(1, min(4, (QT * C - Kp - slack) / (QT * kBM)));
                    const int room_q = QT * C - Gq * QT * kBM;
                    uint32_t thr0 = 0u;
                    for (int m = 0; m < nquad; ++m) {
                        PT_MARK(1);
                        aborted |= !wait_bar_warp(bar(BTM_FULL + acc), acc_ph, sy);
                        PT_MARK(2);
                        ptx::tc_fence_after();
                        float svq[QS];
                        head_sums_ql(acc, svq);   // kQuad implies H >= 64
                        if (++acc == 2) { acc = 0; acc_ph ^= 1; }
                        float sv = svq[0];
                        if (kHalfQ) {
                            float *pt = part + (tile_seq & 1) * (4 * kBM);
                            pt[sl * kBM + qr * 32 + own] = sv;
                            ptx::named_bar_sync(1, kEpiThreads);
                            if (owner) sv += pt[(sl + 1) * kBM + qr * 32 + own];
                        }
                        ++tile_seq;
                        const int tj = m * QT + qbase;   // this warp's pool tile of the unit
                        const int pool_local = (t.i0 + tj) * kBM + qr * 32 + own;
                        const int pool_g = t.pool_base + pool_local;
                        if (p.fp8 && pool_g < p.P_total) sv *= p.pk_scale[pool_g];
                        sv = __fadd_rn(sv, 0.f);   // folds -0 into +0
                        PT_MARK(3);
                        if (owner) {
                            const bool ps = tj < npt && pool_local < nc0 && fkey(sv) > thr0;
                            const unsigned bal = __ballot_sync(kFull, ps);
                            if (bal != 0u) {
                                int base = 0;
                                if (lane == 0) base = atomicAdd(&qcnt[0], __popc(bal));
                                base = __shfl_sync(kFull, base, 0);
                                if (ps) {
                                    const int d = base + __popc(bal & lt);
                                    cs[d] = sv;
                                    ci[d] = pool_g;
                                }
                            }
                        }
                        PT_MARK(4);
                        if ((m % Gq) == Gq - 1 && m != nquad - 1) {
                            ptx::named_bar_sync(1, kEpiThreads);
                            if (qcnt[0] > room_q) {
                                // all sixteen warps prune the lone query's area
                                const int nn = group_select<kEpiWarps>(cs, ci, qcnt[0], Kp, false,
                                                                       slack, 0, etid, hist0, gs0,
                                                                       &thr_s[0]);
                                if (etid == 0) qcnt[0] = nn;
                                ptx::named_bar_sync(1, kEpiThreads);
                                thr0 = thr_s[0];
                            }
                            PT_MARK(5);
                        }
                    }
                } else {
                    tiles(std::false_type{});
                }
            } else if constexpr (kDirect) {
                if (direct) tiles(std::true_type{});
                else tiles(std::false_type{});
            } else {
                tiles(std::false_type{});
            }
            // after an abort the loop ran on to the tile's end without waiting
            // (its scores are garbage); all warps leave here together
            if (aborted && lane == 0) *agree_tm = 1u;
            PT_MARK(1);
            ptx::named_bar_sync(1, kEpiThreads);   // also: w staging is rewritten next
            if (*agree_tm != 0u) break;
            if (p.mode == 1) continue;

            // final selection, pool order and output: every group on its own queries
            bool emit = true;
            if constexpr (kFew) {
                if (ti_slots[2].splits > 1)
                    emit = split_unit_end(ti_slots + 2, nq, QT, Kp, C, cs, ci, qcnt, thr_s, hist, gs,
                                          g, gtid, etid, misc + 2, p.part_idx, p.part_score,
                                          p.part_cnt, p.tile_ctr);
            }
            for (int q = g; kDirect && q < nq && emit && direct; q += kGroups) {
                const int64_t row = static_cast<int64_t>(t.t0 + q) * Kp;
                const int nc_q = min((tau0 + q + 1) / p.kp, t.pool_count);
                const int n = group_select_direct(cd + q * CD, nc_q, Kp, t.pool_base, g, gtid,
                                                  hist, gs, p.pool_idx + row, p.pool_score + row);
                for (int e = n + gtid; e < Kp; e += kGroupThreads) {
                    p.pool_idx[row + e] = -1;
                    p.pool_score[row + e] = -INFINITY;
                }
            }
            bool lone_done = false;
            if constexpr (kQuad) {
                if (nq == 1 && emit && !direct) {
                    // a lone query: all sixteen warps select and store it
                    constexpr int NW = kEpiWarps;
                    int n = qcnt[0];
                    if (n > Kp) {
                        group_select<NW>(cs, ci, n, Kp, true, 0, 0, etid, hist0, gs0, &thr_s[0]);
                        n = Kp;
                    }
                    const int64_t row = static_cast<int64_t>(t.t0) * Kp;
                    const int nc_q = min((tau0 + 1) / p.kp, t.pool_count);
                    const int words = (nc_q + 31) / 32;
                    if (words <= QT * C - n) {
                        group_rank_store<NW>(cs, ci, n, t.pool_base, words, 0, etid, gs0,
                                             p.pool_idx + row, p.pool_score + row);
                    } else {
                        group_sort_by_pool<NW>(cs, ci, n, 0, etid);
                        for (int e = etid; e < n; e += kEpiThreads) {
                            p.pool_idx[row + e] = ci[e];
                            p.pool_score[row + e] = cs[e];
                        }
                    }
                    for (int e = n + etid; e < Kp; e += kEpiThreads) {
                        p.pool_idx[row + e] = -1;
                        p.pool_score[row + e] = -INFINITY;
                    }
                    lone_done = true;
                }
            }
            for (int q = g; q < nq && emit && !direct && !lone_done; q += kGroups) {
                int n = qcnt[q];
                float *csq = cs + q * C;
                int *ciq = ci + q * C;
                if (n > Kp) {
                    group_select(csq, ciq, n, Kp, true, 0, g, gtid, hist, gs, &thr_s[q]);
                    n = Kp;
                }
                const int64_t row = static_cast<int64_t>(t.t0 + q) * Kp;
                const int nc_q = min((tau0 + q + 1) / p.kp, t.pool_count);   // visible local pools
                const int words = (nc_q + 31) / 32;
                if (words <= (kQuad && nq == 1 ? QT * C : C) - n) {
                    group_rank_store(csq, ciq, n, t.pool_base, words, g, gtid, gs,
                                     p.pool_idx + row, p.pool_score + row);
                } else {
                    group_sort_by_pool(csq, ciq, n, g, gtid);
                    for (int e = gtid; e < n; e += kGroupThreads) {
                        p.pool_idx[row + e] = ciq[e];
                        p.pool_score[row + e] = csq[e];
                    }
                }
                for (int e = n + gtid; e < Kp; e += kGroupThreads) {
                    p.pool_idx[row + e] = -1;
                    p.pool_score[row + e] = -INFINITY;
                }
            }
            group_bar(g);
            for (int q = g; q < QT; q += kGroups) {
                if (gtid == 0) {
                    qcnt[q] = 0;
                    thr_s[q] = 0u;
                }
            }
            ptx::named_bar_sync(1, kEpiThreads);
            PT_MARK(6);
        }
        PT_MARK(7);
        if (lane == 0) PT_FLUSH(24);
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
    __shared__ int s_ntiles;
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

// Sum over the block (1024 threads); every thread gets the total.
__device__ int block_sum(int v, int *red)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    v = __reduce_add_sync(kFull, v);
    __syncthreads();   // red reuse
    if (lane == 0) red[wid] = v;
    __syncthreads();
    int tot = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) tot += red[w];
    return tot;
}

// Exclusive prefix over the block in thread order; *total gets the sum.
__device__ int block_exclusive_scan(int v, int *red, int *total)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += o;
    }
    __syncthreads();   // red reuse
    if (lane == 31) red[wid] = incl;
    __syncthreads();
    int before = 0, tot = 0;
    for (int w = 0; w < static_cast<int>(blockDim.x >> 5); ++w) {
        if (w < wid) before += red[w];
        tot += red[w];
    }
    *total = tot;
    return before + incl - v;
}

// Split-pool schedule (one block of 1024 threads, one query tile per thread).
// The W pool tiles of all query tiles are cut into units of about
// W / (4 * grid) pool tiles (at least kSplitMinTiles): a query tile with more
// pool tiles becomes min(splits_max, ceil(npt / U)) units of nearly equal
// length, U doubling until the split units fit the `slots` partial lists.
// Table: the split units first (tile by tile; their table positions are their
// partial-list slots), then the unsplit query tiles.  Also validates
// cu_seqlens and resets the tile counter, the status word and the per-tile
// arrival counters.
__global__ void __launch_bounds__(1024)
    split_schedule_kernel(const int32_t *cu, const int32_t *q_pos, const int32_t *cu_pools,
                          int n_docs, int T, int P_total, int QT, int kp, int grid, int slots,
                          int splits_max, int *ws, int *units, int *ctr)
{
    __shared__ int s_nt;
    __shared__ int red[32];
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
        if (nt > static_cast<int>(blockDim.x)) ok = 0;
        s_nt = ok ? nt : 0;
        ws[WS_COUNTER] = 0;
        ws[WS_STATUS] = ok ? 0 : KPOOL_STATUS_BAD_SEQLENS;
    }
    __syncthreads();
    const int nt = s_nt;
    const int g = threadIdx.x;
    int t0 = 0, d = 0, npt = 0;
    if (g < nt) {
        int i = g;
        if (cu != nullptr) {
            int acc = 0;
            for (d = 0; d < n_docs; ++d) {
                const int n = (cu[d + 1] - cu[d] + QT - 1) / QT;
                if (g < acc + n) break;
                acc += n;
            }
            i = g - acc;
        }
        const int doc_start = cu != nullptr ? cu[d] : 0;
        const int doc_end = cu != nullptr ? cu[d + 1] : T;
        const int pool_count = cu != nullptr ? cu_pools[d + 1] - cu_pools[d] : P_total;
        const int pos = (q_pos != nullptr ? q_pos[d] : 0) + i * QT;
        t0 = doc_start + i * QT;
        const int nq = min(QT, doc_end - t0);
        const int nc_last = min((pos + nq) / kp, pool_count);   // as pool_tiles_of
        npt = (nc_last + kBM - 1) / kBM;
    }
    const int W = block_sum(min(npt, 1 << 20), red);
    int U = max(kSplitMinTiles, (W + 4 * grid - 1) / (4 * grid));
    int sp = 1;
    for (int iter = 0; iter < 31; ++iter) {
        sp = npt > U ? min(splits_max, (npt + U - 1) / U) : 1;
        if (block_sum(sp > 1 ? sp : 0, red) <= slots) break;
        U *= 2;
    }
    if (block_sum(sp > 1 ? sp : 0, red) > slots) sp = 1;   // (not reached: U outgrows every npt)
    int n_split = 0, n_whole = 0;
    const int ex_s = block_exclusive_scan(sp > 1 ? sp : 0, red, &n_split);
    const int ex_w = block_exclusive_scan(g < nt && sp == 1 ? 1 : 0, red, &n_whole);
    int4 *u4 = reinterpret_cast<int4 *>(units);
    if (g < nt) {
        ctr[g] = 0;
        if (sp > 1) {
            for (int k = 0; k < sp; ++k) {
                const int at = ex_s + k;
                u4[2 * at] = make_int4(t0, d, static_cast<int>(static_cast<int64_t>(k) * npt / sp),
                                       static_cast<int>(static_cast<int64_t>(k + 1) * npt / sp));
                u4[2 * at + 1] = make_int4(ex_s, sp, g, k);
            }
        } else {
            const int at = n_split + ex_w;
            u4[2 * at] = make_int4(t0, d, 0, npt);
            u4[2 * at + 1] = make_int4(-1, 1, g, 0);
        }
    }
    if (threadIdx.x == 0) ws[WS_NTILES] = n_split + n_whole;
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

// Limit of one pipeline wait, for every scoring launch of the process
// (kpool_debug_set_wait_limit_ns; tests lower it to make waits expire).
std::atomic<uint64_t> g_wait_limit_ns{kTimeoutNs};

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

template <int H, bool kFew, bool kDirect>
int launch_hf(const Layout &L, const CUtensorMap &mq, const CUtensorMap &mpk, const Params &prm,
              int grid, cudaStream_t s)
{
    const int smem = static_cast<int>(L.total) + 1024;
    KPOOL_CUDA_CHECK(cudaFuncSetAttribute(score_kernel<H, kFew, kDirect>,
                                          cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    score_kernel<H, kFew, kDirect><<<grid, kThreads, smem, s>>>(mq, mpk, prm);
    KPOOL_CUDA_CHECK(cudaGetLastError());
    return KPOOL_OK;
}

// Three instantiations: the split-pool schedule for calls with few query
// tiles; direct mode for calls whose documents are short on average (at most
// 4C pools each: their short tiles skip the threshold filter); and the long
// prefill loop, which carries no code of the other two.
template <int H>
int launch_h(const ScoreArgs &a, const Layout &L, const CUtensorMap &mq, const CUtensorMap &mpk,
             const Params &prm, int grid, cudaStream_t s)
{
    if (prm.units != nullptr) return launch_hf<H, true, false>(L, mq, mpk, prm, grid, s);
    if (a.mode == 0 && a.P_total <= 4 * static_cast<int64_t>(L.C) * a.n_docs)
        return launch_hf<H, false, true>(L, mq, mpk, prm, grid, s);
    return launch_hf<H, false, false>(L, mq, mpk, prm, grid, s);
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

#ifdef KPOOL_PHASE_TIMERS
extern "C" KPOOL_API int kpool_debug_phase_timers(unsigned long long *out32, int reset)
{
    KPOOL_CUDA_CHECK(cudaDeviceSynchronize());
    KPOOL_CUDA_CHECK(cudaMemcpyFromSymbol(out32, g_phase_timers, 32 * sizeof(unsigned long long)));
    if (reset) {
        static const unsigned long long zero[32] = {};
        KPOOL_CUDA_CHECK(cudaMemcpyToSymbol(g_phase_timers, zero, sizeof zero));
    }
    return KPOOL_OK;
}
#endif

size_t score_workspace_bytes(int64_t T, int H, int n_docs)
{
    const int64_t QT = qt_of(H);
    const int64_t max_tiles = (T + QT - 1) / QT + n_docs;
    size_t b = WS_TABLE_INTS * 4 + static_cast<size_t>(max_tiles) * 8;
    return (b + 255) & ~static_cast<size_t>(255);
}

namespace {

// Workspace layout of the split-pool schedule (offsets in ints from the
// workspace base), after the header and the one-unit-per-tile table.
struct SplitLayout {
    int ok;               // the call may use the split-pool schedule
    int slots;            // partial lists (split units) per call, at most
    int max_units;
    int64_t units_off, ctr_off, cnt_off, idx_off, score_off;
    size_t bytes;
};

SplitLayout split_layout(int64_t T, int H, int n_docs, int Kp)
{
    SplitLayout s{};
    const int64_t QT = qt_of(H);
    const int64_t max_tiles = (T + QT - 1) / QT + n_docs;
    const size_t base = score_workspace_bytes(T, H, n_docs);
    s.bytes = base;
    if (Kp <= 0 || max_tiles > kSplitMaxQT) return s;
    s.slots = static_cast<int>(std::max<int64_t>(1, kSplitEntries / (QT * Kp)));
    s.max_units = kSplitMaxQT + s.slots;
    int64_t off = static_cast<int64_t>(base / 4);
    s.units_off = off; off += static_cast<int64_t>(s.max_units) * 8;
    s.ctr_off = off;   off += kSplitMaxQT;
    s.cnt_off = off;   off += static_cast<int64_t>(s.slots) * QT;
    off = (off + 63) & ~static_cast<int64_t>(63);
    s.idx_off = off;   off += static_cast<int64_t>(s.slots) * QT * Kp;
    s.score_off = off; off += static_cast<int64_t>(s.slots) * QT * Kp;
    s.bytes = (static_cast<size_t>(off) * 4 + 255) & ~static_cast<size_t>(255);
    s.ok = 1;
    return s;
}

}  // namespace

size_t score_workspace_split_bytes(int64_t T, int H, int n_docs, int Kp)
{
    return split_layout(T, H, n_docs, Kp).bytes;
}

uint64_t set_wait_limit_ns(uint64_t ns)
{
    return g_wait_limit_ns.exchange(ns == 0 ? kTimeoutNs : ns);
}

uint64_t get_wait_limit_ns() { return g_wait_limit_ns.load(std::memory_order_relaxed); }

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
    // few query tiles (decode, short chunks) with room in the workspace: split
    // their pool lists over the CTAs (C >= 2 Kp lets a merge append a whole
    // partial list after at most one compaction).  That instantiation streams
    // pooled keys through one more stage: its units are memory-bound.
    const SplitLayout SL = split_layout(a.T, a.H, a.n_docs, a.Kp);
    const Layout Lf = make_layout(a.H, a.D, a.fp8, a.fp8 ? 4 : 3);
    const bool split = a.mode == 0 && SL.ok && a.ws_bytes >= SL.bytes && Lf.C >= 2 * a.Kp;
    const Layout L = split ? Lf : make_layout(a.H, a.D, a.fp8);
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
    prm.q_pos = a.q_pos;
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
    prm.wait_limit_ns = g_wait_limit_ns.load(std::memory_order_relaxed);
    prm.L = L;

    int grid;
    if (split) {
        prm.units = a.ws + SL.units_off;
        prm.tile_ctr = a.ws + SL.ctr_off;
        prm.part_cnt = a.ws + SL.cnt_off;
        prm.part_idx = a.ws + SL.idx_off;
        prm.part_score = reinterpret_cast<float *>(a.ws + SL.score_off);
        grid = num_sms();
        split_schedule_kernel<<<1, kSplitMaxQT, 0, s>>>(
            a.cu_seqlens, a.q_pos, a.cu_pools, a.n_docs, static_cast<int>(a.T),
            static_cast<int>(a.P_total), QT, a.kpool, grid, SL.slots, kSplitMaxSplits, a.ws,
            prm.units, prm.tile_ctr);
    } else {
        schedule_kernel<<<1, 1024, 0, s>>>(a.cu_seqlens, a.n_docs, static_cast<int>(a.T), QT,
                                           static_cast<int>(max_tiles), a.ws);
        grid = static_cast<int>(std::min<int64_t>(num_sms(), max_tiles));
    }
    KPOOL_CUDA_CHECK(cudaGetLastError());
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
