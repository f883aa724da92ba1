/*
 * Plain CPU oracle for the KPool DSA indexer (test infrastructure).
 *
 * THIS FILE IS TEST INFRASTRUCTURE.  Only the tests, the smoke check and the
 * CPU-baseline leg of the benchmark may load it.  It shares no code, header,
 * table or helper with the CUDA library: every rounding routine below is
 * written from the number-format definitions, the Hadamard matrix is built
 * explicitly, scores are formed in double precision and selection is a full
 * sort.  Nothing here is blocked, fused or reordered beyond what the method's
 * definition states.
 *
 * Sources (page titles and sections):
 *   [MG]  Megatron-LM PR "GLM5.3 Flash (KDA + mHC + KPool DSA) support + FP8",
 *         Changes section 3 "KPool DSA indexer + NoPE" (pooling, FP32
 *         accumulation, BF16 pooled key, top-k over index_topk // kpool pools,
 *         expansion, always_select_tail, packed-THD restart, FP32 head weights;
 *         the FP8 emulation chain FP32 Hadamard -> BF16 -> E4M3 with a
 *         power-of-two row scale), and the Testing section
 *         (test_kpool_causal_tail: full causal prefix under the budget;
 *         FP8 emulation against a Hadamard-matrix reference).
 *   [SK]  SkyRL PR "GLM-5.3-Flash (glm5_next) Megatron support", commit
 *         "k-pool indexer": per-dimension softmax over each pool's slots of
 *         gate_score + ape, weighting the keys; per-segment compression.
 *   [XT]  xtuner PR "GLM-5.3-Flash F5: NoPE DSA + KPool indexer", Summary and
 *         commit notes: relu homogeneity (head_dim^-0.5 movable into w);
 *         causal [start, end) pool ranges.
 *
 * Readings of points the pages leave open:
 *   - A pool is a candidate for query t iff its last token is <= t
 *     (complete causal pools); the tail is t's own pool only when that pool
 *     is incomplete at t, i.e. (tau+1) mod kp != 0.
 *   - A trailing partial pool of a document is never compressed or scored.
 *   - Ties in selection go to the lower pool index; output pools ascend;
 *     token rows ascend with the tail last; padding is -1 (score -inf).
 *   - Pool and token indices are global (packed) indices.
 *   - FP8: orthonormal Sylvester-order Hadamard (scale 128^-1/2), computed
 *     exactly here (double, exact sum of +-1 terms); s = 2^ceil(log2(amax/448))
 *     over the BF16 row, s = 1 for an all-zero row; E4M3 RNE, satfinite.
 *
 * Pins: tests/test_oracle_pins.py checks every function here against
 * closed forms, library routines and brute force (no function is left
 * unpinned).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Number formats, from their definitions.                              */
/* ------------------------------------------------------------------ */

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 stored fraction bits.  The
 * upper 16 bits of an IEEE binary32 word, so decoding is a shift. */
double ora_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round half to even of a double that is already an integer or half-integer
 * scaled value: returns the nearest integer, ties to the even one. */
static double round_half_even(double r)
{
    double fl = floor(r);
    double diff = r - fl;
    if (diff > 0.5) return fl + 1.0;
    if (diff < 0.5) return fl;
    /* exact tie */
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Round a double to bfloat16, round-to-nearest-even, once.  Precision is 8
 * significant bits; the smallest normal is 2^-126 and subnormals step by
 * 2^-133.  Values whose rounded magnitude reaches 2^128 become infinity. */
uint16_t ora_bf16_from_double(double x)
{
    if (isnan(x)) return 0x7FC0;
    double ax = fabs(x);
    double r;
    if (ax == 0.0) {
        r = 0.0;
    } else if (isinf(x)) {
        r = INFINITY;
    } else {
        int e;
        frexp(ax, &e);               /* ax = m * 2^e, m in [0.5, 1) */
        int ex = e - 1;              /* ax in [2^ex, 2^(ex+1)) */
        if (ex < -126) ex = -126;    /* subnormal range: fixed quantum */
        double q = ldexp(1.0, ex - 7);
        r = round_half_even(ax / q) * q;
        if (r >= ldexp(1.0, 128)) r = INFINITY;
    }
    float f = (float)(signbit(x) ? -r : r);   /* exact: r has <= 8 bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* E4M3 (OCP FP8): 1 sign, 4 exponent (bias 7), 3 fraction bits; exponent
 * field 0 is subnormal (step 2^-9); no infinities; S.1111.111 is NaN, so the
 * largest finite magnitude is 1.75 * 2^8 = 448. */
double ora_e4m3_to_double(uint8_t c)
{
    int s = (c >> 7) & 1;
    int E = (c >> 3) & 0xF;
    int M = c & 7;
    double v;
    if (E == 0xF && M == 7) return NAN;
    if (E == 0) v = ldexp((double)M, -9);
    else v = ldexp(1.0 + M / 8.0, E - 7);
    return s ? -v : v;
}

/* Round to E4M3, nearest-even, saturating to +-448 (satfinite). */
uint8_t ora_e4m3_from_double(double x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double ax = fabs(x);
    if (isnan(x)) return 0x7F;
    if (ax == 0.0) return sign;
    double r;
    if (isinf(ax)) {
        r = 448.0;
    } else {
        int e;
        frexp(ax, &e);
        int ex = e - 1;
        if (ex < -6) ex = -6;        /* subnormal range: quantum 2^-9 */
        double q = ldexp(1.0, ex - 3);
        r = round_half_even(ax / q) * q;
        if (r > 448.0) r = 448.0;
    }
    if (r == 0.0) return sign;
    /* encode r exactly */
    if (r < ldexp(1.0, -6)) {
        int M = (int)(r / ldexp(1.0, -9));
        return (uint8_t)(sign | M);
    }
    int e;
    frexp(r, &e);
    int ex = e - 1;                   /* r in [2^ex, 2^(ex+1)) */
    int M = (int)((r / ldexp(1.0, ex) - 1.0) * 8.0);
    int E = ex + 7;
    return (uint8_t)(sign | (E << 3) | M);
}

/* ------------------------------------------------------------------ */
/* Document / pool bookkeeping ([MG] packed THD restarts pools).        */
/* ------------------------------------------------------------------ */

/* cu_pools[d] = sum over earlier documents of floor(L/kp); returns total. */
int64_t ora_cu_pools(const int32_t *cu_seqlens, int n_docs, int kp, int32_t *cu_pools)
{
    int64_t acc = 0;
    cu_pools[0] = 0;
    for (int d = 0; d < n_docs; d++) {
        int64_t L = (int64_t)cu_seqlens[d + 1] - cu_seqlens[d];
        acc += L / kp;
        cu_pools[d + 1] = (int32_t)acc;
    }
    return acc;
}

static int doc_of_token(const int32_t *cu_seqlens, int n_docs, int64_t t)
{
    for (int d = 0; d < n_docs; d++)
        if (t >= cu_seqlens[d] && t < cu_seqlens[d + 1]) return d;
    return -1;
}

/* ------------------------------------------------------------------ */
/* Compression ([MG] section 3, [SK] k-pool commit).                    */
/* ------------------------------------------------------------------ */

/* For every complete pool j of every document and every dimension d:
 *   a_s   = gate[i_s, d] + ape[s, d]             (s = slot 0..kp-1)
 *   alpha = softmax over s of a_s
 *   pk    = bf16_rne( sum_s alpha_s * k[i_s, d] )
 * with i_s = doc_start + j*kp + s, in double, rounded once.
 * pk_exact (optional) receives the unrounded double value; pk_cond
 * (optional) the condition scale sum_s alpha_s * |k[i_s, d]| of the sum. */
void ora_compress(const uint16_t *k, const uint16_t *gate, const float *ape,
                  const int32_t *cu_seqlens, int n_docs, int D, int kp,
                  uint16_t *pk_out, double *pk_exact, double *pk_cond)
{
    int32_t *cu_pools = (int32_t *)malloc(sizeof(int32_t) * (n_docs + 1));
    ora_cu_pools(cu_seqlens, n_docs, kp, cu_pools);
    for (int doc = 0; doc < n_docs; doc++) {
        int64_t start = cu_seqlens[doc];
        int64_t npool = (int64_t)cu_pools[doc + 1] - cu_pools[doc];
#pragma omp parallel for schedule(static)
        for (int64_t j = 0; j < npool; j++) {
            double a[64];
            for (int d = 0; d < D; d++) {
                double m = -INFINITY;
                for (int s = 0; s < kp; s++) {
                    int64_t i = start + j * kp + s;
                    a[s] = ora_bf16_to_double(gate[i * D + d]) + (double)ape[s * D + d];
                    if (a[s] > m) m = a[s];
                }
                double z = 0.0;
                for (int s = 0; s < kp; s++) z += exp(a[s] - m);
                double acc = 0.0, cond = 0.0;
                for (int s = 0; s < kp; s++) {
                    int64_t i = start + j * kp + s;
                    double alpha = exp(a[s] - m) / z;
                    acc += alpha * ora_bf16_to_double(k[i * D + d]);
                    cond += alpha * fabs(ora_bf16_to_double(k[i * D + d]));
                }
                int64_t g = cu_pools[doc] + j;
                pk_out[g * D + d] = ora_bf16_from_double(acc);
                if (pk_exact) pk_exact[g * D + d] = acc;
                if (pk_cond) pk_cond[g * D + d] = cond;
            }
        }
    }
    free(cu_pools);
}

/* The key path in front of compression (Megatron-LM PR, Changes section 4:
 * linear_wk and k_norm run unquantized, in BF16; section 3 and the SkyRL
 * commit "k-pool indexer": the BF16 per-token compression gate).  For every
 * token t, with W = [W_k; W_g] of shape [2D, hidden] (rows are output
 * features, as a linear layer's weight):
 *   kproj[t, j] = bf16_rne( sum_i x[t, i] * W[j, i] )          j < D
 *   gate[t, j]  = bf16_rne( sum_i x[t, i] * W[D + j, i] )      j < D
 *   mu = mean_j kproj[t, j],  var = mean_j (kproj[t, j] - mu)^2
 *   k[t, j]     = bf16_rne( (kproj[t, j] - mu) / sqrt(var + eps) * gamma[j] + beta[j] )
 * (k_norm read as a LayerNorm with weight and bias, biased variance), each
 * formed in double and rounded once.  The exact (unrounded) values are
 * returned when the pointers are non-NULL, and k_cond receives the
 * normalisation's condition scale (|kproj - mu| + mean |kproj|) * rs * |gamma|
 * + |beta| per element. */
void ora_project_keys(const uint16_t *x, const uint16_t *w, const float *gamma,
                      const float *beta, double eps, int64_t T, int hidden, int D,
                      uint16_t *k_out, uint16_t *gate_out, double *kproj_exact,
                      double *k_exact, double *gate_exact, double *k_cond)
{
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; t++) {
        double kp[512];
        double mu = 0.0;
        for (int j = 0; j < 2 * D; j++) {
            double acc = 0.0;
            for (int i = 0; i < hidden; i++)
                acc += ora_bf16_to_double(x[t * hidden + i]) * ora_bf16_to_double(w[(int64_t)j * hidden + i]);
            if (j < D) {
                if (kproj_exact) kproj_exact[t * D + j] = acc;
                kp[j] = ora_bf16_to_double(ora_bf16_from_double(acc));
                mu += kp[j];
            } else {
                if (gate_exact) gate_exact[t * D + j - D] = acc;
                gate_out[t * D + j - D] = ora_bf16_from_double(acc);
            }
        }
        mu /= D;
        double var = 0.0;
        for (int j = 0; j < D; j++) var += (kp[j] - mu) * (kp[j] - mu);
        var /= D;
        const double rs = 1.0 / sqrt(var + eps);
        double mabs = 0.0;
        for (int j = 0; j < D; j++) mabs += fabs(kp[j]);
        mabs /= D;
        for (int j = 0; j < D; j++) {
            const double v = (kp[j] - mu) * rs * (double)gamma[j] + (double)beta[j];
            if (k_exact) k_exact[t * D + j] = v;
            /* condition scale of the normalisation: the terms whose rounding
             * errors a finite-precision evaluation adds up */
            if (k_cond)
                k_cond[t * D + j] = (fabs(kp[j] - mu) + mabs) * rs * fabs((double)gamma[j]) +
                                    fabs((double)beta[j]);
            k_out[t * D + j] = ora_bf16_from_double(v);
        }
    }
}

/* Softmax weights of one pool (for the sum-to-one pin). */
void ora_pool_weights(const uint16_t *gate, const float *ape, int64_t first_token,
                      int D, int kp, double *alpha /* [kp, D] */)
{
    for (int d = 0; d < D; d++) {
        double m = -INFINITY;
        for (int s = 0; s < kp; s++) {
            double a = ora_bf16_to_double(gate[(first_token + s) * D + d]) + (double)ape[s * D + d];
            if (a > m) m = a;
        }
        double z = 0.0;
        for (int s = 0; s < kp; s++) {
            double a = ora_bf16_to_double(gate[(first_token + s) * D + d]) + (double)ape[s * D + d];
            z += exp(a - m);
        }
        for (int s = 0; s < kp; s++) {
            double a = ora_bf16_to_double(gate[(first_token + s) * D + d]) + (double)ape[s * D + d];
            alpha[s * D + d] = exp(a - m) / z;
        }
    }
}

/* ------------------------------------------------------------------ */
/* FP8 input emulation ([MG] section 3: FP32 Hadamard -> BF16 -> E4M3     */
/* with a power-of-two row scale; Testing: Hadamard-matrix reference).  */
/* ------------------------------------------------------------------ */

/* Sylvester-order Hadamard entry: H[i][j] = (-1)^popcount(i & j). */
static int hadamard_sign(int i, int j)
{
    return (__builtin_popcount((unsigned)(i & j)) & 1) ? -1 : 1;
}

/* Fill the explicit n x n Hadamard matrix (entries +-1, unnormalised). */
void ora_hadamard_matrix(int n, double *out)
{
    for (int i = 0; i < n; i++)
        for (int j = 0; j < n; j++) out[i * n + j] = (double)hadamard_sign(i, j);
}

/* Smallest power of two s with amax <= 448 * s; 1 for an all-zero row. */
double ora_pow2_scale(double amax)
{
    if (amax == 0.0) return 1.0;
    int e = -160;
    while (448.0 * ldexp(1.0, e) < amax) e++;
    while (e > -160 && 448.0 * ldexp(1.0, e - 1) >= amax) e--;
    return ldexp(1.0, e);
}

/* One row of n=D values (bf16) -> E4M3 codes and scale:
 *   y = (H x) / sqrt(D)      explicit matrix, double
 *   b = bf16_rne(y)
 *   s = pow2_scale(max |b|)
 *   c = e4m3_rne_satfinite(b / s)
 * y_out / b_out (optional) receive the intermediate values. */
void ora_fp8_rows(const uint16_t *x, int64_t rows, int D, uint8_t *codes, float *scales,
                  double *y_out, uint16_t *b_out)
{
    double *Hm = (double *)malloc(sizeof(double) * D * D);
    ora_hadamard_matrix(D, Hm);
    double norm = 1.0 / sqrt((double)D);
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; r++) {
        double xv[256], bv[256];
        for (int d = 0; d < D; d++) xv[d] = ora_bf16_to_double(x[r * D + d]);
        double amax = 0.0;
        for (int i = 0; i < D; i++) {
            double acc = 0.0;
            for (int j = 0; j < D; j++) acc += Hm[i * D + j] * xv[j];
            double y = acc * norm;
            uint16_t b = ora_bf16_from_double(y);
            if (y_out) y_out[r * D + i] = y;
            if (b_out) b_out[r * D + i] = b;
            bv[i] = ora_bf16_to_double(b);
            if (fabs(bv[i]) > amax) amax = fabs(bv[i]);
        }
        double s = ora_pow2_scale(amax);
        scales[r] = (float)s;
        for (int i = 0; i < D; i++) codes[r * D + i] = ora_e4m3_from_double(bv[i] / s);
    }
    free(Hm);
}

/* ------------------------------------------------------------------ */
/* Scoring and selection.                                               */
/* ------------------------------------------------------------------ */

/* Operands: either bf16 (qs == NULL) or E4M3 codes with per-row scales.
 * q is [T, H, D]; pk is [P, D].  Values are decoded to double once (exact:
 * bf16 -> double, and e4m3 * power-of-two scale -> double). */
typedef struct {
    const void *q;       /* uint16 bf16 or uint8 e4m3 */
    const float *qs;     /* [T, H] scales, NULL for bf16 */
    const float *w;      /* [T, H] */
    const void *pk;      /* uint16 bf16 or uint8 e4m3 */
    const float *pks;    /* [P] scales, NULL for bf16 */
    int fp8;
    int H, D;
    int64_t P;
    double *pkd;         /* decoded pooled keys [P, D] */
} ora_operands;

static double q_elem(const ora_operands *o, int64_t t, int h, int d)
{
    int64_t i = (t * o->H + h) * (int64_t)o->D + d;
    if (!o->fp8) return ora_bf16_to_double(((const uint16_t *)o->q)[i]);
    return ora_e4m3_to_double(((const uint8_t *)o->q)[i]) * (double)o->qs[t * o->H + h];
}

static double pk_elem(const ora_operands *o, int64_t p, int d)
{
    int64_t i = p * (int64_t)o->D + d;
    if (!o->fp8) return ora_bf16_to_double(((const uint16_t *)o->pk)[i]);
    return ora_e4m3_to_double(((const uint8_t *)o->pk)[i]) * (double)o->pks[p];
}

static void ops_init(ora_operands *o, const void *q, const float *qs, const float *w,
                     const void *pk, const float *pks, int fp8, int H, int D, int64_t P)
{
    o->q = q; o->qs = qs; o->w = w; o->pk = pk; o->pks = pks; o->fp8 = fp8;
    o->H = H; o->D = D; o->P = P;
    o->pkd = (double *)malloc(sizeof(double) * (size_t)(P > 0 ? P : 1) * D);
    for (int64_t p = 0; p < P; p++)
        for (int d = 0; d < D; d++) o->pkd[p * D + d] = pk_elem(o, p, d);
}

static void ops_free(ora_operands *o) { free(o->pkd); }

/* qd: decoded q row of token t, [H, D] */
static void decode_q(const ora_operands *o, int64_t t, double *qd)
{
    for (int h = 0; h < o->H; h++)
        for (int d = 0; d < o->D; d++) qd[h * o->D + d] = q_elem(o, t, h, d);
}

/* score[t,p] = sum_h w[t,h] * relu( sum_d q[t,h,d] * pk[p,d] );
 * cond[t,p]  = sum_h |w[t,h]| * relu(...)   (the condition scale used by
 * the parity tolerance). */
static void score_pair(const ora_operands *o, const double *qd, int64_t t, int64_t p,
                       double *score, double *cond)
{
    const double *kd = o->pkd + p * o->D;
    double sc = 0.0, cd = 0.0;
    for (int h = 0; h < o->H; h++) {
        const double *qh = qd + h * o->D;
        double x = 0.0;
        for (int d = 0; d < o->D; d++) x += qh[d] * kd[d];
        double r = x > 0.0 ? x : 0.0;
        double wv = (double)o->w[t * o->H + h];
        sc += wv * r;
        cd += fabs(wv) * r;
    }
    *score = sc;
    *cond = cd;
}

/* Number of complete causal pools for document-local position tau. */
static int64_t n_complete(int64_t tau, int kp) { return (tau + 1) / kp; }

/* Where query rows sit.  Document d's query rows are [cu_q[d], cu_q[d+1]); its
 * i-th query row is at document-local position q_pos[d] + i (q_pos NULL: 0, the
 * plain case where every key token is also a query).  Its keys are the tokens
 * [cu_k[d], cu_k[d+1]) with floor(L_k / kp) complete pools.  A query sees the
 * complete pools j < min(floor((tau+1)/kp), pools of its document). */
typedef struct {
    const int32_t *cu_q;
    const int32_t *q_pos;
    const int32_t *cu_k;
    const int32_t *cu_pools;
    int n_docs;
} ora_layout;

static int layout_row(const ora_layout *L, int64_t t, int64_t *tau, int64_t *nc, int kp)
{
    int d = doc_of_token(L->cu_q, L->n_docs, t);
    if (d < 0) return -1;
    *tau = (L->q_pos ? L->q_pos[d] : 0) + (t - L->cu_q[d]);
    int64_t npool = (int64_t)L->cu_pools[d + 1] - L->cu_pools[d];
    int64_t c = n_complete(*tau, kp);
    *nc = c < npool ? c : npool;
    return d;
}

/* Scores for an explicit list of (query row, global pool) pairs.  A pair
 * whose pool is not a visible complete pool of the row's document gets
 * -inf / 0. */
void ora_score_pairs_at(const void *q, const float *qs, const float *w, const void *pk,
                        const float *pks, int fp8, const int32_t *cu_q, const int32_t *q_pos,
                        const int32_t *cu_k, int n_docs, int H, int D, int kp, int64_t P,
                        const int64_t *rows, const int64_t *pools, int64_t n_pairs,
                        double *score_out, double *cond_out)
{
    ora_operands o;
    ops_init(&o, q, qs, w, pk, pks, fp8, H, D, P);
    int32_t *cu_pools = (int32_t *)malloc(sizeof(int32_t) * (n_docs + 1));
    ora_cu_pools(cu_k, n_docs, kp, cu_pools);
    ora_layout L = {cu_q, q_pos, cu_k, cu_pools, n_docs};
#pragma omp parallel
    {
        double *qd = (double *)malloc(sizeof(double) * H * D);
#pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < n_pairs; i++) {
            int64_t t = rows[i], p = pools[i], tau, nc;
            int doc = layout_row(&L, t, &tau, &nc, kp);
            int64_t j = doc < 0 ? -1 : p - cu_pools[doc];
            if (doc < 0 || j < 0 || j >= nc) {
                score_out[i] = -INFINITY;
                cond_out[i] = 0.0;
                continue;
            }
            decode_q(&o, t, qd);
            score_pair(&o, qd, t, p, &score_out[i], &cond_out[i]);
        }
        free(qd);
    }
    free(cu_pools);
    ops_free(&o);
}

void ora_score_pairs(const void *q, const float *qs, const float *w, const void *pk,
                     const float *pks, int fp8, const int32_t *cu_seqlens, int n_docs,
                     int H, int D, int kp, int64_t P, const int64_t *rows, const int64_t *pools,
                     int64_t n_pairs, double *score_out, double *cond_out)
{
    ora_score_pairs_at(q, qs, w, pk, pks, fp8, cu_seqlens, NULL, cu_seqlens, n_docs, H, D, kp, P,
                       rows, pools, n_pairs, score_out, cond_out);
}

typedef struct {
    double s;
    int64_t p;
} cand;

/* Order: score descending, then pool index ascending. */
static int cand_cmp(const void *a, const void *b)
{
    const cand *x = (const cand *)a, *y = (const cand *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->p < y->p) ? -1 : (x->p > y->p);
}

static int i64_cmp(const void *a, const void *b)
{
    int64_t x = *(const int64_t *)a, y = *(const int64_t *)b;
    return (x > y) - (x < y);
}

/* Selection for a list of query rows ([MG] top-k over index_topk // kpool
 * pools; all pools when fewer are visible).  For each row r:
 *   sel[r, 0..Kp)     selected global pools, ascending, -1 padded
 *   sel_score[r, ..]  their scores (-inf padded)
 *   kth[r], kth_cond[r]  score and condition scale of the Kp-th best pool
 *                     (NaN / 0 when the row selects all of its pools)
 *   n_sel[r]          number of selected pools. */
void ora_select_rows_at(const void *q, const float *qs, const float *w, const void *pk,
                        const float *pks, int fp8, const int32_t *cu_q, const int32_t *q_pos,
                        const int32_t *cu_k, int n_docs, int H, int D, int kp, int64_t P, int Kp,
                        const int64_t *rows, int64_t n_rows, int32_t *sel, double *sel_score,
                        double *kth, double *kth_cond, int32_t *n_sel)
{
    ora_operands o;
    ops_init(&o, q, qs, w, pk, pks, fp8, H, D, P);
    int32_t *cu_pools = (int32_t *)malloc(sizeof(int32_t) * (n_docs + 1));
    ora_cu_pools(cu_k, n_docs, kp, cu_pools);
    ora_layout L = {cu_q, q_pos, cu_k, cu_pools, n_docs};
#pragma omp parallel
    {
        double *qd = (double *)malloc(sizeof(double) * H * D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; r++) {
            int64_t t = rows[r], tau, nc;
            int doc = layout_row(&L, t, &tau, &nc, kp);
            cand *c = (cand *)malloc(sizeof(cand) * (nc > 0 ? nc : 1));
            double *conds = (double *)malloc(sizeof(double) * (nc > 0 ? nc : 1));
            double *scores = (double *)malloc(sizeof(double) * (nc > 0 ? nc : 1));
            decode_q(&o, t, qd);
            for (int64_t j = 0; j < nc; j++) {
                c[j].p = cu_pools[doc] + j;
                score_pair(&o, qd, t, c[j].p, &scores[j], &conds[j]);
                c[j].s = scores[j];
            }
            qsort(c, (size_t)nc, sizeof(cand), cand_cmp);
            int64_t ns = nc < Kp ? nc : Kp;
            n_sel[r] = (int32_t)ns;
            if (nc > Kp) {
                kth[r] = c[Kp - 1].s;
                kth_cond[r] = conds[c[Kp - 1].p - cu_pools[doc]];
            } else {
                kth[r] = NAN;
                kth_cond[r] = 0.0;
            }
            /* ascending pool order for output */
            int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (ns > 0 ? ns : 1));
            for (int64_t i = 0; i < ns; i++) idx[i] = c[i].p;
            qsort(idx, (size_t)ns, sizeof(int64_t), i64_cmp);
            for (int64_t i = 0; i < Kp; i++) {
                if (i < ns) {
                    sel[r * Kp + i] = (int32_t)idx[i];
                    sel_score[r * Kp + i] = scores[idx[i] - cu_pools[doc]];
                } else {
                    sel[r * Kp + i] = -1;
                    sel_score[r * Kp + i] = -INFINITY;
                }
            }
            free(idx);
            free(scores);
            free(conds);
            free(c);
        }
        free(qd);
    }
    free(cu_pools);
    ops_free(&o);
}

void ora_select_rows(const void *q, const float *qs, const float *w, const void *pk,
                     const float *pks, int fp8, const int32_t *cu_seqlens, int n_docs,
                     int H, int D, int kp, int64_t P, int Kp, const int64_t *rows, int64_t n_rows,
                     int32_t *sel, double *sel_score, double *kth, double *kth_cond,
                     int32_t *n_sel)
{
    ora_select_rows_at(q, qs, w, pk, pks, fp8, cu_seqlens, NULL, cu_seqlens, n_docs, H, D, kp, P,
                       Kp, rows, n_rows, sel, sel_score, kth, kth_cond, n_sel);
}

/* Full score rows (small cases): out[r, p] for every global pool p, -inf
 * where p is not a complete causal pool of the row's document. */
void ora_score_rows_full(const void *q, const float *qs, const float *w, const void *pk,
                         const float *pks, int fp8, const int32_t *cu_seqlens, int n_docs,
                         int H, int D, int kp, int64_t P_total, const int64_t *rows,
                         int64_t n_rows, double *out, double *cond_out)
{
    ora_operands o;
    ops_init(&o, q, qs, w, pk, pks, fp8, H, D, P_total);
    int32_t *cu_pools = (int32_t *)malloc(sizeof(int32_t) * (n_docs + 1));
    ora_cu_pools(cu_seqlens, n_docs, kp, cu_pools);
#pragma omp parallel
    {
        double *qd = (double *)malloc(sizeof(double) * H * D);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; r++) {
            int64_t t = rows[r];
            int doc = doc_of_token(cu_seqlens, n_docs, t);
            int64_t tau = t - cu_seqlens[doc];
            int64_t nc = n_complete(tau, kp);
            decode_q(&o, t, qd);
            for (int64_t p = 0; p < P_total; p++) {
                int64_t j = p - cu_pools[doc];
                if (j >= 0 && j < nc) {
                    score_pair(&o, qd, t, p, &out[r * P_total + p], &cond_out[r * P_total + p]);
                } else {
                    out[r * P_total + p] = -INFINITY;
                    cond_out[r * P_total + p] = 0.0;
                }
            }
        }
        free(qd);
    }
    free(cu_pools);
    ops_free(&o);
}

/* ------------------------------------------------------------------ */
/* Expansion + causal tail ([MG] section 3: expand to token indices,     */
/* always_select_tail appends the incomplete causal pool).              */
/* ------------------------------------------------------------------ */

/* Row r (query rows[r]) of width W = Kp*kp + kp - 1:
 *   tokens of each selected pool (ascending pools, kp tokens each), then
 *   the tail tokens t-((tau+1) mod kp)+1 .. t when tail is on and the query's
 *   own pool is incomplete, then -1 padding.  sel holds the pool lists
 *   [n_rows, Kp] (global pools, -1 padded). */
void ora_expand_rows_at(const int32_t *sel, const int32_t *cu_q, const int32_t *q_pos,
                        const int32_t *cu_k, int n_docs, int kp, int Kp, int tail,
                        const int64_t *rows, int64_t n_rows, int32_t *out)
{
    int64_t W = (int64_t)Kp * kp + kp - 1;
    int32_t *cu_pools = (int32_t *)malloc(sizeof(int32_t) * (n_docs + 1));
    ora_cu_pools(cu_k, n_docs, kp, cu_pools);
    ora_layout L = {cu_q, q_pos, cu_k, cu_pools, n_docs};
    for (int64_t r = 0; r < n_rows; r++) {
        int64_t t = rows[r], tau, nc;
        int doc = layout_row(&L, t, &tau, &nc, kp);
        int64_t pos = 0;
        for (int64_t i = 0; i < Kp; i++) {
            int32_t g = sel[r * Kp + i];
            if (g < 0) continue;
            int64_t j = g - cu_pools[doc];
            for (int s = 0; s < kp; s++) out[r * W + pos++] = (int32_t)(cu_k[doc] + j * kp + s);
        }
        if (tail) {
            int64_t rem = (tau + 1) % kp;
            for (int64_t i = rem - 1; i >= 0; i--)
                out[r * W + pos++] = (int32_t)(cu_k[doc] + tau - i);
        }
        while (pos < W) out[r * W + pos++] = -1;
    }
    free(cu_pools);
}

void ora_expand_rows(const int32_t *sel, const int32_t *cu_seqlens, int n_docs, int kp, int Kp,
                     int tail, const int64_t *rows, int64_t n_rows, int32_t *out)
{
    ora_expand_rows_at(sel, cu_seqlens, NULL, cu_seqlens, n_docs, kp, Kp, tail, rows, n_rows, out);
}

/* ------------------------------------------------------------------ */
/* The sparse attention that consumes the indexer's selection: xtuner   */
/* PR "GLM-5.3-Flash F5: NoPE DSA + KPool indexer + clamped SwiGLU",    */
/* Summary (NoPE DeepSeek sparse attention; a SparseMLA forward of the  */
/* FlashMLA kind over the selected token indices) and Megatron-LM PR    */
/* "GLM5.3 Flash", Changes section 3, "NoPE" (the absorbed query has no */
/* positional slice).  In the absorbed form every head of query t       */
/* attends over the latent rows c[j] of the selected tokens, which      */
/* serve as keys and as values:                                         */
/*   s_j   = scale * sum_d q[t, h, d] * c[j, d]      j in tok[r, :], j >= 0 */
/*   lse   = log sum_j exp(s_j)                                         */
/*   o[d]  = sum_j exp(s_j - lse) * c[j, d]                             */
/* in double.  A listed index counts once per listing; -1 entries are   */
/* skipped; a row without tokens gets o = 0 and lse = -inf.             */
/* ------------------------------------------------------------------ */
void ora_sparse_attn(const uint16_t *q, const uint16_t *c, const int32_t *tok, int W, int H,
                     int Dc, double scale, const int64_t *rows, int64_t n_rows, double *o_out,
                     double *lse_out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < n_rows; r++) {
        const int64_t t = rows[r];
        const int32_t *tr = tok + r * (int64_t)W;
        double *s = (double *)malloc(sizeof(double) * (W > 0 ? W : 1));
        for (int h = 0; h < H; h++) {
            const uint16_t *qh = q + (t * H + h) * (int64_t)Dc;
            double m = -INFINITY;
            for (int j = 0; j < W; j++) {
                if (tr[j] < 0) continue;
                double acc = 0.0;
                for (int d = 0; d < Dc; d++)
                    acc += ora_bf16_to_double(qh[d]) * ora_bf16_to_double(c[(int64_t)tr[j] * Dc + d]);
                s[j] = scale * acc;
                if (s[j] > m) m = s[j];
            }
            double *oh = o_out + (r * H + h) * (int64_t)Dc;
            for (int d = 0; d < Dc; d++) oh[d] = 0.0;
            if (m == -INFINITY) {
                lse_out[r * H + h] = -INFINITY;
                continue;
            }
            double z = 0.0;
            for (int j = 0; j < W; j++)
                if (tr[j] >= 0) z += exp(s[j] - m);
            for (int j = 0; j < W; j++) {
                if (tr[j] < 0) continue;
                const double p = exp(s[j] - m) / z;
                for (int d = 0; d < Dc; d++)
                    oh[d] += p * ora_bf16_to_double(c[(int64_t)tr[j] * Dc + d]);
            }
            lse_out[r * H + h] = m + log(z);
        }
        free(s);
    }
}

int ora_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
