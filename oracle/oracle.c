/*
 * oracle.c -- plain fp64 CPU oracle for block-causal and staircase attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this code.  It shares nothing
 * with the CUDA path (no headers, no helpers, no tables) and is never called
 * by the product library.
 *
 * What it computes (the plain definition, no tiling, no online softmax):
 *   - ORL announcement thread (24vids.com mirror), highlight 3: attention for
 *     block-diffusion LMs is *block-causal*: a sequence is cut into blocks of
 *     B tokens; a query sees every key of its own block (bidirectionally) and
 *     every key of all earlier blocks.
 *   - Same thread, Insight 3, and ORL paper card (thelatestinai.com),
 *     Figure 3 caption: training replays packed trajectories with a
 *     *staircase* kernel: after a clean prefix of P tokens sit K copies of
 *     the active block (one per denoising step); every copy sees the prefix
 *     and itself only.
 *   - The attention itself is ordinary scaled-dot-product softmax attention
 *     (the thread compares it with FlashAttention), with the natural-log
 *     log-sum-exp of each query row kept for the backward pass, and the
 *     textbook softmax-attention gradients.
 *
 * Readings taken where the pages are silent (each one listed in the design
 * notes of the repository):
 *   - staircase prefix rows are queries too and are block-causal inside the
 *     prefix (block size = copy length); they never see copies;
 *   - when a sequence has fewer queries than keys (a decode step), query row i
 *     sits at key position p = i + (Lk - Lq) (aligned to the end);
 *   - GQA: query head h reads KV head floor(h / G), G = Hq / Hkv;
 *   - LSE is the natural logarithm;
 *   - several active blocks per trajectory (the announcement thread's
 *     "irregular trajectories", Insight 3): the copies of each active block
 *     form a group after the prefix, and a group's copies see the clean keys
 *     before their block's position (the prompt and the clean blocks before
 *     it) and themselves only -- the multi-block staircase below.
 *
 * Layout of every array handed in (one sequence at a time, row-major fp64):
 *   Q, dO, O, dQ : [Lq][Hq][d]     K, V, dK, dV : [Lk][Hkv][d]
 *   LSE          : [Hq][Lq]
 *
 * The parallel loops only split independent rows / columns across threads;
 * each row is still computed by the plain definition.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BLOCK_CAUSAL 0
#define ORACLE_STAIRCASE 1
#define ORACLE_STAIRCASE_MULTI 2

/* A sequence's mask.  The multi-block staircase (several active blocks per
 * trajectory, the "irregular trajectories" of the announcement thread,
 * Insight 3) generalises the staircase: after the clean prefix [0, P) come
 * n_groups groups of copies; group g holds copies[g] copies of one active
 * block (B tokens each), and its copies see the clean keys [0, visible[g])
 * -- the prompt and the clean blocks before that active block -- and their
 * own copy only.  The staircase is one group with visible[0] = P. */
typedef struct {
    int kind, B, P;
    int n_groups;
    const int32_t *copies;
    const int32_t *visible;
} oracle_mask_t;

/* allowed(i, j): may local query row i attend to local key j?
 * Block-causal (announcement thread, highlight 3):
 *     floor(j / B) <= floor(p / B),                p = i + (Lk - Lq).
 * Staircase (announcement thread, Insight 3; paper card, Figure 3):
 *     row in the prefix (p < P):  j < P  and  floor(j / B) <= floor(p / B)
 *     row in copy c = floor((p - P) / B):  j < P  or  floor((j - P) / B) == c */
static int allowed_m(const oracle_mask_t *mk, int Lq, int Lk, int i, int j)
{
    const int B = mk->B, P = mk->P;
    if (i < 0 || i >= Lq || j < 0 || j >= Lk || B <= 0) return 0;
    long p = (long)i + (long)(Lk - Lq);
    if (mk->kind == ORACLE_BLOCK_CAUSAL) return (j / B) <= (p / B);
    if (p < P) return j < P && (j / B) <= (p / B);
    if (mk->kind == ORACLE_STAIRCASE) {
        if (j < P) return 1;
        return ((long)j - P) / B == (p - P) / B;
    }
    /* multi-block staircase: find the row's group, then its own copy */
    long start = P;
    for (int g = 0; g < mk->n_groups; ++g) {
        const long span = (long)mk->copies[g] * B;
        if (p < start + span) {
            const long c0 = start + ((p - start) / B) * B;
            return j < mk->visible[g] || (j >= c0 && j < c0 + B);
        }
        start += span;
    }
    return 0;
}

static oracle_mask_t simple_mask(int kind, int B, int P)
{
    oracle_mask_t mk = {kind, B, P, 0, NULL, NULL};
    return mk;
}

static oracle_mask_t multi_mask(int B, int P, int n_groups, const int32_t *copies,
                                const int32_t *visible)
{
    oracle_mask_t mk = {ORACLE_STAIRCASE_MULTI, B, P, n_groups, copies, visible};
    return mk;
}

int oracle_allowed(int kind, int B, int P, int Lq, int Lk, int i, int j)
{
    const oracle_mask_t mk = simple_mask(kind, B, P);
    return allowed_m(&mk, Lq, Lk, i, j);
}

int oracle_allowed_multi(int B, int P, int n_groups, const int32_t *copies,
                         const int32_t *visible, int L, int i, int j)
{
    const oracle_mask_t mk = multi_mask(B, P, n_groups, copies, visible);
    return allowed_m(&mk, L, L, i, j);
}

static void mask_m(const oracle_mask_t *mk, int Lq, int Lk, uint8_t *M)
{
    for (int i = 0; i < Lq; ++i)
        for (int j = 0; j < Lk; ++j)
            M[(size_t)i * Lk + j] = (uint8_t)allowed_m(mk, Lq, Lk, i, j);
}

/* The explicit mask of one sequence, M[i*Lk + j] in {0,1}. */
void oracle_mask(int kind, int B, int P, int Lq, int Lk, uint8_t *M)
{
    const oracle_mask_t mk = simple_mask(kind, B, P);
    mask_m(&mk, Lq, Lk, M);
}

void oracle_mask_multi(int B, int P, int n_groups, const int32_t *copies, const int32_t *visible,
                       int L, uint8_t *M)
{
    const oracle_mask_t mk = multi_mask(B, P, n_groups, copies, visible);
    mask_m(&mk, L, L, M);
}

static long long count_pairs_m(const oracle_mask_t *mk, int Lq, int Lk)
{
    long long n = 0;
    for (int i = 0; i < Lq; ++i)
        for (int j = 0; j < Lk; ++j)
            n += allowed_m(mk, Lq, Lk, i, j);
    return n;
}

/* Number of allowed (i, j) pairs of one sequence (per head). */
long long oracle_count_pairs(int kind, int B, int P, int Lq, int Lk)
{
    const oracle_mask_t mk = simple_mask(kind, B, P);
    return count_pairs_m(&mk, Lq, Lk);
}

long long oracle_count_pairs_multi(int B, int P, int n_groups, const int32_t *copies,
                                   const int32_t *visible, int L)
{
    const oracle_mask_t mk = multi_mask(B, P, n_groups, copies, visible);
    return count_pairs_m(&mk, L, L);
}

static int max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

int oracle_num_threads(void) { return max_threads(); }

/* One query row of one head: fill mrow (mask row), S (scores, -inf where
 * masked), P (probabilities), and return LSE.  O row (d values) written. */
static double row_forward(const oracle_mask_t *mk, int Lq, int Lk, int Hq, int Hkv, int d,
                          double scale, const double *Q, const double *K, const double *V,
                          int h, int i, uint8_t *mrow, double *S, double *Pr, double *Orow)
{
    const int G = Hq / Hkv;
    const int kvh = h / G;
    const double *q = Q + ((size_t)i * Hq + h) * d;
    for (int j = 0; j < Lk; ++j) mrow[j] = (uint8_t)allowed_m(mk, Lq, Lk, i, j);
    /* S_ij = scale * <Q_i, K_j>, -inf where not allowed */
    double m = -INFINITY;
    for (int j = 0; j < Lk; ++j) {
        if (!mrow[j]) { S[j] = -INFINITY; continue; }
        const double *k = K + ((size_t)j * Hkv + kvh) * d;
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += q[c] * k[c];
        S[j] = scale * acc;
        if (S[j] > m) m = S[j];
    }
    /* P = softmax_j(S); LSE = ln sum_j exp(S_ij) */
    double Z = 0.0;
    for (int j = 0; j < Lk; ++j) {
        Pr[j] = mrow[j] ? exp(S[j] - m) : 0.0;
        Z += Pr[j];
    }
    for (int j = 0; j < Lk; ++j) Pr[j] /= Z;
    /* O_i = sum_j P_ij V_j */
    for (int c = 0; c < d; ++c) Orow[c] = 0.0;
    for (int j = 0; j < Lk; ++j) {
        if (!mrow[j]) continue;
        const double *v = V + ((size_t)j * Hkv + kvh) * d;
        for (int c = 0; c < d; ++c) Orow[c] += Pr[j] * v[c];
    }
    return m + log(Z);
}

/* Forward for one sequence, query heads [h_lo, h_hi).  rows == NULL: every
 * row, outputs indexed by row; else only rows[0..nrows), outputs indexed by
 * position in that list (O: [nrows][Hq][d], LSE: [Hq][nrows]). */
static void fwd_seq_m(const oracle_mask_t *mk, int Lq, int Lk, int Hq, int Hkv, int d,
                      double scale, const double *Q, const double *K, const double *V, int h_lo,
                      int h_hi, const int32_t *rows, int nrows, double *O, double *LSE)
{
    const int nr = rows ? nrows : Lq;
    const long ntask = (long)(h_hi - h_lo) * nr;
#pragma omp parallel
    {
        uint8_t *mrow = (uint8_t *)malloc((size_t)Lk + 1);
        double *S = (double *)malloc(sizeof(double) * ((size_t)Lk + 1));
        double *Pr = (double *)malloc(sizeof(double) * ((size_t)Lk + 1));
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < ntask; ++t) {
            const int h = h_lo + (int)(t / nr);
            const int r = (int)(t % nr);
            const int i = rows ? rows[r] : r;
            double *Orow = O + ((size_t)r * Hq + h) * d;
            LSE[(size_t)h * nr + r] = row_forward(mk, Lq, Lk, Hq, Hkv, d, scale, Q, K, V, h, i,
                                                  mrow, S, Pr, Orow);
        }
        free(mrow);
        free(S);
        free(Pr);
    }
}

void oracle_fwd_seq(int kind, int B, int P, int Lq, int Lk, int Hq, int Hkv, int d, double scale,
                    const double *Q, const double *K, const double *V, int h_lo, int h_hi,
                    const int32_t *rows, int nrows, double *O, double *LSE)
{
    const oracle_mask_t mk = simple_mask(kind, B, P);
    fwd_seq_m(&mk, Lq, Lk, Hq, Hkv, d, scale, Q, K, V, h_lo, h_hi, rows, nrows, O, LSE);
}

void oracle_fwd_seq_multi(int B, int P, int n_groups, const int32_t *copies,
                          const int32_t *visible, int L, int Hq, int Hkv, int d, double scale,
                          const double *Q, const double *K, const double *V, int h_lo, int h_hi,
                          const int32_t *rows, int nrows, double *O, double *LSE)
{
    const oracle_mask_t mk = multi_mask(B, P, n_groups, copies, visible);
    fwd_seq_m(&mk, L, L, Hq, Hkv, d, scale, Q, K, V, h_lo, h_hi, rows, nrows, O, LSE);
}

/* Backward for one sequence, KV heads [kvh_lo, kvh_hi) (and their G query
 * heads).  Textbook softmax-attention gradients:
 *   dV = P^T dO;  dP = dO V^T;  D_i = sum_c dO_ic O_ic;  dS = P o (dP - D);
 *   dQ = scale dS K;  dK = scale dS^T Q;  dK, dV summed over the G query
 *   heads that share a KV head.
 * qrows (or NULL = all Lq rows) selects the dQ rows computed; dQ indexed by
 * position in that list: [nq][Hq][d].  krows (or NULL = all Lk keys) selects
 * the dK/dV rows computed: [nk][Hkv][d].  Only heads in range are written.
 * P_ij for a key column is exp(S_ij - LSE_i), the same softmax. */
static void bwd_seq_m(const oracle_mask_t *mk, int Lq, int Lk, int Hq, int Hkv, int d,
                      double scale, const double *Q, const double *K, const double *V,
                      const double *dO, int kvh_lo, int kvh_hi, const int32_t *qrows, int nq,
                      const int32_t *krows, int nk, double *dQ, double *dK, double *dV)
{
    const int G = Hq / Hkv;
    const int h_lo = kvh_lo * G, h_hi = kvh_hi * G;
    const int nqr = qrows ? nq : Lq;
    const int nkr = krows ? nk : Lk;

    /* Which query rows are needed: the dQ rows, and every row that sees one of
     * the requested keys. */
    uint8_t *need = (uint8_t *)calloc((size_t)Lq + 1, 1);
    for (int r = 0; r < nqr; ++r) need[qrows ? qrows[r] : r] = 1;
#pragma omp parallel for schedule(static)
    for (int i = 0; i < Lq; ++i) {
        if (need[i]) continue;
        for (int r = 0; r < nkr; ++r)
            if (allowed_m(mk, Lq, Lk, i, krows ? krows[r] : r)) { need[i] = 1; break; }
    }
    int32_t *qpos = (int32_t *)malloc(sizeof(int32_t) * ((size_t)Lq + 1));
    for (int i = 0; i < Lq; ++i) qpos[i] = -1;
    if (qrows)
        for (int r = 0; r < nq; ++r) qpos[qrows[r]] = r;
    else
        for (int i = 0; i < Lq; ++i) qpos[i] = i;

    /* Per needed row and head: LSE_i, D_i, and (for dQ rows) dQ_i. */
    double *LSE = (double *)malloc(sizeof(double) * ((size_t)Lq * Hq + 1));
    double *Dv = (double *)malloc(sizeof(double) * ((size_t)Lq * Hq + 1));
    const long ntask = (long)(h_hi - h_lo) * Lq;
#pragma omp parallel
    {
        uint8_t *mrow = (uint8_t *)malloc((size_t)Lk + 1);
        double *S = (double *)malloc(sizeof(double) * ((size_t)Lk + 1));
        double *Pr = (double *)malloc(sizeof(double) * ((size_t)Lk + 1));
        double *Orow = (double *)malloc(sizeof(double) * ((size_t)d + 1));
#pragma omp for schedule(dynamic, 4)
        for (long t = 0; t < ntask; ++t) {
            const int h = h_lo + (int)(t / Lq);
            const int i = (int)(t % Lq);
            if (!need[i]) continue;
            const int kvh = h / G;
            const double lse = row_forward(mk, Lq, Lk, Hq, Hkv, d, scale, Q, K, V, h, i, mrow, S,
                                           Pr, Orow);
            const double *dout = dO + ((size_t)i * Hq + h) * d;
            double D = 0.0;
            for (int c = 0; c < d; ++c) D += dout[c] * Orow[c];
            LSE[(size_t)i * Hq + h] = lse;
            Dv[(size_t)i * Hq + h] = D;
            if (qpos[i] < 0) continue;
            double *dq = dQ + ((size_t)qpos[i] * Hq + h) * d;
            for (int c = 0; c < d; ++c) dq[c] = 0.0;
            for (int j = 0; j < Lk; ++j) {
                if (!mrow[j]) continue;
                const double *v = V + ((size_t)j * Hkv + kvh) * d;
                const double *k = K + ((size_t)j * Hkv + kvh) * d;
                double dp = 0.0;
                for (int c = 0; c < d; ++c) dp += dout[c] * v[c];
                const double ds = Pr[j] * (dp - D);
                for (int c = 0; c < d; ++c) dq[c] += scale * ds * k[c];
            }
        }
        free(mrow);
        free(S);
        free(Pr);
        free(Orow);
    }

    /* Per requested key and KV head: dK_j, dV_j over every row and head of
     * the group that sees key j. */
    const long ktask = (long)(kvh_hi - kvh_lo) * nkr;
#pragma omp parallel for schedule(dynamic, 4)
    for (long t = 0; t < ktask; ++t) {
        const int kvh = kvh_lo + (int)(t / nkr);
        const int r = (int)(t % nkr);
        const int j = krows ? krows[r] : r;
        double *dk = dK + ((size_t)r * Hkv + kvh) * d;
        double *dv = dV + ((size_t)r * Hkv + kvh) * d;
        for (int c = 0; c < d; ++c) { dk[c] = 0.0; dv[c] = 0.0; }
        const double *k = K + ((size_t)j * Hkv + kvh) * d;
        const double *v = V + ((size_t)j * Hkv + kvh) * d;
        for (int h = kvh * G; h < (kvh + 1) * G; ++h) {
            for (int i = 0; i < Lq; ++i) {
                if (!allowed_m(mk, Lq, Lk, i, j)) continue;
                const double *q = Q + ((size_t)i * Hq + h) * d;
                const double *dout = dO + ((size_t)i * Hq + h) * d;
                double s = 0.0, dp = 0.0;
                for (int c = 0; c < d; ++c) { s += q[c] * k[c]; dp += dout[c] * v[c]; }
                const double p = exp(scale * s - LSE[(size_t)i * Hq + h]);
                const double ds = p * (dp - Dv[(size_t)i * Hq + h]);
                for (int c = 0; c < d; ++c) {
                    dv[c] += p * dout[c];
                    dk[c] += scale * ds * q[c];
                }
            }
        }
    }
    free(need);
    free(qpos);
    free(LSE);
    free(Dv);
}

void oracle_bwd_seq(int kind, int B, int P, int Lq, int Lk, int Hq, int Hkv, int d, double scale,
                    const double *Q, const double *K, const double *V, const double *dO,
                    int kvh_lo, int kvh_hi, const int32_t *qrows, int nq, const int32_t *krows,
                    int nk, double *dQ, double *dK, double *dV)
{
    const oracle_mask_t mk = simple_mask(kind, B, P);
    bwd_seq_m(&mk, Lq, Lk, Hq, Hkv, d, scale, Q, K, V, dO, kvh_lo, kvh_hi, qrows, nq, krows, nk,
              dQ, dK, dV);
}

void oracle_bwd_seq_multi(int B, int P, int n_groups, const int32_t *copies,
                          const int32_t *visible, int L, int Hq, int Hkv, int d, double scale,
                          const double *Q, const double *K, const double *V, const double *dO,
                          int kvh_lo, int kvh_hi, const int32_t *qrows, int nq,
                          const int32_t *krows, int nk, double *dQ, double *dK, double *dV)
{
    const oracle_mask_t mk = multi_mask(B, P, n_groups, copies, visible);
    bwd_seq_m(&mk, L, L, Hq, Hkv, d, scale, Q, K, V, dO, kvh_lo, kvh_hi, qrows, nq, krows, nk, dQ,
              dK, dV);
}

/* ------------------------------------------------------------------------
 * FP8 E4M3 (OCP 8-bit floating point, E4M3 variant), the KV-cache format of
 * the decode engine on the ORL paper card (Table 11 caption: the NVFP4
 * configurations use an FP8 KV cache).  Bit layout s eeee mmm, exponent bias
 * 7; exponent field 0 holds the subnormals m * 2^-9; field 1..15 holds
 * (1 + m/8) * 2^(e-7), except s 1111 111, which is NaN; there are no
 * infinities, so the largest finite magnitude is 1.75 * 2^8 = 448.
 * Quantising a value: round to the nearest representable magnitude, ties to
 * the even code; a magnitude that rounds above 448 saturates to 448; NaN
 * stays NaN.
 * ---------------------------------------------------------------------- */
double oracle_e4m3_decode(unsigned char c)
{
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

unsigned char oracle_e4m3_encode(float x)
{
    const unsigned char sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (unsigned char)(sign | 0x7F);
    const double a = fabs((double)x);
    /* spacing of the representable magnitudes around a: 2^-9 below 2^-6
     * (subnormals and the first binade), else 2^(floor(log2 a) - 3) */
    double q;
    if (a < ldexp(1.0, -6)) {
        q = ldexp(1.0, -9);
    } else {
        int ex;
        frexp(a, &ex); /* a = f * 2^ex, f in [0.5, 1): floor(log2 a) = ex - 1 */
        q = ldexp(1.0, ex - 1 - 3);
    }
    /* a / q is exact (q is a power of two); rint rounds ties to even */
    double v = rint(a / q) * q;
    if (v > 448.0) v = 448.0;
    if (v == 0.0) return sign;
    if (v < ldexp(1.0, -6)) return (unsigned char)(sign | (int)(v / ldexp(1.0, -9)));
    int ex;
    frexp(v, &ex);
    const int e = ex - 1 + 7;                             /* biased exponent */
    const int m = (int)((v / ldexp(1.0, ex - 1) - 1.0) * 8.0); /* exact */
    return (unsigned char)(sign | (e << 3) | m);
}

void oracle_e4m3_encode_array(const float *x, long n, unsigned char *out)
{
    for (long i = 0; i < n; ++i) out[i] = oracle_e4m3_encode(x[i]);
}

void oracle_e4m3_decode_array(const unsigned char *c, long n, double *out)
{
    for (long i = 0; i < n; ++i) out[i] = oracle_e4m3_decode(c[i]);
}
