/*
 * linattn.c -- plain, sequential float64 reference for the causal
 * cos-re-weighted linear-attention scan (cosFormer).
 *
 * TEST INFRASTRUCTURE ONLY, like oracle.c: the tests, the package smoke check
 * and the benchmark's CPU-baseline leg are its only callers; it shares no
 * code, header, table or helper with the CUDA library, and the library never
 * calls it.
 *
 * What it computes (per head, queries Q_1..Q_N, keys K_1..K_N, values
 * V_1..V_N in R^d, a re-weighting length M > 0, positions i, j = 1..N):
 *
 *     Q'_i = ReLU(Q_i),  K'_j = ReLU(K_j)
 *     s_ij = (Q'_i . K'_j) cos(pi/2 * (i - j) / M)
 *     o_i  = sum_{j<=i} s_ij V_j / sum_{j<=i} s_ij      (0 where the sum is 0)
 *
 * Source: LG AI Research blog "[ICLR 2022] Part 1: Efficient Transformer",
 * section "cosFormer" and its equations: the similarity is the dot product of the ReLU feature maps of
 * query and key (the non-negative decomposable map the section settles on),
 * re-weighted by cos(pi/2 (i - j) / M) so that near positions weigh more.
 * By the cosine sum formula the weight splits into
 * cos(pi i/2M) cos(pi j/2M) + sin(pi i/2M) sin(pi j/2M), so with
 * Q^cos_i = Q'_i cos(pi i/2M), Q^sin_i = Q'_i sin(pi i/2M) and the same for K
 * the output is
 *
 *     o_i = (Q^cos_i S^cos_i + Q^sin_i S^sin_i) / (Q^cos_i z^cos_i + Q^sin_i z^sin_i)
 *
 * with S^cos_i = sum_j (K^cos_j)^T V_j (a d x d matrix), z^cos_i = sum_j K^cos_j
 * (a d vector), and likewise for sin.  The section writes the sums over all
 * j = 1..N (every query sees every key); the prefix form here sums j <= i,
 * which makes S and z running sums over the sequence: a prefix scan whose
 * state is (S^cos, S^sin, z^cos, z^sin).  Readings: the sums run over
 * j <= i (causal); M is a caller argument (cosFormer takes the sequence
 * length); a zero denominator (no key shares a positive coordinate with the
 * query) gives o_i = 0.
 *
 * Inputs are float32 arrays (bfloat16 data is widened first, exactly); all
 * arithmetic is double, cos/sin are libm's.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double relu_d(float x) { return x > 0.0f ? (double)x : 0.0; }

static double half_pi(void) { return 2.0 * atan(1.0); }

/* The definition written out: for every i, the weighted average over      */
/* j <= i with the weight s_ij computed directly from (i - j).  O(N^2 d).   */
void oracle_la_bruteforce(const float *Q, const float *K, const float *V,
                          int64_t N, int64_t d, double M, double *O)
{
    const double hp = half_pi();
    double *num = (double *)malloc((size_t)(d > 0 ? d : 1) * sizeof(double));
    for (int64_t i = 0; i < N; ++i) {
        double den = 0.0;
        for (int64_t c = 0; c < d; ++c) num[c] = 0.0;
        for (int64_t j = 0; j <= i; ++j) {
            double dot = 0.0;
            for (int64_t c = 0; c < d; ++c)
                dot += relu_d(Q[i * d + c]) * relu_d(K[j * d + c]);
            double s = dot * cos(hp * (double)(i - j) / M);
            den += s;
            for (int64_t c = 0; c < d; ++c) num[c] += s * (double)V[j * d + c];
        }
        for (int64_t c = 0; c < d; ++c) O[i * d + c] = den != 0.0 ? num[c] / den : 0.0;
    }
    free(num);
}

/* The decomposed form as a prefix scan, token by token.  State layout:     */
/* Sc, Ss [d, d] row-major (row = key coordinate, column = value            */
/* coordinate), zc, zs [d].  If init_* are non-NULL the scan starts from    */
/* that state and positions continue from pos0 (position of the first token */
/* is pos0 + 1); otherwise from zero and pos0 = 0.  O (may be NULL) gets    */
/* every o_i; the final state is written to the *_out arrays (may be NULL). */
int oracle_la_scan(const float *Q, const float *K, const float *V, int64_t N, int64_t d,
                   double M, int64_t pos0, const double *init_Sc, const double *init_Ss,
                   const double *init_zc, const double *init_zs, double *O,
                   double *Sc_out, double *Ss_out, double *zc_out, double *zs_out)
{
    const double hp = half_pi();
    size_t dd = (size_t)(d > 0 ? d : 1);
    double *Sc = (double *)calloc(dd * dd, sizeof(double));
    double *Ss = (double *)calloc(dd * dd, sizeof(double));
    double *zc = (double *)calloc(dd, sizeof(double));
    double *zs = (double *)calloc(dd, sizeof(double));
    double *kp = (double *)malloc(dd * sizeof(double));
    double *qp = (double *)malloc(dd * sizeof(double));
    if (!Sc || !Ss || !zc || !zs || !kp || !qp) {
        free(Sc); free(Ss); free(zc); free(zs); free(kp); free(qp);
        return 1;
    }
    if (init_Sc) memcpy(Sc, init_Sc, (size_t)(d * d) * sizeof(double));
    if (init_Ss) memcpy(Ss, init_Ss, (size_t)(d * d) * sizeof(double));
    if (init_zc) memcpy(zc, init_zc, (size_t)d * sizeof(double));
    if (init_zs) memcpy(zs, init_zs, (size_t)d * sizeof(double));
    for (int64_t t = 0; t < N; ++t) {
        double pos = (double)(pos0 + t + 1);          /* 1-based position */
        double ct = cos(hp * pos / M), st = sin(hp * pos / M);
        /* add token t's key/value to the running sums */
        for (int64_t a = 0; a < d; ++a) kp[a] = relu_d(K[t * d + a]);
        for (int64_t a = 0; a < d; ++a) {
            double kc = kp[a] * ct, ks = kp[a] * st;
            zc[a] += kc;
            zs[a] += ks;
            for (int64_t b = 0; b < d; ++b) {
                double v = (double)V[t * d + b];
                Sc[a * d + b] += kc * v;
                Ss[a * d + b] += ks * v;
            }
        }
        if (!O) continue;
        /* read out with the query of the same position */
        for (int64_t a = 0; a < d; ++a) qp[a] = relu_d(Q[t * d + a]);
        double den = 0.0;
        for (int64_t a = 0; a < d; ++a) den += qp[a] * ct * zc[a] + qp[a] * st * zs[a];
        for (int64_t b = 0; b < d; ++b) {
            double num = 0.0;
            for (int64_t a = 0; a < d; ++a)
                num += qp[a] * ct * Sc[a * d + b] + qp[a] * st * Ss[a * d + b];
            O[t * d + b] = den != 0.0 ? num / den : 0.0;
        }
    }
    if (Sc_out) memcpy(Sc_out, Sc, (size_t)(d * d) * sizeof(double));
    if (Ss_out) memcpy(Ss_out, Ss, (size_t)(d * d) * sizeof(double));
    if (zc_out) memcpy(zc_out, zc, (size_t)d * sizeof(double));
    if (zs_out) memcpy(zs_out, zs, (size_t)d * sizeof(double));
    free(Sc); free(Ss); free(zc); free(zs); free(kp); free(qp);
    return 0;
}
