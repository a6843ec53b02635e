/*
 * oracle.c -- plain, sequential float64 reference for the softmax-attention
 * prefix scan.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the oracle that the CUDA library is
 * checked against.  Only the tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load or call it.  It shares no code,
 * header, table or helper with the CUDA library, and the library never calls
 * it.  It is deliberately slow and unblocked: one head at a time, one token
 * at a time, in the order the method is written.
 *
 * What it computes (per head, for a query q in R^d, keys k_1..k_N and values
 * v_1..v_N in R^d):
 *
 *     s_i = q . k_i                                    (unscaled dot product)
 *     o_t = sum_{i<=t} exp(s_i) v_i / sum_{i<=t} exp(s_i)   for t = 1..N
 *
 * Sources:
 *  - "Self-attention Does Not Need O(n^2) Memory" review, section 2
 *    "Algorithm": the score is the dot product of the query with key i; the
 *    running vector sum v* and scalar sum s* start at zero, each (k_i, v_i)
 *    pair adds v_i e^{s_i} and e^{s_i}, and the result is v* divided by s*
 *    once the keys are consumed (the softmax division moved to the end).
 *  - "Attention as an RNN" review, "Proposed method": attention is a
 *    many-to-one RNN; its many-to-many output (every prefix t) is what the
 *    parallel prefix scan computes, exactly, not approximately; the state has
 *    a constant size and is updated one token at a time.
 *  - Section 3 "Numerical Stability" of the memory-efficient-attention review
 *    names the need for a stabilising trick but its body is missing.  The
 *    reading taken here is the standard one: carry the running maximum m of
 *    the scores and keep the sums rescaled by exp(-m), so the state is
 *    (m, u, w) = (max_i s_i, sum_i exp(s_i - m) v_i, sum_i exp(s_i - m)).
 *    When a new maximum M appears the old sums are multiplied by exp(m - M).
 *
 * Inputs are float32 arrays (bfloat16 inputs are widened to float32 by the
 * caller, which is exact); everything is computed in double.  exp() is the C
 * library's double exp.  Build: gcc -O2 (no -ffast-math), see build.py.
 *
 * Parity pins: every function here is checked by tests/test_oracle.py
 * against brute force, closed forms, a hand-derived rational worked example,
 * invariances and a long-double run (see that file's header).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Score: s_t = sum_j q[j] * k_t[j], j ascending, in double.                 */
/* ("Self-attention Does Not Need O(n^2) Memory" review, section 2.)        */
/* ------------------------------------------------------------------------ */
void oracle_scores(const float *q, const float *K, int64_t N, int64_t d,
                   double *s)
{
    for (int64_t t = 0; t < N; ++t) {
        double acc = 0.0;
        for (int64_t j = 0; j < d; ++j)
            acc += (double)q[j] * (double)K[t * d + j];
        s[t] = acc;
    }
}

/* ------------------------------------------------------------------------ */
/* The sequential recurrence given the scores.                              */
/*                                                                          */
/* State (m, u[d], w); identity (-inf, 0, 0).  For each token t in order:   */
/*     M = max(m, s_t)                                                      */
/*     a = exp(m - M)   (0 when m is -inf: the empty prefix)                */
/*     b = exp(s_t - M)                                                     */
/*     u = a*u + b*v_t ;  w = a*w + b ;  m = M                              */
/*     o_t = u / w        (inclusive: token t is part of its own prefix)    */
/*                                                                          */
/* init_m/init_u/init_w give a starting state (NULL = identity); this is    */
/* the constant-size RNN state of the Aaren review's "Proposed method",     */
/* so a stream can be continued from a saved state.                          */
/* O may be NULL (only the final state is returned).                        */
/* ------------------------------------------------------------------------ */
void oracle_scan_scores(const double *s, const float *V, int64_t N, int64_t d,
                        const double *init_m, const double *init_u,
                        const double *init_w, double *O, double *m_out,
                        double *u_out, double *w_out)
{
    double m = -INFINITY, w = 0.0;
    double *u = (double *)calloc((size_t)(d > 0 ? d : 1), sizeof(double));
    if (init_m && init_u && init_w) {
        m = *init_m;
        w = *init_w;
        for (int64_t j = 0; j < d; ++j) u[j] = init_u[j];
    }
    for (int64_t t = 0; t < N; ++t) {
        double M = (s[t] > m) ? s[t] : m;
        double a = (m == -INFINITY) ? 0.0 : exp(m - M);
        double b = exp(s[t] - M);
        for (int64_t j = 0; j < d; ++j)
            u[j] = a * u[j] + b * (double)V[t * d + j];
        w = a * w + b;
        m = M;
        if (O)
            for (int64_t j = 0; j < d; ++j) O[t * d + j] = u[j] / w;
    }
    if (m_out) *m_out = m;
    if (w_out) *w_out = w;
    if (u_out)
        for (int64_t j = 0; j < d; ++j) u_out[j] = u[j];
    free(u);
}

/* Scores then recurrence, one head: the whole path in one call.  The scores */
/* of a head are held in a scratch array of N doubles.                       */
int oracle_scan(const float *q, const float *K, const float *V, int64_t N,
                int64_t d, const double *init_m, const double *init_u,
                const double *init_w, double *O, double *m_out, double *u_out,
                double *w_out)
{
    double *s = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!s) return 1;
    oracle_scores(q, K, N, d, s);
    oracle_scan_scores(s, V, N, d, init_m, init_u, init_w, O, m_out, u_out,
                       w_out);
    free(s);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Brute force: for every prefix t, the textbook softmax over s_1..s_t,     */
/* weights applied to v_1..v_t.  O(N^2 d); small N only.  This is the plain */
/* definition of the many-to-many output, independent of the recurrence.   */
/* ------------------------------------------------------------------------ */
void oracle_bruteforce(const double *s, const float *V, int64_t N, int64_t d,
                       double *O)
{
    for (int64_t t = 0; t < N; ++t) {
        double mx = s[0];
        for (int64_t i = 1; i <= t; ++i)
            if (s[i] > mx) mx = s[i];
        double den = 0.0;
        for (int64_t i = 0; i <= t; ++i) den += exp(s[i] - mx);
        for (int64_t j = 0; j < d; ++j) {
            double num = 0.0;
            for (int64_t i = 0; i <= t; ++i)
                num += exp(s[i] - mx) * (double)V[i * d + j];
            O[t * d + j] = num / den;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* The associative operator on states.                                      */
/*   (m_a,u_a,w_a) (+) (m_b,u_b,w_b) = (M, e^{m_a-M} u_a + e^{m_b-M} u_b,    */
/*                                          e^{m_a-M} w_a + e^{m_b-M} w_b)  */
/* with M = max(m_a, m_b); the identity (-inf, 0, 0) is returned unchanged  */
/* when both sides are the identity (exp(-inf - -inf) would be NaN).        */
/* ------------------------------------------------------------------------ */
void oracle_combine(double m_a, const double *u_a, double w_a, double m_b,
                    const double *u_b, double w_b, int64_t d, double *m_o,
                    double *u_o, double *w_o)
{
    double M = (m_a > m_b) ? m_a : m_b;
    if (M == -INFINITY) {
        *m_o = -INFINITY;
        *w_o = 0.0;
        for (int64_t j = 0; j < d; ++j) u_o[j] = 0.0;
        return;
    }
    double ea = (m_a == -INFINITY) ? 0.0 : exp(m_a - M);
    double eb = (m_b == -INFINITY) ? 0.0 : exp(m_b - M);
    for (int64_t j = 0; j < d; ++j) u_o[j] = ea * u_a[j] + eb * u_b[j];
    *w_o = ea * w_a + eb * w_b;
    *m_o = M;
}

/* ------------------------------------------------------------------------ */
/* Hillis-Steele inclusive scan of the operator above over the leaves       */
/* (s_t, v_t, 1): ceil(log2 N) rounds; in the round with offset k every     */
/* position t >= k becomes x[t-k] (+) x[t], from a second buffer so a round */
/* reads only the previous round's values.  O(N log N d).  This is the      */
/* parallel prefix scan the Aaren review names, run serially; it must give  */
/* the same outputs as the sequential recurrence.                           */
/* ------------------------------------------------------------------------ */
int oracle_hillis_steele(const double *s, const float *V, int64_t N,
                         int64_t d, double *O)
{
    int64_t stride = d + 2; /* [m, w, u_0..u_{d-1}] */
    double *x = (double *)malloc((size_t)(N > 0 ? N : 1) * stride * sizeof(double));
    double *y = (double *)malloc((size_t)(N > 0 ? N : 1) * stride * sizeof(double));
    if (!x || !y) {
        free(x);
        free(y);
        return 1;
    }
    for (int64_t t = 0; t < N; ++t) {
        x[t * stride + 0] = s[t];
        x[t * stride + 1] = 1.0;
        for (int64_t j = 0; j < d; ++j)
            x[t * stride + 2 + j] = (double)V[t * d + j];
    }
    for (int64_t k = 1; k < N; k *= 2) {
        for (int64_t t = 0; t < N; ++t) {
            double *dst = y + t * stride;
            const double *b = x + t * stride;
            if (t >= k) {
                const double *a = x + (t - k) * stride;
                oracle_combine(a[0], a + 2, a[1], b[0], b + 2, b[1], d, &dst[0],
                               dst + 2, &dst[1]);
            } else {
                memcpy(dst, b, (size_t)stride * sizeof(double));
            }
        }
        double *tmp = x;
        x = y;
        y = tmp;
    }
    for (int64_t t = 0; t < N; ++t)
        for (int64_t j = 0; j < d; ++j)
            O[t * d + j] = x[t * stride + 2 + j] / x[t * stride + 1];
    free(x);
    free(y);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The same sequential recurrence in long double, results rounded to double */
/* on output.  Used only to bound the double oracle's own rounding error.   */
/* ------------------------------------------------------------------------ */
int oracle_scan_longdouble(const float *q, const float *K, const float *V,
                           int64_t N, int64_t d, double *O, double *m_out,
                           double *u_out, double *w_out)
{
    long double m = -INFINITY, w = 0.0L;
    long double *u = (long double *)calloc((size_t)(d > 0 ? d : 1), sizeof(long double));
    if (!u) return 1;
    for (int64_t t = 0; t < N; ++t) {
        long double s = 0.0L;
        for (int64_t j = 0; j < d; ++j)
            s += (long double)q[j] * (long double)K[t * d + j];
        long double M = (s > m) ? s : m;
        long double a = (m == -INFINITY) ? 0.0L : expl(m - M);
        long double b = expl(s - M);
        for (int64_t j = 0; j < d; ++j)
            u[j] = a * u[j] + b * (long double)V[t * d + j];
        w = a * w + b;
        m = M;
        if (O)
            for (int64_t j = 0; j < d; ++j) O[t * d + j] = (double)(u[j] / w);
    }
    if (m_out) *m_out = (double)m;
    if (w_out) *w_out = (double)w;
    if (u_out)
        for (int64_t j = 0; j < d; ++j) u_out[j] = (double)u[j];
    free(u);
    return 0;
}
