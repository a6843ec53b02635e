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

/* ======================================================================== */
/* Differentiation of the many-to-many output.                              */
/*                                                                          */
/* The memory-efficient-attention review reports its method for inference   */
/* and for differentiation (its abstract and section 5.2, whose body the    */
/* page lacks); the Aaren review calls the RNN form exact and               */
/* differentiable ("Proposed method").  For one head and an upstream        */
/* gradient g_t = dL/do_t (t = 1..N), with p_{t,i} = e^{s_i} / sum_{j<=t}   */
/* e^{s_j} for i <= t (so o_t = sum_{i<=t} p_{t,i} v_i):                     */
/*                                                                          */
/*   dL/dv_i = sum_{t>=i} p_{t,i} g_t                                       */
/*   dL/ds_i = sum_{t>=i} p_{t,i} (g_t . v_i - g_t . o_t)                   */
/*   dL/dq   = sum_i dL/ds_i k_i ,   dL/dk_i = dL/ds_i q                    */
/*                                                                          */
/* (the softmax Jacobian dp_{t,i}/ds_j = p_{t,i} (1[i=j] - p_{t,j})).       */
/* ======================================================================== */

/* Log of the softmax denominator of every prefix:                          */
/*   lse_t = log sum_{i<=t} e^{s_i}, evaluated as max + log(sum e^{s-max})  */
/* over the whole prefix (no running form).  O(N^2); used by the pins.      */
void oracle_lse_direct(const double *s, int64_t N, double *lse)
{
    for (int64_t t = 0; t < N; ++t) {
        double top = s[0];
        for (int64_t i = 1; i <= t; ++i) top = (s[i] > top) ? s[i] : top;
        double acc = 0.0;
        for (int64_t i = 0; i <= t; ++i) acc += exp(s[i] - top);
        lse[t] = top + log(acc);
    }
}

/* The definition above written out: O(N^2 d), small N only.  ds may be    */
/* NULL.  dq [d], dK [N,d], dV [N,d], ds [N] are written.                    */
void oracle_backward_bruteforce(const float *q, const float *K, const float *V,
                                const float *G, int64_t N, int64_t d,
                                double *dq, double *dK, double *dV, double *ds)
{
    double *s = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    double *p = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    double *o = (double *)malloc((size_t)(d > 0 ? d : 1) * sizeof(double));
    double *dsl = (double *)calloc((size_t)(N > 0 ? N : 1), sizeof(double));
    for (int64_t i = 0; i < N; ++i) {
        double acc = 0.0;
        for (int64_t j = 0; j < d; ++j) acc += (double)q[j] * (double)K[i * d + j];
        s[i] = acc;
    }
    for (int64_t x = 0; x < N * d; ++x) dV[x] = 0.0;
    for (int64_t t = 0; t < N; ++t) {
        /* softmax weights of prefix t and its output o_t */
        double top = s[0];
        for (int64_t i = 1; i <= t; ++i) top = (s[i] > top) ? s[i] : top;
        double z = 0.0;
        for (int64_t i = 0; i <= t; ++i) z += exp(s[i] - top);
        for (int64_t i = 0; i <= t; ++i) p[i] = exp(s[i] - top) / z;
        for (int64_t j = 0; j < d; ++j) {
            double acc = 0.0;
            for (int64_t i = 0; i <= t; ++i) acc += p[i] * (double)V[i * d + j];
            o[j] = acc;
        }
        double go = 0.0;
        for (int64_t j = 0; j < d; ++j) go += (double)G[t * d + j] * o[j];
        for (int64_t i = 0; i <= t; ++i) {
            double gv = 0.0;
            for (int64_t j = 0; j < d; ++j) {
                dV[i * d + j] += p[i] * (double)G[t * d + j];
                gv += (double)G[t * d + j] * (double)V[i * d + j];
            }
            dsl[i] += p[i] * (gv - go);
        }
    }
    for (int64_t j = 0; j < d; ++j) dq[j] = 0.0;
    for (int64_t i = 0; i < N; ++i)
        for (int64_t j = 0; j < d; ++j) {
            dq[j] += dsl[i] * (double)K[i * d + j];
            dK[i * d + j] = dsl[i] * (double)q[j];
        }
    if (ds)
        for (int64_t i = 0; i < N; ++i) ds[i] = dsl[i];
    free(s);
    free(p);
    free(o);
    free(dsl);
}

/* The same gradients in O(N d): the sums over t >= i run backwards, token  */
/* by token, as the two suffix sums                                         */
/*   R_i = sum_{t>=i} e^{lse_i - lse_t} g_t,                                */
/*   D_i = sum_{t>=i} e^{lse_i - lse_t} (g_t . o_t)                         */
/* (every weight <= 1, as lse never decreases along the sequence), so that  */
/*   R_i = g_i + e^{lse_i - lse_{i+1}} R_{i+1}   (same for D),              */
/*   dL/dv_i = e^{s_i - lse_i} R_i,                                         */
/*   dL/ds_i = e^{s_i - lse_i} (v_i . R_i - D_i).                           */
/* lse_t and o_t come from a forward pass in the running form (the          */
/* recurrence of oracle_scan_scores, with lse_t = m_t + log w_t).           */
/* ds may be NULL.  Returns nonzero when scratch allocation fails.          */
int oracle_backward(const float *q, const float *K, const float *V,
                    const float *G, int64_t N, int64_t d, double *dq,
                    double *dK, double *dV, double *ds)
{
    double *s = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    double *lse = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    double *O = (double *)malloc((size_t)(N > 0 ? N : 1) * (d > 0 ? d : 1) * sizeof(double));
    double *R = (double *)calloc((size_t)(d > 0 ? d : 1), sizeof(double));
    if (!s || !lse || !O || !R) {
        free(s);
        free(lse);
        free(O);
        free(R);
        return 1;
    }
    oracle_scores(q, K, N, d, s);
    /* forward: running maximum and rescaled sum give lse_t; outputs o_t */
    {
        double run_max = -INFINITY, run_sum = 0.0;
        for (int64_t t = 0; t < N; ++t) {
            double hi = (s[t] > run_max) ? s[t] : run_max;
            run_sum = run_sum * ((run_max == -INFINITY) ? 0.0 : exp(run_max - hi)) + exp(s[t] - hi);
            run_max = hi;
            lse[t] = run_max + log(run_sum);
        }
        oracle_scan_scores(s, V, N, d, NULL, NULL, NULL, O, NULL, NULL, NULL);
    }
    /* backward: suffix sums from the last token down */
    double D = 0.0;
    for (int64_t j = 0; j < d; ++j) dq[j] = 0.0;
    for (int64_t i = N - 1; i >= 0; --i) {
        if (i + 1 < N) {
            double decay = exp(lse[i] - lse[i + 1]);
            for (int64_t j = 0; j < d; ++j) R[j] *= decay;
            D *= decay;
        }
        double go = 0.0, vr = 0.0;
        for (int64_t j = 0; j < d; ++j) {
            go += (double)G[i * d + j] * O[i * d + j];
            R[j] += (double)G[i * d + j];
        }
        D += go;
        double pii = exp(s[i] - lse[i]);
        for (int64_t j = 0; j < d; ++j) {
            dV[i * d + j] = pii * R[j];
            vr += (double)V[i * d + j] * R[j];
        }
        double dsi = pii * (vr - D);
        for (int64_t j = 0; j < d; ++j) {
            dK[i * d + j] = dsi * (double)q[j];
            dq[j] += dsi * (double)K[i * d + j];
        }
        if (ds) ds[i] = dsi;
    }
    free(s);
    free(lse);
    free(O);
    free(R);
    return 0;
}

/* lse_t of every prefix in the running form (as oracle_backward's forward  */
/* pass); the value the library's forward writes next to O for a backward.  */
int oracle_lse(const float *q, const float *K, int64_t N, int64_t d, double *lse)
{
    double *s = (double *)malloc((size_t)(N > 0 ? N : 1) * sizeof(double));
    if (!s) return 1;
    oracle_scores(q, K, N, d, s);
    double run_max = -INFINITY, run_sum = 0.0;
    for (int64_t t = 0; t < N; ++t) {
        double hi = (s[t] > run_max) ? s[t] : run_max;
        run_sum = run_sum * ((run_max == -INFINITY) ? 0.0 : exp(run_max - hi)) + exp(s[t] - hi);
        run_max = hi;
        lse[t] = run_max + log(run_sum);
    }
    free(s);
    return 0;
}
