"""Pins for the float64 oracle: checks against things other than the oracle.

Each pin_* function raises AssertionError on failure.  tests/test_oracle.py
runs them against the real oracle, and against deliberately broken copies of
oracle.c to show that each plausible mistake (a dropped term, a wrong sign, a
wrong index, a transposed operand) fails at least one pin.

What pins what:
  worked example   hand-derived rational example of the definition
                   (tests/golden/rational_worked_example.txt)
  brute force      per-prefix textbook softmax on tiny inputs
  last row         o_N equals single-query softmax attention, computed with
                   numpy's matmul and scipy.special.softmax
  scores           q . k_t equals numpy's matmul
  shift            adding a constant to every score leaves O unchanged and
                   shifts m by that constant
  equal scores     q = 0 gives the prefix means cumsum(V)/t
  Hillis-Steele    the parallel-scan order of the same operator agrees
  operator laws    associativity, commutativity, identity
  first output     o_1 = v_1
  one-hot          a score 60 above the rest makes o_t that token's v
  bounds           o_t inside the convex hull of v_1..v_t, 1 <= w <= N,
                   m = max s
  long double      the same recurrence in long double agrees to ~1e-14
  large scores     |s| up to 5000 (exp would overflow without rescaling)
  continuation     scanning [A; B] equals scanning B from A's final state
  running sum      the unscaled running sums of the memory-efficient-attention
                   review (section 2) agree when the scores are moderate
Differentiation (gradients of L = sum_t g_t . o_t):
  finite diff.     central differences of L computed by an independent numpy
                   forward (per-prefix scipy.special.softmax, matmuls)
  suffix sums      the O(N d) backward equals the O(N^2 d) definition
  shift            sum_i dL/ds_i = 0 (L does not change when every score
                   moves by the same constant)
  one token        o_1 = v_1, so dL/dv_1 = g_1 and every score gradient is 0
  equal scores     q = 0: dL/dv_i = sum_{t>=i} g_t / t
  log-sum-exp      lse_t (running form) equals scipy.special.logsumexp of
                   every prefix and the per-prefix direct form
  large scores     |s| in the hundreds: the backward stays finite and agrees
Causal cos-re-weighted linear attention (cosFormer):
  worked example   hand-derived outputs and final state, exact in a + b sqrt3
                   (tests/golden/cosformer_worked_example.txt)
  definition       the decomposed prefix sums equal the O(N^2 d) definition
  ReLU linear att. M -> infinity gives causal ReLU linear attention written
                   with numpy matrix products
  prefix means     equal similarities, M -> infinity: cumsum(V) / i
  invariances      query-row and key scaling, ReLU of negative coordinates,
                   value shift, causality, o_1 = v_1, box bounds
  zero query       a query with no positive coordinate gives o_i = 0
  continuation     scanning [A; B] equals scanning B from A's state
"""
import os
from fractions import Fraction

import numpy as np
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def _rel(a, b):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    return float(np.max(np.abs(a - b)) / max(1e-300, float(np.max(np.abs(b)))))


def read_fixture_r3(name):
    """Like read_fixture, but keys ending in _r3 hold a,b pairs (a + b*sqrt3),
    returned as float64 arrays; other keys as float64 arrays of fractions."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            key = key.strip()
            rows = []
            for r in rest.split("|"):
                if key.endswith("_r3"):
                    vals = []
                    for x in r.split():
                        a, b = x.split(",")
                        vals.append(float(Fraction(a)) + float(Fraction(b)) * np.sqrt(3.0))
                    rows.append(vals)
                else:
                    rows.append([float(Fraction(x)) for x in r.split()])
            out[key] = np.array(rows, dtype=np.float64)
    return out


def read_fixture(name):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, rest = line.split(":", 1)
            rows = [[Fraction(x) for x in r.split()] for r in rest.split("|")]
            vals[key.strip()] = rows
    return vals


def pin_worked_example():
    fx = read_fixture("rational_worked_example.txt")
    e = [float(x) for x in fx["scores_exp"][0]]
    s = np.log(np.array(e))
    V = np.array([[float(x) for x in r] for r in fx["V"]], dtype=np.float32)
    want = np.array([[float(x) for x in r] for r in fx["O"]])
    O, m, u, w = oracle.scan_scores(s, V)
    assert np.max(np.abs(O - want)) < 1e-14, (O, want)
    assert abs(np.exp(m) - float(fx["m_exp"][0][0])) < 1e-13
    assert abs(w - float(fx["w"][0][0])) < 1e-14
    assert np.max(np.abs(u - np.array([float(x) for x in fx["u"][0]]))) < 1e-14
    for alt in (oracle.bruteforce(s, V), oracle.hillis_steele(s, V)):
        assert np.max(np.abs(alt - want)) < 1e-14


def pin_bruteforce():
    r = _rng(11)
    for N, d, scale in ((1, 3, 1.0), (2, 4, 1.0), (7, 16, 3.0), (64, 8, 10.0), (200, 5, 30.0)):
        q = r.standard_normal(d).astype(np.float32)
        K = (scale * r.standard_normal((N, d))).astype(np.float32)
        V = r.standard_normal((N, d)).astype(np.float32)
        O, m, u, w = oracle.scan(q, K, V)
        s = oracle.scores(q, K)
        Ob = oracle.bruteforce(s, V)
        assert _rel(O, Ob) < 1e-12, (N, d, _rel(O, Ob))


def pin_last_row():
    r = _rng(12)
    for N, d in ((1, 4), (33, 16), (300, 64)):
        q = r.standard_normal(d).astype(np.float32)
        K = (2 * r.standard_normal((N, d))).astype(np.float32)
        V = r.standard_normal((N, d)).astype(np.float32)
        O, m, u, w = oracle.scan(q, K, V)
        s_np = K.astype(np.float64) @ q.astype(np.float64)
        ref = scipy.special.softmax(s_np) @ V.astype(np.float64)
        assert _rel(O[-1], ref) < 1e-12
        assert abs(m - s_np.max()) <= 1e-12 * max(1.0, abs(s_np.max()))
        assert abs(w - np.exp(s_np - s_np.max()).sum()) < 1e-10 * N
        assert _rel(u / w, ref) < 1e-12


def pin_scores():
    r = _rng(13)
    q = r.standard_normal(64).astype(np.float32)
    K = r.standard_normal((100, 64)).astype(np.float32)
    s = oracle.scores(q, K)
    ref = K.astype(np.float64) @ q.astype(np.float64)
    assert np.max(np.abs(s - ref)) < 1e-12


def pin_shift():
    r = _rng(14)
    N, d = 150, 8
    s = 5 * r.standard_normal(N)
    V = r.standard_normal((N, d)).astype(np.float32)
    O0, m0, u0, w0 = oracle.scan_scores(s, V)
    for c in (100.0, -700.0, 0.5):
        O1, m1, u1, w1 = oracle.scan_scores(s + c, V)
        assert _rel(O1, O0) < 1e-12
        assert abs(m1 - (m0 + c)) < 1e-9
        assert abs(w1 - w0) < 1e-12 * w0
        assert _rel(u1, u0) < 1e-12


def pin_equal_scores():
    r = _rng(15)
    for N, d in ((1, 4), (97, 16)):
        q = np.zeros(d, dtype=np.float32)
        K = r.standard_normal((N, d)).astype(np.float32)
        V = r.standard_normal((N, d)).astype(np.float32)
        O, m, u, w = oracle.scan(q, K, V)
        ref = np.cumsum(V.astype(np.float64), axis=0) / np.arange(1, N + 1)[:, None]
        assert _rel(O, ref) < 1e-12
        assert m == 0.0 and abs(w - N) < 1e-9


def pin_hillis_steele():
    r = _rng(16)
    for N, d in ((1, 2), (2, 3), (3, 4), (100, 8), (257, 5), (64, 16)):
        s = 20 * r.standard_normal(N)
        V = r.standard_normal((N, d)).astype(np.float32)
        O, m, u, w = oracle.scan_scores(s, V)
        Oh = oracle.hillis_steele(s, V)
        assert _rel(Oh, O) < 1e-12, (N, d)


def _state(r, d, m=None):
    m = float(10 * r.standard_normal()) if m is None else m
    return m, r.standard_normal(d), float(abs(r.standard_normal()) + 0.1)


def _same_state(a, b, tol=1e-12):
    # compare as functions of the represented sums: rebase b to a's m
    ma, ua, wa = a
    mb, ub, wb = b
    if ma == -np.inf or mb == -np.inf:
        return ma == mb and wa == wb == 0.0 and not np.any(ua) and not np.any(ub)
    f = np.exp(mb - ma)
    return (abs(ma - mb) < 1e-12 * max(1.0, abs(ma))
            and abs(wb * f - wa) <= tol * abs(wa)
            and np.max(np.abs(ub * f - ua)) <= tol * max(1e-300, np.max(np.abs(ua))))


def pin_operator_laws():
    r = _rng(17)
    d = 6
    ident = (-np.inf, np.zeros(d), 0.0)
    for _ in range(50):
        a, b, c = _state(r, d), _state(r, d), _state(r, d)
        ab_c = oracle.combine(oracle.combine(a, b), c)
        a_bc = oracle.combine(a, oracle.combine(b, c))
        assert _same_state(ab_c, a_bc)
        assert _same_state(oracle.combine(a, b), oracle.combine(b, a))
        assert _same_state(oracle.combine(ident, a), a)
        assert _same_state(oracle.combine(a, ident), a)
    assert _same_state(oracle.combine(ident, ident), ident)
    # the operator on two leaves equals the two-token softmax (closed form)
    v1, v2 = r.standard_normal(d), r.standard_normal(d)
    m, u, w = oracle.combine((1.5, v1, 1.0), (-0.5, v2, 1.0))
    p = 1.0 / (1.0 + np.exp(-2.0))
    assert m == 1.5 and np.max(np.abs(u / w - (p * v1 + (1 - p) * v2))) < 1e-14


def pin_first_output():
    r = _rng(18)
    for d in (1, 16, 128):
        q = r.standard_normal(d).astype(np.float32)
        K = r.standard_normal((5, d)).astype(np.float32)
        V = r.standard_normal((5, d)).astype(np.float32)
        O, m, u, w = oracle.scan(q, K, V)
        assert np.array_equal(O[0], V[0].astype(np.float64))


def pin_one_hot():
    r = _rng(19)
    N, d, star = 64, 8, 20
    s = r.standard_normal(N)
    s[star] = s.max() + 60.0
    V = r.standard_normal((N, d)).astype(np.float32)
    O, m, u, w = oracle.scan_scores(s, V)
    assert np.max(np.abs(O[star:] - V[star].astype(np.float64))) < N * np.exp(-55)
    assert _rel(O[:star], oracle.bruteforce(s[:star], V[:star])) < 1e-12


def pin_bounds():
    r = _rng(20)
    N, d = 120, 8
    s = 15 * r.standard_normal(N)
    V = r.standard_normal((N, d)).astype(np.float32)
    O, m, u, w = oracle.scan_scores(s, V)
    Vd = V.astype(np.float64)
    lo = np.minimum.accumulate(Vd, axis=0)
    hi = np.maximum.accumulate(Vd, axis=0)
    assert np.all(O >= lo - 1e-12) and np.all(O <= hi + 1e-12)
    assert m == s.max()
    assert 1.0 <= w <= N
    for t in (1, 2, 10, 57):   # the prefix states obey the same bounds
        _, mt, ut, wt = oracle.scan_scores(s[:t], V[:t], want_O=False)
        assert mt == s[:t].max() and 1.0 <= wt <= t


def pin_long_double():
    r = _rng(21)
    q = r.standard_normal(16).astype(np.float32)
    K = (4 * r.standard_normal((256, 16))).astype(np.float32)
    V = r.standard_normal((256, 16)).astype(np.float32)
    O, m, u, w = oracle.scan(q, K, V)
    Ol, ml, ul, wl = oracle.scan_longdouble(q, K, V)
    assert _rel(O, Ol) < 1e-13
    assert abs(m - ml) < 1e-13 * max(1.0, abs(ml))
    assert abs(w - wl) < 1e-13 * wl and _rel(u, ul) < 1e-13


def pin_large_scores():
    r = _rng(22)
    N, d = 90, 4
    s = 2000 * r.standard_normal(N)
    s[::7] = 5000.0 - r.random(len(s[::7]))
    V = r.uniform(-1, 1, (N, d)).astype(np.float32)
    O, m, u, w = oracle.scan_scores(s, V)
    assert np.all(np.isfinite(O)) and np.isfinite(w) and np.all(np.isfinite(u))
    assert _rel(O, oracle.bruteforce(s, V)) < 1e-12


def pin_continuation():
    r = _rng(23)
    N, d = 200, 8
    q = r.standard_normal(d).astype(np.float32)
    K = (3 * r.standard_normal((N, d))).astype(np.float32)
    V = r.standard_normal((N, d)).astype(np.float32)
    O, m, u, w = oracle.scan(q, K, V)
    for cut in (1, 50, 199):
        _, ma, ua, wa = oracle.scan(q, K[:cut], V[:cut], want_O=False)
        Ob, mb, ub, wb = oracle.scan(q, K[cut:], V[cut:], init=(ma, ua, wa))
        assert _rel(Ob, O[cut:]) < 1e-12
        assert _same_state((m, u, w), (mb, ub, wb))


def pin_running_sum():
    # the memory-efficient-attention review's section 2 algorithm taken as
    # written: unscaled sums v* += v e^s, s* += e^s, output v*/s* (scores kept
    # moderate so e^s cannot overflow)
    r = _rng(24)
    N, d = 80, 6
    s = 3 * r.standard_normal(N)
    V = r.standard_normal((N, d)).astype(np.float32)
    vstar = np.zeros(d)
    sstar = 0.0
    ref = np.empty((N, d))
    for t in range(N):
        vstar = vstar + V[t].astype(np.float64) * np.exp(s[t])
        sstar = sstar + np.exp(s[t])
        ref[t] = vstar / sstar
    O, m, u, w = oracle.scan_scores(s, V)
    assert _rel(O, ref) < 1e-12


def _numpy_loss(q, K, V, G):
    """L = sum_t G_t . o_t with o_t the per-prefix softmax of q.k_i over V,
    in numpy float64 (independent of the oracle's C code)."""
    s = K @ q
    total = 0.0
    for t in range(len(s)):
        p = scipy.special.softmax(s[:t + 1])
        total += float(G[t] @ (p @ V[:t + 1]))
    return total


def _small(seed, N, d, scale=1.0):
    r = _rng(seed)
    f = lambda *shape: r.standard_normal(shape).astype(np.float32)
    return f(d) * np.float32(scale), f(N, d), f(N, d), f(N, d)


def pin_backward_finite_differences():
    for seed, N, d in ((1, 6, 3), (2, 11, 4), (3, 1, 2)):
        q, K, V, G = _small(seed, N, d)
        dq, dK, dV, _ = oracle.backward_bruteforce(q, K, V, G)
        q64, K64, V64, G64 = (x.astype(np.float64) for x in (q, K, V, G))
        h = 1e-5
        r = _rng(100 + seed)
        checks = [("q", j, None) for j in range(d)]
        checks += [("K", int(r.integers(N)), int(r.integers(d))) for _ in range(4)]
        checks += [("V", int(r.integers(N)), int(r.integers(d))) for _ in range(4)]
        for name, a, b in checks:
            base = {"q": q64, "K": K64, "V": V64}[name]
            plus, minus = base.copy(), base.copy()
            idx = (a,) if b is None else (a, b)
            plus[idx] += h
            minus[idx] -= h
            args_p = {"q": q64, "K": K64, "V": V64, name: plus}
            args_m = {"q": q64, "K": K64, "V": V64, name: minus}
            fd = (_numpy_loss(args_p["q"], args_p["K"], args_p["V"], G64) -
                  _numpy_loss(args_m["q"], args_m["K"], args_m["V"], G64)) / (2 * h)
            an = {"q": dq, "K": dK, "V": dV}[name][idx]
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(fd)), (name, idx, fd, an)


def pin_backward_suffix_sums():
    for seed, N, d in ((4, 1, 1), (5, 2, 3), (6, 17, 5), (7, 40, 8)):
        q, K, V, G = _small(seed, N, d, scale=2.0)
        ref = oracle.backward_bruteforce(q, K, V, G)
        got = oracle.backward(q, K, V, G)
        # dL/ds_i is a difference of two sums that nearly cancel: a few
        # hundred ulps of float64 apart at most when both are right
        for a, b in zip(got, ref):
            assert _rel(a, b) < 1e-10


def pin_backward_shift():
    q, K, V, G = _small(8, 30, 6, scale=3.0)
    _, _, _, ds = oracle.backward(q, K, V, G)
    assert abs(float(np.sum(ds))) <= 1e-12 * float(np.sum(np.abs(ds)))


def pin_backward_one_token():
    q, K, V, G = _small(9, 1, 5)
    dq, dK, dV, ds = oracle.backward(q, K, V, G)
    assert np.array_equal(dV[0], G[0].astype(np.float64))
    assert abs(ds[0]) <= 1e-15 and np.max(np.abs(dq)) <= 1e-15 and np.max(np.abs(dK)) <= 1e-15


def pin_backward_equal_scores():
    _, K, V, G = _small(10, 25, 4)
    q = np.zeros(4, dtype=np.float32)
    _, _, dV, _ = oracle.backward(q, K, V, G)
    t = np.arange(1, 26, dtype=np.float64)[:, None]
    ref = np.cumsum((G.astype(np.float64) / t)[::-1], axis=0)[::-1]
    assert _rel(dV, ref) < 1e-13


def pin_lse():
    q, K, _, _ = _small(11, 50, 6, scale=4.0)
    got = oracle.lse(q, K)
    s = oracle.scores(q, K)
    ref = np.array([scipy.special.logsumexp(s[:t + 1]) for t in range(len(s))])
    assert _rel(got, ref) < 1e-13
    assert _rel(oracle.lse_direct(s), ref) < 1e-13


def pin_backward_large_scores():
    q, K, V, G = _small(12, 60, 4)
    K = (K * np.float32(60.0)).astype(np.float32)    # scores of several hundred
    s = oracle.scores(q, K)
    assert np.max(np.abs(s)) > 150
    got = oracle.backward(q, K, V, G)
    ref = oracle.backward_bruteforce(q, K, V, G)
    for a, b in zip(got, ref):
        assert np.all(np.isfinite(a))
        assert _rel(a, b) < 1e-11


# ---------------------------------------------------------------------------
# Causal cos-re-weighted linear attention (cosFormer section of the LG AI
# Research "Efficient Transformer" review).
# ---------------------------------------------------------------------------

def _la_inputs(seed, N, d, neg=True):
    r = _rng(seed)
    Q = r.standard_normal((N, d)).astype(np.float32)
    K = r.standard_normal((N, d)).astype(np.float32)
    V = r.standard_normal((N, d)).astype(np.float32)
    if not neg:
        Q, K = np.abs(Q), np.abs(K)
    return Q, K, V


def pin_la_worked_example():
    fx = read_fixture_r3("cosformer_worked_example.txt")
    M = float(fx["M"][0][0])
    Q, K, V = (fx[k].astype(np.float32) for k in ("Q", "K", "V"))
    num, den = fx["num_r3"], fx["den_r3"][:, 0]
    want = np.where(den[:, None] != 0, num / np.where(den == 0, 1, den)[:, None], 0.0)
    Ob = oracle.la_bruteforce(Q, K, V, M)
    O, (Sc, Ss, zc, zs) = oracle.la_scan(Q, K, V, M)
    assert np.max(np.abs(Ob - want)) < 1e-14, (Ob, want)
    assert np.max(np.abs(O - want)) < 1e-13, (O, want)
    assert np.max(np.abs(zc - fx["zc_r3"][0])) < 1e-13 and np.max(np.abs(zs - fx["zs_r3"][0])) < 1e-13
    assert np.max(np.abs(Sc - fx["Sc_r3"])) < 1e-13, (Sc, fx["Sc_r3"])
    assert np.max(np.abs(Ss - fx["Ss_r3"])) < 1e-13, (Ss, fx["Ss_r3"])


def pin_la_scan_equals_definition():
    """The decomposed prefix sums equal the definition (two different
    computations: cos of the difference vs the cosine sum formula)."""
    for seed, N, d, Mf in ((1, 1, 4, 1.0), (2, 7, 3, 1.0), (3, 64, 16, 1.0), (4, 200, 8, 2.5),
                           (5, 150, 32, 40.0)):
        Q, K, V = _la_inputs(seed, N, d)
        M = Mf * N
        Ob = oracle.la_bruteforce(Q, K, V, M)
        O, _ = oracle.la_scan(Q, K, V, M)
        assert _rel(O, Ob) < 1e-12, (N, d, _rel(O, Ob))


def pin_la_relu_linear_attention():
    """M -> infinity removes the re-weighting (every cos is 1): the output is
    causal linear attention with the ReLU feature map, written with numpy
    matrix products (the masked similarity matrix, normalised by its row
    sums)."""
    for seed, N, d in ((6, 50, 8), (7, 120, 16)):
        Q, K, V = _la_inputs(seed, N, d)
        Qp, Kp = np.maximum(Q.astype(np.float64), 0), np.maximum(K.astype(np.float64), 0)
        P = np.tril(Qp @ Kp.T)
        rs = P.sum(axis=1, keepdims=True)
        want = np.where(rs > 0, (P @ V.astype(np.float64)) / np.where(rs > 0, rs, 1), 0.0)
        for got in (oracle.la_bruteforce(Q, K, V, 1e300), oracle.la_scan(Q, K, V, 1e300)[0]):
            assert _rel(got, want) < 1e-12, _rel(got, want)


def pin_la_prefix_means():
    """All similarities equal and M -> infinity: o_i is the mean of v_1..v_i."""
    N, d = 40, 5
    Q = np.full((N, d), 0.5, np.float32)
    K = np.full((N, d), 2.0, np.float32)
    V = _la_inputs(8, N, d)[2]
    want = np.cumsum(V.astype(np.float64), axis=0) / np.arange(1, N + 1)[:, None]
    for got in (oracle.la_bruteforce(Q, K, V, 1e300), oracle.la_scan(Q, K, V, 1e300)[0]):
        assert _rel(got, want) < 1e-13


def pin_la_invariances():
    """Scaling a query row or all keys by c > 0 (powers of two, so the inputs
    stay exact) leaves O unchanged; negative
    coordinates of Q and K act as zeros (the ReLU map); adding a constant
    vector to every value adds it to every output; o_i does not depend on
    tokens after i; o_1 = v_1; each o_i lies in the box spanned by v_1..v_i."""
    N, d = 80, 12
    Q, K, V = _la_inputs(9, N, d)
    M = float(N)
    O, _ = oracle.la_scan(Q, K, V, M)
    c = np.float32(2.0) ** (np.arange(N) % 7 - 3).astype(np.float32)[:, None]   # exact scalings
    assert _rel(oracle.la_scan(Q * c, K, V, M)[0], O) < 1e-13
    assert _rel(oracle.la_scan(Q, K * np.float32(4.0), V, M)[0], O) < 1e-13
    Qn = np.where(Q > 0, Q, np.float32(-7.0)); Kn = np.where(K > 0, K, np.float32(-0.5))
    assert _rel(oracle.la_scan(Qn, Kn, V, M)[0], O) < 1e-15
    Vq = (np.round(V * 1024) / 1024).astype(np.float32)           # dyadic: V + shift stays exact
    shift = np.arange(-5, d - 5).astype(np.float32)
    O = oracle.la_scan(Q, K, Vq, M)[0]
    Os = oracle.la_scan(Q, K, Vq + shift, M)[0]
    sim = np.tril(np.maximum(Q.astype(np.float64), 0) @ np.maximum(K.astype(np.float64), 0).T)
    live = np.any(sim > 0, axis=1)          # rows with a non-zero denominator
    assert np.max(np.abs(Os[live] - (O[live] + shift))) < 1e-12
    O, V = oracle.la_scan(Q, K, V, M)[0], V
    K2, V2 = K.copy(), V.copy()
    K2[50:] = _la_inputs(10, N - 50, d)[1]; V2[50:] = 9.0
    assert np.max(np.abs(oracle.la_scan(Q, K2, V2, M)[0][:50] - O[:50])) == 0.0
    assert np.max(np.abs(oracle.la_bruteforce(Q, K2, V2, M)[:50] - oracle.la_bruteforce(Q, K, V, M)[:50])) == 0.0
    if np.dot(np.maximum(Q[0], 0), np.maximum(K[0], 0)) > 0:
        assert np.max(np.abs(O[0] - V[0])) < 1e-15
    lo = np.minimum.accumulate(V.astype(np.float64), axis=0)
    hi = np.maximum.accumulate(V.astype(np.float64), axis=0)
    assert np.all(O[live] >= lo[live] - 1e-12) and np.all(O[live] <= hi[live] + 1e-12)


def pin_la_zero_query():
    """A query with no positive coordinate has zero similarity to every key:
    its output is 0 (the reading for an empty weighted average)."""
    Q, K, V = _la_inputs(11, 30, 6)
    Q[[0, 7, 29]] = -np.abs(Q[[0, 7, 29]])
    for got in (oracle.la_bruteforce(Q, K, V, 30.0), oracle.la_scan(Q, K, V, 30.0)[0]):
        assert np.all(got[[0, 7, 29]] == 0.0) and np.all(np.isfinite(got))


def pin_la_continuation():
    """Scanning [A; B] equals scanning B from A's final state with positions
    continued (and both final states agree)."""
    N, d, cut = 90, 10, 37
    Q, K, V = _la_inputs(12, N, d)
    M = float(N)
    O, st = oracle.la_scan(Q, K, V, M)
    _, stA = oracle.la_scan(Q[:cut], K[:cut], V[:cut], M, want_O=False)
    OB, stB = oracle.la_scan(Q[cut:], K[cut:], V[cut:], M, init=stA, pos0=cut)
    assert _rel(OB, O[cut:]) < 1e-13
    for a, b in zip(stB, st):
        assert _rel(a, b) < 1e-13


ALL_PINS = [
    pin_worked_example, pin_bruteforce, pin_last_row, pin_scores, pin_shift,
    pin_equal_scores, pin_hillis_steele, pin_operator_laws, pin_first_output,
    pin_one_hot, pin_bounds, pin_long_double, pin_large_scores, pin_continuation,
    pin_running_sum, pin_backward_finite_differences, pin_backward_suffix_sums,
    pin_backward_shift, pin_backward_one_token, pin_backward_equal_scores, pin_lse,
    pin_backward_large_scores, pin_la_worked_example, pin_la_scan_equals_definition,
    pin_la_relu_linear_attention, pin_la_prefix_means, pin_la_invariances, pin_la_zero_query,
    pin_la_continuation,
]
