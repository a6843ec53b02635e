"""Float64 oracle for the softmax-attention prefix scan and the causal
cos-re-weighted linear-attention scan (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, the package smoke check and the
benchmark's CPU-baseline leg are the only callers.  The CUDA library and its
Python binding never import this package, and this package imports nothing
from them.  All arithmetic lives in oracle.c (plain sequential C in double)
and linattn.c; this module only converts numpy arrays and calls them.

Inputs are float32 numpy arrays (bfloat16 data must be widened to float32
first, which is exact).  Outputs are float64.
"""
import contextlib
import ctypes
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

_lib = None
_override = None

_f32p = ctypes.POINTER(ctypes.c_float)
_f64p = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def _bind(path):
    lib = ctypes.CDLL(path)
    lib.oracle_scores.argtypes = [_f32p, _f32p, _i64, _i64, _f64p]
    lib.oracle_scores.restype = None
    lib.oracle_scan_scores.argtypes = [_f64p, _f32p, _i64, _i64, _f64p, _f64p,
                                       _f64p, _f64p, _f64p, _f64p, _f64p]
    lib.oracle_scan_scores.restype = None
    lib.oracle_scan.argtypes = [_f32p, _f32p, _f32p, _i64, _i64, _f64p, _f64p,
                                _f64p, _f64p, _f64p, _f64p, _f64p]
    lib.oracle_scan.restype = ctypes.c_int
    lib.oracle_bruteforce.argtypes = [_f64p, _f32p, _i64, _i64, _f64p]
    lib.oracle_bruteforce.restype = None
    lib.oracle_combine.argtypes = [ctypes.c_double, _f64p, ctypes.c_double,
                                   ctypes.c_double, _f64p, ctypes.c_double, _i64,
                                   _f64p, _f64p, _f64p]
    lib.oracle_combine.restype = None
    lib.oracle_hillis_steele.argtypes = [_f64p, _f32p, _i64, _i64, _f64p]
    lib.oracle_hillis_steele.restype = ctypes.c_int
    lib.oracle_scan_longdouble.argtypes = [_f32p, _f32p, _f32p, _i64, _i64,
                                           _f64p, _f64p, _f64p, _f64p]
    lib.oracle_scan_longdouble.restype = ctypes.c_int
    lib.oracle_lse_direct.argtypes = [_f64p, _i64, _f64p]
    lib.oracle_lse_direct.restype = None
    lib.oracle_lse.argtypes = [_f32p, _f32p, _i64, _i64, _f64p]
    lib.oracle_lse.restype = ctypes.c_int
    lib.oracle_backward_bruteforce.argtypes = [_f32p, _f32p, _f32p, _f32p, _i64, _i64,
                                               _f64p, _f64p, _f64p, _f64p]
    lib.oracle_backward_bruteforce.restype = None
    lib.oracle_backward.argtypes = [_f32p, _f32p, _f32p, _f32p, _i64, _i64,
                                    _f64p, _f64p, _f64p, _f64p]
    lib.oracle_backward.restype = ctypes.c_int
    lib.oracle_la_bruteforce.argtypes = [_f32p, _f32p, _f32p, _i64, _i64, ctypes.c_double, _f64p]
    lib.oracle_la_bruteforce.restype = None
    lib.oracle_la_scan.argtypes = [_f32p, _f32p, _f32p, _i64, _i64, ctypes.c_double, _i64,
                                   _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p, _f64p]
    lib.oracle_la_scan.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _override is not None:
        return _override
    if _lib is None:
        _lib = _bind(_build.build())
    return _lib


@contextlib.contextmanager
def using_library(path):
    """Run the wrappers against another build of oracle.c (the tests use this
    to check that deliberately broken copies fail the pins)."""
    global _override
    prev = _override
    _override = _bind(path)
    try:
        yield
    finally:
        _override = prev


def _f32(x):
    return np.ascontiguousarray(x, dtype=np.float32)


def _f64(x):
    return np.ascontiguousarray(x, dtype=np.float64)


def _p32(a):
    return a.ctypes.data_as(_f32p)


def _p64(a):
    return None if a is None else a.ctypes.data_as(_f64p)


def scores(q, K):
    """s_t = q . k_t in double; q [d], K [N, d]."""
    q, K = _f32(q), _f32(K)
    N, d = K.shape
    s = np.empty(N, dtype=np.float64)
    _load().oracle_scores(_p32(q), _p32(K), N, d, _p64(s))
    return s


def _init_arrays(init, d):
    if init is None:
        return None, None, None
    m0, u0, w0 = init
    return (np.array([m0], dtype=np.float64), _f64(np.reshape(u0, (d,))),
            np.array([w0], dtype=np.float64))


def scan_scores(s, V, init=None, want_O=True):
    """Sequential recurrence from given scores; returns (O or None, m, u, w)."""
    s, V = _f64(s), _f32(V)
    N, d = V.shape
    m0, u0, w0 = _init_arrays(init, d)
    O = np.empty((N, d), dtype=np.float64) if want_O else None
    m = np.empty(1); w = np.empty(1); u = np.empty(d)
    _load().oracle_scan_scores(_p64(s), _p32(V), N, d, _p64(m0), _p64(u0), _p64(w0),
                               _p64(O), _p64(m), _p64(u), _p64(w))
    return O, float(m[0]), u, float(w[0])


def scan(q, K, V, init=None, want_O=True, out=None):
    """One head: scores then recurrence.  Returns (O [N,d] or None, m, u [d], w).
    `out` (optional, float64 C-contiguous [N, d]) receives O in place of a
    fresh array."""
    q, K, V = _f32(q), _f32(K), _f32(V)
    N, d = K.shape
    m0, u0, w0 = _init_arrays(init, d)
    if out is not None:
        if out.dtype != np.float64 or out.shape != (N, d) or not out.flags.c_contiguous:
            raise ValueError("out must be a C-contiguous float64 array of shape [N, d]")
        O = out
    else:
        O = np.empty((N, d), dtype=np.float64) if want_O else None
    m = np.empty(1); w = np.empty(1); u = np.empty(d)
    rc = _load().oracle_scan(_p32(q), _p32(K), _p32(V), N, d, _p64(m0), _p64(u0),
                             _p64(w0), _p64(O), _p64(m), _p64(u), _p64(w))
    if rc != 0:
        raise MemoryError("oracle_scan: allocation failed")
    return O, float(m[0]), u, float(w[0])


def bruteforce(s, V):
    """Per-prefix direct softmax, O(N^2 d)."""
    s, V = _f64(s), _f32(V)
    N, d = V.shape
    O = np.empty((N, d), dtype=np.float64)
    _load().oracle_bruteforce(_p64(s), _p32(V), N, d, _p64(O))
    return O


def combine(a, b):
    """The associative operator on states a = (m, u, w), b = (m, u, w)."""
    ma, ua, wa = a
    mb, ub, wb = b
    ua, ub = _f64(ua), _f64(ub)
    d = ua.shape[0]
    m = np.empty(1); w = np.empty(1); u = np.empty(d)
    _load().oracle_combine(float(ma), _p64(ua), float(wa), float(mb), _p64(ub),
                           float(wb), d, _p64(m), _p64(u), _p64(w))
    return float(m[0]), u, float(w[0])


def hillis_steele(s, V):
    """Hillis-Steele scan of the operator over leaves (s_t, v_t, 1)."""
    s, V = _f64(s), _f32(V)
    N, d = V.shape
    O = np.empty((N, d), dtype=np.float64)
    if _load().oracle_hillis_steele(_p64(s), _p32(V), N, d, _p64(O)) != 0:
        raise MemoryError("oracle_hillis_steele: allocation failed")
    return O


def scan_longdouble(q, K, V):
    """The recurrence in long double (rounded to double on output)."""
    q, K, V = _f32(q), _f32(K), _f32(V)
    N, d = K.shape
    O = np.empty((N, d), dtype=np.float64)
    m = np.empty(1); w = np.empty(1); u = np.empty(d)
    if _load().oracle_scan_longdouble(_p32(q), _p32(K), _p32(V), N, d, _p64(O),
                                      _p64(m), _p64(u), _p64(w)) != 0:
        raise MemoryError("oracle_scan_longdouble: allocation failed")
    return O, float(m[0]), u, float(w[0])


def lse_direct(s):
    """log sum_{i<=t} e^{s_i} of every prefix t, each prefix summed afresh."""
    s = _f64(s)
    out = np.empty(len(s), dtype=np.float64)
    _load().oracle_lse_direct(_p64(s), len(s), _p64(out))
    return out


def lse(q, K):
    """log sum_{i<=t} e^{q.k_i} of every prefix t, in the running form."""
    q, K = _f32(q), _f32(K)
    N, d = K.shape
    out = np.empty(N, dtype=np.float64)
    if _load().oracle_lse(_p32(q), _p32(K), N, d, _p64(out)) != 0:
        raise MemoryError("oracle_lse: allocation failed")
    return out


def backward_bruteforce(q, K, V, G):
    """Gradients of L = sum_t G_t . o_t from their definition, O(N^2 d).
    Returns (dq [d], dK [N,d], dV [N,d], ds [N]) in float64."""
    q, K, V, G = _f32(q), _f32(K), _f32(V), _f32(G)
    N, d = K.shape
    dq = np.empty(d); dK = np.empty((N, d)); dV = np.empty((N, d)); ds = np.empty(N)
    _load().oracle_backward_bruteforce(_p32(q), _p32(K), _p32(V), _p32(G), N, d, _p64(dq),
                                       _p64(dK), _p64(dV), _p64(ds))
    return dq, dK, dV, ds


def backward(q, K, V, G):
    """The same gradients by backward suffix sums, O(N d).
    Returns (dq [d], dK [N,d], dV [N,d], ds [N]) in float64."""
    q, K, V, G = _f32(q), _f32(K), _f32(V), _f32(G)
    N, d = K.shape
    dq = np.empty(d); dK = np.empty((N, d)); dV = np.empty((N, d)); ds = np.empty(N)
    if _load().oracle_backward(_p32(q), _p32(K), _p32(V), _p32(G), N, d, _p64(dq), _p64(dK),
                               _p64(dV), _p64(ds)) != 0:
        raise MemoryError("oracle_backward: allocation failed")
    return dq, dK, dV, ds


def backward_heads(q, K, V, G, threads=1):
    """backward() for independent heads: q [BH,d], K/V/G [BH,N,d].
    Returns (dq [BH,d], dK, dV [BH,N,d], ds [BH,N])."""
    q, K, V, G = _f32(q), _f32(K), _f32(V), _f32(G)
    BH, N, d = K.shape
    dq = np.empty((BH, d)); dK = np.empty((BH, N, d)); dV = np.empty((BH, N, d))
    ds = np.empty((BH, N))

    def one(h):
        dq[h], dK[h], dV[h], ds[h] = backward(q[h], K[h], V[h], G[h])

    if threads <= 1:
        for h in range(BH):
            one(h)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, range(BH)))
    return dq, dK, dV, ds


def scan_heads(q, K, V, threads=1, want_O=True):
    """Independent heads: q [BH, d], K/V [BH, N, d].  Each head is one call of
    scan(); with threads > 1 the heads run on a thread pool (ctypes releases
    the GIL during the call).  Returns (O [BH,N,d] or None, m [BH], u [BH,d],
    w [BH])."""
    q, K, V = _f32(q), _f32(K), _f32(V)
    BH, N, d = K.shape
    O = np.empty((BH, N, d), dtype=np.float64) if want_O else None
    m = np.empty(BH); w = np.empty(BH); u = np.empty((BH, d))

    def one(h):
        o_h, m[h], u[h], w[h] = scan(q[h], K[h], V[h], want_O=want_O)
        if want_O:
            O[h] = o_h

    if threads <= 1:
        for h in range(BH):
            one(h)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, range(BH)))
    return O, m, u, w


def _opt64(a):
    return None if a is None else _p64(a)


def la_bruteforce(Q, K, V, M):
    """Causal cos-re-weighted linear attention from its definition, O(N^2 d):
    o_i = sum_{j<=i} s_ij v_j / sum_{j<=i} s_ij with
    s_ij = relu(Q_i) . relu(K_j) cos(pi/2 (i - j) / M).  Returns O [N,d]."""
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    N, d = K.shape
    O = np.empty((N, d))
    _load().oracle_la_bruteforce(_p32(Q), _p32(K), _p32(V), N, d, float(M), _p64(O))
    return O


def la_scan(Q, K, V, M, init=None, pos0=0, want_O=True, out=None):
    """The same output by the decomposed prefix sums, O(N d^2).  init =
    (Sc, Ss, zc, zs) continues a scan whose last token had position pos0.
    Returns (O [N,d] or None, (Sc [d,d], Ss [d,d], zc [d], zs [d])).  `out`
    (optional, float64 C-contiguous [N, d]) receives O in place of a fresh
    array."""
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    N, d = K.shape
    if out is not None:
        if out.dtype != np.float64 or out.shape != (N, d) or not out.flags.c_contiguous:
            raise ValueError("out must be a C-contiguous float64 array of shape [N, d]")
        O = out
    else:
        O = np.empty((N, d)) if want_O else None
    Sc = np.empty((d, d)); Ss = np.empty((d, d)); zc = np.empty(d); zs = np.empty(d)
    ini = [None] * 4 if init is None else [_f64(x) for x in init]
    if _load().oracle_la_scan(_p32(Q), _p32(K), _p32(V), N, d, float(M), int(pos0),
                              *(_opt64(x) for x in ini), _opt64(O), _p64(Sc), _p64(Ss),
                              _p64(zc), _p64(zs)) != 0:
        raise MemoryError("oracle_la_scan: allocation failed")
    return O, (Sc, Ss, zc, zs)


def la_heads(Q, K, V, M, threads=1, want_O=True):
    """la_scan() for independent heads: Q/K/V [BH,N,d].  Returns (O [BH,N,d]
    or None, (Sc [BH,d,d], Ss [BH,d,d], zc [BH,d], zs [BH,d]))."""
    Q, K, V = _f32(Q), _f32(K), _f32(V)
    BH, N, d = K.shape
    O = np.empty((BH, N, d)) if want_O else None
    Sc = np.empty((BH, d, d)); Ss = np.empty((BH, d, d)); zc = np.empty((BH, d))
    zs = np.empty((BH, d))

    def one(h):
        o, (Sc[h], Ss[h], zc[h], zs[h]) = la_scan(Q[h], K[h], V[h], M, want_O=want_O)
        if want_O:
            O[h] = o

    if threads <= 1:
        for h in range(BH):
            one(h)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(one, range(BH)))
    return O, (Sc, Ss, zc, zs)


def lib_path():
    return os.path.abspath(_build.LIB)
