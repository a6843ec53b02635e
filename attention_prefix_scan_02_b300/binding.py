"""Python binding of libaaren: the C ABI of include/aaren.h under the same
names, taking torch tensors.

This module only marshals arguments (checks dtypes, shapes, devices and
contiguity, passes data pointers and the current CUDA stream) and turns
error codes into exceptions.  Every step of the computation runs in the
library's CUDA kernels; there is no CPU fallback: if libaaren.so is missing
or fails to load, every call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libaaren.so")
CHECKED_LIB_PATH = os.path.join(_HERE, "libaaren_checked.so")   # -DAAREN_CHECKED build

AAREN_OK = 0
AAREN_ERR_INVALID = 1
AAREN_ERR_UNSUPPORTED = 2
AAREN_ERR_CUDA = 3
AAREN_ERR_LOOKBACK_TIMEOUT = 4
AAREN_ERR_BOUNDS = 5
AAREN_ERR_LOAD_TIMEOUT = 6
AAREN_ERR_WORKSPACE = 7

AAREN_F32 = 0
AAREN_BF16 = 1
AAREN_BF16_F32OUT = 2

# every symbol include/aaren.h declares
EXPORTS = (
    "aaren_scan_forward", "aaren_scan_forward_ex", "aaren_scan_workspace_bytes",
    "aaren_state_init", "aaren_step", "aaren_check", "aaren_status_string",
    "aaren_abi_version", "aaren_debug_set_fault", "aaren_scan_chunk_tokens",
    "aaren_scan_forward_noalloc", "aaren_scan_reduce", "aaren_reduce_workspace_bytes",
    "aaren_scan_forward_stats", "aaren_scan_backward", "aaren_backward_workspace_bytes",
    "aaren_linattn_forward", "aaren_debug_drop_arrival", "aaren_backward_chunk_tokens",
    "aaren_checked_build", "aaren_debug_bounds_probe",
)

# size of the fixed device scratch of aaren_scan_forward_noalloc (include/aaren.h)
AAREN_NOALLOC_SCRATCH_BYTES = 16 * 1024 * 1024

_lib = None

_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32


class AarenError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} (status {code})")


def load(path: str | None = None):
    """Load libaaren.so (once) and declare its signatures.  Raises if absent."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libaaren.so not found at {p}: build it with "
            "`python -m attention_prefix_scan_02_b300.build` (no CPU fallback exists)")
    lib = ctypes.CDLL(p)
    lib.aaren_scan_forward.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32, _vp]
    lib.aaren_scan_forward.restype = _i32
    lib.aaren_scan_forward_ex.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32,
                                          _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.aaren_scan_forward_ex.restype = _i32
    lib.aaren_scan_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64]
    lib.aaren_scan_workspace_bytes.restype = ctypes.c_size_t
    lib.aaren_state_init.argtypes = [_vp, _vp, _vp, _i64, _i64, _vp]
    lib.aaren_state_init.restype = _i32
    lib.aaren_step.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp]
    lib.aaren_step.restype = _i32
    lib.aaren_check.argtypes = [_vp]
    lib.aaren_check.restype = _i32
    lib.aaren_status_string.argtypes = [_i32]
    lib.aaren_status_string.restype = ctypes.c_char_p
    lib.aaren_abi_version.argtypes = []
    lib.aaren_abi_version.restype = _i32
    lib.aaren_debug_set_fault.argtypes = [_i64, _i64]
    lib.aaren_debug_set_fault.restype = _i32
    lib.aaren_scan_chunk_tokens.argtypes = [_i64, _i32]
    lib.aaren_scan_chunk_tokens.restype = _i64
    lib.aaren_debug_drop_arrival.argtypes = [_i64]
    lib.aaren_debug_drop_arrival.restype = _i32
    lib.aaren_backward_chunk_tokens.argtypes = [_i64, _i32]
    lib.aaren_backward_chunk_tokens.restype = _i64
    lib.aaren_checked_build.argtypes = []
    lib.aaren_checked_build.restype = _i32
    lib.aaren_debug_bounds_probe.argtypes = [_i64]
    lib.aaren_debug_bounds_probe.restype = _i32
    lib.aaren_scan_forward_noalloc.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32, _vp]
    lib.aaren_scan_forward_noalloc.restype = _i32
    lib.aaren_scan_reduce.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32,
                                      _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_size_t, _vp]
    lib.aaren_scan_reduce.restype = _i32
    lib.aaren_reduce_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64]
    lib.aaren_reduce_workspace_bytes.restype = ctypes.c_size_t
    lib.aaren_scan_forward_stats.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, _i32,
                                             _vp, ctypes.c_size_t, _vp]
    lib.aaren_scan_forward_stats.restype = _i32
    lib.aaren_scan_backward.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i64, _i64,
                                        _i64, _i64, _i32, _vp, ctypes.c_size_t, _vp]
    lib.aaren_scan_backward.restype = _i32
    lib.aaren_backward_workspace_bytes.argtypes = [_i64, _i64, _i64, _i64]
    lib.aaren_backward_workspace_bytes.restype = ctypes.c_size_t
    lib.aaren_linattn_forward.argtypes = [_vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64, ctypes.c_double,
                                          _i64, _i32, _vp, _vp, _vp, _vp, _vp]
    lib.aaren_linattn_forward.restype = _i32
    if path is None:
        _lib = lib
    return lib


@contextlib.contextmanager
def using_library(path: str):
    """Route every call of this module to another build of the library (the
    tests run the checked build, libaaren_checked.so, this way)."""
    global _lib
    prev = _lib
    _lib = load(path)
    try:
        yield _lib
    finally:
        _lib = prev


def status_string(code: int) -> str:
    return load().aaren_status_string(int(code)).decode()


def _raise(code: int, where: str):
    if code != AAREN_OK:
        raise AarenError(code, where)


def _stream_handle(stream) -> int | None:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream or None
    return int(stream) or None


def _ptr(t: torch.Tensor | None) -> int | None:
    return None if t is None else (t.data_ptr() or None)


def dtype_code(in_dtype: torch.dtype, out_dtype: torch.dtype) -> int:
    if in_dtype == torch.float32 and out_dtype == torch.float32:
        return AAREN_F32
    if in_dtype == torch.bfloat16 and out_dtype == torch.bfloat16:
        return AAREN_BF16
    if in_dtype == torch.bfloat16 and out_dtype == torch.float32:
        return AAREN_BF16_F32OUT
    raise ValueError(f"unsupported dtype pair: inputs {in_dtype}, output {out_dtype}")


def _check_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda:
            raise ValueError("tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError("tensors must be contiguous")


def _check_state(m, u, w, n, d):
    given = [x is not None for x in (m, u, w)]
    if any(given) and not all(given):
        raise ValueError("a state is given as all of (m, u, w) or none")
    if all(given):
        _check_cuda(m, u, w)
        for x in (m, u, w):
            if x.dtype != torch.float32:
                raise ValueError("state tensors are float32")
        if m.numel() != n or w.numel() != n or u.numel() != n * d:
            raise ValueError("state shapes must be m [n], u [n, d], w [n]")


def aaren_scan_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().aaren_scan_workspace_bytes(B, H, N, d))


def aaren_scan_chunk_tokens(d: int, dtype: int) -> int:
    return int(load().aaren_scan_chunk_tokens(d, dtype))


def aaren_backward_chunk_tokens(d: int, dtype: int) -> int:
    return int(load().aaren_backward_chunk_tokens(d, dtype))


def aaren_scan_forward(q, K, V, O, stream=None):
    """O[b,h,t] = softmax-weighted mean of V[b,h,:t+1] with weights e^{q.k}.
    q [B,H,d], K/V/O [B,H,N,d]; O is written."""
    return aaren_scan_forward_ex(q, K, V, O, stream=stream)


def aaren_scan_forward_ex(q, K, V, O, m_in=None, u_in=None, w_in=None, m_out=None,
                          u_out=None, w_out=None, workspace=None, stream=None):
    """aaren_scan_forward with optional starting state (m_in, u_in, w_in), final
    state (m_out, u_out, w_out) and a caller workspace (a CUDA uint8 tensor of
    at least aaren_scan_workspace_bytes bytes)."""
    lib = load()
    if K.dim() != 4:
        raise ValueError("K must be [B, H, N, d]")
    B, H, N, d = K.shape
    if tuple(V.shape) != (B, H, N, d) or tuple(O.shape) != (B, H, N, d):
        raise ValueError("K, V and O must have the same shape [B, H, N, d]")
    if tuple(q.shape) != (B, H, d):
        raise ValueError("q must be [B, H, d]")
    if q.dtype != K.dtype or V.dtype != K.dtype:
        raise ValueError("q, K and V must share one dtype")
    _check_cuda(q, K, V, O, workspace)
    _check_state(m_in, u_in, w_in, B * H, d)
    _check_state(m_out, u_out, w_out, B * H, d)
    code = dtype_code(K.dtype, O.dtype)
    ws_bytes = 0
    if workspace is not None:
        ws_bytes = workspace.numel() * workspace.element_size()
    rc = lib.aaren_scan_forward_ex(
        _ptr(q), _ptr(K), _ptr(V), _ptr(O), B, H, N, d, code,
        _ptr(m_in), _ptr(u_in), _ptr(w_in), _ptr(m_out), _ptr(u_out), _ptr(w_out),
        _ptr(workspace), ws_bytes, _stream_handle(stream))
    _raise(rc, "aaren_scan_forward_ex")
    return O


def aaren_scan_forward_noalloc(q, K, V, O, stream=None):
    """aaren_scan_forward without any device allocation: the carry workspace is
    the library's fixed device array (see include/aaren.h for the limit and
    the rule that calls overlapping on the GPU race)."""
    lib = load()
    if K.dim() != 4 or tuple(V.shape) != tuple(K.shape) or tuple(O.shape) != tuple(K.shape):
        raise ValueError("K, V and O must have the same shape [B, H, N, d]")
    B, H, N, d = K.shape
    if tuple(q.shape) != (B, H, d) or q.dtype != K.dtype or V.dtype != K.dtype:
        raise ValueError("q must be [B, H, d] and share the dtype of K and V")
    _check_cuda(q, K, V, O)
    rc = lib.aaren_scan_forward_noalloc(_ptr(q), _ptr(K), _ptr(V), _ptr(O), B, H, N, d,
                                        dtype_code(K.dtype, O.dtype), _stream_handle(stream))
    _raise(rc, "aaren_scan_forward_noalloc")
    return O


def aaren_reduce_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().aaren_reduce_workspace_bytes(B, H, N, d))


def aaren_scan_reduce(q, K, V, o_last=None, m_in=None, u_in=None, w_in=None, m_out=None,
                      u_out=None, w_out=None, workspace=None, stream=None):
    """Many-to-one output: o_last [B*H, d] = o_N of each head (or None), and
    the final state (m_out, u_out, w_out) when given; no per-token output.
    q [B,H,d], K/V [B,H,N,d]; optional starting state (m_in, u_in, w_in)."""
    lib = load()
    if K.dim() != 4 or tuple(V.shape) != tuple(K.shape):
        raise ValueError("K and V must have the same shape [B, H, N, d]")
    B, H, N, d = K.shape
    if tuple(q.shape) != (B, H, d) or q.dtype != K.dtype or V.dtype != K.dtype:
        raise ValueError("q must be [B, H, d] and share the dtype of K and V")
    if o_last is not None and o_last.numel() != B * H * d:
        raise ValueError("o_last must hold [B*H, d]")
    _check_cuda(q, K, V, o_last, workspace)
    _check_state(m_in, u_in, w_in, B * H, d)
    _check_state(m_out, u_out, w_out, B * H, d)
    code = dtype_code(K.dtype, o_last.dtype if o_last is not None else
                      (torch.float32 if K.dtype == torch.float32 else torch.bfloat16))
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.aaren_scan_reduce(
        _ptr(q), _ptr(K), _ptr(V), _ptr(o_last), B, H, N, d, code,
        _ptr(m_in), _ptr(u_in), _ptr(w_in), _ptr(m_out), _ptr(u_out), _ptr(w_out),
        _ptr(workspace), ws_bytes, _stream_handle(stream))
    _raise(rc, "aaren_scan_reduce")
    return o_last


def aaren_backward_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(load().aaren_backward_workspace_bytes(B, H, N, d))


def aaren_scan_forward_stats(q, K, V, O, stats, workspace=None, stream=None):
    """aaren_scan_forward that also writes stats [B,H,N,2] float32: the
    (m_t, w_t) of every prefix, which aaren_scan_backward needs."""
    lib = load()
    B, H, N, d = K.shape
    if tuple(V.shape) != (B, H, N, d) or tuple(O.shape) != (B, H, N, d) or tuple(q.shape) != (B, H, d):
        raise ValueError("q [B,H,d], K/V/O [B,H,N,d]")
    if stats.dtype != torch.float32 or stats.numel() != B * H * N * 2:
        raise ValueError("stats must be float32 [B, H, N, 2]")
    _check_cuda(q, K, V, O, stats, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.aaren_scan_forward_stats(_ptr(q), _ptr(K), _ptr(V), _ptr(O), _ptr(stats), B, H, N, d,
                                      dtype_code(K.dtype, O.dtype), _ptr(workspace), ws_bytes,
                                      _stream_handle(stream))
    _raise(rc, "aaren_scan_forward_stats")
    return O, stats


def aaren_scan_backward(q, K, V, O, dO, stats, dq, dK, dV, workspace=None, stream=None):
    """Gradients dq [B*H,d], dK, dV [B,H,N,d] (float32, written) of the
    many-to-many output, given its upstream gradient dO and the forward's
    O and stats."""
    lib = load()
    B, H, N, d = K.shape
    for t in (V, O, dO, dK, dV):
        if tuple(t.shape) != (B, H, N, d):
            raise ValueError("K, V, O, dO, dK, dV must be [B, H, N, d]")
    if tuple(q.shape) != (B, H, d) or dq.numel() != B * H * d:
        raise ValueError("q must be [B, H, d] and dq hold [B*H, d]")
    if O.dtype != dO.dtype:
        raise ValueError("O and dO share the output dtype")
    for t in (dq, dK, dV, stats):
        if t.dtype != torch.float32:
            raise ValueError("gradients and stats are float32")
    _check_cuda(q, K, V, O, dO, stats, dq, dK, dV, workspace)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = lib.aaren_scan_backward(_ptr(q), _ptr(K), _ptr(V), _ptr(O), _ptr(dO), _ptr(stats),
                                 _ptr(dq), _ptr(dK), _ptr(dV), B, H, N, d,
                                 dtype_code(K.dtype, O.dtype), _ptr(workspace), ws_bytes,
                                 _stream_handle(stream))
    _raise(rc, "aaren_scan_backward")
    return dq, dK, dV


def aaren_state_init(m, u, w, stream=None):
    """Identity state (-inf, 0, 0): m [n], u [n, d], w [n] (float32)."""
    n, d = u.shape
    _check_state(m, u, w, n, d)
    rc = load().aaren_state_init(_ptr(m), _ptr(u), _ptr(w), n, d, _stream_handle(stream))
    _raise(rc, "aaren_state_init")


def aaren_step(q, m, u, w, k_t, v_t, o_t, stream=None):
    """One token per stream: q, k_t, v_t, o_t [n, d]; state m [n], u [n, d], w [n]
    updated in place; o_t written."""
    n, d = k_t.shape
    for t in (q, v_t, o_t):
        if tuple(t.shape) != (n, d):
            raise ValueError("q, k_t, v_t and o_t must be [n, d]")
    if q.dtype != k_t.dtype or v_t.dtype != k_t.dtype:
        raise ValueError("q, k_t and v_t must share one dtype")
    _check_cuda(q, k_t, v_t, o_t)
    _check_state(m, u, w, n, d)
    code = dtype_code(k_t.dtype, o_t.dtype)
    rc = load().aaren_step(_ptr(q), _ptr(m), _ptr(u), _ptr(w), _ptr(k_t), _ptr(v_t),
                           _ptr(o_t), n, d, code, _stream_handle(stream))
    _raise(rc, "aaren_step")


def aaren_check(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status."""
    return int(load().aaren_check(_stream_handle(stream)))


def aaren_debug_set_fault(never_publish_chunk: int = -1, wait_limit_ns: int = 0):
    _raise(load().aaren_debug_set_fault(never_publish_chunk, wait_limit_ns),
           "aaren_debug_set_fault")


def aaren_debug_drop_arrival(chunk: int = -1):
    _raise(load().aaren_debug_drop_arrival(chunk), "aaren_debug_drop_arrival")


def aaren_debug_bounds_probe(offset: int = 0):
    _raise(load().aaren_debug_bounds_probe(offset), "aaren_debug_bounds_probe")


def aaren_checked_build() -> bool:
    return bool(load().aaren_checked_build())


def aaren_abi_version() -> int:
    return int(load().aaren_abi_version())


# ---- conveniences (allocation + the calls above) ---------------------------

def scan_forward(q, K, V, out_dtype=None, init=None, return_state=False, workspace=None,
                 stream=None):
    """Allocate O (and the final state when asked) and run aaren_scan_forward_ex.
    init = (m, u, w) starting state or None.  Returns O, or (O, (m, u, w))."""
    out_dtype = out_dtype or K.dtype
    O = torch.empty(K.shape, dtype=out_dtype, device=K.device)
    B, H, N, d = K.shape
    m_in = u_in = w_in = None
    if init is not None:
        m_in, u_in, w_in = init
    m_out = u_out = w_out = None
    if return_state:
        m_out = torch.empty(B * H, dtype=torch.float32, device=K.device)
        u_out = torch.empty(B * H, d, dtype=torch.float32, device=K.device)
        w_out = torch.empty(B * H, dtype=torch.float32, device=K.device)
    aaren_scan_forward_ex(q, K, V, O, m_in, u_in, w_in, m_out, u_out, w_out, workspace, stream)
    return (O, (m_out, u_out, w_out)) if return_state else O


def scan_reduce(q, K, V, out_dtype=None, init=None, return_state=False, workspace=None,
                stream=None):
    """Allocate o_N [B, H, d] (and the final state when asked) and run
    aaren_scan_reduce.  Returns o_N, or (o_N, (m, u, w))."""
    out_dtype = out_dtype or K.dtype
    B, H, N, d = K.shape
    o = torch.empty(B, H, d, dtype=out_dtype, device=K.device)
    m_in = u_in = w_in = None
    if init is not None:
        m_in, u_in, w_in = init
    m_out = u_out = w_out = None
    if return_state:
        m_out = torch.empty(B * H, dtype=torch.float32, device=K.device)
        u_out = torch.empty(B * H, d, dtype=torch.float32, device=K.device)
        w_out = torch.empty(B * H, dtype=torch.float32, device=K.device)
    aaren_scan_reduce(q, K, V, o, m_in, u_in, w_in, m_out, u_out, w_out, workspace, stream)
    return (o, (m_out, u_out, w_out)) if return_state else o


def new_reduce_workspace(B, H, N, d, device="cuda"):
    nbytes = aaren_reduce_workspace_bytes(B, H, N, d)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def scan_forward_train(q, K, V, out_dtype=None, stream=None):
    """Forward for a later backward: returns (O, stats)."""
    out_dtype = out_dtype or K.dtype
    B, H, N, d = K.shape
    O = torch.empty(K.shape, dtype=out_dtype, device=K.device)
    stats = torch.empty(B, H, N, 2, dtype=torch.float32, device=K.device)
    return aaren_scan_forward_stats(q, K, V, O, stats, stream=stream)


def scan_backward(q, K, V, O, dO, stats, workspace=None, stream=None):
    """Allocate and return (dq [B,H,d], dK, dV [B,H,N,d]) in float32."""
    B, H, N, d = K.shape
    dq = torch.empty(B, H, d, dtype=torch.float32, device=K.device)
    dK = torch.empty(K.shape, dtype=torch.float32, device=K.device)
    dV = torch.empty(K.shape, dtype=torch.float32, device=K.device)
    aaren_scan_backward(q, K, V, O, dO, stats, dq, dK, dV, workspace, stream)
    return dq, dK, dV


def new_backward_workspace(B, H, N, d, device="cuda"):
    nbytes = aaren_backward_workspace_bytes(B, H, N, d)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def new_workspace(B, H, N, d, device="cuda"):
    nbytes = aaren_scan_workspace_bytes(B, H, N, d)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def aaren_linattn_forward(Q, K, V, O, M, pos0=0, S_in=None, z_in=None, S_out=None, z_out=None,
                          stream=None):
    """Causal cos-re-weighted linear attention (include/aaren.h):
    Q, K, V [B,H,N,64] bfloat16, O [B,H,N,64] bfloat16 or float32; states
    S [B,H,2,64,64], z [B,H,2,64] float32 (or None)."""
    _check_cuda(Q, K, V, O, S_in, z_in, S_out, z_out)
    if Q.dim() != 4 or Q.shape != K.shape or K.shape != V.shape or O.shape != K.shape:
        raise ValueError("Q, K, V, O must all be [B, H, N, d]")
    if not (Q.dtype == K.dtype == V.dtype):
        raise ValueError("Q, K, V must share a dtype")
    B, H, N, d = K.shape
    for S, z in ((S_in, z_in), (S_out, z_out)):
        if (S is None) != (z is None):
            raise ValueError("a state is given as both of (S, z) or neither")
        if S is not None:
            if S.dtype != torch.float32 or z.dtype != torch.float32:
                raise ValueError("state tensors are float32")
            if S.numel() != B * H * 2 * d * d or z.numel() != B * H * 2 * d:
                raise ValueError("state shapes must be S [B,H,2,d,d], z [B,H,2,d]")
    rc = load().aaren_linattn_forward(_ptr(Q), _ptr(K), _ptr(V), _ptr(O), B, H, N, d, float(M),
                                      int(pos0), dtype_code(K.dtype, O.dtype), _ptr(S_in),
                                      _ptr(z_in), _ptr(S_out), _ptr(z_out), _stream_handle(stream))
    _raise(rc, "aaren_linattn_forward")
    return O


def linattn_forward(Q, K, V, M=None, out_dtype=None, init=None, pos0=0, return_state=False,
                    stream=None):
    """Allocate O (and the final state when asked) and run
    aaren_linattn_forward.  M defaults to the sequence length pos0 + N
    (at least 1).
    Returns O, or (O, (S, z))."""
    out_dtype = out_dtype or K.dtype
    B, H, N, d = K.shape
    M = float(max(pos0 + N, 1)) if M is None else float(M)
    O = torch.empty(K.shape, dtype=out_dtype, device=K.device)
    S_in = z_in = S_out = z_out = None
    if init is not None:
        S_in, z_in = init
    if return_state:
        S_out = torch.empty(B, H, 2, d, d, dtype=torch.float32, device=K.device)
        z_out = torch.empty(B, H, 2, d, dtype=torch.float32, device=K.device)
    aaren_linattn_forward(Q, K, V, O, M, pos0, S_in, z_in, S_out, z_out, stream)
    return (O, (S_out, z_out)) if return_state else O
