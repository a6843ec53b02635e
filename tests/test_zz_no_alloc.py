"""The allocation-free scan entry point (aaren_scan_forward_noalloc).

Some callers cannot allocate device memory: a plugin or an embedded library
whose host framework owns the GPU's memory and forbids outside cudaMalloc,
or a latency-critical loop that cannot risk an allocator call that may block
or fail when memory is full.  For them the scan's carry workspace is a fixed
array inside the library.  The GPU test calls the entry point through the
C ABI twice in a row (the second call finds the first call's leftovers in the
shared array) and compares each result with the regular aaren_scan_forward
and with the float64 oracle, at the tolerances of the other parity tests.  It
also checks that the calls take nothing from the device's stream-ordered
pool and leave the device's free memory unchanged.  This file is collected
last so that a run stopping at the first failure has run every other test
before it; it also passes on its own in a fresh process.
"""
import ctypes
import os
import re

import pytest
import torch

import oracle
from attention_prefix_scan_02_b300 import binding, inputs
from tests.parity import TOL_BF16, TOL_F32, rowwise_rel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# CUmemPool_attribute values of the CUDA driver API
_POOL_RESERVED_CURRENT = 5
_POOL_USED_HIGH = 8


def test_scratch_size_matches_the_header():
    text = open(os.path.join(ROOT, "include", "aaren.h")).read()
    m = re.search(r"#define AAREN_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", text)
    assert m is not None
    assert int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == binding.AAREN_NOALLOC_SCRATCH_BYTES


def test_noalloc_rejects_oversized_problems_before_any_cuda_call():
    """Host-only: the size check comes first, so null tensors never matter."""
    lib = binding.load()
    B, H, N, d = 1, 64, 1 << 20, 128
    assert binding.aaren_scan_workspace_bytes(B, H, N, d) > binding.AAREN_NOALLOC_SCRATCH_BYTES
    rc = lib.aaren_scan_forward_noalloc(None, None, None, None, B, H, N, d, binding.AAREN_BF16, None)
    assert rc == binding.AAREN_ERR_WORKSPACE
    assert lib.aaren_scan_forward_noalloc(None, None, None, None, 1, 1, 8, 48, binding.AAREN_BF16,
                                          None) == binding.AAREN_ERR_UNSUPPORTED
    assert lib.aaren_scan_forward_noalloc(None, None, None, None, 1, -1, 8, 64, binding.AAREN_BF16,
                                          None) == binding.AAREN_ERR_INVALID


class _DefaultPool:
    """The current device's default stream-ordered memory pool, read through
    the CUDA driver API (the pool cudaMallocAsync draws from)."""

    def __init__(self):
        self.cu = ctypes.CDLL("libcuda.so.1")
        dev = ctypes.c_int()
        assert self.cu.cuDeviceGet(ctypes.byref(dev), torch.cuda.current_device()) == 0
        self.pool = ctypes.c_void_p()
        assert self.cu.cuDeviceGetDefaultMemPool(ctypes.byref(self.pool), dev) == 0

    def get(self, attr):
        v = ctypes.c_uint64()
        assert self.cu.cuMemPoolGetAttribute(self.pool, attr, ctypes.byref(v)) == 0
        return v.value

    def reset_used_high(self):
        zero = ctypes.c_uint64(0)
        assert self.cu.cuMemPoolSetAttribute(self.pool, _POOL_USED_HIGH, ctypes.byref(zero)) == 0


def _call(lib, q, K, V, O, code):
    B, H, N, d = K.shape
    stream = torch.cuda.current_stream().cuda_stream or None
    return lib.aaren_scan_forward_noalloc(q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                          B, H, N, d, code, stream)


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["bf16_f32out", "f32_ragged"])
def test_noalloc_matches_the_regular_scan_and_the_oracle_on_two_calls(case):
    lib = binding.load()
    if case == "bf16_f32out":
        wl = inputs.custom(2, 4, 3000, 128, dtype="bf16", seed=123)
        out_t, code, tol = torch.float32, binding.AAREN_BF16_F32OUT, TOL_BF16
    else:
        wl = inputs.custom(3, 2, 1000 + 37, 64, dtype="f32", seed=124)
        out_t, code, tol = torch.float32, binding.AAREN_F32, TOL_F32
    assert binding.aaren_scan_workspace_bytes(wl.B, wl.H, wl.N, wl.d) <= \
        binding.AAREN_NOALLOC_SCRATCH_BYTES
    qc, Kc, Vc = inputs.batch_inputs(wl)
    q, K, V = qc.cuda(), Kc.cuda(), Vc.cuda()
    f = lambda t: t.float().reshape(-1, *t.shape[2:]).numpy()
    Oref, *_ = oracle.scan_heads(f(qc), f(Kc), f(Vc), threads=inputs.default_threads())
    Oref = Oref.reshape(wl.B, wl.H, wl.N, wl.d)
    O_reg = torch.empty(K.shape, dtype=out_t, device="cuda")
    binding.aaren_scan_forward(q, K, V, O_reg)
    assert binding.aaren_check() == binding.AAREN_OK
    outs = [torch.full(K.shape, float("nan"), dtype=out_t, device="cuda") for _ in range(2)]
    torch.cuda.synchronize()
    pool = _DefaultPool()
    pool.reset_used_high()
    reserved0 = pool.get(_POOL_RESERVED_CURRENT)
    free0, _ = torch.cuda.mem_get_info()
    for O in outs:
        assert _call(lib, q, K, V, O, code) == binding.AAREN_OK
        assert binding.aaren_check() == binding.AAREN_OK
    free1, _ = torch.cuda.mem_get_info()
    assert pool.get(_POOL_USED_HIGH) == 0, "the call drew on the stream-ordered pool"
    assert pool.get(_POOL_RESERVED_CURRENT) == reserved0
    assert free1 == free0, f"device free memory moved by {free0 - free1} bytes"
    for O in outs:
        assert torch.isfinite(O).all()
        assert rowwise_rel(O.cpu(), O_reg.cpu().numpy()) <= tol
        assert rowwise_rel(O.cpu(), Oref) <= tol
