"""The allocation-free scan entry point (aaren_scan_forward_noalloc).

Callers that must not allocate device memory (their GPU memory belongs to
another allocator, or they cannot risk an allocator call in a latency-critical
loop) use this entry point; its carry workspace is a fixed array inside the
library.  The GPU test calls it through the C ABI twice in a row -- the second
call finds the first call's leftovers in the shared array -- and compares each
result with the regular aaren_scan_forward at the tolerances of the other
parity tests.  This file is collected last so that a run stopping at the first
failure has run every other test before it; it also passes on its own in a
fresh process.
"""
import ctypes
import os
import re

import pytest
import torch

from attention_prefix_scan_02_b300 import binding, inputs
from tests.parity import TOL_BF16, TOL_F32, rowwise_rel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_scratch_size_matches_the_header():
    text = open(os.path.join(ROOT, "include", "aaren.h")).read()
    m = re.search(r"#define AAREN_NOALLOC_SCRATCH_BYTES \((\d+)u \* (\d+)u \* (\d+)u\)", text)
    assert m is not None
    assert int(m.group(1)) * int(m.group(2)) * int(m.group(3)) == binding.AAREN_NOALLOC_SCRATCH_BYTES


def _call(lib, q, K, V, O, code):
    B, H, N, d = K.shape
    stream = torch.cuda.current_stream().cuda_stream or None
    return lib.aaren_scan_forward_noalloc(q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(),
                                          B, H, N, d, code, stream)


@pytest.mark.gpu
@pytest.mark.parametrize("case", ["bf16_f32out", "f32_ragged"])
def test_noalloc_matches_the_regular_scan_on_two_calls(case):
    lib = binding.load()
    if case == "bf16_f32out":
        wl = inputs.custom(2, 4, 3000, 128, dtype="bf16", seed=123)
        out_t, code, tol = torch.float32, binding.AAREN_BF16_F32OUT, TOL_BF16
    else:
        wl = inputs.custom(3, 2, 1000 + 37, 64, dtype="f32", seed=124)
        out_t, code, tol = torch.float32, binding.AAREN_F32, TOL_F32
    assert binding.aaren_scan_workspace_bytes(wl.B, wl.H, wl.N, wl.d) <= \
        binding.AAREN_NOALLOC_SCRATCH_BYTES
    q, K, V = inputs.batch_inputs(wl, device="cuda")
    O_ref = torch.empty(K.shape, dtype=out_t, device="cuda")
    binding.aaren_scan_forward(q, K, V, O_ref)
    assert binding.aaren_check() == binding.AAREN_OK
    for _ in range(2):
        O = torch.full(K.shape, float("nan"), dtype=out_t, device="cuda")
        assert _call(lib, q, K, V, O, code) == binding.AAREN_OK
        assert binding.aaren_check() == binding.AAREN_OK
        assert torch.isfinite(O).all()
        assert rowwise_rel(O.cpu(), O_ref.cpu().numpy()) <= tol


@pytest.mark.gpu
def test_noalloc_rejects_problems_beyond_its_scratch():
    lib = binding.load()
    B, H, N, d = 1, 64, 1 << 20, 128
    assert binding.aaren_scan_workspace_bytes(B, H, N, d) > binding.AAREN_NOALLOC_SCRATCH_BYTES
    # distinct, aligned addresses that are never dereferenced: the size check
    # rejects the call on the host before anything is launched
    elems = B * H * N * d * 2
    base = 1 << 44
    ptrs = [ctypes.c_void_p(base + i * (elems + 4096)) for i in range(4)]
    rc = lib.aaren_scan_forward_noalloc(*ptrs, B, H, N, d, binding.AAREN_BF16, None)
    assert rc == binding.AAREN_ERR_WORKSPACE
    assert binding.aaren_check() == binding.AAREN_OK
