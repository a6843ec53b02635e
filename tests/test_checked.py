"""The bounds-checked build of the library (libaaren_checked.so, the same
source compiled with -DAAREN_CHECKED), in place of a memory checker.

In that build every kernel tests each extent it computes -- rows of a global
tensor, a workspace slot, a bulk or tensor copy, a shared-memory stage --
against its buffer before the access; a violation skips the access and makes
aaren_check report AAREN_ERR_BOUNDS.  The guard bands of test_guard.py see
writes past a buffer; these checks also cover reads.  Here the ragged-length
parity cases of every entry point (lengths that end inside a chunk or a
tile, every d and dtype) and the guard-band cases run against the checked
build: each must give the same results and report no violation.  A probe
shifts the index one check tests (never an address) to show that a
violation is reported and its accesses are skipped."""
import os

import pytest
import torch

from attention_prefix_scan_02_b300 import binding, build
from tests import test_backward, test_edge, test_guard, test_linattn, test_reduce, test_step


def test_checked_library_is_built_and_exports_the_abi():
    """Host only: the checked build exists beside the regular one and says so."""
    build.build_checked()
    assert os.path.exists(binding.CHECKED_LIB_PATH)
    with binding.using_library(binding.CHECKED_LIB_PATH):
        assert binding.aaren_checked_build()
        assert binding.aaren_abi_version() == 2
    assert not binding.aaren_checked_build()


@pytest.fixture
def checked():
    """Route the binding to the checked library for one test; afterwards no
    violation (or any other device status) may be pending."""
    with binding.using_library(binding.CHECKED_LIB_PATH):
        yield
        assert binding.aaren_check() == binding.AAREN_OK


DT3 = ["f32", "bf16", "bf16_f32out"]


@pytest.mark.gpu
@pytest.mark.parametrize("dt", DT3)
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_scan_ragged_lengths(checked, d, dt):
    test_edge.test_ragged_lengths(d, dt)


@pytest.mark.gpu
def test_scan_many_short_heads(checked):
    test_edge.test_many_short_heads()


@pytest.mark.gpu
@pytest.mark.parametrize("dt", ["f32", "bf16_f32out"])
def test_scan_continuation(checked, dt):
    test_edge.test_continuation_from_a_saved_state(dt)


@pytest.mark.gpu
@pytest.mark.parametrize("dt", DT3)
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_reduce_ragged_lengths(checked, d, dt):
    test_reduce.test_ragged_lengths(d, dt)


@pytest.mark.gpu
@pytest.mark.parametrize("dt", DT3)
@pytest.mark.parametrize("d", [16, 64, 128])
def test_backward_ragged_lengths(checked, d, dt):
    test_backward.test_ragged_lengths(d, dt)


@pytest.mark.gpu
@pytest.mark.parametrize("dt", DT3)
@pytest.mark.parametrize("d", [16, 64, 128])
def test_step_shapes(checked, d, dt):
    test_step.test_step_all_shapes(d, dt)


@pytest.mark.gpu
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_linattn_ragged_lengths(checked, out):
    test_linattn.test_ragged_lengths(out)


@pytest.mark.gpu
def test_linattn_continuation(checked):
    test_linattn.test_continuation_from_a_state()


@pytest.mark.gpu
@pytest.mark.parametrize("io", test_guard.DTYPES, ids=DT3)
@pytest.mark.parametrize("d", [16, 128])
def test_guard_bands(checked, d, io):
    test_guard.test_scan_forward_writes_stay_in_bounds(d, io)
    test_guard.test_reduce_writes_stay_in_bounds(d, io)
    test_guard.test_step_writes_stay_in_bounds(d, io)
    if d == 128:
        test_guard.test_backward_writes_stay_in_bounds(d, io)


@pytest.mark.gpu
@pytest.mark.parametrize("out_t", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_guard_bands_linattn(checked, out_t):
    test_guard.test_linattn_writes_stay_in_bounds(out_t)


def _probe_step(n=40, d=64):
    q = torch.randn(n, d, device="cuda")
    k = torch.randn(n, d, device="cuda")
    v = torch.randn(n, d, device="cuda")
    o = torch.full((n, d), float("nan"), device="cuda")
    m = torch.empty(n, device="cuda"); u = torch.empty(n, d, device="cuda"); w = torch.empty(n, device="cuda")
    binding.aaren_state_init(m, u, w)
    assert binding.aaren_check() == binding.AAREN_OK
    try:
        binding.aaren_debug_bounds_probe(n)   # every stream's index tests as out of range
        binding.aaren_step(q, m, u, w, k, v, o)
        rc = binding.aaren_check()
    finally:
        binding.aaren_debug_bounds_probe(0)
    return rc, o, m, u, w


@pytest.mark.gpu
def test_a_violation_is_reported_and_its_access_skipped():
    with binding.using_library(binding.CHECKED_LIB_PATH):
        rc, o, m, u, w = _probe_step()
        assert rc == binding.AAREN_ERR_BOUNDS
        assert torch.isnan(o).all()                      # no output row was written
        assert torch.isinf(m).all() and (w == 0).all() and (u == 0).all()   # state untouched
        assert binding.aaren_check() == binding.AAREN_OK   # the report was cleared
    # the regular build carries no checks: the probe changes nothing there
    rc, o, m, u, w = _probe_step()
    assert rc == binding.AAREN_OK
    assert torch.isfinite(o).all()
