"""Error paths on the GPU: argument errors on real device tensors, and the
bounded cross-block carry wait.

The wait test plants a chunk whose carry is never published (a flag nothing
sets) with a short wait limit: its successors must give up, report
AAREN_ERR_LOOKBACK_TIMEOUT through aaren_check, and leave the context usable
(a following scan is correct).  No GPU fault, trap or hang is involved."""
import time

import pytest
import torch

import oracle
from attention_prefix_scan_02_b300 import binding, inputs
from tests.parity import TOL_F32, rowwise_rel

pytestmark = pytest.mark.gpu


def test_binding_rejects_bad_shapes_and_dtypes():
    q = torch.randn(1, 2, 64, device="cuda")
    K = torch.randn(1, 2, 100, 64, device="cuda")
    with pytest.raises(ValueError):
        binding.aaren_scan_forward(q, K, K.clone(), torch.empty(1, 2, 99, 64, device="cuda"))
    with pytest.raises(ValueError):
        binding.aaren_scan_forward(q.half(), K.half(), K.half(), torch.empty_like(K))
    with pytest.raises(ValueError):
        binding.aaren_scan_forward(q, K.transpose(2, 3), K, K.clone())


def test_abi_rejects_bad_device_arguments():
    lib = binding.load()
    q = torch.randn(1, 2, 64, device="cuda")
    K = torch.randn(1, 2, 101, 64, device="cuda")
    V = torch.randn(1, 2, 101, 64, device="cuda")
    O = torch.empty_like(K)
    args = lambda qq, kk, vv, oo: (qq, kk, vv, oo, 1, 2, 100, 64, binding.AAREN_F32, None)
    ok = lib.aaren_scan_forward(*args(q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr()))
    assert ok == binding.AAREN_OK
    # misaligned K (4 bytes off a 16-byte boundary)
    rc = lib.aaren_scan_forward(*args(q.data_ptr(), K.data_ptr() + 4, V.data_ptr(), O.data_ptr()))
    assert rc == binding.AAREN_ERR_INVALID
    # O aliasing V
    rc = lib.aaren_scan_forward(*args(q.data_ptr(), K.data_ptr(), V.data_ptr(), V.data_ptr() + 256))
    assert rc == binding.AAREN_ERR_INVALID
    # workspace too small, or misaligned
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    rc = lib.aaren_scan_forward_ex(q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), 1, 2, 100,
                                   64, 0, None, None, None, None, None, None, ws.data_ptr(), 16, None)
    assert rc == binding.AAREN_ERR_WORKSPACE
    big = binding.new_workspace(1, 2, 100, 64)
    rc = lib.aaren_scan_forward_ex(q.data_ptr(), K.data_ptr(), V.data_ptr(), O.data_ptr(), 1, 2, 100,
                                   64, 0, None, None, None, None, None, None, big.data_ptr() + 16,
                                   big.numel() - 16, None)
    assert rc == binding.AAREN_ERR_WORKSPACE
    assert binding.aaren_check() == binding.AAREN_OK


def test_carry_wait_gives_up_and_context_survives():
    d = 64
    wl = inputs.custom(1, 2, 40 * 128 + 5, d, seed=5)
    q, K, V = inputs.batch_inputs(wl)
    qg, Kg, Vg = q.cuda(), K.cuda(), V.cuda()
    C = binding.aaren_scan_chunk_tokens(d, binding.AAREN_F32)
    assert C == 128
    try:
        binding.aaren_debug_set_fault(never_publish_chunk=5, wait_limit_ns=20_000_000)
        t0 = time.time()
        binding.scan_forward(qg, Kg, Vg)
        rc = binding.aaren_check()
        elapsed = time.time() - t0
    finally:
        binding.aaren_debug_set_fault(-1, 0)
    assert rc == binding.AAREN_ERR_LOOKBACK_TIMEOUT
    assert elapsed < 10.0
    # the status word was cleared and the context still works
    assert binding.aaren_check() == binding.AAREN_OK
    O = binding.scan_forward(qg, Kg, Vg)
    assert binding.aaren_check() == binding.AAREN_OK
    f = lambda t: t.reshape(-1, *t.shape[2:]).numpy()
    Oref, *_ = oracle.scan_heads(f(q), f(K), f(V))
    assert rowwise_rel(O.cpu().reshape(Oref.shape), Oref) <= TOL_F32
