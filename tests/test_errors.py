"""Error paths on the GPU: argument errors on real device tensors, and every
kind of bounded device wait made to give up.

Each wait test sets a testing hook and a short wait limit (20 ms): a chunk
whose carry is never published (a flag nothing sets), or a barrier arrival
inside a block that is withheld.  The waits on it must give up, report the
right status through aaren_check, and leave the context usable (the next
call matches the oracle).  Covered: the look-back of the persistent scan
and of the one-chunk-per-block scan, the persistent scan's hand-offs inside a
block, the backward pass's look-forward, and the linear attention's
tensor-core pipeline.  No GPU fault, trap or hang is involved: every wait is
bounded and every copy or product in flight is waited for before a block
leaves."""
import os
import time

import pytest
import torch

import oracle
from attention_prefix_scan_02_b300 import binding, inputs
from tests.parity import TOL_BF16, TOL_F32, rowwise_rel

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


def _oracle_check(q, K, V, O, tol):
    f = lambda t: t.float().reshape(-1, *t.shape[2:]).numpy()
    Oref, *_ = oracle.scan_heads(f(q), f(K), f(V))
    assert rowwise_rel(O.cpu().float().reshape(Oref.shape), Oref) <= tol


def _faulted(expected, run, never_publish=-1, drop=-1, limit_ns=20_000_000):
    """Run `run()` with a testing hook set and a short wait limit; return the
    status aaren_check reports and the seconds it took."""
    try:
        binding.aaren_debug_set_fault(never_publish_chunk=never_publish, wait_limit_ns=limit_ns)
        binding.aaren_debug_drop_arrival(drop)
        t0 = time.time()
        run()
        rc = binding.aaren_check()
        elapsed = time.time() - t0
    finally:
        binding.aaren_debug_set_fault(-1, 0)
        binding.aaren_debug_drop_arrival(-1)
    assert rc == expected, binding.status_string(rc)
    assert elapsed < 10.0
    # the status word was cleared and the context still works
    assert binding.aaren_check() == binding.AAREN_OK


# (d, input dtype): which kernel serves it -- float32 d = 64 and every
# bfloat16 size run on the persistent kernel, other float32 sizes on the
# one-chunk-per-block kernel
CARRY_CASES = {"pipe_f32_d64": (64, "f32"), "block_f32_d128": (128, "f32"),
               "pipe_bf16_d128": (128, "bf16")}


@pytest.mark.parametrize("case", sorted(CARRY_CASES))
def test_carry_wait_gives_up_and_context_survives(case):
    """A chunk whose carry is never published: its successors' look-back
    waits give up (AAREN_ERR_LOOKBACK_TIMEOUT), and the next scan is right."""
    d, dt = CARRY_CASES[case]
    code = binding.AAREN_F32 if dt == "f32" else binding.AAREN_BF16_F32OUT
    C = binding.aaren_scan_chunk_tokens(d, code)
    assert C == (64 if case == "block_f32_d128" else 128)
    wl = inputs.custom(1, 2, 40 * C + 5, d, dtype=dt, seed=5)
    q, K, V = inputs.batch_inputs(wl)
    qg, Kg, Vg = q.cuda(), K.cuda(), V.cuda()
    _faulted(binding.AAREN_ERR_LOOKBACK_TIMEOUT,
             lambda: binding.scan_forward(qg, Kg, Vg, out_dtype=torch.float32), never_publish=5)
    O = binding.scan_forward(qg, Kg, Vg, out_dtype=torch.float32)
    assert binding.aaren_check() == binding.AAREN_OK
    _oracle_check(q, K, V, O, TOL_F32 if dt == "f32" else TOL_BF16)


@pytest.mark.parametrize("d,dt", [(128, "bf16"), (64, "f32")])
def test_in_block_hand_off_gives_up_and_context_survives(d, dt):
    """The persistent scan's first compute warp of one chunk withholds its
    aggregate from its group: the group's waits give up
    (AAREN_ERR_LOAD_TIMEOUT; the chunk's successors then also give up on its
    carry), every warp leaves with no copy in flight, and the next scan on
    the same context is right."""
    code = binding.AAREN_F32 if dt == "f32" else binding.AAREN_BF16_F32OUT
    C = binding.aaren_scan_chunk_tokens(d, code)
    wl = inputs.custom(2, 3, 30 * C + 17, d, dtype=dt, seed=6)
    q, K, V = inputs.batch_inputs(wl)
    qg, Kg, Vg = q.cuda(), K.cuda(), V.cuda()
    _faulted(binding.AAREN_ERR_LOAD_TIMEOUT,
             lambda: binding.scan_forward(qg, Kg, Vg, out_dtype=torch.float32), drop=36)
    O = binding.scan_forward(qg, Kg, Vg, out_dtype=torch.float32)
    assert binding.aaren_check() == binding.AAREN_OK
    _oracle_check(q, K, V, O, TOL_F32 if dt == "f32" else TOL_BF16)


@pytest.mark.parametrize("d,dt", [(64, "bf16"), (128, "f32")])
def test_backward_look_forward_gives_up_and_context_survives(d, dt):
    """A backward chunk whose suffix is never published: the chunks before it
    give up their look-forward (AAREN_ERR_LOOKBACK_TIMEOUT); the next
    backward on the same context matches the oracle's gradients."""
    from tests.test_backward import TOL, TOL_DV, grad_errors, upstream
    in_t = torch.bfloat16 if dt == "bf16" else torch.float32
    code = binding.AAREN_BF16_F32OUT if dt == "bf16" else binding.AAREN_F32
    C = binding.aaren_backward_chunk_tokens(d, code)
    assert C > 0
    wl = inputs.custom(1, 2, 25 * C + 9, d, dtype=dt, seed=7)
    q, K, V = inputs.batch_inputs(wl)
    G = upstream(1, 2, wl.N, d, torch.float32, seed=7)
    qg, Kg, Vg, Gg = q.cuda(), K.cuda(), V.cuda(), G.cuda()
    O, stats = binding.scan_forward_train(qg, Kg, Vg, out_dtype=torch.float32)
    assert binding.aaren_check() == binding.AAREN_OK
    _faulted(binding.AAREN_ERR_LOOKBACK_TIMEOUT,
             lambda: binding.scan_backward(qg, Kg, Vg, O, Gg, stats), never_publish=12)
    dq, dK, dV = binding.scan_backward(qg, Kg, Vg, O, Gg, stats)
    assert binding.aaren_check() == binding.AAREN_OK
    f = lambda t: t.float().reshape(-1, *t.shape[2:]).numpy()
    ref = oracle.backward_heads(f(q), f(K), f(V), f(G))
    e_v, e_k, e_q = grad_errors(f(q), f(K), f(V), f(dq.cpu()), f(dK.cpu()), f(dV.cpu()), ref)
    key = "f32" if dt == "f32" else "bf16_f32out"
    assert e_v <= TOL_DV[key] and e_k <= TOL[key] and e_q <= TOL[key]


_LINATTN_CHILD = r"""
import sys, time
sys.path.insert(0, sys.argv[1])
import numpy as np, torch
import oracle
from attention_prefix_scan_02_b300 import binding, inputs
wl = inputs.custom(1, 1, 300, 64, dtype="bf16", seed=11, kind="tokens")
Q, K, V = inputs.token_inputs(wl)
Qg, Kg, Vg = Q.cuda(), K.cuda(), V.cuda()
binding.aaren_debug_set_fault(-1, 20_000_000)
binding.aaren_debug_drop_arrival(1)
t0 = time.time()
binding.linattn_forward(Qg, Kg, Vg, out_dtype=torch.float32)
rc = binding.aaren_check()
dt = time.time() - t0
binding.aaren_debug_set_fault(-1, 0)
binding.aaren_debug_drop_arrival(-1)
assert rc == binding.AAREN_ERR_LOAD_TIMEOUT, binding.status_string(rc)
assert dt < 10.0
assert binding.aaren_check() == binding.AAREN_OK
O = binding.linattn_forward(Qg, Kg, Vg, out_dtype=torch.float32)
assert binding.aaren_check() == binding.AAREN_OK
f = lambda t: t.float().reshape(-1, *t.shape[2:]).numpy()
Oref = oracle.la_scan(f(Q)[0], f(K)[0], f(V)[0], 300.0)[0]
err = float(np.max(np.max(np.abs(O.cpu().numpy().reshape(Oref.shape) - Oref), -1)
                  / np.maximum(np.max(np.abs(Oref), -1), 1e-30)))
assert err <= 1e-4, err
print("LINATTN_ABORT_OK", dt)
"""


def test_linattn_wait_gives_up_and_context_survives():
    """The linear attention's MMA warp never hears that chunk 1's weighted
    keys are ready: its wait gives up, the CTA aborts (every warpgroup leaves
    at a chunk boundary, the MMAs in flight drain, tensor memory is freed),
    aaren_check reports AAREN_ERR_LOAD_TIMEOUT, and the next call on the same
    context is right.  Runs in a child process of its own: one head of 300
    tokens, one CTA."""
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    res = subprocess.run([sys.executable, "-c", _LINATTN_CHILD, root], capture_output=True, text=True,
                         timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "LINATTN_ABORT_OK" in res.stdout
