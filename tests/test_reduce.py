"""GPU parity of the many-to-one form (aaren_scan_reduce, through the C ABI)
against the float64 oracle: o_N of every head and the final state (m, u, w),
on the named workloads, ragged lengths around the part and batch sizes,
every d and dtype, a starting state, the empty sequence, and against the
scan's own last output.

The oracle's o_N is u_N / w_N of its final state (the definition of the last
prefix output).  Tolerances are those of the scan: float32 2e-5, bfloat16
inputs 2e-3 (row-wise relative error), bfloat16 output within one bfloat16
ulp of the rounded oracle value."""
import numpy as np
import pytest
import torch

import oracle
from attention_prefix_scan_02_b300 import binding, inputs
from tests.parity import (TOL_BF16, TOL_F32, bf16_ulp_violations, rowwise_rel, state_errors)

pytestmark = pytest.mark.gpu

THREADS = inputs.default_threads()
DTYPES = {
    "f32": (torch.float32, torch.float32, TOL_F32),
    "bf16": (torch.bfloat16, torch.bfloat16, TOL_BF16),
    "bf16_f32out": (torch.bfloat16, torch.float32, TOL_BF16),
}


def report(name, **vals):
    print("PARITY", name, " ".join(f"{k}={v:.3e}" if isinstance(v, float) else f"{k}={v}"
                                   for k, v in vals.items()))


def oracle_final(q, K, V, init=None):
    """Final state and o_N of every head from the oracle (no per-token output)."""
    B, H, N, d = K.shape
    f = lambda t: t.to(torch.float32).reshape(-1, *t.shape[2:]).numpy()
    if init is None:
        _, m, u, w = oracle.scan_heads(f(q), f(K), f(V), threads=THREADS, want_O=False)
    else:
        qs, Ks, Vs = f(q), f(K), f(V)
        m = np.empty(B * H); u = np.empty((B * H, d)); w = np.empty(B * H)
        for h in range(B * H):
            _, m[h], u[h], w[h] = oracle.scan(qs[h], Ks[h], Vs[h], init=(init[0][h], init[1][h],
                                                                         init[2][h]), want_O=False)
    return u / w[:, None], m, u, w


def check(name, o, state, ref, tol, out_bf16):
    oref, mref, uref, wref = ref
    o = o.reshape(len(mref), -1).cpu()
    assert torch.isfinite(o.float()).all()
    em, ew, eu = state_errors(*(x.cpu() for x in state), mref, uref, wref)
    if out_bf16:
        bad = bf16_ulp_violations(o, oref)
        report(name, bf16_ulp_violations=bad, o_rowwise_rel=rowwise_rel(o.float(), oref), m=em, w=ew, u=eu)
        assert bad == 0
    else:
        err = rowwise_rel(o, oref)
        report(name, o_rowwise_rel=err, m=em, w=ew, u=eu)
        assert err <= tol
    assert em <= tol and ew <= tol and eu <= tol


def run(q, K, V, out_t, init=None):
    o, st = binding.scan_reduce(q.cuda(), K.cuda(), V.cuda(), out_dtype=out_t, init=init,
                                return_state=True)
    assert binding.aaren_check() == binding.AAREN_OK
    return o, st


@pytest.mark.parametrize("name,out", [("tiny", "f32"), ("bf16_4k", "f32"), ("bf16_4k", "bf16"),
                                      ("stress", "f32")])
def test_named_workloads(name, out):
    wl = inputs.WORKLOADS[name]
    q, K, V = inputs.batch_inputs(wl)
    out_t = torch.float32 if out == "f32" else torch.bfloat16
    tol = TOL_F32 if wl.dtype == "f32" else TOL_BF16
    o, st = run(q, K, V, out_t)
    check(f"reduce_{name}_{out}out", o, st, oracle_final(q, K, V), tol, out == "bf16")


@pytest.mark.parametrize("out", ["bf16", "f32"])
def test_long_workload_every_head(out):
    """The 2^20-token workload at full size: o_N and the final state of all
    16 heads against the oracle, head by head."""
    from concurrent.futures import ThreadPoolExecutor
    wl = inputs.WORKLOADS["long"]
    q, K, V = inputs.batch_inputs(wl, device="cuda")
    out_t = torch.float32 if out == "f32" else torch.bfloat16
    o, st = binding.scan_reduce(q, K, V, out_dtype=out_t, return_state=True)
    assert binding.aaren_check() == binding.AAREN_OK
    del K, V

    def one(h):
        qh, Kh, Vh = inputs.head_inputs(wl, 0, h)
        _, m, u, w = oracle.scan(qh, Kh, Vh, want_O=False)
        return m, u, w

    with ThreadPoolExecutor(max_workers=max(1, min(THREADS, 8))) as ex:
        res = list(ex.map(one, range(wl.H)))
    mref = np.array([r[0] for r in res]); uref = np.array([r[1] for r in res])
    wref = np.array([r[2] for r in res])
    check(f"reduce_long_{out}out", o, st, (uref / wref[:, None], mref, uref, wref), TOL_BF16,
          out == "bf16")


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_ragged_lengths(d, dt):
    in_t, out_t, tol = DTYPES[dt]
    for N in (1, 7, 8, 9, 63, 64, 65, 1000, 4099):
        wl = inputs.custom(2, 3, N, d, dtype="f32" if dt == "f32" else "bf16", seed=3000 + N + d)
        q, K, V = inputs.batch_inputs(wl)
        o, st = run(q, K, V, out_t)
        check(f"reduce_ragged_d{d}_{dt}_N{N}", o, st, oracle_final(q, K, V), tol,
              out_t == torch.bfloat16)


@pytest.mark.parametrize("dt", ["f32", "bf16_f32out"])
def test_starting_state_continues_the_sequence(dt):
    """o_N and the state of (first part, then second part from the first
    part's state) equal those of the whole sequence."""
    in_t, out_t, tol = DTYPES[dt]
    wl = inputs.custom(2, 2, 3000, 64, dtype="f32" if dt == "f32" else "bf16", seed=77)
    q, K, V = inputs.batch_inputs(wl)
    cut = 1234
    _, st1 = run(q, K[:, :, :cut].contiguous(), V[:, :, :cut].contiguous(), out_t)
    o2, st2 = run(q, K[:, :, cut:].contiguous(), V[:, :, cut:].contiguous(), out_t, init=st1)
    check(f"reduce_continue_{dt}", o2, st2, oracle_final(q, K, V), tol, False)


def test_empty_sequence_with_a_starting_state():
    wl = inputs.custom(1, 3, 500, 32, seed=5)
    q, K, V = inputs.batch_inputs(wl)
    _, st = run(q, K, V, torch.float32)
    E = torch.empty(1, 3, 0, 32)
    o0, st0 = run(q, E, E, torch.float32, init=st)
    m, u, w = (x.cpu() for x in st)
    assert torch.equal(st0[0].cpu(), m) and torch.equal(st0[2].cpu(), w)
    assert torch.equal(st0[1].cpu(), u)
    assert torch.allclose(o0.reshape(3, 32).cpu(), u / w[:, None], rtol=1e-6, atol=0)


def test_state_only_and_output_only():
    wl = inputs.custom(2, 2, 777, 128, dtype="bf16", seed=6)
    q, K, V = (t.cuda() for t in inputs.batch_inputs(wl))
    o = torch.empty(4, 128, device="cuda")
    binding.aaren_scan_reduce(q, K, V, o)
    m = torch.empty(4, device="cuda"); u = torch.empty(4, 128, device="cuda")
    w = torch.empty(4, device="cuda")
    binding.aaren_scan_reduce(q, K, V, None, m_out=m, u_out=u, w_out=w)
    assert binding.aaren_check() == binding.AAREN_OK
    assert torch.allclose(o, u / w[:, None], rtol=1e-6, atol=0)


@pytest.mark.parametrize("dt", list(DTYPES))
def test_agrees_with_the_scans_last_output(dt):
    in_t, out_t, tol = DTYPES[dt]
    wl = inputs.custom(4, 2, 5000, 64, dtype="f32" if dt == "f32" else "bf16", seed=9)
    q, K, V = (t.cuda() for t in inputs.batch_inputs(wl))
    O, (ms, us, ws) = binding.scan_forward(q, K, V, out_dtype=out_t, return_state=True)
    o, (mr, ur, wr) = binding.scan_reduce(q, K, V, out_dtype=out_t, return_state=True)
    assert binding.aaren_check() == binding.AAREN_OK
    last = O[:, :, -1].float().reshape(8, 64).cpu()
    red = o.float().reshape(8, 64).cpu()
    if out_t == torch.bfloat16:
        # both are roundings of values within float32 error: at most 1 ulp apart
        assert bf16_ulp_violations(red, last.double().numpy()) == 0
    else:
        assert rowwise_rel(red, last.double().numpy()) <= 2 * tol
    em, ew, eu = state_errors(mr.cpu(), ur.cpu(), wr.cpu(), ms.cpu().double().numpy(),
                              us.cpu().double().numpy(), ws.cpu().double().numpy())
    assert em <= 2 * tol and ew <= 2 * tol and eu <= 2 * tol


def test_caller_workspace_reused():
    wl = inputs.custom(1, 4, 20000, 128, dtype="bf16", seed=10)
    q, K, V = (t.cuda() for t in inputs.batch_inputs(wl))
    ws = binding.new_reduce_workspace(1, 4, 20000, 128)
    ws.fill_(0xAB)   # contents need no initialisation
    a = binding.scan_reduce(q, K, V, out_dtype=torch.float32, workspace=ws)
    b = binding.scan_reduce(q, K, V, out_dtype=torch.float32, workspace=ws)
    assert binding.aaren_check() == binding.AAREN_OK
    assert torch.equal(a, b)   # same launch shape, same combine order: bitwise equal
    ref = oracle_final(q.cpu(), K.cpu(), V.cpu())
    assert rowwise_rel(a.reshape(4, 128).cpu(), ref[0]) <= TOL_BF16
