"""GPU edge cases and end-to-end invariants of the scan, through the C ABI.

Ragged lengths around the chunk size, every d and dtype, empty inputs,
continuation from a saved state, shift invariance, equal scores, the first
output, many short heads, workspace reuse."""
import numpy as np
import pytest
import torch

import oracle
from attention_prefix_scan_02_b300 import binding, inputs
from tests.parity import (TOL_BF16, TOL_F32, bf16_ulp_violations, rowwise_rel, state_errors)

pytestmark = pytest.mark.gpu

DTYPES = {
    "f32": (torch.float32, torch.float32, TOL_F32),
    "bf16": (torch.bfloat16, torch.bfloat16, TOL_BF16),
    "bf16_f32out": (torch.bfloat16, torch.float32, TOL_BF16),
}
CODE = {"f32": binding.AAREN_F32, "bf16": binding.AAREN_BF16,
        "bf16_f32out": binding.AAREN_BF16_F32OUT}


def oracle_all(q, K, V, init=None):
    B, H, N, d = K.shape
    f = lambda t: t.to(torch.float32).reshape(-1, *t.shape[2:]).numpy()
    qs, Ks, Vs = f(q), f(K), f(V)
    O = np.empty((B * H, N, d)); m = np.empty(B * H); u = np.empty((B * H, d)); w = np.empty(B * H)
    for h in range(B * H):
        st = None if init is None else (init[0][h], init[1][h], init[2][h])
        O[h], m[h], u[h], w[h] = oracle.scan(qs[h], Ks[h], Vs[h], init=st)
    return O.reshape(B, H, N, d), m, u, w


def compare(O, state, ref, tol, out_bf16):
    Oref, mref, uref, wref = ref
    m, u, w = (x.cpu() for x in state)
    if out_bf16:
        assert bf16_ulp_violations(O.cpu(), Oref) == 0
    else:
        assert rowwise_rel(O.cpu(), Oref) <= tol
    em, ew, eu = state_errors(m, u, w, mref, uref, wref)
    assert em <= tol and ew <= tol and eu <= tol


def make(B, H, N, d, dt, seed=100, kind="normal"):
    wl = inputs.custom(B, H, N, d, dtype="f32" if dt == "f32" else "bf16", seed=seed, kind=kind)
    return inputs.batch_inputs(wl)


@pytest.mark.parametrize("dt", list(DTYPES))
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_ragged_lengths(d, dt):
    in_t, out_t, tol = DTYPES[dt]
    C = binding.aaren_scan_chunk_tokens(d, CODE[dt])
    for N in (1, 2, 31, 33, C - 1, C, C + 1, 5 * C + 17):
        q, K, V = make(2, 3, N, d, dt, seed=1000 + N + d)
        O, st = binding.scan_forward(q.cuda(), K.cuda(), V.cuda(), out_dtype=out_t,
                                     return_state=True)
        assert binding.aaren_check() == 0
        compare(O, st, oracle_all(q, K, V), tol, out_t == torch.bfloat16)


def test_many_short_heads():
    q, K, V = make(64, 64, 40, 64, "bf16", seed=7)
    O, st = binding.scan_forward(q.cuda(), K.cuda(), V.cuda(), out_dtype=torch.float32,
                                 return_state=True)
    assert binding.aaren_check() == 0
    compare(O, st, oracle_all(q, K, V), TOL_BF16, False)


def test_empty_inputs():
    d = 64
    for B, H, N in ((0, 4, 10), (2, 0, 10), (2, 3, 0)):
        q = torch.randn(B, H, d, device="cuda")
        K = torch.randn(B, H, N, d, device="cuda")
        O = torch.full((B, H, N, d), 7.0, device="cuda")
        binding.aaren_scan_forward(q, K, K.clone(), O)
        assert binding.aaren_check() == 0
    # N = 0 with a final state: identity, or the starting state
    q = torch.randn(2, 3, d, device="cuda")
    K = torch.empty(2, 3, 0, d, device="cuda")
    O, (m, u, w) = binding.scan_forward(q, K, K.clone(), return_state=True)
    torch.cuda.synchronize()
    assert torch.all(m == -float("inf")) and torch.all(u == 0) and torch.all(w == 0)
    init = (torch.randn(6, device="cuda"), torch.randn(6, d, device="cuda"),
            torch.rand(6, device="cuda") + 1)
    O, (m, u, w) = binding.scan_forward(q, K, K.clone(), init=init, return_state=True)
    torch.cuda.synchronize()
    assert torch.equal(m, init[0]) and torch.equal(u, init[1]) and torch.equal(w, init[2])


@pytest.mark.parametrize("dt", ["f32", "bf16_f32out"])
def test_continuation_from_a_saved_state(dt):
    """Scanning [A; B] equals scanning A, then B starting from A's final state
    (the constant-size RNN state carried between calls)."""
    in_t, out_t, tol = DTYPES[dt]
    d = 64
    q, K, V = make(2, 2, 1000, d, dt, seed=21)
    qg, Kg, Vg = q.cuda(), K.cuda(), V.cuda()
    O_full, st_full = binding.scan_forward(qg, Kg, Vg, out_dtype=out_t, return_state=True)
    for cut in (1, 129, 700):
        _, st_a = binding.scan_forward(qg, Kg[:, :, :cut].contiguous(), Vg[:, :, :cut].contiguous(),
                                       out_dtype=out_t, return_state=True)
        O_b, st_b = binding.scan_forward(qg, Kg[:, :, cut:].contiguous(), Vg[:, :, cut:].contiguous(),
                                         out_dtype=out_t, init=st_a, return_state=True)
        assert binding.aaren_check() == 0
        ref = oracle_all(q, K, V)
        assert rowwise_rel(O_b.cpu(), ref[0][:, :, cut:]) <= tol
        em, ew, eu = state_errors(*(x.cpu() for x in st_b), *ref[1:])
        assert em <= tol and ew <= tol and eu <= tol
        assert rowwise_rel(O_b.cpu(), O_full[:, :, cut:].cpu()) <= 2 * tol


def test_shift_invariance_end_to_end():
    """k_i -> k_i + a q shifts every score by a |q|^2: the output is unchanged."""
    d = 64
    q, K, V = make(2, 2, 700, d, "f32", seed=31)
    a = 3.0
    K2 = (K.double() + a * q.double()[:, :, None, :]).float()
    O1 = binding.scan_forward(q.cuda(), K.cuda(), V.cuda())
    O2 = binding.scan_forward(q.cuda(), K2.cuda(), V.cuda())
    assert binding.aaren_check() == 0
    # the shifted keys are rounded to float32, so compare each against its own oracle
    ref2 = oracle_all(q, K2, V)[0]
    assert rowwise_rel(O2.cpu(), ref2) <= TOL_F32
    assert rowwise_rel(O1.cpu(), O2.cpu()) <= 1e-3


def test_equal_scores_give_prefix_means():
    d = 32
    q, K, V = make(1, 2, 500, d, "f32", seed=41)
    q.zero_()
    O = binding.scan_forward(q.cuda(), K.cuda(), V.cuda()).cpu().double()
    assert binding.aaren_check() == 0
    ref = torch.cumsum(V.double(), dim=2) / torch.arange(1, 501, dtype=torch.float64)[:, None]
    assert rowwise_rel(O, ref.numpy()) <= TOL_F32


def test_first_output_is_first_value():
    q, K, V = make(3, 2, 300, 128, "f32", seed=51)
    O = binding.scan_forward(q.cuda(), K.cuda(), V.cuda()).cpu()
    assert binding.aaren_check() == 0
    assert torch.equal(O[:, :, 0], V[:, :, 0])


def test_large_logits_stay_finite():
    q, K, V = make(2, 2, 3000, 64, "f32", seed=61, kind="stress")
    K = K * 4          # scores in the thousands
    O, st = binding.scan_forward(q.cuda(), K.cuda(), V.cuda(), return_state=True)
    assert binding.aaren_check() == 0
    assert torch.isfinite(O).all() and torch.isfinite(st[1]).all()
    ref = oracle_all(q, K, V)
    assert rowwise_rel(O.cpu(), ref[0]) <= TOL_F32


def test_workspace_needs_no_initialisation_and_is_reusable():
    d = 128
    q, K, V = make(1, 4, 3000, d, "bf16", seed=71)
    qg, Kg, Vg = q.cuda(), K.cuda(), V.cuda()
    ws = binding.new_workspace(1, 4, 3000, d)
    ws.fill_(0xA5)
    ref = oracle_all(q, K, V)
    for _ in range(3):
        O, st = binding.scan_forward(qg, Kg, Vg, out_dtype=torch.float32, return_state=True,
                                     workspace=ws)
        assert binding.aaren_check() == 0
        compare(O, st, ref, TOL_BF16, False)


def test_streams_are_respected():
    d = 64
    q, K, V = make(2, 4, 2000, d, "bf16", seed=81)
    qg, Kg, Vg = q.cuda(), K.cuda(), V.cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        O = binding.scan_forward(qg, Kg, Vg, out_dtype=torch.float32)
    assert binding.aaren_check(s) == 0
    assert rowwise_rel(O.cpu(), oracle_all(q, K, V)[0]) <= TOL_BF16


@pytest.mark.parametrize("graph", [False, True])
def test_scan_reads_inputs_written_just_before_it(graph):
    """Two scans on one workspace, each reading q, K and V from buffers that
    copy kernels refill just before it on the same stream.  The scan kernel
    is launched as a programmatic dependent of its workspace zeroing, which
    itself follows the copies in stream order, so the scan must read nothing
    before the copies (and the earlier scan's use of the workspace) are
    complete: each output matches the oracle on its own inputs."""
    d, N = 64, 5 * 128 + 17
    sets = [make(2, 3, N, d, "bf16", seed=s) for s in (61, 62)]
    refs = [oracle_all(q, K, V) for q, K, V in sets]
    dev = [tuple(t.cuda() for t in s) for s in sets]
    qb = torch.empty_like(dev[0][0])
    Kb = torch.empty_like(dev[0][1])
    Vb = torch.empty_like(dev[0][2])
    outs = [torch.empty(Kb.shape, dtype=torch.float32, device="cuda") for _ in sets]
    states = [tuple(torch.empty(s, device="cuda") for s in ((2, 3), (2, 3, d), (2, 3))) for _ in sets]
    ws = torch.empty(binding.aaren_scan_workspace_bytes(2, 3, N, d), dtype=torch.uint8, device="cuda")

    def body():
        for (q, K, V), O, (m, u, w) in zip(dev, outs, states):
            qb.copy_(q)
            Kb.copy_(K)
            Vb.copy_(V)
            binding.aaren_scan_forward_ex(qb, Kb, Vb, O, m_out=m, u_out=u, w_out=w, workspace=ws)

    if graph:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            body()
        g.replay()
    else:
        body()
    torch.cuda.synchronize()
    assert binding.aaren_check() == 0
    for O, st, ref in zip(outs, states, refs):
        compare(O, st, ref, TOL_BF16, False)
