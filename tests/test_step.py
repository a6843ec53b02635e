"""GPU parity of the streaming one-token update (aaren_step) on the streaming
workload: 256 streams x 8 heads, d = 64, float32, 4096 tokens fed one step at
a time.  Every step's output of every stream and every final state must
match the oracle, and the last outputs and final states must match
aaren_scan_forward run on the same sequences."""
import numpy as np
import pytest
import torch

import oracle
from attention_prefix_scan_02_b300 import binding, inputs
from tests.parity import TOL_BF16, TOL_F32, rowwise_rel, state_errors

pytestmark = pytest.mark.gpu


def stream_inputs(wl):
    q, K, V = inputs.batch_inputs(wl)            # [B,H,d], [B,H,N,d]; B = streams
    n = wl.B * wl.H
    return q, K, V, n


def run_steps(q, K, V, n, out_dtype, graph=False):
    B, H, N, d = K.shape
    qs = q.reshape(n, d).cuda()
    Ks = K.permute(2, 0, 1, 3).reshape(N, n, d).contiguous().cuda()
    Vs = V.permute(2, 0, 1, 3).reshape(N, n, d).contiguous().cuda()
    Os = torch.empty((N, n, d), dtype=out_dtype, device="cuda")
    m = torch.empty(n, device="cuda")
    u = torch.empty(n, d, device="cuda")
    w = torch.empty(n, device="cuda")
    binding.aaren_state_init(m, u, w)
    if not graph:
        for t in range(N):
            binding.aaren_step(qs, m, u, w, Ks[t], Vs[t], Os[t])
    else:
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for t in range(N):
                binding.aaren_step(qs, m, u, w, Ks[t], Vs[t], Os[t])
        g.replay()
    assert binding.aaren_check() == 0
    return Os, m, u, w


def test_stream_workload_steps_match_oracle_and_scan():
    wl = inputs.WORKLOADS["stream"]
    q, K, V, n = stream_inputs(wl)
    N, d = wl.N, wl.d
    Os, m, u, w = run_steps(q, K, V, n, torch.float32)
    # oracle: every stream's final state and last output
    f = lambda t: t.reshape(n, *t.shape[2:]).numpy()
    Oref, mref, uref, wref = oracle.scan_heads(f(q), f(K), f(V), threads=inputs.default_threads(),
                                               want_O=False)
    em, ew, eu = state_errors(m.cpu(), u.cpu(), w.cpu(), mref, uref, wref)
    last_ref = uref / wref[:, None]
    e_last = rowwise_rel(Os[-1].cpu(), last_ref)
    print(f"PARITY stream_steps m={em:.3e} w={ew:.3e} u={eu:.3e} o_last={e_last:.3e}")
    assert max(em, ew, eu, e_last) <= TOL_F32
    # the parallel scan on the same sequences
    O_scan, (ms, us, ws) = binding.scan_forward(q.cuda(), K.cuda(), V.cuda(), return_state=True)
    assert binding.aaren_check() == 0
    es = state_errors(ms.cpu(), us.cpu(), ws.cpu(), mref, uref, wref)
    assert max(es) <= TOL_F32
    O_scan = O_scan.reshape(n, N, d)
    # every step's output of every stream, and the scan's output at every
    # prefix, 256 streams at a time (the oracle's float64 outputs of all 2048
    # streams would take 4.3 GB)
    qn, Kn, Vn = f(q), f(K), f(V)
    worst_step = worst_scan = 0.0
    for i0 in range(0, n, 256):
        i1 = min(n, i0 + 256)
        Oref_b, *_ = oracle.scan_heads(qn[i0:i1], Kn[i0:i1], Vn[i0:i1],
                                       threads=inputs.default_threads())
        e = rowwise_rel(Os[:, i0:i1].permute(1, 0, 2).contiguous().cpu(), Oref_b)
        assert e <= TOL_F32, f"streams {i0}..{i1 - 1}: every-step error {e:.3e}"
        worst_step = max(worst_step, e)
        e = rowwise_rel(O_scan[i0:i1].cpu(), Oref_b)
        assert e <= TOL_F32, f"streams {i0}..{i1 - 1}: scan output error {e:.3e}"
        worst_scan = max(worst_scan, e)
        del Oref_b
    print(f"PARITY stream_steps_every_output o={worst_step:.3e} scan_every_output o={worst_scan:.3e}")
    d_last = rowwise_rel(Os[-1].cpu(), O_scan[:, -1].cpu().numpy())
    print(f"PARITY stream_step_vs_scan o_last={d_last:.3e}")
    assert d_last <= 2 * TOL_F32


def test_steps_in_a_cuda_graph_match_plain_launches():
    wl = inputs.custom(16, 8, 300, 64, seed=4, kind="stream")
    q, K, V, n = stream_inputs(wl)
    O1, m1, u1, w1 = run_steps(q, K, V, n, torch.float32)
    O2, m2, u2, w2 = run_steps(q, K, V, n, torch.float32, graph=True)
    assert torch.equal(O1, O2) and torch.equal(m1, m2) and torch.equal(u1, u2)


@pytest.mark.parametrize("graph", [False, True])
def test_step_reads_inputs_written_just_before_it(graph):
    """Each step reads k_t and v_t from one buffer that a copy kernel refills
    just before it on the same stream.  A step is launched as a programmatic
    dependent of the kernel before it, so it must read only once that copy
    has completed: the outputs equal those of steps reading every token's
    inputs from their own rows."""
    wl = inputs.custom(8, 8, 200, 64, seed=46, kind="stream")
    q, K, V, n = stream_inputs(wl)
    O_ref, m_ref, u_ref, w_ref = run_steps(q, K, V, n, torch.float32)
    B, H, N, d = K.shape
    qs = q.reshape(n, d).cuda()
    Ks = K.permute(2, 0, 1, 3).reshape(N, n, d).contiguous().cuda()
    Vs = V.permute(2, 0, 1, 3).reshape(N, n, d).contiguous().cuda()
    kbuf = torch.empty(n, d, device="cuda")
    vbuf = torch.empty(n, d, device="cuda")
    Os = torch.empty((N, n, d), device="cuda")
    m = torch.empty(n, device="cuda")
    u = torch.empty(n, d, device="cuda")
    w = torch.empty(n, device="cuda")

    def body():
        binding.aaren_state_init(m, u, w)
        for t in range(N):
            kbuf.copy_(Ks[t])
            vbuf.copy_(Vs[t])
            binding.aaren_step(qs, m, u, w, kbuf, vbuf, Os[t])

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
    assert torch.equal(Os, O_ref)
    assert torch.equal(m, m_ref) and torch.equal(u, u_ref) and torch.equal(w, w_ref)


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("dt", ["f32", "bf16", "bf16_f32out"])
def test_step_all_shapes(d, dt):
    in_dtype = "f32" if dt == "f32" else "bf16"
    out_t = torch.bfloat16 if dt == "bf16" else torch.float32
    tol = TOL_F32 if dt == "f32" else TOL_BF16
    wl = inputs.custom(3, 5, 70, d, dtype=in_dtype, seed=90 + d, kind="stream")
    q, K, V, n = stream_inputs(wl)
    Os, m, u, w = run_steps(q, K, V, n, out_t)
    f = lambda t: t.float().reshape(n, *t.shape[2:]).numpy()
    Oref, mref, uref, wref = oracle.scan_heads(f(q), f(K), f(V))
    em, ew, eu = state_errors(m.cpu(), u.cpu(), w.cpu(), mref, uref, wref)
    assert max(em, ew, eu) <= tol
    O = Os.float().permute(1, 0, 2).cpu().numpy()
    err = rowwise_rel(O, Oref)
    bound = tol if dt != "bf16" else TOL_BF16 + 2.0 ** -8
    assert err <= bound


def test_step_continues_a_scan():
    """Prefill with the scan, then continue the same streams with steps."""
    wl = inputs.custom(4, 4, 600, 64, seed=44, kind="stream")
    q, K, V, n = stream_inputs(wl)
    cut = 450
    d = wl.d
    _, (m, u, w) = binding.scan_forward(q.cuda(), K[:, :, :cut].contiguous().cuda(),
                                        V[:, :, :cut].contiguous().cuda(), return_state=True)
    qs = q.reshape(n, d).cuda()
    o = torch.empty(n, d, device="cuda")
    for t in range(cut, wl.N):
        binding.aaren_step(qs, m, u, w, K[:, :, t].reshape(n, d).contiguous().cuda(),
                           V[:, :, t].reshape(n, d).contiguous().cuda(), o)
    assert binding.aaren_check() == 0
    f = lambda t: t.reshape(n, *t.shape[2:]).numpy()
    Oref, mref, uref, wref = oracle.scan_heads(f(q), f(K), f(V))
    em, ew, eu = state_errors(m.cpu(), u.cpu(), w.cpu(), mref, uref, wref)
    assert max(em, ew, eu) <= TOL_F32
    assert rowwise_rel(o.cpu(), Oref[:, -1]) <= TOL_F32
