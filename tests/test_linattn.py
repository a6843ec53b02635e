"""GPU parity of the causal cos-re-weighted linear attention
(aaren_linattn_forward, through the C ABI) against the float64 oracle
(oracle.la_scan, pinned to the definition, a hand-derived worked example and
the ReLU-linear-attention special case).

Tolerance (derived from the arithmetic; the pages fix none for this method):
bfloat16 inputs are exact, every product runs on the tensor cores with
float32 accumulation, and every operand the method rounds (the intra-chunk
weights A, the position-weighted keys, the state S) is carried as a bfloat16
pair hi + lo, i.e. with about 16 significant bits.  What remains is float32
accumulation error: about 1e-5 row-wise relative in a float64 emulation of
the same chunked arithmetic.  TOL_LA = 1e-4 leaves a 10x margin and still
fails if any one hi/lo pair loses its low half (that alone costs 2e-3 to
3e-3).  Row-wise relative error as for the scan (||o_i - ref||_inf /
||ref||_inf); bfloat16 outputs within one bfloat16 ulp of the rounded oracle
value; states relative to the largest entry of the head's S (resp. z)."""
import numpy as np
import pytest
import torch

import oracle
from attention_prefix_scan_02_b300 import binding, inputs
from tests.parity import bf16_ulp_violations, rowwise_rel

pytestmark = pytest.mark.gpu

THREADS = inputs.default_threads()
TOL_LA = 1e-4


def report(name, **vals):
    print("PARITY", name, " ".join(f"{k}={v:.3e}" if isinstance(v, float) else f"{k}={v}"
                                   for k, v in vals.items()))


def f32(t):
    return t.to(torch.float32).reshape(-1, *t.shape[2:]).cpu().numpy()


def ref_heads(Q, K, V, M, init=None, pos0=0):
    """Oracle outputs and final states of every head: O [BH,N,d], S [BH,2,d,d], z [BH,2,d]."""
    Qn, Kn, Vn = f32(Q), f32(K), f32(V)
    BH, N, d = Kn.shape
    O = np.empty((BH, N, d)); S = np.empty((BH, 2, d, d)); z = np.empty((BH, 2, d))
    from concurrent.futures import ThreadPoolExecutor

    def one(h):
        ini = None
        if init is not None:
            Si, zi = (x.reshape(BH, 2, *x.shape[3:]).cpu().double().numpy() for x in init)
            ini = (Si[h, 0], Si[h, 1], zi[h, 0], zi[h, 1])
        o, (Sc, Ss, zc, zs) = oracle.la_scan(Qn[h], Kn[h], Vn[h], M, init=ini, pos0=pos0)
        O[h] = o; S[h, 0] = Sc; S[h, 1] = Ss; z[h, 0] = zc; z[h, 1] = zs

    with ThreadPoolExecutor(max_workers=max(1, min(THREADS, 16))) as ex:
        list(ex.map(one, range(BH)))
    return O, S, z


def state_err(S, z, Sr, zr):
    S = S.reshape(Sr.shape).cpu().double().numpy(); z = z.reshape(zr.shape).cpu().double().numpy()
    eS = max(float(np.max(np.abs(S[h] - Sr[h])) / max(1e-30, float(np.max(np.abs(Sr[h])))))
             for h in range(len(Sr)))
    ez = max(float(np.max(np.abs(z[h] - zr[h])) / max(1e-30, float(np.max(np.abs(zr[h])))))
             for h in range(len(zr)))
    return eS, ez


def check_out(name, O, ref, out_t):
    BH = ref.shape[0]
    o = O.reshape(BH, *O.shape[2:]).cpu()
    assert torch.isfinite(o.float()).all()
    if out_t == torch.bfloat16:
        bad = bf16_ulp_violations(o, ref)
        report(name, bf16_ulp_violations=bad, rowwise=rowwise_rel(o.float(), ref))
        assert bad == 0
    else:
        err = rowwise_rel(o, ref)
        report(name, rowwise=err)
        assert err <= TOL_LA


def run(Q, K, V, out_t, M=None, init=None, pos0=0):
    out = binding.linattn_forward(Q.cuda(), K.cuda(), V.cuda(), M=M, out_dtype=out_t,
                                  init=None if init is None else tuple(x.cuda() for x in init),
                                  pos0=pos0, return_state=True)
    assert binding.aaren_check() == binding.AAREN_OK
    return out


def workload(B, H, N, seed):
    return inputs.token_inputs(inputs.custom(B, H, N, 64, dtype="bf16", seed=seed, kind="tokens"))


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_small_sequences(out):
    out_t = torch.float32 if out == "f32" else torch.bfloat16
    Q, K, V = workload(1, 2, 300, 71)
    O, (S, z) = run(Q, K, V, out_t)
    Or, Sr, zr = ref_heads(Q, K, V, 300.0)
    check_out(f"la_small_{out}", O, Or, out_t)
    eS, ez = state_err(S, z, Sr, zr)
    report(f"la_small_{out}_state", S=eS, z=ez)
    assert eS <= TOL_LA and ez <= TOL_LA


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_ragged_lengths(out):
    out_t = torch.float32 if out == "f32" else torch.bfloat16
    for N in (1, 2, 63, 127, 128, 129, 255, 256, 257, 1000):
        Q, K, V = workload(1, 3, N, 7000 + N)
        O, (S, z) = run(Q, K, V, out_t)
        Or, Sr, zr = ref_heads(Q, K, V, float(N))
        check_out(f"la_ragged_{out}_N{N}", O, Or, out_t)
        eS, ez = state_err(S, z, Sr, zr)
        assert eS <= TOL_LA and ez <= TOL_LA, (N, eS, ez)


def test_more_heads_than_sms():
    """320 heads: every CTA walks several heads (state reset between them)."""
    Q, K, V = workload(2, 160, 257, 72)
    O, (S, z) = run(Q, K, V, torch.float32)
    Or, Sr, zr = ref_heads(Q, K, V, 257.0)
    check_out("la_320_heads", O, Or, torch.float32)
    eS, ez = state_err(S, z, Sr, zr)
    report("la_320_heads_state", S=eS, z=ez)
    assert eS <= TOL_LA and ez <= TOL_LA


@pytest.mark.parametrize("Mf", [1.0, 3.0, 50.0])
def test_reweighting_length(Mf):
    Q, K, V = workload(1, 2, 700, 73)
    M = Mf * 700
    O, _ = run(Q, K, V, torch.float32, M=M)
    Or, _, _ = ref_heads(Q, K, V, M)
    check_out(f"la_M{Mf}", O, Or, torch.float32)


def test_continuation_from_a_state():
    """(first part, then the rest from its state with positions continued)
    equals the whole sequence."""
    Q, K, V = workload(2, 2, 1500, 74)
    cut = 611
    sl = lambda t, a, b: t[:, :, a:b].contiguous()
    M = 1500.0
    _, st1 = run(sl(Q, 0, cut), sl(K, 0, cut), sl(V, 0, cut), torch.float32, M=M)
    O2, (S2, z2) = run(sl(Q, cut, 1500), sl(K, cut, 1500), sl(V, cut, 1500), torch.float32, M=M,
                       init=st1, pos0=cut)
    Or, Sr, zr = ref_heads(Q, K, V, M)
    check_out("la_continue", O2, Or[:, cut:], torch.float32)
    eS, ez = state_err(S2, z2, Sr, zr)
    assert eS <= TOL_LA and ez <= TOL_LA


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_positions_past_single_precision(out):
    """Positions that continue from near 2^24, where their conversion to
    single precision stops being exact (the kernel forms each angle as
    float(position) / (2M) in single precision)."""
    out_t = torch.float32 if out == "f32" else torch.bfloat16
    Q, K, V = workload(1, 2, 300, 77)
    pos0 = (1 << 24) - 150
    M = float(pos0 + 300)
    O, (S, z) = run(Q, K, V, out_t, M=M, pos0=pos0)
    Or, Sr, zr = ref_heads(Q, K, V, M, pos0=pos0)
    check_out(f"la_far_positions_{out}", O, Or, out_t)
    eS, ez = state_err(S, z, Sr, zr)
    report(f"la_far_positions_{out}_state", S=eS, z=ez)
    assert eS <= TOL_LA and ez <= TOL_LA


def test_zero_queries_give_zero_rows():
    Q, K, V = workload(1, 2, 400, 75)
    rows = [0, 5, 127, 128, 333]
    Q[:, :, rows] = -Q[:, :, rows].abs() - 0.5
    O, _ = run(Q, K, V, torch.float32)
    assert torch.all(O[:, :, rows] == 0)
    Or, _, _ = ref_heads(Q, K, V, 400.0)
    live = [i for i in range(400) if i not in rows]
    check_out("la_zero_rows", O[:, :, live], Or[:, live], torch.float32)


def test_empty_sequence_copies_the_state():
    Q, K, V = workload(1, 2, 200, 76)
    _, (S, z) = run(Q, K, V, torch.float32)
    E = torch.empty(1, 2, 0, 64, dtype=torch.bfloat16)
    _, (S0, z0) = run(E, E, E, torch.float32, init=(S, z), pos0=200)
    assert torch.equal(S0.cpu(), S.cpu()) and torch.equal(z0.cpu(), z.cpu())
    _, (Sz, zz) = run(E, E, E, torch.float32)
    assert torch.count_nonzero(Sz).item() == 0 and torch.count_nonzero(zz).item() == 0


def test_full_workload_sampled():
    """The linattn workload at full size (64 x 16 heads x 2048 tokens, bf16
    in and out): 12 heads spread over the batch against the oracle, outputs
    and final states."""
    wl = inputs.WORKLOADS["linattn"]
    Q, K, V = inputs.token_inputs(wl, device="cuda")
    O, (S, z) = binding.linattn_forward(Q, K, V, return_state=True)
    assert binding.aaren_check() == binding.AAREN_OK
    heads = [(0, 0), (0, 15), (7, 3), (20, 8), (31, 1), (32, 12), (40, 5), (47, 9), (55, 14),
             (60, 2), (63, 0), (63, 15)]
    from concurrent.futures import ThreadPoolExecutor

    def one(bh):
        b, h = bh
        Qh, Kh, Vh = inputs.head_token_inputs(wl, b, h)
        o, (Sc, Ss, zc, zs) = oracle.la_scan(Qh, Kh, Vh, float(wl.N))
        return bh, o, np.stack([Sc, Ss]), np.stack([zc, zs])

    with ThreadPoolExecutor(max_workers=max(1, min(THREADS, 12))) as ex:
        res = list(ex.map(one, heads))
    bad = 0; e_s = e_z = 0.0; e_row = 0.0
    for (b, h), o, Sr, zr in res:
        bad += bf16_ulp_violations(O[b, h].cpu(), o)
        e_row = max(e_row, rowwise_rel(O[b, h].float().cpu(), o))
        es, ez = state_err(S[b, h][None], z[b, h][None], Sr[None], zr[None])
        e_s, e_z = max(e_s, es), max(e_z, ez)
    report("la_full_workload", bf16_ulp_violations=bad, rowwise=e_row, S=e_s, z=e_z)
    assert bad == 0 and e_s <= TOL_LA and e_z <= TOL_LA
