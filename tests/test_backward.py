"""GPU parity of the backward pass (aaren_scan_forward_stats +
aaren_scan_backward, through the C ABI) against the float64 oracle's
gradients (oracle.backward, itself pinned to the definition and to finite
differences), on seeded inputs and upstream gradients.

Metrics (gradients are float32 for every dtype):
  dV    row-wise relative error, as for the forward output;
  dK, dq   relative to the size of what they are computed from.  dL/ds_i =
        p_i (v_i . R_i - D_i) is a difference of two sums that can nearly
        cancel (always, when one score dominates: then every dL/ds is ~0), so
        its float32 error is bounded by the summands, not by the result:
        S_i = |v_i| |dV_i| + |dL/ds_i - v_i . dV_i|  (= p_i |v_i| |R_i| + p_i |D_i|,
        from the oracle).  The checks are
          max |dK - ref| <= tol * max_i S_i * max|q|,
          max |dq - ref| <= tol * sum_i S_i max|k_i|.
Tolerances: float32 inputs and outputs 2e-5 (as the forward) for dK and
dq, 5e-5 for dV: dV_i = p_i R_i where R_i sums g over the whole rest of the
sequence (16384 tokens in the stress workload) with a rounded decay factor
per token, and unlike the forward's o_t = u_t / w_t no division cancels the
correlated part of that rounding.  bfloat16 inputs with a float32 O and dO:
2e-3 (as the forward).  A bfloat16 O and dO carry the output's own rounding
(2^-9 relative) into g_t . o_t, so D_i and with it dL/ds carry it too: 4e-3
(2^-8) for those."""
import numpy as np
import pytest
import torch

import oracle
from attention_prefix_scan_02_b300 import binding, inputs
from tests.parity import rowwise_rel

pytestmark = pytest.mark.gpu

THREADS = inputs.default_threads()
TOL = {"f32": 2e-5, "bf16_f32out": 2e-3, "bf16": 4e-3}          # dK, dq
TOL_DV = {"f32": 5e-5, "bf16_f32out": 2e-3, "bf16": 4e-3}       # dV rows
TYPES = {"f32": (torch.float32, torch.float32), "bf16_f32out": (torch.bfloat16, torch.float32),
         "bf16": (torch.bfloat16, torch.bfloat16)}


def report(name, **vals):
    print("PARITY", name, " ".join(f"{k}={v:.3e}" if isinstance(v, float) else f"{k}={v}"
                                   for k, v in vals.items()))


def upstream(B, H, N, d, out_t, seed):
    """dL/dO ~ N(0, 1), stored in the output type."""
    wl = inputs.custom(B, H, N, d, dtype="bf16" if out_t == torch.bfloat16 else "f32",
                       seed=seed + 7777)
    return inputs.batch_inputs(wl)[2]


def scale_rel(a, ref):
    a = np.asarray(a, np.float64)
    ref = np.asarray(ref, np.float64)
    return float(np.max(np.abs(a - ref)) / max(1e-30, float(np.max(np.abs(ref)))))


def summand_scale(Vh, rdV, rds):
    """S_i = |v_i| |dV_i| + |ds_i - v_i . dV_i| for one head (float64)."""
    Vh = np.asarray(Vh, np.float64)
    vdv = np.sum(Vh * rdV, axis=-1)
    return np.linalg.norm(Vh, axis=-1) * np.linalg.norm(rdV, axis=-1) + np.abs(rds - vdv)


def grad_errors(q, K, V, dq, dK, dV, ref):
    """(dV row-wise, dK and dq against the summand scale), worst head."""
    rq, rK, rV, rds = ref
    e_v = rowwise_rel(dV, rV) if dV.size else 0.0
    e_k = e_q = 0.0
    for h in range(len(rq)):
        if K.shape[1] == 0:
            continue
        S = summand_scale(V[h], rV[h], rds[h])
        sk = float(np.max(S)) * float(np.max(np.abs(q[h])))
        sq = float(np.sum(S * np.max(np.abs(K[h]), axis=-1)))
        e_k = max(e_k, float(np.max(np.abs(dK[h] - rK[h]))) / max(sk, 1e-30))
        e_q = max(e_q, float(np.max(np.abs(dq[h] - rq[h]))) / max(sq, 1e-30))
    return e_v, e_k, e_q


def run_case(name, q, K, V, G, dt):
    in_t, out_t = TYPES[dt]
    qc, Kc, Vc, Gc = q.cuda(), K.cuda(), V.cuda(), G.cuda()
    O, stats = binding.scan_forward_train(qc, Kc, Vc, out_dtype=out_t)
    dq, dK, dV = binding.scan_backward(qc, Kc, Vc, O, Gc, stats)
    assert binding.aaren_check() == binding.AAREN_OK
    B, H, N, d = K.shape
    f = lambda t: t.to(torch.float32).reshape(-1, *t.shape[2:]).numpy()
    qs, Ks, Vs = f(q), f(K), f(V)
    ref = oracle.backward_heads(qs, Ks, Vs, f(G), threads=THREADS)
    dq, dK, dV = (x.cpu().numpy().reshape(B * H, *x.shape[2:]) for x in (dq, dK, dV))
    assert np.all(np.isfinite(dq)) and np.all(np.isfinite(dK)) and np.all(np.isfinite(dV))
    e_v, e_k, e_q = grad_errors(qs, Ks, Vs, dq, dK, dV, ref)
    report(name, dV_rowwise=e_v, dK=e_k, dq=e_q, dK_vs_own_max=scale_rel(dK, ref[1]))
    assert e_v <= TOL_DV[dt] and e_k <= TOL[dt] and e_q <= TOL[dt]
    return O, stats


def test_stats_give_every_prefix_log_sum_exp():
    wl = inputs.custom(2, 3, 3000, 64, seed=41)
    q, K, V = inputs.batch_inputs(wl)
    O, stats = binding.scan_forward_train(q.cuda(), K.cuda(), V.cuda())
    O_plain = binding.scan_forward(q.cuda(), K.cuda(), V.cuda())
    assert binding.aaren_check() == binding.AAREN_OK
    # saving the statistics changes nothing (the cross-chunk carry folds its
    # predecessors in a timing-dependent grouping, so up to float32 rounding)
    assert rowwise_rel(O.cpu(), O_plain.cpu().double().numpy()) <= 1e-6
    st = stats.cpu().numpy().reshape(6, 3000, 2).astype(np.float64)
    lse = st[..., 0] + np.log(st[..., 1])
    qs, Ks = q.reshape(6, 64).numpy(), K.reshape(6, 3000, 64).numpy()
    ref = np.stack([oracle.lse(qs[h], Ks[h]) for h in range(6)])
    err = float(np.max(np.abs(lse - ref) / np.maximum(1.0, np.abs(ref))))
    report("stats_lse", rel=err)
    assert err <= 1e-5


@pytest.mark.parametrize("dt", ["f32", "bf16_f32out", "bf16"])
def test_random_sequences(dt):
    in_t, out_t = TYPES[dt]
    wl = inputs.custom(2, 2, 2500, 64, dtype="f32" if dt == "f32" else "bf16", seed=42)
    q, K, V = inputs.batch_inputs(wl)
    G = upstream(2, 2, 2500, 64, out_t, 42)
    run_case(f"bwd_random_{dt}", q, K, V, G, dt)


def test_tiny_workload():
    wl = inputs.WORKLOADS["tiny"]
    q, K, V = inputs.batch_inputs(wl)
    G = upstream(wl.B, wl.H, wl.N, wl.d, torch.float32, wl.seed)
    run_case("bwd_tiny_f32", q, K, V, G, "f32")


def test_stress_workload():
    wl = inputs.WORKLOADS["stress"]
    q, K, V = inputs.batch_inputs(wl)
    G = upstream(wl.B, wl.H, wl.N, wl.d, torch.float32, wl.seed)
    run_case("bwd_stress_f32", q, K, V, G, "f32")


@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_bf16_4k_workload(out):
    wl = inputs.WORKLOADS["bf16_4k"]
    q, K, V = inputs.batch_inputs(wl)
    dt = "bf16_f32out" if out == "f32" else "bf16"
    G = upstream(wl.B, wl.H, wl.N, wl.d, TYPES[dt][1], wl.seed)
    run_case(f"bwd_bf16_4k_{out}out", q, K, V, G, dt)


@pytest.mark.parametrize("dt", ["f32", "bf16_f32out", "bf16"])
@pytest.mark.parametrize("d", [16, 32, 64, 128])
def test_ragged_lengths(d, dt):
    in_t, out_t = TYPES[dt]
    for N in (1, 2, 31, 33, 63, 65, 128, 129, 1000):
        wl = inputs.custom(1, 3, N, d, dtype="f32" if dt == "f32" else "bf16", seed=5000 + N + d)
        q, K, V = inputs.batch_inputs(wl)
        G = upstream(1, 3, N, d, out_t, 5000 + N + d)
        run_case(f"bwd_ragged_d{d}_{dt}_N{N}", q, K, V, G, dt)


def test_empty_sequence_gives_zero_query_gradient():
    q = torch.randn(1, 2, 32).cuda()
    E = torch.empty(1, 2, 0, 32).cuda()
    st = torch.empty(1, 2, 0, 2).cuda()
    dq = torch.full((2, 32), 7.0, device="cuda")
    binding.aaren_scan_backward(q, E, E, E, E, st, dq, E.clone(), E.clone())
    assert binding.aaren_check() == binding.AAREN_OK
    assert torch.count_nonzero(dq).item() == 0


def test_long_workload_sampled():
    """The 2^20-token workload at full size (bf16 in, f32 O and dO): dq of
    every head and dK, dV of two heads against the oracle."""
    from concurrent.futures import ThreadPoolExecutor
    wl = inputs.WORKLOADS["long"]
    q, K, V = inputs.batch_inputs(wl, device="cuda")
    G = upstream(wl.B, wl.H, wl.N, wl.d, torch.float32, wl.seed).cuda()
    O, stats = binding.scan_forward_train(q, K, V, out_dtype=torch.float32)
    dq, dK, dV = binding.scan_backward(q, K, V, O, G, stats)
    assert binding.aaren_check() == binding.AAREN_OK
    sampled = (0, wl.H - 1)
    dK_s = {h: dK[0, h].cpu().numpy() for h in sampled}
    dV_s = {h: dV[0, h].cpu().numpy() for h in sampled}
    dq = dq.reshape(wl.H, wl.d).cpu().numpy()
    Gc = G.cpu()
    del K, V, O, dK, dV

    def one(h):
        qh, Kh, Vh = inputs.head_inputs(wl, 0, h)
        rq, rK, rV, rds = oracle.backward(qh, Kh, Vh, Gc[0, h].numpy())
        S = summand_scale(Vh, rV, rds)
        out = {"q": float(np.max(np.abs(dq[h] - rq))) /
                    float(np.sum(S * np.max(np.abs(Kh), axis=-1)))}
        if h in sampled:
            out["k"] = float(np.max(np.abs(dK_s[h] - rK))) / (float(np.max(S)) * float(np.max(np.abs(qh))))
            out["v"] = rowwise_rel(dV_s[h], rV)
        return h, out

    with ThreadPoolExecutor(max_workers=max(1, min(THREADS, 8))) as ex:
        res = dict(ex.map(one, range(wl.H)))
    e_q = max(r["q"] for r in res.values())
    e_k = max(res[h]["k"] for h in sampled)
    e_v = max(res[h]["v"] for h in sampled)
    report("bwd_long_bf16_f32out", dV_rowwise=e_v, dK_scale=e_k, dq=e_q)
    assert e_q <= TOL["bf16_f32out"] and e_k <= TOL["bf16_f32out"] and e_v <= TOL["bf16_f32out"]
