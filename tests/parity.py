"""Comparison metrics for the parity tests (GPU result vs the float64 oracle).

Readings of "max relative error" (the plainest well-posed ones):
  * output rows: err = max over heads and tokens t of
    ||o_t - o_t_ref||_inf / ||o_t_ref||_inf  (element-wise relative error is
    ill-posed where a component of o_t is near 0);
  * bfloat16 output: every element equals the bfloat16 rounding (to nearest
    even) of the oracle value or one of its two neighbours (1 ulp), up to the
    float32 arithmetic error before the rounding, which is absolute on the
    row's scale (slack 2e-5 * ||o_t_ref||_inf: a component near 0 may sit
    several of its own tiny ulps away); bfloat16 rounding alone can exceed
    2e-3 relative, so a 2e-3 bound cannot apply to bfloat16 outputs;
  * final states (defined only up to (m + c, u e^-c, w e^-c)): m within tol
    (relative, floor 1), then u and w rebased to the oracle's m and compared
    relative (u row-wise as above).
"""
import numpy as np
import torch

import oracle

TOL_F32 = 2e-5     # float32 inputs and outputs
TOL_BF16 = 2e-3    # bfloat16 inputs, float32 accumulation, float32 output


def to_np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().to("cpu", torch.float32).numpy() if x.dtype == torch.bfloat16 \
            else x.detach().cpu().numpy()
    return np.asarray(x)


def rowwise_rel(o, ref):
    """max over rows of ||o - ref||_inf / ||ref||_inf (last axis = row)."""
    o = np.asarray(to_np(o), dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    num = np.max(np.abs(o - ref), axis=-1)
    den = np.maximum(np.max(np.abs(ref), axis=-1), 1e-30)
    return float(np.max(num / den)) if num.size else 0.0


def bf16_round(x):
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64))
    return t.to(torch.bfloat16).to(torch.float32).numpy()


def bf16_ulp_violations(o_bf16, ref, row_slack=TOL_F32, verbose=True):
    """Number of elements further than 1 bf16 ulp (+ row_slack * row max)
    from RNE(ref)."""
    o = to_np(o_bf16).astype(np.float64)
    ref = np.asarray(ref, np.float64)
    r = bf16_round(ref).astype(np.float64)
    mag = np.maximum(np.abs(r), np.float64(2.0 ** -126))
    ulp = 2.0 ** (np.floor(np.log2(mag)) - 7)
    slack = row_slack * np.max(np.abs(ref), axis=-1, keepdims=True)
    excess = np.abs(o - r) - ulp * (1 + 1e-9) - slack
    bad = int(np.count_nonzero(excess > 0))
    if bad and verbose:
        i = np.unravel_index(np.argmax(excess), excess.shape)
        print(f"bf16 violation: {bad} elements; worst at {i}: gpu={o[i]!r} ref={ref[i]!r} "
              f"rne={r[i]!r} ulp={ulp[i]!r} rowmax={np.max(np.abs(ref[i[:-1]]))!r}")
    return bad


def state_errors(m, u, w, m_ref, u_ref, w_ref):
    """(m error, w error, u error) after rebasing to the reference m."""
    m = np.asarray(to_np(m), np.float64).reshape(-1)
    w = np.asarray(to_np(w), np.float64).reshape(-1)
    u = np.asarray(to_np(u), np.float64).reshape(len(m), -1)
    m_ref = np.asarray(m_ref, np.float64).reshape(-1)
    w_ref = np.asarray(w_ref, np.float64).reshape(-1)
    u_ref = np.asarray(u_ref, np.float64).reshape(len(m_ref), -1)
    em = float(np.max(np.abs(m - m_ref) / np.maximum(1.0, np.abs(m_ref))))
    f = np.exp(m - m_ref)
    ew = float(np.max(np.abs(w * f - w_ref) / w_ref))
    eu = rowwise_rel(u * f[:, None], u_ref)
    return em, ew, eu


def compare_head_by_blocks(O_head, q, K, V, bf16_out, rows=1 << 16):
    """One head's whole output O_head (a CPU tensor [N, d]) against the
    oracle, `rows` tokens at a time.  At each block boundary the oracle
    continues from its own float64 state, which is the same arithmetic as one
    pass over the head, so host memory stays bounded at any N.
    Returns (row-wise relative error, bf16 ulp violations (0 unless
    bf16_out), all finite, the oracle's final state (m, u, w))."""
    N = K.shape[0]
    state = None
    err, bad, finite = 0.0, 0, True
    for r0 in range(0, N, rows):
        r1 = min(N, r0 + rows)
        Oref, m, u, w = oracle.scan(q, K[r0:r1], V[r0:r1], init=state)
        state = (m, u, w)
        blk = O_head[r0:r1]
        finite = finite and bool(torch.isfinite(blk.float()).all())
        err = max(err, rowwise_rel(blk.float(), Oref))
        if bf16_out:
            bad += bf16_ulp_violations(blk, Oref)
    return err, bad, finite, state
