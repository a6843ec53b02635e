"""The parity tests' own comparison helpers, on the CPU: the block-wise
comparison of a long head must see exactly what one pass of the oracle sees,
and must catch a wrong value in any block."""
import numpy as np
import torch

import oracle
from attention_prefix_scan_02_b300 import inputs
from tests.parity import TOL_F32, compare_head_by_blocks


def _head():
    wl = inputs.custom(1, 1, 1000, 32, dtype="bf16", seed=77)
    return inputs.head_inputs(wl, 0, 0)


def test_blockwise_oracle_state_equals_one_pass():
    q, K, V = _head()
    Oref, m, u, w = oracle.scan(q, K, V)
    O = torch.from_numpy(Oref.astype(np.float32))
    err, bad, finite, (mb, ub, wb) = compare_head_by_blocks(O, q, K, V, False, rows=96)
    assert finite and bad == 0
    assert err <= 1e-7                       # only the float32 rounding of O
    assert mb == m and wb == w and np.array_equal(ub, u)   # the same arithmetic, bit for bit


def test_blockwise_comparison_catches_a_wrong_row_in_any_block():
    q, K, V = _head()
    Oref, *_ = oracle.scan(q, K, V)
    for row in (0, 95, 96, 500, 999):
        O = torch.from_numpy(Oref.astype(np.float32))
        O[row, 3] += 1e-3 * float(np.max(np.abs(Oref[row])))
        err, *_ = compare_head_by_blocks(O, q, K, V, False, rows=96)
        assert err > TOL_F32, row
        Ob = O.to(torch.bfloat16)
        Ob[row, 5] = -Ob[row, 5] + 0.5
        _, bad, *_ = compare_head_by_blocks(Ob, q, K, V, True, rows=96)
        assert bad >= 1, row


def test_blockwise_comparison_flags_non_finite_output():
    q, K, V = _head()
    Oref, *_ = oracle.scan(q, K, V)
    O = torch.from_numpy(Oref.astype(np.float32))
    O[700, 0] = float("nan")
    _, _, finite, _ = compare_head_by_blocks(O, q, K, V, False, rows=96)
    assert not finite
