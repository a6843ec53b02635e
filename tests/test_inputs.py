"""The seeded input generators: determinism and the workload recipes."""
import numpy as np
import torch

from attention_prefix_scan_02_b300 import inputs


def test_heads_are_deterministic_and_distinct():
    wl = inputs.custom(2, 3, 70, 16, seed=5)
    a = inputs.head_inputs(wl, 1, 2)
    b = inputs.head_inputs(wl, 1, 2)
    c = inputs.head_inputs(wl, 0, 2)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)
    assert not np.array_equal(a[1], c[1])


def test_blocks_make_long_heads_independent_of_block_boundaries():
    wl = inputs.custom(1, 1, inputs.BLOCK_ROWS + 10, 16, seed=6)
    q, K, V = inputs.head_inputs(wl, 0, 0)
    assert K.shape == (inputs.BLOCK_ROWS + 10, 16) and K.dtype == np.float32
    short = inputs.custom(1, 1, 100, 16, seed=6)
    _, K2, _ = inputs.head_inputs(short, 0, 0)
    assert np.array_equal(K[:100], K2)          # same stream for the first block


def test_batch_matches_heads_for_any_thread_count():
    wl = inputs.custom(2, 2, 33, 32, dtype="bf16", seed=7)
    q1, K1, V1 = inputs.batch_inputs(wl, threads=1)
    q4, K4, V4 = inputs.batch_inputs(wl, threads=4)
    assert K1.dtype == torch.bfloat16 and K1.shape == (2, 2, 33, 32)
    assert torch.equal(K1, K4) and torch.equal(V1, V4) and torch.equal(q1, q4)
    qh, Kh, Vh = inputs.head_inputs(wl, 1, 0)
    assert np.array_equal(K1[1, 0].float().numpy(), Kh)
    assert np.array_equal(q1[1, 0].float().numpy(), qh)


def test_bf16_rounding_is_nearest_even():
    x = np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, 1.0 + 2 ** -9], dtype=np.float32)
    r = inputs.round_bf16(x)
    assert list(r) == [1.0, 1.0 + 4 * 2 ** -8, 1.0]


def test_stress_recipe():
    wl = inputs.custom(1, 1, 500, 64, seed=2, kind="stress")
    q, K, V = inputs.head_inputs(wl, 0, 0)
    spikes = np.arange(96, 500, 97)
    assert np.array_equal(K[spikes], np.tile(np.float32(3.0) * q, (len(spikes), 1)))
    rest = np.setdiff1d(np.arange(500), spikes)
    assert 6.0 < K[rest].std() < 10.0           # 8 x N(0,1)
    assert V.min() >= -1.0 and V.max() < 1.0


def test_stream_recipe_shares_the_query_across_streams():
    wl = inputs.WORKLOADS["stream"]
    small = inputs.custom(3, wl.H, 8, wl.d, seed=wl.seed, kind="stream")
    q0, _, _ = inputs.head_inputs(small, 0, 5)
    q2, K2, _ = inputs.head_inputs(small, 2, 5)
    _, K0, _ = inputs.head_inputs(small, 0, 5)
    assert np.array_equal(q0, q2) and not np.array_equal(K0, K2)


def test_named_workloads():
    w = inputs.WORKLOADS
    assert (w["tiny"].B, w["tiny"].H, w["tiny"].N, w["tiny"].d, w["tiny"].dtype) == (1, 1, 256, 16, "f32")
    assert (w["bf16_4k"].B, w["bf16_4k"].H, w["bf16_4k"].N, w["bf16_4k"].d) == (8, 4, 4096, 64)
    assert (w["stress"].B, w["stress"].H, w["stress"].N, w["stress"].d) == (4, 8, 16384, 64)
    assert (w["long"].B, w["long"].H, w["long"].N, w["long"].d, w["long"].dtype) == (1, 16, 1 << 20, 128, "bf16")
    assert (w["stream"].B, w["stream"].H, w["stream"].N, w["stream"].d) == (256, 8, 4096, 64)


def test_batch_offset_draws_a_shard_of_a_larger_batch():
    """Rank r of a multi-GPU run draws batch entries [r B, (r + 1) B): the
    shards of all ranks together are the batch of world * B sequences."""
    small = inputs.custom(1, 2, 40, 16, seed=21)
    big = inputs.custom(3, 2, 40, 16, seed=21)
    qb, Kb, Vb = inputs.batch_inputs(big)
    for r in range(3):
        q, K, V = inputs.batch_inputs(small, b0=r)
        assert torch.equal(q[0], qb[r]) and torch.equal(K[0], Kb[r]) and torch.equal(V[0], Vb[r])


def test_token_recipe_matches_heads_and_shards():
    """One query per token (the linear-attention workload): the batch tensors
    equal the per-head draws for any thread count, bf16 values are the
    rounded float32 draws, queries differ per token, and b0 selects a shard
    of a larger batch."""
    wl = inputs.custom(2, 3, 40, 64, dtype="bf16", seed=5, kind="tokens")
    Q1, K1, V1 = inputs.token_inputs(wl, threads=1)
    Q4, K4, V4 = inputs.token_inputs(wl, threads=4)
    assert Q1.shape == (2, 3, 40, 64) and Q1.dtype == torch.bfloat16
    assert torch.equal(Q1, Q4) and torch.equal(K1, K4) and torch.equal(V1, V4)
    Qh, Kh, Vh = inputs.head_token_inputs(wl, 1, 2)
    assert np.array_equal(Q1[1, 2].float().numpy(), Qh)
    assert np.array_equal(K1[1, 2].float().numpy(), Kh)
    assert np.array_equal(V1[1, 2].float().numpy(), Vh)
    assert np.array_equal(inputs.round_bf16(Qh), Qh)
    assert not np.array_equal(Qh[0], Qh[1])
    big = inputs.custom(4, 3, 40, 64, dtype="bf16", seed=5, kind="tokens")
    Qs, Ks, Vs = inputs.token_inputs(big, b0=0)
    sub = inputs.custom(2, 3, 40, 64, dtype="bf16", seed=5, kind="tokens")
    Qb, Kb, Vb = inputs.token_inputs(sub, b0=2)
    assert torch.equal(Qs[2:], Qb) and torch.equal(Ks[2:], Kb) and torch.equal(Vs[2:], Vb)


def test_linattn_workload_shape():
    wl = inputs.WORKLOADS["linattn"]
    assert (wl.B, wl.H, wl.N, wl.d, wl.dtype, wl.kind) == (64, 16, 2048, 64, "bf16", "tokens")
    # 1024 heads over 148 SMs: the busiest SM takes 7 heads against 6.9 on average
    assert -(-wl.heads // 148) == 7
