"""Write bounds of every entry point, checked with guard bands.

Without a memory checker on the GPU, each buffer a call writes is placed
inside a larger allocation whose head and tail (the guard bands) hold a
fixed byte pattern.  After the call both bands must be unchanged, on ragged
sizes that end inside a chunk or a tile and on single-token heads, so a
kernel that writes one element past (or before) any of its outputs, its
final state or its workspace fails here.  The inputs must be unchanged too.

The guarded outputs are also compared with the same call on plain
allocations, which shows the kernel wrote the whole output and nothing
depends on where it sits: bitwise where the combination order is fixed (the
reduce, the linear attention, the step), and to rounding where a decoupled
look-back folds whatever mix of aggregates and inclusive prefixes it finds
at run time (the forward scan and its final state).  Their values against
the oracle are the parity tests' business."""
import math

import pytest
import torch

from attention_prefix_scan_02_b300 import binding

pytestmark = pytest.mark.gpu

GUARD = 4096      # bytes on each side; a multiple of 16 keeps the body 16-byte aligned
PATTERN = 0xA5


class Guarded:
    """A tensor of `shape` and `dtype` between two guard bands."""

    def __init__(self, shape, dtype):
        esz = torch.empty((), dtype=dtype).element_size()
        self.nbytes = math.prod(shape) * esz
        total = 2 * GUARD + ((self.nbytes + 15) // 16) * 16
        self.raw = torch.full((total,), PATTERN, dtype=torch.uint8, device="cuda")
        self.t = self.raw[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.nbytes:]
        return bool((head == PATTERN).all()) and bool((tail == PATTERN).all())


def _inputs(B, H, N, d, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    q = torch.randn(B, H, d, device="cuda", generator=g).to(dtype)
    K = torch.randn(B, H, N, d, device="cuda", generator=g).to(dtype)
    V = torch.randn(B, H, N, d, device="cuda", generator=g).to(dtype)
    return q, K, V


def _same(a, b):
    torch.testing.assert_close(a.float(), b.float(), rtol=0, atol=0, equal_nan=True)


def _close(a, b):
    """Equal up to the rounding of a different combination order: a few
    float32 ulps, or one bfloat16 ulp of the output."""
    rtol = 2 ** -7 if a.dtype == torch.bfloat16 else 1e-5
    torch.testing.assert_close(a.float(), b.float(), rtol=rtol, atol=1e-6)


DTYPES = [(torch.float32, torch.float32), (torch.bfloat16, torch.bfloat16),
          (torch.bfloat16, torch.float32)]
SIZES = [1, 3, 33, 129, 300]


@pytest.mark.parametrize("d", [16, 32, 64, 128])
@pytest.mark.parametrize("io", DTYPES, ids=["f32", "bf16", "bf16_f32out"])
def test_scan_forward_writes_stay_in_bounds(d, io):
    in_t, out_t = io
    B, H = 1, 3
    for N in SIZES:
        q, K, V = _inputs(B, H, N, d, in_t, seed=N + d)
        K0, V0, q0 = K.clone(), V.clone(), q.clone()
        O = Guarded((B, H, N, d), out_t)
        m, u, w = Guarded((B * H,), torch.float32), Guarded((B * H, d), torch.float32), \
            Guarded((B * H,), torch.float32)
        ws = Guarded((binding.aaren_scan_workspace_bytes(B, H, N, d),), torch.uint8)
        binding.aaren_scan_forward_ex(q, K, V, O.t, m_out=m.t, u_out=u.t, w_out=w.t, workspace=ws.t)
        assert binding.aaren_check() == binding.AAREN_OK
        for name, x in (("O", O), ("m", m), ("u", u), ("w", w), ("workspace", ws)):
            assert x.intact(), f"{name} guard band overwritten at N={N}, d={d}"
        _same(K, K0); _same(V, V0); _same(q, q0)
        Op = torch.empty(B, H, N, d, dtype=out_t, device="cuda")
        mp, up, wp = (torch.empty(B * H, device="cuda"), torch.empty(B * H, d, device="cuda"),
                      torch.empty(B * H, device="cuda"))
        binding.aaren_scan_forward_ex(q, K, V, Op, m_out=mp, u_out=up, w_out=wp)
        assert binding.aaren_check() == binding.AAREN_OK
        _close(O.t, Op); _close(m.t, mp); _close(u.t, up); _close(w.t, wp)

        On = Guarded((B, H, N, d), out_t)
        binding.aaren_scan_forward_noalloc(q, K, V, On.t)
        assert binding.aaren_check() == binding.AAREN_OK
        assert On.intact(), f"noalloc O guard band overwritten at N={N}, d={d}"
        _close(On.t, Op)


@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("io", DTYPES, ids=["f32", "bf16", "bf16_f32out"])
def test_reduce_writes_stay_in_bounds(d, io):
    in_t, out_t = io
    B, H = 2, 3
    for N in SIZES:
        q, K, V = _inputs(B, H, N, d, in_t, seed=3 * N + d)
        o = Guarded((B * H, d), out_t)
        m, u, w = Guarded((B * H,), torch.float32), Guarded((B * H, d), torch.float32), \
            Guarded((B * H,), torch.float32)
        ws = Guarded((binding.aaren_reduce_workspace_bytes(B, H, N, d),), torch.uint8)
        binding.aaren_scan_reduce(q, K, V, o.t, m_out=m.t, u_out=u.t, w_out=w.t, workspace=ws.t)
        assert binding.aaren_check() == binding.AAREN_OK
        for name, x in (("o_N", o), ("m", m), ("u", u), ("w", w), ("workspace", ws)):
            assert x.intact(), f"{name} guard band overwritten at N={N}, d={d}"
        op = torch.empty(B * H, d, dtype=out_t, device="cuda")
        binding.aaren_scan_reduce(q, K, V, op)
        assert binding.aaren_check() == binding.AAREN_OK
        _same(o.t, op)


@pytest.mark.parametrize("d", [32, 128])
@pytest.mark.parametrize("io", DTYPES, ids=["f32", "bf16", "bf16_f32out"])
def test_backward_writes_stay_in_bounds(d, io):
    in_t, out_t = io
    B, H = 1, 2
    for N in (1, 33, 300):
        q, K, V = _inputs(B, H, N, d, in_t, seed=5 * N + d)
        O = Guarded((B, H, N, d), out_t)
        stats = Guarded((B, H, N, 2), torch.float32)
        wsf = Guarded((binding.aaren_scan_workspace_bytes(B, H, N, d),), torch.uint8)
        binding.aaren_scan_forward_stats(q, K, V, O.t, stats.t, workspace=wsf.t)
        assert binding.aaren_check() == binding.AAREN_OK
        for name, x in (("O", O), ("stats", stats), ("workspace", wsf)):
            assert x.intact(), f"forward_stats {name} guard band overwritten at N={N}, d={d}"
        g = torch.Generator(device="cuda")
        g.manual_seed(N)
        dO = torch.randn(B, H, N, d, device="cuda", generator=g).to(out_t)
        dq, dK, dV = Guarded((B * H, d), torch.float32), Guarded((B, H, N, d), torch.float32), \
            Guarded((B, H, N, d), torch.float32)
        wsb = Guarded((binding.aaren_backward_workspace_bytes(B, H, N, d),), torch.uint8)
        binding.aaren_scan_backward(q, K, V, O.t, dO, stats.t, dq.t, dK.t, dV.t, workspace=wsb.t)
        assert binding.aaren_check() == binding.AAREN_OK
        for name, x in (("dq", dq), ("dK", dK), ("dV", dV), ("workspace", wsb)):
            assert x.intact(), f"backward {name} guard band overwritten at N={N}, d={d}"
        assert bool(torch.isfinite(dK.t).all()) and bool(torch.isfinite(dV.t).all())
        assert bool(torch.isfinite(dq.t).all())


@pytest.mark.parametrize("d", [16, 64, 128])
@pytest.mark.parametrize("io", DTYPES, ids=["f32", "bf16", "bf16_f32out"])
def test_step_writes_stay_in_bounds(d, io):
    in_t, out_t = io
    for n in (1, 5, 129):
        g = torch.Generator(device="cuda")
        g.manual_seed(n + d)
        q, k, v = (torch.randn(n, d, device="cuda", generator=g).to(in_t) for _ in range(3))
        m, u, w = Guarded((n,), torch.float32), Guarded((n, d), torch.float32), Guarded((n,), torch.float32)
        o = Guarded((n, d), out_t)
        binding.aaren_state_init(m.t, u.t, w.t)
        for _ in range(3):
            binding.aaren_step(q, m.t, u.t, w.t, k, v, o.t)
        assert binding.aaren_check() == binding.AAREN_OK
        for name, x in (("m", m), ("u", u), ("w", w), ("o_t", o)):
            assert x.intact(), f"{name} guard band overwritten at n={n}, d={d}"
        # three steps with one (k, v) are the mean of three equal values: o = v
        torch.testing.assert_close(o.t.float(), v.float(), rtol=1e-6, atol=1e-6)


@pytest.mark.parametrize("out_t", [torch.bfloat16, torch.float32], ids=["bf16", "f32"])
def test_linattn_writes_stay_in_bounds(out_t):
    B, H, d = 1, 3, 64
    for N in (1, 127, 129, 300):
        g = torch.Generator(device="cuda")
        g.manual_seed(7 * N)
        Q, K, V = (torch.randn(B, H, N, d, device="cuda", generator=g).to(torch.bfloat16) for _ in range(3))
        Q0, K0, V0 = Q.clone(), K.clone(), V.clone()
        O = Guarded((B, H, N, d), out_t)
        S, z = Guarded((B, H, 2, d, d), torch.float32), Guarded((B, H, 2, d), torch.float32)
        binding.aaren_linattn_forward(Q, K, V, O.t, float(N), S_out=S.t, z_out=z.t)
        assert binding.aaren_check() == binding.AAREN_OK
        for name, x in (("O", O), ("S", S), ("z", z)):
            assert x.intact(), f"{name} guard band overwritten at N={N}"
        _same(Q, Q0); _same(K, K0); _same(V, V0)
        Op = torch.empty(B, H, N, d, dtype=out_t, device="cuda")
        Sp, zp = torch.empty(B, H, 2, d, d, device="cuda"), torch.empty(B, H, 2, d, device="cuda")
        binding.aaren_linattn_forward(Q, K, V, Op, float(N), S_out=Sp, z_out=zp)
        assert binding.aaren_check() == binding.AAREN_OK
        _same(O.t, Op); _same(S.t, Sp); _same(z.t, zp)
