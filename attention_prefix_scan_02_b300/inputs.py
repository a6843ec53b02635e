"""Seeded synthetic inputs for the softmax-attention prefix scan.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
callers; it holds none of the method's arithmetic (no scores, exponentials or
sums), only the recipes that draw q, K and V.

Recipe (deterministic, independent of thread count):
  * Every (tensor, b, h) has its own stream: numpy PCG64 seeded with
    SeedSequence([seed, tensor_id, b, h, block]), tensor_id 0 = q, 1 = K,
    2 = V.  Long heads are cut into blocks of BLOCK_ROWS rows, each with its
    own stream, so one head can be drawn in parallel and any head can be
    regenerated on its own.
  * Normal draws are float32 standard normals (numpy's float32 ziggurat),
    drawn row-major [rows, d].  Uniform U(-1, 1) draws are 2x - 1 with x a
    float32 uniform on [0, 1) (exact in float32).
  * bfloat16 workloads round the float32 draws to bfloat16 with
    round-to-nearest-even (torch's conversion); the oracle is fed those
    identical rounded values widened back to float32 (exact).

Workloads (name -> shape and value recipe):
  tiny        B=1, H=1, N=256, d=16, f32, seed 0: q, K, V ~ N(0,1).
  bf16_4k     B=8, H=4, N=4096, d=64, bf16 storage, seed 1: q, K, V ~ N(0,1).
  stress      B=4, H=8, N=16384, d=64, f32, seed 2: q ~ N(0,1); K ~ 8 N(0,1);
              then every 97th key (0-based i with (i+1) % 97 == 0) is set to
              3q, so the running maximum jumps sharply; V ~ U(-1, 1).
  long        B=1, H=16, N=2^20, d=128, bf16 storage, seed 3: q, K, V ~ N(0,1).
  stream      256 streams x H=8, N=4096 steps, d=64, f32, seed 4: one query
              per head drawn once (stream index 0 of the q stream) and shared
              by all 256 streams, as a learned query is; K, V ~ N(0,1) per
              (stream, head).
  linattn     B=64, H=16, N=2048, d=64, bf16 storage, seed 5: the causal
              linear-attention (cosFormer) workload, one query per token:
              Q, K, V ~ N(0,1), each [N, d] per head (Q drawn like K from the
              q stream).  Re-weighting length M = N.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass

import numpy as np

BLOCK_ROWS = 1 << 16

TENSOR_Q, TENSOR_K, TENSOR_V = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str   # storage dtype of q, K, V: "f32" or "bf16"
    seed: int
    kind: str    # "normal", "stress", "stream" or "tokens" (a query per token)

    @property
    def heads(self) -> int:
        return self.B * self.H


WORKLOADS = {
    "tiny": Workload("tiny", 1, 1, 256, 16, "f32", 0, "normal"),
    "bf16_4k": Workload("bf16_4k", 8, 4, 4096, 64, "bf16", 1, "normal"),
    "stress": Workload("stress", 4, 8, 16384, 64, "f32", 2, "stress"),
    "long": Workload("long", 1, 16, 1 << 20, 128, "bf16", 3, "normal"),
    "stream": Workload("stream", 256, 8, 4096, 64, "f32", 4, "stream"),
    "linattn": Workload("linattn", 64, 16, 2048, 64, "bf16", 5, "tokens"),
}


def custom(B, H, N, d, dtype="f32", seed=100, kind="normal", name="custom") -> Workload:
    """A workload of any shape with one of the value recipes above."""
    return Workload(name, B, H, N, d, dtype, seed, kind)


def _rng(seed, tensor_id, b, h, block):
    return np.random.Generator(np.random.PCG64(
        np.random.SeedSequence([seed, tensor_id, b, h, block])))


def _normal_rows(seed, tensor_id, b, h, rows, d, out=None):
    out = np.empty((rows, d), dtype=np.float32) if out is None else out
    for blk, r0 in enumerate(range(0, rows, BLOCK_ROWS)):
        r1 = min(rows, r0 + BLOCK_ROWS)
        _rng(seed, tensor_id, b, h, blk).standard_normal(
            (r1 - r0, d), dtype=np.float32, out=out[r0:r1])
    return out


def _uniform_rows(seed, tensor_id, b, h, rows, d):
    out = np.empty((rows, d), dtype=np.float32)
    for blk, r0 in enumerate(range(0, rows, BLOCK_ROWS)):
        r1 = min(rows, r0 + BLOCK_ROWS)
        x = _rng(seed, tensor_id, b, h, blk).random((r1 - r0, d), dtype=np.float32)
        out[r0:r1] = np.float32(2.0) * x - np.float32(1.0)
    return out


def round_bf16(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (RNE) and widen back to float32."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(
        torch.bfloat16).to(torch.float32).numpy()


def head_query(wl: Workload, b: int, h: int) -> np.ndarray:
    """q for head (b, h), float32 [d] (bf16-rounded for bf16 workloads)."""
    qb = 0 if wl.kind == "stream" else b
    q = _normal_rows(wl.seed, TENSOR_Q, qb, h, 1, wl.d)[0]
    return round_bf16(q) if wl.dtype == "bf16" else q


def head_inputs(wl: Workload, b: int, h: int):
    """(q [d], K [N, d], V [N, d]) for head (b, h) as float32 numpy arrays
    holding the workload's stored values (bf16-rounded for bf16 workloads)."""
    q = head_query(wl, b, h)
    if wl.kind == "stress":
        K = _normal_rows(wl.seed, TENSOR_K, b, h, wl.N, wl.d)
        K *= np.float32(8.0)
        idx = np.arange(96, wl.N, 97)
        K[idx] = np.float32(3.0) * q
        V = _uniform_rows(wl.seed, TENSOR_V, b, h, wl.N, wl.d)
    else:
        K = _normal_rows(wl.seed, TENSOR_K, b, h, wl.N, wl.d)
        V = _normal_rows(wl.seed, TENSOR_V, b, h, wl.N, wl.d)
    if wl.dtype == "bf16":
        K, V = round_bf16(K), round_bf16(V)
    return q, K, V


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def batch_inputs(wl: Workload, device=None, threads: int | None = None, b0: int = 0):
    """All heads as torch tensors in the storage dtype:
    q [B, H, d], K [B, H, N, d], V [B, H, N, d].

    Row b of the result holds batch entry b0 + b of the recipe (a shard of a
    larger batch: with b0 = r * B, rank r of a multi-GPU run draws its own
    heads).  Heads are drawn on a thread pool and copied into the (optionally
    device) tensors one head at a time, so host memory holds only a few
    heads."""
    import torch
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    dev = torch.device("cpu") if device is None else torch.device(device)
    q = torch.empty((wl.B, wl.H, wl.d), dtype=tdt, device=dev)
    K = torch.empty((wl.B, wl.H, wl.N, wl.d), dtype=tdt, device=dev)
    V = torch.empty((wl.B, wl.H, wl.N, wl.d), dtype=tdt, device=dev)
    threads = threads or default_threads()

    def one(bh):
        b, h = divmod(bh, wl.H)
        qh, Kh, Vh = head_inputs(wl, b0 + b, h)
        return bh, qh, Kh, Vh

    workers = min(threads, max(1, wl.heads))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        for w0 in range(0, wl.heads, workers):   # bounded: one wave of heads in memory
            for bh, qh, Kh, Vh in ex.map(one, range(w0, min(wl.heads, w0 + workers))):
                b, h = divmod(bh, wl.H)
                q[b, h].copy_(torch.from_numpy(qh).to(tdt))
                K[b, h].copy_(torch.from_numpy(Kh).to(tdt))
                V[b, h].copy_(torch.from_numpy(Vh).to(tdt))
    return q, K, V


def head_token_inputs(wl: Workload, b: int, h: int):
    """(Q [N, d], K [N, d], V [N, d]) of head (b, h) for workloads with one
    query per token, float32 numpy holding the stored values."""
    Q = _normal_rows(wl.seed, TENSOR_Q, b, h, wl.N, wl.d)
    K = _normal_rows(wl.seed, TENSOR_K, b, h, wl.N, wl.d)
    V = _normal_rows(wl.seed, TENSOR_V, b, h, wl.N, wl.d)
    if wl.dtype == "bf16":
        Q, K, V = round_bf16(Q), round_bf16(K), round_bf16(V)
    return Q, K, V


def token_inputs(wl: Workload, device=None, threads: int | None = None, b0: int = 0):
    """Q, K, V [B, H, N, d] torch tensors in the storage dtype (one query per
    token); batch entries b0 .. b0 + B - 1 of the recipe."""
    import torch
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    dev = torch.device("cpu") if device is None else torch.device(device)
    out = [torch.empty((wl.B, wl.H, wl.N, wl.d), dtype=tdt, device=dev) for _ in range(3)]
    threads = threads or default_threads()

    def one(bh):
        b, h = divmod(bh, wl.H)
        return bh, head_token_inputs(wl, b0 + b, h)

    workers = min(threads, max(1, wl.heads))
    with ThreadPoolExecutor(max_workers=workers) as ex:
        for w0 in range(0, wl.heads, workers):
            for bh, arrs in ex.map(one, range(w0, min(wl.heads, w0 + workers))):
                b, h = divmod(bh, wl.H)
                for t, a in zip(out, arrs):
                    t[b, h].copy_(torch.from_numpy(a).to(tdt))
    return tuple(out)
