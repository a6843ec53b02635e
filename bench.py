#!/usr/bin/env python3
"""Benchmark of the softmax-attention prefix scan on one or more B300 GPUs.

One step = one aaren_scan_forward over the whole workload (scores, chunk
scan, cross-chunk carry, output), inputs resident in HBM.  The default
workload is the long sequence: B=1, H=16, N=2^20 tokens, d=128, q/K/V
bfloat16 ~ N(0,1) (seed 3), bfloat16 output, float32 arithmetic.  Its inputs
(8.6 GB of K and V) are far larger than L2 (126 MB), so no L2 flush is needed
between steps.

Prints ONE JSON line (rank 0):
  value      head-tokens/s (B*H*N per step / mean step time, all ranks)
  roofline   HBM roofline of the scan kernel: algorithmic bytes (K and V read
             once, O written once) per launch / mean launch time, against the
             measured HBM copy peak
  e2e        the same metric through the C ABI with host buffers: per step
             host->device copy of q, K, V from pinned memory, the scan, and the
             device->host copy of O
  cpu_baseline  the float64 oracle timed on this host's cores on a bounded
             sample of the same workload
With torchrun (N > 1) every rank runs its own copy of the workload (heads are
independent: no collective on the data path), the step time is the maximum
over ranks and value counts the head-tokens of all ranks (weak scaling).

`--impl reference` times the float64 oracle instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_HBM_GBS = 6400.0
CPU_SAMPLE_TOKENS = 1 << 18      # per head, cpu_baseline leg
CPU_SAMPLE_MIN_S = 1.0           # cpu_baseline: repeat the sample until this much wall time
CPU_SAMPLE_RUNS = 3              # cpu_baseline: timed runs averaged
CPU_SAMPLE_MAX_PASSES = 100000   # passes are bounded by time (CPU_SAMPLE_MIN_S), not count
METRIC = "Aaren scan tokens/s and achieved HBM GB/s (% of B300 peak), 1 GPU"


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="long", choices=["tiny", "bf16_4k", "stress", "long"])
    ap.add_argument("--heads", type=int, default=0, help="override H (profiling small cases)")
    ap.add_argument("--batch", type=int, default=0, help="override B (profiling small cases)")
    ap.add_argument("--tokens", type=int, default=0, help="override N (profiling small cases)")
    ap.add_argument("--out-dtype", default="", choices=["", "bf16", "f32"])
    ap.add_argument("--op", default="scan", choices=["scan", "reduce", "backward", "step", "linattn"],
                    help="scan: every prefix output (the headline); reduce: the many-to-one "
                         "form (o_N and the final state only); backward: dq, dK, dV of the "
                         "scan from O, dO and the saved per-prefix statistics; step: the "
                         "one-token update of many streams (the stream workload); linattn: "
                         "the causal cos-re-weighted linear attention (the linattn workload)")
    return ap.parse_args()


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(x, dist, device):
    """The largest of every rank's `x` (a step time); `dist` is
    torch.distributed with an initialised process group, or None for one
    rank.  Every rank gets the result."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, step_ms):
    """Units processed by all ranks per second, each rank doing the same
    `units_per_rank` in a step of `step_ms` (the slowest rank's): weak
    scaling, so the job's work grows with the number of ranks."""
    return world * units_per_rank / (step_ms * 1e-3)


def e2e_pieces(wl):
    """Head ranges [h0, h1) of the flattened B*H heads for the end-to-end
    leg's copy/compute overlap: up to 8 pieces of at least 2 heads (a piece
    of a single long head leaves the look-back too deep to keep up with the
    copies); a workload under 256 MB of K and V is one piece."""
    in_b = 2 if wl.dtype == "bf16" else 4
    if wl.heads * wl.N * wl.d * 2 * in_b < (1 << 28) or wl.heads < 4:
        return [(0, wl.heads)]
    n = min(8, wl.heads // 2)
    bounds = [round(i * wl.heads / n) for i in range(n + 1)]
    return [(bounds[i], bounds[i + 1]) for i in range(n)]


def workload(args):
    from attention_prefix_scan_02_b300 import inputs
    wl = inputs.WORKLOADS[args.workload]
    if args.heads or args.tokens or args.batch:
        wl = inputs.custom(args.batch or wl.B, args.heads or wl.H, args.tokens or wl.N, wl.d, wl.dtype, wl.seed,
                           wl.kind, wl.name if not args.tokens else f"{wl.name}_N{args.tokens}")
    return wl


# a GPU spin queued ahead of a start event (before the first timed launch,
# and after each L2 flush): about 0.15 ms at 2 GHz, longer than the host
# needs to issue the launch, so the GPU never idles inside the timed window
# waiting for it.  The spin itself is outside every timed window.
SPIN_CYCLES = 300_000


def needs_flush(wl):
    """True when one step's K and V (under 256 MB) could stay in the 126 MB
    L2 between steps: the bench then flushes L2 before every timed launch."""
    in_b = 2 if wl.dtype == "bf16" else 4
    return wl.heads * wl.N * wl.d * 2 * in_b < (1 << 28)


def flush_l2(flush):
    """Evict K and V from L2 (a write of twice its size), then queue the GPU
    spin so the next launch is already queued when its start event runs."""
    import torch
    flush.fill_(1.0)
    torch.cuda._sleep(SPIN_CYCLES)


def describe(wl, out):
    recipe = {"normal": "q, K, V ~ N(0,1)",
              "stress": "q ~ N(0,1), K ~ 8 N(0,1), every 97th key = 3q, V ~ U(-1,1)",
              "stream": "per-head q shared by streams, K, V ~ N(0,1)"}[wl.kind]
    return {"workload": f"{wl.name}: B={wl.B} H={wl.H} N={wl.N} d={wl.d}, {wl.dtype} in, {out} out, "
                        f"{recipe}, seed {wl.seed}",
            "B": wl.B, "H": wl.H, "N": wl.N, "d": wl.d, "in_dtype": wl.dtype, "out_dtype": out,
            "l2": ("L2 flushed (a write of 2x its size) before every timed launch, then a GPU spin so the "
                   "launch is queued before its start event") if needs_flush(wl)
            else "no flush: K+V per step larger than the 126 MB L2"}


# the source files each profiled kernel is built from (its own code, what it
# includes, and the host file that picks its launch shape)
KERNEL_SOURCES = {
    "k_scan_pipe": ["scan_pipe_kernel.cuh", "scan_kernel.cuh", "common.cuh", "ptx.cuh", "aaren_api.cu"],
    "k_linattn": ["linattn_kernel.cuh", "tc.cuh", "scan_kernel.cuh", "common.cuh", "ptx.cuh", "aaren_api.cu"],
}


def kernel_source_hash(kernel):
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "attention_prefix_scan_02_b300", "csrc")
    for fn in sorted(KERNEL_SOURCES[kernel]):
        with open(os.path.join(csrc, fn), "rb") as f:
            h.update(fn.encode() + f.read())
    return h.hexdigest()[:16]


def profiled_traffic(wl, out, record="scan_long_bf16_traffic.json", kernel="k_scan_pipe"):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current source of the kernel with this head size, dtype and output
    type; else None.  When the capture is of a smaller case (the full launch
    is too large for a multi-pass capture), reads are scaled to this launch's
    head-tokens (every input byte is read once, so reads grow in proportion),
    and writes are the algorithmic output bytes less the capture's write
    shortfall: the tail of the output still in L2 when the kernel ends, a
    fixed residue of the L2's size, not a per-token rate."""
    path = os.path.join(ROOT, "profiles", record)
    try:
        with open(path) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("kernel_source_sha") != kernel_source_hash(kernel):
        return None
    if (rec.get("d") != wl.d or rec.get("in_dtype") != wl.dtype or rec.get("out_dtype") != out):
        return None
    try:
        cap_tokens = rec["head_tokens"]
        alg_w = rec["algorithmic_write_bytes_per_head_token"]
        reads = rec["dram_bytes_read"] / cap_tokens * wl.heads * wl.N
        residue = max(0.0, cap_tokens * alg_w - rec["dram_bytes_write"])
        writes = max(0.0, wl.heads * wl.N * alg_w - residue)
    except (KeyError, TypeError, ZeroDivisionError):
        return None
    return int(reads + writes)


def measured_peak():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            mp = json.load(f)
        return float(mp["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs, copy read+write)"
    except (OSError, ValueError, KeyError):
        return FALLBACK_HBM_GBS, "fallback (6.4 TB/s, earlier B300 measurement)"


class ClockSampler:
    """nvidia-smi clock and throttle-reason samples every 20 ms; summary()
    keeps the samples taken inside [begin, end] (host wall clock), the timed
    region (or, when it is shorter than the sampling period, the samples
    nearest to it)."""
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = None
        self.begin = None
        self.end = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "20"],
                stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    def summary(self):
        import datetime
        if self.proc is None or self.path is None:
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                    rows.append((ts, float(parts[1]), float(parts[2]), parts[5:9]))
                except ValueError:
                    continue
        os.unlink(self.path)
        if not rows:
            return None
        inside = [r for r in rows if self.begin is not None and self.begin <= r[0] <= self.end]
        where = "inside the timed region"
        if not inside and self.begin is not None:
            mid = 0.5 * (self.begin + self.end)
            inside = sorted(rows, key=lambda r: abs(r[0] - mid))[:2]
            where = "nearest to the timed region (shorter than the sampling period)"
        rows = inside or rows
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, _, r in rows for i, v in enumerate(r) if v == "Active"})
        return {"sm_mhz": statistics.median(r[1] for r in rows), "sm_max_mhz": max(r[2] for r in rows),
                "reasons": reasons, "samples": len(rows), "samples_taken": where}


class OracleTimer:
    """The float64 oracle, as it stands, timed on this host's cores.  `items`
    holds one head's inputs each; `fn(item, out)` runs the oracle on one head
    writing its output into `out`.  Inputs are drawn, every output array is
    allocated and first-touched, and the thread pool is started before any
    clock starts; warm(min_s) then runs untimed passes for `min_s` seconds
    (drawing the inputs uses torch's CPU thread pool, whose idle workers keep
    spinning on the cores for a while afterwards), so a timed pass is the
    oracle's own work on quiet cores.  run(min_s) repeats whole passes over
    the items until `min_s` seconds have elapsed and returns (head-tokens/s,
    seconds, passes)."""

    def __init__(self, fn, items, tokens, d, threads):
        import numpy as np
        from concurrent.futures import ThreadPoolExecutor
        self.fn, self.items, self.tokens, self.threads = fn, items, tokens, threads
        self.outs = [np.ones((tokens, d), dtype=np.float64) for _ in items]
        self.pool = ThreadPoolExecutor(max_workers=threads) if threads > 1 else None

    def warm(self, min_s):
        t0 = time.perf_counter()
        while True:
            self.one_pass()
            if time.perf_counter() - t0 >= min_s:
                break

    def _one(self, i):
        self.fn(self.items[i], self.outs[i])

    def one_pass(self):
        if self.pool is None:
            for i in range(len(self.items)):
                self._one(i)
        else:
            list(self.pool.map(self._one, range(len(self.items))))

    def run(self, min_s):
        passes = 0
        t0 = time.perf_counter()
        while True:
            self.one_pass()
            passes += 1
            dt = time.perf_counter() - t0
            if dt >= min_s or passes >= CPU_SAMPLE_MAX_PASSES:
                break
        return passes * len(self.items) * self.tokens / dt, dt, passes

    def close(self):
        if self.pool is not None:
            self.pool.shutdown()
        self.outs = []


def scan_oracle_timer(wl, tokens_per_head, threads, heads=None):
    """OracleTimer over the first `tokens_per_head` tokens of the first
    `heads` heads (all by default) of workload `wl`."""
    import oracle
    from attention_prefix_scan_02_b300 import inputs
    n = min(tokens_per_head, wl.N)
    sub = inputs.custom(wl.B, wl.H, n, wl.d, wl.dtype, wl.seed, wl.kind, wl.name)
    hs = [(b, h) for b in range(wl.B) for h in range(wl.H)][:heads or wl.heads]
    items = [inputs.head_inputs(sub, b, h) for b, h in hs]
    return OracleTimer(lambda x, out: oracle.scan(*x, out=out), items, n, wl.d, min(threads, len(items)))


def cpu_baseline_leg(wl, threads):
    """The oracle on the scan workload's sample: all host threads over the
    first CPU_SAMPLE_TOKENS tokens of every head, and one thread over the
    first CPU_SAMPLE_TOKENS / 4 tokens of head 0."""
    t = scan_oracle_timer(wl, CPU_SAMPLE_TOKENS, threads)
    t.warm(CPU_SAMPLE_MIN_S)
    runs = [t.run(CPU_SAMPLE_MIN_S) for _ in range(CPU_SAMPLE_RUNS)]   # as the reference arm's steps
    rate = statistics.mean(r for r, _, _ in runs)
    dt = sum(d for _, d, _ in runs)
    passes = sum(n for _, _, n in runs)
    n, nh, used = t.tokens, len(t.items), t.threads
    t.close()
    cpu = {"value": rate, "unit": "head-tokens/s", "cores": used, "kind": "oracle",
           "sample": f"the first {n} tokens of all {nh} heads ({n * nh} head-tokens): the mean of "
                     f"{CPU_SAMPLE_RUNS} runs of at least {CPU_SAMPLE_MIN_S:.0f} s ({passes} passes, "
                     f"{dt:.1f} s wall on {used} threads, about {dt * used:.0f} CPU-seconds), after "
                     f"{CPU_SAMPLE_MIN_S:.0f} s of untimed passes"}
    t1 = scan_oracle_timer(wl, CPU_SAMPLE_TOKENS // 4, 1, heads=1)
    t1.warm(0.2)
    r1, dt1, passes1 = t1.run(CPU_SAMPLE_MIN_S)
    t1.close()
    cpu["single_thread"] = {"value": r1, "unit": "head-tokens/s", "cores": 1,
                            "sample": f"the first {t1.tokens} tokens of head 0, {passes1} passes, "
                                      f"{dt1:.1f} s"}
    return cpu


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def run_reference(args):
    """The oracle arm: the float64 oracle timed on this host's cores, one
    step = repeated passes over the cpu_baseline leg's sample (the first
    CPU_SAMPLE_TOKENS tokens of every head, one thread per head) for at
    least CPU_SAMPLE_MIN_S seconds, so the two report one measurement."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    wl = workload(args)
    out = args.out_dtype or wl.dtype
    threads = min(host_cores(), wl.heads)
    timer = scan_oracle_timer(wl, CPU_SAMPLE_TOKENS, threads)
    timer.warm(CPU_SAMPLE_MIN_S)
    rates = []
    for i in range(args.warmup + args.steps):
        r, dt, passes = timer.run(CPU_SAMPLE_MIN_S if i >= args.warmup else 0.0)
        if i >= args.warmup:
            rates.append((r, dt, passes))
    n, nh, used = timer.tokens, len(timer.items), timer.threads
    timer.close()
    sample = (f"each step: passes over the first {n} tokens of all {nh} heads ({n * nh} head-tokens) "
              f"for at least {CPU_SAMPLE_MIN_S:.0f} s on {used} threads "
              f"({statistics.mean(p for _, _, p in rates):.1f} passes a step on average)")
    value = statistics.mean(r for r, _, _ in rates)
    line = {"impl": "reference", "metric": METRIC,
            "value": value, "unit": "head-tokens/s", "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(dt for _, dt, _ in rates),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": describe(wl, out),
            "cpu_baseline": {"value": value, "unit": "head-tokens/s", "cores": used,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": "head-tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    from attention_prefix_scan_02_b300 import binding, build, inputs
    build.build()
    wl = workload(args)
    out = args.out_dtype or wl.dtype
    out_t = torch.bfloat16 if out == "bf16" else torch.float32
    in_t = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    warmup = max(3, args.warmup)

    # CPU baseline first (host memory is freed before the GPU legs)
    cpu = None
    if rank == 0:
        cpu = cpu_baseline_leg(wl, min(host_cores(), wl.heads))

    # rank r draws batch entries [r B, (r + 1) B) of the recipe: the ranks
    # together process a batch of world * B sequences (weak scaling)
    q, K, V = inputs.batch_inputs(wl, device="cuda", b0=rank * wl.B)
    reduce = args.op == "reduce"
    backward = args.op == "backward"
    O = torch.empty((wl.B, wl.H, wl.d) if reduce else K.shape, dtype=out_t, device="cuda")
    if reduce:
        ws = binding.new_reduce_workspace(wl.B, wl.H, wl.N, wl.d)
    elif backward:
        ws = binding.new_backward_workspace(wl.B, wl.H, wl.N, wl.d)
        # the step's forward (untimed) and an upstream gradient dL/dO ~ N(0, 1)
        stats = torch.empty(wl.B, wl.H, wl.N, 2, dtype=torch.float32, device="cuda")
        binding.aaren_scan_forward_stats(q, K, V, O, stats)
        gwl = inputs.custom(wl.B, wl.H, wl.N, wl.d, dtype=out, seed=wl.seed + 7777)
        dO = inputs.batch_inputs(gwl, device="cuda", b0=rank * wl.B)[2]
        g_q = torch.empty(wl.B, wl.H, wl.d, dtype=torch.float32, device="cuda")
        g_K = torch.empty(K.shape, dtype=torch.float32, device="cuda")
        g_V = torch.empty(K.shape, dtype=torch.float32, device="cuda")
    else:
        ws = binding.new_workspace(wl.B, wl.H, wl.N, wl.d)
    stream = torch.cuda.current_stream()
    in_b = 2 if wl.dtype == "bf16" else 4
    out_b = 2 if out == "bf16" else 4
    elems = wl.heads * wl.N * wl.d
    # algorithmic bytes: K, V read once (+ O written once for the scan); the
    # backward reads K, V, O, dO and the per-prefix (m, w) once and writes
    # dK, dV (float32) once
    if backward:
        alg_bytes = elems * (2 * in_b + 2 * out_b + 2 * 4) + wl.heads * wl.N * 8
    else:
        alg_bytes = elems * (2 * in_b + (0 if reduce else out_b))
    tokens = wl.heads * wl.N
    flush = None
    if needs_flush(wl):                             # small workloads sit in L2: flush it
        flush = torch.empty(2 * torch.cuda.get_device_properties(0).L2_cache_size // 4 + 1,
                            dtype=torch.float32, device="cuda")

    def call(q, K, V, O):
        if reduce:
            binding.aaren_scan_reduce(q, K, V, O, workspace=ws, stream=stream)
        elif backward:
            binding.aaren_scan_backward(q, K, V, O, dO, stats, g_q, g_K, g_V, workspace=ws,
                                        stream=stream)
        else:
            binding.aaren_scan_forward_ex(q, K, V, O, workspace=ws, stream=stream)

    def step():
        call(q, K, V, O)

    for _ in range(warmup):
        if flush is not None:
            flush_l2(flush)
        step()
    if binding.aaren_check() != binding.AAREN_OK:
        raise SystemExit("device status error during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        clocks.begin = time.time()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(SPIN_CYCLES)   # the host issues the first launches meanwhile
        t_start.record(stream)
        for i in range(args.steps):
            if flush is not None:
                flush_l2(flush)
            starts[i].record(stream)
            step()
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        clocks.end = time.time()
    if dist is not None:
        dist.barrier()
    status = binding.aaren_check()
    if status != binding.AAREN_OK:
        raise SystemExit(f"device status error in the timed region: {binding.status_string(status)}")
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    mean_launch_ms = statistics.mean(launch_ms)
    launch_spread = {"launch_ms_median": statistics.median(launch_ms), "launch_ms_min": min(launch_ms)}
    step_ms = mean_launch_ms if flush is not None else t_start.elapsed_time(t_end) / args.steps
    step_ms = max_over_ranks(step_ms, dist, "cuda")

    # end to end through the C ABI with host buffers
    e2e = None
    if backward:
        e2e = {"value": None, "not_measured": "the backward's host copies (K, V, O, dO in; dK, dV "
                                              "out: 34 GB a step at full size) are not timed; see the "
                                              "scan's line for the end-to-end figure"}
    if (rank == 0 or world > 1) and not backward:
        hq = torch.empty(q.shape, dtype=in_t, pin_memory=True)
        hK = torch.empty(K.shape, dtype=in_t, pin_memory=True)
        hV = torch.empty(V.shape, dtype=in_t, pin_memory=True)
        hO = torch.empty(O.shape, dtype=out_t, pin_memory=True)
        hq.copy_(q); hK.copy_(K); hV.copy_(V)
        dq, dK, dV, dO = q, K, V, O          # device buffers are reused
        e2e_steps = max(1, min(args.steps, 3))
        pieces = e2e_pieces(wl)
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in pieces]
        ev_done = [torch.cuda.Event() for _ in pieces]
        flat = lambda t: t.view(wl.heads, *t.shape[2:])
        hKf, hVf, dKf, dVf = flat(hK), flat(hV), flat(dK), flat(dV)
        hqf, dqf = hq.view(wl.heads, wl.d), dq.view(wl.heads, wl.d)
        hOf, dOf = hO.view(wl.heads, *O.shape[2:]), dO.view(wl.heads, *O.shape[2:])

        def e2e_step():
            """Heads in pieces: the host->device copy of piece i+1 (copy
            stream), the call on piece i (the compute stream) and the
            device->host copy of piece i-1 (a second copy stream) overlap, so
            the two transfer directions run at once."""
            s_in.wait_stream(stream)
            s_out.wait_stream(stream)
            with torch.cuda.stream(s_in):
                dq.copy_(hq, non_blocking=True)
            for i, (h0, h1) in enumerate(pieces):
                with torch.cuda.stream(s_in):
                    dKf[h0:h1].copy_(hKf[h0:h1], non_blocking=True)
                    dVf[h0:h1].copy_(hVf[h0:h1], non_blocking=True)
                    ev_in[i].record(s_in)
                stream.wait_event(ev_in[i])
                n = h1 - h0
                sub = lambda t: t[h0:h1].view(1, n, *t.shape[1:])
                call(sub(dqf), sub(dKf), sub(dVf), sub(dOf))
                ev_done[i].record(stream)
                s_out.wait_event(ev_done[i])
                with torch.cuda.stream(s_out):
                    hOf[h0:h1].copy_(dOf[h0:h1], non_blocking=True)
            stream.wait_stream(s_out)

        e2e_step()
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        b.record(stream)
        torch.cuda.synchronize()
        e2e_ms = a.elapsed_time(b) / e2e_steps
        e2e_ms = max_over_ranks(e2e_ms, dist, "cuda")
        if binding.aaren_check() != binding.AAREN_OK:
            raise SystemExit("device status error in the end-to-end leg")
        h2d = (hq.numel() + hK.numel() + hV.numel()) * in_b
        e2e = {"value": whole_job_rate(tokens, world, e2e_ms), "unit": "head-tokens/s",
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": hO.numel() * out_b,
               "ms_per_step": e2e_ms, "steps": e2e_steps,
               "path": ("pinned host q,K,V -> device, aaren_scan_reduce, device o_N -> pinned host"
                        if reduce else
                        "pinned host q,K,V -> device, aaren_scan_forward_ex, device O -> pinned host"),
               "pieces": f"{len(pieces)} piece(s) of heads; the host->device copy, the call and the "
                         f"device->host copy of consecutive pieces overlap on three streams"}
        del hq, hK, hV, hO

    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0

    peak, peak_src = measured_peak()
    achieved = alg_bytes / (mean_launch_ms * 1e-3) / 1e9
    traffic = None if (reduce or backward) else profiled_traffic(wl, out)
    line = {
        "metric": METRIC,
        "value": whole_job_rate(tokens, world, step_ms),
        "unit": "head-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "io_dtype": f"{wl.dtype} in, {out} out", "data": "synthetic",
        "config": dict(describe(wl, out), op=args.op, global_batch=world * wl.B,
                       parallelism=f"independent sequences, {world} rank(s), no collective"),
        # a scan call launches the workspace zeroing (k_zero_ws) and the scan;
        # the reduce and the backward zero theirs with a driver memset
        "gpu_launches": args.steps if (reduce or backward) else 2 * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "algorithmic_bytes_per_launch": alg_bytes, "launch_ms": mean_launch_ms,
                     **launch_spread, "peak_source": peak_src,
                     "kernel": "k_scan_reduce" if reduce else "k_scan_bwd" if backward else
                               ("k_scan_pipe" if (wl.dtype == "bf16" or wl.d == 64) else "k_scan_fwd")},
        "cpu_baseline": cpu,
        "e2e": e2e,
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def run_step(args):
    """The constant-memory one-token update of many streams: every stream of
    the stream workload (256 x 8 = 2048 streams, d = 64, float32) advances
    by one token per aaren_step call, for all 4096 tokens.  Timed two ways:
    plain launches through the binding (each call pays the host launch
    cost), and the same 4096 calls captured once in a CUDA graph and
    replayed (the device time of a step).  A step moves 1.6 MB of K, V and
    O (plus 1.1 MB of state read and written): it is launch-bound."""
    import torch

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    from attention_prefix_scan_02_b300 import binding, build, inputs
    build.build()
    wl = inputs.WORKLOADS["stream"]
    n, d, T = wl.heads, wl.d, wl.N
    q, K, V = inputs.batch_inputs(wl, b0=rank * wl.B)
    qs = q.reshape(n, d).cuda()
    Ks = K.permute(2, 0, 1, 3).reshape(T, n, d).contiguous().cuda()
    Vs = V.permute(2, 0, 1, 3).reshape(T, n, d).contiguous().cuda()
    del K, V
    Os = torch.empty((T, n, d), dtype=torch.float32, device="cuda")
    m = torch.empty(n, device="cuda"); u = torch.empty(n, d, device="cuda")
    w = torch.empty(n, device="cuda")
    stream = torch.cuda.current_stream()

    def sequence():
        binding.aaren_state_init(m, u, w, stream=stream)
        for t in range(T):
            binding.aaren_step(qs, m, u, w, Ks[t], Vs[t], Os[t], stream=stream)

    warmup = max(3, args.warmup)
    steps = max(1, min(args.steps, 5))
    for _ in range(warmup):
        sequence()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(steps):
        sequence()
    b.record(stream)
    torch.cuda.synchronize()
    plain_us = a.elapsed_time(b) * 1e3 / (steps * T)

    gs = torch.cuda.Stream()
    gs.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=gs):
        binding.aaren_state_init(m, u, w)
        for t in range(T):
            binding.aaren_step(qs, m, u, w, Ks[t], Vs[t], Os[t])
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        clocks.begin = time.time()
        a.record(stream)
        for _ in range(steps):
            g.replay()
        b.record(stream)
        torch.cuda.synchronize()
        clocks.end = time.time()
    graph_us = a.elapsed_time(b) * 1e3 / (steps * T)
    if binding.aaren_check() != binding.AAREN_OK:
        raise SystemExit("device status error in the step benchmark")
    if rank != 0:
        return 0
    step_bytes = n * d * 4 * 3            # k_t, v_t read, o_t written
    peak, peak_src = measured_peak()
    line = {
        "metric": METRIC + " (one-token step of many streams)",
        "value": world * n / (graph_us * 1e-6), "unit": "head-tokens/s",
        "n_gpus": world, "steps": steps, "warmup": warmup,
        "ms_per_step": graph_us * 1e-3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": f"stream: {wl.B} streams x {wl.H} heads = {n} streams, d={d}, "
                               f"{T} tokens each, f32, seed {wl.seed}", "op": "step",
                   "l2": "state and one token per stream are L2-resident by design"},
        "gpu_launches": steps * (T + 1),
        "step_us": {"cuda_graph": graph_us, "plain_launches": plain_us},
        "roofline": {"bound": "launch", "achieved": step_bytes / (graph_us * 1e-6) / 1e9,
                     "peak": peak, "unit": "GB/s", "frac": step_bytes / (graph_us * 1e-6) / 1e9 / peak,
                     "traffic": None, "algorithmic_bytes_per_launch": step_bytes,
                     "peak_source": peak_src, "kernel": "k_step"},
        "e2e": {"value": world * n / (plain_us * 1e-6), "unit": "head-tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0,
                "path": "plain aaren_step calls through the binding, device-resident tokens"},
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    return 0


LA_CPU_TOKENS = 512        # oracle sample: leading tokens of each sampled head
LA_CPU_HEADS = 64


def la_oracle_timer(wl, tokens, heads, threads):
    """OracleTimer for the float64 linear-attention oracle over the first
    `tokens` tokens of the first `heads` heads of workload `wl`."""
    import oracle
    from attention_prefix_scan_02_b300 import inputs
    n = min(tokens, wl.N)
    sub_wl = inputs.custom(wl.B, wl.H, n, wl.d, wl.dtype, wl.seed, wl.kind, wl.name)
    hs = [(b, h) for b in range(wl.B) for h in range(wl.H)][:heads]
    items = [inputs.head_token_inputs(sub_wl, b, h) for b, h in hs]
    M = float(wl.N)
    return OracleTimer(lambda x, out: oracle.la_scan(*x, M, out=out), items, n, wl.d,
                       min(threads, len(items)))


def run_linattn(args):
    """The causal cos-re-weighted linear attention on the linattn workload
    (B=64, H=16, N=2048, d=64, bf16 in; one query per token): one
    aaren_linattn_forward per step, inputs resident in HBM (1.07 GB of Q, K,
    V, larger than L2).  Algorithmic bytes: Q, K, V read once and O written
    once per head-token."""
    import torch

    rank, world, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from attention_prefix_scan_02_b300 import binding, build, inputs
    build.build()
    wl = inputs.WORKLOADS["linattn"]
    if args.batch:   # a smaller case for profiling: fewer sequences of the same recipe
        wl = inputs.custom(args.batch, wl.H, wl.N, wl.d, wl.dtype, wl.seed, wl.kind, f"{wl.name}_B{args.batch}")
    out = args.out_dtype or wl.dtype
    out_t = torch.bfloat16 if out == "bf16" else torch.float32
    warmup = max(3, args.warmup)
    cpu = None
    if rank == 0:
        t = la_oracle_timer(wl, LA_CPU_TOKENS, LA_CPU_HEADS, host_cores())
        t.warm(CPU_SAMPLE_MIN_S)
        rate, dt, passes = t.run(CPU_SAMPLE_MIN_S)
        n, nh, used = t.tokens, len(t.items), t.threads
        t.close()
        cpu = {"value": rate, "unit": "head-tokens/s", "cores": used, "kind": "oracle",
               "sample": f"the first {n} tokens of {nh} heads ({n * nh} head-tokens), {passes} passes, "
                         f"{dt:.1f} s wall on {used} threads"}
        t1 = la_oracle_timer(wl, LA_CPU_TOKENS, 1, 1)
        t1.warm(0.2)
        r1, dt1, passes1 = t1.run(CPU_SAMPLE_MIN_S)
        t1.close()
        cpu["single_thread"] = {"value": r1, "unit": "head-tokens/s", "cores": 1,
                                "sample": f"the first {t1.tokens} tokens of head 0, {passes1} passes, "
                                          f"{dt1:.1f} s"}
    Q, K, V = inputs.token_inputs(wl, device="cuda", b0=rank * wl.B)
    O = torch.empty(K.shape, dtype=out_t, device="cuda")
    stream = torch.cuda.current_stream()
    M = float(wl.N)

    def call(Q, K, V, O):
        binding.aaren_linattn_forward(Q, K, V, O, M, stream=stream)

    for _ in range(warmup):
        call(Q, K, V, O)
    if binding.aaren_check() != binding.AAREN_OK:
        raise SystemExit("device status error during warm-up")
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    with ClockSampler(local) as clocks:
        time.sleep(0.3)
        clocks.begin = time.time()
        t_start = torch.cuda.Event(enable_timing=True)
        t_end = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(SPIN_CYCLES)   # the host issues the first launches meanwhile
        t_start.record(stream)
        for i in range(args.steps):
            starts[i].record(stream)
            call(Q, K, V, O)
            ends[i].record(stream)
        t_end.record(stream)
        torch.cuda.synchronize()
        clocks.end = time.time()
    if dist is not None:
        dist.barrier()
    status = binding.aaren_check()
    if status != binding.AAREN_OK:
        raise SystemExit(f"device status error in the timed region: {binding.status_string(status)}")
    launch_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    mean_launch_ms = statistics.mean(launch_ms)
    launch_spread = {"launch_ms_median": statistics.median(launch_ms), "launch_ms_min": min(launch_ms)}
    step_ms = max_over_ranks(t_start.elapsed_time(t_end) / args.steps, dist, "cuda")
    tokens = wl.heads * wl.N
    elems = tokens * wl.d
    out_b = 2 if out == "bf16" else 4
    alg_bytes = elems * (3 * 2 + out_b)

    # end to end with pinned host buffers: Q, K, V in and O out inside the timed region
    hQ, hK, hV = (torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (Q, K, V))
    hO = torch.empty(O.shape, dtype=out_t, pin_memory=True)
    hQ.copy_(Q); hK.copy_(K); hV.copy_(V)
    e2e_steps = max(1, min(args.steps, 3))
    pieces = e2e_pieces(wl)
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    ev_in = [torch.cuda.Event() for _ in pieces]
    ev_done = [torch.cuda.Event() for _ in pieces]
    flat = lambda t: t.view(wl.heads, *t.shape[2:])
    hf = [flat(t) for t in (hQ, hK, hV)]
    df = [flat(t) for t in (Q, K, V)]
    hOf, dOf = flat(hO), flat(O)

    def e2e_step():
        """Heads in pieces, the copies in and out of consecutive pieces
        overlapping the calls (three streams), as for the scan."""
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for i, (h0, h1) in enumerate(pieces):
            with torch.cuda.stream(s_in):
                for d_, h_ in zip(df, hf):
                    d_[h0:h1].copy_(h_[h0:h1], non_blocking=True)
                ev_in[i].record(s_in)
            stream.wait_event(ev_in[i])
            sub = lambda t: t[h0:h1].view(1, h1 - h0, *t.shape[1:])
            call(*(sub(t) for t in df), sub(dOf))
            ev_done[i].record(stream)
            s_out.wait_event(ev_done[i])
            with torch.cuda.stream(s_out):
                hOf[h0:h1].copy_(dOf[h0:h1], non_blocking=True)
        stream.wait_stream(s_out)

    e2e_step()
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True); b = torch.cuda.Event(enable_timing=True)
    a.record(stream)
    for _ in range(e2e_steps):
        e2e_step()
    b.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(a.elapsed_time(b) / e2e_steps, dist, "cuda")
    if binding.aaren_check() != binding.AAREN_OK:
        raise SystemExit("device status error in the end-to-end leg")
    if rank != 0:
        if dist is not None:
            dist.destroy_process_group()
        return 0
    peak, peak_src = measured_peak()
    achieved = alg_bytes / (mean_launch_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC + " (causal cos-re-weighted linear attention)",
        "value": whole_job_rate(tokens, world, step_ms), "unit": "head-tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": f"linattn: B={wl.B} H={wl.H} N={wl.N} d={wl.d}, bf16 in, {out} out, "
                               f"Q, K, V ~ N(0,1) (a query per token), M = N, seed {wl.seed}",
                   "op": "linattn", "global_batch": world * wl.B,
                   "parallelism": f"independent sequences, {world} rank(s), no collective",
                   "l2": f"no flush: Q, K, V per step ({3 * wl.heads * wl.N * wl.d * 2 / 1e9:.2f} GB) larger than "
                         f"the 126 MB L2"},
        "gpu_launches": args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "traffic": profiled_traffic(wl, out, "linattn_bf16_traffic.json", "k_linattn"),
                     "algorithmic_bytes_per_launch": alg_bytes, "launch_ms": mean_launch_ms,
                     **launch_spread, "peak_source": peak_src, "kernel": "k_linattn"},
        "cpu_baseline": cpu,
        "e2e": {"value": whole_job_rate(tokens, world, e2e_ms), "unit": "head-tokens/s",
                "h2d_bytes_per_step": 3 * elems * 2, "d2h_bytes_per_step": elems * out_b,
                "ms_per_step": e2e_ms, "steps": e2e_steps,
                "path": "pinned host Q,K,V -> device, aaren_linattn_forward, device O -> pinned host",
                "pieces": f"{len(pieces)} piece(s) of heads; the host->device copy, the call and the "
                          f"device->host copy of consecutive pieces overlap on three streams"},
        "clocks": clocks.summary(),
    }
    print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference" and args.op == "linattn":
        rank, _, _ = dist_env()
        if rank != 0:
            return 0
        from attention_prefix_scan_02_b300 import inputs
        wl = inputs.WORKLOADS["linattn"]
        timer = la_oracle_timer(wl, LA_CPU_TOKENS, LA_CPU_HEADS, host_cores())
        timer.warm(CPU_SAMPLE_MIN_S)
        rates = []
        for i in range(args.warmup + args.steps):
            r, dt, passes = timer.run(CPU_SAMPLE_MIN_S if i >= args.warmup else 0.0)
            if i >= args.warmup:
                rates.append((r, dt))
        n, nh, used = timer.tokens, len(timer.items), timer.threads
        timer.close()
        value = statistics.mean(r for r, _ in rates)
        print(json.dumps({"impl": "reference", "metric": METRIC + " (causal cos-re-weighted linear attention)",
                          "value": value, "unit": "head-tokens/s", "n_gpus": args.gpus, "steps": args.steps,
                          "warmup": args.warmup, "ms_per_step": 1e3 * statistics.mean(dt for _, dt in rates),
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
                          "data": "synthetic", "config": {"workload": "linattn", "op": "linattn"},
                          "cpu_baseline": {"value": value, "unit": "head-tokens/s", "cores": used,
                                           "kind": "oracle",
                                           "sample": f"each step: passes over the first {n} tokens of {nh} "
                                                     f"heads for at least {CPU_SAMPLE_MIN_S:.0f} s on "
                                                     f"{used} threads"},
                          "e2e": {"value": value, "unit": "head-tokens/s", "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return 0
    if args.op == "linattn":
        return run_linattn(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.op == "step":
        return run_step(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
