"""The multi-rank path of bench.py on CPU: two gloo ranks (one process
each, rendezvous on 127.0.0.1).  Heads are independent, so ranks run
their own copies of the workload with no collective on the data path; the
only communication is the barrier and the maximum of the step times, and
the reported rate counts every rank's head-tokens (weak scaling).  The
oracle arm runs on rank 0 alone."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, step_ms, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        worst = bench.max_over_ranks(step_ms[rank], dist, "cpu")
        rate = bench.whole_job_rate(1000, world, worst)
        out[rank] = (worst, rate)
    finally:
        dist.destroy_process_group()


def test_two_ranks_take_the_slowest_step_and_count_all_units():
    world, port = 2, free_port()
    step_ms = [2.0, 3.0]
    manager = mp.get_context("spawn").Manager()
    out = manager.dict()
    mp.start_processes(_rank_main, args=(world, port, step_ms, out), nprocs=world,
                       start_method="spawn", join=True)
    for r in range(world):
        worst, rate = out[r]
        assert worst == 3.0
        assert rate == pytest.approx(2 * 1000 / 3e-3)


def test_one_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(1.5, None, "cpu") == 1.5
    assert bench.whole_job_rate(10, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_prints_on_rank_0_only():
    """Under torchrun the other ranks of the oracle arm exit 0 without work
    (checked here for rank 1 of 2 through the environment torchrun sets)."""
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "1", "--warmup", "0"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0
    assert res.stdout.strip() == ""


def test_reference_arm_line_on_rank_0():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    res = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--workload", "tiny", "--steps", "2", "--warmup", "1"],
                         env=env, capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    line = json.loads(res.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle"
    assert line["e2e"]["h2d_bytes_per_step"] == 0
