"""The N-rank host logic of bench.py, run as two gloo ranks on the CPU.

bench.py runs one process per GPU as independent replicas of the same
workload (the path shards without any exchange); only the timing uses a
collective: each rank's time is replaced by the slowest rank's, and the
job's throughput is the per-rank rate at that time times the rank count.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.barrier(world)
        slowest = bench.max_over_ranks(times[rank], world, device="cpu")
        bench.barrier(world)
        out[rank] = (slowest, bench.job_rate(1.0 / slowest, world))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(0.010, 0.013), (0.020, 0.005)])
def test_two_ranks_take_the_slowest_time_and_sum_rates(times):
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.start_processes(_worker, args=(world, _free_port(), times, out), nprocs=world, start_method="spawn")
        res = dict(out)
    slowest = max(times)
    for r in range(world):
        got_slowest, rate = res[r]
        assert got_slowest == pytest.approx(slowest)
        assert rate == pytest.approx(world / slowest)


def test_single_rank_is_unchanged():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.5, 1) == 0.5
    assert bench.job_rate(3.0, 1) == 3.0


def test_reference_arm_under_torchrun_prints_once():
    """Launched as the driver launches it for N > 1, the reference arm runs
    on rank 0 alone: one JSON line, every rank exits 0."""
    import json
    import subprocess
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "1", "--cpu-seconds", "1"]
    r = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip().startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
