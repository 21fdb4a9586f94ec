"""The benchmark's multi-rank logic on the CPU: two gloo ranks on
127.0.0.1, as torch.distributed.run would start them.  Each rank runs its
own replica of the product; the job's time is the slowest rank's, and the
whole-job throughput counts every rank's flops.  The reference arm prints
from rank 0 only; the other ranks exit 0 without work.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.slowest_rank_ms(times[rank], dist, "cpu")
        value = bench.job_tflops(world, 2.0 * 8192 ** 3, 10, ms)
        out[rank] = (ms, value)
    finally:
        dist.destroy_process_group()


def test_slowest_rank_and_whole_job_throughput():
    world, port = 2, _free_port()
    times = [7.0, 9.5]          # ms for 10 steps on each rank
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
    for rank in range(world):
        ms, value = out[rank]
        assert ms == 9.5, "every rank must see the slowest rank's time"
        assert value == pytest.approx(world * 2.0 * 8192 ** 3 * 10 / 9.5e-3 / 1e12)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.slowest_rank_ms(3.25) == 3.25
    assert bench.job_tflops(1, 2e12, 4, 8.0) == pytest.approx(1000.0)


@pytest.mark.parametrize("rank", [0, 1])
def test_reference_arm_prints_from_rank_zero_only(rank):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1")
    proc = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2", "--steps", "1",
                           "--warmup", "0", "--case", "gemm_512_f16_alpha1.5_beta0.5"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert proc.returncode == 0, proc.stderr
    lines = [l for l in proc.stdout.splitlines() if l.strip()]
    if rank == 0:
        line = json.loads(lines[-1])
        assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    else:
        assert lines == []
