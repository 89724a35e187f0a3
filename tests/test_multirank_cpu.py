"""The N > 1 path of bench.py on CPU: world-size-2 gloo ranks, each timing its
own replica.  The job's time is the slowest rank's (max over ranks) and its
throughput the total work over that time; the reference arm runs on rank 0
only."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, _ = bench.dist_env()
    dist = bench.dist_init(ws, "gloo")
    bench.barrier(dist)
    slowest = bench.max_over_ranks(dist, times[r])
    out[r] = (slowest, bench.job_throughput(ws, 1e12, 10, slowest))
    dist.destroy_process_group()


def test_max_over_ranks_and_job_throughput_gloo():
    world = 2
    times = [40.0, 55.0]  # ms for 10 steps on each rank
    mgr = mp.get_context("spawn").Manager()  # no fork of this (threaded) process
    out = mgr.dict()
    mp.spawn(_rank_main, args=(world, _free_port(), times, out), nprocs=world, join=True)
    for r in range(world):
        slowest, value = out[r]
        assert slowest == 55.0
        # 2 ranks x 10 steps x 1e12 FLOP in 55 ms
        assert value == pytest.approx(2 * 10 * 1e12 / 0.055 / 1e12)


def test_reference_arm_prints_on_rank_zero_only(tmp_path):
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
