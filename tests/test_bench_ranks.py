"""bench.py's replica path with two ranks on CPU (gloo): the slowest rank's
time and the whole-job rate every rank computes from it; the reference arm's
other ranks exit without work."""
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.rank_barrier(world)
        ms = [12.5, 20.0][rank]  # this rank's timed region
        slowest = bench.max_over_ranks(ms, world, "cpu")
        out[rank] = (slowest, bench.whole_job_rate(112.0, world, slowest))
        bench.rank_barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_slowest_time_and_the_whole_job_rate():
    world = 2
    out = mp.Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), out), nprocs=world, start_method="spawn")
    assert out[0] == out[1]
    slowest, rate = out[0]
    assert slowest == 20.0
    assert rate == pytest.approx(2 * 112.0 / 0.020)  # units of both ranks over the slowest time


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.rank_barrier(1)
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.whole_job_rate(112.0, 1, 250.0) == pytest.approx(448.0)


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--steps", "3", "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
