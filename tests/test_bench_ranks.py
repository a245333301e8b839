"""The multi-rank path of bench.py on the CPU: two gloo ranks, each running
its own replica, agree on the slowest rank's step time, and the whole-job
value counts the work of both ranks over that time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench._max_over_ranks(times[rank], world, "cpu")
        dist.barrier()
        out[rank] = ms
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [(2.0, 3.5), (4.25, 1.0)])
def test_two_ranks_take_the_slowest_step(times):
    world = 2
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_rank, args=(world, _free_port(), times, out), nprocs=world, join=True)
    assert out[0] == out[1] == max(times)


def test_job_value_counts_every_rank():
    flop = 1.3e12  # one rank's work per step
    one = bench._job_value(flop, 2.0, 1)
    assert one == pytest.approx(flop / 2e-3 / 1e12)
    # two replicas in the time of the slower one: twice the work, same time
    assert bench._job_value(flop, 2.0, 2) == pytest.approx(2 * one)
    assert bench._max_over_ranks(1.75, 1, "cpu") == 1.75


def test_reference_arm_runs_on_rank_zero_only():
    """Under torchrun the oracle's timing runs on rank 0 alone; another rank
    exits 0 at once without output."""
    import subprocess
    import sys
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(os.path.dirname(bench.__file__), "bench.py"),
                        "--impl", "reference", "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
