"""bench.py's multi-GPU arithmetic on the host: two gloo ranks on the CPU.

Every rank runs the same workload on its own GPU with no exchange between
ranks (weak scaling, replicas only), so the job's time per step is the
slowest rank's and its rate is the rows of all ranks over that time.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        ms = bench.max_over_ranks(times[rank], world)
        out[rank] = ms
    finally:
        dist.destroy_process_group()


@pytest.mark.timeout(120)
def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    times = [3.0, 5.5]
    out = mp.get_context("spawn").Manager().dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), times, out), nprocs=world,
                       start_method="spawn", join=True)
    assert out[0] == out[1] == max(times)


def test_whole_job_rate_counts_every_rank():
    # 64 rows per rank, 2 ms per step, 4 ranks: 4 * 64 / 2e-3 rows/s.
    assert bench.whole_job_rate(64, 2.0, 4) == pytest.approx(128000.0)
    assert bench.whole_job_rate(64, 2.0, 1) == pytest.approx(32000.0)


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(7.25, 1) == 7.25
