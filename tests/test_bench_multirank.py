"""The benchmark's multi-rank bookkeeping on CPU (gloo, world size 2): every rank
decodes its own batch with no collective on the data path, and the job's time is
the slowest rank's, reached by an all-reduce(MAX) of the per-rank times."""
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


def _rank_main(rank, world, port, times, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        assert (r, w, local) == (rank, world, rank)
        ms = bench.max_over_ranks(times[rank], w, torch.device("cpu"))
        out[rank] = ms
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank():
    world, port = 2, _free_port()
    times = [0.031, 0.045]
    out = mp.Manager().dict()
    mp.spawn(_rank_main, args=(world, port, times, out), nprocs=world, join=True)
    assert out[0] == pytest.approx(0.045) and out[1] == pytest.approx(0.045)


def test_single_rank_keeps_its_time_and_job_value_counts_all_ranks():
    assert bench.max_over_ranks(0.0321, 1, torch.device("cpu")) == 0.0321
    # 2 ranks x 150,994,944 B in 0.0321 ms per step
    assert bench.job_gbps(150994944, 2, 0.0321) == pytest.approx(2 * 150994944 / 0.0321e-3 / 1e9)
    assert bench.job_gbps(150994944, 1, 0.0321) == pytest.approx(4703.9, rel=1e-4)
