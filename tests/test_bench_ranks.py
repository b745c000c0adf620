"""bench.py's multi-rank arithmetic on two gloo ranks (CPU): timing is the
maximum over ranks and the reported value is the whole job's work over it."""
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


def _rank_main(rank, world, port):
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", init_method="tcp://127.0.0.1:%d" % port, rank=rank, world_size=world)
    try:
        elapsed = [40.0, 55.5][rank]                       # this rank's timed region, ms
        slowest = bench.max_over_ranks(elapsed, dist, "cpu")
        assert slowest == 55.5
        value = bench.job_throughput(2.0e12, 10, world, slowest)
        assert abs(value - 2.0e12 * 10 * world / 0.0555 / 1e12) < 1e-9
        env_ws, env_rank, _ = bench.dist_env()
        assert (env_ws, env_rank) == (1, 0) or env_ws == world
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_max():
    port = _free_port()
    mp.spawn(_rank_main, args=(2, port), nprocs=2, join=True)


def test_single_process_defaults():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(12.5) == 12.5
    assert bench.job_throughput(1e12, 5, 1, 1000.0) == pytest.approx(5.0)
