"""The benchmark's multi-rank arithmetic on CPU: two gloo ranks (one process
each, 127.0.0.1) time different steps; every rank must see the slowest rank's
time, and the whole-job figure counts both ranks' bytes over that time."""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = [2.0, 3.5][rank]                       # rank 1 is the slow one
        t = bench.max_over_ranks(ms, dist, "cpu")
        out[rank] = (t, bench.job_gbs(277381376, world, t))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    world = 2
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_rank, args=(world, _free_port(), out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 3.5
    assert res[0][1] == pytest.approx(2 * 277381376 / 3.5e-3 / 1e9)


def test_single_process_is_identity():
    assert bench.max_over_ranks(1.25, None, "cpu") == 1.25
    assert bench.job_gbs(1e9, 1, 1000.0) == pytest.approx(1.0)
