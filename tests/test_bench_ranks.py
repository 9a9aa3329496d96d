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


def test_bench_starts_its_own_replica_ranks():
    """`bench.py --gpus 2` run without torchrun starts two ranks itself (one
    process each, gloo here); both join, and rank 0's line reports the job."""
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items()
           if k not in ("RANK", "WORLD_SIZE", "LOCAL_RANK", "MASTER_ADDR", "MASTER_PORT")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--launcher-selftest"], env=env, capture_output=True, text=True,
                       timeout=180)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [json.loads(x) for x in r.stdout.splitlines() if x.startswith("{")]
    assert len(lines) == 1                          # rank 0 alone prints
    line = lines[0]
    assert line["n_gpus"] == 2 and line["ranks_joined"] == 2
    assert line["ms_per_step"] == 2.0               # the slower rank's time
    assert line["job_gbs_for_1GB_per_rank"] == pytest.approx(2 * 1e9 / 2e-3 / 1e9)


def test_bench_refuses_a_rank_count_mismatch():
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2",
                        "--launcher-selftest"], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode != 0 and "WORLD_SIZE=1" in r.stderr
