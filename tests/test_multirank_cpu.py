"""The N > 1 host path of bench.py on CPU: two gloo ranks (127.0.0.1).

Under torchrun every rank runs its own replica of the workload (weak
scaling, no collective on the data path); the only cross-rank steps are the
barrier around the timed region and the maximum of the per-rank times, and
the reported value is every rank's work over that slowest time."""

import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench._barrier(world)
        slowest = bench._max_over_ranks(times[rank], world)
        bench._barrier(world)
        q.put((rank, slowest, bench._aggregate(1.0e12, world, slowest)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time_and_sum_the_work():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    times = [4.0, 5.0]   # ms per step of rank 0 and rank 1
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        got = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in procs)
    # both ranks see the slowest rank's time; the value counts both ranks' work
    assert [g[0] for g in got] == [0, 1]
    assert all(g[1] == 5.0 for g in got)
    assert all(g[2] == pytest.approx(2 * 1.0e12 / 5.0e-3 / 1e12) for g in got)


def test_single_rank_needs_no_process_group():
    assert bench._max_over_ranks(3.25, 1) == 3.25
    assert bench._aggregate(2.0e12, 1, 4.0) == pytest.approx(500.0)
