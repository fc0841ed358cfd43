"""Host logic of the multi-GPU bench on CPU ranks (gloo, world size 2):
every rank runs its own replica, the job time is the maximum over ranks and
throughput counts all ranks' tokens (weak scaling, no data-path collective)."""
from __future__ import annotations

import os
import socket
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, local = bench.dist_env()
        times = bench.max_over_ranks([10.0 * (rank + 1), 5.0 - rank])
        tput = bench.job_tokens_per_s(64, 100, w, times[0])
        q.put((r, w, local, times, tput))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_job_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, (r, w, local, times, tput) in enumerate(res):
        assert (r, w, local) == (rank, 2, rank)
        assert times == [20.0, 5.0]  # the slowest rank's time, element-wise
        assert abs(tput - 64 * 100 * 2 / 0.020) < 1e-6


def test_single_process_is_a_noop():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5]) == [1.5, 2.5]
    assert bench.job_tokens_per_s(1, 1000, 1, 50.0) == 20000.0
