"""The benchmark's N > 1 host logic (replicas, max-over-ranks time, summed
work) on two gloo ranks on the CPU."""
from __future__ import annotations

import os
import socket

import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, q):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import torch.distributed as dist

    import bench
    r, local, w = bench.dist_init()
    assert (r, local, w) == (rank, rank, world)
    bench.barrier(w)
    t = bench.max_over_ranks(1.0 + rank, w)      # rank times 1.0 and 2.0 -> 2.0
    work = bench.sum_over_ranks(10.0 * (rank + 1), w)  # 10 + 20 -> 30
    q.put((rank, t, work))
    dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    assert res == [(0, 2.0, 30.0), (1, 2.0, 30.0)]
