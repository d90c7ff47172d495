"""The multi-GPU path on CPU: two gloo ranks combine their timings and unit
counts the way bench.py does under torchrun (max of times, sum of units), and
each rank draws its own requests.  The data path itself has no collective."""
from __future__ import annotations

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench

    t_dev = [0.5, 0.8][rank]
    t_e2e = [0.9, 0.7][rank]
    out = bench.combine_ranks(t_dev, t_e2e, 100 + rank, 10 * (rank + 1), 1000.0 * (rank + 1),
                              True, torch.device("cpu"))
    seeds = bench.rank_seed(303, rank)
    q.put((rank, out, seeds))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_combination():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict()
    for _ in range(2):
        rank, out, seed = q.get(timeout=120)
        res[rank] = (out, seed)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in range(2):
        t_dev, t_e2e, misses, e2e, alg = res[r][0]
        assert t_dev == pytest.approx(0.8) and t_e2e == pytest.approx(0.9)
        assert misses == 201 and e2e == 30 and alg == 3000.0
    assert res[0][1] != res[1][1]
