"""The multi-rank plumbing of bench.py (replicas: timing reduction only),
run as two gloo ranks on the CPU."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        t = bench.reduce_max(10.0 + rank, "cpu")         # slowest rank decides the time
        u = bench.reduce_sum(100.0 * (rank + 1), "cpu")  # units processed by all ranks
        bench.barrier()
        q.put((rank, ws, r, t, u))
    finally:
        dist.destroy_process_group()


def test_two_rank_reductions():
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
    for rank, ws, r, t, u in res:
        assert ws == 2 and r == rank
        assert t == 11.0          # max over ranks
        assert u == 300.0         # sum over ranks


def test_single_process_reductions_are_identity():
    import bench
    assert bench.reduce_max(3.5, "cpu") == 3.5
    assert bench.reduce_sum(2.0, "cpu") == 2.0
