"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2): the
job's time is the slowest rank's, its work the sum over ranks, and every rank
agrees on both.  Rows are independent, so ranks share no data; this is the
only cross-rank exchange there is."""
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
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t, u = bench.aggregate_over_ranks(10.0 * (rank + 1), 1000.0 + rank, world)
        # a rank that finishes early still waits for the others' numbers
        dist.barrier()
        q.put((rank, t, u))
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    for rank, t, u in got:
        assert t == 20.0          # max over ranks
        assert u == 2001.0        # sum over ranks


def test_single_process_passthrough():
    import bench
    assert bench.aggregate_over_ranks(3.5, 7.0, 1) == (3.5, 7.0)
