"""The N > 1 path of bench.py on CPU ranks (gloo, world size 2).

Each rank scores its own batch with no collective on the data path; the
only exchange is the reduction of the timing (max over ranks) and of the
kept-row count (sum over ranks) that bench.py reports.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [120.5, 98.25][rank]
    kept = [36258, 35001][rank]
    out[rank] = bench.reduce_over_ranks(ms, kept, world, "cpu")
    dist.destroy_process_group()


def test_reduce_over_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(world):
            assert out[r] == (120.5, 36258.0 + 35001.0)


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.reduce_over_ranks(10.0, 7, 1, "cpu") == (10.0, 7.0)
