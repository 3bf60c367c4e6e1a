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


def _vocab_rank(rank, world, port, out):
    # vocabulary-parallel scoring on CPU ranks: each rank reduces its shard of
    # W to per-row (m, s, u, t) partials, one all_gather exchanges them, and
    # every rank merges them into the whole vocabulary's log-prob / entropy
    import numpy as np
    import torch
    import torch.distributed as dist
    from oracle import lmhead_oracle as O
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(80)
    N, H, V = 50, 16, 90
    h = rng.standard_normal((N, H))
    W = 2.0 * rng.standard_normal((V, H)) / 4.0
    y = rng.integers(0, V, N)
    keep = (rng.random(N) < 0.7).astype(np.uint8)
    bounds = [0, 37, 90]
    a, b = bounds[rank], bounds[rank + 1]
    mine = torch.from_numpy(O.shard_partials(h, W[a:b], a, y, keep))
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine)
    merged = O.merge_shard_partials(torch.stack(gathered).numpy(), keep)
    full = O.forward(h, W, y, keep)
    out[rank] = max(float(np.abs(g - f).max()) for g, f in zip(merged, full))
    dist.destroy_process_group()


def test_vocab_parallel_exchange_on_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_vocab_rank, args=(r, world, port, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(world):
            assert out[r] < 1e-12
