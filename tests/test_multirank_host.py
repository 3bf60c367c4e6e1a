"""The N > 1 path of bench.py on CPU ranks (gloo, world size 2).

Each rank scores its own batch; the data path's one exchange is the
all-reduce of the weight gradient after the backward (the library's
allreduce_weight_grad, run here on CPU tensors with the oracle's per-rank
gradients), and bench.py reduces the timing (max over ranks) and the
kept-row count (sum over ranks).  How bench.py treats --gpus is checked
without starting ranks, and the reference arm (CPU only) runs under two
launcher ranks.
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


def _dp_rank(rank, world, port, out):
    # data-parallel backward on CPU ranks: each rank takes its half of the
    # batch, computes its weight gradient (the oracle stands in for the GPU
    # backward), and allreduce_weight_grad sums them: the result must be the
    # whole batch's weight gradient on every rank
    import numpy as np
    import torch
    import torch.distributed as dist
    from oracle import lmhead_oracle as O
    from sft_keep_mask_gb300.api import allreduce_weight_grad
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    rng = np.random.default_rng(81)
    N, H, V = 60, 16, 70
    h = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H)) / 4.0
    y = rng.integers(0, V, N)
    keep = (rng.random(N) < 0.6).astype(np.uint8)
    g_lp = rng.standard_normal(N)
    g_ent = 0.1 * rng.standard_normal(N)
    rows = slice(0, 27) if rank == 0 else slice(27, N)
    _, dW_mine = O.backward(h[rows], W, y[rows], keep[rows], g_lp[rows], g_ent[rows])
    dW = torch.from_numpy(dW_mine.copy())
    allreduce_weight_grad(dW)
    _, dW_all = O.backward(h, W, y, keep, g_lp, g_ent)
    out[rank] = (float(np.abs(dW.numpy() - dW_all).max()), float(np.abs(dW_all).max()),
                 float(np.abs(dW_mine - dW_all).max()))
    dist.destroy_process_group()


def test_data_parallel_weight_gradient_on_two_gloo_ranks():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_dp_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        for r in range(world):
            err, scale, own = out[r]
            assert err < 1e-12 * max(scale, 1.0)
            assert own > 1e-3 * scale  # one rank's half alone is not the answer


def test_allreduce_weight_grad_without_a_process_group_is_the_identity():
    import torch
    from sft_keep_mask_gb300.api import allreduce_weight_grad
    g = torch.arange(6.0).reshape(2, 3)
    assert torch.equal(allreduce_weight_grad(g.clone()), g)


def test_gpus_flag_is_honoured():
    import bench
    assert bench.launch_plan(1, {}) == "run"
    assert bench.launch_plan(4, {}) == "spawn"           # no launcher: start 4 ranks
    assert bench.launch_plan(2, {"WORLD_SIZE": "2"}) == "run"
    assert bench.launch_plan(1, {"WORLD_SIZE": "1"}) == "run"
    assert "8" in bench.launch_plan(8, {"WORLD_SIZE": "2"})  # never report n_gpus != N
    assert bench.launch_plan(0, {}) != "run"


def test_data_parallel_ranks_share_the_weight_and_not_the_batch():
    # bench.py's ranks draw their batches from per-rank seeds and the weight
    # from the workload's seed, as data-parallel replicas of one model
    from sft_keep_mask_gb300 import synth
    base = synth.workload("tiny", N=64, H=16, V=50)
    r0 = synth.make_inputs(synth.workload("tiny", N=64, H=16, V=50, seed=base.seed), "cpu",
                           weight_seed=base.seed)
    r1 = synth.make_inputs(synth.workload("tiny", N=64, H=16, V=50, seed=base.seed + 100),
                           "cpu", weight_seed=base.seed)
    import torch
    assert torch.equal(r0["weight"], r1["weight"])
    assert not torch.equal(r0["hidden"], r1["hidden"])
    # and each draw is reproducible
    again = synth.make_inputs(synth.workload("tiny", N=64, H=16, V=50, seed=base.seed + 100),
                              "cpu", weight_seed=base.seed)
    assert torch.equal(r1["hidden"], again["hidden"]) and torch.equal(r1["weight"],
                                                                      again["weight"])


def test_reference_arm_under_two_launcher_ranks_prints_one_line():
    # launched as the driver launches N = 2 (torch.distributed.run, 127.0.0.1):
    # rank 0 alone times the oracle and prints the line; the other rank exits 0
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}",
           os.path.join(root, "bench.py"), "--impl", "reference", "--gpus", "2",
           "--workload", "tiny", "--steps", "1", "--warmup", "1"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    r = subprocess.run(cmd, capture_output=True, text=True, cwd=root, timeout=600, env=env)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
