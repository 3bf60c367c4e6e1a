"""The multi-rank forms with the library's own kernels: two processes share the
GPU, each runs its part through the C ABI, and they exchange their results
over gloo on CPU copies (no kernel of one process ever waits on the other).

* Vocabulary-parallel ([P2] gemini review: one reduction after the loop;
  greptile / cursor reviews: each shard returns its d_logits @ W_shard): rank
  r holds W[a_r:b_r], computes its per-row (m, s, u, t) partials with
  lmhead_fwd_shard, the partials are all-gathered, every rank merges them with
  lmhead_merge_shards, runs lmhead_bwd_shard on its shard and the hidden-
  gradient partials are summed by an all-reduce.  Against the float64 oracle
  of the whole vocabulary.
* Data-parallel: rank r scores its half of the batch with lmhead_fwd /
  lmhead_bwd and allreduce_weight_grad sums the weight gradients.  Against the
  oracle of the whole batch, and against one process scoring the whole batch.
"""

import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from oracle import lmhead_oracle as O
from sft_keep_mask_gb300 import synth
from tests._util import assert_frob_close, assert_rows_close, to64

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
W_TINY = dict(seed=71, N=700, H=192, V=5000)
BOUNDS = [0, 2201, 5000]   # uneven, unaligned vocabulary shards


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import sys
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    torch.cuda.set_device(0)
    return dist


def _vocab_rank(rank, world, port, out):
    dist = _init(rank, world, port)
    from sft_keep_mask_gb300 import lmhead as L
    from sft_keep_mask_gb300 import synth as S
    from sft_keep_mask_gb300.api import LMHeadScorer
    w = S.workload("tiny", **W_TINY)
    inp = S.make_inputs(w, device="cuda")
    N, H, V = w.N, w.H, w.V
    a, b = BOUNDS[rank], BOUNDS[rank + 1]
    Wr = inp["weight"][a:b].contiguous()
    keep = inp["keep"]
    sc = LMHeadScorer(N, H, b - a, chunk_rows=256)
    part = torch.empty(N, 4, device="cuda")
    L.lmhead_fwd_shard(inp["hidden"], Wr, a, V, inp["targets"], keep, True, part, sc.workspace,
                       256)
    mine = part.cpu()
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine)
    parts = torch.stack(gathered).cuda()
    lp = torch.empty(N, device="cuda")
    ent = torch.empty(N, device="cuda")
    lse = torch.empty(N, device="cuda")
    L.lmhead_merge_shards(parts, keep, True, lp, ent, lse)
    dh_r = torch.empty(N, H, dtype=torch.bfloat16, device="cuda")
    dW_r = torch.empty(b - a, H, device="cuda")
    L.lmhead_bwd_shard(inp["hidden"], Wr, a, V, inp["targets"], keep, lse, ent,
                       inp["grad_logprob"], inp["grad_entropy"], dh_r, dW_r, False, sc.workspace,
                       256)
    torch.cuda.synchronize()
    dh = dh_r.float().cpu()
    dist.all_reduce(dh)
    out[rank] = dict(status=sc.status(), lp=lp.cpu().numpy(), ent=ent.cpu().numpy(),
                     lse=lse.cpu().numpy(), dh=dh.numpy(), dW=dW_r.cpu().numpy())
    dist.destroy_process_group()


def _data_rank(rank, world, port, out):
    dist = _init(rank, world, port)
    from sft_keep_mask_gb300 import synth as S
    from sft_keep_mask_gb300.api import LMHeadScorer, allreduce_weight_grad
    w = S.workload("tiny", **W_TINY)
    inp = S.make_inputs(w, device="cuda")
    half = w.N // 2
    rows = slice(0, half) if rank == 0 else slice(half, w.N)
    args = [inp[k][rows].contiguous() for k in ("hidden", "targets", "keep", "grad_logprob",
                                                 "grad_entropy")]
    hidden, targets, keep, g_lp, g_ent = args
    sc = LMHeadScorer(hidden.shape[0], w.H, w.V, chunk_rows=256)
    lp, ent, lse = sc.forward(hidden, inp["weight"], targets, keep)
    dh, dW = sc.backward(hidden, inp["weight"], targets, keep, lse, ent, g_lp, g_ent)
    torch.cuda.synchronize()
    dW_cpu = dW.cpu()
    allreduce_weight_grad(dW_cpu)
    out[rank] = dict(status=sc.status(), lp=lp.cpu().numpy(), dh=dh.float().cpu().numpy(),
                     dW=dW_cpu.numpy())
    dist.destroy_process_group()


def _run(target):
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=target, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(600)
            assert p.exitcode == 0
        return [dict(out[r]) for r in range(world)]


def _oracle():
    w = synth.workload("tiny", **W_TINY)
    inp = synth.make_inputs(w, device="cuda")
    h, W = to64(inp["hidden"]), to64(inp["weight"])
    y = inp["targets"].cpu().numpy()
    k = inp["keep"].cpu().numpy()
    fwd = O.forward(h, W, y, k)
    bwd = O.backward(h, W, y, k, inp["grad_logprob"].cpu().double().numpy(),
                     inp["grad_entropy"].cpu().double().numpy())
    return w, inp, fwd, bwd


def test_vocabulary_parallel_ranks_with_the_library():
    res = _run(_vocab_rank)
    w, _, (olp, oent, olse), (odh, odW) = _oracle()
    for r, d in enumerate(res):
        assert d["status"] == 0
        assert_rows_close(d["lp"].astype(np.float64), olp, f"logprob (rank {r})")
        assert_rows_close(d["ent"].astype(np.float64), oent, f"entropy (rank {r})")
        assert_rows_close(d["lse"].astype(np.float64), olse, f"lse (rank {r})")
        assert_frob_close(d["dh"].astype(np.float64), odh, f"dhidden (rank {r})")
    dW = np.concatenate([res[0]["dW"], res[1]["dW"]]).astype(np.float64)
    assert_frob_close(dW, odW, "dW (shards side by side)")


def test_data_parallel_ranks_with_the_library():
    from sft_keep_mask_gb300.api import LMHeadScorer
    res = _run(_data_rank)
    w, inp, (olp, _, _), (odh, odW) = _oracle()
    assert all(d["status"] == 0 for d in res)
    assert_rows_close(np.concatenate([res[0]["lp"], res[1]["lp"]]).astype(np.float64), olp,
                      "logprob (ranks' halves)")
    assert_frob_close(np.concatenate([res[0]["dh"], res[1]["dh"]]).astype(np.float64), odh,
                      "dhidden (ranks' halves)")
    for r in range(2):
        assert_frob_close(res[r]["dW"].astype(np.float64), odW, f"all-reduced dW (rank {r})")
    # one process scoring the whole batch: the same sum up to fp32 rounding
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=256)
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"])
    _, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"], lse, ent,
                        inp["grad_logprob"], inp["grad_entropy"])
    torch.cuda.synchronize()
    whole = dW.cpu().double().numpy()
    err = np.linalg.norm(res[0]["dW"] - whole) / np.linalg.norm(whole)
    assert err < 1e-5 and np.array_equal(res[0]["dW"], res[1]["dW"])
