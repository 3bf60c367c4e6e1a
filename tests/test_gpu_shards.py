"""Vocabulary-parallel entry points on one GPU: the vocabulary is split into
uneven shards, each scored by lmhead_fwd_shard / lmhead_bwd_shard, the
partials merged by lmhead_merge_shards and the hidden-gradient partials summed
as a caller would; the result must match the float64 oracle of the whole
vocabulary."""

import numpy as np
import pytest
import torch

from oracle import lmhead_oracle as O
from sft_keep_mask_gb300 import lmhead as L
from sft_keep_mask_gb300 import synth
from sft_keep_mask_gb300.api import LMHeadScorer
from tests._util import assert_frob_close, assert_rows_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.mark.parametrize("bounds", [[0, 2600, 5000], [0, 1000, 1001 + 999, 3333, 5000]])
def test_shards_merge_to_the_whole_vocabulary(bounds):
    w = synth.workload("tiny", seed=70, N=700, H=192, V=5000)
    inp = synth.make_inputs(w, device=DEV)
    keep = inp["keep"]
    N, H, V = w.N, w.H, w.V
    shards = list(zip(bounds[:-1], bounds[1:]))
    parts = torch.empty(len(shards), N, 4, device=DEV)
    scorers = []
    for r, (a, b) in enumerate(shards):
        sc = LMHeadScorer(N, H, b - a, chunk_rows=256)
        scorers.append(sc)
        Wr = inp["weight"][a:b].contiguous()
        L.lmhead_fwd_shard(inp["hidden"], Wr, a, V, inp["targets"], keep, True, parts[r],
                           sc.workspace, 256)
    lp = torch.empty(N, device=DEV)
    ent = torch.empty(N, device=DEV)
    lse = torch.empty(N, device=DEV)
    L.lmhead_merge_shards(parts, keep, True, lp, ent, lse)
    dh = torch.zeros(N, H, dtype=torch.float32, device=DEV)
    dW = torch.empty(V, H, device=DEV)
    for r, (a, b) in enumerate(shards):
        sc = LMHeadScorer(N, H, b - a, chunk_rows=256)
        scorers.append(sc)
        Wr = inp["weight"][a:b].contiguous()
        dh_r = torch.empty(N, H, dtype=torch.bfloat16, device=DEV)
        L.lmhead_bwd_shard(inp["hidden"], Wr, a, V, inp["targets"], keep, lse, ent,
                           inp["grad_logprob"], inp["grad_entropy"], dh_r, dW[a:b], False,
                           sc.workspace, 256)
        dh += dh_r.float()  # the caller's reduction over shards
    torch.cuda.synchronize()
    assert all(sc.status() == 0 for sc in scorers)
    h, W = to64(inp["hidden"]), to64(inp["weight"])
    y = inp["targets"].cpu().numpy()
    k = keep.cpu().numpy()
    olp, oent, olse = O.forward(h, W, y, k)
    assert_rows_close(lp.cpu().double().numpy(), olp, "logprob")
    assert_rows_close(ent.cpu().double().numpy(), oent, "entropy")
    assert_rows_close(lse.cpu().double().numpy(), olse, "lse")
    odh, odW = O.backward(h, W, y, k, inp["grad_logprob"].cpu().double().numpy(),
                          inp["grad_entropy"].cpu().double().numpy())
    assert_frob_close(dh.cpu().double().numpy(), odh, "dhidden (sum of shards)")
    assert_frob_close(dW.cpu().double().numpy(), odW, "dW (concatenated shards)")
    # the shard partials themselves against the oracle's shard partials
    for r, (a, b) in enumerate(shards):
        op = O.shard_partials(h, W[a:b], a, y, k)
        got = parts[r].cpu().double().numpy()
        kept = k == 1
        np.testing.assert_allclose(got[kept, 0], op[kept, 0], atol=1e-4)
        np.testing.assert_allclose(got[kept, 1], op[kept, 1], rtol=1e-4)
        assert (got[~kept, 0] == -np.inf).all() and (got[~kept, 1] == 0).all()


def test_shard_arguments_are_checked():
    w = synth.workload("tiny", seed=71, N=64, H=64, V=1000)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(64, 64, 500)
    parts = torch.empty(64, 4, device=DEV)
    with pytest.raises(L.LmheadError):
        # a 400-row shard starting at 700 runs past V_total = 1000
        L.lmhead_fwd_shard(inp["hidden"], inp["weight"][600:].contiguous(), 700, 1000,
                           inp["targets"], None, True, parts, sc.workspace)
