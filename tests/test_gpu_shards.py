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


def _shards_case(w, bounds, chunk=256, grad_entropy=True, keep=None):
    """Scores w's vocabulary in the shards given by `bounds`, merges and sums
    them as a caller would, and checks everything against the oracle."""
    inp = synth.make_inputs(w, device=DEV)
    keep = inp["keep"] if keep is None else keep
    g_ent = inp["grad_entropy"] if grad_entropy else None
    N, H, V = w.N, w.H, w.V
    shards = list(zip(bounds[:-1], bounds[1:]))
    parts = torch.empty(len(shards), N, 4, device=DEV)
    scorers = []
    for r, (a, b) in enumerate(shards):
        sc = LMHeadScorer(N, H, b - a, chunk_rows=chunk)
        scorers.append(sc)
        Wr = inp["weight"][a:b].contiguous()
        L.lmhead_fwd_shard(inp["hidden"], Wr, a, V, inp["targets"], keep, True, parts[r],
                           sc.workspace, chunk)
    lp = torch.empty(N, device=DEV)
    ent = torch.empty(N, device=DEV)
    lse = torch.empty(N, device=DEV)
    L.lmhead_merge_shards(parts, keep, True, lp, ent, lse)
    dh = torch.zeros(N, H, dtype=torch.float32, device=DEV)
    dW = torch.empty(V, H, device=DEV)
    for r, (a, b) in enumerate(shards):
        sc = LMHeadScorer(N, H, b - a, chunk_rows=chunk)
        scorers.append(sc)
        Wr = inp["weight"][a:b].contiguous()
        dh_r = torch.empty(N, H, dtype=torch.bfloat16, device=DEV)
        L.lmhead_bwd_shard(inp["hidden"], Wr, a, V, inp["targets"], keep, lse, ent,
                           inp["grad_logprob"], g_ent, dh_r, dW[a:b], False,
                           sc.workspace, chunk)
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
                          None if g_ent is None else g_ent.cpu().double().numpy())
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


@pytest.mark.parametrize("bounds", [[0, 2600, 5000], [0, 1000, 1001 + 999, 3333, 5000]])
def test_shards_merge_to_the_whole_vocabulary(bounds):
    _shards_case(synth.workload("tiny", seed=70, N=700, H=192, V=5000), bounds)


def test_random_shard_partitions():
    # seeded problems: 1 to 6 shards cut at random (unaligned) vocabulary
    # rows, vocabularies down to one token, chunk sizes, metric-only or
    # differentiable entropy, sparse and dense keep masks
    rng = np.random.default_rng(75)
    for case in range(10):
        N = int(rng.integers(1, 1500))
        H = int(rng.choice([8, 64, 136, 520]))
        V = int(rng.integers(1, 9000))
        nshard = int(rng.integers(1, min(6, V) + 1))
        cuts = sorted(rng.choice(np.arange(1, V), size=nshard - 1, replace=False)) if V > 1 else []
        bounds = [0, *[int(c) for c in cuts], V]
        w = synth.workload("tiny", seed=760 + case, N=N, H=H, V=V)
        keep = torch.from_numpy((rng.random(N) < float(rng.choice([0.05, 0.5, 1.0])))
                                .astype(np.uint8)).to(DEV)
        _shards_case(w, bounds, chunk=int(rng.choice([256, 512, 1024])),
                     grad_entropy=bool(rng.integers(0, 2)), keep=keep)


def test_shard_arguments_are_checked():
    w = synth.workload("tiny", seed=71, N=64, H=64, V=1000)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(64, 64, 500)
    parts = torch.empty(64, 4, device=DEV)
    with pytest.raises(L.LmheadError):
        # a 400-row shard starting at 700 runs past V_total = 1000
        L.lmhead_fwd_shard(inp["hidden"], inp["weight"][600:].contiguous(), 700, 1000,
                           inp["targets"], None, True, parts, sc.workspace)
