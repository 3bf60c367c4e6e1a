"""Parity of the CUDA path (through the C ABI) with the float64 oracle.

Integer work (keep mask, compaction, Nk) must match bit for bit; logprob,
entropy and lse within 1e-3 absolute; dhidden and dW within 1e-2 relative
Frobenius error (bf16 inputs, fp32 accumulation, bf16 logit gradient).
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import lmhead_oracle as O
from sft_keep_mask_gb300 import lmhead as L
from sft_keep_mask_gb300 import synth
from sft_keep_mask_gb300.api import LMHeadScorer
from tests._util import (assert_frob_close, assert_rows_close, gpu_keep, oracle_keep,
                         seq_offsets, to64)

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _run_both(w, chunk_rows=0, want_entropy=True, grad_entropy=True, keep_override="auto",
              accumulate=False, check_bwd=True, blocksparse=False, active_frac=1.0):
    inp = synth.make_inputs(w, device=DEV, active_frac=active_frac)
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=chunk_rows, blocksparse=blocksparse)
    if isinstance(keep_override, str):
        keep = gpu_keep(sc, inp)
        keep_np = oracle_keep(inp)
        np.testing.assert_array_equal(keep.cpu().numpy(), keep_np)
    elif keep_override is None:
        keep, keep_np = None, None
    else:
        keep_np = keep_override
        keep = torch.from_numpy(keep_np).to(DEV)
    g_ent = inp["grad_entropy"] if grad_entropy else None
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep, want_entropy)
    out = dict(lp=lp, ent=ent, lse=lse)
    dW0 = None
    if check_bwd:
        # with accumulation the gradient is added to a seeded prior one
        if accumulate:
            g = torch.Generator(device=DEV).manual_seed(w.seed)
            dW0 = torch.randn(w.V, w.H, generator=g, device=DEV)
        dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                             inp["grad_logprob"], g_ent,
                             dweight=None if dW0 is None else dW0.clone(), accumulate=accumulate)
        out.update(dh=dh, dW=dW)
    torch.cuda.synchronize()
    assert sc.status() == 0

    h, W = to64(inp["hidden"]), to64(inp["weight"])
    y = inp["targets"].cpu().numpy()
    olp, oent, olse = O.forward(h, W, y, keep_np, want_entropy)
    assert_rows_close(lp.cpu().double().numpy(), olp, "logprob")
    assert_rows_close(lse.cpu().double().numpy(), olse, "lse")
    if want_entropy:
        assert_rows_close(ent.cpu().double().numpy(), oent, "entropy")
    skipped = np.zeros(w.N, bool) if keep_np is None else keep_np == 0
    assert (lp.cpu().numpy()[skipped] == 0).all() and (lse.cpu().numpy()[skipped] == 0).all()
    if check_bwd:
        odh, odW = O.backward(h, W, y, keep_np, inp["grad_logprob"].cpu().double().numpy(),
                              None if g_ent is None else g_ent.cpu().double().numpy())
        if dW0 is not None:
            odW = odW + dW0.cpu().double().numpy()
        assert_frob_close(to64(out["dh"]), odh, "dhidden")
        assert_frob_close(out["dW"].cpu().double().numpy(), odW, "dW")
        assert (out["dh"].cpu()[torch.from_numpy(skipped)] == 0).all()
    return inp, keep, keep_np, out, sc


def test_tiny_forward_backward_with_entropy_gradient():
    _run_both(synth.workload("tiny"))


def test_multi_tile_ragged_multi_chunk():
    # N, H, V not multiples of the tiles; 4 chunks of 256 kept rows; packed
    # sequences build the keep mask on the device
    w = synth.workload("moe30b_rl", N=3000, H=384, V=5000)
    _run_both(w, chunk_rows=256)


def test_metric_only_entropy_and_no_entropy():
    w = synth.workload("tiny", seed=7, N=700, H=192, V=3000)
    _run_both(w, want_entropy=True, grad_entropy=False)
    _run_both(w, want_entropy=False, grad_entropy=False)


def test_keep_none_scores_every_row():
    w = synth.workload("tiny", seed=8, N=300, H=128, V=2100)
    _run_both(w, keep_override=None)


def test_empty_keep_mask():
    w = synth.workload("tiny", seed=9, N=200, H=64, V=1000)
    inp, keep, _, out, sc = _run_both(w, keep_override=np.zeros(200, np.uint8))
    assert not out["lp"].any() and not out["lse"].any() and not out["ent"].any()
    assert not out["dh"].any() and not out["dW"].any()
    # with accumulation the weight gradient is left as it was
    dW = torch.full((w.V, w.H), 3.0, device=DEV)
    sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, out["lse"], out["ent"],
                inp["grad_logprob"], inp["grad_entropy"], dweight=dW, accumulate=True)
    torch.cuda.synchronize()
    assert (dW == 3.0).all()


def test_single_kept_row_and_vocab_tail():
    w = synth.workload("tiny", seed=10, N=64, H=64, V=257)
    keep = np.zeros(64, np.uint8)
    keep[37] = 1
    _run_both(w, keep_override=keep)


def test_gradient_accumulation_and_determinism():
    w = synth.workload("tiny", seed=11, N=640, H=256, V=4100)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=256)
    keep = inp["keep"]
    args = (inp["hidden"], inp["weight"], inp["targets"], keep)
    lp1, ent1, lse1 = sc.forward(*args)
    lp2, ent2, lse2 = sc.forward(*args)
    assert torch.equal(lp1, lp2) and torch.equal(ent1, ent2) and torch.equal(lse1, lse2)
    g = (inp["grad_logprob"], inp["grad_entropy"])
    dh1, dW1 = sc.backward(*args, lse1, ent1, *g)
    dh2, dW2 = sc.backward(*args, lse1, ent1, *g)
    assert torch.equal(dh1, dh2) and torch.equal(dW1, dW2)
    sc.backward(*args, lse1, ent1, *g, dweight=dW2, accumulate=True)
    torch.cuda.synchronize()
    assert torch.allclose(dW2, 2 * dW1, rtol=1e-6, atol=1e-7)


def test_peaked_rows():
    w = synth.workload("tiny", seed=12, N=300, H=256, V=4096, w_scale=16.0)
    inp, _, _, out, _ = _run_both(w)
    lp = out["lp"].cpu().numpy()
    assert (lp <= 1e-5).all()


def test_compaction_and_expand_bit_exact():
    rng = np.random.default_rng(13)
    for n in (1, 255, 4096, 4097, 20000):
        keep_np = (rng.random(n) < 0.37).astype(np.uint8)
        y = torch.from_numpy(rng.integers(0, 50, n)).to(DEV)
        sc = LMHeadScorer(n, 64, 50)
        idx, yc, nk = sc.compact(torch.from_numpy(keep_np).to(DEV), y)
        oidx, onk, oyc = O.compact(keep_np, y.cpu().numpy(), 50)
        assert int(nk.item()) == onk
        np.testing.assert_array_equal(idx[:onk].cpu().numpy(), oidx)
        np.testing.assert_array_equal(yc[:onk].cpu().numpy(), oyc)
        src = torch.arange(n, dtype=torch.float32, device=DEV) + 1
        dst = torch.full((n,), 7.0, device=DEV)
        L.lmhead_expand(src, idx, nk, n, dst)
        want = np.zeros(n, np.float32)
        want[oidx] = np.arange(onk, dtype=np.float32) + 1
        np.testing.assert_array_equal(dst.cpu().numpy(), want)


def test_keep_mask_builder_bit_exact():
    rng = np.random.default_rng(14)
    lens = [int(x) for x in rng.integers(1, 300, 40)]
    n = sum(lens)
    comps = [((rng.random(n) < p) * rng.standard_normal(n)).astype(np.float32)
             for p in (0.3, 0.1, 0.05)]
    sc = LMHeadScorer(n, 64, 50)
    t = [torch.from_numpy(c).to(DEV) for c in comps]
    for k in range(1, 4):
        keep = sc.keep_mask(*(t[:k] + [None] * (3 - k)), seq_lens=lens)
        np.testing.assert_array_equal(keep.cpu().numpy(), O.build_keep_mask(comps[:k], lens))


def test_target_out_of_range_sets_status():
    w = synth.workload("tiny", seed=15, N=128, H=64, V=500)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V)
    keep = torch.zeros(w.N, dtype=torch.uint8, device=DEV)
    keep[5] = 1
    y = inp["targets"].clone()
    y[6] = -100          # skipped row: never read
    sc.forward(inp["hidden"], inp["weight"], y, keep)
    assert sc.status() == 0
    y[5] = w.V           # kept row out of range
    sc.forward(inp["hidden"], inp["weight"], y, keep)
    assert sc.status() == L.LMHEAD_ETARGET


def test_no_allocation_inside_calls():
    w = synth.workload("tiny", seed=16, N=512, H=256, V=4096)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V)
    lp = torch.empty(w.N, device=DEV)
    ent = torch.empty(w.N, device=DEV)
    lse = torch.empty(w.N, device=DEV)
    dh = torch.empty_like(inp["hidden"])
    dW = torch.empty(w.V, w.H, device=DEV)
    torch.cuda.synchronize()
    base = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"], out=(lp, ent, lse))
    sc.backward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"], lse, ent,
                inp["grad_logprob"], inp["grad_entropy"], dweight=dW, dhidden=dh)
    torch.cuda.synchronize()
    assert torch.cuda.max_memory_allocated() == base


# ------------------------------------------------------------ full sizes

def _sampled_rows_check(w, inp, keep, out, count, with_bwd):
    """Oracle on sampled kept rows (row-local outputs) of a full-size batch."""
    kept = torch.nonzero(keep).flatten().cpu().numpy() if keep is not None else np.arange(w.N)
    pick = kept[synth.sample_rows(len(kept), count, w.seed)]
    rows = torch.from_numpy(pick).to(DEV)
    W = to64(inp["weight"])
    h = to64(inp["hidden"][rows])
    y = inp["targets"][rows].cpu().numpy()
    g1 = inp["grad_logprob"][rows].cpu().double().numpy() if with_bwd else None
    g2 = (inp["grad_entropy"][rows].cpu().double().numpy()
          if with_bwd and inp["grad_entropy"] is not None else None)
    lp, ent, lse, dh, _ = O.score_rows(h, W, y, g1, g2)
    assert_rows_close(out["lp"][rows].cpu().double().numpy(), lp, "logprob (sampled)")
    assert_rows_close(out["ent"][rows].cpu().double().numpy(), ent, "entropy (sampled)")
    assert_rows_close(out["lse"][rows].cpu().double().numpy(), lse, "lse (sampled)")
    if with_bwd:
        assert_frob_close(to64(out["dh"][rows]), dh, "dhidden (sampled rows)")


def test_full_size_qwen3_4b_forward_sampled():
    w = synth.workload("qwen3_4b")
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V)
    keep = gpu_keep(sc, inp)
    np.testing.assert_array_equal(keep.cpu().numpy(), oracle_keep(inp))
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep)
    torch.cuda.synchronize()
    assert sc.status() == 0
    k = keep.bool()
    assert (lp[k] <= 1e-5).all()
    assert (ent[k] >= -1e-5).all() and (ent[k] <= math.log(w.V) + 1e-4).all()
    assert (lp[~k] == 0).all() and (ent[~k] == 0).all()
    _sampled_rows_check(w, inp, keep, dict(lp=lp, ent=ent, lse=lse), 48, False)


def test_row_offsets_past_two_to_the_31_elements():
    # N x H = 2.46e9 elements: every kept row from 2^31 / H = 524288 on starts
    # past the 32-bit element range of hidden and dhidden.  Only kept rows are
    # read, so the others stay zero; V is small so that the oracle checks the
    # whole dW and every kept row.
    N, H, V = 600000, 4096, 3000
    first_far = (1 << 31) // H
    rng = np.random.default_rng(2031)
    near = rng.choice(first_far, 1000, replace=False)
    far = first_far + rng.choice(N - first_far, 1000, replace=False)
    kept = np.sort(np.concatenate([near, far]))
    keep_np = np.zeros(N, np.uint8)
    keep_np[kept] = 1
    g = torch.Generator(device=DEV).manual_seed(2031)
    hidden = torch.zeros(N, H, dtype=torch.bfloat16, device=DEV)
    rows = torch.from_numpy(kept).to(DEV)
    hidden[rows] = torch.randn(len(kept), H, generator=g, device=DEV).to(torch.bfloat16)
    weight = (torch.randn(V, H, generator=g, device=DEV) / math.sqrt(H)).to(torch.bfloat16)
    targets = torch.randint(0, V, (N,), generator=g, device=DEV)
    g_lp = torch.randn(N, generator=g, device=DEV)
    g_ent = 0.1 * torch.randn(N, generator=g, device=DEV)
    keep = torch.from_numpy(keep_np).to(DEV)
    sc = LMHeadScorer(N, H, V)
    lp, ent, lse = sc.forward(hidden, weight, targets, keep)
    dh, dW = sc.backward(hidden, weight, targets, keep, lse, ent, g_lp, g_ent)
    torch.cuda.synchronize()
    assert sc.status() == 0
    olp, oent, olse, odh, odW = O.score_rows(to64(hidden[rows]), to64(weight),
                                             targets[rows].cpu().numpy(),
                                             g_lp[rows].cpu().double().numpy(),
                                             g_ent[rows].cpu().double().numpy())
    assert_rows_close(lp[rows].cpu().double().numpy(), olp, "logprob (rows past 2^31 elements)")
    assert_rows_close(ent[rows].cpu().double().numpy(), oent, "entropy")
    assert_rows_close(lse[rows].cpu().double().numpy(), olse, "lse")
    assert_frob_close(to64(dh[rows]), odh, "dhidden (rows past 2^31 elements)")
    assert_frob_close(dW.cpu().double().numpy(), odW, "dW")
    skipped = torch.from_numpy(np.flatnonzero(keep_np == 0)[-1000:]).to(DEV)  # far rows
    assert (dh[skipped] == 0).all() and (lp[skipped] == 0).all()


def test_full_size_qwen3_4b_forward_backward_metric_only_sampled():
    # the Qwen3-4B head's fwd + bwd with the entropy as a metric only (no
    # entropy gradient, [P2] How it works): sampled rows against the oracle
    w = synth.workload("qwen3_4b")
    inp = synth.make_inputs(w, device=DEV)
    assert inp["grad_entropy"] is None
    sc = LMHeadScorer(w.N, w.H, w.V)
    keep = gpu_keep(sc, inp)
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep)
    dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                         inp["grad_logprob"], None)
    torch.cuda.synchronize()
    assert sc.status() == 0
    _sampled_rows_check(w, inp, keep, dict(lp=lp, ent=ent, lse=lse, dh=dh), 32, True)
    k = keep.bool()
    assert (dh[~k] == 0).all() and (lp[~k] == 0).all()
    col = dW.double().sum(0)
    assert col.abs().max().item() <= 1e-3 * dW.double().abs().sum(0).max().item()


def test_full_size_half_kept_forward_backward_sampled():
    # the bench's workload: 64K packed tokens, half of them kept
    w = synth.workload("moe30b_rl_half")
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V)
    keep = gpu_keep(sc, inp)
    np.testing.assert_array_equal(keep.cpu().numpy(), oracle_keep(inp))
    assert int(keep.sum().item()) == 32767
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep)
    dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                         inp["grad_logprob"], inp["grad_entropy"])
    torch.cuda.synchronize()
    assert sc.status() == 0
    _sampled_rows_check(w, inp, keep, dict(lp=lp, ent=ent, lse=lse, dh=dh), 24, True)
    k = keep.bool()
    assert (dh[~k] == 0).all()
    col = dW.double().sum(0)
    assert col.abs().max().item() <= 1e-3 * dW.double().abs().sum(0).max().item()


_DEPTH = {}


def _full_depth_case():
    """8192 kept rows of 9000 at H = 4096 and V = 3000, with the oracle's
    whole dhidden and dW (computed once for the variants that reuse it)."""
    if not _DEPTH:
        w = synth.workload("moe30b_rl", seed=33, N=9000, V=3000)
        inp = synth.make_inputs(w, device=DEV)
        keep_np = np.zeros(w.N, np.uint8)
        keep_np[np.random.default_rng(33).choice(w.N, 8192, replace=False)] = 1
        odh, odW = O.backward(to64(inp["hidden"]), to64(inp["weight"]),
                              inp["targets"].cpu().numpy(), keep_np,
                              inp["grad_logprob"].cpu().double().numpy(),
                              inp["grad_entropy"].cpu().double().numpy())
        _DEPTH.update(w=w, inp=inp, keep_np=keep_np, odh=odh, odW=odW)
    return _DEPTH


@pytest.mark.parametrize("variant", ["pair", "single", "wide"])
def test_weight_gradient_at_full_chunk_depth(monkeypatch, variant):
    # one chunk of 8192 kept rows: the dW contraction runs over K = 8192 (128
    # K blocks, deeper than a default-bench chunk) for all 16 column tiles of
    # H = 4096; the whole dW is compared element-wise, written and
    # accumulated onto a prior gradient
    monkeypatch.setenv("LMHEAD_GEMM", variant)
    c = _full_depth_case()
    w, inp, keep_np = c["w"], c["inp"], c["keep_np"]
    keep = torch.from_numpy(keep_np).to(DEV)
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=8192)
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep)
    g = (inp["grad_logprob"], inp["grad_entropy"])
    dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent, *g)
    prior = torch.randn(w.V, w.H, generator=torch.Generator(device=DEV).manual_seed(5),
                        device=DEV)
    acc = prior.clone()
    sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent, *g, dweight=acc,
                accumulate=True)
    torch.cuda.synchronize()
    assert sc.status() == 0
    assert int(sc.kept_rows().item()) == 8192
    assert_frob_close(dW.cpu().double().numpy(), c["odW"], "dW (K = 8192)")
    assert_frob_close((acc.double() - prior.double()).cpu().numpy(), c["odW"],
                      "accumulated dW (K = 8192)")
    assert_frob_close(to64(dh), c["odh"], "dhidden (K = 8192)")


def test_full_size_moe30b_rl_forward_backward_sampled():
    w = synth.workload("moe30b_rl")
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V)
    keep = gpu_keep(sc, inp)
    np.testing.assert_array_equal(keep.cpu().numpy(), oracle_keep(inp))
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep)
    dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                         inp["grad_logprob"], inp["grad_entropy"])
    torch.cuda.synchronize()
    assert sc.status() == 0
    _sampled_rows_check(w, inp, keep, dict(lp=lp, ent=ent, lse=lse, dh=dh), 24, True)
    k = keep.bool()
    assert (dh[~k] == 0).all()
    # every row's logit gradient sums to zero over the vocabulary, so the
    # columns of dW sum to (nearly) zero
    col = dW.double().sum(0)
    assert col.abs().max().item() <= 1e-3 * dW.double().abs().sum(0).max().item()


def test_full_vocab_slice_weight_gradient():
    # full H and V, a 192-row slice: the oracle computes the whole dW
    w = synth.workload("moe30b_rl", N=192)
    keep_np = (np.random.default_rng(17).random(w.N) < 0.5).astype(np.uint8)
    _run_both(w, keep_override=keep_np, chunk_rows=64)


# ------------------------------------------------------ one-CTA GEMM variant

@pytest.fixture
def single_cta(monkeypatch):
    # the library reads LMHEAD_GEMM on every call; "single" selects the
    # one-CTA tcgen05 kernel (128 x 256 tiles) instead of the CTA pairs
    monkeypatch.setenv("LMHEAD_GEMM", "single")
    yield


def test_single_cta_variant_tiny(single_cta):
    _run_both(synth.workload("tiny"))


def test_single_cta_variant_ragged_multi_chunk(single_cta):
    _run_both(synth.workload("moe30b_rl", N=3000, H=384, V=5000), chunk_rows=256)


def test_single_cta_variant_empty_and_single_row(single_cta):
    w = synth.workload("tiny", seed=10, N=64, H=64, V=257)
    keep = np.zeros(64, np.uint8)
    keep[37] = 1
    _run_both(w, keep_override=keep)
    _run_both(w, keep_override=np.zeros(64, np.uint8))


def test_variants_agree_bitwise(monkeypatch):
    # the three kernels accumulate every logit over K in the same order, so
    # with dHidden's K range left whole their outputs agree bit for bit (split,
    # which tiles form the split tail depends on each variant's tile count;
    # each variant's split dHidden is checked against the oracle by the
    # parity suite)
    w = synth.workload("tiny", seed=21, N=900, H=320, V=3000)
    inp = synth.make_inputs(w, device=DEV)
    res = []
    monkeypatch.setenv("LMHEAD_DH_SPLIT", "1")
    for variant in ("pair", "single", "wide"):
        monkeypatch.setenv("LMHEAD_GEMM", variant)  # the previous value comes back after the test
        sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=256)
        lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"])
        dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"], lse,
                             ent, inp["grad_logprob"], inp["grad_entropy"])
        torch.cuda.synchronize()
        res.append((lp, ent, lse, dh, dW))
    for other in res[1:]:
        for a, b in zip(res[0], other):
            assert torch.equal(a, b)


_TAIL_ORACLE = {}


@pytest.mark.parametrize("variant", ["pair", "single", "wide"])
@pytest.mark.parametrize("share", ["2", "3", "4"])
def test_dhidden_tail_tiles_split_into_up_to_four_parts(monkeypatch, variant, share):
    # 2560 kept rows in one chunk, H = 2048, V = 8000 (125 K blocks): on 76
    # CTA pairs the 80 pair tiles run one whole wave and a tail of 4 tiles
    # cut into K parts, the 160 one-CTA tiles on 152 CTAs likewise (8 tail
    # tiles), and the 40 wide tiles form a tail alone (in two rounds of parts
    # with 3 or 4 parts allowed); the whole dhidden -- rows written directly
    # and rows summed from partials -- against the oracle
    monkeypatch.setenv("LMHEAD_GEMM", variant)
    monkeypatch.setenv("LMHEAD_DH_SPLIT", share)
    w = synth.workload("tiny", seed=41, N=2560, H=2048, V=8000)
    inp = synth.make_inputs(w, device=DEV)
    keep = torch.ones(w.N, dtype=torch.uint8, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=2560)
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep)
    dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                         inp["grad_logprob"], inp["grad_entropy"])
    dh2, _ = sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                         inp["grad_logprob"], inp["grad_entropy"])
    torch.cuda.synchronize()
    assert sc.status() == 0
    assert torch.equal(dh, dh2)  # the partial sums are added in a fixed order
    if "ref" not in _TAIL_ORACLE:
        h, W = to64(inp["hidden"]), to64(inp["weight"])
        y = inp["targets"].cpu().numpy()
        _TAIL_ORACLE["ref"] = O.backward(h, W, y, np.ones(w.N, np.uint8),
                                            inp["grad_logprob"].cpu().double().numpy(),
                                            inp["grad_entropy"].cpu().double().numpy())
    odh, odW = _TAIL_ORACLE["ref"]
    assert_frob_close(to64(dh), odh, "dhidden")
    assert_frob_close(dW.cpu().double().numpy(), odW, "dW")
    # every row on its own as well: a tile whose partial sums were dropped or
    # added twice shows up in its rows even when the whole matrix passes
    got = to64(dh)
    rel = np.linalg.norm(got - odh, axis=1) / np.linalg.norm(odh, axis=1)
    assert rel.max() < 2e-2, rel.max()


def test_wide_tiles_chosen_per_contraction(monkeypatch):
    # LMHEAD_WIDE names the contractions on 256 x 512 tiles (the rest on
    # 256 x 256): each choice matches the oracle, and the forward results
    # agree bit for bit across choices (every variant accumulates a logit
    # over K in the same order)
    monkeypatch.delenv("LMHEAD_GEMM", raising=False)  # it would take precedence
    w = synth.workload("tiny", seed=33, N=1500, H=1024, V=6000)
    first = None
    for wide in ("none", "fwd,dz", "dh", "dw,dh", "fwd,dz,dh,dw"):
        monkeypatch.setenv("LMHEAD_WIDE", wide)  # restored after the test
        _, _, _, out, _ = _run_both(w, chunk_rows=512)
        fwd = [out[k].clone() for k in ("lp", "ent", "lse")]
        if first is None:
            first = fwd
        for a, b in zip(first, fwd):
            assert torch.equal(a, b), wide


@pytest.mark.parametrize("nk", [255, 256, 257, 511, 513, 1000])
def test_chunk_boundaries(nk):
    # the kept rows are cut into equal 256-aligned chunks on the device; Nk
    # around chunk multiples exercises the first / last chunk bounds
    w = synth.workload("tiny", seed=30 + nk, N=1100, H=64, V=300)
    keep = np.zeros(w.N, np.uint8)
    keep[np.random.default_rng(nk).choice(w.N, nk, replace=False)] = 1
    _run_both(w, keep_override=keep, chunk_rows=256)


@pytest.mark.parametrize("variant", ["pair", "single", "wide"])
@pytest.mark.parametrize("N,H,V", [(1, 8, 1), (5, 16, 2), (33, 64, 7), (300, 8, 300),
                                   (70, 24, 129)])
def test_tiny_and_degenerate_shapes(monkeypatch, variant, N, H, V):
    # shapes smaller than one tile in every dimension: TMA boxes reach past the
    # tensor (zero fill), V = 1 makes every logprob and entropy exactly 0
    monkeypatch.setenv("LMHEAD_GEMM", variant)
    w = synth.workload("tiny", seed=90 + N + V, N=N, H=H, V=V)
    _run_both(w, keep_override=np.ones(N, np.uint8))
    if N > 1:
        keep = np.zeros(N, np.uint8)
        keep[::2] = 1
        _run_both(w, keep_override=keep)


# ------------------------------------------------ block-sparse tile skipping

@pytest.mark.parametrize("variant", ["pair", "single", "wide"])
def test_blocksparse_matches_the_oracle(monkeypatch, variant):
    monkeypatch.setenv("LMHEAD_GEMM", variant)
    # contiguous active suffixes (the entropy-bonus layout), ragged H and V,
    # several chunks of active tiles
    w = synth.workload("entropy_bonus", N=5000, H=320, V=3001)
    _run_both(w, chunk_rows=512, blocksparse=True, active_frac=0.4)
    # scattered keep mask: almost every tile is active
    _run_both(synth.workload("tiny", seed=140, N=700, H=192, V=1500), blocksparse=True)


def test_blocksparse_edge_cases():
    w = synth.workload("tiny", seed=141, N=300, H=64, V=700)
    _run_both(w, keep_override=None, blocksparse=True)
    _run_both(w, keep_override=np.zeros(300, np.uint8), blocksparse=True)
    one = np.zeros(300, np.uint8)
    one[299] = 1  # a kept row in the last, partial tile
    _run_both(w, keep_override=one, blocksparse=True, chunk_rows=256)


def test_blocksparse_forward_equals_compaction_bitwise():
    # a row's logits accumulate in the same order wherever the row sits, so
    # the forward results of the two strategies agree bit for bit
    w = synth.workload("entropy_bonus", N=6144, H=256, V=4000)
    inp = synth.make_inputs(w, device=DEV, active_frac=0.7)
    outs = []
    for bs in (False, True):
        sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=1024, blocksparse=bs)
        keep = gpu_keep(sc, inp)
        lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep)
        dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                             inp["grad_logprob"], inp["grad_entropy"])
        torch.cuda.synchronize()
        assert sc.status() == 0
        outs.append((lp, ent, lse, dh, dW))
    (a, b) = outs
    for x, y in zip(a[:3], b[:3]):
        assert torch.equal(x, y)
    assert torch.allclose(a[3].float(), b[3].float(), rtol=2e-2, atol=1e-3)
    assert torch.allclose(a[4], b[4], rtol=1e-4, atol=1e-5)


def _full_size_fwd_bwd(w, active_frac=1.0, rows=16):
    """Returns the device memory the scoring calls added (their outputs)."""
    inp = synth.make_inputs(w, device=DEV, active_frac=active_frac)
    sc = LMHeadScorer(w.N, w.H, w.V)
    keep = gpu_keep(sc, inp)
    np.testing.assert_array_equal(keep.cpu().numpy(), oracle_keep(inp))
    torch.cuda.synchronize()
    before = torch.cuda.memory_allocated()
    torch.cuda.reset_peak_memory_stats()
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep)
    dh, dW = sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                         inp["grad_logprob"], inp["grad_entropy"])
    torch.cuda.synchronize()
    added = torch.cuda.max_memory_allocated() - before
    assert sc.status() == 0
    _sampled_rows_check(w, inp, keep, dict(lp=lp, ent=ent, lse=lse, dh=dh), rows, True)
    k = keep.bool()
    assert (lp[~k] == 0).all() and (dh[~k] == 0).all()
    col = dW.sum(0, dtype=torch.float64)
    l1 = torch.linalg.vector_norm(dW, 1, dim=0)
    assert col.abs().max().item() <= 1e-3 * l1.max().item()
    return added


def test_full_size_entropy_bonus_sampled():
    _full_size_fwd_bwd(synth.workload("entropy_bonus"), active_frac=0.64)


def test_full_size_long_context_sampled():
    # the largest workload: N = 262144 rows, H = 5120; no [N, V] buffer exists
    w = synth.workload("long_context")
    added = _full_size_fwd_bwd(w, rows=12)
    # only the outputs (logprob, entropy, lse, dhidden, dW) are allocated
    outputs = w.N * 4 * 3 + w.N * w.H * 2 + w.V * w.H * 4
    assert added <= outputs + (1 << 20)
    assert added < 0.1 * w.N * w.V * 2


def test_random_shape_sweep(monkeypatch):
    # seeded random problems: shapes, keep densities, chunk sizes, GEMM
    # variant and strategy all vary; every one must match the oracle
    rng = np.random.default_rng(2026)
    for case in range(12):
        N = int(rng.integers(1, 1500))
        H = int(rng.choice([8, 16, 64, 136, 256, 520]))
        V = int(rng.integers(1, 4200))
        chunk = int(rng.choice([0, 256, 512, 768]))
        density = float(rng.choice([0.0, 0.05, 0.5, 1.0]))
        keep = (rng.random(N) < density).astype(np.uint8)
        variant = str(rng.choice(["pair", "single", "wide"]))
        bs = bool(rng.integers(0, 2))
        ent = bool(rng.integers(0, 2))
        monkeypatch.setenv("LMHEAD_GEMM", variant)  # restored after the test
        w = synth.workload("tiny", seed=300 + case, N=N, H=H, V=V)
        _run_both(w, chunk_rows=chunk, keep_override=keep, blocksparse=bs, grad_entropy=ent)


def test_random_sweep_of_schedules_and_accumulation(monkeypatch):
    # seeded random problems up to 6000 rows and 2048 columns, over the
    # dHidden split caps (whole tiles, tails in 2-4 K parts, as the tile count
    # and fill fall), the GEMM variants and the default per-contraction
    # choice, both strategies, entropy gradient on or off and dW accumulated
    # onto a prior gradient or written; every one must match the oracle
    if os.environ.get("LMHEAD_GEMM"):
        pytest.skip("picks the GEMM variant of every case itself")
    rng = np.random.default_rng(7)
    for case in range(30):
        while True:
            N = int(rng.integers(1, 6000))
            H = int(rng.choice([8, 24, 64, 136, 256, 512, 520, 1024, 1536, 2048]))
            V = int(rng.integers(1, 30000))
            if N * H * V <= 3e9:
                break
        chunk = int(rng.choice([0, 256, 512, 768, 1280, 2048, 4096]))
        density = float(rng.choice([0.0, 0.02, 0.3, 0.7, 1.0]))
        keep = (rng.random(N) < density).astype(np.uint8)
        variant = str(rng.choice(["pair", "single", "wide", "default"]))
        split = str(rng.choice(["1", "2", "3", "4"]))
        bs = bool(rng.integers(0, 2))
        ent = bool(rng.integers(0, 2))
        acc = bool(rng.integers(0, 2))
        if variant == "default":
            monkeypatch.delenv("LMHEAD_GEMM", raising=False)
        else:
            monkeypatch.setenv("LMHEAD_GEMM", variant)
        monkeypatch.setenv("LMHEAD_DH_SPLIT", split)  # both restored after the test
        w = synth.workload("tiny", seed=1000 + case, N=N, H=H, V=V)
        _run_both(w, chunk_rows=chunk, keep_override=keep, blocksparse=bs, grad_entropy=ent,
                  accumulate=acc)


@pytest.mark.parametrize("variant", ["pair", "single", "wide"])
def test_wide_hidden_and_long_vocabulary(monkeypatch, variant):
    # H = 8192: 128 K steps in the projections and 32 column tiles in dHidden
    # and dW; V = 200000: 782 vocabulary tiles ending in a 64-wide tail, so
    # the last dZ box and the last dW rows reach past the matrix and are
    # clipped by the output maps
    monkeypatch.setenv("LMHEAD_GEMM", variant)
    _run_both(synth.workload("tiny", seed=510, N=520, H=8192, V=3000), chunk_rows=256)
    _run_both(synth.workload("tiny", seed=511, N=96, H=256, V=200000), chunk_rows=256)


@pytest.mark.parametrize("variant", ["pair", "single", "wide"])
def test_widest_hidden_and_largest_vocabulary(monkeypatch, variant):
    # H = 16384: 256 K steps in the projections, 64 column tiles in dHidden
    # and dW; V = 262144 (a 256K vocabulary): 1024 vocabulary tiles and
    # 4096 K steps in dHidden
    monkeypatch.setenv("LMHEAD_GEMM", variant)
    _run_both(synth.workload("tiny", seed=512, N=300, H=16384, V=1500), chunk_rows=256)
    _run_both(synth.workload("tiny", seed=513, N=80, H=512, V=262144), chunk_rows=256)


def test_expand_skips_and_reports_out_of_range_indices():
    # lmhead_expand takes idx and Nk from the caller: entries outside [0, N)
    # (and Nk > N) are skipped and reported as LMHEAD_EBOUNDS.  dst sits inside
    # a larger guarded buffer, so nothing lands outside memory the test owns.
    n, guard = 100, 64
    buf = torch.full((n + 2 * guard,), -5.0, device=DEV)
    dst = buf[guard:guard + n]
    src = torch.arange(1, 9, dtype=torch.float32, device=DEV)
    idx = torch.tensor([3, -1, 50, n, 99, n + 5, 0, 7], dtype=torch.int32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lmhead_expand(src, idx, torch.tensor([8], dtype=torch.int32, device=DEV), n, dst, st)
    torch.cuda.synchronize()
    assert int(st.item()) == L.LMHEAD_EBOUNDS
    want = np.zeros(n, np.float32)
    for k, r in enumerate(idx.tolist()):
        if 0 <= r < n:
            want[r] = k + 1
    np.testing.assert_array_equal(dst.cpu().numpy(), want)
    assert (buf[:guard] == -5.0).all() and (buf[guard + n:] == -5.0).all()
    # Nk larger than N: the first N entries are expanded and the excess reported
    st.zero_()
    src2 = torch.arange(1, n + 1, dtype=torch.float32, device=DEV)
    idx2 = torch.arange(n - 1, -1, -1, dtype=torch.int32, device=DEV)
    L.lmhead_expand(src2, idx2, torch.tensor([n + 40], dtype=torch.int32, device=DEV), n, dst, st)
    torch.cuda.synchronize()
    assert int(st.item()) == L.LMHEAD_EBOUNDS
    np.testing.assert_array_equal(dst.cpu().numpy(), np.arange(n, 0, -1, dtype=np.float32))
    # valid input leaves the status word alone
    st.zero_()
    L.lmhead_expand(src2, idx2, torch.tensor([n], dtype=torch.int32, device=DEV), n, dst, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0


def test_millions_of_rows_and_a_hundred_chunks():
    # N = 2.1 M rows (513 compaction blocks), about 1.05 M kept rows in 129
    # chunks of 8192, with a tiny head so the oracle stays cheap
    _run_both(synth.workload("tiny", seed=520, N=2_100_000, H=8, V=20))


def test_numerical_extremes():
    N, H, V = 300, 64, 1000
    sc = LMHeadScorer(N, H, V, chunk_rows=256)
    g = torch.Generator(device=DEV)
    g.manual_seed(530)
    h = torch.randn(N, H, generator=g, device=DEV).to(torch.bfloat16)
    y = torch.randint(0, V, (N,), generator=g, device=DEV)
    y[0], y[1] = 0, V - 1  # the first and last vocabulary ids
    keep = torch.ones(N, dtype=torch.uint8, device=DEV)
    # identical W rows: every logit of a row is equal -> uniform distribution
    Wu = torch.randn(1, H, generator=g, device=DEV).repeat(V, 1).to(torch.bfloat16)
    lp, ent, lse = sc.forward(h, Wu, y, keep)
    torch.cuda.synchronize()
    assert sc.status() == 0
    np.testing.assert_allclose(lp.cpu().numpy(), -np.log(V), atol=1e-4)
    np.testing.assert_allclose(ent.cpu().numpy(), np.log(V), atol=1e-4)
    # very peaked rows (W x 100): logits of order 100, no overflow, lp <= 0,
    # entropy >= 0, and the oracle's values
    Wp = (torch.randn(V, H, generator=g, device=DEV) * (100.0 / np.sqrt(H))).to(torch.bfloat16)
    lp, ent, lse = sc.forward(h, Wp, y, keep)
    g_lp = torch.randn(N, generator=g, device=DEV)
    g_ent = 0.1 * torch.randn(N, generator=g, device=DEV)
    dh, dW = sc.backward(h, Wp, y, keep, lse, ent, g_lp, g_ent)
    torch.cuda.synchronize()
    assert sc.status() == 0
    for t in (lp, ent, lse, dh.float(), dW):
        assert torch.isfinite(t).all()
    assert (lp <= 1e-5).all() and (ent >= -1e-5).all()
    olp, oent, olse = O.forward(to64(h), to64(Wp), y.cpu().numpy(), None)
    assert_rows_close(lp.cpu().double().numpy(), olp, "logprob")
    assert_rows_close(ent.cpu().double().numpy(), oent, "entropy")
    assert_rows_close(lse.cpu().double().numpy(), olse, "lse")
    odh, odW = O.backward(to64(h), to64(Wp), y.cpu().numpy(), None, to64(g_lp), to64(g_ent))
    assert_frob_close(to64(dh), odh, "dhidden")
    assert_frob_close(dW.cpu().double().numpy(), odW, "dW")
