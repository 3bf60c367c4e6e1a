"""Scoring of existing logits (selective_log_softmax) against the oracle.

Float32 logprob / entropy / lse within 1e-3 of the float64 oracle, logit
gradient within 1e-2 relative Frobenius error (bf16 output) or 1e-5 (float32
output); skipped rows exactly zero.
"""

import math

import numpy as np
import pytest
import torch

from oracle import lmhead_oracle as O
from sft_keep_mask_gb300 import lmhead as L
from sft_keep_mask_gb300 import synth
from tests._util import assert_frob_close, assert_rows_close, frob_rel

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run(d, keep_np=None, grad_entropy=True, want_entropy=True):
    z = d["logits"]
    N, V = z.shape
    keep = None if keep_np is None else torch.from_numpy(keep_np).to(DEV)
    lp = torch.empty(N, device=DEV)
    ent = torch.empty(N, device=DEV)
    lse = torch.empty(N, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    L.lmhead_selective_log_softmax_fwd(z, d["targets"], keep, want_entropy, lp, ent, lse, st)
    dz = torch.empty(N, V, dtype=z.dtype, device=DEV)
    ge = d["grad_entropy"] if grad_entropy else None
    L.lmhead_selective_log_softmax_bwd(z, d["targets"], keep, lse, ent, d["grad_logprob"], ge,
                                       dz, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    z64 = z.float().cpu().double().numpy()
    y = d["targets"].cpu().numpy()
    olp, oent, olse = O.selective_log_softmax(z64, y, keep_np, want_entropy)
    assert_rows_close(lp.cpu().double().numpy(), olp, "logprob")
    assert_rows_close(lse.cpu().double().numpy(), olse, "lse")
    if want_entropy:
        assert_rows_close(ent.cpu().double().numpy(), oent, "entropy")
    odz = O.selective_log_softmax_backward(
        z64, y, keep_np, d["grad_logprob"].cpu().double().numpy(),
        ge.cpu().double().numpy() if ge is not None else None)
    got = dz.float().cpu().double().numpy()
    if z.dtype == torch.bfloat16:
        assert_frob_close(got, odz, "dlogits")
    else:
        assert frob_rel(got, odz) <= 1e-5
    if keep_np is not None:
        off = keep_np == 0
        assert (lp.cpu().numpy()[off] == 0).all() and not dz.cpu()[torch.from_numpy(off)].any()
    return lp, ent, lse, dz


@pytest.mark.parametrize("V", [5000, 5003])
def test_bf16_logits_vector_and_scalar_paths(V):
    d = synth.make_logits(300, V, seed=50, device=DEV)
    keep = (np.random.default_rng(50).random(300) < 0.6).astype(np.uint8)
    _run(d, keep)


def test_strided_rows_and_metric_only_entropy():
    d = synth.make_logits(200, 4000, seed=51, device=DEV, ld=4096)
    assert d["logits"].stride(0) == 4096
    _run(d, None, grad_entropy=False)
    _run(d, None, grad_entropy=False, want_entropy=False)


def test_random_sweep_of_shapes_strides_and_dtypes():
    # seeded problems: row counts, vocabularies down to one token, bf16 or
    # fp32 logits, row strides that keep rows 16-byte aligned or not (the
    # vector and the scalar path), logit scales, keep densities, and the
    # entropy as a loss term, a metric or absent
    rng = np.random.default_rng(57)
    for case in range(12):
        N = int(rng.integers(1, 600))
        V = int(rng.integers(1, 20000))
        dtype = torch.bfloat16 if rng.integers(0, 2) else torch.float32
        ld = V + int(rng.choice([0, 1, 3, 8, 64]))
        d = synth.make_logits(N, V, seed=580 + case, std=float(rng.choice([0.5, 2.0, 8.0])),
                              dtype=dtype, device=DEV, ld=ld)
        density = float(rng.choice([0.0, 0.3, 1.0, -1.0]))  # -1: no mask
        keep = None if density < 0 else (rng.random(N) < density).astype(np.uint8)
        ge = bool(rng.integers(0, 2))
        want = True if ge else bool(rng.integers(0, 2))
        _run(d, keep, grad_entropy=ge, want_entropy=want)


def test_float32_logits():
    d = synth.make_logits(150, 3001, seed=52, dtype=torch.float32, device=DEV)
    _run(d, None)


def test_large_negative_logprob_is_not_quantised():
    # a target logit 40 below every other: log p = -40 - log(V - 1 + e^-40);
    # bf16 has a spacing of 0.25 at this magnitude, the float32 result must
    # be far closer than that
    V = 4096
    z = torch.zeros(4, V, dtype=torch.bfloat16, device=DEV)
    y = torch.tensor([7, 100, 2000, 4095], device=DEV)
    z[torch.arange(4), y] = -40.0
    lp = torch.empty(4, device=DEV)
    ent = torch.empty(4, device=DEV)
    lse = torch.empty(4, device=DEV)
    L.lmhead_selective_log_softmax_fwd(z, y, None, True, lp, ent, lse)
    torch.cuda.synchronize()
    want = -40.0 - math.log(V - 1 + math.exp(-40.0))
    assert np.abs(lp.cpu().double().numpy() - want).max() < 1e-3


def test_target_out_of_range_sets_status():
    d = synth.make_logits(16, 300, seed=53, device=DEV)
    y = d["targets"].clone()
    y[3] = 300
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    lp = torch.empty(16, device=DEV)
    lse = torch.empty(16, device=DEV)
    L.lmhead_selective_log_softmax_fwd(d["logits"], y, None, False, lp, None, lse, st)
    torch.cuda.synchronize()
    assert int(st.item()) == L.LMHEAD_ETARGET


def test_full_size_sampled_rows():
    # the shape of the pull request's measurements: N=16384, V=151936, bf16
    N, V = 16384, 151936
    d = synth.make_logits(N, V, seed=54, device=DEV)
    z = d["logits"]
    lp = torch.empty(N, device=DEV)
    ent = torch.empty(N, device=DEV)
    lse = torch.empty(N, device=DEV)
    L.lmhead_selective_log_softmax_fwd(z, d["targets"], None, True, lp, ent, lse)
    dz = torch.empty_like(z)
    L.lmhead_selective_log_softmax_bwd(z, d["targets"], None, lse, ent, d["grad_logprob"],
                                       d["grad_entropy"], dz)
    torch.cuda.synchronize()
    rows = torch.from_numpy(synth.sample_rows(N, 32, 54)).to(DEV)
    z64 = z[rows].float().cpu().double().numpy()
    y = d["targets"][rows].cpu().numpy()
    olp, oent, olse = O.selective_log_softmax(z64, y)
    assert_rows_close(lp[rows].cpu().double().numpy(), olp, "logprob")
    assert_rows_close(ent[rows].cpu().double().numpy(), oent, "entropy")
    assert_rows_close(lse[rows].cpu().double().numpy(), olse, "lse")
    odz = O.selective_log_softmax_backward(z64, y, None,
                                           d["grad_logprob"][rows].cpu().double().numpy(),
                                           d["grad_entropy"][rows].cpu().double().numpy())
    assert_frob_close(dz[rows].float().cpu().double().numpy(), odz, "dlogits (sampled rows)")
