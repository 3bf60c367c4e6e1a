"""The autograd op ``hidden_to_logprobs`` against the float64 oracle.

A loss built from the op's outputs is differentiated by torch autograd; the
gradients that reach ``hidden`` and ``weight`` (or ``main_grad``) come from
lmhead_bwd and must match the oracle's backward of the same loss.
"""

import numpy as np
import pytest
import torch

from oracle import lmhead_oracle as O
from sft_keep_mask_gb300 import lmhead as L
from sft_keep_mask_gb300 import synth
from sft_keep_mask_gb300.autograd import hidden_to_logprobs, workspace_status
from tests._util import assert_frob_close, assert_rows_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _inputs(seed=300, N=700, H=192, V=3000):
    w = synth.workload("tiny", seed=seed, N=N, H=H, V=V)
    return w, synth.make_inputs(w, device=DEV)


def _leaves(inp):
    h = inp["hidden"].clone().requires_grad_(True)
    W = inp["weight"].clone().requires_grad_(True)
    return h, W


def test_entropy_in_the_loss_matches_the_oracle():
    w, inp = _inputs()
    h, W = _leaves(inp)
    lp, ent = hidden_to_logprobs(h, W, inp["targets"], inp["keep"], return_entropy=True,
                                 entropy_requires_grad=True, chunk_rows=256)
    loss = (inp["grad_logprob"] * lp).sum() + (inp["grad_entropy"] * ent).sum()
    loss.backward()
    torch.cuda.synchronize()
    assert workspace_status(h, W, 256) == 0
    keep = inp["keep"].cpu().numpy()
    y = inp["targets"].cpu().numpy()
    olp, oent, _ = O.forward(to64(h), to64(W), y, keep)
    odh, odW = O.backward(to64(h), to64(W), y, keep, to64(inp["grad_logprob"]),
                          to64(inp["grad_entropy"]))
    assert_rows_close(lp.detach().cpu().double().numpy(), olp, "logprob")
    assert_rows_close(ent.detach().cpu().double().numpy(), oent, "entropy")
    assert h.grad.dtype == torch.bfloat16 and W.grad.dtype == torch.bfloat16
    assert_frob_close(to64(h.grad), odh, "dhidden")
    assert_frob_close(to64(W.grad), odW, "dW")
    # rows outside the keep mask get exactly zero gradient
    assert not h.grad[inp["keep"] == 0].any()


def test_metric_only_entropy_has_no_gradient():
    w, inp = _inputs(seed=301)
    h, W = _leaves(inp)
    lp, ent = hidden_to_logprobs(h, W, inp["targets"], inp["keep"], return_entropy=True)
    assert not ent.requires_grad
    (inp["grad_logprob"] * lp).sum().backward()
    keep = inp["keep"].cpu().numpy()
    y = inp["targets"].cpu().numpy()
    odh, odW = O.backward(to64(h), to64(W), y, keep, to64(inp["grad_logprob"]))
    assert_frob_close(to64(h.grad), odh, "dhidden")
    assert_frob_close(to64(W.grad), odW, "dW")


def test_logprob_only_bool_mask_and_main_grad_accumulation():
    w, inp = _inputs(seed=302)
    h, W = _leaves(inp)
    main = torch.full((w.V, w.H), 0.25, dtype=torch.float32, device=DEV)
    keep_bool = inp["keep"].bool()
    lp = hidden_to_logprobs(h, W, inp["targets"], keep_bool, main_grad=main)
    assert isinstance(lp, torch.Tensor)
    (inp["grad_logprob"] * lp).sum().backward()
    torch.cuda.synchronize()
    assert W.grad is None  # the gradient went into main_grad
    keep = inp["keep"].cpu().numpy()
    y = inp["targets"].cpu().numpy()
    olp, _, _ = O.forward(to64(h), to64(W), y, keep, want_entropy=False)
    odh, odW = O.backward(to64(h), to64(W), y, keep, to64(inp["grad_logprob"]))
    assert_rows_close(lp.detach().cpu().double().numpy(), olp, "logprob")
    assert_frob_close(to64(h.grad), odh, "dhidden")
    assert_frob_close(main.cpu().double().numpy() - 0.25, odW, "dW accumulated in main_grad")


def test_unused_logprob_with_entropy_loss_and_every_row_kept():
    # only the entropy enters the loss; keep_mask None scores every row
    w, inp = _inputs(seed=303, N=300, H=128, V=2100)
    h, W = _leaves(inp)
    _, ent = hidden_to_logprobs(h, W, inp["targets"], None, return_entropy=True,
                                entropy_requires_grad=True)
    (inp["grad_entropy"] * ent).sum().backward()
    y = inp["targets"].cpu().numpy()
    zeros = np.zeros(w.N)
    odh, odW = O.backward(to64(h), to64(W), y, None, zeros, to64(inp["grad_entropy"]))
    assert_frob_close(to64(h.grad), odh, "dhidden")
    assert_frob_close(to64(W.grad), odW, "dW")


def test_bad_target_on_a_kept_row_is_reported():
    w, inp = _inputs(seed=304, N=200, H=64, V=1000)
    y = inp["targets"].clone()
    kept = int(torch.nonzero(inp["keep"])[0])
    y[kept] = w.V  # out of range on a kept row
    h, W = _leaves(inp)
    hidden_to_logprobs(h, W, y, inp["keep"])
    assert workspace_status(h, W) == L.LMHEAD_ETARGET


def test_changing_batch_size_reuses_one_workspace():
    # RL batches change N from step to step: the op keeps one workspace per
    # (device, H, V, chunk) and grows it only when a larger N needs more
    from sft_keep_mask_gb300 import autograd as A
    H, V = 128, 2100
    sizes = []
    for i, N in enumerate((700, 300, 650, 900, 500)):
        w, inp = _inputs(seed=310 + i, N=N, H=H, V=V)
        h, W = _leaves(inp)
        lp = hidden_to_logprobs(h, W, inp["targets"], inp["keep"], chunk_rows=256)
        (inp["grad_logprob"] * lp).sum().backward()
        keep = inp["keep"].cpu().numpy()
        y = inp["targets"].cpu().numpy()
        odh, odW = O.backward(to64(h), to64(W), y, keep, to64(inp["grad_logprob"]))
        assert_frob_close(to64(h.grad), odh, "dhidden")
        assert_frob_close(to64(W.grad), odW, "dW")
        ws = A.workspace_for(N, H, V, 256, h.device)
        sizes.append(ws.numel())
    keys = [k for k in A._workspaces if k[2:] == (H, V, 256)]
    assert len(keys) == 1
    # grew only for the two sizes larger than every earlier one
    assert len(set(sizes)) <= 2


def test_backward_saves_no_full_vocabulary_activation():
    # twinkle pull request #283, section 1: the backward must not keep a
    # full-vocabulary activation alive.  Every tensor the op saves is either
    # one of its inputs (no new memory) or a per-row vector (lse, entropy):
    # the extra bytes grow with the rows, never with rows x vocabulary.
    extra = {}
    for N in (512, 1024):
        w, inp = _inputs(seed=310, N=N, H=128, V=20000)
        h, W = _leaves(inp)
        inputs = {t.data_ptr() for t in (h, W, inp["targets"], inp["keep"])}
        saved = []

        def pack(t):
            saved.append((t.data_ptr(), tuple(t.shape), t.numel() * t.element_size()))
            return t

        with torch.autograd.graph.saved_tensors_hooks(pack, lambda t: t):
            lp, ent = hidden_to_logprobs(h, W, inp["targets"], inp["keep"],
                                         return_entropy=True, entropy_requires_grad=True)
        (lp.sum() + ent.sum()).backward()
        torch.cuda.synchronize()
        assert h.grad is not None and W.grad is not None
        new = [(shape, b) for ptr, shape, b in saved if ptr not in inputs]
        assert all(w.V not in shape for shape, _ in new), new
        extra[N] = sum(b for _, b in new)
    assert extra[512] == 512 * 8 and extra[1024] == 1024 * 8  # lse + entropy, fp32
