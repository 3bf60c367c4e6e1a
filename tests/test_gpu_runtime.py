"""Runtime behaviour of the C ABI: CUDA-graph capture of a whole forward +
backward step and the device-side kept-row count."""

import numpy as np
import pytest
import torch

from sft_keep_mask_gb300 import lmhead as L
from sft_keep_mask_gb300 import synth
from sft_keep_mask_gb300.api import LMHeadScorer

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_forward_backward_step_replays_from_a_cuda_graph():
    w = synth.workload("moe30b_rl", seed=130, N=2048, H=256, V=3000)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=512)
    off = np.zeros(len(inp["seq_lens"]) + 1, np.int32)
    off[1:] = np.cumsum(inp["seq_lens"])
    offsets = torch.from_numpy(off).to(DEV)
    keep = torch.empty(w.N, dtype=torch.uint8, device=DEV)
    lp = torch.empty(w.N, device=DEV)
    ent = torch.empty(w.N, device=DEV)
    lse = torch.empty(w.N, device=DEV)
    dh = torch.empty_like(inp["hidden"])
    dW = torch.empty(w.V, w.H, device=DEV)

    def step():
        s = torch.cuda.current_stream()
        L.lmhead_build_keep_mask(inp["components"][0], None, None, offsets, keep, s)
        L.lmhead_fwd(inp["hidden"], inp["weight"], inp["targets"], keep, True, lp, ent, lse,
                     sc.workspace, 512, s)
        L.lmhead_bwd(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                     inp["grad_logprob"], inp["grad_entropy"], dh, dW, False, sc.workspace,
                     512, s)

    step()  # eager; also the one-time per-process set-up of the library
    torch.cuda.synchronize()
    want = [t.clone() for t in (keep, lp, ent, lse, dh, dW)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for t in (keep, lp, ent, lse, dh, dW):
        t.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert sc.status() == 0
    for got, exp in zip((keep, lp, ent, lse, dh, dW), want):
        assert torch.equal(got, exp)


def test_kept_rows_on_the_device():
    w = synth.workload("tiny", seed=131, N=999, H=64, V=500)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V)
    sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"])
    torch.cuda.synchronize()
    assert int(sc.kept_rows().item()) == int(inp["keep"].sum().item())
