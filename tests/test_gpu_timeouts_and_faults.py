"""Failure detection without a GPU fault.

* Host sites: with LMHEAD_FAULT naming a site the call returns an error code
  instead of launching, and the next call without it works.
* Device waits: with LMHEAD_FAULT=stall the GEMM producer issues no loads, so
  nothing ever completes the pipeline barriers; every wait gives up after its
  time limit, the kernel returns, the status word reads LMHEAD_ETIMEOUT, the
  timeout record names a wait on filled stages or on a finished accumulator
  (the waits the missing loads starve), and the context stays usable for the
  next call, which clears the record.
* Guard bands: bytes around the workspace and the outputs are unchanged by a
  forward + backward (no out-of-bounds writes).
"""

import numpy as np
import pytest
import torch

from oracle import lmhead_oracle as O
from sft_keep_mask_gb300 import lmhead as L
from sft_keep_mask_gb300 import synth
from sft_keep_mask_gb300.api import LMHeadScorer
from tests._util import assert_rows_close, to64

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _small():
    w = synth.workload("tiny", seed=120, N=200, H=128, V=1000)
    return w, synth.make_inputs(w, device=DEV)


def _check_forward(w, inp, sc):
    lp, ent, lse = sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"])
    torch.cuda.synchronize()
    assert sc.status() == 0
    olp, oent, olse = O.forward(to64(inp["hidden"]), to64(inp["weight"]),
                                inp["targets"].cpu().numpy(), inp["keep"].cpu().numpy())
    assert_rows_close(lp.cpu().double().numpy(), olp, "logprob")
    assert_rows_close(ent.cpu().double().numpy(), oent, "entropy")


@pytest.mark.parametrize("site", ["tensor_map", "launch"])
def test_host_fault_sites_return_an_error_and_recover(monkeypatch, site):
    w, inp = _small()
    sc = LMHeadScorer(w.N, w.H, w.V)
    monkeypatch.setenv("LMHEAD_FAULT", site)
    with pytest.raises(L.LmheadError) as e:
        sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"])
    assert e.value.code == L.LMHEAD_ECUDA
    monkeypatch.delenv("LMHEAD_FAULT")
    _check_forward(w, inp, sc)


@pytest.mark.parametrize("variant", ["pair", "single", "wide"])
def test_stalled_pipeline_times_out_and_the_context_survives(monkeypatch, variant):
    w, inp = _small()
    sc = LMHeadScorer(w.N, w.H, w.V)
    monkeypatch.setenv("LMHEAD_GEMM", variant)
    monkeypatch.setenv("LMHEAD_FAULT", "stall")
    sc.forward(inp["hidden"], inp["weight"], inp["targets"], inp["keep"])
    assert sc.status() == L.LMHEAD_ETIMEOUT
    site, cta = L.lmhead_get_timeout_record(sc.workspace)
    # the MMA issuer starves on a filled stage, the epilogue on a finished
    # accumulator: whichever gave up first is recorded
    assert site in (3, 4) and 0 <= cta < 1024
    monkeypatch.delenv("LMHEAD_FAULT")
    _check_forward(w, inp, sc)
    assert L.lmhead_get_timeout_record(sc.workspace) is None


def test_guard_bands_around_workspace_and_outputs():
    w = synth.workload("moe30b_rl", seed=121, N=1500, H=320, V=3000)
    inp = synth.make_inputs(w, device=DEV)
    sc = LMHeadScorer(w.N, w.H, w.V, chunk_rows=256)
    keep = sc.keep_mask(inp["components"][0], seq_lens=inp["seq_lens"])
    G = 1 << 16

    def guarded(n, dtype):
        buf = torch.empty(n * torch.tensor([], dtype=dtype).element_size() + 2 * G,
                          dtype=torch.uint8, device=DEV)
        buf.fill_(0xA5)
        return buf, buf[G:G + n * torch.tensor([], dtype=dtype).element_size()].view(dtype)

    ws_buf, ws = guarded(sc.workspace.numel(), torch.uint8)
    sc.workspace = ws
    lp_buf, lp = guarded(w.N, torch.float32)
    ent_buf, ent = guarded(w.N, torch.float32)
    lse_buf, lse = guarded(w.N, torch.float32)
    dh_buf, dh = guarded(w.N * w.H, torch.bfloat16)
    dW_buf, dW = guarded(w.V * w.H, torch.float32)
    sc.forward(inp["hidden"], inp["weight"], inp["targets"], keep, out=(lp, ent, lse))
    sc.backward(inp["hidden"], inp["weight"], inp["targets"], keep, lse, ent,
                inp["grad_logprob"], inp["grad_entropy"], dweight=dW.view(w.V, w.H),
                dhidden=dh.view(w.N, w.H))
    torch.cuda.synchronize()
    assert sc.status() == 0
    for name, buf in (("workspace", ws_buf), ("logprob", lp_buf), ("entropy", ent_buf),
                      ("lse", lse_buf), ("dhidden", dh_buf), ("dW", dW_buf)):
        head = buf[:G].cpu().numpy()
        tail = buf[-G:].cpu().numpy()
        assert (head == 0xA5).all() and (tail == 0xA5).all(), f"{name} guard band overwritten"


def test_host_memory_passed_as_a_device_buffer_is_refused():
    # a pinned host buffer where device memory is expected: the call returns
    # LMHEAD_EINVAL from its pointer check and launches nothing
    w, inp = _small()
    sc = LMHeadScorer(w.N, w.H, w.V)
    lib = L.lib()
    out = [torch.empty(w.N, dtype=torch.float32, device=DEV) for _ in range(3)]
    host_keep = inp["keep"].cpu().pin_memory()
    stream = torch.cuda.current_stream().cuda_stream
    torch.cuda.synchronize()
    before = L.lmhead_launch_count()
    code = lib.lmhead_fwd(inp["hidden"].data_ptr(), inp["weight"].data_ptr(),
                          inp["targets"].data_ptr(), host_keep.data_ptr(), w.N, w.H, w.V, 1,
                          out[0].data_ptr(), out[1].data_ptr(), out[2].data_ptr(), 0,
                          sc.workspace.data_ptr(), sc.workspace.numel(), stream)
    assert code == L.LMHEAD_EINVAL
    assert L.lmhead_launch_count() == before
    _check_forward(w, inp, sc)  # the next valid call works
