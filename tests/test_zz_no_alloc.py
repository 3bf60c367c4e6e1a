"""lmhead_compact_noalloc: compaction for callers that cannot allocate.

Callers with no device allocator of their own (a plugin inside a framework
whose caching allocator owns the GPU memory, or a service that must not call
cudaMalloc after start-up) use this entry point: its scratch lives in a fixed
array inside the library, so they pass only inputs and outputs.  This test
calls it through the C ABI twice in a row, on different inputs, and checks
each result against lmhead_compact (the workspace entry point) bit for bit.
It sits in its own file, collected last.
"""

import ctypes

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

DEV = "cuda"
MAX_ROWS = 16777216  # LMHEAD_NOALLOC_MAX_ROWS


def _noalloc(L):
    fn = L.lmhead_compact_noalloc
    vp = ctypes.c_void_p
    fn.restype = ctypes.c_int
    fn.argtypes = [vp, vp, ctypes.c_int64, ctypes.c_int, vp, vp, vp, vp, vp]
    return fn


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_noalloc_compaction_matches_workspace_entry_point():
    from sft_keep_mask_gb300 import lmhead

    L = lmhead.lib()
    fn = _noalloc(L)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    rng = np.random.default_rng(2024)
    V = 151936
    # calls in a row with different sizes and masks: each reuses the scratch
    # the one before left behind; 8192 rows fill exactly two scan blocks of
    # 4096, so the last block is a full one
    for call, (n, p_keep) in enumerate([(100003, 0.55), (37000, 0.2), (8192, 0.5)]):
        keep = torch.from_numpy((rng.random(n) < p_keep).astype(np.uint8)).to(DEV)
        y = torch.from_numpy(rng.integers(0, V, n)).to(DEV)
        outs = []
        for which in ("workspace", "noalloc"):
            idx = torch.full((n,), -1, dtype=torch.int32, device=DEV)
            yc = torch.full((n,), -1, dtype=torch.int32, device=DEV)
            nk = torch.full((1,), -1, dtype=torch.int32, device=DEV)
            if which == "workspace":
                ws = torch.empty(lmhead.lmhead_workspace_size(n, 8, V, 0, 0), dtype=torch.uint8,
                                 device=DEV)
                lmhead.lmhead_compact(keep, y, V, idx, yc, nk, ws)
                st = lmhead.lmhead_get_status(ws)
            else:
                d_st = torch.full((1,), -7, dtype=torch.int32, device=DEV)
                code = fn(_p(keep), _p(y), n, V, _p(idx), _p(yc), _p(nk), _p(d_st), stream)
                assert code == 0, f"call {call}: status {code}"
                torch.cuda.synchronize()
                st = int(d_st.item())
            outs.append((idx.cpu(), yc.cpu(), int(nk.item()), st))
        (i0, y0, n0, s0), (i1, y1, n1, s1) = outs
        assert s0 == 0 and s1 == 0
        assert n0 == n1 == int(keep.sum().item())
        assert torch.equal(i0[:n0], i1[:n1])
        assert torch.equal(y0[:n0], y1[:n1])


def test_noalloc_rejects_oversize_and_reports_bad_targets():
    from sft_keep_mask_gb300 import lmhead

    L = lmhead.lib()
    fn = _noalloc(L)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    fake = ctypes.c_void_p(1 << 20)
    assert fn(None, fake, MAX_ROWS + 1, 10, fake, fake, fake, fake, stream) == 1
    n = 5000
    keep = torch.ones(n, dtype=torch.uint8, device=DEV)
    y = torch.zeros(n, dtype=torch.int64, device=DEV)
    y[4321] = 10  # out of range for V = 10
    idx = torch.empty(n, dtype=torch.int32, device=DEV)
    yc = torch.empty(n, dtype=torch.int32, device=DEV)
    nk = torch.empty(1, dtype=torch.int32, device=DEV)
    d_st = torch.zeros(1, dtype=torch.int32, device=DEV)
    assert fn(_p(keep), _p(y), n, 10, _p(idx), _p(yc), _p(nk), _p(d_st), stream) == 0
    torch.cuda.synchronize()
    assert int(d_st.item()) == lmhead.LMHEAD_ETARGET
    y[4321] = 9  # a clean call clears the status it reports
    assert fn(_p(keep), _p(y), n, 10, _p(idx), _p(yc), _p(nk), _p(d_st), stream) == 0
    torch.cuda.synchronize()
    assert int(d_st.item()) == 0 and int(nk.item()) == n


def test_noalloc_empty_batch_writes_zero_kept_rows():
    # N = 0 launches nothing: Nk is written as 0 and the status cleared
    from sft_keep_mask_gb300 import lmhead

    L = lmhead.lib()
    fn = _noalloc(L)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    one = torch.zeros(1, dtype=torch.int64, device=DEV)  # any device buffer; N = 0 reads none
    idx = torch.empty(1, dtype=torch.int32, device=DEV)
    yc = torch.empty(1, dtype=torch.int32, device=DEV)
    nk = torch.full((1,), 77, dtype=torch.int32, device=DEV)
    d_st = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    assert fn(None, _p(one), 0, 10, _p(idx), _p(yc), _p(nk), _p(d_st), stream) == 0
    torch.cuda.synchronize()
    assert int(nk.item()) == 0 and int(d_st.item()) == 0
