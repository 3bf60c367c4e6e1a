"""Host-side checks of the C ABI that need no GPU.

The library must load, export every function that ``include/lmhead.h``
declares, size its workspace as documented, and reject bad arguments with a
status code before touching the device.
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "lmhead.h")


@pytest.fixture(scope="module")
def L():
    from sft_keep_mask_gb300 import build as b
    b.build()
    from sft_keep_mask_gb300 import lmhead
    return lmhead.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(lmhead_[a-z_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for want in ("lmhead_workspace_size", "lmhead_compact", "lmhead_fwd", "lmhead_bwd",
                 "lmhead_expand", "lmhead_build_keep_mask", "lmhead_get_status",
                 "lmhead_strerror"):
        assert want in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in _declared() if not hasattr(L, n)]
    assert not missing, missing


def test_strerror_and_version(L):
    from sft_keep_mask_gb300 import lmhead
    assert lmhead.lmhead_strerror(0) == "ok"
    assert "workspace" in lmhead.lmhead_strerror(2)
    assert "sm_103a" in lmhead.lmhead_version()


def test_workspace_size_formula(L):
    from sft_keep_mask_gb300 import lmhead
    f = lmhead.lmhead_workspace_size
    assert f(-1, 64, 64) == 0 and f(10, 0, 64) == 0 and f(10, 64, 0) == 0
    # grows with the chunk, not with [N, V]: doubling N at a fixed chunk adds
    # only O(N) bytes
    H, V = 4096, 151936
    a = f(65536, H, V, True, 8192)
    b = f(131072, H, V, True, 8192)
    assert b - a < 65536 * 64
    assert a < 65536 * V * 2 / 4  # far below a bf16 [N, V] logit buffer
    # chunk buffers: dz [C, V] bf16 + h_c [C, H] bf16 + partials [V/256, C] x 16 B
    # + dHidden tail partials [4, C, H] fp32
    C = 8192
    core = C * V * 2 + C * H * 2 + (V // 256 + 1) * C * 16 + 4 * C * H * 4
    assert core <= a <= core + 65536 * 48 + 4096


def _fake(addr=1 << 20):
    return ctypes.c_void_p(addr)


def test_bad_arguments_return_einval_without_a_device(L):
    N, H, V = 16, 64, 128
    ws = _fake()
    big = 1 << 40
    # H not a multiple of 8
    assert L.lmhead_fwd(_fake(), _fake(), _fake(), None, N, 60, V, 1, _fake(), _fake(), _fake(),
                        0, ws, big, None) == 1
    # NULL hidden
    assert L.lmhead_fwd(None, _fake(), _fake(), None, N, H, V, 1, _fake(), _fake(), _fake(),
                        0, ws, big, None) == 1
    # entropy requested but NULL
    assert L.lmhead_fwd(_fake(), _fake(), _fake(), None, N, H, V, 1, _fake(), None, _fake(),
                        0, ws, big, None) == 1
    # unaligned hidden
    assert L.lmhead_fwd(_fake((1 << 20) + 2), _fake(), _fake(), None, N, H, V, 1, _fake(),
                        _fake(), _fake(), 0, ws, big, None) == 1
    # workspace too small
    assert L.lmhead_fwd(_fake(), _fake(), _fake(), None, N, H, V, 1, _fake(), _fake(), _fake(),
                        0, ws, 1024, None) == 2
    # unaligned workspace
    assert L.lmhead_fwd(_fake(), _fake(), _fake(), None, N, H, V, 1, _fake(), _fake(), _fake(),
                        0, _fake((1 << 20) + 16), big, None) == 1
    # backward: grad_entropy without entropy
    assert L.lmhead_bwd(_fake(), _fake(), _fake(), None, N, H, V, _fake(), None, _fake(),
                        _fake(), _fake(), _fake(), 0, 0, ws, big, None) == 1
    # backward: NULL dweight
    assert L.lmhead_bwd(_fake(), _fake(), _fake(), None, N, H, V, _fake(), _fake(), _fake(),
                        _fake(), _fake(), None, 0, 0, ws, big, None) == 1
    # expand / compact / keep mask argument checks
    assert L.lmhead_expand(None, _fake(), _fake(), N, _fake(), None, None) == 1
    assert L.lmhead_compact(None, None, N, V, _fake(), _fake(), _fake(), ws, big, None) == 1
    assert L.lmhead_build_keep_mask(None, None, None, None, 1, N, _fake(), None) == 1


def test_valid_call_without_a_gpu_reports_unsupported(L):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    N, H, V = 16, 64, 128
    assert L.lmhead_fwd(_fake(), _fake(), _fake(), None, N, H, V, 1, _fake(), _fake(), _fake(),
                        0, _fake(), 1 << 40, None) == 6


def test_binding_refuses_a_missing_library(monkeypatch, tmp_path):
    from sft_keep_mask_gb300 import lmhead
    monkeypatch.setattr(lmhead, "_lib", None)
    monkeypatch.setattr(lmhead, "_LIB_PATH", str(tmp_path / "nope.so"))
    with pytest.raises(RuntimeError, match="missing"):
        lmhead.lib()


def test_autograd_op_rejects_bad_arguments_before_any_call():
    import torch
    from sft_keep_mask_gb300 import hidden_to_logprobs
    h = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(16, 8, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError, match="return_entropy"):
        hidden_to_logprobs(h, W, y, entropy_requires_grad=True)
    with pytest.raises(TypeError, match="main_grad"):
        hidden_to_logprobs(h, W, y, main_grad=torch.zeros(16, 8, dtype=torch.bfloat16))
    with pytest.raises(TypeError, match="main_grad"):
        hidden_to_logprobs(h, W, y, main_grad=torch.zeros(8, 16))


def test_binding_runs_each_call_on_its_tensors_device():
    import torch
    from sft_keep_mask_gb300 import lmhead
    assert lmhead._device_of(None, None) is None
    with pytest.raises(TypeError, match="CUDA"):
        lmhead._device_of(torch.zeros(2))  # host tensors never reach the library


def test_workspace_size_never_decreases_with_n(L):
    # a workspace sized for N_max serves every smaller batch (the header's
    # promise, which LMHeadScorer and the autograd op rely on)
    from sft_keep_mask_gb300 import lmhead
    f = lmhead.lmhead_workspace_size
    for H, V, C in ((8, 20, 256), (4096, 151936, 0), (192, 3000, 768)):
        prev = 0
        for N in list(range(0, 3000, 7)) + [8191, 8192, 8193, 65536, 262144]:
            cur = f(N, H, V, True, C)
            assert cur >= prev, (H, V, C, N)
            prev = cur
