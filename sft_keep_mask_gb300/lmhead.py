"""Thin Python binding of the C ABI in ``include/lmhead.h``.

Argument marshalling only: each function takes torch tensors already on the
GPU, passes their device pointers and the current CUDA stream to the function
of the same name in ``liblmhead.so``, and raises ``LmheadError`` on a non-OK
status.  Every step of the scoring path runs in the library's own kernels;
there is no fallback, and a missing library is an error.
"""

from __future__ import annotations

import ctypes
import os

import torch

# LMHEAD_LIBRARY=debug selects the build with device-side index checks.
_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib",
                         "liblmhead_debug.so" if os.environ.get("LMHEAD_LIBRARY") == "debug"
                         else "liblmhead.so")
_lib = None

LMHEAD_OK = 0
LMHEAD_EINVAL = 1
LMHEAD_EWORKSPACE = 2
LMHEAD_ETARGET = 3
LMHEAD_ECUDA = 4
LMHEAD_ETIMEOUT = 5
LMHEAD_EUNSUPPORTED = 6
LMHEAD_EBOUNDS = 7
DEFAULT_CHUNK_ROWS = 8192


class LmheadError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {lmhead_strerror(code)} (status {code})")


_VP = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int
_SIGS = {
    "lmhead_workspace_size": (ctypes.c_size_t, [_I64, _I32, _I32, _I32, _I32]),
    "lmhead_build_keep_mask": (_I32, [_VP, _VP, _VP, _VP, ctypes.c_int32, _I64, _VP, _VP]),
    "lmhead_compact": (_I32, [_VP, _VP, _I64, _I32, _VP, _VP, _VP, _VP, ctypes.c_size_t, _VP]),
    "lmhead_fwd": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _I32, _VP, _VP, _VP, _I32, _VP,
                          ctypes.c_size_t, _VP]),
    "lmhead_bwd": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _VP, _VP, _VP, _VP, _VP, _VP,
                          _I32, _I32, _VP, ctypes.c_size_t, _VP]),
    "lmhead_expand": (_I32, [_VP, _VP, _VP, _I64, _VP, _VP, _VP]),
    "lmhead_fwd_blocksparse": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _I32, _VP, _VP, _VP,
                                      _I32, _VP, ctypes.c_size_t, _VP]),
    "lmhead_bwd_blocksparse": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _VP, _VP, _VP, _VP,
                                      _VP, _VP, _I32, _I32, _VP, ctypes.c_size_t, _VP]),
    "lmhead_fwd_shard": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _I64, _I64, _I32, _VP, _I32,
                                _VP, ctypes.c_size_t, _VP]),
    "lmhead_merge_shards": (_I32, [_VP, _I32, _VP, _I64, _I32, _VP, _VP, _VP, _VP]),
    "lmhead_bwd_shard": (_I32, [_VP, _VP, _VP, _VP, _I64, _I32, _I32, _I64, _I64, _VP, _VP, _VP,
                                _VP, _VP, _VP, _I32, _I32, _VP, ctypes.c_size_t, _VP]),
    "lmhead_selective_log_softmax_fwd": (_I32, [_VP, _I32, _I64, _VP, _VP, _I64, _I32, _I32, _VP,
                                                _VP, _VP, _VP, _VP]),
    "lmhead_selective_log_softmax_bwd": (_I32, [_VP, _I32, _I64, _VP, _VP, _I64, _I32, _VP, _VP,
                                                _VP, _VP, _VP, _I64, _VP, _VP]),
    "lmhead_get_status": (_I32, [_VP, _VP]),
    "lmhead_get_timeout_record": (ctypes.c_int32, [_VP, _VP]),
    "lmhead_workspace_kept_rows": (_VP, [_VP]),
    "lmhead_strerror": (ctypes.c_char_p, [_I32]),
    "lmhead_profile_enable": (None, [_I32]),
    "lmhead_profile_kinds": (_I32, []),
    "lmhead_profile_kind_name": (ctypes.c_char_p, [_I32]),
    "lmhead_profile_read": (_I32, [ctypes.POINTER(ctypes.c_int64), ctypes.POINTER(ctypes.c_double)]),
    "lmhead_launch_count": (ctypes.c_int64, []),
    "lmhead_version": (ctypes.c_char_p, []),
}


def library_path() -> str:
    return _LIB_PATH


def lib():
    """The loaded ``liblmhead.so``; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(
                f"{_LIB_PATH} is missing: build the CUDA library first "
                "(python -c 'import __graft_entry__ as g; g.build()')")
        handle = ctypes.CDLL(_LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _lib = handle
    return _lib


def _p(t):
    return None if t is None else _VP(t.data_ptr())


def _s(stream, device=None):
    s = torch.cuda.current_stream(device) if stream is None else stream
    return _VP(s.cuda_stream)


def _device_of(*tensors):
    """The one CUDA device of the given tensors (None ignored); the library
    launches on the current device, so every call runs under this one."""
    dev = None
    for t in tensors:
        if t is None:
            continue
        if not t.is_cuda:
            raise TypeError("every tensor argument must be a CUDA tensor")
        if dev is None:
            dev = t.device
        elif t.device != dev:
            raise ValueError(f"tensors on different devices ({dev} and {t.device})")
    return dev


def _call(name, tensors, *args, stream=None):
    """Runs lib().<name>(*args, stream) on the tensors' device and returns the
    status code."""
    dev = _device_of(*tensors)
    if dev is None:
        return getattr(lib(), name)(*args, _s(stream))
    with torch.cuda.device(dev):
        return getattr(lib(), name)(*args, _s(stream, dev))


def _check(code, where):
    if code != LMHEAD_OK:
        raise LmheadError(code, where)


def _need(t, dtype, name, numel=None):
    if t is None:
        return
    if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
        raise TypeError(f"{name} must be a contiguous CUDA tensor of {dtype}")
    if numel is not None and t.numel() != numel:
        raise ValueError(f"{name} must have {numel} elements, has {t.numel()}")


def lmhead_strerror(code: int) -> str:
    return lib().lmhead_strerror(int(code)).decode()


def lmhead_version() -> str:
    return lib().lmhead_version().decode()


def lmhead_workspace_size(N: int, H: int, V: int, want_entropy: bool = True,
                          chunk_rows: int = 0) -> int:
    return int(lib().lmhead_workspace_size(N, H, V, int(want_entropy), chunk_rows))


def lmhead_build_keep_mask(loss_mask, ce_weight, kl_weight, seq_offsets, keep, stream=None):
    N = keep.numel()
    for name, t in (("loss_mask", loss_mask), ("ce_weight", ce_weight), ("kl_weight", kl_weight)):
        _need(t, torch.float32, name, N)
    _need(seq_offsets, torch.int32, "seq_offsets")
    _need(keep, torch.uint8, "keep")
    code = _call("lmhead_build_keep_mask", (loss_mask, ce_weight, kl_weight, seq_offsets, keep),
                 _p(loss_mask), _p(ce_weight), _p(kl_weight), _p(seq_offsets),
                 seq_offsets.numel() - 1, N, _p(keep), stream=stream)
    _check(code, "lmhead_build_keep_mask")


def lmhead_compact(keep, targets, V, idx, targets_c, d_nk, workspace, stream=None):
    N = targets.numel()
    _need(keep, torch.uint8, "keep", N)
    _need(targets, torch.int64, "targets")
    _need(idx, torch.int32, "idx", N)
    _need(targets_c, torch.int32, "targets_c", N)
    _need(d_nk, torch.int32, "d_nk", 1)
    _need(workspace, torch.uint8, "workspace")
    code = _call("lmhead_compact", (keep, targets, idx, targets_c, d_nk, workspace),
                 _p(keep), _p(targets), N, V, _p(idx), _p(targets_c), _p(d_nk), _p(workspace),
                 workspace.numel(), stream=stream)
    _check(code, "lmhead_compact")


def lmhead_fwd(hidden, weight, targets, keep, want_entropy, logprob, entropy, lse, workspace,
               chunk_rows=0, stream=None, _entry="lmhead_fwd"):
    N, H = hidden.shape
    V = weight.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight", V * H)
    _need(targets, torch.int64, "targets", N)
    _need(keep, torch.uint8, "keep", N)
    _need(logprob, torch.float32, "logprob", N)
    _need(entropy, torch.float32, "entropy", N)
    _need(lse, torch.float32, "lse", N)
    _need(workspace, torch.uint8, "workspace")
    code = _call(_entry, (hidden, weight, targets, keep, logprob, entropy, lse, workspace),
                 _p(hidden), _p(weight), _p(targets), _p(keep), N, H, V,
                 int(bool(want_entropy)), _p(logprob), _p(entropy), _p(lse), int(chunk_rows),
                 _p(workspace), workspace.numel(), stream=stream)
    _check(code, _entry)


def lmhead_bwd(hidden, weight, targets, keep, lse, entropy, grad_logprob, grad_entropy, dhidden,
               dweight, dw_accumulate, workspace, chunk_rows=0, stream=None, _entry="lmhead_bwd"):
    N, H = hidden.shape
    V = weight.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight, torch.bfloat16, "weight", V * H)
    _need(targets, torch.int64, "targets", N)
    _need(keep, torch.uint8, "keep", N)
    _need(lse, torch.float32, "lse", N)
    _need(entropy, torch.float32, "entropy", N)
    _need(grad_logprob, torch.float32, "grad_logprob", N)
    _need(grad_entropy, torch.float32, "grad_entropy", N)
    _need(dhidden, torch.bfloat16, "dhidden", N * H)
    _need(dweight, torch.float32, "dweight", V * H)
    _need(workspace, torch.uint8, "workspace")
    code = _call(_entry, (hidden, weight, targets, keep, lse, entropy, grad_logprob,
                          grad_entropy, dhidden, dweight, workspace),
                 _p(hidden), _p(weight), _p(targets), _p(keep), N, H, V, _p(lse), _p(entropy),
                 _p(grad_logprob), _p(grad_entropy), _p(dhidden), _p(dweight),
                 int(bool(dw_accumulate)), int(chunk_rows), _p(workspace), workspace.numel(),
                 stream=stream)
    _check(code, _entry)


def lmhead_fwd_blocksparse(hidden, weight, targets, keep, want_entropy, logprob, entropy, lse,
                           workspace, chunk_rows=0, stream=None):
    lmhead_fwd(hidden, weight, targets, keep, want_entropy, logprob, entropy, lse, workspace,
               chunk_rows, stream, _entry="lmhead_fwd_blocksparse")


def lmhead_bwd_blocksparse(hidden, weight, targets, keep, lse, entropy, grad_logprob,
                           grad_entropy, dhidden, dweight, dw_accumulate, workspace, chunk_rows=0,
                           stream=None):
    lmhead_bwd(hidden, weight, targets, keep, lse, entropy, grad_logprob, grad_entropy, dhidden,
               dweight, dw_accumulate, workspace, chunk_rows, stream,
               _entry="lmhead_bwd_blocksparse")


def lmhead_fwd_shard(hidden, weight_shard, v_begin, V_total, targets, keep, want_entropy,
                     partials, workspace, chunk_rows=0, stream=None):
    N, H = hidden.shape
    Vs = weight_shard.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight_shard, torch.bfloat16, "weight_shard", Vs * H)
    _need(targets, torch.int64, "targets", N)
    _need(keep, torch.uint8, "keep", N)
    _need(partials, torch.float32, "partials", N * 4)
    _need(workspace, torch.uint8, "workspace")
    code = _call("lmhead_fwd_shard", (hidden, weight_shard, targets, keep, partials, workspace),
                 _p(hidden), _p(weight_shard), _p(targets), _p(keep), N, H, Vs, int(v_begin),
                 int(V_total), int(bool(want_entropy)), _p(partials), int(chunk_rows),
                 _p(workspace), workspace.numel(), stream=stream)
    _check(code, "lmhead_fwd_shard")


def lmhead_merge_shards(partials, keep, want_entropy, logprob, entropy, lse, stream=None):
    S, N = partials.shape[0], partials.shape[1]
    _need(partials, torch.float32, "partials", S * N * 4)
    _need(keep, torch.uint8, "keep", N)
    _need(logprob, torch.float32, "logprob", N)
    _need(entropy, torch.float32, "entropy", N)
    _need(lse, torch.float32, "lse", N)
    code = _call("lmhead_merge_shards", (partials, keep, logprob, entropy, lse),
                 _p(partials), S, _p(keep), N, int(bool(want_entropy)), _p(logprob),
                 _p(entropy), _p(lse), stream=stream)
    _check(code, "lmhead_merge_shards")


def lmhead_bwd_shard(hidden, weight_shard, v_begin, V_total, targets, keep, lse, entropy,
                     grad_logprob, grad_entropy, dhidden_partial, dweight_shard, dw_accumulate,
                     workspace, chunk_rows=0, stream=None):
    N, H = hidden.shape
    Vs = weight_shard.shape[0]
    _need(hidden, torch.bfloat16, "hidden")
    _need(weight_shard, torch.bfloat16, "weight_shard", Vs * H)
    _need(targets, torch.int64, "targets", N)
    _need(keep, torch.uint8, "keep", N)
    _need(lse, torch.float32, "lse", N)
    _need(entropy, torch.float32, "entropy", N)
    _need(grad_logprob, torch.float32, "grad_logprob", N)
    _need(grad_entropy, torch.float32, "grad_entropy", N)
    _need(dhidden_partial, torch.bfloat16, "dhidden_partial", N * H)
    _need(dweight_shard, torch.float32, "dweight_shard", Vs * H)
    _need(workspace, torch.uint8, "workspace")
    code = _call("lmhead_bwd_shard", (hidden, weight_shard, targets, keep, lse, entropy,
                                       grad_logprob, grad_entropy, dhidden_partial,
                                       dweight_shard, workspace),
                 _p(hidden), _p(weight_shard), _p(targets), _p(keep), N, H, Vs, int(v_begin),
                 int(V_total), _p(lse), _p(entropy), _p(grad_logprob), _p(grad_entropy),
                 _p(dhidden_partial), _p(dweight_shard), int(bool(dw_accumulate)),
                 int(chunk_rows), _p(workspace), workspace.numel(), stream=stream)
    _check(code, "lmhead_bwd_shard")


def lmhead_expand(src, idx, d_nk, N, dst, d_status=None, stream=None):
    _need(src, torch.float32, "src")
    _need(idx, torch.int32, "idx")
    _need(d_nk, torch.int32, "d_nk", 1)
    _need(dst, torch.float32, "dst", N)
    _need(d_status, torch.int32, "d_status", 1)
    code = _call("lmhead_expand", (src, idx, d_nk, dst, d_status), _p(src), _p(idx), _p(d_nk), N,
                 _p(dst), _p(d_status), stream=stream)
    _check(code, "lmhead_expand")


def _logits_dtype(t):
    if t.dtype == torch.bfloat16:
        return 0
    if t.dtype == torch.float32:
        return 1
    raise TypeError("logits must be bf16 or float32")


def _rows(t, name):
    if not t.is_cuda or t.dim() != 2 or t.stride(1) != 1:
        raise TypeError(f"{name} must be a 2-D CUDA tensor with unit column stride")
    return t.stride(0)


def lmhead_selective_log_softmax_fwd(logits, targets, keep, want_entropy, logprob, entropy, lse,
                                     d_status=None, stream=None):
    N, V = logits.shape
    ld = _rows(logits, "logits")
    _need(targets, torch.int64, "targets", N)
    _need(keep, torch.uint8, "keep", N)
    _need(logprob, torch.float32, "logprob", N)
    _need(entropy, torch.float32, "entropy", N)
    _need(lse, torch.float32, "lse", N)
    _need(d_status, torch.int32, "d_status", 1)
    code = _call("lmhead_selective_log_softmax_fwd",
                 (logits, targets, keep, logprob, entropy, lse, d_status),
                 _p(logits), _logits_dtype(logits), ld, _p(targets), _p(keep), N, V,
                 int(bool(want_entropy)), _p(logprob), _p(entropy), _p(lse), _p(d_status),
                 stream=stream)
    _check(code, "lmhead_selective_log_softmax_fwd")


def lmhead_selective_log_softmax_bwd(logits, targets, keep, lse, entropy, grad_logprob,
                                     grad_entropy, dlogits, d_status=None, stream=None):
    N, V = logits.shape
    ld = _rows(logits, "logits")
    ld_out = _rows(dlogits, "dlogits")
    if dlogits.dtype != logits.dtype or tuple(dlogits.shape) != (N, V):
        raise TypeError("dlogits must match the logits' shape and dtype")
    _need(targets, torch.int64, "targets", N)
    _need(keep, torch.uint8, "keep", N)
    _need(lse, torch.float32, "lse", N)
    _need(entropy, torch.float32, "entropy", N)
    _need(grad_logprob, torch.float32, "grad_logprob", N)
    _need(grad_entropy, torch.float32, "grad_entropy", N)
    _need(d_status, torch.int32, "d_status", 1)
    code = _call("lmhead_selective_log_softmax_bwd",
                 (logits, targets, keep, lse, entropy, grad_logprob, grad_entropy, dlogits,
                  d_status),
                 _p(logits), _logits_dtype(logits), ld, _p(targets), _p(keep), N, V, _p(lse),
                 _p(entropy), _p(grad_logprob), _p(grad_entropy), _p(dlogits), ld_out,
                 _p(d_status), stream=stream)
    _check(code, "lmhead_selective_log_softmax_bwd")


def lmhead_get_status(workspace, stream=None) -> int:
    """Device status of the last call on this workspace (synchronises)."""
    return int(_call("lmhead_get_status", (workspace,), _p(workspace), stream=stream))


# Pipeline waits named by lmhead_get_timeout_record (site codes 1 .. 6).
TIMEOUT_SITES = {1: "producer: free stage", 2: "MMA issuer: released accumulator",
                 3: "MMA issuer: filled stage", 4: "epilogue: finished accumulator",
                 5: "producer: drain of its loads", 6: "MMA issuer: drain of its MMAs"}


def lmhead_get_timeout_record(workspace, stream=None):
    """(site, cta) of the first pipeline wait that gave up in the last call on
    this workspace, or None if none did (synchronises)."""
    rec = int(_call("lmhead_get_timeout_record", (workspace,), _p(workspace), stream=stream))
    if rec < 0:
        raise LmheadError(LMHEAD_ECUDA, "lmhead_get_timeout_record")
    return None if rec == 0 else (rec >> 24, rec & 0xFFFFFF)


def lmhead_workspace_kept_rows(workspace):
    """A 1-element int32 CUDA tensor viewing Nk in the workspace (no copy)."""
    addr = lib().lmhead_workspace_kept_rows(_p(workspace))
    off = addr - workspace.data_ptr()
    return workspace[off:off + 4].view(torch.int32)


def lmhead_profile_enable(on: bool = True):
    lib().lmhead_profile_enable(int(bool(on)))


def lmhead_profile_read():
    """{kernel kind: (launches, total device ms)} since the last read."""
    L = lib()
    k = L.lmhead_profile_kinds()
    launches = (ctypes.c_int64 * k)()
    ms = (ctypes.c_double * k)()
    _check(L.lmhead_profile_read(launches, ms), "lmhead_profile_read")
    return {L.lmhead_profile_kind_name(i).decode(): (int(launches[i]), float(ms[i]))
            for i in range(k)}


def lmhead_launch_count() -> int:
    return int(lib().lmhead_launch_count())
