"""Autograd op over the C ABI: per-row target log-probability (and entropy)
straight from hidden states and the LM-head weight, skipping rows outside the
keep mask.

This is the interface of the fused op in SkyRL pull request #2374,
"feat(megatron): fuse LM-head entropy for RL" (Overview): one projection
returns the log-probability of every row's target and, with
``return_entropy``, its entropy; ``entropy_requires_grad`` decides whether
the entropy is a logged metric or a term of the loss that gets its own
gradient.  The keep mask is the one of prime-rl pull request #3326, "Don't
compute the logprobs and their gradients for masked tokens" (Overview): a
row outside it reads 0 and takes no part in either gradient.

Forward is ``lmhead_fwd``, backward ``lmhead_bwd`` (the logits are
recomputed, never stored).  The weight gradient is the library's fp32
accumulator: pass ``main_grad`` (an fp32 [V, H] tensor) to have it added
there in place, in which case ``weight`` receives no ``.grad``; otherwise
the fp32 gradient is cast to the weight's dtype by torch for autograd.
Everything else is argument marshalling; no step of the scoring runs outside
the library.  Device-side errors (a kept row whose target is outside
[0, V)) are reported through ``workspace_status``.

Calls for the same head (device, H, V, chunk_rows) share one workspace, so
they must be ordered on one stream (as forward and backward of a training
step are); work on other streams needs its own ``LMHeadScorer``.
"""

from __future__ import annotations

import torch

from . import lmhead as L

_workspaces: dict = {}


def workspace_for(N: int, H: int, V: int, chunk_rows: int, device) -> torch.Tensor:
    """A workspace for N rows of this head on `device`.

    One buffer is kept per (device, H, V, chunk_rows) and reused for any N
    whose workspace fits in it (the library lays the workspace out from N and
    only needs enough bytes), so a batch size that changes from step to step
    does not allocate a new workspace each time; it grows by a quarter beyond
    the largest size asked for so far when it is too small.
    """
    dev = torch.device(device)
    if dev.index is None:
        dev = torch.device(dev.type, torch.cuda.current_device())
    key = (dev.type, dev.index, H, V, chunk_rows)
    need = max(L.lmhead_workspace_size(N, H, V, True, chunk_rows), 256)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < need:
        if ws is not None:
            need += need // 4
            del _workspaces[key]
            ws = None
        ws = torch.empty(need, dtype=torch.uint8, device=dev)
        _workspaces[key] = ws
    return ws


def workspace_status(hidden: torch.Tensor, weight: torch.Tensor, chunk_rows: int = 0) -> int:
    """Device status word of the last call on the workspace of this shape
    (synchronises the current stream): 0 if every call went through."""
    N, H = hidden.shape
    ws = workspace_for(N, H, weight.shape[0], chunk_rows, hidden.device)
    return L.lmhead_get_status(ws)


def _mask(keep):
    if keep is None:
        return None
    if keep.dtype == torch.bool:
        return keep.view(torch.uint8)
    return keep


class _HiddenToLogprobs(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, weight, targets, keep, return_entropy, entropy_requires_grad,
                chunk_rows, main_grad):
        N, H = hidden.shape
        V = weight.shape[0]
        dev = hidden.device
        ws = workspace_for(N, H, V, chunk_rows, dev)
        lp = torch.empty(N, dtype=torch.float32, device=dev)
        lse = torch.empty(N, dtype=torch.float32, device=dev)
        ent = torch.empty(N, dtype=torch.float32, device=dev) if return_entropy else None
        L.lmhead_fwd(hidden, weight, targets, keep, return_entropy, lp, ent, lse, ws, chunk_rows)
        ctx.save_for_backward(hidden, weight, targets, keep, lse,
                              ent if entropy_requires_grad else None)
        ctx.entropy_requires_grad = entropy_requires_grad
        ctx.chunk_rows = chunk_rows
        ctx.main_grad = main_grad
        ctx.weight_dtype = weight.dtype
        if ent is None:
            return lp
        if not entropy_requires_grad:
            ctx.mark_non_differentiable(ent)
        return lp, ent

    @staticmethod
    def backward(ctx, *grads):
        hidden, weight, targets, keep, lse, ent = ctx.saved_tensors
        N, H = hidden.shape
        V = weight.shape[0]
        g_lp = grads[0]
        g_lp = (torch.zeros(N, dtype=torch.float32, device=hidden.device) if g_lp is None
                else g_lp.contiguous())
        g_ent = None
        if ctx.entropy_requires_grad and len(grads) > 1 and grads[1] is not None:
            g_ent = grads[1].contiguous()
        ws = workspace_for(N, H, V, ctx.chunk_rows, hidden.device)
        dhidden = torch.empty_like(hidden)
        main = ctx.main_grad
        dW = main if main is not None else torch.empty(V, H, dtype=torch.float32,
                                                       device=hidden.device)
        L.lmhead_bwd(hidden, weight, targets, keep, lse, ent if g_ent is not None else None,
                     g_lp, g_ent, dhidden, dW, main is not None, ws, ctx.chunk_rows)
        dweight = None if main is not None else dW.to(ctx.weight_dtype)
        return dhidden, dweight, None, None, None, None, None, None


def hidden_to_logprobs(hidden, weight, targets, keep_mask=None, return_entropy=False,
                       entropy_requires_grad=False, chunk_rows=0, main_grad=None):
    """Log-probability of each row's target under softmax(hidden @ weight.T).

    hidden    [N, H] bf16, contiguous, on the GPU
    weight    [V, H] bf16, contiguous (the LM head)
    targets   [N] int64: the token each row predicts (read on kept rows only,
              which must hold 0 <= target < V)
    keep_mask [N] bool or uint8, or None for every row kept
    return_entropy        also return the entropy of each row's distribution
    entropy_requires_grad the entropy is a loss term (its gradient flows back);
                          otherwise it is a metric without gradient
    chunk_rows            kept rows per chunk (0: the library's default)
    main_grad             optional fp32 [V, H] buffer that the weight
                          gradient is added to in place

    Returns logprob [N] fp32, or (logprob, entropy), with 0 on rows outside
    the keep mask.
    """
    if entropy_requires_grad and not return_entropy:
        raise ValueError("entropy_requires_grad needs return_entropy")
    if main_grad is not None and (main_grad.dtype != torch.float32 or
                                  main_grad.shape != weight.shape):
        raise TypeError("main_grad must be an fp32 tensor shaped like weight")
    return _HiddenToLogprobs.apply(hidden, weight, targets, _mask(keep_mask),
                                   bool(return_entropy), bool(entropy_requires_grad),
                                   int(chunk_rows), main_grad)
