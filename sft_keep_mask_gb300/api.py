"""Convenience layer over the C ABI: allocates outputs and the workspace.

Every computation is one of the ``lmhead_*`` calls; this module only creates
torch tensors for their outputs and keeps one workspace per shape.
"""

from __future__ import annotations

import torch

from . import lmhead as L


class LMHeadScorer:
    """Fused LM-head scoring for fixed (N, H, V, chunk_rows)."""

    def __init__(self, N: int, H: int, V: int, chunk_rows: int = 0, device="cuda"):
        self.N, self.H, self.V = N, H, V
        self.chunk_rows = chunk_rows
        self.device = torch.device(device)
        nbytes = L.lmhead_workspace_size(N, H, V, True, chunk_rows)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)

    def keep_mask(self, loss_mask=None, ce_weight=None, kl_weight=None, seq_lens=None,
                  stream=None):
        """Keep mask after the next-token shift from token-aligned loss components."""
        lens = torch.as_tensor(seq_lens, dtype=torch.int64)
        offsets = torch.zeros(lens.numel() + 1, dtype=torch.int32)
        offsets[1:] = torch.cumsum(lens, 0).to(torch.int32)
        offsets = offsets.to(self.device)
        keep = torch.empty(self.N, dtype=torch.uint8, device=self.device)
        L.lmhead_build_keep_mask(loss_mask, ce_weight, kl_weight, offsets, keep, stream)
        return keep

    def compact(self, keep, targets, stream=None):
        idx = torch.empty(self.N, dtype=torch.int32, device=self.device)
        yc = torch.empty(self.N, dtype=torch.int32, device=self.device)
        nk = torch.empty(1, dtype=torch.int32, device=self.device)
        L.lmhead_compact(keep, targets, self.V, idx, yc, nk, self.workspace, stream)
        return idx, yc, nk

    def forward(self, hidden, weight, targets, keep=None, want_entropy=True, stream=None,
                out=None):
        if out is None:
            out = (torch.empty(self.N, dtype=torch.float32, device=self.device),
                   torch.empty(self.N, dtype=torch.float32, device=self.device)
                   if want_entropy else None,
                   torch.empty(self.N, dtype=torch.float32, device=self.device))
        lp, ent, lse = out
        L.lmhead_fwd(hidden, weight, targets, keep, want_entropy, lp, ent, lse, self.workspace,
                     self.chunk_rows, stream)
        return lp, ent, lse

    def backward(self, hidden, weight, targets, keep, lse, entropy, grad_logprob,
                 grad_entropy=None, dweight=None, accumulate=False, stream=None, dhidden=None):
        if dhidden is None:
            dhidden = torch.empty_like(hidden)
        if dweight is None:
            dweight = torch.empty(self.V, self.H, dtype=torch.float32, device=self.device)
        L.lmhead_bwd(hidden, weight, targets, keep, lse, entropy, grad_logprob, grad_entropy,
                     dhidden, dweight, accumulate, self.workspace, self.chunk_rows, stream)
        return dhidden, dweight

    def kept_rows(self):
        """Nk of the last call on this workspace, as a 1-element int32 CUDA
        tensor (read it after the call has completed; no host sync here)."""
        return L.lmhead_workspace_kept_rows(self.workspace)

    def status(self, stream=None) -> int:
        return L.lmhead_get_status(self.workspace, stream)
