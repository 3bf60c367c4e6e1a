"""Convenience layer over the C ABI: allocates outputs and the workspace.

Every computation is one of the ``lmhead_*`` calls; this module only creates
torch tensors for their outputs and keeps one workspace per shape.
"""

from __future__ import annotations

import torch

from . import lmhead as L


class LMHeadScorer:
    """Fused LM-head scoring for one head (H, V, chunk_rows) and batches of up
    to N rows.

    The workspace is sized for N rows and serves any batch of at most N rows
    (the library lays it out from each call's row count, and a smaller batch
    needs no more bytes), so batch sizes that change from step to step reuse
    it; outputs are sized by each call's batch.
    """

    def __init__(self, N: int, H: int, V: int, chunk_rows: int = 0, device="cuda",
                 blocksparse: bool = False):
        """blocksparse: score the active 256-row tiles in place instead of
        compacting the kept rows (lmhead_fwd_blocksparse / _bwd_blocksparse)."""
        self.N, self.H, self.V = N, H, V
        self.blocksparse = blocksparse
        self.chunk_rows = chunk_rows
        self.device = torch.device(device)
        nbytes = L.lmhead_workspace_size(N, H, V, True, chunk_rows)
        self.workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=self.device)

    def _rows(self, n: int) -> int:
        if n > self.N:
            raise ValueError(f"batch of {n} rows exceeds this scorer's capacity of {self.N}")
        return n

    def keep_mask(self, loss_mask=None, ce_weight=None, kl_weight=None, seq_lens=None,
                  stream=None):
        """Keep mask after the next-token shift from token-aligned loss components."""
        comps = [c for c in (loss_mask, ce_weight, kl_weight) if c is not None]
        n = self._rows(comps[0].numel() if comps else self.N)
        lens = torch.as_tensor(seq_lens, dtype=torch.int64)
        offsets = torch.zeros(lens.numel() + 1, dtype=torch.int32)
        offsets[1:] = torch.cumsum(lens, 0).to(torch.int32)
        offsets = offsets.to(self.device)
        keep = torch.empty(n, dtype=torch.uint8, device=self.device)
        L.lmhead_build_keep_mask(loss_mask, ce_weight, kl_weight, offsets, keep, stream)
        return keep

    def compact(self, keep, targets, stream=None):
        n = self._rows(targets.numel())
        idx = torch.empty(n, dtype=torch.int32, device=self.device)
        yc = torch.empty(n, dtype=torch.int32, device=self.device)
        nk = torch.empty(1, dtype=torch.int32, device=self.device)
        L.lmhead_compact(keep, targets, self.V, idx, yc, nk, self.workspace, stream)
        return idx, yc, nk

    def forward(self, hidden, weight, targets, keep=None, want_entropy=True, stream=None,
                out=None):
        n = self._rows(hidden.shape[0])
        if out is None:
            out = (torch.empty(n, dtype=torch.float32, device=self.device),
                   torch.empty(n, dtype=torch.float32, device=self.device)
                   if want_entropy else None,
                   torch.empty(n, dtype=torch.float32, device=self.device))
        lp, ent, lse = out
        fwd = L.lmhead_fwd_blocksparse if self.blocksparse else L.lmhead_fwd
        fwd(hidden, weight, targets, keep, want_entropy, lp, ent, lse, self.workspace,
            self.chunk_rows, stream)
        return lp, ent, lse

    def backward(self, hidden, weight, targets, keep, lse, entropy, grad_logprob,
                 grad_entropy=None, dweight=None, accumulate=False, stream=None, dhidden=None):
        self._rows(hidden.shape[0])
        if dhidden is None:
            dhidden = torch.empty_like(hidden)
        if dweight is None:
            dweight = torch.empty(self.V, self.H, dtype=torch.float32, device=self.device)
        bwd = L.lmhead_bwd_blocksparse if self.blocksparse else L.lmhead_bwd
        bwd(hidden, weight, targets, keep, lse, entropy, grad_logprob, grad_entropy, dhidden,
            dweight, accumulate, self.workspace, self.chunk_rows, stream)
        return dhidden, dweight

    def kept_rows(self):
        """Nk of the last call on this workspace, as a 1-element int32 CUDA
        tensor (read it after the call has completed; no host sync here)."""
        return L.lmhead_workspace_kept_rows(self.workspace)

    def status(self, stream=None) -> int:
        return L.lmhead_get_status(self.workspace, stream)


class StepPipeline:
    """Runs steps whose inputs live in pinned host memory, keeping the GPU busy
    across steps: the host-to-device copy of step i+1's inputs overlaps the
    computation of step i, and the host reads step i's results while step
    i+1 is already queued.

    step_fn(*device_inputs) enqueues one step on the current stream (e.g. the
    keep mask, lmhead_fwd and lmhead_bwd calls); result_fn() returns the
    device tensors to read back after every step (e.g. logprob and entropy).
    Two sets of device input buffers and two sets of pinned result buffers
    alternate; a side stream does the copies, ordered with events.
    """

    def __init__(self, step_fn, result_fn, host_inputs, device="cuda"):
        self.device = torch.device(device)
        self.step_fn = step_fn
        self.result_fn = result_fn
        self.copy_stream = torch.cuda.Stream(self.device)
        self.bufs = [[None if t is None else torch.empty_like(t, device=self.device)
                      for t in host_inputs] for _ in range(2)]
        self.ready = [torch.cuda.Event() for _ in range(2)]
        self.free = [torch.cuda.Event() for _ in range(2)]
        self.done = [torch.cuda.Event() for _ in range(2)]
        for e in self.free:
            e.record(torch.cuda.current_stream(self.device))
        self.host_results = None

    def _prefetch(self, slot, host_inputs):
        with torch.cuda.stream(self.copy_stream):
            self.copy_stream.wait_event(self.free[slot])
            for d, h in zip(self.bufs[slot], host_inputs):
                if d is not None:
                    d.copy_(h, non_blocking=True)
            self.ready[slot].record(self.copy_stream)

    def run(self, batches):
        """Runs one step per batch (a list of pinned host tensors each), reading
        every step's results back; returns the host copies of the last step's."""
        compute = torch.cuda.current_stream(self.device)
        if not batches:
            return None
        pending = None
        self._prefetch(0, batches[0])
        for i in range(len(batches)):
            slot = i % 2
            if i + 1 < len(batches):
                self._prefetch(1 - slot, batches[i + 1])
            compute.wait_event(self.ready[slot])
            self.step_fn(*self.bufs[slot])
            self.free[slot].record(compute)
            res = self.result_fn()
            if self.host_results is None:
                self.host_results = [[torch.empty(r.shape, dtype=r.dtype).pin_memory()
                                      for r in res] for _ in range(2)]
            for h, r in zip(self.host_results[slot], res):
                h.copy_(r, non_blocking=True)
            self.done[slot].record(compute)
            if pending is not None:
                pending.synchronize()  # step i-1's results are on the host
            pending = self.done[slot]
        pending.synchronize()
        return self.host_results[(len(batches) - 1) % 2]


def allreduce_weight_grad(dweight, group=None):
    """Data-parallel sum of the weight gradient over the ranks of `group`.

    Rows are independent for logprob, entropy and dhidden, so data-parallel
    ranks score their own batches; the weight gradient is the one exchange:
    one all-reduce after the backward (SkyRL pull request #2374, gemini review:
    a single reduction after the loop, not one per chunk).  This is the
    caller's collective (torch.distributed: NCCL between GPUs, gloo on CPU
    tensors), issued on the current stream; with one rank it does nothing.
    """
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(dweight, op=dist.ReduceOp.SUM, group=group)
    return dweight
