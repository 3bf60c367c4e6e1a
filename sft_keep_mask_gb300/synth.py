"""Seeded synthetic inputs for the fused LM-head scoring path.

This module only draws random numbers and lays out packed sequences.  It holds
none of the scoring arithmetic (no shift, no compaction, no softmax), so both
the CUDA library's tests and the float64 oracle can take their inputs from it.

Workloads (seed = workload number):

1. ``tiny``          N=256, H=256, V=4096; keep ~ Bernoulli(0.5).
2. ``qwen3_4b``      N=16384, H=2560, V=151936, W scaled x4 (peaked rows);
                     two packed sequences of 8192, 40% prompt / 60% completion.
3. ``moe30b_rl``     N=65536, H=4096, V=151936; sequences of length
                     ~U[512, 8192] packed to exactly N, prompt fraction
                     ~U[0.3, 0.7] masked (55% of the rows kept in the seed-3
                     draw).
   ``moe30b_rl_half`` the same packed sequences with the prompt fraction
                     exactly 0.5 (the first half of every sequence masked):
                     half the rows kept (49.98%) whatever the seed.
4. ``entropy_bonus`` N=16384, H=4096, V=131072; 16 sequences of 1024 whose
                     last round(f * 1024) tokens are active, f a parameter.
5. ``long_context``  N=262144, H=5120, V=151936; alternating prompt spans
                     ~U[768, 12288] and completion spans ~U[256, 4096].

Every workload draws hidden ~ N(0, 1) and W ~ N(0, 1/H) (times ``w_scale``)
in bf16, targets ~ U[0, V), grad_logprob ~ N(0, 1) and grad_entropy either
~ N(0, 0.1), the constant -0.01, or absent (metric-only entropy).
"""

from __future__ import annotations

import dataclasses

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    seed: int
    N: int
    H: int
    V: int
    w_scale: float = 1.0
    mask: str = "bernoulli"          # bernoulli | two_seq | packed | suffix | alternating
    grad_entropy: str = "normal"     # normal | const | none
    want_entropy: bool = True
    prompt_frac: tuple = (0.3, 0.7)  # packed: bounds of the uniform prompt fraction


WORKLOADS = {
    "tiny": Workload("tiny", 1, 256, 256, 4096, 1.0, "bernoulli", "normal"),
    "qwen3_4b": Workload("qwen3_4b", 2, 16384, 2560, 151936, 4.0, "two_seq", "none"),
    "moe30b_rl": Workload("moe30b_rl", 3, 65536, 4096, 151936, 1.0, "packed", "const"),
    "moe30b_rl_half": Workload("moe30b_rl_half", 3, 65536, 4096, 151936, 1.0, "packed", "const",
                               prompt_frac=(0.5, 0.5)),
    "entropy_bonus": Workload("entropy_bonus", 4, 16384, 4096, 131072, 1.0, "suffix", "const"),
    "long_context": Workload("long_context", 5, 262144, 5120, 151936, 1.0, "alternating", "const"),
}


def workload(name: str, **overrides) -> Workload:
    """The named workload, optionally with fields replaced (e.g. a smaller N)."""
    return dataclasses.replace(WORKLOADS[name], **overrides)


def _spans(rng: np.random.Generator, w: Workload, active_frac: float):
    """Token-aligned loss mask (float32 0/1) and packed sequence lengths."""
    n = w.N
    mask = np.zeros(n, dtype=np.float32)
    lens = []
    if w.mask == "two_seq":
        half = n // 2
        for s in (0, half):
            length = half if s == 0 else n - half
            p = int(round(0.4 * length))
            mask[s + p:s + length] = 1.0
            lens.append(length)
    elif w.mask == "packed":
        pos = 0
        while pos < n:
            length = int(rng.integers(512, 8193))
            length = min(length, n - pos)
            frac = float(rng.uniform(*w.prompt_frac))
            p = int(round(frac * length))
            mask[pos + p:pos + length] = 1.0
            lens.append(length)
            pos += length
    elif w.mask == "suffix":
        seq = 1024
        for s in range(0, n, seq):
            length = min(seq, n - s)
            a = int(round(active_frac * length))
            mask[s + length - a:s + length] = 1.0
            lens.append(length)
    elif w.mask == "alternating":
        pos = 0
        seq_start = 0
        # one packed sequence per (prompt, completion) pair
        while pos < n:
            p = int(rng.integers(768, 12289))
            c = int(rng.integers(256, 4097))
            p = min(p, n - pos)
            c = min(c, n - pos - p)
            mask[pos + p:pos + p + c] = 1.0
            pos += p + c
            lens.append(pos - seq_start)
            seq_start = pos
    else:
        raise ValueError(f"workload {w.name} has no span layout")
    return mask, lens


def make_inputs(w: Workload, device="cpu", active_frac: float = 1.0,
                keep_all: bool = False, weight_seed=None):
    """Draw one batch of the workload.

    weight_seed: draw W from its own generator with this seed (data-parallel
    ranks share the weight and draw their batches from per-rank seeds);
    None draws it from the workload's generator, between hidden and targets.

    Returns a dict with
      hidden [N,H] bf16, weight [V,H] bf16, targets [N] int64,
      grad_logprob [N] f32, grad_entropy [N] f32 or None,
      and either ``keep`` [N] uint8 (Bernoulli workloads, or every row kept
      when ``keep_all``) or ``components`` (list of token-aligned [N] f32 loss
      masks) with ``seq_lens`` (packed sequence lengths).
    All tensors are on ``device``; draws on CUDA use a CUDA generator.
    """
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed)
    rng = np.random.default_rng(w.seed)
    hidden = torch.randn(w.N, w.H, generator=g, device=dev, dtype=torch.float32)
    hidden = hidden.to(torch.bfloat16)
    std = w.w_scale / float(np.sqrt(w.H))
    weight = torch.empty(w.V, w.H, device=dev, dtype=torch.bfloat16)
    gw = g
    if weight_seed is not None:
        gw = torch.Generator(device=dev)
        gw.manual_seed(weight_seed)
    rows = 8192
    for r in range(0, w.V, rows):
        blk = torch.randn(min(rows, w.V - r), w.H, generator=gw, device=dev,
                          dtype=torch.float32)
        weight[r:r + blk.shape[0]] = (blk * std).to(torch.bfloat16)
    targets = torch.randint(0, w.V, (w.N,), generator=g, device=dev, dtype=torch.int64)
    g_lp = torch.randn(w.N, generator=g, device=dev, dtype=torch.float32)
    if w.grad_entropy == "normal":
        g_ent = 0.1 * torch.randn(w.N, generator=g, device=dev, dtype=torch.float32)
    elif w.grad_entropy == "const":
        g_ent = torch.full((w.N,), -0.01, device=dev, dtype=torch.float32)
    else:
        g_ent = None
    out = dict(hidden=hidden, weight=weight, targets=targets,
               grad_logprob=g_lp, grad_entropy=g_ent)
    if keep_all:
        out["keep"] = torch.ones(w.N, dtype=torch.uint8, device=dev)
    elif w.mask == "bernoulli":
        u = torch.rand(w.N, generator=g, device=dev)
        out["keep"] = (u < 0.5).to(torch.uint8)
    else:
        mask, lens = _spans(rng, w, active_frac)
        out["components"] = [torch.from_numpy(mask).to(dev)]
        out["seq_lens"] = lens
    return out


def sample_rows(n_kept: int, count: int, seed: int):
    """``count`` distinct positions in [0, n_kept), sorted (a seeded draw)."""
    rng = np.random.default_rng(1000 + seed)
    count = min(count, n_kept)
    return np.sort(rng.choice(n_kept, size=count, replace=False))


def make_logits(N: int, V: int, seed: int, std: float = 2.0, dtype=torch.bfloat16,
                device="cpu", ld: int = 0):
    """Logits ~ N(0, std^2) of shape [N, V] (row stride ld >= V when given),
    targets ~ U[0, V), grad_logprob ~ N(0, 1) and grad_entropy ~ N(0, 0.1).
    The shape of twinkle pull request #283's measurements is N=16384,
    V=151936."""
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    width = max(ld, V)
    z = torch.empty(N, width, dtype=dtype, device=dev)
    rows = 2048
    for r in range(0, N, rows):
        blk = torch.randn(min(rows, N - r), width, generator=g, device=dev)
        z[r:r + blk.shape[0]] = (blk * std).to(dtype)
    targets = torch.randint(0, V, (N,), generator=g, device=dev, dtype=torch.int64)
    g_lp = torch.randn(N, generator=g, device=dev)
    g_ent = 0.1 * torch.randn(N, generator=g, device=dev)
    return dict(logits=z[:, :V], targets=targets, grad_logprob=g_lp, grad_entropy=g_ent)
