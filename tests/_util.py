"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the float64 oracle on the same seeded inputs, and compare."""

import numpy as np
import torch

from oracle import lmhead_oracle as O

ATOL_ROW = 1e-3      # |d logprob|, |d entropy|, |d lse| (absolute)
RTOL_FRO = 1e-2      # relative Frobenius error of dhidden and dW


def seq_offsets(lens, device="cuda"):
    off = np.zeros(len(lens) + 1, dtype=np.int32)
    off[1:] = np.cumsum(lens)
    return torch.from_numpy(off).to(device)


def to64(t):
    return t.detach().float().cpu().double().numpy()


def gpu_keep(scorer, inp):
    """Keep mask of an input dict: given directly or built on the GPU."""
    if "keep" in inp:
        return inp["keep"]
    comps = inp["components"]
    return scorer.keep_mask(comps[0], comps[1] if len(comps) > 1 else None,
                            comps[2] if len(comps) > 2 else None, seq_lens=inp["seq_lens"])


def oracle_keep(inp):
    if "keep" in inp:
        return inp["keep"].cpu().numpy().astype(np.uint8)
    return O.build_keep_mask([c.cpu().numpy() for c in inp["components"]], inp["seq_lens"])


def frob_rel(got, want):
    num = np.linalg.norm((got - want).ravel())
    den = np.linalg.norm(want.ravel())
    return num / den if den > 0 else num


def assert_rows_close(got, want, what):
    err = np.abs(got - want).max() if got.size else 0.0
    assert err <= ATOL_ROW, f"{what}: max abs error {err:.3e} > {ATOL_ROW}"


def assert_frob_close(got, want, what):
    err = frob_rel(got, want)
    assert err <= RTOL_FRO, f"{what}: relative Frobenius error {err:.3e} > {RTOL_FRO}"
