"""Float64 CPU oracle for fused LM-head scoring with a keep mask.

TEST INFRASTRUCTURE ONLY.  Nothing in the product imports this module: only
``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / reference
arm of ``bench.py`` may call it.  It shares no code, table or constant with the
CUDA library and imports nothing from it.

It is the plain definition of what the fused path computes, written out in
float64 with the full ``[Nk, V]`` logits materialised.  The bf16 inputs are
upcast exactly (every bf16 value is an exact float64).

Sources (web pages; cited by title and section):

* [P1] prime-rl pull request #3326, "Don't compute the logprobs and their
  gradients for tokens no loss component reads" -- maintainer comment on where
  the FLOPs go (the ``[N,4096] @ [4096,151936]`` vocab matmul), and the
  "Overview" of the change: keep only positions that the RL loss mask, the CE
  weights or the ref-KL weights read after the next-token shift; compact ->
  chunked logprob/entropy -> expand back; skipped positions get zero logprobs
  and entropy.
* [P2] SkyRL pull request #2374, "feat(megatron): fuse LM-head entropy for RL"
  -- "How it works" (one projection gives the selected-token log-prob and the
  entropy; metric-only entropy adds no gradient work; entropy-loss mode keeps
  the entropy derivative) and the gemini-code-assist review (entropy is
  ``-(p * log p).sum(-1)`` over the vocabulary; the backward reuses the saved
  forward entropy).
* [P3] twinkle pull request #283, "Fix three memory defects in the Megatron
  path", section "1. selective_log_softmax pins one full-vocab copy per row"
  -- float32 results for bf16 input, softmax recomputed in backward.

Readings taken where the pages are silent (each also listed in the design
notes of the repository):

* The keep mask handed to the scoring functions is aligned to hidden rows:
  row ``i`` predicts token ``i+1``.  ``build_keep_mask`` derives it from the
  per-token loss components (row i is kept iff some component is non-zero at
  token i+1 of the same packed sequence; the last row of each sequence is
  never kept).
* ``keep is None`` keeps every row.
* Targets on kept rows must lie in ``[0, V)``; targets on skipped rows are
  never read.
* Skipped rows: logprob = entropy = lse = 0, hidden gradient 0, and no
  contribution to the weight gradient.
* Natural logarithms; temperature 1, no bias, no soft-cap.
* With ``g_ent is None`` (metric-only entropy) the entropy term is absent from
  the logit gradient.

Also the scoring of logits that already exist ([P3] section 1,
``selective_log_softmax``): the same log-prob / entropy / lse definitions and
their logit gradient, applied to a given ``[N, V]`` logit matrix.

Parity status: every function here is pinned by ``tests/test_oracle.py``
(closed forms, invariants, brute force on tiny inputs, central finite
differences).  No function is "parity unpinned".
"""

from __future__ import annotations

import numpy as np


class OracleTargetError(ValueError):
    """A kept row carries a target outside ``[0, V)``."""


def build_keep_mask(components, seq_lens):
    """Rows whose next token is read by some loss component.

    [P1] "Overview": the vocab matmul runs only on positions that the RL
    loss_mask, the CE weights or the ref-KL weights use, after the usual
    next-token shift.  Row ``i`` of the hidden states scores token ``i+1``,
    so row ``i`` is kept iff ``components[c][i+1] != 0`` for some ``c`` and
    ``i+1`` lies in the same packed sequence as ``i``.

    components : list of 1-D arrays of length N (token-aligned weights or 0/1
                 masks; any non-zero value counts).
    seq_lens   : lengths of the packed sequences, summing to N.
    returns    : uint8 array [N] of 0/1.
    """
    comps = [np.asarray(c) for c in components]
    n = int(comps[0].shape[0])
    if int(np.sum(seq_lens)) != n:
        raise ValueError("sequence lengths must sum to N")
    read = np.zeros(n, dtype=bool)
    for c in comps:
        read |= c != 0
    keep = np.zeros(n, dtype=np.uint8)
    start = 0
    for length in seq_lens:
        length = int(length)
        for i in range(start, start + length - 1):
            keep[i] = 1 if read[i + 1] else 0
        start += length
    return keep


def compact(keep, targets, V):
    """Stable compaction of the kept rows.

    [P1] "Overview": compact -> score -> expand.  The order of the kept rows
    is their order in the packed batch (ascending row index).

    returns idx (int32 [Nk], ascending), Nk (int), targets_c (int32 [Nk]).
    Raises OracleTargetError if a kept row's target is outside [0, V).
    """
    targets = np.asarray(targets).astype(np.int64)
    n = targets.shape[0]
    if keep is None:
        keep = np.ones(n, dtype=np.uint8)
    keep = np.asarray(keep)
    idx = [i for i in range(n) if keep[i] != 0]
    idx = np.asarray(idx, dtype=np.int32)
    yc = targets[idx] if idx.size else np.zeros(0, np.int64)
    if idx.size and (yc.min() < 0 or yc.max() >= V):
        raise OracleTargetError("target outside [0, V) on a kept row")
    return idx, int(idx.size), yc.astype(np.int32)


def _kept_logits(h, W, idx):
    """z = h[idx] @ W^T in float64: the materialised [Nk, V] logits.

    [P1] maintainer comment: hidden -> logits is the ``[N, H] @ [H, V]``
    vocab matmul; here only the kept rows are projected.
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    return h[idx] @ W.T


def _log_softmax(z):
    """log p = z - lse with lse = max z + log sum exp(z - max z), per row."""
    zmax = z.max(axis=1, keepdims=True)
    lse = zmax[:, 0] + np.log(np.exp(z - zmax).sum(axis=1))
    return z - lse[:, None], lse


def forward(h, W, targets, keep=None, want_entropy=True):
    """Selected-token log-prob, entropy and lse of every row.

    [P2] "How it works": one projection yields the selected-token log-prob
    and the entropy; the gemini-code-assist review gives the entropy as
    ``-(p * log p)`` summed over the vocabulary.  [P3] section 1: results in
    float (here float64).  [P1] "Overview": skipped rows get zeros.

    h [N, H], W [V, H] (any float dtype; upcast to float64), targets [N] int,
    keep [N] 0/1 or None.  Returns (logprob, entropy, lse), float64 [N] each;
    entropy is all zeros when ``want_entropy`` is false.
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    n = h.shape[0]
    V = W.shape[0]
    idx, nk, yc = compact(keep, targets, V)
    lp = np.zeros(n)
    ent = np.zeros(n)
    lse = np.zeros(n)
    if nk == 0:
        return lp, ent, lse
    z = _kept_logits(h, W, idx)
    logp, l = _log_softmax(z)
    lp[idx] = logp[np.arange(nk), yc]
    lse[idx] = l
    if want_entropy:
        p = np.exp(logp)
        ent[idx] = -(p * logp).sum(axis=1)
    return lp, ent, lse


def backward(h, W, targets, keep, g_lp, g_ent=None):
    """Gradients of L = sum_i g_lp[i] * logprob[i] + g_ent[i] * entropy[i].

    With p = softmax(z) and y the target of the row:
      d logprob / d z_v = 1[v = y] - p_v
      d entropy / d z_v = -p_v (log p_v + entropy)
    so dz_v = g_lp (1[v=y] - p_v) - g_ent p_v (log p_v + entropy)
    ([P2] "How it works": entropy-loss mode keeps the entropy derivative in the
    fused backward; metric-only entropy adds none, i.e. ``g_ent is None``).
    Then dh = dz @ W and dW = dz^T @ h over the kept rows ([P2] greptile and
    cursor reviews: the hidden gradient is ``d_logits @ W``; weight gradients
    per weight row).  Skipped rows get dh = 0 and add nothing to dW ([P1]).

    Returns (dh float64 [N, H], dW float64 [V, H]).
    """
    h = np.asarray(h, dtype=np.float64)
    W = np.asarray(W, dtype=np.float64)
    n, H = h.shape
    V = W.shape[0]
    idx, nk, yc = compact(keep, targets, V)
    dh = np.zeros((n, H))
    dW = np.zeros((V, H))
    if nk == 0:
        return dh, dW
    z = _kept_logits(h, W, idx)
    logp, _ = _log_softmax(z)
    p = np.exp(logp)
    onehot = np.zeros_like(p)
    onehot[np.arange(nk), yc] = 1.0
    g1 = np.asarray(g_lp, dtype=np.float64)[idx]
    dz = g1[:, None] * (onehot - p)
    if g_ent is not None:
        g2 = np.asarray(g_ent, dtype=np.float64)[idx]
        ent = -(p * logp).sum(axis=1)
        dz = dz - g2[:, None] * p * (logp + ent[:, None])
    dh[idx] = dz @ W
    dW = dz.T @ h[idx]
    return dh, dW


def score_rows(h_rows, W, targets_rows, g_lp_rows=None, g_ent_rows=None,
               want_entropy=True):
    """Forward (and, given g_lp_rows, backward) for a set of kept rows.

    The same definitions as ``forward``/``backward`` applied to rows that are
    all kept; used on sampled rows of a full-size batch, where each row's
    outputs and hidden gradient depend on that row alone.  Returns
    (logprob, entropy, lse, dh or None, dW contribution or None).
    """
    h_rows = np.asarray(h_rows, dtype=np.float64)
    r = h_rows.shape[0]
    keep = np.ones(r, dtype=np.uint8)
    lp, ent, lse = forward(h_rows, W, targets_rows, keep, want_entropy)
    if g_lp_rows is None:
        return lp, ent, lse, None, None
    dh, dW = backward(h_rows, W, targets_rows, keep, g_lp_rows, g_ent_rows)
    return lp, ent, lse, dh, dW


def selective_log_softmax(z, targets, keep=None, want_entropy=True):
    """Log-prob of the target, entropy and lse of rows of given logits.

    [P3] section 1 ("selective_log_softmax pins one full-vocab copy per row"):
    log_softmax of each row computed in float (here float64), the target's
    log-prob gathered, and the entropy -(p * log p) summed over the
    vocabulary ([P2] gemini-code-assist review).  Rows with keep == 0 get 0.

    z [N, V] (any float dtype; upcast to float64), targets [N] int,
    keep [N] 0/1 or None.  Returns (logprob, entropy, lse), float64 [N].
    """
    z = np.asarray(z, dtype=np.float64)
    n, V = z.shape
    idx, nk, yc = compact(keep, targets, V)
    lp = np.zeros(n)
    ent = np.zeros(n)
    lse = np.zeros(n)
    if nk == 0:
        return lp, ent, lse
    logp, l = _log_softmax(z[idx])
    lp[idx] = logp[np.arange(nk), yc]
    lse[idx] = l
    if want_entropy:
        ent[idx] = -(np.exp(logp) * logp).sum(axis=1)
    return lp, ent, lse


def selective_log_softmax_backward(z, targets, keep, g_lp, g_ent=None):
    """Gradient of sum_i g_lp[i] logprob[i] + g_ent[i] entropy[i] w.r.t. z.

    The same logit gradient as ``backward``:
    dz_v = g_lp (1[v=y] - p_v) - g_ent p_v (log p_v + entropy); rows with
    keep == 0 get 0.  Returns dz, float64 [N, V].
    """
    z = np.asarray(z, dtype=np.float64)
    n, V = z.shape
    idx, nk, yc = compact(keep, targets, V)
    dz = np.zeros((n, V))
    if nk == 0:
        return dz
    logp, _ = _log_softmax(z[idx])
    p = np.exp(logp)
    onehot = np.zeros_like(p)
    onehot[np.arange(nk), yc] = 1.0
    g1 = np.asarray(g_lp, dtype=np.float64)[idx]
    d = g1[:, None] * (onehot - p)
    if g_ent is not None:
        g2 = np.asarray(g_ent, dtype=np.float64)[idx]
        ent = -(p * logp).sum(axis=1)
        d = d - g2[:, None] * p * (logp + ent[:, None])
    dz[idx] = d
    return dz


def shard_partials(h, W_shard, v_begin, targets, keep=None):
    """Per-row partial reductions over one vocabulary shard.

    [P2] gemini-code-assist review: with the LM head split over the vocabulary
    (tensor parallel), each rank reduces its own logits and a single exchange
    after the chunk loop completes the log-softmax and the entropy.  For the
    shard W_shard = W[v_begin : v_begin + Vs] and each kept row:
      m = max_v z_v,  s = sum_v exp(z_v - m),
      u = sum_v exp(z_v - m) (z_v - m),
      t = z_y if v_begin <= y < v_begin + Vs else -inf.
    Skipped rows get (-inf, 0, 0, -inf).  Returns float64 [N, 4].
    """
    h = np.asarray(h, dtype=np.float64)
    W_shard = np.asarray(W_shard, dtype=np.float64)
    n = h.shape[0]
    Vs = W_shard.shape[0]
    targets = np.asarray(targets).astype(np.int64)
    if keep is None:
        keep = np.ones(n, dtype=np.uint8)
    out = np.zeros((n, 4))
    out[:, 0] = -np.inf
    out[:, 3] = -np.inf
    idx = np.flatnonzero(np.asarray(keep))
    if idx.size == 0:
        return out
    z = h[idx] @ W_shard.T
    m = z.max(axis=1)
    e = np.exp(z - m[:, None])
    out[idx, 0] = m
    out[idx, 1] = e.sum(axis=1)
    out[idx, 2] = (e * (z - m[:, None])).sum(axis=1)
    local = targets[idx] - v_begin
    inside = (local >= 0) & (local < Vs)
    rows = np.flatnonzero(inside)
    out[idx[rows], 3] = z[rows, local[rows]]
    return out


def merge_shard_partials(partials, keep=None):
    """Log-prob, entropy and lse of every row from the shards' partials.

    With M = max_r m_r, S = sum_r s_r e^(m_r - M),
    U = sum_r e^(m_r - M) (u_r + s_r (m_r - M)):
      lse = M + log S, logprob = t - lse (t from the shard holding y),
      entropy = log S - U / S.
    partials float [R, N, 4]; skipped rows (keep == 0) get 0.
    """
    P = np.asarray(partials, dtype=np.float64)
    R, n, _ = P.shape
    if keep is None:
        keep = np.ones(n, dtype=np.uint8)
    lp = np.zeros(n)
    ent = np.zeros(n)
    lse = np.zeros(n)
    for i in np.flatnonzero(np.asarray(keep)):
        M = P[:, i, 0].max()
        w = np.exp(P[:, i, 0] - M)
        S = (P[:, i, 1] * w).sum()
        U = (w * (P[:, i, 2] + P[:, i, 1] * (P[:, i, 0] - M))).sum()
        t = P[:, i, 3].max()
        lse[i] = M + np.log(S)
        lp[i] = t - lse[i]
        ent[i] = np.log(S) - U / S
    return lp, ent, lse
