"""Pins of the C float64 oracle (oracle/lmhead_oracle_c.c), no GPU needed.

It must agree with the numpy oracle -- an independent statement of the same
definition, itself pinned by brute force, closed forms and finite
differences in test_oracle.py -- to rounding (1e-12 relative), and meet
closed forms of its own:
  * W = 0: every logit is 0, so logprob = -log V, entropy = log V, lse =
    log V, dhidden = 0 and dW[v, :] = sum_r g_lp,r (1[v = y_r] - 1/V) h_r
    (the entropy term vanishes: log p_v + entropy = 0 for uniform p);
  * V = 1: logprob = entropy = 0, lse = z_0, and no gradient at all;
  * a target outside [0, V) is refused.
"""

import math

import numpy as np
import pytest

from oracle import lmhead_oracle as O
from oracle import lmhead_oracle_c as C


def _case(seed, R, H, V, scale=0.5):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((R, H))
    W = scale * rng.standard_normal((V, H))
    y = rng.integers(0, V, R)
    g_lp = rng.standard_normal(R)
    g_ent = 0.1 * rng.standard_normal(R)
    return h, W, y, g_lp, g_ent


def _close(a, b, tol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    assert np.abs(a - b).max() <= tol * max(1.0, np.abs(b).max())


@pytest.mark.parametrize("R,H,V", [(1, 8, 2), (5, 16, 129), (13, 40, 700), (4, 3, 1000)])
@pytest.mark.parametrize("entropy_grad", [True, False])
def test_agrees_with_the_numpy_oracle(R, H, V, entropy_grad):
    h, W, y, g_lp, g_ent = _case(R * 1000 + V, R, H, V)
    ge = g_ent if entropy_grad else None
    got = C.score_rows(h, W, y, g_lp, ge)
    want = O.score_rows(h, W, y, g_lp, ge)
    for a, b in zip(got, want):
        _close(a, b)


def test_forward_only_leaves_no_gradient():
    h, W, y, _, _ = _case(3, 6, 16, 50)
    lp, ent, lse, dh, dW = C.score_rows(h, W, y)
    assert dh is None and dW is None
    _close(lp, O.score_rows(h, W, y)[0])


def test_zero_weight_closed_form():
    R, H, V = 9, 12, 37
    h, W, y, g_lp, g_ent = _case(4, R, H, V)
    W[:] = 0.0
    lp, ent, lse, dh, dW = C.score_rows(h, W, y, g_lp, g_ent)
    _close(lp, np.full(R, -math.log(V)), 1e-14)
    _close(ent, np.full(R, math.log(V)), 1e-14)
    _close(lse, np.full(R, math.log(V)), 1e-14)
    assert np.abs(dh).max() == 0.0
    onehot = np.zeros((R, V))
    onehot[np.arange(R), y] = 1.0
    want = ((onehot - 1.0 / V) * g_lp[:, None]).T @ h
    _close(dW, want, 1e-13)


def test_single_token_vocabulary():
    h, W, y, g_lp, g_ent = _case(5, 4, 10, 1)
    lp, ent, lse, dh, dW = C.score_rows(h, W, y, g_lp, g_ent)
    assert np.abs(lp).max() == 0.0 and np.abs(ent).max() == 0.0
    _close(lse, h @ W[0], 1e-14)
    assert np.abs(dh).max() == 0.0 and np.abs(dW).max() == 0.0


def test_out_of_range_target_is_refused():
    h, W, y, g_lp, g_ent = _case(6, 3, 8, 20)
    y[1] = 20
    with pytest.raises(ValueError):
        C.score_rows(h, W, y, g_lp, g_ent)


def test_threads_reported():
    assert C.threads() >= 1
