"""Pins of the float64 oracle to facts fixed outside the oracle itself.

Each test checks the oracle against one of: a hand-worked fixture in
``tests/golden/``, a closed form, an invariant of the mathematics, a library
routine the definition reduces to, brute force on a tiny input, or central
finite differences of the forward.  A plausible slip in the oracle (a dropped
entropy term, a wrong sign, an off-by-one in the shift, a transposed operand)
fails at least one of them.
"""

import math
import os

import numpy as np
import pytest

from oracle import lmhead_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _problem(seed, N, H, V, scale=1.0, keep_p=0.6):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((N, H))
    W = rng.standard_normal((V, H)) * scale / math.sqrt(H)
    y = rng.integers(0, V, N)
    keep = (rng.random(N) < keep_p).astype(np.uint8)
    g_lp = rng.standard_normal(N)
    g_ent = 0.3 * rng.standard_normal(N)
    return h, W, y, keep, g_lp, g_ent


def _read_golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                out[k.strip()] = v.split()
            else:
                parts = line.split()
                out[(parts[0], parts[1])] = float(parts[2])
    return out


# ---------------------------------------------------------------- keep mask

def test_keep_mask_golden_fixture():
    g = _read_golden("keep_mask_shift.txt")
    lens = [int(x) for x in g["seq_lens"]]
    comps = [np.array([float(x) for x in g[k]]) for k in ("loss_mask", "ce_weight", "kl_weight")]
    want = np.array([int(x) for x in g["keep"]], dtype=np.uint8)
    got = O.build_keep_mask(comps, lens)
    np.testing.assert_array_equal(got, want)


def test_keep_mask_last_row_of_each_sequence_is_zero():
    rng = np.random.default_rng(3)
    lens = [7, 1, 12, 5]
    n = sum(lens)
    comps = [np.ones(n), (rng.random(n) < 0.5).astype(float)]
    keep = O.build_keep_mask(comps, lens)
    ends = np.cumsum(lens) - 1
    assert (keep[ends] == 0).all()
    others = np.setdiff1d(np.arange(n), ends)
    assert (keep[others] == 1).all()  # component 0 reads every token


def test_keep_mask_is_union_of_components_shifted():
    rng = np.random.default_rng(4)
    lens = [40, 25, 35]
    n = sum(lens)
    a = (rng.random(n) < 0.3).astype(float)
    b = (rng.random(n) < 0.3) * rng.standard_normal(n)  # non-binary weights
    keep = O.build_keep_mask([a, b], lens)
    union = O.build_keep_mask([np.logical_or(a != 0, b != 0).astype(float)], lens)
    np.testing.assert_array_equal(keep, union)
    # a single sequence reduces to a shift by one: keep[i] = read[i+1]
    single = O.build_keep_mask([a], [n])
    np.testing.assert_array_equal(single[:-1], (a[1:] != 0).astype(np.uint8))
    assert single[-1] == 0


# --------------------------------------------------------------- compaction

def test_compaction_matches_flatnonzero():
    rng = np.random.default_rng(5)
    for n in (0, 1, 17, 1000):
        keep = (rng.random(n) < 0.4).astype(np.uint8)
        y = rng.integers(0, 50, n)
        idx, nk, yc = O.compact(keep, y, 50)
        np.testing.assert_array_equal(idx, np.flatnonzero(keep))
        assert nk == int(keep.sum())
        np.testing.assert_array_equal(yc, y[np.flatnonzero(keep)])


def test_compaction_none_keeps_everything():
    y = np.arange(9) % 4
    idx, nk, yc = O.compact(None, y, 4)
    assert nk == 9
    np.testing.assert_array_equal(idx, np.arange(9))


def test_target_out_of_range_on_kept_row_raises():
    keep = np.array([1, 0, 1], dtype=np.uint8)
    with pytest.raises(O.OracleTargetError):
        O.compact(keep, np.array([0, 1, 7]), 5)
    with pytest.raises(O.OracleTargetError):
        O.compact(keep, np.array([-1, 1, 2]), 5)
    # an ignore index on a skipped row is never read
    idx, nk, _ = O.compact(keep, np.array([0, -100, 4]), 5)
    assert nk == 2


# ------------------------------------------------------------------ forward

def _brute_forward_row(hrow, W, y):
    """Pure-Python loops: logits, max, log-sum-exp, entropy."""
    V, H = len(W), len(hrow)
    z = [sum(hrow[k] * W[v][k] for k in range(H)) for v in range(V)]
    m = max(z)
    s = sum(math.exp(zv - m) for zv in z)
    lse = m + math.log(s)
    ent = 0.0
    for zv in z:
        p = math.exp(zv - lse)
        ent -= p * (zv - lse)
    return z[y] - lse, ent, lse


def test_forward_matches_brute_force_tiny():
    h, W, y, keep, _, _ = _problem(11, 6, 5, 9, scale=2.0)
    lp, ent, lse = O.forward(h, W, y, keep)
    for i in range(6):
        if keep[i]:
            b = _brute_forward_row(list(h[i]), [list(r) for r in W], int(y[i]))
            assert abs(lp[i] - b[0]) < 1e-12
            assert abs(ent[i] - b[1]) < 1e-12
            assert abs(lse[i] - b[2]) < 1e-12
        else:
            assert lp[i] == 0.0 and ent[i] == 0.0 and lse[i] == 0.0


def test_forward_two_way_golden():
    g = _read_golden("closed_forms.txt")
    h = np.array([[1.0]])
    W = np.array([[0.0], [math.log(3.0)]])
    lp, ent, lse = O.forward(h, W, np.array([0]), None)
    assert abs(lp[0] - g[("two_way", "logprob")]) < 1e-14
    assert abs(ent[0] - g[("two_way", "entropy")]) < 1e-14
    assert abs(lse[0] - g[("two_way", "lse")]) < 1e-14


@pytest.mark.parametrize("V", [4096, 151936])
def test_forward_zero_weight_is_uniform(V):
    g = _read_golden("closed_forms.txt")
    rng = np.random.default_rng(1)
    H = 8
    h = rng.standard_normal((3, H))
    W = np.zeros((V, H))
    y = np.array([0, V // 2, V - 1])
    lp, ent, lse = O.forward(h, W, y, None)
    want = g[(f"uniform_{V}", "entropy")]
    np.testing.assert_allclose(ent, want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse, want, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lp, -want, rtol=0, atol=1e-12)


def test_forward_binary_vocab_closed_form():
    rng = np.random.default_rng(2)
    h = rng.standard_normal((50, 4))
    W = rng.standard_normal((2, 4))
    y = rng.integers(0, 2, 50)
    lp, ent, _ = O.forward(h, W, y, None)
    z = h @ W.T
    d = z[np.arange(50), 1 - y] - z[np.arange(50), y]
    softplus = np.logaddexp(0.0, d)
    np.testing.assert_allclose(lp, -softplus, rtol=0, atol=1e-12)
    q = 1.0 / (1.0 + np.exp(-d))  # probability of the other token
    hb = -(q * np.log(q) + (1 - q) * np.log1p(-q))
    np.testing.assert_allclose(ent, hb, rtol=0, atol=1e-12)


def test_forward_single_token_vocab():
    rng = np.random.default_rng(3)
    h = rng.standard_normal((4, 6))
    W = rng.standard_normal((1, 6))
    lp, ent, lse = O.forward(h, W, np.zeros(4, int), None)
    np.testing.assert_allclose(lp, 0.0, atol=1e-15)
    np.testing.assert_allclose(ent, 0.0, atol=1e-15)
    np.testing.assert_allclose(lse, (h @ W.T)[:, 0], atol=1e-12)


def test_forward_invariants_random():
    h, W, y, keep, _, _ = _problem(12, 200, 16, 300, scale=3.0)
    lp, ent, lse = O.forward(h, W, y, keep)
    k = keep.astype(bool)
    assert (lp[k] <= 0).all()
    assert (ent[k] >= 0).all() and (ent[k] <= math.log(300) + 1e-12).all()
    # log-sum-exp is bounded by max z and max z + log V
    zmax = (h @ W.T).max(axis=1)
    assert (lse[k] >= zmax[k] - 1e-12).all()
    assert (lse[k] <= zmax[k] + math.log(300) + 1e-12).all()


def test_forward_uniform_logit_shift_invariance():
    h, W, y, keep, _, _ = _problem(13, 40, 12, 70)
    c = np.random.default_rng(0).standard_normal(12)
    lp0, ent0, lse0 = O.forward(h, W, y, keep)
    lp1, ent1, lse1 = O.forward(h, W + c[None, :], y, keep)
    np.testing.assert_allclose(lp1, lp0, atol=1e-11)
    np.testing.assert_allclose(ent1, ent0, atol=1e-11)
    np.testing.assert_allclose(lse1, lse0 + (h @ c) * keep, atol=1e-11)


def test_forward_vocab_permutation_invariance():
    h, W, y, keep, _, _ = _problem(14, 30, 10, 64)
    perm = np.random.default_rng(1).permutation(64)
    inv = np.argsort(perm)
    lp0, ent0, lse0 = O.forward(h, W, y, keep)
    lp1, ent1, lse1 = O.forward(h, W[perm], inv[y], keep)
    np.testing.assert_allclose(lp1, lp0, atol=1e-12)
    np.testing.assert_allclose(ent1, ent0, atol=1e-12)
    np.testing.assert_allclose(lse1, lse0, atol=1e-12)


def test_forward_peaked_rows():
    # z[i, y_i] exceeds every other logit of row i by at least 39:
    # p_y -> 1, so logprob -> 0 and entropy -> 0 (bounded by (V-1) e^-39 terms)
    rng = np.random.default_rng(15)
    n, V = 20, 50
    h = np.eye(n)
    W = 0.1 * rng.standard_normal((V, n))
    y = rng.integers(0, V, n)
    W[y, np.arange(n)] += 40.0
    lp, ent, _ = O.forward(h, W, y, None)
    assert (lp <= 0).all() and (lp > -V * math.exp(-39.0)).all()
    assert (ent >= 0).all() and (ent < V * 41 * math.exp(-39.0)).all()


def test_forward_row_independence_and_zero_fill():
    h, W, y, keep, _, _ = _problem(16, 60, 8, 40)
    lp0, ent0, lse0 = O.forward(h, W, y, keep)
    flip = keep.copy()
    flip[::3] = 1 - flip[::3]
    lp1, ent1, lse1 = O.forward(h, W, y, flip)
    both = (keep == 1) & (flip == 1)
    np.testing.assert_array_equal(lp0[both], lp1[both])
    np.testing.assert_array_equal(ent0[both], ent1[both])
    off = keep == 0
    assert (lp0[off] == 0).all() and (ent0[off] == 0).all() and (lse0[off] == 0).all()


def test_forward_without_entropy():
    h, W, y, keep, _, _ = _problem(17, 30, 8, 40)
    lp0, ent0, lse0 = O.forward(h, W, y, keep, want_entropy=True)
    lp1, ent1, lse1 = O.forward(h, W, y, keep, want_entropy=False)
    np.testing.assert_array_equal(lp0, lp1)
    np.testing.assert_array_equal(lse0, lse1)
    assert (ent1 == 0).all()


def test_forward_empty_keep():
    h, W, y, _, _, _ = _problem(18, 5, 4, 7)
    lp, ent, lse = O.forward(h, W, y, np.zeros(5, np.uint8))
    assert not lp.any() and not ent.any() and not lse.any()


# ----------------------------------------------------------------- backward

def _loss(h, W, y, keep, g_lp, g_ent):
    lp, ent, _ = O.forward(h, W, y, keep)
    out = float(np.sum(g_lp * lp))
    if g_ent is not None:
        out += float(np.sum(g_ent * ent))
    return out


@pytest.mark.parametrize("with_entropy", [True, False])
def test_backward_central_finite_differences(with_entropy):
    h, W, y, keep, g_lp, g_ent = _problem(21, 4, 8, 16, scale=2.0, keep_p=0.7)
    keep[:] = [1, 0, 1, 1]
    ge = g_ent if with_entropy else None
    dh, dW = O.backward(h, W, y, keep, g_lp, ge)
    eps = 1e-5
    num_h = np.zeros_like(h)
    for i in range(h.shape[0]):
        for k in range(h.shape[1]):
            hp, hm = h.copy(), h.copy()
            hp[i, k] += eps
            hm[i, k] -= eps
            num_h[i, k] = (_loss(hp, W, y, keep, g_lp, ge) - _loss(hm, W, y, keep, g_lp, ge)) / (2 * eps)
    num_W = np.zeros_like(W)
    for v in range(W.shape[0]):
        for k in range(W.shape[1]):
            Wp, Wm = W.copy(), W.copy()
            Wp[v, k] += eps
            Wm[v, k] -= eps
            num_W[v, k] = (_loss(h, Wp, y, keep, g_lp, ge) - _loss(h, Wm, y, keep, g_lp, ge)) / (2 * eps)
    assert np.linalg.norm(dh - num_h) <= 1e-6 * np.linalg.norm(num_h)
    assert np.linalg.norm(dW - num_W) <= 1e-6 * np.linalg.norm(num_W)
    assert (dh[1] == 0).all()


def test_backward_weight_grad_columns_sum_to_zero():
    h, W, y, keep, g_lp, g_ent = _problem(22, 50, 12, 80)
    _, dW = O.backward(h, W, y, keep, g_lp, g_ent)
    scale = np.abs(dW).max()
    np.testing.assert_allclose(dW.sum(axis=0), 0.0, atol=1e-12 * max(scale, 1) * 80)


def test_backward_hidden_grad_unchanged_by_common_weight_shift():
    h, W, y, keep, g_lp, g_ent = _problem(23, 30, 10, 40)
    c = np.random.default_rng(2).standard_normal(10)
    dh0, _ = O.backward(h, W, y, keep, g_lp, g_ent)
    dh1, _ = O.backward(h, W + c[None, :], y, keep, g_lp, g_ent)
    np.testing.assert_allclose(dh1, dh0, atol=1e-11)


def test_backward_zero_weight_closed_form():
    h, W, y, keep, g_lp, g_ent = _problem(24, 25, 6, 30)
    W = np.zeros_like(W)
    dh, dW = O.backward(h, W, y, keep, g_lp, g_ent)
    assert not dh.any()
    V = 30
    want = np.zeros((V, 6))
    for i in range(25):
        if keep[i]:
            dz = -g_lp[i] / V * np.ones(V)
            dz[y[i]] += g_lp[i]
            want += np.outer(dz, h[i])
    np.testing.assert_allclose(dW, want, atol=1e-12)


def test_backward_skipping_equals_zeroed_gradients():
    h, W, y, keep, g_lp, g_ent = _problem(25, 40, 8, 33)
    dh, dW = O.backward(h, W, y, keep, g_lp, g_ent)
    k = keep.astype(float)
    dh_all, dW_all = O.backward(h, W, y, None, g_lp * k, g_ent * k)
    np.testing.assert_allclose(dW, dW_all, atol=1e-12)
    np.testing.assert_allclose(dh, dh_all, atol=1e-12)
    assert (dh[keep == 0] == 0).all()


def test_backward_metric_only_entropy_equals_zero_entropy_grad():
    h, W, y, keep, g_lp, _ = _problem(26, 20, 8, 30)
    a = O.backward(h, W, y, keep, g_lp, None)
    b = O.backward(h, W, y, keep, g_lp, np.zeros(20))
    np.testing.assert_allclose(a[0], b[0], atol=1e-15)
    np.testing.assert_allclose(a[1], b[1], atol=1e-15)


def test_score_rows_matches_full_batch():
    h, W, y, keep, g_lp, g_ent = _problem(27, 30, 8, 20)
    lp, ent, lse = O.forward(h, W, y, keep)
    dh, _ = O.backward(h, W, y, keep, g_lp, g_ent)
    rows = np.flatnonzero(keep)[:5]
    r = O.score_rows(h[rows], W, y[rows], g_lp[rows], g_ent[rows])
    np.testing.assert_allclose(r[0], lp[rows], atol=1e-13)
    np.testing.assert_allclose(r[1], ent[rows], atol=1e-13)
    np.testing.assert_allclose(r[2], lse[rows], atol=1e-13)
    np.testing.assert_allclose(r[3], dh[rows], atol=1e-13)


# ------------------------------------------- scoring of existing logits

def test_sls_brute_force_and_zero_fill():
    rng = np.random.default_rng(40)
    z = 3.0 * rng.standard_normal((7, 11))
    y = rng.integers(0, 11, 7)
    keep = np.array([1, 0, 1, 1, 0, 1, 1], np.uint8)
    lp, ent, lse = O.selective_log_softmax(z, y, keep)
    for i in range(7):
        if not keep[i]:
            assert lp[i] == 0 and ent[i] == 0 and lse[i] == 0
            continue
        row = list(z[i])
        m = max(row)
        l = m + math.log(sum(math.exp(v - m) for v in row))
        e = -sum(math.exp(v - l) * (v - l) for v in row)
        assert abs(lp[i] - (row[y[i]] - l)) < 1e-12
        assert abs(ent[i] - e) < 1e-12 and abs(lse[i] - l) < 1e-12


def test_sls_closed_forms():
    g = _read_golden("closed_forms.txt")
    V = 4096
    lp, ent, lse = O.selective_log_softmax(np.full((2, V), 1.5), np.array([3, 9]))
    np.testing.assert_allclose(ent, g[("uniform_4096", "entropy")], atol=1e-12)
    np.testing.assert_allclose(lp, -g[("uniform_4096", "entropy")], atol=1e-12)
    np.testing.assert_allclose(lse, 1.5 + g[("uniform_4096", "entropy")], atol=1e-12)
    lp, ent, lse = O.selective_log_softmax(np.array([[0.0, math.log(3.0)]]), np.array([0]))
    assert abs(lp[0] - g[("two_way", "logprob")]) < 1e-14
    assert abs(ent[0] - g[("two_way", "entropy")]) < 1e-14


def test_sls_row_shift_invariance():
    rng = np.random.default_rng(41)
    z = rng.standard_normal((20, 50))
    y = rng.integers(0, 50, 20)
    c = 100 * rng.standard_normal(20)
    a = O.selective_log_softmax(z, y)
    b = O.selective_log_softmax(z + c[:, None], y)
    np.testing.assert_allclose(b[0], a[0], atol=1e-10)
    np.testing.assert_allclose(b[1], a[1], atol=1e-10)
    np.testing.assert_allclose(b[2], a[2] + c, atol=1e-10)


def test_sls_agrees_with_the_fused_forward_and_backward():
    h, W, y, keep, g_lp, g_ent = _problem(42, 30, 12, 40)
    z = h @ W.T
    for a, b in zip(O.selective_log_softmax(z, y, keep), O.forward(h, W, y, keep)):
        np.testing.assert_allclose(a, b, atol=1e-12)
    dz = O.selective_log_softmax_backward(z, y, keep, g_lp, g_ent)
    dh, dW = O.backward(h, W, y, keep, g_lp, g_ent)
    np.testing.assert_allclose(dz @ W, dh, atol=1e-11)
    np.testing.assert_allclose(dz.T @ h, dW, atol=1e-11)


@pytest.mark.parametrize("with_entropy", [True, False])
def test_sls_backward_finite_differences(with_entropy):
    rng = np.random.default_rng(43)
    z = 2.0 * rng.standard_normal((3, 9))
    y = rng.integers(0, 9, 3)
    keep = np.array([1, 1, 0], np.uint8)
    g1 = rng.standard_normal(3)
    g2 = 0.5 * rng.standard_normal(3) if with_entropy else None

    def loss(zz):
        lp, ent, _ = O.selective_log_softmax(zz, y, keep)
        return float(np.sum(g1 * lp) + (np.sum(g2 * ent) if g2 is not None else 0.0))

    dz = O.selective_log_softmax_backward(z, y, keep, g1, g2)
    num = np.zeros_like(z)
    eps = 1e-5
    for i in range(3):
        for v in range(9):
            zp, zm = z.copy(), z.copy()
            zp[i, v] += eps
            zm[i, v] -= eps
            num[i, v] = (loss(zp) - loss(zm)) / (2 * eps)
    assert np.linalg.norm(dz - num) <= 1e-7 * max(np.linalg.norm(num), 1.0)
    np.testing.assert_allclose(dz.sum(axis=1), 0.0, atol=1e-12)
    assert not dz[2].any()


# --------------------------------------------- vocabulary-parallel shards

def test_shard_merge_equals_full_forward():
    # splitting the vocabulary into shards and merging their partials gives
    # the forward of the whole vocabulary (any split, uneven shards)
    h, W, y, keep, _, _ = _problem(60, 40, 16, 101, scale=3.0)
    full = O.forward(h, W, y, keep)
    for bounds in ([0, 101], [0, 50, 101], [0, 7, 8, 64, 101]):
        parts = np.stack([O.shard_partials(h, W[a:b], a, y, keep)
                          for a, b in zip(bounds[:-1], bounds[1:])])
        got = O.merge_shard_partials(parts, keep)
        for g, f in zip(got, full):
            np.testing.assert_allclose(g, f, atol=1e-12)


def test_shard_partials_closed_form():
    # a shard of W = 0 has z = 0: m = 0, s = Vs, u = 0; t = 0 iff y inside
    h = np.ones((3, 4))
    y = np.array([2, 9, 15])
    P = O.shard_partials(h, np.zeros((6, 4)), 8, y)
    np.testing.assert_allclose(P[:, 0], 0.0)
    np.testing.assert_allclose(P[:, 1], 6.0)
    np.testing.assert_allclose(P[:, 2], 0.0)
    assert P[0, 3] == -np.inf and P[1, 3] == 0.0 and P[2, 3] == -np.inf


def test_shard_backward_sums_to_full_backward():
    # dz of a shard uses the global lse / entropy; the hidden gradient is the
    # sum over shards of dz_shard @ W_shard, dW is the concatenation
    h, W, y, keep, g_lp, g_ent = _problem(61, 30, 12, 77)
    dh, dW = O.backward(h, W, y, keep, g_lp, g_ent)
    z = h @ W.T
    dz = O.selective_log_softmax_backward(z, y, keep, g_lp, g_ent)
    dh_sum = np.zeros_like(dh)
    for a, b in ((0, 30), (30, 77)):
        dh_sum += dz[:, a:b] @ W[a:b]
        np.testing.assert_allclose(dz[:, a:b].T @ h, dW[a:b], atol=1e-12)
    np.testing.assert_allclose(dh_sum, dh, atol=1e-12)
