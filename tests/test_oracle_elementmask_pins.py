"""Pins for the oracle's element mask.

"Understanding FlashAttention" (Attention) says a mask is elementwise and independent of the scores,
causal masking being one kind among several; (What is left to the implementation) warns that a row
whose keys are all masked has max -inf.  The oracle takes a boolean mask broadcastable to
[B, H, Nq, Nk] (true = the key may be seen), intersected with the band, excludes masked keys
outright (weight exactly 0), and gives a row with no visible key o = 0 and L = -inf.  These tests
pin that with closed forms, a 50-digit brute force and finite differences of the gradients.
"""

import math

import numpy as np
import pytest

import oracle


def _band_visible(i, j, Nq, Nk, wl, wr):
    c = i + Nk - Nq
    return (wr < 0 or j <= c + wr) and (wl < 0 or j >= c - wl)


def test_permutation_mask_picks_one_value_per_row():
    # row i sees key pi(i) only: o_i = v_pi(i) exactly and L_i = scale q_i . k_pi(i)
    rng = np.random.default_rng(60)
    Nq = Nk = 9
    d, scale = 5, 0.4
    q = rng.standard_normal((1, 1, Nq, d))
    k, v = (rng.standard_normal((1, 1, Nk, d)) for _ in range(2))
    pi = rng.permutation(Nk)
    mask = np.zeros((Nq, Nk), dtype=bool)
    mask[np.arange(Nq), pi] = True
    o, lse = oracle.attention(q, k, v, scale=scale, mask=mask)
    for i in range(Nq):
        np.testing.assert_array_equal(o[0, 0, i], v[0, 0, pi[i]])
        assert math.isclose(lse[0, 0, i], scale * float(q[0, 0, i] @ k[0, 0, pi[i]]), rel_tol=1e-14, abs_tol=1e-15)


def test_zero_scores_give_the_mean_of_the_visible_values():
    # q = 0: every visible key has score 0, so o_i is the mean of the visible values and
    # L_i = log(number of visible keys); rows with no visible key give o = 0, L = -inf
    rng = np.random.default_rng(61)
    B, H, Nq, Nk, d = 2, 3, 7, 11, 4
    q = np.zeros((B, H, Nq, d))
    k, v = (rng.standard_normal((B, H, Nk, d)) for _ in range(2))
    mask = rng.random((B, H, Nq, Nk)) < 0.4
    mask[0, 1, 3] = False  # one empty row
    o, lse = oracle.attention(q, k, v, scale=1.0, mask=mask)
    for b in range(B):
        for h in range(H):
            for i in range(Nq):
                vis = np.nonzero(mask[b, h, i])[0]
                if vis.size == 0:
                    assert np.all(o[b, h, i] == 0.0) and lse[b, h, i] == -np.inf
                    continue
                np.testing.assert_allclose(o[b, h, i], v[b, h, vis].mean(axis=0), rtol=0, atol=1e-14)
                assert math.isclose(lse[b, h, i], math.log(vis.size), rel_tol=0, abs_tol=1e-14)


@pytest.mark.parametrize("band", [(-1, -1), (-1, 0), (2, 1)])
def test_closed_form_log_weights_under_mask_and_band(band):
    # d = 1, q = 1, k_j = ln(c_j) / scale: scores ln(c_j) for every row, so p_ij = c_j m_ij / sum c m over
    # the keys both the mask and the band leave visible; v_j = e_j picks the weights out one by one
    rng = np.random.default_rng(62)
    Nq, Nk, scale = 6, 8, 0.5
    c = rng.uniform(0.2, 3.0, Nk)
    q = np.ones((1, 1, Nq, 1))
    k = (np.log(c) / scale).reshape(1, 1, Nk, 1)
    mask = rng.random((Nq, Nk)) < 0.6
    o_cols = []
    for t in range(Nk):
        v = np.zeros((1, 1, Nk, 1))
        v[0, 0, t, 0] = 1.0
        o, lse = oracle.attention(q, k, v, scale=scale, window=band, mask=mask)
        o_cols.append(o[0, 0, :, 0])
    P = np.stack(o_cols, axis=1)
    for i in range(Nq):
        vis = np.array([mask[i, j] and _band_visible(i, j, Nq, Nk, *band) for j in range(Nk)])
        if not vis.any():
            assert np.all(P[i] == 0.0) and lse[0, 0, i] == -np.inf
            continue
        w = np.where(vis, c, 0.0)
        np.testing.assert_allclose(P[i], w / w.sum(), rtol=1e-13, atol=1e-16)
        assert math.isclose(lse[0, 0, i], math.log(w.sum()), rel_tol=1e-13)


def test_all_true_mask_and_broadcast_forms():
    rng = np.random.default_rng(63)
    B, H, Nq, Nk, d = 2, 3, 5, 9, 4
    q, k, v = (rng.standard_normal((B, H, n, d)) for n in (Nq, Nk, Nk))
    o0, l0 = oracle.attention(q, k, v, causal=True)
    o1, l1 = oracle.attention(q, k, v, causal=True, mask=np.ones((Nq, Nk), dtype=bool))
    np.testing.assert_array_equal(o0, o1)
    np.testing.assert_array_equal(l0, l1)
    # one mask for every (b, h), one per batch entry shared by its heads, one per (b, h)
    m2 = rng.random((Nq, Nk)) < 0.5
    m3 = rng.random((B, 1, Nq, Nk)) < 0.5
    for m in (m2, m3):
        full = np.broadcast_to(m, (B, H, Nq, Nk)).copy()
        oa, la = oracle.attention(q, k, v, mask=m)
        ob, lb = oracle.attention(q, k, v, mask=full)
        np.testing.assert_array_equal(oa, ob)
        np.testing.assert_array_equal(la, lb)
    # the rows helper and the probabilities take the same mask
    rows = np.array([0, 7, 13, 29])
    o_r, l_r = oracle.attention_rows(q, k, v, rows, mask=m3)
    oa, la = oracle.attention(q, k, v, mask=m3)
    np.testing.assert_array_equal(o_r, oa.reshape(-1, d)[rows])
    np.testing.assert_array_equal(l_r, la.reshape(-1)[rows])
    p = oracle.attention_probs(q[1, 2], k[1, 2], mask=m3[1, 0])
    assert np.all(p[~m3[1, 0]] == 0.0)
    np.testing.assert_allclose(p @ v[1, 2], oa[1, 2], rtol=0, atol=1e-14)


def test_mask_is_not_ignored():
    # the negative control: the same call without the mask misses the closed form
    rng = np.random.default_rng(64)
    q = np.zeros((1, 1, 4, 2))
    k, v = (rng.standard_normal((1, 1, 6, 2)) for _ in range(2))
    mask = np.zeros((4, 6), dtype=bool)
    mask[:, :2] = True
    o, _ = oracle.attention(q, k, v, scale=1.0)
    assert np.abs(o[0, 0] - v[0, 0, :2].mean(axis=0)).max() > 1e-3


def test_element_masks_match_50_digit_brute_force():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(65)
    for (Nq, Nk, d, band) in [(4, 6, 3, (-1, -1)), (6, 4, 2, (-1, 0)), (5, 5, 2, (1, 1))]:
        q, k, v = (rng.standard_normal((1, 1, n, d)) * 2 for n in (Nq, Nk, Nk))
        mask = rng.random((Nq, Nk)) < 0.55
        mask[1] = False
        o, lse = oracle.attention(q, k, v, window=band, scale=0.7, mask=mask)
        for i in range(Nq):
            keys = [j for j in range(Nk) if mask[i, j] and _band_visible(i, j, Nq, Nk, *band)]
            if not keys:
                assert np.all(o[0, 0, i] == 0.0) and lse[0, 0, i] == -np.inf
                continue
            xs = [mpmath.mpf(0.7) * mpmath.fsum(mpmath.mpf(q[0, 0, i, t]) * mpmath.mpf(k[0, 0, j, t]) for t in range(d))
                  for j in keys]
            es = [mpmath.e ** x for x in xs]
            z = mpmath.fsum(es)
            for t in range(d):
                exact = mpmath.fsum(e * mpmath.mpf(v[0, 0, j, t]) for e, j in zip(es, keys)) / z
                assert abs(o[0, 0, i, t] - float(exact)) <= 1e-14 * max(1.0, abs(float(exact)))
            assert abs(lse[0, 0, i] - float(mpmath.log(z))) <= 1e-14 * max(1.0, abs(float(mpmath.log(z))))


def test_element_mask_gradients_match_50_digit_central_difference():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    h = mpmath.mpf("1e-22")
    rng = np.random.default_rng(66)
    Nq, Nk, d, scale = 3, 4, 2, 0.6
    mask = np.array([[1, 0, 1, 1], [0, 0, 0, 0], [0, 1, 1, 0]], dtype=bool)  # row 1 empty, key 0 seen once

    def f(q, k, v, g):
        total = mpmath.mpf(0)
        for i in range(Nq):
            keys = [j for j in range(Nk) if mask[i, j]]
            if not keys:
                continue
            xs = [mpmath.mpf(scale) * mpmath.fsum(q[i][t] * k[j][t] for t in range(d)) for j in keys]
            mx = max(xs)
            es = [mpmath.e ** (x - mx) for x in xs]
            z = mpmath.fsum(es)
            for t in range(d):
                total += mpmath.fsum(e * v[j][t] for e, j in zip(es, keys)) / z * g[i][t]
        return total

    q, k, v, g = (rng.standard_normal((1, 1, n, d)) for n in (Nq, Nk, Nk, Nq))
    grads = oracle.attention_backward(q, k, v, g, scale=scale, mask=mask)
    mats = [[[mpmath.mpf(float(x)) for x in row] for row in a[0, 0]] for a in (q, k, v, g)]
    for which, grad in enumerate(grads):
        for r in range(len(mats[which])):
            for t in range(d):
                plus = [[list(row) for row in m] for m in mats]
                minus = [[list(row) for row in m] for m in mats]
                plus[which][r][t] += h
                minus[which][r][t] -= h
                num = (f(*plus) - f(*minus)) / (2 * h)
                assert abs(grad[0, 0, r, t] - float(num)) <= 1e-13 * max(1.0, abs(float(num))), (which, r, t)
    assert np.all(grads[0][0, 0, 1] == 0.0)  # the empty row has dq = 0
    # a key nobody sees gets dk = dv = 0
    mask2 = mask.copy()
    mask2[:, 3] = False
    g2 = oracle.attention_backward(q, k, v, g, scale=scale, mask=mask2)
    assert np.all(g2[1][0, 0, 3] == 0.0) and np.all(g2[2][0, 0, 3] == 0.0)
