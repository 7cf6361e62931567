"""Pins for the oracle's banded masks and its rows with no visible key.

"Understanding FlashAttention" (Attention) says masks are elementwise, independent of the scores,
and that causal masking is one kind among several; (What is left to the implementation) warns
that a row whose keys are all masked has max -inf.  The oracle reads masks as bottom-right
aligned bands (window_left, window_right) and gives a row with no visible key o = 0, L = -inf.
These tests pin that reading with closed forms, an independent tiled restatement, a 50-digit
brute force, and finite differences of the gradients.
"""

import math

import numpy as np
import pytest

import oracle


def _visible(i, j, Nq, Nk, wl, wr):
    # the band, as stated in the reading (bottom-right aligned; -1 = unbounded)
    c = i + Nk - Nq
    return (wr < 0 or j <= c + wr) and (wl < 0 or j >= c - wl)


BANDS = [(-1, -1), (-1, 0), (0, 0), (2, 0), (3, 1), (0, 2), (-1, 1), (1, -1)]


@pytest.mark.parametrize("Nq,Nk", [(5, 5), (3, 7), (7, 3)])
def test_single_key_window_picks_the_diagonal_value(Nq, Nk):
    # (0, 0): row i sees exactly key i + Nk - Nq, so o_i = v_{i+off} and L_i = scale q_i.k_{i+off};
    # rows whose diagonal key does not exist see nothing: o = 0, L = -inf.
    rng = np.random.default_rng(40)
    d, scale = 4, 0.6
    q = rng.standard_normal((1, 1, Nq, d))
    k, v = (rng.standard_normal((1, 1, Nk, d)) for _ in range(2))
    o, lse = oracle.attention(q, k, v, window=(0, 0), scale=scale)
    off = Nk - Nq
    for i in range(Nq):
        j = i + off
        if 0 <= j < Nk:
            np.testing.assert_array_equal(o[0, 0, i], v[0, 0, j])
            assert math.isclose(lse[0, 0, i], scale * float(q[0, 0, i] @ k[0, 0, j]), rel_tol=1e-14, abs_tol=1e-15)
        else:
            assert np.all(o[0, 0, i] == 0.0) and lse[0, 0, i] == -np.inf


def test_causal_with_more_queries_than_keys_empties_the_top_rows():
    rng = np.random.default_rng(41)
    Nq, Nk, d = 6, 4, 3
    q = rng.standard_normal((1, 1, Nq, d))
    k, v = (rng.standard_normal((1, 1, Nk, d)) for _ in range(2))
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.5)
    assert np.all(o[0, 0, :2] == 0.0) and np.all(lse[0, 0, :2] == -np.inf)
    np.testing.assert_array_equal(o[0, 0, 2], v[0, 0, 0])  # row 2 sees key 0 only
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse[0, 0, 2:]))


@pytest.mark.parametrize("band", BANDS)
def test_band_closed_form_log_weights(band):
    # scores ln(c_j), independent of the row: p_ij = c_j / sum_{visible j'} c_j'.  With v_j a one-hot
    # vector at a permuted position times (j + 1), O_i[perm j] = p_ij (j + 1) exactly.
    Nq, Nk, scale = 4, 7, 0.5
    wl, wr = band
    c = np.arange(1, Nk + 1, dtype=np.float64) * 1.25
    q = np.zeros((1, 1, Nq, Nk))
    q[..., 0] = 1.0
    k = np.zeros((1, 1, Nk, Nk))
    k[0, 0, :, 0] = np.log(c) / scale
    perm = np.roll(np.arange(Nk), 2)
    v = np.zeros((1, 1, Nk, Nk))
    for j in range(Nk):
        v[0, 0, j, perm[j]] = j + 1.0
    o, lse = oracle.attention(q, k, v, window=band, scale=scale)
    for i in range(Nq):
        vis = [j for j in range(Nk) if _visible(i, j, Nq, Nk, wl, wr)]
        expect = np.zeros(Nk)
        for j in vis:
            expect[perm[j]] = c[j] / c[vis].sum() * (j + 1)
        np.testing.assert_allclose(o[0, 0, i], expect, rtol=1e-13, atol=1e-15)
        if vis:
            assert math.isclose(lse[0, 0, i], math.log(c[vis].sum()), rel_tol=1e-14)
        else:
            assert lse[0, 0, i] == -np.inf


def test_none_and_causal_bands_are_the_named_masks():
    rng = np.random.default_rng(42)
    q, k, v = (rng.standard_normal((2, 2, 9, 5)) for _ in range(3))
    for causal, band in ((False, (-1, -1)), (True, (-1, 0))):
        a = oracle.attention(q, k, v, causal=causal, scale=0.4)
        b = oracle.attention(q, k, v, window=band, scale=0.4)
        np.testing.assert_array_equal(a[0], b[0])
        np.testing.assert_array_equal(a[1], b[1])


@pytest.mark.parametrize("w", [4, 32, 128])
def test_symmetric_band_equals_tiled_local_window(w):
    # The tiled FlashAttention-2 restatement in test_oracle_pins keeps |i - j| < w/2; for Nq == Nk
    # that is the band (w/2 - 1, w/2 - 1).
    from test_oracle_pins import _tiled_forward
    rng = np.random.default_rng(43)
    n, d = 256, 16
    Q, K, V = (rng.standard_normal((n, d)) for _ in range(3))
    o, lse = oracle.attention(Q[None, None], K[None, None], V[None, None], window=(w // 2 - 1, w // 2 - 1),
                              scale=0.25)
    Ot, Lt = _tiled_forward(Q, K, V, 0.25, 64, 64, window=w)
    np.testing.assert_allclose(o[0, 0], Ot, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse[0, 0], Lt, rtol=0, atol=1e-13)


def test_bands_match_50_digit_brute_force():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(44)
    for (Nq, Nk, d) in [(4, 6, 3), (6, 4, 2), (5, 5, 2)]:
        q, k, v = (rng.standard_normal((1, 1, n, d)) * 2 for n in (Nq, Nk, Nk))
        for band in BANDS:
            wl, wr = band
            o, lse = oracle.attention(q, k, v, window=band, scale=0.7)
            for i in range(Nq):
                keys = [j for j in range(Nk) if _visible(i, j, Nq, Nk, wl, wr)]
                if not keys:
                    assert np.all(o[0, 0, i] == 0.0) and lse[0, 0, i] == -np.inf
                    continue
                xs = [mpmath.mpf(0.7) * mpmath.fsum(mpmath.mpf(q[0, 0, i, t]) * mpmath.mpf(k[0, 0, j, t])
                                                    for t in range(d)) for j in keys]
                es = [mpmath.e ** x for x in xs]
                z = mpmath.fsum(es)
                for t in range(d):
                    exact = mpmath.fsum(e * mpmath.mpf(v[0, 0, j, t]) for e, j in zip(es, keys)) / z
                    assert abs(o[0, 0, i, t] - float(exact)) <= 1e-14 * max(1.0, abs(float(exact)))
                assert abs(lse[0, 0, i] - float(mpmath.log(z))) <= 1e-14 * max(1.0, abs(float(mpmath.log(z))))


def test_band_gradients_match_50_digit_central_difference():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    h = mpmath.mpf("1e-22")
    rng = np.random.default_rng(45)

    def f(q, k, v, g, scale, Nq, Nk, wl, wr):
        total = mpmath.mpf(0)
        for i in range(Nq):
            keys = [j for j in range(Nk) if _visible(i, j, Nq, Nk, wl, wr)]
            if not keys:
                continue
            xs = [scale * mpmath.fsum(q[i][t] * k[j][t] for t in range(len(q[0]))) for j in keys]
            mx = max(xs)
            es = [mpmath.e ** (x - mx) for x in xs]
            z = mpmath.fsum(es)
            for t in range(len(q[0])):
                total += mpmath.fsum(e * v[j][t] for e, j in zip(es, keys)) / z * g[i][t]
        return total

    for (Nq, Nk, d, band) in [(3, 4, 2, (1, 0)), (4, 3, 2, (-1, 0)), (3, 3, 2, (0, 1))]:
        wl, wr = band
        q, k, v, g = (rng.standard_normal((1, 1, n, d)) for n in (Nq, Nk, Nk, Nq))
        scale = 0.6
        grads = oracle.attention_backward(q, k, v, g, window=band, scale=scale)
        mats = [[[mpmath.mpf(float(x)) for x in row] for row in a[0, 0]] for a in (q, k, v, g)]
        for which, grad in enumerate(grads):
            for r in range(len(mats[which])):
                for t in range(d):
                    plus = [[list(row) for row in m] for m in mats]
                    minus = [[list(row) for row in m] for m in mats]
                    plus[which][r][t] += h
                    minus[which][r][t] -= h
                    num = (f(*plus, mpmath.mpf(scale), Nq, Nk, wl, wr) - f(*minus, mpmath.mpf(scale), Nq, Nk, wl, wr)) / (2 * h)
                    assert abs(grad[0, 0, r, t] - float(num)) <= 1e-13 * max(1.0, abs(float(num))), (band, which, r, t)
        # rows with no visible key have zero dQ
        for i in range(Nq):
            if not any(_visible(i, j, Nq, Nk, wl, wr) for j in range(Nk)):
                assert np.all(grads[0][0, 0, i] == 0.0)
