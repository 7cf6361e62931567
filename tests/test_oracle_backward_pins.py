"""Pins for the oracle's attention gradients ("Flash Attention: The Hidden Gem", Phase 2).

The oracle computes dQ, dK, dV from the softmax Jacobian.  None of these tests restates that
computation.  They check it against the derivative's own definition (a 50-digit central
difference of the scalar f = sum(O * G), and an fp64 one through the pinned forward), against
closed forms (one key, two keys, identical keys) and against invariants that follow from the
forward's symmetries.  A dropped scale, a wrong sign on D, a transposed dS or P, or a mask
slip in the backward fails at least one of them.
"""

import math

import numpy as np
import pytest

import oracle


def _f_mp(mpmath, q, k, v, g, scale, causal):
    """f = sum_i sum_t O_it G_it, O by the attention definition, in mpmath arithmetic."""
    Nq, d = len(q), len(q[0])
    Nk = len(k)
    total = mpmath.mpf(0)
    for i in range(Nq):
        keys = [j for j in range(Nk) if (not causal) or j <= i + Nk - Nq]
        xs = [scale * mpmath.fsum(q[i][t] * k[j][t] for t in range(d)) for j in keys]
        mx = max(xs)
        es = [mpmath.e ** (x - mx) for x in xs]
        z = mpmath.fsum(es)
        for t in range(d):
            o = mpmath.fsum(e * v[j][t] for e, j in zip(es, keys)) / z
            total += o * g[i][t]
    return total


def test_gradients_match_50_digit_central_difference():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    h = mpmath.mpf("1e-22")
    rng = np.random.default_rng(31)
    for (Nq, Nk, d, causal) in [(1, 1, 1, False), (2, 3, 2, False), (3, 3, 2, True), (2, 4, 3, True),
                                 (3, 2, 2, False)]:
        q, k, v, g = (rng.standard_normal((1, 1, n, d)) for n in (Nq, Nk, Nk, Nq))
        scale = 0.8 / math.sqrt(d)
        dq, dk, dv = oracle.attention_backward(q, k, v, g, causal=causal, scale=scale)
        mats = [[[mpmath.mpf(float(x)) for x in row] for row in a[0, 0]] for a in (q, k, v, g)]
        sc = mpmath.mpf(scale)
        for which, grad in ((0, dq), (1, dk), (2, dv)):
            rows = len(mats[which])
            for r in range(rows):
                for t in range(d):
                    plus = [[list(row) for row in m] for m in mats]
                    minus = [[list(row) for row in m] for m in mats]
                    plus[which][r][t] += h
                    minus[which][r][t] -= h
                    num = (_f_mp(mpmath, *plus[:3], plus[3], sc, causal)
                           - _f_mp(mpmath, *minus[:3], minus[3], sc, causal)) / (2 * h)
                    assert abs(grad[0, 0, r, t] - float(num)) <= 1e-13 * max(1.0, abs(float(num))), (
                        Nq, Nk, d, causal, which, r, t)


@pytest.mark.parametrize("causal", [False, True])
def test_gradients_match_fp64_central_difference_through_forward(causal):
    # The forward is pinned on its own; differentiating it numerically checks the backward at a
    # size with several heads and a ragged causal offset (Nq < Nk).
    rng = np.random.default_rng(32)
    B, H, Nq, Nk, d = 1, 2, 5, 7, 4
    q, k, v, g = (rng.standard_normal((B, H, n, d)) for n in (Nq, Nk, Nk, Nq))
    scale = 0.45
    dq, dk, dv = oracle.attention_backward(q, k, v, g, causal=causal, scale=scale)
    eps = 1e-6

    def f(qq, kk, vv):
        o, _ = oracle.attention(qq, kk, vv, causal=causal, scale=scale)
        return float(np.sum(o * g))

    for which, grad in ((0, dq), (1, dk), (2, dv)):
        base = [q, k, v]
        num = np.zeros_like(grad)
        for idx in np.ndindex(*grad.shape):
            p = [a.copy() for a in base]
            m = [a.copy() for a in base]
            p[which][idx] += eps
            m[which][idx] -= eps
            num[idx] = (f(*p) - f(*m)) / (2 * eps)
        np.testing.assert_allclose(grad, num, rtol=0, atol=2e-8)


def test_one_key_closed_form():
    # A single key gets weight 1 whatever the scores: O_i = v, so dQ = dK = 0 and dV = sum_i G_i.
    rng = np.random.default_rng(33)
    q, g = (rng.standard_normal((2, 3, 6, 5)) for _ in range(2))
    k, v = (rng.standard_normal((2, 3, 1, 5)) for _ in range(2))
    dq, dk, dv = oracle.attention_backward(q, k, v, g, scale=0.7)
    assert np.all(dq == 0) and np.all(dk == 0)
    np.testing.assert_allclose(dv[:, :, 0], g.sum(axis=2), rtol=0, atol=1e-13)


def test_two_keys_closed_form_sigmoid():
    # With two keys the row's weight on key 0 is p = sigmoid(scale * q.(k0 - k1)), and
    # f_i = G_i.(p v0 + (1-p) v1).  Hence, with c_i = p(1-p) G_i.(v0 - v1):
    #   dq_i = scale c_i (k0 - k1),  dk0 = scale sum_i c_i q_i = -dk1,
    #   dv0 = sum_i p_i G_i,  dv1 = sum_i (1 - p_i) G_i.
    rng = np.random.default_rng(34)
    Nq, d, scale = 4, 3, 0.9
    q, g = (rng.standard_normal((1, 1, Nq, d)) for _ in range(2))
    k, v = (rng.standard_normal((1, 1, 2, d)) for _ in range(2))
    dq, dk, dv = oracle.attention_backward(q, k, v, g, scale=scale)
    Q, G, K, V = q[0, 0], g[0, 0], k[0, 0], v[0, 0]
    p = 1.0 / (1.0 + np.exp(-scale * (Q @ (K[0] - K[1]))))
    c = p * (1 - p) * (G @ (V[0] - V[1]))
    np.testing.assert_allclose(dq[0, 0], scale * c[:, None] * (K[0] - K[1])[None, :], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk[0, 0, 0], scale * (c @ Q), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk[0, 0, 1], -scale * (c @ Q), rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv[0, 0, 0], p @ G, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv[0, 0, 1], (1 - p) @ G, rtol=0, atol=1e-14)


def test_identical_keys_give_zero_dq():
    # Equal keys give every query the uniform distribution whatever q is: dQ = 0.
    rng = np.random.default_rng(35)
    q, g = (rng.standard_normal((1, 2, 5, 4)) for _ in range(2))
    k = np.broadcast_to(rng.standard_normal((1, 2, 1, 4)), (1, 2, 6, 4)).copy()
    v = rng.standard_normal((1, 2, 6, 4))
    dq, _, dv = oracle.attention_backward(q, k, v, g, scale=0.6)
    np.testing.assert_allclose(dq, 0.0, rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, np.broadcast_to(g.sum(axis=2, keepdims=True) / 6, dv.shape), atol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_invariants_from_forward_symmetries(causal):
    rng = np.random.default_rng(36)
    B, H, Nq, Nk, d = 2, 2, 9, 13, 6
    q, g = (rng.standard_normal((B, H, Nq, d)) for _ in range(2))
    k, v = (rng.standard_normal((B, H, Nk, d)) for _ in range(2))
    scale = 0.37
    dq, dk, dv = oracle.attention_backward(q, k, v, g, causal=causal, scale=scale)
    # Adding one vector to every key adds a per-row constant to the visible scores: P, and so f,
    # do not move.  The derivative along that direction is sum_j dK_j = 0.
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, rtol=0, atol=1e-12)
    # Scaling Q by a and K by 1/a leaves every score unchanged: sum Q.dQ = sum K.dK per head.
    np.testing.assert_allclose(np.einsum("bhnd,bhnd->bh", q, dq), np.einsum("bhnd,bhnd->bh", k, dk),
                               rtol=0, atol=1e-12)
    # Every row of P sums to 1, so sum_j dV_j = sum_i G_i; f is linear in V, so dV ignores V.
    np.testing.assert_allclose(dv.sum(axis=2), g.sum(axis=2), rtol=0, atol=1e-12)
    _, _, dv2 = oracle.attention_backward(q, k, 3 * v + 1, g, causal=causal, scale=scale)
    np.testing.assert_allclose(dv2, dv, rtol=0, atol=1e-13)
    # f is linear in G: the gradients for 2G are twice those for G.
    dq2, dk2, dv3 = oracle.attention_backward(q, k, v, 2 * g, causal=causal, scale=scale)
    np.testing.assert_allclose(dq2, 2 * dq, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk2, 2 * dk, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv3, 2 * dv, rtol=0, atol=1e-13)


def test_causal_last_key_sees_only_the_last_row():
    # With Nq = Nk and the causal mask, key N-1 is visible to row N-1 alone, where its weight is
    # p = exp(x_last) / sum: dV_{N-1} = p G_{N-1}.
    rng = np.random.default_rng(37)
    n, d, scale = 6, 3, 0.5
    q, k, v, g = (rng.standard_normal((1, 1, n, d)) for _ in range(4))
    _, _, dv = oracle.attention_backward(q, k, v, g, causal=True, scale=scale)
    x = scale * (k[0, 0] @ q[0, 0, n - 1])
    p_last = np.exp(x[-1] - x.max()) / np.exp(x - x.max()).sum()
    np.testing.assert_allclose(dv[0, 0, n - 1], p_last * g[0, 0, n - 1], rtol=0, atol=1e-14)
    # Key 0 is visible to every row: its dV gathers all of them, so it differs from row 0's share.
    assert np.max(np.abs(dv[0, 0, 0] - g[0, 0, 0])) > 1e-3


def test_pins_reject_plausible_backward_mistakes():
    """Outputs with a dropped scale or a flipped D sign (dS = P(dP + D)) are separated from the
    oracle's by the closed form and the invariants above."""
    rng = np.random.default_rng(38)
    Nq, d, scale = 4, 3, 0.9
    q, g = (rng.standard_normal((1, 1, Nq, d)) for _ in range(2))
    k, v = (rng.standard_normal((1, 1, 2, d)) for _ in range(2))
    dq, dk, dv = oracle.attention_backward(q, k, v, g, scale=scale)
    Q, G, K, V = q[0, 0], g[0, 0], k[0, 0], v[0, 0]
    p = 1.0 / (1.0 + np.exp(-scale * (Q @ (K[0] - K[1]))))
    c = p * (1 - p) * (G @ (V[0] - V[1]))
    want_dq = scale * c[:, None] * (K[0] - K[1])[None, :]
    assert np.max(np.abs(dq[0, 0] / scale - want_dq)) > 1e-3        # dropped scale
    # A flipped D sign breaks sum_j dS_ij = 0, hence sum_j dK_j = 0; build such dK from the same
    # P and dP and check that the invariant catches it.
    P = np.stack([p, 1 - p], axis=1)
    dP = G @ V.T
    D = (dP * P).sum(axis=1, keepdims=True)
    bad_dk = scale * (P * (dP + D)).T @ Q
    assert np.max(np.abs(bad_dk.sum(axis=0))) > 1e-3
    assert np.max(np.abs(dk[0, 0].sum(axis=0))) < 1e-13
