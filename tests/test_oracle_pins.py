"""Pins for the fp64 oracle, checked against what the pages and the mathematics fix.

None of these tests re-types the oracle's formulas: they use values printed on the pages,
closed forms, a 50-digit brute force, and independent restatements of the per-key and tiled
recurrences.  Each is chosen so that a plausible slip in the oracle (a dropped scale, a wrong
mask index, swapped K and V, a log in the wrong base, a missing rescale) fails at least one.
"""

import math
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden(name):
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out[key] = vals
    return out


# ---------------------------------------------------------------------------------------------
# "FlashAttention: attention was never compute-bound", Online softmax: the whole idea (demo 2)
# ---------------------------------------------------------------------------------------------

def _demo2_row():
    """A 32-score row that reproduces demo 2's printed figures.

    The first six correct weights are the printed ones.  Block 1 holds them plus two weights of
    0.005; blocks 2 and 3 hold sixteen equal weights below block 1's maximum; block 4 holds one
    dominant weight W and seven equal weights.  With scores x = ln(w) and sum(w) = 1, softmax(x)
    is w itself.  Without the rescale, every block scored against an older maximum is too large
    by W / max(block 1), so the broken weights sum to
        1 / (A * W / max1 + (1 - A)),   A = mass of blocks 1-3,
    which fixes A for the printed sum 0.190131; W = 0.8063 makes the largest error
    W * (1 - 0.190131) print as 6.53e-01.
    """
    g = _golden("fa_io_demo2.txt")
    first6 = np.array([float(x) for x in g["correct_first6"]])
    target_sum = float(g["norescale_weight_sum"][0])
    W = 0.8063
    max1 = first6.max()
    A = (1.0 / target_sum - 1.0) / (W / max1 - 1.0)
    a = 0.005
    u = (A - first6.sum() - 2 * a) / 16.0
    r = (1.0 - A - W) / 7.0
    assert 0 < u < max1 and 0 < r < W and a < max1
    w = np.concatenate([first6, [a, a], np.full(16, u), [r, r, r, W, r, r, r, r]])
    return np.log(w), w, target_sum, g


def test_demo2_online_softmax_matches_ordinary_and_printed_weights():
    x, w, _, g = _demo2_row()
    ordinary = oracle.softmax(x)
    online = oracle.online_softmax(x, block=8, rescale=True)
    # closed form: softmax(ln w) = w when sum(w) = 1
    np.testing.assert_allclose(ordinary, w / w.sum(), rtol=1e-14, atol=0)
    # the page prints a max abs diff of 0.00e+00; fp64 reassociation allows a few ulp
    assert np.max(np.abs(ordinary - online)) <= 4 * np.finfo(np.float64).eps
    printed = [float(s) for s in g["online_first6"]]
    assert [f"{v:.6f}" for v in online[:6]] == [f"{v:.6f}" for v in printed]


def test_demo2_no_rescale_reproduces_printed_failure():
    x, w, target_sum, g = _demo2_row()
    ordinary = oracle.softmax(x)
    broken = oracle.online_softmax(x, block=8, rescale=False)
    assert abs(broken.sum() - target_sum) < 1e-12
    assert f"{np.max(np.abs(ordinary - broken)):.2e}" == g["ordinary_vs_norescale_max_abs_diff"][0]
    assert [f"{v:.6f}" for v in broken[:6]] == g["broken_first6"]
    # invariant: every broken weight is the correct one times the broken sum
    np.testing.assert_allclose(broken, ordinary * broken.sum(), rtol=1e-13, atol=0)


def test_demo2_printed_columns_satisfy_the_invariant():
    """The printed 'broken' column equals 'correct' x 0.190131 to print precision."""
    g = _golden("fa_io_demo2.txt")
    correct = np.array([float(s) for s in g["correct_first6"]])
    broken = np.array([float(s) for s in g["broken_first6"]])
    s = float(g["norescale_weight_sum"][0])
    assert np.all(np.abs(correct * s - broken) <= 5e-7 + 5e-7 * s)


def test_online_softmax_bit_exact_when_max_in_first_block():
    rng = np.random.default_rng(11)
    x = rng.standard_normal(32)
    x[3] = 10.0  # global max in block 1: every later correction factor is exp(0) = 1 exactly
    assert np.array_equal(oracle.online_softmax(x, 8, True), oracle.softmax(x))
    # and then dropping the rescale changes nothing
    assert np.array_equal(oracle.online_softmax(x, 8, False), oracle.softmax(x))


def test_no_rescale_fails_whenever_max_rises_late():
    rng = np.random.default_rng(12)
    for trial in range(20):
        x = rng.standard_normal(32) * 2
        x[24 + trial % 8] = 12.0  # max in block 4
        ordinary = oracle.softmax(x)
        broken = oracle.online_softmax(x, 8, False)
        assert broken.sum() < 1 - 1e-3
        assert np.max(np.abs(broken - ordinary)) > 1e-3
        good = oracle.online_softmax(x, 8, True)
        assert np.max(np.abs(good - ordinary)) <= 4 * np.finfo(np.float64).eps


@pytest.mark.parametrize("block", [1, 3, 8, 32, 100])
def test_online_softmax_any_block_size(block):
    rng = np.random.default_rng(13)
    x = rng.standard_normal(97) * 5
    np.testing.assert_allclose(oracle.online_softmax(x, block), oracle.softmax(x), rtol=1e-14, atol=1e-17)


# ---------------------------------------------------------------------------------------------
# "Understanding FlashAttention", Online softmax: (g, s) at the last element
# ---------------------------------------------------------------------------------------------

def test_online_normalizer_last_element_is_max_and_sum():
    rng = np.random.default_rng(14)
    for n in [1, 2, 8, 1000]:
        x = list(rng.random(n))
        g, s = oracle.online_normalizer(x)
        m = max(x)
        assert g == m
        assert math.isclose(s, math.fsum(math.exp(v - m) for v in x), rel_tol=1e-12)


def test_online_normalizer_closed_form_log_integers():
    # x_i = ln(i): g_N = ln N and s_N = sum_i i/N = (N + 1)/2
    for n in [1, 5, 64, 1001]:
        x = np.log(np.arange(1, n + 1, dtype=np.float64))
        g, s = oracle.online_normalizer(x)
        assert g == x[-1]
        assert math.isclose(s, (n + 1) / 2, rel_tol=1e-12)


def test_softmax_overflow_safety_scores_near_800():
    # scores near 800 overflow a plain exp ("Now break it": [nan nan nan nan]); safe softmax
    # must equal the softmax of the shifted row
    x = np.array([800.0, 801.0, 799.5, 800.25])
    y = oracle.softmax(x)
    assert np.all(np.isfinite(y))
    e = np.exp(x - 800.0)
    np.testing.assert_allclose(y, e / e.sum(), rtol=1e-15)
    assert np.all(np.isfinite(oracle.online_softmax(x, 2)))


# ---------------------------------------------------------------------------------------------
# Attention: closed forms and special cases
# ---------------------------------------------------------------------------------------------

def _log_weight_problem(Nq, Nk, scale):
    """q = e_0 for every row; k_j = ln(c_j)/scale e_0 so the scaled score is ln(c_j); v_j is
    (j + 1) times a one-hot vector at a permuted position.  Then p_j = c_j / sum(c) and
    O[perm[j]] = p_j (j + 1) exactly."""
    d = Nk
    c = np.arange(1, Nk + 1, dtype=np.float64) * 1.5
    q = np.zeros((1, 1, Nq, d))
    q[..., 0] = 1.0
    k = np.zeros((1, 1, Nk, d))
    k[0, 0, :, 0] = np.log(c) / scale
    perm = np.roll(np.arange(Nk), 1)
    v = np.zeros((1, 1, Nk, d))
    for j in range(Nk):
        v[0, 0, j, perm[j]] = j + 1.0
    return q, k, v, c, perm


@pytest.mark.parametrize("scale", [0.125, 0.7])
def test_attention_closed_form_noncausal(scale):
    Nq, Nk = 3, 6
    q, k, v, c, perm = _log_weight_problem(Nq, Nk, scale)
    o, lse = oracle.attention(q, k, v, causal=False, scale=scale)
    expect = np.zeros(Nk)
    for j in range(Nk):
        expect[perm[j]] = c[j] / c.sum() * (j + 1)
    for i in range(Nq):
        np.testing.assert_allclose(o[0, 0, i], expect, rtol=1e-13, atol=1e-15)
        assert math.isclose(lse[0, 0, i], math.log(c.sum()), rel_tol=1e-14)


def test_attention_closed_form_causal_bottom_right():
    scale = 0.5
    Nq, Nk = 3, 6  # row i sees keys j <= i + 3
    q, k, v, c, perm = _log_weight_problem(Nq, Nk, scale)
    o, lse = oracle.attention(q, k, v, causal=True, scale=scale)
    for i in range(Nq):
        vis = i + (Nk - Nq) + 1
        expect = np.zeros(Nk)
        for j in range(vis):
            expect[perm[j]] = c[j] / c[:vis].sum() * (j + 1)
        np.testing.assert_allclose(o[0, 0, i], expect, rtol=1e-13, atol=1e-15)
        assert math.isclose(lse[0, 0, i], math.log(c[:vis].sum()), rel_tol=1e-14)


def test_attention_causal_first_row_is_first_value():
    rng = np.random.default_rng(15)
    q, k, v = (rng.standard_normal((2, 3, 9, 16)) for _ in range(3))
    scale = 0.3
    o, lse = oracle.attention(q, k, v, causal=True, scale=scale)
    np.testing.assert_array_equal(o[:, :, 0], v[:, :, 0])
    np.testing.assert_allclose(lse[:, :, 0], scale * np.einsum("bht,bht->bh", q[:, :, 0], k[:, :, 0]),
                               rtol=1e-14)


def test_attention_identical_keys_gives_mean_of_values():
    rng = np.random.default_rng(16)
    Nq, Nk, d = 5, 7, 8
    q = rng.standard_normal((1, 2, Nq, d))
    k = np.broadcast_to(rng.standard_normal((1, 2, 1, d)), (1, 2, Nk, d)).copy()
    v = rng.standard_normal((1, 2, Nk, d))
    scale = 0.25
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal=causal, scale=scale)
        for h in range(2):
            for i in range(Nq):
                vis = (i + Nk - Nq + 1) if causal else Nk
                np.testing.assert_allclose(o[0, h, i], v[0, h, :vis].mean(axis=0), rtol=1e-13, atol=1e-15)
                x = scale * q[0, h, i] @ k[0, h, 0]
                assert math.isclose(lse[0, h, i], x + math.log(vis), rel_tol=1e-13, abs_tol=1e-14)


def test_attention_rows_sum_to_one_and_ones_values():
    rng = np.random.default_rng(17)
    q = rng.standard_normal((1, 1, 33, 16)) * 3
    k = rng.standard_normal((1, 1, 40, 16)) * 3
    for causal in (False, True):
        p = oracle.attention_probs(q[0, 0], k[0, 0], causal=causal, scale=0.25)
        np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
        if causal:
            for i in range(33):
                assert np.all(p[i, i + 7 + 1:] == 0) and np.all(p[i, : i + 7 + 1] > 0)
        o, _ = oracle.attention(q, k, np.ones((1, 1, 40, 16)), causal=causal, scale=0.25)
        np.testing.assert_allclose(o, 1.0, rtol=0, atol=1e-14)


def test_attention_shift_invariance_large_logits():
    """Adding a constant c to every score of a row leaves O unchanged and shifts L by c.
    Done by appending a dimension (q: C, k: 1), with scale * C = 800 (scores near 800)."""
    rng = np.random.default_rng(18)
    q, k, v = (rng.standard_normal((1, 2, 12, 8)) for _ in range(3))
    scale = 0.5
    C = 800.0 / scale
    q2 = np.concatenate([q, np.full((1, 2, 12, 1), C)], axis=-1)
    k2 = np.concatenate([k, np.ones((1, 2, 12, 1))], axis=-1)
    v2 = np.concatenate([v, np.zeros((1, 2, 12, 1))], axis=-1)
    for causal in (False, True):
        o, lse = oracle.attention(q, k, v, causal=causal, scale=scale)
        o2, lse2 = oracle.attention(q2, k2, v2, causal=causal, scale=scale)
        assert np.all(np.isfinite(o2)) and np.all(np.isfinite(lse2))
        np.testing.assert_allclose(o2[..., :8], o, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse2 - 800.0, lse, rtol=0, atol=1e-12)


def test_attention_matches_50_digit_brute_force():
    mpmath = pytest.importorskip("mpmath")
    mpmath.mp.dps = 50
    rng = np.random.default_rng(19)
    for (Nq, Nk, d, causal) in [(1, 1, 1, False), (2, 3, 2, False), (4, 4, 4, True), (3, 4, 3, True),
                                 (4, 2, 4, False)]:
        if causal and Nq > Nk:
            continue
        q, k, v = (rng.standard_normal((1, 1, n, d)) * 2 for n in (Nq, Nk, Nk))
        scale = 1.0 / math.sqrt(d)
        o, lse = oracle.attention(q, k, v, causal=causal, scale=scale)
        for i in range(Nq):
            keys = [j for j in range(Nk) if (not causal) or j <= i + Nk - Nq]
            xs = [mpmath.mpf(scale) * mpmath.fsum(mpmath.mpf(q[0, 0, i, t]) * mpmath.mpf(k[0, 0, j, t])
                                                  for t in range(d)) for j in keys]
            es = [mpmath.e ** x for x in xs]
            z = mpmath.fsum(es)
            for t in range(d):
                exact = mpmath.fsum(e * mpmath.mpf(v[0, 0, j, t]) for e, j in zip(es, keys)) / z
                assert abs(o[0, 0, i, t] - float(exact)) <= 1e-14 * max(1.0, abs(float(exact)))
            assert abs(lse[0, 0, i] - float(mpmath.log(z))) <= 1e-14 * max(1.0, abs(float(mpmath.log(z))))


def test_attention_rows_equals_full():
    rng = np.random.default_rng(20)
    q, k, v = (rng.standard_normal((2, 2, 21, 8)) for _ in range(3))
    o, lse = oracle.attention(q, k, v, causal=True, scale=0.4)
    rows = np.array([0, 5, 20, 21, 40, 83])
    o_r, lse_r = oracle.attention_rows(q, k, v, rows, causal=True, scale=0.4)
    np.testing.assert_array_equal(o_r, o.reshape(-1, 8)[rows])
    np.testing.assert_array_equal(lse_r, lse.reshape(-1)[rows])


# ---------------------------------------------------------------------------------------------
# Independent restatements: the per-key fused recurrence and the tiled loop nest
# ---------------------------------------------------------------------------------------------

def _per_key_recurrence(q, k, v, scale):
    """"Understanding FlashAttention", Merging the two loops: one key at a time, the output is
    kept normalised at every step, so after key m it is the attention over the first m keys."""
    N, D = len(q), len(q[0])
    out = []
    for n in range(N):
        a = [0.0] * D
        g = s = None
        for m in range(len(k)):
            x = scale * sum(q[n][t] * k[m][t] for t in range(D))
            if g is None:
                g, s = x, 1.0
                a = [v[m][t] for t in range(D)]
                continue
            g_new = max(g, x)
            shrink = math.exp(g - g_new)
            e = math.exp(x - g_new)
            s_new = s * shrink + e
            a = [(a[t] * s * shrink + e * v[m][t]) / s_new for t in range(D)]
            g, s = g_new, s_new
        out.append(a)
    return out


def test_per_key_recurrence_equals_oracle():
    rng = np.random.default_rng(21)
    N, M, D = 6, 11, 5
    q, k, v = rng.random((N, D)), rng.random((M, D)), rng.random((M, D))
    scale = 0.9
    a = _per_key_recurrence(q.tolist(), k.tolist(), v.tolist(), scale)
    o, _ = oracle.attention(q[None, None], k[None, None], v[None, None], causal=False, scale=scale)
    for n in range(N):
        for t in range(D):
            assert math.isclose(a[n][t], o[0, 0, n, t], rel_tol=1e-9)


def _tiled_forward(Q, K, V, scale, Br, Bc, causal=False, window=None):
    """FlashAttention-2 forward loop nest ("Flash Attention: The Hidden Gem", The Algorithm):
    outer loop over query tiles with (m, l, O) per row, inner loop over key/value tiles with the
    correction factor, one normalisation at the end, L = m + log l.  `window` restricts each
    query to keys with |i - j| < window/2 (the page's local-window negative control)."""
    n, d = Q.shape
    nk = K.shape[0]
    O = np.zeros((n, d))
    L = np.zeros(n)
    for i0 in range(0, n, Br):
        Qi = Q[i0:i0 + Br]
        rows = np.arange(i0, i0 + len(Qi))[:, None]
        m = np.full((len(Qi), 1), -np.inf)
        l = np.zeros((len(Qi), 1))
        Oi = np.zeros((len(Qi), d))
        for j0 in range(0, nk, Bc):
            S = scale * (Qi @ K[j0:j0 + Bc].T)
            cols = np.arange(j0, j0 + S.shape[1])[None, :]
            if causal:
                S = np.where(cols <= rows + (nk - n), S, -np.inf)
            if window is not None:
                S = np.where(np.abs(cols - rows) < window // 2, S, -np.inf)
            m_new = np.maximum(m, S.max(axis=1, keepdims=True))
            safe = np.where(np.isfinite(m_new), m_new, 0.0)
            P = np.exp(S - safe)
            corr = np.exp(np.where(np.isfinite(m), m - safe, -np.inf))
            l = corr * l + P.sum(axis=1, keepdims=True)
            Oi = corr * Oi + P @ V[j0:j0 + Bc]
            m = m_new
        O[i0:i0 + Br] = Oi / l
        L[i0:i0 + Br] = (m + np.log(l))[:, 0]
    return O, L


@pytest.mark.parametrize("n", [128, 256, 1024])
def test_tiled_equals_oracle_to_fp64_noise(n):
    # "FlashAttention: attention was never compute-bound", tiling demo: tiled and standard attention
    # agree to fp64 rounding (~1e-16)
    rng = np.random.default_rng(22 + n)
    d = 64
    Q, K, V = (rng.standard_normal((n, d)) for _ in range(3))
    scale = 1 / 8
    O, L = _tiled_forward(Q, K, V, scale, 64, 64)
    o, lse = oracle.attention(Q[None, None], K[None, None], V[None, None], scale=scale)
    assert np.max(np.abs(O - o[0, 0])) < 1e-13
    assert np.max(np.abs(L - lse[0, 0])) < 1e-12


def test_tiled_worked_example_shapes_causal_and_not():
    # "The Algorithm" worked example: N = 8, d = 128, Br = Bc = 2, Tr = Tc = 4
    rng = np.random.default_rng(23)
    Q, K, V = (rng.standard_normal((8, 128)) for _ in range(3))
    scale = 1 / math.sqrt(128)
    for causal in (False, True):
        O, L = _tiled_forward(Q, K, V, scale, 2, 2, causal=causal)
        o, lse = oracle.attention(Q[None, None], K[None, None], V[None, None], causal=causal, scale=scale)
        assert np.max(np.abs(O - o[0, 0])) < 1e-13
        assert np.max(np.abs(L - lse[0, 0])) < 1e-13


def test_local_window_negative_control_fails_tolerance():
    # "Exact means exact": a 128-wide local window is a different function (diff ~0.32)
    rng = np.random.default_rng(24)
    n, d = 512, 64
    Q, K, V = (rng.standard_normal((n, d)) for _ in range(3))
    o, _ = oracle.attention(Q[None, None], K[None, None], V[None, None], scale=1 / 8)
    Ow, _ = _tiled_forward(Q, K, V, 1 / 8, 64, 64, window=128)
    assert np.max(np.abs(Ow - o[0, 0])) > 2e-2


def test_oracle_detects_planted_mask_and_operand_mistakes():
    """The pins above separate the oracle from its plausible mutations: a causal mask that is
    off by one, swapped K and V, or a missing scale all change the closed-form answer."""
    scale = 0.5
    q, k, v, c, perm = _log_weight_problem(3, 6, scale)
    o_good, _ = oracle.attention(q, k, v, causal=True, scale=scale)
    o_kv, _ = oracle.attention(q, v, k, causal=True, scale=scale)
    o_ns, _ = oracle.attention(q, k, v, causal=True, scale=1.0)
    o_nc, _ = oracle.attention(q, k, v, causal=False, scale=scale)
    for bad in (o_kv, o_ns, o_nc):
        assert np.max(np.abs(bad - o_good)) > 1e-3
