"""GPU parity of the banded masks (fattn_fwd_masked, fattn_bwd_masked, fattn_decode_masked) against
the fp64 oracle.

A band (window_left, window_right) lets query row i see key j iff
i + off - window_left <= j <= i + off + window_right, off = Nk - Nq, -1 = unbounded side.  Rows
with no visible key must come out as o = 0, L = -inf (and dq = 0); keys that no query sees as
dk = dv = 0.  Chunked prefill (a block of queries against a longer key sequence, causal,
bottom-right aligned) must reproduce the matching rows of the full prefill exactly.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_utils import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, to64
from test_backward_parity import compare_grads

pytestmark = pytest.mark.gpu

CASES = [
    # B, H, Nq, Nk, d, (window_left, window_right)
    (1, 2, 300, 300, 64, (127, 0)),      # sliding window of 128 keys
    (1, 2, 300, 300, 64, (0, 0)),        # one key per row
    (1, 2, 300, 300, 128, (63, 64)),     # symmetric local band
    (1, 2, 200, 333, 64, (100, 0)),      # chunk against a longer cache, windowed
    (1, 2, 333, 200, 64, (-1, 0)),       # causal with Nq > Nk: the top 133 rows see nothing
    (2, 2, 513, 513, 128, (255, 0)),
    (1, 1, 1000, 1000, 64, (1, 1)),
    (2, 2, 257, 600, 64, (-1, 50)),      # keys up to 50 past the diagonal
    (1, 2, 256, 640, 64, (0, 0)),        # keys 0..383 are seen by no query
    (1, 2, 640, 256, 128, (10, -1)),     # rows above the band's left edge see nothing
    (1, 1, 5, 7, 64, (2, 1)),
]


@pytest.fixture(scope="module")
def fa():
    import exact_attention_31_gb300 as fa
    fa.lib()
    return fa


def _inputs(B, H, Nq, Nk, d, seed):
    from exact_attention_31_gb300.workloads import make_dout, make_qkv
    q, k, v, _ = make_qkv(B, H, Nq, Nk, d, seed, device="cuda")
    return q, k, v, make_dout(B, H, Nq, d, seed, device="cuda")


def compare_masked(o, lse, o_ref, lse_ref, what):
    o = to64(o).reshape(o_ref.shape)
    lse = to64(lse).reshape(lse_ref.shape)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(lse), empty), f"{what}: rows with no visible key differ"
    assert np.all(o[empty] == 0.0), f"{what}: rows with no visible key must be 0"
    full = ~empty
    err = np.abs(o[full] - o_ref[full])
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    assert err.max(initial=0.0) <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (what, err.max(), err.mean())
    if full.any():
        assert np.abs(lse[full] - lse_ref[full]).max() <= LSE_MAX_ABS, what
    return int(empty.sum())


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}q{}k{}d{}w{}_{}".format(*c[:5], *c[5]))
def test_forward_band_matches_oracle(fa, case):
    B, H, Nq, Nk, d, band = case
    q, k, v, _ = _inputs(B, H, Nq, Nk, d, seed=4000 + Nq + 3 * Nk + d + band[0])
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_fwd(q, k, v, window=band, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), window=band, scale=scale)
    compare_masked(o, lse, o_ref, lse_ref, str(case))


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}q{}k{}d{}w{}_{}".format(*c[:5], *c[5]))
def test_backward_band_matches_oracle(fa, case):
    B, H, Nq, Nk, d, band = case
    q, k, v, do = _inputs(B, H, Nq, Nk, d, seed=5000 + Nq + 3 * Nk + d + band[1])
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_fwd(q, k, v, window=band, scale=scale)
    dq, dk, dv = fa.fattn_bwd(q, k, v, o, lse, do, window=band, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    ref = oracle.attention_backward(to64(q), to64(k), to64(v), to64(do), window=band, scale=scale)
    compare_grads((dq, dk, dv), ref, what=str(case))
    # exact zeros where the mask leaves nothing
    _, lse_ref = oracle.attention(to64(q), to64(k), to64(v), window=band, scale=scale)
    empty_rows = np.isneginf(lse_ref)
    assert np.all(to64(dq)[empty_rows] == 0.0)
    unseen = np.all(ref[2] == 0.0, axis=-1) & np.all(ref[1] == 0.0, axis=-1)
    assert np.all(to64(dk)[unseen] == 0.0) and np.all(to64(dv)[unseen] == 0.0)


@pytest.mark.parametrize("d", [64, 128])
def test_named_bands_equal_the_plain_entry_point(fa, d):
    q, k, v, _ = _inputs(1, 2, 384, 500, d, seed=4100 + d)
    for causal, band in ((True, (-1, 0)), (False, (-1, -1))):
        o1, l1 = fa.fattn_fwd(q, k, v, causal=causal)
        o2, l2 = fa.fattn_fwd(q, k, v, window=band)
        torch.cuda.synchronize()
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("d,N,c", [(64, 1000, 300), (128, 1000, 77), (64, 2048, 128)])
def test_chunked_prefill_reproduces_the_full_prefill(fa, d, N, c):
    # A chunk of the last c queries against all N keys (causal, bottom-right aligned) is the same
    # computation, row for row, as those rows of the full causal prefill.
    q, k, v, _ = _inputs(1, 2, N, N, d, seed=4200 + N + c)
    o_full, l_full = fa.fattn_fwd(q, k, v, causal=True)
    qc = q[:, :, N - c:].contiguous()
    o_chunk, l_chunk = fa.fattn_fwd(qc, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o_chunk, o_full[:, :, N - c:]) and torch.equal(l_chunk, l_full[:, :, N - c:])


def test_masked_rejects_bad_windows(fa):
    q, k, v, _ = _inputs(1, 1, 64, 64, 64, seed=4300)
    with pytest.raises(fa.FattnError):
        fa.fattn_fwd(q, k, v, window=(-2, 0))
    with pytest.raises(fa.FattnError):
        fa.fattn_fwd(q, k, v, window=(0, -5))


@pytest.mark.parametrize("Nk,W,d,splits", [(300, 1, 64, 0), (300, 64, 128, 0), (300, 65, 64, 2), (4096, 1000, 128, 0),
                                           (4096, 1000, 64, 7), (4096, 5000, 128, 0), (1, 1, 64, 0), (129, 128, 64, 1)])
def test_decode_sliding_window_matches_oracle(fa, Nk, W, d, splits):
    # One query per (b, h) at position Nk - 1 sees the last W keys.
    from exact_attention_31_gb300.workloads import make_qkv
    q, k, v, _ = make_qkv(2, 3, 1, Nk, d, seed=4400 + Nk + W + d, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_decode(q, k, v, window=(W - 1, 0), num_splits=splits, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), window=(W - 1, 0), scale=scale)
    compare_masked(o, lse, o_ref, lse_ref, f"decode Nk={Nk} W={W} d={d} splits={splits}")
    # the same band through the prefill kernel with Nq = 1
    o2, lse2 = fa.fattn_fwd(q, k, v, window=(W - 1, 0), scale=scale)
    torch.cuda.synchronize()
    assert torch.allclose(o.float(), o2.float(), atol=2e-2) and torch.allclose(lse, lse2, atol=1e-3)
