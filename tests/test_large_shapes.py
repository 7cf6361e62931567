"""GPU parity at size extremes the other tests do not reach: long sequences (a 32K-token causal
prefill, a 256K-key decode, the backward at 8K tokens, an element mask over 32K keys), many heads
in one call, and the FP8 forward at 16K tokens.  Outputs are compared with the fp64 oracle on
sampled rows (every gradient of one 8K head), at the tolerances of the regular parity tests; these
catch 32-bit index overflows and scheduling edge cases of the persistent grid and the split count.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_utils import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_31_gb300 as fa
    fa.lib()
    return fa


def _compare_rows(o, lse, q, k, v, rows, band, scale, what):
    o_ref, lse_ref = oracle.attention_rows(to64(q), to64(k), to64(v), rows, window=band, scale=scale)
    d = q.shape[-1]
    o_k = to64(o).reshape(-1, d)[rows]
    l_k = to64(lse).reshape(-1)[rows]
    err = np.abs(o_k - o_ref)
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (what, err.max(), err.mean())
    assert np.abs(l_k - lse_ref).max() <= LSE_MAX_ABS, what


def test_prefill_32k_tokens_causal(fa):
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, N, d = 1, 2, 32768, 64
    q, k, v, _ = make_qkv(B, H, N, N, d, 9500, device="cuda")
    o, lse = fa.fattn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    per_head = np.array([0, 1, 127, 128, 255, 256, 4095, 16383, 16384, 32767 - 128, 32766, 32767])
    rows = np.concatenate([bh * N + per_head for bh in range(B * H)])
    _compare_rows(o, lse, q, k, v, rows, (-1, 0), 1 / math.sqrt(d), "N=32768 causal")


def test_decode_256k_keys(fa):
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, Nk, d = 1, 2, 262144, 128
    q, k, v, _ = make_qkv(B, H, 1, Nk, d, 9501, device="cuda")
    o, lse = fa.fattn_decode(q, k, v)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), scale=1 / math.sqrt(d))
    assert np.abs(to64(o) - o_ref).max() <= O_MAX_ABS
    assert np.abs(to64(lse) - lse_ref).max() <= LSE_MAX_ABS


def test_4096_heads_in_one_call(fa):
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, N, d = 64, 64, 130, 64
    q, k, v, _ = make_qkv(B, H, N, N, d, 9502, device="cuda")
    o, lse = fa.fattn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    rng = np.random.default_rng(9502)
    rows = np.unique(np.concatenate([rng.choice(B * H * N, 300, replace=False), [0, B * H * N - 1]]))
    _compare_rows(o, lse, q, k, v, rows, (-1, 0), 1 / math.sqrt(d), "4096 heads")


def test_fp8_16k_tokens_causal(fa):
    from exact_attention_31_gb300.workloads import make_qkv_fp8
    B, H, N, d = 1, 2, 16384, 128
    (q8, k8, v8), (qs, ks, vs), _ = make_qkv_fp8(B, H, N, N, d, 9503, device="cuda")
    o, lse = fa.fattn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    from test_fp8_parity import _deq, check_bound
    per_head = np.array([0, 127, 128, 8191, 16383])
    rows = np.concatenate([bh * N + per_head for bh in range(B * H)])
    check_bound(o, lse, _deq(q8, qs), _deq(k8, ks), _deq(v8, vs), (-1, 0), 1 / math.sqrt(d), rows=rows,
                what="fp8 N=16384")


def test_backward_8k_tokens_causal(fa):
    # one head of 8192 tokens: 64 key-tile CTAs, the longest walking 64 query tiles; every gradient
    # against the oracle's (one head is one oracle thread: about half a minute), relative to its
    # magnitude as in the regular backward tests
    from exact_attention_31_gb300.workloads import make_dout, make_qkv
    from test_backward_parity import GRAD_MAX_REL, GRAD_MEAN_REL
    B, H, N, d = 1, 1, 8192, 64
    q, k, v, _ = make_qkv(B, H, N, N, d, 9504, device="cuda")
    do = make_dout(B, H, N, d, 9504, device="cuda")
    scale = 1 / math.sqrt(d)
    o, lse = fa.fattn_fwd(q, k, v, causal=True, scale=scale)
    dq, dk, dv = fa.fattn_bwd(q, k, v, o, lse, do, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    refs = oracle.attention_backward(to64(q), to64(k), to64(v), to64(do), causal=True, scale=scale)
    for name, got, ref in zip(("dq", "dk", "dv"), (dq, dk, dv), refs):
        err = np.abs(to64(got) - ref)
        assert err.max() <= GRAD_MAX_REL * np.abs(ref).max(), (name, err.max(), np.abs(ref).max())
        assert err.mean() <= GRAD_MEAN_REL * np.abs(ref).mean(), (name, err.mean(), np.abs(ref).mean())


def test_element_mask_32k_keys(fa):
    # 4096 queries against 32,768 keys under one mask for both heads: block-sparse (a seeded half of
    # the 128 x 128 blocks hidden) with random bits inside one block in eight, and a row that sees
    # nothing; the summary's bit words span four 64-bit words per query tile
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, Nq, Nk, d = 1, 2, 4096, 32768, 64
    q, k, v, _ = make_qkv(B, H, Nq, Nk, d, 9505, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(9505)
    blocks = torch.rand((Nq // 128, Nk // 128), generator=g, device="cuda") < 0.5
    part = torch.rand((Nq // 128, Nk // 128), generator=g, device="cuda") < 0.125
    mask = blocks.repeat_interleave(128, 0).repeat_interleave(128, 1)
    noise = torch.rand((Nq, Nk), generator=g, device="cuda") < 0.5
    mask = torch.where(part.repeat_interleave(128, 0).repeat_interleave(128, 1), mask & noise, mask)
    mask[1000] = False
    del noise
    o, lse = fa.fattn_fwd(q, k, v, scale=0.125, mask=fa.pack_mask(mask))
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    per_head = np.array([0, 1, 127, 128, 999, 1000, 1001, 2047, 2048, 4095])
    rows = np.concatenate([bh * Nq + per_head for bh in range(B * H)])
    m = mask.cpu().numpy()
    o_ref, lse_ref = oracle.attention_rows(to64(q), to64(k), to64(v), rows, scale=0.125, mask=m)
    o_k = to64(o).reshape(-1, d)[rows]
    l_k = to64(lse).reshape(-1)[rows]
    empty = np.isin(rows % Nq, [1000])
    assert np.all(o_k[empty] == 0.0) and np.all(l_k[empty] == -np.inf)
    err = np.abs(o_k[~empty] - o_ref[~empty])
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (err.max(), err.mean())
    assert np.abs(l_k[~empty] - lse_ref[~empty]).max() <= LSE_MAX_ABS
