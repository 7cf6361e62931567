"""GPU parity of the FP8 forward (fattn_fwd_fp8) against the fp64 oracle on the dequantised inputs.

The pages give FP8 no accuracy contract ("Flash Attention: The Hidden Gem", section FA1, FA2, FA3
only says it costs some precision), so the one in fattn.h is stated from the arithmetic and checked
here element by element:
    |o - o_exact| <= 2^-4 * sum_j p_j |v_j| + 2^-9 |o_exact| + (2^-15 n + 2^-16) max |v|,
    |lse - lse_exact| <= 2^-20 |lse_exact| + 1e-5,
where o_exact, lse_exact and sum_j p_j |v_j| come from the oracle (the last as the attention of the
same q, k with |v| as values).
"""

import math

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_31_gb300 as fa
    fa.lib()
    return fa


def _deq(t8, s):
    return t8.float().cpu().double().numpy() * s


def check_bound(o, lse, q, k, v, band, scale, rows=None, what=""):
    """Compare the kernel's (o, lse) with the oracle; rows = None for all rows, else sampled rows."""
    absv = np.abs(v)
    if rows is None:
        o_ref, lse_ref = oracle.attention(q, k, v, window=band, scale=scale)
        pv_abs, _ = oracle.attention(q, k, absv, window=band, scale=scale)
        o_k = o.float().cpu().double().numpy()
        l_k = lse.cpu().double().numpy()
    else:  # flat row indices (b*H + h)*Nq + i
        o_ref, lse_ref = oracle.attention_rows(q, k, v, rows, window=band, scale=scale)
        pv_abs, _ = oracle.attention_rows(q, k, absv, rows, window=band, scale=scale)
        o_k = o.float().cpu().double().numpy().reshape(-1, q.shape[3])[rows]
        l_k = lse.cpu().double().numpy().reshape(-1)[rows]
    Nq, Nk = q.shape[2], k.shape[2]
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l_k), empty), what
    assert np.all(o_k[empty] == 0.0), what
    full = ~empty
    vmax_bh = absv.reshape(absv.shape[0] * absv.shape[1], -1).max(axis=1)  # per (b, h)
    if rows is None:
        vmax = vmax_bh.reshape(absv.shape[0], absv.shape[1], 1, 1)
    else:
        vmax = vmax_bh[np.asarray(rows) // Nq][:, None]
    bound = 2.0 ** -4 * pv_abs + 2.0 ** -9 * np.abs(o_ref) + (2.0 ** -15 * Nk + 2.0 ** -16) * vmax
    err = np.abs(o_k - o_ref)
    worst = np.max(np.where(full[..., None], err - bound, -np.inf))
    assert worst <= 0.0, f"{what}: output error exceeds the stated bound by {worst:.3e}"
    if full.any():
        lerr = np.abs(l_k[full] - lse_ref[full])
        assert np.all(lerr <= 2.0 ** -20 * np.abs(lse_ref[full]) + 1e-5), (what, lerr.max())
    return float(err[full].max(initial=0.0)), float(err[full].mean()) if full.any() else 0.0


CASES = [
    # B, H, Nq, Nk, band
    (1, 2, 200, 200, (-1, 0)),
    (1, 2, 128, 128, (-1, -1)),
    (2, 2, 257, 333, (100, 0)),      # sliding window, chunk against a longer cache
    (1, 3, 333, 200, (-1, 0)),       # rows above the diagonal see nothing
    (1, 1, 1000, 1000, (-1, -1)),
    (1, 2, 77, 5, (-1, -1)),         # fewer keys than one tile
    (1, 1, 300, 300, (0, 0)),        # one key per row
]


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}q{}k{}w{}_{}".format(*c[:4], *c[4]))
def test_fp8_forward_within_stated_bound(fa, case, d):
    from exact_attention_31_gb300.workloads import make_qkv_fp8
    B, H, Nq, Nk, band = case
    (q8, k8, v8), (qs, ks, vs), boosted = make_qkv_fp8(B, H, Nq, Nk, d, 9000 + Nq + Nk + band[0] + d, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_fwd_fp8(q8, k8, v8, qs, ks, vs, window=band, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    check_bound(o, lse, _deq(q8, qs), _deq(k8, ks), _deq(v8, vs), band, scale, what=str(case))


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_b4h16_n2048_boosted_rows_sampled(fa, causal):
    # The d = 128 configuration with 1 % of query rows scaled x8 (a sharper softmax), quantised to e4m3;
    # sampled rows of four heads, and every boosted row of the first head.
    from exact_attention_31_gb300.workloads import make_qkv_fp8
    (q8, k8, v8), (qs, ks, vs), boosted = make_qkv_fp8(4, 16, 2048, 2048, 128, 9100, device="cuda", boost_frac=0.01)
    scale = 1.0 / math.sqrt(128)
    band = (-1, 0) if causal else (-1, -1)
    o, lse = fa.fattn_fwd_fp8(q8, k8, v8, qs, ks, vs, window=band, scale=scale)
    torch.cuda.synchronize()
    Nq = 2048
    per_head = np.unique(np.concatenate([np.arange(0, Nq, 97), [Nq - 1]]))
    rows = [bh * Nq + per_head for bh in (0, 5, 37, 63)] + [boosted[0].cpu().numpy()]
    rows = np.unique(np.concatenate(rows))
    check_bound(o, lse, _deq(q8, qs), _deq(k8, ks), _deq(v8, vs), band, scale, rows=rows, what=f"causal={causal}")


def test_fp8_b1h32_n8192_d64_causal_sampled(fa):
    # The d = 64 long-sequence configuration (B1 H32 N8192 causal) in e4m3, 1 % of query rows scaled x8;
    # sampled rows of four heads (the first and last rows of every 256-row unit among them) and
    # every boosted row of the first head.
    from exact_attention_31_gb300.workloads import make_qkv_fp8
    B, H, N, d = 1, 32, 8192, 64
    (q8, k8, v8), (qs, ks, vs), boosted = make_qkv_fp8(B, H, N, N, d, 9150, device="cuda", boost_frac=0.01)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    per_head = np.unique(np.concatenate([np.arange(0, N, 331), np.arange(0, N, 256), np.arange(255, N, 256)]))
    rows = [bh * N + per_head for bh in (0, 9, 22, 31)] + [boosted[0].cpu().numpy()]
    rows = np.unique(np.concatenate(rows))
    check_bound(o, lse, _deq(q8, qs), _deq(k8, ks), _deq(v8, vs), (-1, 0), scale, rows=rows, what="d64 N8192")


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_descales_enter_exactly(fa, d):
    # Doubling v_descale doubles O exactly (it multiplies the fp32 normaliser), and moving a factor 2
    # from scale to q_descale leaves the exponent's fp32 coefficient, and so every output, unchanged.
    from exact_attention_31_gb300.workloads import make_qkv_fp8
    (q8, k8, v8), (qs, ks, vs), boosted = make_qkv_fp8(1, 2, 256, 256, d, 9200 + d, device="cuda")
    sc = 1.0 / math.sqrt(d)
    o1, l1 = fa.fattn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True, scale=sc)
    o2, l2 = fa.fattn_fwd_fp8(q8, k8, v8, qs, ks, 2 * vs, causal=True, scale=sc)
    o3, l3 = fa.fattn_fwd_fp8(q8, k8, v8, 2 * qs, ks, vs, causal=True, scale=sc / 2)
    torch.cuda.synchronize()
    assert torch.equal(o2.float(), 2 * o1.float()) and torch.equal(l1, l2)
    assert torch.equal(o1, o3) and torch.equal(l1, l3)


def test_fp8_rejects_other_head_dims(fa):
    q = torch.zeros((1, 1, 64, 96), dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(fa.FattnError) as e:
        fa.fattn_fwd_fp8(q, q, q, 1.0, 1.0, 1.0, workspace=torch.empty(4096, dtype=torch.uint8, device="cuda"))
    assert e.value.status == 2


def _random_cases(n=12, seed=0xF8):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        Nq, Nk = int(rng.integers(1, 600)), int(rng.integers(1, 600))
        kind = int(rng.integers(0, 4))
        band = [(-1, -1), (-1, 0), (int(rng.integers(0, 300)), 0),
                (int(rng.integers(0, 200)), int(rng.integers(0, 200)))][kind]
        out.append((B, H, Nq, Nk, band))
    return out


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", _random_cases(), ids=lambda c: "b{}h{}q{}k{}w{}_{}".format(*c[:4], *c[4]))
def test_fp8_random_shapes_within_stated_bound(fa, case, d):
    from exact_attention_31_gb300.workloads import make_qkv_fp8
    B, H, Nq, Nk, band = case
    (q8, k8, v8), (qs, ks, vs), _ = make_qkv_fp8(B, H, Nq, Nk, d, 9300 + 3 * Nq + Nk + d, device="cuda")
    scale = 0.9 / math.sqrt(d)
    o, lse = fa.fattn_fwd_fp8(q8, k8, v8, qs, ks, vs, window=band, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    check_bound(o, lse, _deq(q8, qs), _deq(k8, ks), _deq(v8, vs), band, scale, what=str(case))
