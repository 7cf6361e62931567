"""GPU parity of fattn_fwd (the tcgen05 prefill kernel) against the fp64 oracle.

Every output is compared element by element, the full-size workloads included.  All inputs come from the
seeded generator in exact_attention_31_gb300.workloads.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_utils import compare, oracle_full, to64

pytestmark = pytest.mark.gpu

SHAPES = [
    # B, H, Nq, Nk, d, causal
    (1, 1, 128, 128, 64, False),
    (1, 1, 1, 1, 64, False),
    (1, 1, 1, 1, 128, True),
    (1, 2, 5, 7, 64, True),
    (2, 3, 300, 300, 64, True),
    (2, 3, 300, 300, 64, False),
    (1, 2, 200, 333, 64, False),
    (1, 2, 77, 333, 128, True),
    (2, 2, 513, 513, 128, False),
    (2, 2, 513, 513, 128, True),
    (1, 3, 256, 1000, 64, True),
    (1, 1, 640, 640, 128, True),
    (1, 2, 129, 129, 64, True),
]


@pytest.fixture(scope="module")
def fa():
    import exact_attention_31_gb300 as fa
    fa.lib()
    return fa


def _gen(B, H, Nq, Nk, d, seed, boost_frac=0.0):
    from exact_attention_31_gb300.workloads import make_qkv
    return make_qkv(B, H, Nq, Nk, d, seed, device="cuda", boost_frac=boost_frac)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}h{}q{}k{}d{}{}".format(*s[:5], "c" if s[5] else ""))
def test_prefill_matches_oracle(fa, shape):
    B, H, Nq, Nk, d, causal = shape
    q, k, v, _ = _gen(B, H, Nq, Nk, d, seed=1000 + Nq + 7 * Nk + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_fwd(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_full(q, k, v, causal, scale)
    compare(o, lse, o_ref, lse_ref, what=str(shape))
    assert fa.fattn_last_error() == 0


def test_prefill_scale_and_large_logits(fa):
    # large scores (scale 1, inputs x4): the running max moves a lot between tiles
    q, k, v, _ = _gen(1, 2, 384, 384, 64, seed=77)
    q = (q.float() * 4).to(torch.bfloat16)
    for causal in (False, True):
        o, lse = fa.fattn_fwd(q, k, v, causal=causal, scale=1.0)
        o_ref, lse_ref = oracle_full(q, k, v, causal, 1.0)
        compare(o, lse, o_ref, lse_ref, what=f"large logits causal={causal}")


def test_prefill_without_lse_and_guard_bands(fa):
    B, H, Nq, Nk, d = 1, 2, 200, 200, 128
    q, k, v, _ = _gen(B, H, Nq, Nk, d, seed=78)
    n = B * H * Nq * d
    sentinel = torch.tensor(-12352.0, dtype=torch.bfloat16)
    big = torch.full((n + 2048,), sentinel.item(), dtype=torch.bfloat16, device="cuda")
    o = big[1024:1024 + n].view(B, H, Nq, d)
    lse_big = torch.full((B * H * Nq + 64,), -7.0, dtype=torch.float32, device="cuda")
    lse = lse_big[32:32 + B * H * Nq].view(B, H, Nq)
    fa.fattn_fwd(q, k, v, causal=True, out=o, lse=lse)
    torch.cuda.synchronize()
    assert torch.all(big[:1024] == sentinel.item()) and torch.all(big[1024 + n:] == sentinel.item())
    assert torch.all(lse_big[:32] == -7.0) and torch.all(lse_big[32 + B * H * Nq:] == -7.0)
    o_ref, lse_ref = oracle_full(q, k, v, True, 1 / math.sqrt(d))
    compare(o, lse, o_ref, lse_ref, what="guard bands")
    o2, none = fa.fattn_fwd(q, k, v, causal=True, want_lse=False)
    assert none is None
    assert torch.equal(o2, o)


def test_prefill_is_deterministic(fa):
    q, k, v, _ = _gen(2, 4, 700, 700, 64, seed=79)
    a, la = fa.fattn_fwd(q, k, v, causal=True)
    b, lb = fa.fattn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(a, b) and torch.equal(la, lb)


def test_prefill_uniform_keys_closed_form(fa):
    # identical keys: every visible key gets the same weight, O is the mean of the visible values
    B, H, N, d = 1, 1, 300, 64
    q, k, v, _ = _gen(B, H, N, N, d, seed=80)
    k = k[:, :, :1].expand(B, H, N, d).contiguous()
    o, lse = fa.fattn_fwd(q, k, v, causal=True)
    vv = to64(v)[0, 0]
    mean = np.cumsum(vv, axis=0) / np.arange(1, N + 1)[:, None]
    assert np.max(np.abs(to64(o)[0, 0] - mean)) < 2e-2
    x = to64(q)[0, 0] @ to64(k)[0, 0, 0] / math.sqrt(d)
    assert np.max(np.abs(to64(lse)[0, 0] - (x + np.log(np.arange(1, N + 1))))) < 1e-3


def test_workload_b1h1_n128_d64(fa):
    from exact_attention_31_gb300.workloads import WORKLOADS, make_workload
    w = WORKLOADS["prefill_b1h1_n128_d64"]
    q, k, v, _ = make_workload(w, "cuda")
    o, lse = fa.fattn_fwd(q, k, v, causal=False, scale=w.scale)
    o_ref, lse_ref = oracle_full(q, k, v, False, w.scale)
    compare(o, lse, o_ref, lse_ref, what=w.name)


def test_workload_b1h8_n1024_d64_causal(fa):
    from exact_attention_31_gb300.workloads import WORKLOADS, make_workload
    w = WORKLOADS["prefill_b1h8_n1024_d64"]
    q, k, v, _ = make_workload(w, "cuda")
    o, lse = fa.fattn_fwd(q, k, v, causal=True, scale=w.scale)
    o_ref, lse_ref = oracle_full(q, k, v, True, w.scale)
    compare(o, lse, o_ref, lse_ref, what=w.name)


@pytest.mark.parametrize("causal", [False, True])
def test_workload_b4h16_n2048_d128_boosted_rows(fa, causal):
    # every output of the B4 H16 N2048 d128 workload (1 % of the query rows of each head x8),
    # element by element against the oracle
    from exact_attention_31_gb300.workloads import WORKLOADS, make_workload
    w = WORKLOADS["prefill_b4h16_n2048_d128"]
    q, k, v, boosted = make_workload(w, "cuda")
    o, lse = fa.fattn_fwd(q, k, v, causal=causal, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_full(q, k, v, causal, w.scale)
    s = compare(o, lse, o_ref, lse_ref, what=w.name + (" causal" if causal else ""))
    # the boosted rows on their own (their peaked weights carry the largest errors)
    rows = np.concatenate([bh * w.Nq + boosted[bh].numpy() for bh in range(w.B * w.H)])
    ob = to64(o).reshape(-1, w.d)[rows]
    eb = np.abs(ob - o_ref.reshape(-1, w.d)[rows])
    assert eb.max() <= 2e-2, (eb.max(), s)
    assert np.abs(to64(lse).reshape(-1)[rows] - lse_ref.reshape(-1)[rows]).max() <= 1e-3


def test_workload_b1h32_n8192_d64_causal(fa):
    # every output of the B1 H32 N8192 d64 causal workload, element by element against the oracle
    from exact_attention_31_gb300.workloads import WORKLOADS, make_workload
    w = WORKLOADS["prefill_b1h32_n8192_d64"]
    q, k, v, _ = make_workload(w, "cuda")
    o, lse = fa.fattn_fwd(q, k, v, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_full(q, k, v, True, w.scale)
    compare(o, lse, o_ref, lse_ref, what=w.name)
    # causal row 0 sees only key 0: its output is exactly v_0
    assert torch.equal(o[:, :, 0], v[:, :, 0])


def test_one_tile_items_in_the_last_round(fa):
    # one 256-row unit per head and one head more than SMs: the last round's unit is taken one
    # query tile at a time by two CTAs (and the B1 H8 N1024 and B4 H16 N2048 workloads, whose units
    # do not fill the GPU or leave a half-empty last round, take the same path); every row of the
    # last heads and sampled rows of the others against the oracle
    from parity_utils import oracle_rows
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    B, H, N, d = 1, sms + 1, 256, 64
    q, k, v, _ = _gen(B, H, N, N, d, seed=81)
    o, lse = fa.fattn_fwd(q, k, v, scale=0.125)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(to64(q[:, -2:]), to64(k[:, -2:]), to64(v[:, -2:]), scale=0.125)
    compare(o[:, -2:], lse[:, -2:], o_ref, lse_ref, what="last round in one-tile items")
    rows = np.arange(0, (H - 2) * N, 997)
    o_s, l_s = oracle_rows(q, k, v, rows, False, 0.125)
    assert np.abs(to64(o).reshape(-1, d)[rows] - o_s).max() <= 2e-2
    assert np.abs(to64(lse).reshape(-1)[rows] - l_s).max() <= 1e-3
