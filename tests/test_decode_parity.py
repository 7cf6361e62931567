"""GPU parity of fattn_decode (split-KV kernel + combine kernel) against the fp64 oracle."""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_utils import compare, oracle_full, to64

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_31_gb300 as fa
    fa.lib()
    return fa


def _gen(B, H, Nk, d, seed):
    from exact_attention_31_gb300.workloads import make_qkv
    q, k, v, _ = make_qkv(B, H, 1, Nk, d, seed, device="cuda")
    return q, k, v


CASES = [
    # B, H, Nk, d, num_splits
    (1, 1, 1, 64, 0),
    (1, 1, 1, 128, 1),
    (1, 2, 64, 128, 0),
    (2, 2, 65, 64, 0),
    (2, 2, 65, 64, 2),
    (2, 3, 1000, 128, 0),
    (2, 3, 1000, 128, 1),
    (2, 3, 1000, 128, 5),
    (3, 2, 4097, 64, 0),
    (1, 4, 16384, 128, 0),
    (1, 4, 16384, 128, 7),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}k{}d{}s{}".format(*c))
def test_decode_matches_oracle(fa, case):
    B, H, Nk, d, S = case
    q, k, v = _gen(B, H, Nk, d, seed=2000 + Nk + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_decode(q, k, v, scale=scale, num_splits=S)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_full(q, k, v, False, scale)
    compare(o, lse, o_ref, lse_ref, what=str(case))


def test_decode_split_count_invariance(fa):
    """The combine rule is exact: splitting the keys differently changes only rounding."""
    B, H, Nk, d = 2, 2, 16384, 128
    q, k, v = _gen(B, H, Nk, d, seed=2100)
    outs = []
    for S in (1, 4, 256):
        ws = torch.empty(fa.fattn_decode_workspace_size(B, H, Nk, d, S), dtype=torch.uint8, device="cuda")
        o, lse = fa.fattn_decode(q, k, v, num_splits=S, workspace=ws)
        outs.append((o.float(), lse))
    for o, lse in outs[1:]:
        assert torch.max(torch.abs(o - outs[0][0])).item() <= 2 ** -8
        assert torch.max(torch.abs(lse - outs[0][1])).item() <= 1e-5


def test_decode_equals_prefill_with_one_query(fa):
    B, H, Nk, d = 2, 3, 777, 64
    q, k, v = _gen(B, H, Nk, d, seed=2200)
    od, ld = fa.fattn_decode(q, k, v)
    op, lp = fa.fattn_fwd(q, k, v, causal=False)
    assert torch.max(torch.abs(od.float() - op.float())).item() <= 2 ** -7
    assert torch.max(torch.abs(ld - lp)).item() <= 2e-5


def test_decode_guard_bands_and_workspace_reuse(fa):
    B, H, Nk, d = 2, 2, 300, 128
    q, k, v = _gen(B, H, Nk, d, seed=2300)
    n = B * H * d
    big = torch.full((n + 512,), 3.0, dtype=torch.bfloat16, device="cuda")
    o = big[256:256 + n].view(B, H, 1, d)
    need = fa.fattn_decode_workspace_size(B, H, Nk, d, 0)
    ws = torch.full((need,), 0xFF, dtype=torch.uint8, device="cuda")  # stale contents must not matter
    fa.fattn_decode(q, k, v, out=o, workspace=ws)
    fa.fattn_decode(q, k, v, out=o, workspace=ws)
    torch.cuda.synchronize()
    assert torch.all(big[:256] == 3.0) and torch.all(big[256 + n:] == 3.0)
    o_ref, lse_ref = oracle_full(q, k, v, False, 1 / math.sqrt(d))
    compare(o, None, o_ref, lse_ref, what="decode guard")


@pytest.mark.parametrize("num_splits", [0, 256], ids=["default_splits", "one_state_per_64key_block"])
def test_workload_decode_b32h32_nk16384_d128(fa, num_splits):
    # every (b, h) of the B32 H32 Nk16384 d128 decode, element by element against the oracle, with the
    # default split count and with one partial state per 64-key block; the cache is moved to the host
    # one batch entry (32 heads, 2 x 128 MiB) at a time
    from exact_attention_31_gb300.workloads import WORKLOADS, make_workload
    w = WORKLOADS["decode_b32h32_nk16384_d128"]
    q, k, v, _ = make_workload(w, "cuda")
    o, lse = fa.fattn_decode(q, k, v, scale=w.scale, num_splits=num_splits)
    torch.cuda.synchronize()
    err_sum = 0.0
    for b in range(w.B):
        o_ref, lse_ref = oracle.attention(to64(q[b:b + 1]), to64(k[b:b + 1]), to64(v[b:b + 1]), causal=False,
                                          scale=w.scale)
        s = compare(o[b:b + 1], lse[b:b + 1], o_ref, lse_ref, what=f"{w.name} b{b}")
        err_sum += s["o_mean"]
    assert err_sum / w.B <= 1e-3
