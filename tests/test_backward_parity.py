"""GPU parity of fattn_bwd (the tcgen05 backward kernels) against the fp64 oracle's gradients.

Inputs come from the seeded generators in exact_attention_31_gb300.workloads.  The forward output
O and L fed to the backward are the library's own (fattn_fwd), as a caller would use them; one test
feeds the oracle's O and L instead, so that the backward is checked on its own.  The oracle
differentiates the exact softmax of the same bf16 inputs.

Tolerance.  The kernels round P and dS to bf16 (relative error at most 2^-9) before the products
that consume them, accumulate in fp32, and round dQ, dK, dV to bf16 at the end; O is bf16 too, so
D = rowsum(dO o O) carries O's rounding.  Each gradient is compared relative to its own magnitude:
max |err| <= GRAD_MAX_REL * max |ref| and mean |err| <= GRAD_MEAN_REL * mean |ref|.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_utils import to64

pytestmark = pytest.mark.gpu

GRAD_MAX_REL = 1.5e-2
GRAD_MEAN_REL = 5e-3

SHAPES = [
    # B, H, Nq, Nk, d, causal
    (1, 1, 128, 128, 64, False),
    (1, 1, 1, 1, 64, False),
    (1, 2, 5, 7, 64, True),
    (1, 2, 256, 256, 64, True),
    (2, 3, 300, 300, 64, True),
    (2, 3, 300, 300, 64, False),
    (1, 2, 200, 333, 64, False),
    (1, 2, 77, 333, 64, True),
    (1, 2, 640, 640, 64, True),
    (1, 1, 128, 128, 128, False),
    (1, 1, 1, 1, 128, True),
    (1, 2, 300, 300, 128, True),
    (1, 2, 200, 333, 128, False),
    (2, 2, 513, 513, 128, True),
]


@pytest.fixture(scope="module")
def fa():
    import exact_attention_31_gb300 as fa
    fa.lib()
    return fa


def _inputs(B, H, Nq, Nk, d, seed):
    from exact_attention_31_gb300.workloads import make_dout, make_qkv
    q, k, v, _ = make_qkv(B, H, Nq, Nk, d, seed, device="cuda")
    do = make_dout(B, H, Nq, d, seed, device="cuda")
    return q, k, v, do


def compare_grads(got, ref, what=""):
    out = {}
    for name, g, r in zip(("dq", "dk", "dv"), got, ref):
        g = to64(g).reshape(r.shape)
        assert np.all(np.isfinite(g)), f"{what}: non-finite {name}"
        err = np.abs(g - r)
        ref_max = float(np.abs(r).max())
        ref_mean = float(np.abs(r).mean())
        s = {"max": float(err.max()), "mean": float(err.mean()), "ref_max": ref_max, "ref_mean": ref_mean}
        out[name] = s
        if ref_max == 0.0:
            # e.g. dQ with a single visible key: P = 1 up to the rounding of L, so dS is rounding noise
            assert s["max"] <= 1e-5, f"{what}: {name} should be zero: {s}"
            continue
        assert s["max"] <= GRAD_MAX_REL * ref_max, f"{what}: {name} max err {s}"
        assert s["mean"] <= GRAD_MEAN_REL * ref_mean, f"{what}: {name} mean err {s}"
    return out


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: "b{}h{}q{}k{}d{}{}".format(*s[:5], "c" if s[5] else ""))
def test_backward_matches_oracle(fa, shape):
    B, H, Nq, Nk, d, causal = shape
    q, k, v, do = _inputs(B, H, Nq, Nk, d, seed=2000 + Nq + 7 * Nk + d)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_fwd(q, k, v, causal=causal, scale=scale)
    dq, dk, dv = fa.fattn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    ref = oracle.attention_backward(to64(q), to64(k), to64(v), to64(do), causal=causal, scale=scale)
    s = compare_grads((dq, dk, dv), ref, what=str(shape))
    print(shape, {n: (round(x["max"] / max(x["ref_max"], 1e-300), 5), round(x["mean"] / max(x["ref_mean"], 1e-300), 5))
                  for n, x in s.items()})


@pytest.mark.parametrize("d", [64, 128])
def test_backward_from_oracle_forward(fa, d):
    # The backward alone: O (rounded to bf16) and L come from the fp64 oracle.
    B, H, Nq, Nk, causal = 1, 2, 384, 384, True
    q, k, v, do = _inputs(B, H, Nq, Nk, d, seed=3100 + d)
    scale = 0.7 / math.sqrt(d)
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), causal=causal, scale=scale)
    o = torch.from_numpy(o_ref).to(torch.float32).to(torch.bfloat16).cuda()
    lse = torch.from_numpy(lse_ref).to(torch.float32).cuda()
    dq, dk, dv = fa.fattn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
    torch.cuda.synchronize()
    ref = oracle.attention_backward(to64(q), to64(k), to64(v), to64(do), causal=causal, scale=scale)
    compare_grads((dq, dk, dv), ref, what=f"oracle-forward d={d}")


def test_backward_repeat_and_dirty_workspace(fa):
    # The workspace's contents on entry do not matter; a second call gives the same dK and dV
    # (per-CTA sums, fixed order) and dQ within rounding of the accumulation order.
    B, H, Nq, Nk, d = 1, 2, 512, 512, 64
    q, k, v, do = _inputs(B, H, Nq, Nk, d, seed=3200)
    o, lse = fa.fattn_fwd(q, k, v, causal=True)
    ws = torch.full((fa.fattn_bwd_workspace_size(B, H, Nq, d),), 0x7F, dtype=torch.uint8, device="cuda")
    g1 = [t.clone() for t in fa.fattn_bwd(q, k, v, o, lse, do, causal=True, workspace=ws)]
    g2 = fa.fattn_bwd(q, k, v, o, lse, do, causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert torch.allclose(g1[0].float(), g2[0].float(), rtol=1e-2, atol=1e-3)
    ref = oracle.attention_backward(to64(q), to64(k), to64(v), to64(do), causal=True, scale=1 / 8)
    compare_grads(g2, ref, what="dirty workspace")


def test_backward_large_logits(fa):
    # Scores far from 0 (scaled by 6): P must come from L exactly, not overflow or underflow badly.
    B, H, Nq, Nk, d = 1, 2, 256, 384, 64
    q, k, v, do = _inputs(B, H, Nq, Nk, d, seed=3300)
    q = (q.float() * 6).to(torch.bfloat16)
    o, lse = fa.fattn_fwd(q, k, v, causal=True)
    dq, dk, dv = fa.fattn_bwd(q, k, v, o, lse, do, causal=True)
    torch.cuda.synchronize()
    ref = oracle.attention_backward(to64(q), to64(k), to64(v), to64(do), causal=True, scale=1 / 8)
    compare_grads((dq, dk, dv), ref, what="large logits")


def test_backward_workload_sampled(fa):
    # Full prefill workload B=1, H=32, N=8192, d=64, causal, in the launch configuration the
    # benchmark times; the oracle's gradients are computed for two whole heads.
    from exact_attention_31_gb300.workloads import WORKLOADS, make_dout, make_workload
    w = WORKLOADS["prefill_b1h32_n8192_d64"]
    q, k, v, _ = make_workload(w, device="cuda")
    do = make_dout(w.B, w.H, w.Nq, w.d, w.seed, device="cuda")
    o, lse = fa.fattn_fwd(q, k, v, causal=True, scale=w.scale)
    dq, dk, dv = fa.fattn_bwd(q, k, v, o, lse, do, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    heads = torch.tensor([0, 31], device="cuda")
    pick = lambda t: t.index_select(1, heads)  # noqa: E731
    ref = oracle.attention_backward(to64(pick(q)), to64(pick(k)), to64(pick(v)), to64(pick(do)), causal=True,
                                    scale=w.scale)
    compare_grads((pick(dq), pick(dk), pick(dv)), ref, what="workload heads 0 and 31")


def test_backward_partial_head_group_sampled(fa):
    # B1 H12 N8192 d128 causal: the backward's CTAs walk the heads in groups sized to stay in L2 (8
    # heads here), so the last group holds 4; heads 0 and 11 (first of the first group, last of the
    # partial one) are checked whole against the oracle.
    B, H, N, d = 1, 12, 8192, 128
    q, k, v, do = _inputs(B, H, N, N, d, seed=3400)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_fwd(q, k, v, causal=True, scale=scale)
    dq, dk, dv = fa.fattn_bwd(q, k, v, o, lse, do, causal=True, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    heads = torch.tensor([0, 11], device="cuda")
    pick = lambda t: t.index_select(1, heads)  # noqa: E731
    ref = oracle.attention_backward(to64(pick(q)), to64(pick(k)), to64(pick(v)), to64(pick(do)), causal=True,
                                    scale=scale)
    compare_grads((pick(dq), pick(dk), pick(dv)), ref, what="B1 H12 N8192 d128 heads 0 and 11")
