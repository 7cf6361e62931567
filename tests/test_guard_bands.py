"""Guard bands and reruns for the outputs the prefill/decode tests do not cover: the backward's dQ,
dK and dV, the FP8 forward's O and L, and the element-masked forward's O and L.

Each output is a view into the middle of a larger buffer filled with a sentinel; after the call the
sentinel must be intact on both sides (no store lands outside the output), and the call run again
into fresh buffers must give the same bytes.  dK, dV and every forward output are bit-identical from
run to run (each is produced by one CTA in a fixed order); dQ is accumulated by fp32 TMA reduce-adds
from every key tile, whose arrival order varies, and is compared to a bf16 ulp.
"""

import math

import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fa():
    import exact_attention_31_gb300 as fa
    fa.lib()
    return fa


def guarded(shape, dtype, fill, pad=1024):
    n = math.prod(shape)
    big = torch.full((n + 2 * pad,), fill, dtype=dtype, device="cuda")
    return big, big[pad:pad + n].view(*shape)


def intact(big, n, fill, pad=1024):
    return bool(torch.all(big[:pad] == fill)) and bool(torch.all(big[pad + n:] == fill))


def test_backward_guard_bands_and_rerun(fa):
    from exact_attention_31_gb300.workloads import make_dout, make_qkv
    for d, causal, (B, H, Nq, Nk) in ((64, True, (1, 2, 300, 300)), (128, False, (2, 1, 190, 333))):
        q, k, v, _ = make_qkv(B, H, Nq, Nk, d, 950 + d, "cuda")
        do = make_dout(B, H, Nq, d, 951 + d, "cuda")
        scale = 1 / math.sqrt(d)
        o, lse = fa.fattn_fwd(q, k, v, causal=causal, scale=scale)
        fill = -12352.0
        bq, dq = guarded(q.shape, torch.bfloat16, fill)
        bk, dk = guarded(k.shape, torch.bfloat16, fill)
        bv, dv = guarded(v.shape, torch.bfloat16, fill)
        fa.fattn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale, dq=dq, dk=dk, dv=dv)
        torch.cuda.synchronize()
        for big, t, name in ((bq, dq, "dq"), (bk, dk, "dk"), (bv, dv, "dv")):
            assert intact(big, t.numel(), fill), f"d={d}: a store landed outside {name}"
        dq2, dk2, dv2 = fa.fattn_bwd(q, k, v, o, lse, do, causal=causal, scale=scale)
        torch.cuda.synchronize()
        assert torch.equal(dk, dk2) and torch.equal(dv, dv2), f"d={d}: dK/dV differ between runs"
        torch.testing.assert_close(dq2.float(), dq.float(), rtol=1e-2, atol=2e-3)


def test_fp8_guard_bands_and_rerun(fa):
    from exact_attention_31_gb300.workloads import make_qkv_fp8
    for d in (64, 128):
        (q, k, v), (qs, ks, vs), _ = make_qkv_fp8(1, 3, 260, 390, d, 952 + d, "cuda")
        bo, o = guarded((1, 3, 260, d), torch.bfloat16, -12352.0)
        bl, lse = guarded((1, 3, 260), torch.float32, -7.0, pad=64)
        fa.fattn_fwd_fp8(q, k, v, qs, ks, vs, causal=True, scale=1 / math.sqrt(d), out=o, lse=lse)
        torch.cuda.synchronize()
        assert intact(bo, o.numel(), -12352.0) and intact(bl, lse.numel(), -7.0, pad=64), f"d={d}"
        o2, lse2 = fa.fattn_fwd_fp8(q, k, v, qs, ks, vs, causal=True, scale=1 / math.sqrt(d))
        torch.cuda.synchronize()
        assert torch.equal(o, o2) and torch.equal(lse, lse2), f"FP8 d={d} differs between runs"


def test_element_mask_guard_bands_and_rerun(fa):
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, Nq, Nk, d = 2, 2, 333, 450, 64
    q, k, v, _ = make_qkv(B, H, Nq, Nk, d, 953, "cuda")
    g = torch.Generator(device="cuda").manual_seed(954)
    mask = torch.rand((B, 1, Nq, Nk), generator=g, device="cuda") < 0.3
    mask[0, 0, 17] = False  # a row that sees nothing
    words = fa.pack_mask(mask)
    bo, o = guarded((B, H, Nq, d), torch.bfloat16, -12352.0)
    bl, lse = guarded((B, H, Nq), torch.float32, -7.0, pad=64)
    fa.fattn_fwd(q, k, v, scale=0.125, mask=words, out=o, lse=lse)
    torch.cuda.synchronize()
    assert intact(bo, o.numel(), -12352.0) and intact(bl, lse.numel(), -7.0, pad=64)
    assert torch.all(o[0, :, 17] == 0) and torch.all(lse[0, :, 17] == -math.inf)
    o2, lse2 = fa.fattn_fwd(q, k, v, scale=0.125, mask=words)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, lse2)
