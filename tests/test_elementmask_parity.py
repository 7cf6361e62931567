"""GPU parity of the element-mask forward (fattn_fwd_mask) against the fp64 oracle.

A mask is elementwise and independent of the scores ("Understanding FlashAttention", Attention).  The
library takes it as a bit per (query, key) pair, shared or not over batch and heads, on top of the
band; whole 128 x 128 tiles it hides are skipped and only partly hidden tiles read the bits.  These
tests cover random masks of several densities, rows with no visible key, block-sparse patterns,
masks shared over heads and batch, the band combined with the mask, and identities with the
unmasked entry points, element by element against the oracle at the contract tolerances.
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


def _gen(B, H, Nq, Nk, d, seed):
    from exact_attention_31_gb300.workloads import make_qkv
    q, k, v, _ = make_qkv(B, H, Nq, Nk, d, seed, device="cuda")
    return q, k, v


def _check(o, lse, q, k, v, mask_bool, scale, window, what):
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), scale=scale, window=window, mask=mask_bool)
    o64, l64 = to64(o), to64(lse)
    empty = np.isneginf(lse_ref)
    assert np.array_equal(np.isneginf(l64), empty), what
    assert np.all(o64[empty] == 0.0), what
    err = np.abs(o64 - o_ref)
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (what, err.max(), err.mean())
    if (~empty).any():
        assert np.abs(l64[~empty] - lse_ref[~empty]).max() <= LSE_MAX_ABS, what
    return err


def _random_mask(shape, density, seed, device="cuda"):
    g = torch.Generator(device=device).manual_seed(seed)
    return torch.rand(shape, generator=g, device=device) < density


CASES = [
    # B, H, Nq, Nk, d, mask batch/head shape ("bh", "h1", "11"), density, band
    (1, 2, 300, 300, 64, "bh", 0.5, (-1, -1)),
    (2, 2, 513, 700, 128, "bh", 0.3, (-1, -1)),
    (1, 3, 128, 1000, 64, "11", 0.05, (-1, -1)),
    (2, 3, 260, 260, 64, "b1", 0.7, (-1, 0)),
    (1, 2, 777, 777, 128, "1h", 0.5, (-1, 0)),
    (1, 2, 400, 333, 64, "bh", 0.9, (63, 0)),
    (1, 1, 1, 129, 128, "bh", 0.5, (-1, -1)),
]


def _mask_shape(kind, B, H, Nq, Nk):
    return {"bh": (B, H, Nq, Nk), "b1": (B, 1, Nq, Nk), "1h": (1, H, Nq, Nk), "11": (Nq, Nk)}[kind]


@pytest.mark.parametrize("case", CASES, ids=lambda c: "b{}h{}q{}k{}d{}{}p{}w{}_{}".format(*c[:7], *c[7]))
def test_masked_forward_matches_oracle(fa, case):
    B, H, Nq, Nk, d, kind, density, band = case
    q, k, v = _gen(B, H, Nq, Nk, d, 5000 + Nq + Nk + d)
    mb = _random_mask(_mask_shape(kind, B, H, Nq, Nk), density, 5100 + Nq)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_fwd(q, k, v, scale=scale, window=band, mask=fa.pack_mask(mb))
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    _check(o, lse, q, k, v, mb.cpu().numpy(), scale, band, str(case))


@pytest.mark.parametrize("d", [64, 128])
def test_rows_with_no_visible_key(fa, d):
    B, H, N = 1, 2, 384
    q, k, v = _gen(B, H, N, N, d, 5200 + d)
    mb = _random_mask((B, H, N, N), 0.4, 5201)
    mb[0, 0, 10] = False           # a row of the first tile
    mb[0, 1, 200:260] = False      # rows across a tile boundary
    mb[0, 0, 256:] = False         # the last query tile sees nothing at all
    o, lse = fa.fattn_fwd(q, k, v, mask=fa.pack_mask(mb))
    torch.cuda.synchronize()
    _check(o, lse, q, k, v, mb.cpu().numpy(), 1 / math.sqrt(d), None, "empty rows")
    assert torch.all(o[0, 0, 256:] == 0) and torch.all(torch.isneginf(lse[0, 0, 256:]))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_block_sparse_mask(fa, d, causal):
    # 128 x 128 blocks wholly on or off (skipped), plus some blocks with a random pattern inside
    B, H, N = 1, 2, 1024
    q, k, v = _gen(B, H, N, N, d, 5300 + d + causal)
    g = torch.Generator(device="cuda").manual_seed(5301 + d)
    blocks = torch.rand((B, H, N // 128, N // 128), generator=g, device="cuda") < 0.4
    blocks[..., torch.arange(N // 128), torch.arange(N // 128)] = True  # every row sees its diagonal block
    mb = blocks.repeat_interleave(128, dim=2).repeat_interleave(128, dim=3)
    partial = torch.rand((B, H, N // 128, N // 128), generator=g, device="cuda") < 0.2
    noise = torch.rand((B, H, N, N), generator=g, device="cuda") < 0.5
    pm = partial.repeat_interleave(128, dim=2).repeat_interleave(128, dim=3)
    mb = torch.where(pm, mb & noise, mb)
    o, lse = fa.fattn_fwd(q, k, v, causal=causal, mask=fa.pack_mask(mb))
    torch.cuda.synchronize()
    _check(o, lse, q, k, v, mb.cpu().numpy(), 1 / math.sqrt(d), (-1, 0) if causal else None, "block sparse")


@pytest.mark.parametrize("d", [64, 128])
def test_mask_identities_with_unmasked_entry_points(fa, d):
    # an all-visible mask changes nothing, and a mask that spells out the causal band gives the causal
    # forward: the same tiles, the same arithmetic, the same bytes
    B, H, Nq, Nk = 2, 2, 300, 420
    q, k, v = _gen(B, H, Nq, Nk, d, 5400 + d)
    o0, l0 = fa.fattn_fwd(q, k, v)
    o1, l1 = fa.fattn_fwd(q, k, v, mask=fa.pack_mask(torch.ones((Nq, Nk), dtype=torch.bool, device="cuda")))
    assert torch.equal(o0, o1) and torch.equal(l0, l1)
    i = torch.arange(Nq, device="cuda")[:, None]
    j = torch.arange(Nk, device="cuda")[None, :]
    causal_bits = j <= i + (Nk - Nq)
    oc, lc = fa.fattn_fwd(q, k, v, causal=True)
    om, lm = fa.fattn_fwd(q, k, v, mask=fa.pack_mask(causal_bits))
    torch.cuda.synchronize()
    assert torch.equal(oc, om) and torch.equal(lc, lm)


def test_masked_rows_with_rising_scores_take_the_redo_phase(fa):
    # rows whose scores rise far above their first visible tile's, under a random mask
    from exact_attention_31_gb300.workloads import make_rising_scores
    B, H, N, d = 1, 2, 640, 64
    q, k, v = make_rising_scores(B, H, N, N, d, 5500, device="cuda")
    mb = _random_mask((B, H, N, N), 0.6, 5501)
    before = fa.fattn_fwd_recomputed_rows()
    o, lse = fa.fattn_fwd(q, k, v, mask=fa.pack_mask(mb))
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    assert fa.fattn_fwd_recomputed_rows() > before
    _check(o, lse, q, k, v, mb.cpu().numpy(), 1 / 8, None, "rising scores")


def test_mask_arguments_are_checked(fa):
    L = fa.lib()
    B, H, N, d = 1, 1, 256, 64
    q, k, v = _gen(B, H, N, N, d, 5600)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    words = fa.pack_mask(torch.ones((N, N), dtype=torch.bool, device="cuda"))
    ws = torch.empty(fa.fattn_mask_workspace_size(B, H, N, N), dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream

    def call(mask_ptr, sb, sh, ws_bytes):
        return L.fattn_fwd_mask(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, N, d,
                                mask_ptr, sb, sh, -1, -1, 0.125, ws.data_ptr(), ws_bytes, s)
    assert call(words.data_ptr(), 0, 0, ws.numel()) == 0
    assert call(None, 0, 0, ws.numel()) == 1                    # no mask
    assert call(words.data_ptr() + 4, 0, 0, ws.numel()) == 1    # misaligned
    assert call(words.data_ptr(), -4, 0, ws.numel()) == 1       # negative stride
    assert call(words.data_ptr(), 0, 6, ws.numel()) == 1        # stride not a multiple of 4 words
    assert call(words.data_ptr(), 0, 0, ws.numel() - 1) == 1    # short workspace
    torch.cuda.synchronize()
    assert fa.fattn_mask_row_words(1) == 4 and fa.fattn_mask_row_words(129) == 8 and fa.fattn_mask_row_words(0) == -1


# ------------------------------------------------------------------------------------------------
# Backward under the element mask (fattn_bwd_mask), at the backward's gradient tolerance: each
# gradient within 1.5e-2 of its own largest magnitude (max) and 5e-3 of its mean magnitude (mean).
# ------------------------------------------------------------------------------------------------
GRAD_MAX_REL = 1.5e-2
GRAD_MEAN_REL = 5e-3

BWD_CASES = [
    # B, H, Nq, Nk, d, mask kind, density, band
    (1, 2, 300, 300, 64, "bh", 0.5, (-1, -1)),
    (2, 2, 257, 400, 128, "b1", 0.3, (-1, -1)),
    (1, 3, 640, 640, 64, "11", 0.6, (-1, 0)),
    (1, 2, 513, 513, 128, "bh", 0.8, (-1, 0)),
    (1, 2, 384, 300, 64, "1h", 0.7, (100, 0)),
]


def _grads_close(grads, refs, what):
    for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
        e = np.abs(to64(g) - r)
        scale_max, scale_mean = np.abs(r).max(), np.abs(r).mean()
        if scale_max == 0.0:
            assert e.max() <= 1e-5, (what, name)
            continue
        assert e.max() <= GRAD_MAX_REL * scale_max and e.mean() <= GRAD_MEAN_REL * scale_mean, \
            (what, name, e.max(), scale_max, e.mean(), scale_mean)


@pytest.mark.parametrize("case", BWD_CASES, ids=lambda c: "b{}h{}q{}k{}d{}{}p{}w{}_{}".format(*c[:7], *c[7]))
def test_masked_backward_matches_oracle(fa, case):
    from exact_attention_31_gb300.workloads import make_dout
    B, H, Nq, Nk, d, kind, density, band = case
    q, k, v = _gen(B, H, Nq, Nk, d, 5700 + Nq + Nk + d)
    do = make_dout(B, H, Nq, d, 5700 + Nq, device="cuda")
    mb = _random_mask(_mask_shape(kind, B, H, Nq, Nk), density, 5800 + Nq)
    mb[..., 7, :] = False  # a row with no visible key (dq = 0 there)
    words = fa.pack_mask(mb)
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_fwd(q, k, v, scale=scale, window=band, mask=words)
    grads = fa.fattn_bwd(q, k, v, o, lse, do, scale=scale, window=band, mask=words)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    refs = oracle.attention_backward(to64(q), to64(k), to64(v), to64(do), scale=scale, window=band,
                                     mask=mb.cpu().numpy())
    _grads_close(grads, refs, str(case))
    assert torch.all(grads[0][..., 7, :] == 0)


@pytest.mark.parametrize("d", [64, 128])
def test_block_sparse_backward(fa, d):
    # whole 128 x 128 blocks hidden (skipped by every key tile), a few partial ones, causal band
    from exact_attention_31_gb300.workloads import make_dout
    B, H, N = 1, 2, 768
    q, k, v = _gen(B, H, N, N, d, 5900 + d)
    do = make_dout(B, H, N, d, 5900 + d, device="cuda")
    g = torch.Generator(device="cuda").manual_seed(5901 + d)
    blocks = torch.rand((B, H, N // 128, N // 128), generator=g, device="cuda") < 0.5
    blocks[..., torch.arange(N // 128), torch.arange(N // 128)] = True
    mb = blocks.repeat_interleave(128, dim=2).repeat_interleave(128, dim=3)
    partial = torch.rand((B, H, N // 128, N // 128), generator=g, device="cuda") < 0.25
    noise = torch.rand((B, H, N, N), generator=g, device="cuda") < 0.5
    mb = torch.where(partial.repeat_interleave(128, dim=2).repeat_interleave(128, dim=3), mb & noise, mb)
    words = fa.pack_mask(mb)
    o, lse = fa.fattn_fwd(q, k, v, causal=True, mask=words)
    grads = fa.fattn_bwd(q, k, v, o, lse, do, causal=True, mask=words)
    torch.cuda.synchronize()
    refs = oracle.attention_backward(to64(q), to64(k), to64(v), to64(do), causal=True, mask=mb.cpu().numpy())
    _grads_close(grads, refs, f"block sparse d={d}")


@pytest.mark.parametrize("d", [64, 128])
def test_masked_backward_identities(fa, d):
    # an all-visible mask and a mask spelling out the causal band give the unmasked backward's dk and
    # dv bit for bit (the same tiles and arithmetic); dq, accumulated in no fixed order, within rounding
    from exact_attention_31_gb300.workloads import make_dout
    B, H, Nq, Nk = 1, 2, 300, 420
    q, k, v = _gen(B, H, Nq, Nk, d, 6000 + d)
    do = make_dout(B, H, Nq, d, 6000 + d, device="cuda")
    i = torch.arange(Nq, device="cuda")[:, None]
    j = torch.arange(Nk, device="cuda")[None, :]
    for causal, bits in ((False, torch.ones((Nq, Nk), dtype=torch.bool, device="cuda")), (True, j <= i + (Nk - Nq))):
        o, lse = fa.fattn_fwd(q, k, v, causal=causal)
        g0 = fa.fattn_bwd(q, k, v, o, lse, do, causal=causal)
        g1 = fa.fattn_bwd(q, k, v, o, lse, do, mask=fa.pack_mask(bits))
        torch.cuda.synchronize()
        assert torch.equal(g0[1], g1[1]) and torch.equal(g0[2], g1[2]), causal
        assert (g0[0].float() - g1[0].float()).abs().max().item() <= 2 ** -7 * g0[0].float().abs().max().item()
