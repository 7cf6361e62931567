"""Seeded random sweep of shapes and masks through every compute entry point, against the oracle.

Each case draws B, H, Nq, Nk (not multiples of the 128-row tiles), d in {64, 128} and a band from a
fixed generator, runs the forward and the backward under that band and a windowed decode, and
compares element by element with the fp64 oracle at the tolerances of the dedicated parity tests.
The sizes stay small so that the oracle finishes in seconds.
"""

import math

import numpy as np
import pytest
import torch

import oracle
from parity_utils import to64
from test_backward_parity import compare_grads
from test_mask_parity import compare_masked

pytestmark = pytest.mark.gpu


def _cases(n=24, seed=0x5EED):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(n):
        B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
        Nq, Nk = int(rng.integers(1, 400)), int(rng.integers(1, 400))
        d = int(rng.choice([64, 128]))
        kind = int(rng.integers(0, 4))
        if kind == 0:
            band = (-1, -1)
        elif kind == 1:
            band = (-1, 0)
        elif kind == 2:
            band = (int(rng.integers(0, 300)), 0)
        else:
            band = (int(rng.integers(0, 200)), int(rng.integers(0, 200)))
        out.append((B, H, Nq, Nk, d, band))
    return out


@pytest.fixture(scope="module")
def fa():
    import exact_attention_31_gb300 as fa
    fa.lib()
    return fa


@pytest.mark.parametrize("case", _cases(), ids=lambda c: "b{}h{}q{}k{}d{}w{}_{}".format(*c[:5], *c[5]))
def test_random_shape_forward_backward(fa, case):
    from exact_attention_31_gb300.workloads import make_dout, make_qkv
    B, H, Nq, Nk, d, band = case
    seed = 6000 + 7 * Nq + 13 * Nk + d + band[0]
    q, k, v, _ = make_qkv(B, H, Nq, Nk, d, seed, device="cuda")
    do = make_dout(B, H, Nq, d, seed, device="cuda")
    scale = 0.9 / math.sqrt(d)
    o, lse = fa.fattn_fwd(q, k, v, window=band, scale=scale)
    grads = fa.fattn_bwd(q, k, v, o, lse, do, window=band, scale=scale)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), window=band, scale=scale)
    compare_masked(o, lse, o_ref, lse_ref, str(case))
    ref = oracle.attention_backward(to64(q), to64(k), to64(v), to64(do), window=band, scale=scale)
    compare_grads(grads, ref, what=str(case))


@pytest.mark.parametrize("case", _cases(8, seed=0xDEC0), ids=lambda c: "b{}h{}k{}d{}w{}".format(c[0], c[1], c[3], c[4], c[5][0]))
def test_random_shape_decode(fa, case):
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, _, Nk, d, band = case
    q, k, v, _ = make_qkv(B, H, 1, Nk, d, 6500 + Nk + d, device="cuda")
    scale = 1.0 / math.sqrt(d)
    o, lse = fa.fattn_decode(q, k, v, window=(band[0], 0), scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), window=(band[0], 0), scale=scale)
    compare_masked(o, lse, o_ref, lse_ref, f"decode {case}")
