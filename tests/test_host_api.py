"""GPU checks of the host-buffer entry points (fattn_fwd_host, fattn_decode_host): each chunk of heads
runs the device kernels as its own problem, so the outputs must equal the device calls' outputs bit
for bit, whatever the chunking, for pinned and pageable host memory, and for calls enqueued back to
back on one workspace; and they must match the fp64 oracle.
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


def _host(t, pinned):
    h = t.cpu()
    return h.pin_memory() if pinned else h


FWD_CASES = [
    # B, H, Nq, Nk, d, band, heads_per_chunk, pinned
    (1, 32, 1024, 1024, 64, (-1, 0), 0, True),     # four chunks of eight heads
    (2, 3, 200, 333, 128, (100, 0), 4, True),      # chunks of 4, 2 heads in the last
    (1, 1, 77, 77, 64, (-1, -1), 0, True),         # a single chunk
    (1, 5, 300, 300, 64, (-1, 0), 1, False),       # pageable host memory, one head per chunk
    (2, 2, 333, 200, 128, (-1, 0), 3, True),       # rows above the diagonal see nothing
]


@pytest.mark.parametrize("case", FWD_CASES, ids=lambda c: "b{}h{}q{}k{}d{}w{}_{}c{}{}".format(
    *c[:5], *c[5], c[6], "p" if c[7] else "u"))
def test_fwd_host_equals_device_call(fa, case):
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, Nq, Nk, d, band, hpc, pinned = case
    q, k, v, _ = make_qkv(B, H, Nq, Nk, d, 7000 + Nq + Nk + d, device="cuda")
    o_dev, l_dev = fa.fattn_fwd(q, k, v, window=band)
    hq, hk, hv = (_host(t, pinned) for t in (q, k, v))
    o_h = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=pinned)
    l_h = torch.empty(q.shape[:3], dtype=torch.float32, pin_memory=pinned)
    fa.fattn_fwd_host(hq, hk, hv, window=band, heads_per_chunk=hpc, out=o_h, lse=l_h)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(l_h, l_dev.cpu())


def test_fwd_host_matches_oracle(fa):
    from exact_attention_31_gb300.workloads import make_qkv
    q, k, v, _ = make_qkv(2, 3, 257, 257, 64, 7100, device="cpu")
    o, lse = fa.fattn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True, heads_per_chunk=2)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), causal=True, scale=1 / math.sqrt(64))
    err = np.abs(to64(o) - o_ref)
    assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS
    assert np.abs(to64(lse) - lse_ref).max() <= LSE_MAX_ABS


def test_fwd_host_back_to_back_calls_share_a_workspace(fa):
    # Three calls on different inputs enqueued without a synchronisation in between: each call's
    # copies wait for the previous call's work, so every output is the one of its own inputs.
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, N, d = 1, 6, 384, 64
    ws = torch.empty(fa.fattn_fwd_host_workspace_size(B, H, N, N, d, 2), dtype=torch.uint8, device="cuda")
    runs = []
    for r in range(3):
        q, k, v, _ = make_qkv(B, H, N, N, d, 7200 + r, device="cuda")
        ref = fa.fattn_fwd(q, k, v, causal=True)
        out = fa.fattn_fwd_host(*(t.cpu().pin_memory() for t in (q, k, v)), causal=True, heads_per_chunk=2,
                                workspace=ws)
        runs.append((ref, out))
    torch.cuda.synchronize()
    for (o_d, l_d), (o_h, l_h) in runs:
        assert torch.equal(o_h, o_d.cpu()) and torch.equal(l_h, l_d.cpu())


DEC_CASES = [
    # B, H, Nk, d, window_left, heads_per_chunk, pinned
    (4, 8, 4096, 128, -1, 0, True),
    (2, 3, 1000, 64, 255, 2, True),       # only the last 256 keys are copied
    (1, 5, 300, 128, 5000, 0, False),     # window wider than the cache, pageable memory
    (3, 1, 65, 64, 0, 1, True),           # one visible key
]


@pytest.mark.parametrize("case", DEC_CASES, ids=lambda c: "b{}h{}k{}d{}w{}c{}{}".format(*c[:6], "p" if c[6] else "u"))
def test_decode_host_equals_device_call(fa, case):
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, Nk, d, wl, hpc, pinned = case
    q, k, v, _ = make_qkv(B, H, 1, Nk, d, 7300 + Nk + d + wl, device="cuda")
    window = None if wl < 0 else (wl, 0)
    o_dev, l_dev = fa.fattn_decode(q, k, v, window=window)
    o_h, l_h = fa.fattn_decode_host(*(_host(t, pinned) for t in (q, k, v)), window=window, heads_per_chunk=hpc)
    torch.cuda.synchronize()
    assert fa.fattn_last_error() == 0
    assert torch.equal(o_h, o_dev.cpu()) and torch.equal(l_h, l_dev.cpu())
    o_ref, lse_ref = oracle.attention(to64(q), to64(k), to64(v), window=(wl, 0), scale=1 / math.sqrt(d))
    assert np.abs(to64(o_h) - o_ref).max() <= O_MAX_ABS
    assert np.abs(to64(l_h) - lse_ref).max() <= LSE_MAX_ABS
