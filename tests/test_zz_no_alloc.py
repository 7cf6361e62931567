"""fattn_decode_static: the decode entry point for callers that cannot allocate device memory.

Some users of this library are handed only their inputs, outputs and a stream and may not call
cudaMalloc (a plugin inside a framework that owns every allocation, or a latency-critical path that
cannot afford an allocation's device synchronisation).  For them the library keeps the decode's
partial states in a fixed array compiled into the library.  These tests call that entry point
through the C ABI with raw device pointers and check it against fattn_decode, which uses a
caller-owned workspace, on consecutive calls with different shapes and inputs, and against the fp64
oracle on a shape whose split count has to shrink to fit the array.
This file is collected last on purpose.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

from parity_utils import LSE_MAX_ABS, O_MAX_ABS, O_MEAN_ABS

pytestmark = pytest.mark.gpu

STATIC_BYTES = 8 << 20  # FATTN_DECODE_STATIC_WORKSPACE_BYTES in include/fattn.h


def _raw_static_call(L, q, k, v, o, lse, scale, num_splits):
    vp = ctypes.c_void_p
    stream = vp(torch.cuda.current_stream().cuda_stream)
    B, H, Nk, d = k.shape
    return L.fattn_decode_static(vp(q.data_ptr()), vp(k.data_ptr()), vp(v.data_ptr()), vp(o.data_ptr()),
                                 vp(lse.data_ptr()), B, H, Nk, d, ctypes.c_float(scale), num_splits, stream)


def _close(o_a, l_a, o_b, l_b):
    err = (o_a.float() - o_b.float()).abs()
    assert err.max().item() <= O_MAX_ABS and err.mean().item() <= O_MEAN_ABS
    assert (l_a - l_b).abs().max().item() <= LSE_MAX_ABS


def test_static_workspace_decode_matches_workspace_decode():
    import exact_attention_31_gb300 as fa
    from exact_attention_31_gb300.workloads import make_qkv
    L = fa.lib()
    cases = [
        # B, H, Nk, d, num_splits.  The first fits the array at its default split count (32 splits of
        # 512 keys: 4.1 MiB of partial states); the last two are given split counts.
        (8, 32, 16384, 128, 0),
        (3, 5, 777, 64, 0),
        (2, 4, 3000, 128, 7),
    ]
    for n, (B, H, Nk, d, S) in enumerate(cases):
        q, k, v, _ = make_qkv(B, H, 1, Nk, d, seed=0x5EED + n, device="cuda")
        scale = 1.0 / math.sqrt(d)
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, 1), float("nan"), dtype=torch.float32, device="cuda")
        assert _raw_static_call(L, q, k, v, o, lse, scale, S) == 0
        torch.cuda.synchronize()
        o_ref, l_ref = fa.fattn_decode(q, k, v, scale=scale, num_splits=S)
        torch.cuda.synchronize()
        assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
        _close(o, lse, o_ref, l_ref)
        # same split count, same kernels: the results are identical
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
        # the same call again on the same inputs gives the same bytes (the array's leftovers from
        # the previous call do not leak into the result)
        o2 = torch.empty_like(q)
        lse2 = torch.empty_like(lse)
        assert _raw_static_call(L, q, k, v, o2, lse2, scale, S) == 0
        torch.cuda.synchronize()
        assert torch.equal(o2, o) and torch.equal(lse2, lse)


def test_static_workspace_decode_shrinks_the_split_count_to_fit():
    # The B32 H32 Nk16384 d128 decode: its default 32 splits need 16.6 MiB of partial states, so the
    # entry point lowers the count until they fit the 8 MiB array (15 splits).  The result must equal
    # fattn_decode with that count, match the fp64 oracle on sampled heads, and the calls after the
    # first must not change the device's free memory.
    import exact_attention_31_gb300 as fa
    import oracle
    from exact_attention_31_gb300.workloads import WORKLOADS, make_workload
    L = fa.lib()
    w = WORKLOADS["decode_b32h32_nk16384_d128"]
    q, k, v, _ = make_workload(w, "cuda")
    assert fa.fattn_decode_workspace_size(w.B, w.H, w.Nk, w.d, 0) > STATIC_BYTES
    fitted = None
    for S in range(fa.fattn_decode_num_splits(w.B, w.H, w.Nk, 0), 0, -1):
        if fa.fattn_decode_workspace_size(w.B, w.H, w.Nk, w.d, S) <= STATIC_BYTES:
            fitted = S
            break
    assert fitted == 15
    outs = [(torch.full_like(q, float("nan")), torch.full((w.B, w.H, 1), float("nan"), device="cuda"))
            for _ in range(3)]
    assert _raw_static_call(L, q, k, v, outs[0][0], outs[0][1], w.scale, 0) == 0
    torch.cuda.synchronize()
    free_before, _ = torch.cuda.mem_get_info()
    for o, lse in outs[1:]:
        assert _raw_static_call(L, q, k, v, o, lse, w.scale, 0) == 0
    torch.cuda.synchronize()
    free_after, _ = torch.cuda.mem_get_info()
    assert free_after == free_before
    for o, lse in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(lse, outs[0][1])
    o_ref, l_ref = fa.fattn_decode(q, k, v, scale=w.scale, num_splits=fitted)
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], o_ref) and torch.equal(outs[0][1], l_ref)
    rng = np.random.default_rng(7)
    pairs = [(0, 0), (w.B - 1, w.H - 1)] + [tuple(x) for x in rng.integers(0, [w.B, w.H], size=(14, 2))]
    o, lse = outs[0]
    for b, h in pairs:
        to64 = lambda t: t.detach().cpu().double().numpy()  # noqa: E731
        o_x, l_x = oracle.attention(to64(q[b:b + 1, h:h + 1]), to64(k[b:b + 1, h:h + 1]),
                                    to64(v[b:b + 1, h:h + 1]), causal=False, scale=w.scale)
        err = np.abs(to64(o[b, h]) - o_x[0, 0])
        assert err.max() <= O_MAX_ABS and err.mean() <= O_MEAN_ABS, (b, h, err.max())
        assert abs(float(lse[b, h, 0]) - l_x[0, 0, 0]) <= LSE_MAX_ABS, (b, h)


def test_static_workspace_decode_rejects_sizes_beyond_the_array():
    import exact_attention_31_gb300 as fa
    from exact_attention_31_gb300.workloads import make_qkv
    L = fa.lib()
    B, H, Nk, d = 8, 32, 16384, 128
    need = fa.fattn_decode_workspace_size(B, H, Nk, d, 256)
    assert need > STATIC_BYTES
    q, _, _, _ = make_qkv(B, H, 1, 128, d, seed=1, device="cuda")
    big_k = torch.empty((B, H, Nk, d), dtype=torch.bfloat16, device="cuda")
    o = torch.zeros_like(q)
    lse = torch.zeros((B, H, 1), dtype=torch.float32, device="cuda")
    # an explicit split count whose partial states do not fit: rejected, nothing launched or written
    assert _raw_static_call(L, q, big_k, big_k, o, lse, 0.1, 256) == 1
    torch.cuda.synchronize()
    assert torch.count_nonzero(o).item() == 0 and torch.count_nonzero(lse).item() == 0
    # and through the binding, a clear error
    with pytest.raises(fa.FattnError):
        fa.fattn_decode_static(q, big_k, big_k, num_splits=256)
