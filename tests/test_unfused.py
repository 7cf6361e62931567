"""Standard attention in three kernels (include/fattn_unfused.h, libfattn_unfused.so): the baseline
whose device-memory traffic the fused forward is measured against ("Flash Attention: The Hidden Gem",
Background and Enter Flash Attention).  Host side: the library exports what its header declares and
rejects bad arguments before launching anything.  GPU side: its output against the oracle, element by
element, at the same tolerances as the fused forward (it rounds P to bf16 as the fused kernel does).
"""

import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fattn_unfused.h")


@pytest.fixture(scope="module")
def UL():
    from exact_attention_31_gb300 import _build
    _build.build_unfused()
    import exact_attention_31_gb300 as fa
    return fa.unfused_lib()


def declared():
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    return sorted(set(re.findall(r"\b(fattn_[a-z0-9_]+)\s*\(", text)))


def test_unfused_library_exports_its_header(UL):
    names = declared()
    assert names == ["fattn_fwd_unfused", "fattn_unfused_workspace_size"]
    for n in names:
        assert hasattr(UL, n)


def test_unfused_workspace_size(UL):
    # S fp32 and P bf16, [B, H, Nq, ld] each with ld = Nk rounded up to 8, each region 256-aligned
    def expect(B, H, Nq, Nk):
        ld = (Nk + 7) // 8 * 8
        r = B * H * Nq * ld
        return (r * 4 + 255) // 256 * 256 + (r * 2 + 255) // 256 * 256
    for shape in ((1, 1, 1, 1), (2, 3, 129, 1000), (1, 32, 8192, 8192), (4, 16, 2048, 2048), (1, 1, 5, 13)):
        assert UL.fattn_unfused_workspace_size(*shape) == expect(*shape), shape
    assert UL.fattn_unfused_workspace_size(0, 1, 1, 1) == 0


A = 4096  # a 16-byte-aligned fake address: the checks reject every call below before any CUDA call


@pytest.mark.parametrize("args,expect", [
    ((None, A, A, A, None, 1, 1, 8, 8, 64, 0, 0.125, A, 1 << 20), 1),   # null q
    ((A, A, A, A + 8, None, 1, 1, 8, 8, 64, 0, 0.125, A, 1 << 20), 1),  # misaligned o
    ((A, A, A, A, A + 2, 1, 1, 8, 8, 64, 0, 0.125, A, 1 << 20), 1),     # misaligned lse
    ((A, A, A, A, None, 1, 1, 9, 8, 64, 1, 0.125, A, 1 << 20), 1),      # causal with Nq > Nk
    ((A, A, A, A, None, 1, 1, 8, 8, 64, 0, -1.0, A, 1 << 20), 1),       # negative scale
    ((A, A, A, A, None, 1, 1, 8, 8, 60, 0, 0.125, A, 1 << 20), 2),      # d not a multiple of 8
    ((A, A, A, A, None, 1, 1, 8, 40000, 64, 0, 0.125, A, 1 << 40), 2),  # a score row over 32768 keys
    ((A, A, A, A, None, 1, 1, 8, 8, 64, 0, 0.125, A, 100), 1),          # workspace too small
    ((A, A, A, A, None, 1, 1, 8, 8, 64, 0, 0.125, None, 1 << 20), 1),   # no workspace
])
def test_unfused_rejects_bad_arguments(UL, args, expect):
    assert UL.fattn_fwd_unfused(*args, None) == expect


@pytest.mark.gpu
@pytest.mark.parametrize("B,H,Nq,Nk,d,causal", [
    (1, 2, 384, 384, 64, True),
    (2, 1, 200, 333, 128, False),   # Nk not a multiple of 8: padded score rows
    (1, 3, 129, 1000, 64, True),    # Nq < Nk, bottom-right causal
    (1, 1, 1, 77, 128, False),
    (1, 1, 5, 1, 64, False),
    (1, 2, 64, 4096, 128, True),
])
def test_unfused_matches_oracle(B, H, Nq, Nk, d, causal):
    import torch
    import exact_attention_31_gb300 as fa
    from exact_attention_31_gb300.workloads import make_qkv
    from parity_utils import compare, oracle_full
    q, k, v, _ = make_qkv(B, H, Nq, Nk, d, 960 + d + Nq, "cuda")
    scale = 1 / math.sqrt(d)
    o, lse = fa.fattn_fwd_unfused(q, k, v, causal=causal, scale=scale)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_full(q, k, v, causal, scale)
    compare(o, lse, o_ref, lse_ref, f"unfused {B}x{H}x{Nq}x{Nk} d{d} causal={causal}")


@pytest.mark.gpu
def test_unfused_workload_b1h8_n1024_d64_causal_and_workspace_contents():
    # the small prefill workload in full; the workspace then holds S (fp32) and P (bf16), checked
    # against the oracle's definitions on one head: S = scale q.k, P rows sum to 1, zero above the
    # diagonal
    import numpy as np
    import torch
    import exact_attention_31_gb300 as fa
    from exact_attention_31_gb300.workloads import make_qkv
    from parity_utils import compare, oracle_full, to64
    B, H, N, d = 1, 8, 1024, 64
    q, k, v, _ = make_qkv(B, H, N, N, d, 0xFA77E000 + 2, "cuda")
    scale = 0.125
    ws = torch.empty(fa.fattn_unfused_workspace_size(B, H, N, N), dtype=torch.uint8, device="cuda")
    o, lse = fa.fattn_fwd_unfused(q, k, v, causal=True, scale=scale, workspace=ws)
    torch.cuda.synchronize()
    o_ref, lse_ref = oracle_full(q, k, v, True, scale)
    compare(o, lse, o_ref, lse_ref, "unfused B1 H8 N1024 causal")
    S = ws[:B * H * N * N * 4].view(torch.float32).view(B, H, N, N)
    Pm = ws[(B * H * N * N * 4 + 255) // 256 * 256:][:B * H * N * N * 2].view(torch.bfloat16).view(B, H, N, N)
    s_ref = scale * to64(q[0, 3]) @ to64(k[0, 3]).T
    assert np.abs(to64(S[0, 3]) - s_ref).max() < 1e-4 * max(1.0, np.abs(s_ref).max())
    p = to64(Pm[0, 3])
    assert np.all(np.triu(p, 1) == 0)
    assert np.abs(p.sum(1) - 1).max() < 1e-2
