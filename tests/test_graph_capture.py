"""The device entry points can be captured in a CUDA graph (after one eager call has filled the
library's per-device caches) and replayed on new data in the same buffers; a replay gives what an
eager call on that data gives.  Small, launch-bound problems rely on this.
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


def _fill(dst, seed):
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, N, d = dst[0].shape[0], dst[0].shape[1], dst[1].shape[2], dst[0].shape[3]
    q, k, v, _ = make_qkv(B, H, dst[0].shape[2], N, d, seed, device="cuda")
    for t, s in zip(dst, (q, k, v)):
        t.copy_(s)


@pytest.mark.parametrize("B,H,N,d,causal", [(1, 1, 128, 64, False), (1, 8, 1024, 64, True), (2, 2, 300, 128, True)])
def test_forward_replays_on_new_data(fa, B, H, N, d, causal):
    bufs = [torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    o = torch.empty_like(bufs[0])
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    _fill(bufs, 8000)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fa.fattn_fwd(*bufs, causal=causal, out=o, lse=lse, stream=s)  # fills the per-device caches
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        for _ in range(3):
            fa.fattn_fwd(*bufs, causal=causal, out=o, lse=lse, stream=s)
    for seed in (8001, 8002):
        _fill(bufs, seed)
        g.replay()
        torch.cuda.synchronize()
        o_ref, l_ref = fa.fattn_fwd(*bufs, causal=causal)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
    assert fa.fattn_last_error() == 0


def test_decode_replays_on_new_data(fa):
    B, H, Nk, d = 4, 4, 2000, 128
    q = torch.empty((B, H, 1, d), dtype=torch.bfloat16, device="cuda")
    k, v = (torch.empty((B, H, Nk, d), dtype=torch.bfloat16, device="cuda") for _ in range(2))
    ws = torch.empty(fa.fattn_decode_workspace_size(B, H, Nk, d, 0), dtype=torch.uint8, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, 1), dtype=torch.float32, device="cuda")
    _fill([q, k, v], 8100)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fa.fattn_decode(q, k, v, workspace=ws, out=o, lse=lse, stream=s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fa.fattn_decode(q, k, v, workspace=ws, out=o, lse=lse, stream=s)
    _fill([q, k, v], 8101)
    g.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = fa.fattn_decode(q, k, v)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)


def test_backward_replays_on_new_data(fa):
    from exact_attention_31_gb300.workloads import make_dout
    B, H, N, d = 1, 2, 384, 64
    bufs = [torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    do = torch.empty_like(bufs[0])
    o = torch.empty_like(bufs[0])
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    grads = [torch.empty_like(bufs[0]) for _ in range(3)]
    ws = torch.empty(fa.fattn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")

    def run(stream):
        fa.fattn_fwd(*bufs, causal=True, out=o, lse=lse, stream=stream)
        fa.fattn_bwd(*bufs, o, lse, do, causal=True, workspace=ws, dq=grads[0], dk=grads[1], dv=grads[2],
                     stream=stream)

    _fill(bufs, 8200)
    do.copy_(make_dout(B, H, N, d, 8200, device="cuda"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        run(s)
    _fill(bufs, 8201)
    do.copy_(make_dout(B, H, N, d, 8201, device="cuda"))
    g.replay()
    torch.cuda.synchronize()
    o_ref, l_ref = fa.fattn_fwd(*bufs, causal=True)
    ref = fa.fattn_bwd(*bufs, o_ref, l_ref, do, causal=True)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref)
    # dK and dV have a fixed accumulation order; dQ's order across key tiles is not fixed
    assert torch.equal(grads[1], ref[1]) and torch.equal(grads[2], ref[2])
    rel = (grads[0].float() - ref[0].float()).abs().max() / ref[0].float().abs().max()
    assert rel < 1e-2
    assert math.isfinite(float(rel))


def _capture_and_replay(call, refill, check, reps=2):
    """Eager call (fills the caches), capture `call` twice into a graph on a side stream, then for
    each refill of the inputs replay it and let `check` compare against an eager call."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(s)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(s)
        call(s)
    for r in range(reps):
        refill(r)
        g.replay()
        torch.cuda.synchronize()
        check()


def test_element_mask_forward_and_backward_replay(fa):
    # the tile-summary kernel (and its memset) and the masked kernels in one graph
    from exact_attention_31_gb300.workloads import make_dout
    B, H, N, d = 1, 2, 400, 64
    bufs = [torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    do = torch.empty_like(bufs[0])
    o = torch.empty_like(bufs[0])
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    grads = [torch.empty_like(bufs[0]) for _ in range(3)]
    g = torch.Generator(device="cuda").manual_seed(8100)
    mask = fa.pack_mask(torch.rand((N, N), generator=g, device="cuda") < 0.4)
    mws = torch.empty(fa.fattn_mask_workspace_size(B, H, N, N), dtype=torch.uint8, device="cuda")
    bws = torch.empty(fa.fattn_bwd_mask_workspace_size(B, H, N, N, d), dtype=torch.uint8, device="cuda")

    def call(s):
        fa.fattn_fwd(*bufs, mask=mask, mask_workspace=mws, out=o, lse=lse, stream=s)
        fa.fattn_bwd(*bufs, o, lse, do, mask=mask, workspace=bws, dq=grads[0], dk=grads[1], dv=grads[2], stream=s)

    def refill(r):
        _fill(bufs, 8101 + r)
        do.copy_(make_dout(B, H, N, d, 8110 + r, device="cuda"))

    def check():
        o_ref, l_ref = fa.fattn_fwd(*bufs, mask=mask)
        ref = fa.fattn_bwd(*bufs, o_ref, l_ref, do, mask=mask)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)
        assert torch.equal(grads[1], ref[1]) and torch.equal(grads[2], ref[2])
        torch.testing.assert_close(grads[0].float(), ref[0].float(), rtol=1e-2, atol=2e-3)

    _capture_and_replay(call, refill, check)
    assert fa.fattn_last_error() == 0


@pytest.mark.parametrize("d", [64, 128])
def test_fp8_forward_replays(fa, d):
    # the V transpose and the FP8 kernel in one graph
    from exact_attention_31_gb300.workloads import make_qkv_fp8
    B, H, N = 1, 2, 333
    (q, k, v), (qs, ks, vs), _ = make_qkv_fp8(B, H, N, N, d, 8120, device="cuda")
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    ws = torch.empty(fa.fattn_fwd_fp8_workspace_size(B, H, N, d), dtype=torch.uint8, device="cuda")

    def call(s):
        fa.fattn_fwd_fp8(q, k, v, qs, ks, vs, causal=True, out=o, lse=lse, workspace=ws, stream=s)

    def refill(r):
        (q2, k2, v2), _, _ = make_qkv_fp8(B, H, N, N, d, 8121 + r, device="cuda")
        q.copy_(q2), k.copy_(k2), v.copy_(v2)

    def check():
        o_ref, l_ref = fa.fattn_fwd_fp8(q, k, v, qs, ks, vs, causal=True)
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, l_ref)

    _capture_and_replay(call, refill, check)


def test_allocation_free_decode_replays(fa):
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, Nk, d = 2, 4, 3000, 128
    q, k, v, _ = make_qkv(B, H, 1, Nk, d, 8130, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((B, H, 1), dtype=torch.float32, device="cuda")

    def call(s):
        fa.fattn_decode_static(q, k, v, out=o, lse=lse, stream=s)

    def refill(r):
        q2, k2, v2, _ = make_qkv(B, H, 1, Nk, d, 8131 + r, device="cuda")
        q.copy_(q2), k.copy_(k2), v.copy_(v2)

    def check():
        o_ref, l_ref = fa.fattn_decode(q, k, v)
        torch.cuda.synchronize()
        assert (o.float() - o_ref.float()).abs().max().item() <= 2e-3  # another split count
        assert (lse - l_ref).abs().max().item() <= 1e-4

    _capture_and_replay(call, refill, check)


def test_host_buffer_forward_replays(fa):
    # the host-buffer entry point's copies (on the library's own streams, ordered by events) and
    # kernels are captured into the caller's graph with them
    from exact_attention_31_gb300.workloads import make_qkv
    B, H, N, d = 1, 4, 256, 64
    hq, hk, hv = (torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory() for _ in range(3))
    ho = torch.empty((B, H, N, d), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = torch.empty(fa.fattn_fwd_host_workspace_size(B, H, N, N, d, 2), dtype=torch.uint8, device="cuda")

    def call(s):
        fa.fattn_fwd_host(hq, hk, hv, causal=True, out=ho, lse=hl, heads_per_chunk=2, workspace=ws,
                          device=torch.device("cuda", 0), stream=s)

    def refill(r):
        q, k, v, _ = make_qkv(B, H, N, N, d, 8140 + r, device="cpu")
        hq.copy_(q), hk.copy_(k), hv.copy_(v)

    def check():
        o_ref, l_ref = fa.fattn_fwd(hq.cuda(), hk.cuda(), hv.cuda(), causal=True)
        torch.cuda.synchronize()
        assert torch.equal(ho, o_ref.cpu()) and torch.equal(hl, l_ref.cpu())

    _capture_and_replay(call, refill, check)
