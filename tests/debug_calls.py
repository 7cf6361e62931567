"""Every entry point of the library on small seeded problems, for tests/test_debug_checks.py.

Run as a script with FATTN_DEBUG=1 in the environment, it makes the calls through the debug build
(libfattn_debug.so), reads the device-side checks' record, and saves the outputs and the record to
the file named on the command line; the test makes the same calls through the release build and
compares.  Shapes are small, ragged and cover every kernel: prefill at d = 64 and 128 (causal,
plain, band, element mask, several tiles and a ragged tail), the decode (default split, sliding
window, the allocation-free entry point), the backward (causal, plain, masked), FP8 at both head
dimensions and the host-buffer paths.
"""

import math
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def run(fa, dev):
    from exact_attention_31_gb300.workloads import make_dout, make_qkv, make_qkv_fp8

    out = {}

    def keep(name, *ts):
        out[name] = [t.detach().cpu().clone() for t in ts if t is not None]

    # prefill
    for d, causal, (B, H, Nq, Nk) in ((64, True, (1, 2, 384, 384)), (128, False, (2, 1, 200, 333)),
                                      (64, False, (1, 3, 129, 1000)), (128, True, (1, 2, 300, 520))):
        q, k, v, _ = make_qkv(B, H, Nq, Nk, d, 910 + d + Nq, dev)
        o, lse = fa.fattn_fwd(q, k, v, causal=causal, scale=1 / math.sqrt(d))
        keep(f"fwd_d{d}_{'causal' if causal else 'full'}_{Nq}x{Nk}", o, lse)
    q, k, v, _ = make_qkv(1, 2, 500, 700, 64, 931, dev)
    keep("fwd_band", *fa.fattn_fwd(q, k, v, scale=0.125, window=(150, 20)))
    g = torch.Generator(device=dev).manual_seed(932)
    mask = torch.rand((500, 700), generator=g, device=dev) < 0.4
    mask[:, 256:384] = False  # a hidden block column
    keep("fwd_mask", *fa.fattn_fwd(q, k, v, scale=0.125, causal=True, mask=fa.pack_mask(mask)))

    # decode
    q, k, v, _ = make_qkv(2, 3, 1, 1500, 128, 933, dev)
    keep("decode", *fa.fattn_decode(q, k, v, scale=1 / math.sqrt(128)))
    keep("decode_window", *fa.fattn_decode(q, k, v, scale=1 / math.sqrt(128), window=(200, 0)))
    keep("decode_static", *fa.fattn_decode_static(q, k, v, scale=1 / math.sqrt(128)))
    q, k, v, _ = make_qkv(1, 2, 1, 777, 64, 934, dev)
    keep("decode_d64", *fa.fattn_decode(q, k, v, scale=0.125, num_splits=5))

    # backward
    for d, causal, (B, H, Nq, Nk) in ((64, True, (1, 2, 256, 256)), (128, False, (1, 1, 200, 330)),
                                      (64, False, (2, 1, 130, 260))):
        q, k, v, _ = make_qkv(B, H, Nq, Nk, d, 935 + d + Nq, dev)
        do = make_dout(B, H, Nq, d, 936 + d, dev)
        o, lse = fa.fattn_fwd(q, k, v, causal=causal, scale=1 / math.sqrt(d))
        keep(f"bwd_d{d}_{'causal' if causal else 'full'}", *fa.fattn_bwd(q, k, v, o, lse, do, causal=causal,
                                                                          scale=1 / math.sqrt(d)))
    q, k, v, _ = make_qkv(1, 1, 300, 300, 64, 937, dev)
    do = make_dout(1, 1, 300, 64, 938, dev)
    m = torch.rand((300, 300), generator=g, device=dev) < 0.5
    words = fa.pack_mask(m)
    o, lse = fa.fattn_fwd(q, k, v, scale=0.125, mask=words)
    keep("bwd_mask", *fa.fattn_bwd(q, k, v, o, lse, do, scale=0.125, mask=words))

    # FP8
    for d in (64, 128):
        (q8, k8, v8), (qs, ks, vs), _ = make_qkv_fp8(1, 2, 300, 400, d, 939 + d, dev)
        keep(f"fp8_d{d}", *fa.fattn_fwd_fp8(q8, k8, v8, qs, ks, vs, causal=True, scale=1 / math.sqrt(d)))

    # host-buffer paths
    q, k, v, _ = make_qkv(1, 4, 256, 256, 64, 940, "cpu")
    o, lse = fa.fattn_fwd_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), causal=True, scale=0.125,
                               heads_per_chunk=2, device=dev)
    torch.cuda.synchronize(dev)
    keep("fwd_host", o, lse)
    q, k, v, _ = make_qkv(2, 2, 1, 900, 128, 941, "cpu")
    o, lse = fa.fattn_decode_host(q.pin_memory(), k.pin_memory(), v.pin_memory(), scale=1 / math.sqrt(128),
                                  heads_per_chunk=1, device=dev)
    torch.cuda.synchronize(dev)
    keep("decode_host", o, lse)
    torch.cuda.synchronize(dev)
    return out


if __name__ == "__main__":
    import exact_attention_31_gb300 as fa

    assert fa.fattn_debug_build(), "run with FATTN_DEBUG=1 after building libfattn_debug.so"
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    outs = run(fa, dev)
    rules, first = fa.fattn_debug_take()
    torch.save({"outs": outs, "rules": rules, "first": first, "last_error": fa.fattn_last_error()}, sys.argv[1])
