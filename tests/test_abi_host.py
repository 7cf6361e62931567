"""Host-side checks of the C ABI: the library loads, exports every declared symbol, and rejects bad
arguments before touching the GPU (these calls return before any CUDA call, so they run anywhere).
"""

import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fattn.h")


@pytest.fixture(scope="module")
def L():
    from exact_attention_31_gb300 import _build
    _build.build()
    import exact_attention_31_gb300 as fa
    return fa.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fattn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("fattn_fwd", "fattn_bwd", "fattn_bwd_workspace_size", "fattn_decode",
                     "fattn_decode_workspace_size", "fattn_status_string", "fattn_last_error",
                     "fattn_decode_num_splits"):
        assert required in names


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), f"libfattn.so does not export {name}"


def test_status_strings(L):
    import exact_attention_31_gb300 as fa
    assert fa.fattn_status_string(0) == "FATTN_OK"
    assert fa.fattn_status_string(4) == "FATTN_ERR_TIMEOUT"
    assert fa.fattn_status_string(99) == "FATTN_UNKNOWN_STATUS"


A = 4096  # a 16-byte-aligned fake address: never dereferenced, the checks reject the call first


@pytest.mark.parametrize("args,expect", [
    ((None, A, A, A, None, 1, 1, 8, 8, 64, 0, 0.125), 1),       # null q
    ((A, A, A, A + 2, None, 1, 1, 8, 8, 64, 0, 0.125), 1),      # misaligned o
    ((A, A, A, A, A + 1, 1, 1, 8, 8, 64, 0, 0.125), 1),         # misaligned lse
    ((A, A, A, A, None, 0, 1, 8, 8, 64, 0, 0.125), 1),          # B = 0
    ((A, A, A, A, None, 1, 1, 0, 8, 64, 0, 0.125), 1),          # Nq = 0
    ((A, A, A, A, None, 1, 1, 9, 8, 64, 1, 0.125), 1),          # causal with Nq > Nk
    ((A, A, A, A, None, 1, 1, 8, 8, 64, 2, 0.125), 1),          # causal flag not 0/1
    ((A, A, A, A, None, 1, 1, 8, 8, 64, 0, 0.0), 1),            # scale 0
    ((A, A, A, A, None, 1, 1, 8, 8, 64, 0, float("nan")), 1),   # scale NaN
    ((A, A, A, A, None, 1, 1, 8, 8, 64, 0, float("inf")), 1),   # scale inf
    ((A, A, A, A, None, 1, 1, 8, 8, 96, 0, 0.125), 2),          # d unsupported
    ((A, A, A, A, None, 1, 1, 8, 8, 32, 0, 0.125), 2),
])
def test_fwd_rejects_bad_arguments(L, args, expect):
    assert L.fattn_fwd(*args, None) == expect


def test_decode_split_resolution(L):
    # default: about 8 blocks of 64 keys per split, more splits while B H S < 8192, at most nblk
    assert L.fattn_decode_num_splits(32, 32, 16384, 0) == 32
    assert L.fattn_decode_num_splits(8, 32, 16384, 0) == 32
    assert L.fattn_decode_num_splits(4, 8, 32768, 0) == 256
    assert L.fattn_decode_num_splits(1, 32, 131072, 0) == 256
    assert L.fattn_decode_num_splits(1, 1, 16384, 0) == 256
    assert L.fattn_decode_num_splits(64, 256, 100000, 0) == 196
    assert L.fattn_decode_num_splits(1, 1, 65, 0) == 2
    assert L.fattn_decode_num_splits(1, 1, 1, 0) == 1
    assert L.fattn_decode_num_splits(1, 1, 1000, 16) == 16
    assert L.fattn_decode_num_splits(1, 1, 1000, 17) == -1
    assert L.fattn_decode_num_splits(1, 1, 0, 0) == -1
    assert L.fattn_decode_num_splits(1, 1, 100, -1) == -1
    assert L.fattn_decode_num_splits(0, 1, 100, 0) == -1


def test_decode_workspace_size(L):
    # one fp32 (m, l, O[d]) per (b, h, split), each array padded to 256 bytes
    def pad(x):
        return (x + 255) // 256 * 256
    # the default for B32 H32 Nk16384 is 32 splits (8 blocks of 64 keys each)
    assert L.fattn_decode_workspace_size(32, 32, 16384, 128, 0) == pad(32 * 32 * 32 * 128 * 4) + pad(32 * 32 * 32 * 2 * 4)
    assert L.fattn_decode_workspace_size(32, 32, 16384, 128, 256) == pad(32 * 32 * 256 * 128 * 4) + pad(32 * 32 * 256 * 2 * 4)
    assert L.fattn_decode_workspace_size(1, 1, 1, 64, 0) == 256 + 256
    assert L.fattn_decode_workspace_size(0, 1, 1, 64, 0) == 0
    assert L.fattn_decode_workspace_size(1, 1, 100, 64, 3) == 0


@pytest.mark.parametrize("args,expect", [
    ((None, A, A, A, None, 1, 1, 64, 64, 0.125, 0, A, 1 << 20), 1),
    ((A, A, A, A, None, 1, 1, 64, 64, 0.125, 0, None, 1 << 20), 1),     # no workspace
    ((A, A, A, A, None, 1, 1, 64, 64, 0.125, 0, A, 16), 1),             # workspace too small
    ((A, A, A, A, None, 1, 1, 64, 64, 0.125, 0, A + 8, 1 << 20), 1),    # misaligned workspace
    ((A, A, A, A, None, 1, 1, 0, 64, 0.125, 0, A, 1 << 20), 1),         # Nk = 0
    ((A, A, A, A, None, 1, 1, 64, 64, 0.125, 2, A, 1 << 20), 1),        # more splits than blocks
    ((A, A, A, A, None, 1, 1, 64, 64, -1.0, 0, A, 1 << 20), 1),         # negative scale
    ((A, A, A, A, None, 1, 1, 64, 80, 0.125, 0, A, 1 << 20), 2),        # d unsupported
])
def test_decode_rejects_bad_arguments(L, args, expect):
    assert L.fattn_decode(*args, None) == expect


def test_bwd_workspace_size(L):
    # fp32 dQ accumulator [B*H][Nq_pad][d] plus two [B*H][Nq_pad][16] bf16 term blocks, each padded to 256 B
    def pad(x):
        return (x + 255) // 256 * 256
    assert L.fattn_bwd_workspace_size(1, 32, 8192, 64) == pad(32 * 8192 * 64 * 4) + 2 * pad(32 * 8192 * 32)
    assert L.fattn_bwd_workspace_size(2, 3, 300, 128) == pad(6 * 384 * 128 * 4) + 2 * pad(6 * 384 * 32)
    assert L.fattn_bwd_workspace_size(1, 1, 1, 64) == pad(128 * 64 * 4) + 2 * pad(128 * 32)
    assert L.fattn_bwd_workspace_size(0, 1, 8, 64) == 0


W = 1 << 24  # a large-enough workspace size for the rejections below
BWD_OK = (A, A, A, A, A, A, A, A, A, 1, 1, 8, 8, 64, 0, 0.125, A, W)


def _bwd(**changes):
    names = ["q", "k", "v", "o", "lse", "dout", "dq", "dk", "dv", "B", "H", "Nq", "Nk", "d", "causal", "scale",
             "ws", "ws_bytes"]
    args = list(BWD_OK)
    for k, val in changes.items():
        args[names.index(k)] = val
    return tuple(args)


@pytest.mark.parametrize("args,expect", [
    (_bwd(q=None), 1),
    (_bwd(lse=None), 1),
    (_bwd(dout=None), 1),
    (_bwd(dk=A + 2), 1),                  # misaligned output
    (_bwd(lse=A + 2), 1),                 # misaligned lse
    (_bwd(ws=None), 1),
    (_bwd(ws=A + 16), 1),                 # workspace not 256-byte aligned
    (_bwd(ws_bytes=1024), 1),             # workspace too small
    (_bwd(Nq=0), 1),
    (_bwd(causal=1, Nq=9), 1),            # causal with Nq > Nk
    (_bwd(causal=3), 1),
    (_bwd(scale=0.0), 1),
    (_bwd(scale=float("nan")), 1),
    (_bwd(d=96), 2),
])
def test_bwd_rejects_bad_arguments(L, args, expect):
    assert L.fattn_bwd(*args, None) == expect


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    import exact_attention_31_gb300 as fa
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fattn_fwd(q, q, q)


def _align256(x):
    return (x + 255) // 256 * 256


@pytest.mark.parametrize("B,H,Nq,Nk,d,hpc,chunk", [(1, 32, 8192, 8192, 64, 0, 8), (2, 3, 100, 300, 128, 0, 2),
                                                   (1, 5, 64, 64, 64, 2, 2), (1, 1, 1, 1, 64, 0, 1)])
def test_fwd_host_workspace_size(L, B, H, Nq, Nk, d, hpc, chunk):
    # two slots, each holding Q, K, V, O (bf16) and L (fp32) of `chunk` heads, every part 256-aligned;
    # the default chunk is B*H/4 rounded up
    slot = (_align256(chunk * Nq * d * 2) + 2 * _align256(chunk * Nk * d * 2) + _align256(chunk * Nq * d * 2)
            + _align256(chunk * Nq * 4))
    assert L.fattn_fwd_host_workspace_size(B, H, Nq, Nk, d, hpc) == 2 * slot


def test_fwd_host_workspace_size_rejects(L):
    assert L.fattn_fwd_host_workspace_size(1, 4, 8, 8, 96, 0) == 0     # d
    assert L.fattn_fwd_host_workspace_size(1, 4, 8, 8, 64, 5) == 0     # more heads per chunk than heads
    assert L.fattn_fwd_host_workspace_size(1, 4, 8, 8, 64, -1) == 0
    assert L.fattn_fwd_host_workspace_size(0, 4, 8, 8, 64, 0) == 0


def test_decode_host_workspace_size_copies_only_visible_keys(L):
    # default chunk: B*H/8 rounded up; a window of the last 100 keys stages 100 keys per head
    full = L.fattn_decode_host_workspace_size(2, 8, 4096, 128, -1, 0)
    win = L.fattn_decode_host_workspace_size(2, 8, 4096, 128, 99, 0)
    chunk = 2
    kv_full, kv_win = 2 * _align256(chunk * 4096 * 128 * 2), 2 * _align256(chunk * 100 * 128 * 2)
    assert full - win == 2 * (kv_full - kv_win) + 2 * (_align256(L.fattn_decode_workspace_size(1, chunk, 4096, 128, 0))
                                                      - _align256(L.fattn_decode_workspace_size(1, chunk, 100, 128, 0)))
    assert L.fattn_decode_host_workspace_size(2, 8, 4096, 128, 5000, 0) == full  # window wider than the cache
    assert L.fattn_decode_host_workspace_size(2, 8, 4096, 128, -2, 0) == 0


@pytest.mark.parametrize("change,expect", [
    ({"q": None}, 1), ({"ws": A + 16}, 1), ({"ws_bytes": 1}, 1), ({"B": 0}, 1), ({"wl": -2}, 1),
    ({"scale": float("nan")}, 1), ({"hpc": 9}, 1), ({"d": 80}, 2),
])
def test_fwd_host_rejects_bad_arguments(L, change, expect):
    a = dict(q=A, k=A, v=A, o=A, lse=None, B=1, H=8, Nq=16, Nk=16, d=64, wl=-1, wr=0, scale=0.125, hpc=0,
             ws=A, ws_bytes=1 << 30)
    a.update(change)
    st = L.fattn_fwd_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nq"], a["Nk"], a["d"],
                          a["wl"], a["wr"], a["scale"], a["hpc"], a["ws"], a["ws_bytes"], None)
    assert st == expect


@pytest.mark.parametrize("change,expect", [
    ({"o": None}, 1), ({"ws": A + 8}, 1), ({"ws_bytes": 1}, 1), ({"Nk": 0}, 1), ({"wr": -2}, 1),
    ({"scale": -1.0}, 1), ({"hpc": -3}, 1), ({"d": 32}, 2),
])
def test_decode_host_rejects_bad_arguments(L, change, expect):
    a = dict(q=A, k=A, v=A, o=A, lse=None, B=2, H=4, Nk=300, d=128, wl=-1, wr=-1, scale=0.1, hpc=0,
             ws=A, ws_bytes=1 << 30)
    a.update(change)
    st = L.fattn_decode_host(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"], a["Nk"], a["d"],
                             a["wl"], a["wr"], a["scale"], a["hpc"], a["ws"], a["ws_bytes"], None)
    assert st == expect


def test_mask_row_words_and_workspace(L):
    # four 32-bit words per 128 keys, so every mask row starts on 16 bytes; the summary holds, per
    # head and per 128-row query tile (forward) or 128-key tile (backward), two sets of bits over the
    # other kind of tile in 64-bit words: the larger layout, padded to 256 bytes
    assert L.fattn_mask_row_words(1) == 4 and L.fattn_mask_row_words(128) == 4 and L.fattn_mask_row_words(129) == 8
    assert L.fattn_mask_row_words(0) == -1

    def summary(B, H, Nq, Nk):
        tq, tk = -(-Nq // 128), -(-Nk // 128)
        per_head = max(tq * 2 * -(-tk // 64), tk * 2 * -(-tq // 64)) * 8
        return -(-B * H * per_head // 256) * 256

    assert L.fattn_mask_workspace_size(2, 3, 300, 1000) == summary(2, 3, 300, 1000) == 768
    assert L.fattn_mask_workspace_size(1, 32, 8192, 8192) == summary(1, 32, 8192, 8192) == 32 * 64 * 16
    assert L.fattn_mask_workspace_size(1, 1, 128, 65536) == summary(1, 1, 128, 65536) == 512 * 16
    assert L.fattn_mask_workspace_size(1, 1, 0, 8) == 0


@pytest.mark.parametrize("mask,sb,sh,ws,nbytes,expect", [
    (None, 0, 0, A, 256, 1),    # no mask
    (A + 4, 0, 0, A, 256, 1),   # misaligned mask
    (A, -4, 0, A, 256, 1),      # negative stride
    (A, 0, 2, A, 256, 1),       # stride not a multiple of 4 words
    (A, 0, 0, None, 256, 1),    # no workspace
    (A, 0, 0, A, 255, 1),       # workspace too small
])
def test_fwd_mask_rejects_bad_arguments(L, mask, sb, sh, ws, nbytes, expect):
    L.fattn_fwd_mask.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_void_p, ctypes.c_longlong,
                                                                             ctypes.c_longlong, ctypes.c_int,
                                                                             ctypes.c_int, ctypes.c_float,
                                                                             ctypes.c_void_p, ctypes.c_size_t,
                                                                             ctypes.c_void_p]
    assert L.fattn_fwd_mask(A, A, A, A, None, 1, 1, 8, 8, 64, mask, sb, sh, -1, -1, 0.125, ws, nbytes, None) == expect
