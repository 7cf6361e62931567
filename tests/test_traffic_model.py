"""The traffic and flop model against every table the page "FlashAttention: attention was never
compute-bound" prints (tests/golden/fa_io_traffic_tables.txt), digit for digit, and the algorithmic
bytes the benchmark takes from it.  CPU only."""

import os

import pytest

from exact_attention_31_gb300 import traffic as T

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "fa_io_traffic_tables.txt")


def tables():
    out = {}
    cur = None
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line.startswith("["):
                cur = line[1:line.index("]")]
                out[cur] = {"header": None, "rows": []}
            elif out[cur]["header"] is None:
                out[cur]["header"] = line.split()
            else:
                out[cur]["rows"].append(dict(zip(out[cur]["header"], line.split())))
    return out


TABLES = tables()
F = T.fmt_table_value
D = 64


def test_golden_file_holds_every_table():
    assert set(TABLES) == {"Where the time actually goes", "Tiling: same answer, flat memory",
                           "How big should a tile be?", "The backward pass: pay flops, save bytes",
                           "And no, it is not doing less arithmetic", "Now break it"}


def test_standard_attention_counts():
    for r in TABLES["Where the time actually goes"]["rows"]:
        n = int(r["n"])
        c = T.standard_forward(n, D)
        assert F(c.mb(), 2) == r["hbm_mb"], n
        assert F(c.gflops(), 3) == r["gflops"], n
        assert F(c.bytes_per_flop(), 3) == r["bytes_per_flop"], n
        assert F(100 * T.score_share(n, D), 1) + "%" == r["n2_share"], n


def test_tiled_attention_counts_and_flat_working_set():
    for r in TABLES["Tiling: same answer, flat memory"]["rows"]:
        n = int(r["n"])
        std, fl = T.standard_forward(n, D), T.tiled_forward(n, D, 64, 64)
        assert F(std.peak_elements * T.FP32 / T.KIB, 1) == r["std_peak_kb"], n
        assert F(fl.peak_elements * T.FP32 / T.KIB, 1) == r["flash_peak_kb"], n
        assert F(std.mb(), 2) == r["std_hbm_mb"], n
        assert F(fl.mb(), 2) == r["flash_hbm_mb"], n


def test_block_size_sweep():
    for r in TABLES["How big should a tile be?"]["rows"]:
        b = int(r["block"])
        c = T.tiled_forward(1024, D, b, b)
        kb = T.tile_working_set(b, b, D) * T.FP32 / T.KIB
        assert F(c.mb(), 2) == r["hbm_mb"], b
        assert F(kb, 1) == r["working_set_kb"], b
        assert ("yes" if kb <= 96 else "NO") == r["fits"], b
    assert F(T.standard_forward(1024, D).mb(), 2) == "17.00"


def test_backward_storage_and_flops():
    for r in TABLES["The backward pass: pay flops, save bytes"]["rows"]:
        n = int(r["n"])
        assert F(T.standard_backward_stored(n, D) * T.FP32 / T.MIB, 2) == r["std_stored_mb"], n
        assert F(T.tiled_backward_stored(n, D) * T.FP32 / T.MIB, 2) == r["flash_stored_mb"], n
        assert F(T.standard_backward_flops(n, D) / 1e9, 2) == r["std_gflops"], n
        assert F(T.tiled_backward_flops(n, D) / 1e9, 2) == r["flash_gflops"], n
        extra = T.tiled_backward_flops(n, D) / T.standard_backward_flops(n, D) - 1
        assert F(100 * extra, 0) + "%" == r["extra_flops"], n


def test_same_flops_only_traffic_moves():
    for r in TABLES["And no, it is not doing less arithmetic"]["rows"]:
        n = int(r["n"])
        std, fl = T.standard_forward(n, D), T.tiled_forward(n, D, 64, 64)
        assert F(std.gflops(), 3) == r["std_gflops"] and F(fl.gflops(), 3) == r["flash_gflops"], n
        assert F(std.mb(), 2) == r["std_hbm_mb"] and F(fl.mb(), 2) == r["flash_hbm_mb"], n
        assert F(std.elements / fl.elements, 1) + "x" == r["traffic_cut"], n


def test_keeping_the_full_score_matrix():
    r = TABLES["Now break it"]["rows"][0]
    assert F(T.tile_working_set(64, 64, D) * T.FP32 / T.KIB, 1) == r["flash_peak_kb"]
    assert F(1024 * 1024 * T.FP32 / T.KIB, 1) == r["full_s_kb"]


@pytest.mark.parametrize("mistake", ["s_once", "kv_per_key_tile", "no_score_tile", "no_recompute"])
def test_plausible_mistakes_miss_the_printed_figures(mistake):
    # Each variant drops or swaps one term of the counting rules; each must contradict a printed figure.
    n, d = 8192, D
    if mistake == "s_once":  # S written and read once, P never materialised
        assert F((2.0 * n * n + 4.0 * n * d) * 4 / T.MIB, 2) != "1032.00"
    elif mistake == "kv_per_key_tile":  # K/V re-read per key tile (Bc) and Q per key tile
        e = 2 * 1024 * d + 2 * 1024 * 1024 * d / 16
        assert F(e * 4 / T.MIB, 2) == "32.50"  # equal when Br = Bc ...
        e = 1024 * d * (1024 // 16) + 2 * 1024 * d + 1024 * d  # ... but Q per key tile is not
        assert F(e * 4 / T.MIB, 2) != "32.50"
    elif mistake == "no_score_tile":
        assert F((64 * d + 2 * 64 * d + 2 * 64) * 4 / T.KIB, 1) != "64.5"
    else:
        assert F(T.standard_backward_flops(2048, d) / 1e9, 2) != "3.22"


def test_masked_tiled_counts():
    # causal n = 256, Br = Bc = 64: query tile r visits key tiles 0..r, so K/V move 1+2+3+4 = 10 tiles
    c = T.tiled_forward_general(256, 256, 8, 64, 64, -1, 0)
    assert c.elements == 2 * 256 * 8 + 10 * 2 * 64 * 8
    assert c.flops == 10 * 4 * 64 * 64 * 8
    # a single-key band visits one key tile per query tile
    c = T.tiled_forward_general(256, 256, 8, 64, 64, 0, 0)
    assert c.elements == 2 * 256 * 8 + 4 * 2 * 64 * 8
    assert T.visible_pairs(256, 256, -1, 0) == 256 * 257 // 2
    assert T.visible_pairs(10, 4, -1, 0) == 10  # more queries than keys: the top rows see nothing
    assert T.visible_pairs(300, 300, 63, 0) == 64 * 65 // 2 + (300 - 64) * 64


def test_benchmark_algorithmic_bytes():
    # B1 H32 N8192 d64 causal: Q, K, V in and O out in bf16 (4 x 32 MiB) plus L (1 MiB)
    assert T.fused_forward_bytes(1, 32, 8192, 8192, 64) == 135266304
    # B32 H32 Nk16384 d128 decode: 8 GiB of cache plus q, O (bf16) and L
    assert T.decode_kv_bytes(32, 32, 16384, 128) == 8589934592
    assert T.decode_bytes(32, 32, 16384, 128) == 8589934592 + 2 * 32 * 32 * 128 * 2 + 32 * 32 * 4
    # without cache reuse the causal prefill of 256-row blocks re-reads K/V: far above the compulsory bytes
    assert T.fused_forward_reread_bytes(1, 1, 8192, 8192, 64, Br=256, window_right=0) > \
        4 * T.fused_forward_bytes(1, 1, 8192, 8192, 64)
    assert T.forward_flops(1, 32, 8192, 8192, 64, True) == 274877906944.0


def test_unfused_kernels_count_is_the_standard_count():
    # the three-kernel baseline's byte count, with every element in 4 bytes and no L, is the page's
    # standard column; with the library's types (S fp32, P bf16, bf16 tensors) it is what the
    # benchmark divides the unfused time by
    for r in TABLES["Where the time actually goes"]["rows"]:
        n = int(r["n"])
        b = T.unfused_forward_bytes(1, 1, n, n, D, s_bytes=4, p_bytes=4, elem_bytes=4, with_lse=False)
        assert F(b / T.MIB, 2) == r["hbm_mb"], n
    n, d = 8192, 64
    assert T.unfused_forward_bytes(1, 32, n, n, d) == 32 * (2 * n * d * 2 + 2 * n * n * 4 + 2 * n * n * 2
                                                            + 2 * n * d * 2 + 4 * n)
