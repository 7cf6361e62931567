"""Host-side logic of bench.py: work formulas, the traffic-evidence lookup and the clock summary."""

import os

import bench


def test_work_formulas():
    # 4 * B * H * N^2 * d, halved for causal
    assert bench.prefill_flops(1, 32, 8192, 64, True) == 274877906944.0
    assert bench.prefill_flops(4, 16, 2048, 128, False) == 4 * 4 * 16 * 2048 * 2048 * 128
    # K and V of the decode cache, bf16
    assert bench.decode_kv_bytes(32, 32, 16384, 128) == 8589934592
    # Q, K, V read and O written in bf16, L written in fp32
    assert bench.prefill_bytes(1, 32, 8192, 64) == 4 * 32 * 8192 * 64 * 2 + 32 * 8192 * 4


def test_recorded_traffic_tracks_the_kernel_source(tmp_path, monkeypatch):
    digest = bench.source_digest(bench.PREFILL_KERNEL_SRC)
    f = tmp_path / "traffic.txt"
    f.write_text(f"# comment\nprefill {digest} 123456\ndecode 0000000000000000 999\n")
    monkeypatch.setattr(bench, "TRAFFIC_FILE", str(f))
    assert bench.recorded_traffic("prefill") == 123456.0
    assert bench.recorded_traffic("decode") is None  # source changed since the capture


def test_committed_traffic_file_parses():
    assert os.path.exists(bench.TRAFFIC_FILE)
    with open(bench.TRAFFIC_FILE) as fh:
        kernels = [ln.split()[0] for ln in fh if ln.strip() and not ln.startswith("#")]
    assert sorted(kernels) == ["backward128", "backward64", "decode", "fp8", "fp8_64", "prefill", "unfused"]
    for k in kernels:  # every record names a kernel source the bench knows (a stale one reads as None)
        r = bench.recorded_traffic(k)
        assert r is None or r > 0, k


def test_clock_summary():
    row = lambda sm, hw="Not Active", cap="Not Active": ["0", str(sm), "2070", "900", "0x0", hw, "Not Active",
                                                         "Not Active", cap]
    samples = [(1.0, row(2070)), (2.0, row(2000)), (3.0, row(2070, cap="Active")), (9.0, row(100, hw="Active"))]
    s = bench.summarize_clocks(samples, 0.5, 3.5)
    assert s["sm_mhz"] == 2070 and s["sm_max_mhz"] == 2070 and s["samples"] == 3
    assert s["reasons"] == ["sw_power_cap"]
    # a timed region shorter than the sampling interval takes the nearest sample
    s = bench.summarize_clocks(samples, 8.9, 8.95)
    assert s["samples"] == 1 and s["reasons"] == ["hw_slowdown"]
    assert bench.summarize_clocks([], 0, 1)["sm_mhz"] is None


def test_visible_pairs_counts_the_band():
    # brute-force count of (i, j) with max(0, i - W + 1) <= j <= i
    for N, W in ((10, 4), (7, 7), (9, 20), (33, 1)):
        brute = sum(1 for i in range(N) for j in range(N) if i - (W - 1) <= j <= i)
        assert bench.visible_pairs(N, W - 1) == brute
    assert bench.visible_pairs(12) == 12 * 13 / 2
