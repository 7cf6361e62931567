#!/usr/bin/env python3
"""Benchmark of the exact-attention hot path on GB300.

One step is one pass of the whole path over one batch of synthetic input:
  1. the fused causal prefill forward, B=1, H=32, Nq=Nk=8192, d=64 (fattn_fwd), and
  2. one split-KV decode, B=32, H=32, Nq=1, Nk=16384, d=128 (fattn_decode: split + combine).
`value` is the prefill throughput in TFLOP/s (4*B*H*Nq*Nk*d, halved for causal) from CUDA events
around each prefill launch; the decode's KV-read bandwidth is reported beside it.  `roofline`
describes the step's dominant kernel by time (the decode's split kernel, HBM-bound);
`roofline_prefill` the prefill kernel (tensor-bound).  Before every
timed prefill the L2 is flushed by writing a 512 MiB buffer (the prefill inputs are smaller than
L2); the decode reads 8 GiB, which no cache holds.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU (replicas, no data-path
collective); the timed region is bracketed by a barrier and a device synchronize, the time is the
maximum over ranks, and rank 0 prints one JSON line.  `--impl reference` times the fp64 CPU oracle
on this host's cores on a bounded sample of the same workload (rank 0 only).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "attn fwd TFLOP/s & % BF16 tensor peak; decode KV GB/s vs HBM peak"
PREFILL = dict(name="prefill_b1h32_n8192_d64", B=1, H=32, N=8192, d=64, causal=True)
DECODE = dict(name="decode_b32h32_nk16384_d128", B=32, H=32, Nk=16384, d=128)
FLUSH_BYTES = 512 << 20
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
PREFILL_KERNEL_SRC = os.path.join(ROOT, "exact_attention_31_gb300", "csrc", "prefill_sm103a.cu")
DECODE_KERNEL_SRC = os.path.join(ROOT, "exact_attention_31_gb300", "csrc", "decode_sm103a.cu")
PREFILL_FP8_KERNEL_SRC = os.path.join(ROOT, "exact_attention_31_gb300", "csrc", "prefill_fp8_sm103a.cu")
BACKWARD_KERNEL_SRC = os.path.join(ROOT, "exact_attention_31_gb300", "csrc", "backward_sm103a.cu")
UNFUSED_SRC = os.path.join(ROOT, "exact_attention_31_gb300", "csrc", "unfused_sm103a.cu")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")


# ------------------------------------------------------------------------------------------------
# Algorithmic work per launch
# ------------------------------------------------------------------------------------------------
# The counting rules of the page's traffic counter ("FlashAttention: attention was never
# compute-bound"), pinned against its printed tables in tests/test_traffic_model.py.
from exact_attention_31_gb300 import traffic  # noqa: E402


def prefill_flops(B, H, N, d, causal):
    return traffic.forward_flops(B, H, N, N, d, causal)


def prefill_bytes(B, H, N, d):
    # read Q, K, V once, write O (bf16) and L (fp32): the tiled count with one query tile per head
    return traffic.fused_forward_bytes(B, H, N, N, d)


def visible_pairs(N, window_left=-1):
    """(query, key) pairs a causal prefill of N rows computes, with an optional sliding window of
    window_left + 1 keys (band (window_left, 0), Nq == Nk)."""
    if window_left < 0:
        return N * (N + 1) / 2
    W = window_left + 1
    if W >= N:
        return N * (N + 1) / 2
    return W * (W + 1) / 2 + (N - W) * W


# ex2 rate of one SM (GB300, measured by a microbenchmark: one warp instruction per 4 cycles per
# scheduler) and the GB300's maximum SM clock
EX2_PER_CLOCK_PER_SM = 32
MAX_SM_HZ = 2070e6
# Clock-based dense bf16 rate of one SM's tensor core (8192 FLOP per clock, tcgen05 M = 128 at full
# rate, measured by a microbenchmark) and the nominal HBM3e bandwidth: the second denominators the
# line reports beside the measured peaks (a copy and cuBLAS stop short of both).
TENSOR_FLOP_PER_CLOCK_PER_SM = 8192
NOMINAL_HBM_GBS = 7900.0


def clock_tensor_peak_tflops():
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return TENSOR_FLOP_PER_CLOCK_PER_SM * sms * MAX_SM_HZ / 1e12


def sfu_roofline(P, window_left, ms):
    """The d = 64 prefill's second bound: one ex2 per visible (query, key) pair against the SFU rate."""
    import torch
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    exps = P["B"] * P["H"] * visible_pairs(P["N"], window_left)
    achieved = exps / (ms * 1e-3) / 1e9
    peak = EX2_PER_CLOCK_PER_SM * sms * MAX_SM_HZ / 1e9
    return {"bound": "sfu (ex2)", "achieved": round(achieved, 1), "peak": round(peak, 1), "unit": "Gexp2/s",
            "frac": round(achieved / peak, 4), "exp2_per_launch": exps,
            "peak_source": f"{EX2_PER_CLOCK_PER_SM} ex2 per clock per SM x {sms} SMs x 2070 MHz (maximum SM clock)"}


def backward_flops(B, H, N, d, causal):
    # the five products of the backward (S, dP, dV, dK, dQ), 2*N*N*d each; half under the causal mask
    f = 10.0 * B * H * N * N * d
    return f / 2 if causal else f


def backward_bytes(B, H, N, d):
    # read Q, K, V, O, dO (bf16) and L; write dQ, dK, dV (bf16)
    return traffic.backward_bytes(B, H, N, N, d)


def decode_kv_bytes(B, H, Nk, d):
    return traffic.decode_kv_bytes(B, H, Nk, d)


def decode_bytes(B, H, Nk, d):
    # K and V once, q in, O out (bf16), L out (fp32)
    return traffic.decode_bytes(B, H, Nk, d)


# ------------------------------------------------------------------------------------------------
# Peaks, traffic evidence, clocks
# ------------------------------------------------------------------------------------------------
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {k: float(p[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


def source_digest(path):
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def recorded_traffic(kernel):
    """DRAM bytes per launch from the committed ncu summary, or None when the kernel source has
    changed since the counters were taken.  Lines: `<kernel> <source-sha16> <bytes_per_launch>`."""
    src = {"prefill": PREFILL_KERNEL_SRC, "decode": DECODE_KERNEL_SRC, "backward64": BACKWARD_KERNEL_SRC,
           "backward128": BACKWARD_KERNEL_SRC, "fp8": PREFILL_FP8_KERNEL_SRC, "fp8_64": PREFILL_FP8_KERNEL_SRC,
           "unfused": UNFUSED_SRC}[kernel]
    try:
        digest = source_digest(src)
        with open(TRAFFIC_FILE) as f:
            for line in f:
                parts = line.split()
                if len(parts) >= 3 and parts[0] == kernel and not line.startswith("#"):
                    return float(parts[2]) if parts[1] == digest else None
    except OSError:
        pass
    return None


class ClockSampler:
    """nvidia-smi sampled every 50 ms in the background; samples carry host timestamps."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu_id), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        return self

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0, t1):
        return summarize_clocks(self.samples, t0, t1)


def summarize_clocks(samples, t0, t1):
    inside = [s for t, s in samples if t0 <= t <= t1]
    note = "samples inside the timed region"
    if not inside and samples:
        mid = 0.5 * (t0 + t1)
        inside = [min(samples, key=lambda ts: abs(ts[0] - mid))[1]]
        note = "timed region shorter than the sampling interval: nearest sample"
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0}

    def num(x):
        try:
            return float(x)
        except ValueError:
            return None

    sm = [num(s[1]) for s in inside if num(s[1]) is not None]
    mx = [num(s[2]) for s in inside if num(s[2]) is not None]
    reasons = set()
    for s in inside:
        for name, val in zip(("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"), s[5:9]):
            if val.strip().lower() == "active":
                reasons.add(name)
    return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
            "reasons": sorted(reasons), "samples": len(inside), "note": note}


# ------------------------------------------------------------------------------------------------
# Distributed plumbing (replicas only)
# ------------------------------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world, backend):
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
    return dist if world > 1 else None


def max_over_ranks(x, dist, device):
    if dist is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------------------------------------
# CPU oracle timing (the reference arm and the cpu_baseline figure)
# ------------------------------------------------------------------------------------------------
def oracle_prefill_sample(q, k, v, budget_s, seed=0, threads=None):
    """Time the oracle on random query rows of the prefill workload until `budget_s` has passed,
    on `threads` host threads (default: all).  Returns (flops_done, seconds, rows_done, threads)."""
    import numpy as np
    import oracle
    B, H, N, d = q.shape
    qq = q.reshape(B * H, N, d)
    rng = np.random.default_rng(seed)
    threads = threads or oracle.default_threads()
    flops = 0.0
    rows_done = 0
    t_total = 0.0
    while t_total < budget_s:
        bh = int(rng.integers(0, B * H))
        rows = np.sort(rng.choice(N, size=min(N, 64 * threads), replace=False))
        qf = np.zeros((1, 1, N, d))
        qf[0, 0, rows] = qq[bh, rows]
        kf = k.reshape(B * H, N, d)[bh][None, None]
        vf = v.reshape(B * H, N, d)[bh][None, None]
        t0 = time.perf_counter()
        oracle.attention_rows(qf, kf, vf, rows, causal=True, scale=1 / math.sqrt(d), nthreads=threads)
        t_total += time.perf_counter() - t0
        flops += float(np.sum(4.0 * (rows + 1) * d))  # row i sees i + 1 keys
        rows_done += rows.size
    return flops, t_total, rows_done, threads


def oracle_decode_sample(q, k, v, budget_s, seed=1):
    """Time the oracle on (b, h) pairs of the decode workload; returns (kv_bytes, s, pairs, threads)."""
    import numpy as np
    import oracle
    B, H, Nk, d = k.shape
    rng = np.random.default_rng(seed)
    threads = oracle.default_threads()
    done = 0
    t_total = 0.0
    while t_total < budget_s and done < B * H:
        b, h = int(rng.integers(0, B)), int(rng.integers(0, H))
        qq, kk, vv = q[b:b + 1, h:h + 1], k[b:b + 1, h:h + 1], v[b:b + 1, h:h + 1]
        t0 = time.perf_counter()
        oracle.attention(qq, kk, vv, causal=False, scale=1 / math.sqrt(d), nthreads=threads)
        t_total += time.perf_counter() - t0
        done += 1
    return float(done * Nk * d * 2 * 2), t_total, done, threads


def host_inputs_f64(seed_prefill=0xFA77E004, seed_decode_pairs=0xFA77E005):
    """Seeded inputs for the CPU timing, drawn on the CPU (same recipe as the GPU inputs)."""
    import torch
    from exact_attention_31_gb300.workloads import make_qkv
    P, D = PREFILL, DECODE
    q, k, v, _ = make_qkv(P["B"], P["H"], P["N"], P["N"], P["d"], seed_prefill, "cpu")
    pf = [t.to(torch.float64).numpy() for t in (q, k, v)]
    # the decode sample needs only a few (b, h) pairs: draw a 2 x 2 slice of the same shape recipe
    q2, k2, v2, _ = make_qkv(2, 2, 1, D["Nk"], D["d"], seed_decode_pairs, "cpu")
    df = [t.to(torch.float64).numpy() for t in (q2, k2, v2)]
    return pf, df


def host_cpu():
    """The host the oracle ran on: its logical CPU count and model name (from /proc/cpuinfo, which
    names the part on x86 and gives the implementer and part numbers on Arm)."""
    info = {"cpu_count": os.cpu_count(), "machine": platform.machine()}
    try:
        with open("/proc/cpuinfo") as f:
            text = f.read()
        for key in ("model name", "Model name", "CPU implementer", "CPU part"):
            for line in text.splitlines():
                if line.split(":")[0].strip() == key:
                    info[key.lower().replace(" ", "_")] = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    return info


def cpu_baseline(budget_s=12.0):
    pf, df = host_inputs_f64()
    flops, secs, rows, threads = oracle_prefill_sample(*pf, budget_s=budget_s * 0.6)
    flops1, secs1, rows1, _ = oracle_prefill_sample(*pf, budget_s=budget_s * 0.15, seed=2, threads=1)
    kvb, dsecs, pairs, _ = oracle_decode_sample(*df, budget_s=budget_s * 0.25)
    return {
        "value": flops / secs / 1e12,
        "unit": "TFLOP/s",
        "cores": threads,
        "kind": "oracle",
        "sample": (f"{rows} random query rows of the causal B1 H32 N8192 d64 prefill ({flops / 1e9:.2f} "
                   f"GFLOP in {secs:.1f} s); decode: {pairs} (b,h) pairs of Nk=16384 d=128"),
        "decode_gbs": kvb / dsecs / 1e9,
        "value_1core": flops1 / secs1 / 1e12,
        "sample_1core": f"{rows1} random query rows of the same prefill on one host thread ({secs1:.1f} s)",
        "host": host_cpu(),
    }


# ------------------------------------------------------------------------------------------------
# The GPU arm
# ------------------------------------------------------------------------------------------------
def gpu_id_for_smi(dev):
    import torch
    props = torch.cuda.get_device_properties(dev)
    uuid = getattr(props, "uuid", None)
    if uuid is not None:
        u = str(uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
    ids = [x for x in vis.split(",") if x.strip()]
    return ids[dev.index] if dev.index < len(ids) else dev.index


def run_ours(args):
    import torch
    world, rank, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_attention_31_gb300 as fa
    from exact_attention_31_gb300.workloads import make_qkv
    fa.lib()

    P = dict(PREFILL, H=args.prefill_heads or PREFILL["H"])
    D = dict(DECODE, B=args.decode_batch or DECODE["B"])
    do_prefill = args.workload in ("both", "prefill")
    do_decode = args.workload in ("both", "decode")
    seed = 0xFA77E000
    stream = torch.cuda.current_stream(dev)
    scale_p, scale_d = 1 / math.sqrt(P["d"]), 1 / math.sqrt(D["d"])
    window = (args.window, 0) if args.window >= 0 else None
    if do_prefill:
        q, k, v, _ = make_qkv(P["B"], P["H"], P["N"], P["N"], P["d"], seed + 4, dev)
        o = torch.empty_like(q)
        lse = torch.empty((P["B"], P["H"], P["N"]), dtype=torch.float32, device=dev)
        flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    if do_decode:
        dq, dk, dv, _ = make_qkv(D["B"], D["H"], 1, D["Nk"], D["d"], seed + 5, dev)
        do = torch.empty_like(dq)
        dlse = torch.empty((D["B"], D["H"], 1), dtype=torch.float32, device=dev)
        ws = torch.empty(fa.fattn_decode_workspace_size(D["B"], D["H"], D["Nk"], D["d"], 0),
                         dtype=torch.uint8, device=dev)

    def step(evs=None):
        if do_prefill:
            flush.zero_()
            if evs is not None:
                evs[0].record(stream)
            fa.fattn_fwd(q, k, v, causal=True, scale=scale_p, out=o, lse=lse, stream=stream, window=window)
            if evs is not None:
                evs[1].record(stream)
        if do_decode:
            if evs is not None:
                evs[2].record(stream)
            fa.fattn_decode(dq, dk, dv, scale=scale_d, num_splits=0, workspace=ws, out=do, lse=dlse,
                            stream=stream)
            if evs is not None:
                evs[3].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.fattn_last_error() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout during warm-up")

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for_smi(dev)).start() if args.clocks else None
    if sampler is not None:
        time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    if sampler is not None:
        time.sleep(0.15)
        sampler.stop()
    if fa.fattn_last_error() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout in the timed region")

    total_ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    pre_avg = dec_avg = None
    if do_prefill:
        pre_avg = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps, dist, dev)
    if do_decode:
        dec_avg = max_over_ranks(sum(e[2].elapsed_time(e[3]) for e in evs) / args.steps, dist, dev)

    e2e = None
    if args.e2e_steps > 0:
        e2e = run_e2e(fa, dev, stream, args, q if do_prefill else None, k if do_prefill else None,
                      v if do_prefill else None, dq if do_decode else None, dk if do_decode else None,
                      dv if do_decode else None, scale_p, scale_d)
        if do_prefill:
            e2e["prefill_s"] = max_over_ranks(e2e["prefill_s"], dist, dev)
        if do_decode:
            e2e["decode_s"] = max_over_ranks(e2e["decode_s"], dist, dev)

    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    pf = prefill_flops(P["B"], P["H"], P["N"], P["d"], True)
    if args.window >= 0:
        pf = 4.0 * P["B"] * P["H"] * P["d"] * visible_pairs(P["N"], args.window)
    kv = decode_kv_bytes(D["B"], D["H"], D["Nk"], D["d"])
    line = {"metric": METRIC}
    if do_prefill:
        line.update(value=round(world * pf / (pre_avg * 1e-3) / 1e12, 2), unit="TFLOP/s")
    else:
        line.update(value=round(world * kv / (dec_avg * 1e-3) / 1e9, 1), unit="GB/s")
    name_p = f"prefill_b{P['B']}h{P['H']}_n{P['N']}_d{P['d']} causal"
    if args.window >= 0:
        name_p += f" sliding window {args.window + 1}"
    name_d = f"decode_b{D['B']}h{D['H']}_nk{D['Nk']}_d{D['d']}"
    workload = " + ".join(([name_p] if do_prefill else []) + ([name_d] if do_decode else []))
    line.update({
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(total_ms / args.steps, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic: seeded iid N(0,1) drawn in fp32 and rounded to bf16",
        "config": {
            "workload": workload,
            "l2": ("prefill inputs (96 MiB) are below L2, so a 512 MiB buffer is written before every "
                   "prefill (inside ms_per_step, outside the per-kernel events); the decode reads 8 GiB"),
            "parallelism": f"replicas x{world}",
            "seeds": {"prefill": hex(0xFA77E000 + 4), "decode": hex(0xFA77E000 + 5),
                      "generator": "torch.Generator per tensor; N(0,1) in fp32 rounded to bf16"},
        },
    })
    if do_prefill:
        per_launch = pf / (pre_avg * 1e-3) / 1e12
        line["config"]["prefill"] = {"B": P["B"], "H": P["H"], "Nq": P["N"], "Nk": P["N"], "d": P["d"],
                                     "causal": True, "scale": scale_p, "flops_per_launch": pf,
                                     "window": None if args.window < 0 else [args.window, 0]}
        line["prefill_ms"] = round(pre_avg, 4)
        line["roofline_prefill" if do_decode else "roofline"] = {
            "kernel": "prefill_kernel<64> (fattn_fwd)",
            "bound": "tensor", "achieved": round(per_launch, 2), "peak": peaks["bf16_tflops"],
            "unit": "TFLOP/s", "frac": round(per_launch / peaks["bf16_tflops"], 4),
            "peak_source": f"{peak_src} bf16 burst (cuBLAS bf16 GEMM)",
            "frac_of_clock_peak": round(per_launch / clock_tensor_peak_tflops(), 4),
            "clock_peak": round(clock_tensor_peak_tflops(), 1),
            "traffic": recorded_traffic("prefill"),
            "algorithmic_bytes": prefill_bytes(P["B"], P["H"], P["N"], P["d"]),
            "secondary": sfu_roofline(P, args.window, pre_avg),
        }
    if do_decode:
        dec_bw = decode_bytes(D["B"], D["H"], D["Nk"], D["d"]) / (dec_avg * 1e-3) / 1e9
        line["config"]["decode"] = {"B": D["B"], "H": D["H"], "Nq": 1, "Nk": D["Nk"], "d": D["d"],
                                    "causal": False, "num_splits": fa.fattn_decode_num_splits(D["B"], D["H"], D["Nk"], 0),
                                    "partial_states": "one (m, l, O) per split of about 512 keys (8 blocks of 64)",
                                    "kv_bytes_per_launch": kv}
        line["decode"] = {"value": round(world * kv / (dec_avg * 1e-3) / 1e9, 1), "unit": "GB/s",
                          "ms": round(dec_avg, 4), "frac_of_hbm": round(dec_bw / peaks["hbm_gbs"], 4)}
        rd = {
            "kernel": "decode_split_kernel<128> + decode_combine_kernel<128> (fattn_decode)",
            "bound": "hbm", "achieved": round(dec_bw, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(dec_bw / peaks["hbm_gbs"], 4), "peak_source": f"{peak_src} copy bandwidth",
            "frac_of_nominal_hbm": round(dec_bw / NOMINAL_HBM_GBS, 4), "nominal_hbm": NOMINAL_HBM_GBS,
            "traffic": recorded_traffic("decode"),
            "algorithmic_bytes": decode_bytes(D["B"], D["H"], D["Nk"], D["d"]),
        }
        # The step's dominant kernel by time is the decode's split kernel (about 78 % of the step in
        # the ncu launch list), so its roofline is the line's "roofline"; the prefill's sits beside it.
        line["roofline"] = rd
    if args.configs and do_prefill and window is None and rank == 0:
        line["configs_measured"] = measure_configs(fa, dev, stream, peaks)
    if args.configs and do_decode and rank == 0:
        # the decode with one partial state per 64-key block, the split the workload describes
        ws256 = torch.empty(fa.fattn_decode_workspace_size(D["B"], D["H"], D["Nk"], D["d"], 256), dtype=torch.uint8,
                            device=dev)
        ts = []
        for i in range(8):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fa.fattn_decode(dq, dk, dv, scale=scale_d, num_splits=256, workspace=ws256, out=do, lse=dlse, stream=stream)
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        ms256 = statistics.median(ts[2:])
        bw256 = decode_bytes(D["B"], D["H"], D["Nk"], D["d"]) / (ms256 * 1e-3) / 1e9
        line.setdefault("configs_measured", []).append(
            {"workload": name_d + " one partial state per 64-key block (num_splits 256)", "ms": round(ms256, 4),
             "gbs": round(bw256, 1), "frac": round(bw256 / peaks["hbm_gbs"], 4),
             "frac_of_nominal_hbm": round(bw256 / NOMINAL_HBM_GBS, 4),
             "method": "CUDA events per call, median of 6 after 2 warm calls (the 8 GiB cache exceeds L2)"})
        del ws256
    if args.rising and do_prefill and window is None and rank == 0:
        line["prefill_rising_scores"] = measure_rising_scores(fa, dev, stream, P, pre_avg, peaks)
    if args.configs and do_prefill and window is None and rank == 0:
        line["prefill_block_sparse_mask"] = measure_block_sparse(fa, dev, stream, P, q, k, v, o, lse, peaks)
        line["prefill_unfused_baseline"] = measure_unfused(fa, dev, stream, P, q, k, v, pre_avg, peaks)
    if args.cpu_budget > 0:
        line["cpu_baseline"] = cpu_baseline(budget_s=args.cpu_budget)
    if e2e is not None:
        if do_prefill:
            line["e2e"] = {"value": round(world * pf / e2e["prefill_s"] / 1e12, 3), "unit": "TFLOP/s"}
        else:
            line["e2e"] = {"value": round(world * kv / e2e["decode_s"] / 1e9, 1), "unit": "GB/s"}
        line["e2e"].update({"h2d_bytes_per_step": e2e["h2d"], "d2h_bytes_per_step": e2e["d2h"]})
        if do_prefill and do_decode:
            line["e2e"]["decode_gbs"] = round(world * kv / e2e["decode_s"] / 1e9, 1)
        line["e2e"]["how"] = ("the host-buffer C-ABI calls (fattn_fwd_host / fattn_decode_host) on pinned "
                              "host buffers: every step copies the inputs in and O and L out, in chunks of "
                              "heads overlapping the kernels; timed with CUDA events on the call's stream")
    line["gpu_launches"] = (int(do_prefill) + 2 * int(do_decode)) * args.steps
    line["clocks"] = sampler.summary(t0, t1) if sampler is not None else None
    print(json.dumps(line), flush=True)


def run_backward(args):
    """Time fattn_bwd (pre-pass, fused kernel, dQ pass) on the prefill workload's shape.  This is a
    line of its own, outside the benchmark step: the step is the forward hot path."""
    import torch
    world, rank, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_attention_31_gb300 as fa
    from exact_attention_31_gb300.workloads import make_dout, make_qkv
    fa.lib()
    P = dict(PREFILL, H=args.prefill_heads or PREFILL["H"], d=args.bwd_d or PREFILL["d"])
    B, H, N, d = P["B"], P["H"], P["N"], P["d"]
    seed = 0xFA77E000 + 4
    stream = torch.cuda.current_stream(dev)
    scale = 1 / math.sqrt(d)
    q, k, v, _ = make_qkv(B, H, N, N, d, seed, dev)
    do = make_dout(B, H, N, d, seed, dev)
    window = (args.window, 0) if args.window >= 0 else None
    o, lse = fa.fattn_fwd(q, k, v, causal=True, scale=scale, stream=stream, window=window)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.fattn_bwd_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(evs=None):
        flush.zero_()
        if evs is not None:
            evs[0].record(stream)
        fa.fattn_bwd(q, k, v, o, lse, do, causal=True, scale=scale, dq=dq, dk=dk, dv=dv, workspace=ws, window=window,
                     stream=stream)
        if evs is not None:
            evs[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.fattn_last_error() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for_smi(dev)).start() if args.clocks else None
    if sampler is not None:
        time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    if sampler is not None:
        time.sleep(0.15)
        sampler.stop()
    if fa.fattn_last_error() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout in the timed region")
    total_ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    avg = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps, dist, dev)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    fl = backward_flops(B, H, N, d, True)
    if args.window >= 0:
        fl = 10.0 * B * H * d * visible_pairs(N, args.window)
    tf = fl / (avg * 1e-3) / 1e12
    line = {
        "metric": "attn bwd TFLOP/s (fattn_bwd: pre-pass + fused kernel + dQ pass)",
        "value": round(world * tf, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded iid N(0,1) drawn in fp32 and rounded to bf16 (q, k, v, dO)",
        "config": {"workload": f"backward_b{B}h{H}_n{N}_d{d} causal" +
                               (f" sliding window {args.window + 1}" if args.window >= 0 else ""),
                   "backward": {"B": B, "H": H, "Nq": N, "Nk": N, "d": d, "causal": True, "scale": scale,
                                "flops_per_call": fl},
                   "l2": "a 512 MiB buffer is written before every call (outside the per-call events)",
                   "parallelism": f"replicas x{world}"},
        "bwd_ms": round(avg, 4),
        "roofline": {"kernel": f"fattn_bwd (bwd_prep_kernel<{d}> + bwd_kernel<{d}> + bwd_dq_kernel<{d}>)",
                     "bound": "tensor", "achieved": round(tf, 2), "peak": peaks["bf16_tflops"],
                     "unit": "TFLOP/s", "frac": round(tf / peaks["bf16_tflops"], 4),
                     "peak_source": f"{peak_src} bf16 burst (cuBLAS bf16 GEMM)",
                     "traffic": recorded_traffic(f"backward{d}") if (B, H, N) == (1, 32, 8192) else None,
                     "traffic_kernel": f"bwd_kernel<{d}> alone (ncu)",
                     "algorithmic_bytes": backward_bytes(B, H, N, d)},
        "gpu_launches": 3 * args.steps,
        "clocks": sampler.summary(t0, t1) if sampler is not None else None,
    }
    print(json.dumps(line), flush=True)


def run_fp8(args):
    """Time fattn_fwd_fp8 (V transpose + fused kernel) on B1 H32 N8192 causal, d 128 (or --fp8-d 64),
    with e4m3 inputs.
    A line of its own, outside the benchmark step: the step is the bf16 forward hot path."""
    import torch
    world, rank, local = dist_env()
    dist = init_dist(world, "nccl")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_attention_31_gb300 as fa
    from exact_attention_31_gb300.workloads import make_qkv_fp8
    fa.lib()
    B, H, N, d = 1, args.prefill_heads or 32, 8192, args.fp8_d or 128
    stream = torch.cuda.current_stream(dev)
    scale = 1 / math.sqrt(d)
    (q, k, v), (qs, ks, vs), _ = make_qkv_fp8(B, H, N, N, d, 0xFA77E000 + 6, dev)
    window = (args.window, 0) if args.window >= 0 else (-1, 0)
    o = torch.empty(q.shape, dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    ws = torch.empty(fa.fattn_fwd_fp8_workspace_size(B, H, N, d), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)

    def step(evs=None):
        flush.zero_()
        if evs is not None:
            evs[0].record(stream)
        fa.fattn_fwd_fp8(q, k, v, qs, ks, vs, window=window, scale=scale, out=o, lse=lse, workspace=ws, stream=stream)
        if evs is not None:
            evs[1].record(stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if fa.fattn_last_error() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout during warm-up")
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(gpu_id_for_smi(dev)).start() if args.clocks else None
    if sampler is not None:
        time.sleep(0.3)
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize(dev)
    t0 = time.time()
    start.record(stream)
    for i in range(args.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    t1 = time.time()
    if dist is not None:
        dist.barrier()
    if sampler is not None:
        time.sleep(0.15)
        sampler.stop()
    if fa.fattn_last_error() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout in the timed region")
    total_ms = max_over_ranks(start.elapsed_time(end), dist, dev)
    avg = max_over_ranks(sum(e[0].elapsed_time(e[1]) for e in evs) / args.steps, dist, dev)
    if rank != 0:
        return
    peaks, peak_src = load_peaks()
    pairs = visible_pairs(N, args.window) if args.window >= 0 else N * N / 2  # the causal convention
    fl = 4.0 * B * H * d * pairs
    tf = fl / (avg * 1e-3) / 1e12
    fp8_peak = 2 * peaks["bf16_tflops"]
    line = {
        "metric": "attn fwd TFLOP/s, FP8 e4m3 operands (fattn_fwd_fp8: V transpose + fused kernel)",
        "value": round(world * tf, 2), "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(total_ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "e4m3",
        "data": "synthetic: seeded iid N(0,1) rounded to bf16, then per-tensor e4m3 quantisation",
        "config": {"workload": f"prefill_fp8_b{B}h{H}_n{N}_d{d} causal" +
                               (f" sliding window {args.window + 1}" if args.window >= 0 else ""),
                   "fp8": {"B": B, "H": H, "Nq": N, "Nk": N, "d": d, "band": list(window), "scale": scale,
                           "descales": [qs, ks, vs], "flops_per_call": fl},
                   "l2": "a 512 MiB buffer is written before every call (outside the per-call events)",
                   "parallelism": f"replicas x{world}"},
        "fp8_ms": round(avg, 4),
        "roofline": {"kernel": f"fattn_fwd_fp8 (fwd_fp8_vt_kernel<{d}> + prefill_fp8_kernel<{d}>)", "bound": "tensor",
                     "achieved": round(tf, 2), "peak": fp8_peak, "unit": "TFLOP/s", "frac": round(tf / fp8_peak, 4),
                     "peak_source": f"{peak_src} bf16 burst (cuBLAS bf16 GEMM) x 2, the nominal fp8:bf16 ratio",
                     "traffic": recorded_traffic("fp8" if d == 128 else "fp8_64")
                     if (B, H, N) == (1, 32, 8192) and args.window < 0 else None,
                     "traffic_kernel": "prefill_fp8_kernel alone (ncu)",
                     "algorithmic_bytes": traffic.fp8_forward_bytes(B, H, N, N, d)},
        "gpu_launches": 2 * args.steps,
        "clocks": sampler.summary(t0, t1) if sampler is not None else None,
    }
    print(json.dumps(line), flush=True)


def measure_configs(fa, dev, stream, peaks, iters=50):
    """TFLOP/s of the smaller prefill configurations (single head N128, B1 H8 N1024 causal, B4 H16
    N2048 d128 with 1 % of query rows x8, without and with the causal mask).  These are launch-bound,
    so each is timed as a CUDA graph of `iters` launches, each after a 512 MiB write that flushes L2,
    minus a graph of the writes alone, with CUDA events around the replays (median of 5).  Measured
    outside the benchmark's timed region; the line's `value` stays the N8192 prefill."""
    import torch
    from exact_attention_31_gb300.workloads import WORKLOADS, make_workload
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    side = torch.cuda.Stream(dev)

    def graph_ms(body):
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            body()  # eager once: fills the library's per-device caches before capture
        stream.wait_stream(side)
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=side):
            for _ in range(iters):
                body()
        ts = []
        for _ in range(6):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            g.replay()
            e1.record(stream)
            e1.synchronize()
            ts.append(e0.elapsed_time(e1))
        ts = sorted(ts[1:])
        return ts[len(ts) // 2]

    flush_ms = graph_ms(lambda: flush.zero_())
    out = []
    for name in ("prefill_b1h1_n128_d64", "prefill_b1h8_n1024_d64", "prefill_b4h16_n2048_d128"):
        w = WORKLOADS[name]
        q, k, v, _ = make_workload(w, dev)
        o, lse = torch.empty_like(q), torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
        for causal in w.causal:
            flops = 4.0 * w.B * w.H * w.Nq * w.Nk * w.d / (2 if causal else 1)

            def body():
                flush.zero_()
                fa.fattn_fwd(q, k, v, causal=causal, scale=w.scale, out=o, lse=lse)

            ms = max(graph_ms(body) - flush_ms, 1e-6) / iters
            tf = flops / (ms * 1e-3) / 1e12
            out.append({"workload": name + (" causal" if causal else ""), "ms": round(ms, 5),
                        "tflops": round(tf, 2), "frac": round(tf / peaks["bf16_tflops"], 4)})
        del q, k, v, o, lse
    out.append({"method": f"CUDA graph of {iters} launches, each after a 512 MiB L2-flush write, minus a graph "
                          f"of the writes alone; median of 5 replays"})
    return out


def measure_rising_scores(fa, dev, stream, P, normal_ms, peaks, iters=10):
    """The benchmark prefill's shape on inputs whose scores rise by about 150 log2-units after the
    first 128 keys (every key after the first tile is a large one), so that every query tile but
    each head's first fails the fast path's range check and is computed again with a running max:
    the cost of the redo phase at its worst.  Timed like the benchmark prefill (L2 flushed before
    each launch, CUDA events per launch, mean of `iters`), outside the benchmark's timed region."""
    import torch
    from exact_attention_31_gb300.workloads import make_rising_scores
    B, H, N, d = P["B"], P["H"], P["N"], P["d"]
    q, k, v = make_rising_scores(B, H, N, N, d, 0xFA77E000 + 7, dev, large_from=128)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    scale = 1 / math.sqrt(d)
    before = fa.fattn_fwd_recomputed_rows()
    fa.fattn_fwd(q, k, v, causal=True, scale=scale, out=o, lse=lse, stream=stream)
    torch.cuda.synchronize(dev)
    rows = fa.fattn_fwd_recomputed_rows() - before
    for _ in range(2):
        fa.fattn_fwd(q, k, v, causal=True, scale=scale, out=o, lse=lse, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        fa.fattn_fwd(q, k, v, causal=True, scale=scale, out=o, lse=lse, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    if fa.fattn_last_error() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout on the rising-score inputs")
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / iters
    tf = prefill_flops(B, H, N, d, True) / (ms * 1e-3) / 1e12
    return {"workload": f"prefill_b{B}h{H}_n{N}_d{d} causal, scores rising ~150 log2-units after key 127",
            "rows_failing_range_check": rows, "rows_total": B * H * N, "ms": round(ms, 4),
            "tflops": round(tf, 2), "frac": round(tf / peaks["bf16_tflops"], 4),
            "time_vs_normal_inputs": round(ms / normal_ms, 3)}


def measure_block_sparse(fa, dev, stream, P, q, k, v, o, lse, peaks, iters=10):
    """The benchmark prefill under an element mask shared by every head: causal, with half of the
    128 x 128 blocks below the diagonal hidden (seeded), the diagonal blocks visible, and one block in
    eight with a random pattern inside.  TFLOP/s counts the visible (query, key) pairs only (4 d flops
    each); the time includes the tile-summary pass.  Outside the benchmark's timed region."""
    import torch
    N, d = P["N"], P["d"]
    T = N // 128
    g = torch.Generator(device=dev).manual_seed(0xFA77E000 + 8)
    blocks = torch.rand((T, T), generator=g, device=dev) < 0.5
    blocks[torch.arange(T), torch.arange(T)] = True
    partial = torch.rand((T, T), generator=g, device=dev) < 0.125
    mb = blocks.repeat_interleave(128, 0).repeat_interleave(128, 1)
    noise = torch.rand((N, N), generator=g, device=dev) < 0.5
    mb = torch.where(partial.repeat_interleave(128, 0).repeat_interleave(128, 1), mb & noise, mb)
    mb &= torch.ones((N, N), dtype=torch.bool, device=dev).tril()
    visible = float(mb.sum().item()) * P["B"] * P["H"]
    words = fa.pack_mask(mb)
    del mb, noise
    ws = torch.empty(fa.fattn_mask_workspace_size(P["B"], P["H"], N, N), dtype=torch.uint8, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    scale = 1 / math.sqrt(d)
    for _ in range(3):
        fa.fattn_fwd(q, k, v, causal=True, scale=scale, out=o, lse=lse, mask=words, mask_workspace=ws, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        fa.fattn_fwd(q, k, v, causal=True, scale=scale, out=o, lse=lse, mask=words, mask_workspace=ws, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / iters
    tf = 4.0 * d * visible / (ms * 1e-3) / 1e12
    return {"workload": f"prefill_b{P['B']}h{P['H']}_n{N}_d{d} causal, one element mask for all heads: half of "
                        "the 128x128 blocks below the diagonal hidden, 1 in 8 with random bits inside",
            "visible_pairs": visible, "ms": round(ms, 4), "tflops_visible": round(tf, 2),
            "frac": round(tf / peaks["bf16_tflops"], 4)}


def measure_unfused(fa, dev, stream, P, q, k, v, fused_ms, peaks, iters=10):
    """The same prefill computed as standard attention in three kernels (fattn_fwd_unfused: a cuBLAS
    GEMM writing S in fp32, the softmax kernel writing P in bf16, a cuBLAS GEMM for O), with the L2
    flushed before each call as for the fused launch.  Outside the benchmark's timed region; the
    comparison the pages' memory-traffic argument is about."""
    import torch
    B, H, N, d = P["B"], P["H"], P["N"], P["d"]
    ws = torch.empty(fa.fattn_unfused_workspace_size(B, H, N, N), dtype=torch.uint8, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    scale = 1 / math.sqrt(d)
    for _ in range(3):
        fa.fattn_fwd_unfused(q, k, v, causal=True, scale=scale, out=o, lse=lse, workspace=ws, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(iters)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        fa.fattn_fwd_unfused(q, k, v, causal=True, scale=scale, out=o, lse=lse, workspace=ws, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / iters
    fl = prefill_flops(B, H, N, d, True)
    ub = traffic.unfused_forward_bytes(B, H, N, N, d)
    fb = prefill_bytes(B, H, N, d)
    del ws
    return {"workload": f"prefill_b{B}h{H}_n{N}_d{d} causal as standard attention in three kernels "
                        "(cuBLAS GEMM -> S fp32, unfused_softmax_kernel -> P bf16 and L, cuBLAS GEMM -> O)",
            "ms": round(ms, 4), "tflops": round(fl / (ms * 1e-3) / 1e12, 2),
            "time_vs_fused": round(ms / fused_ms, 2),
            "algorithmic_bytes": ub, "algorithmic_bytes_fused": fb, "bytes_vs_fused": round(ub / fb, 1),
            "achieved_gbs_of_algorithmic_bytes": round(ub / (ms * 1e-3) / 1e9, 1),
            "frac_hbm": round(ub / (ms * 1e-3) / 1e9 / peaks["hbm_gbs"], 4),
            "traffic_unfused_kernels": recorded_traffic("unfused") if H == 32 else None}


def run_unfused(args):
    """The fused prefill and the three-kernel standard attention on the prefill workload's shape, one
    after the other (for the ncu capture of their DRAM traffic; --prefill-heads shrinks it)."""
    import torch
    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    import exact_attention_31_gb300 as fa
    from exact_attention_31_gb300.workloads import make_qkv
    fa.lib()
    P = dict(PREFILL, H=args.prefill_heads or PREFILL["H"])
    B, H, N, d = P["B"], P["H"], P["N"], P["d"]
    stream = torch.cuda.current_stream(dev)
    q, k, v, _ = make_qkv(B, H, N, N, d, 0xFA77E000 + 4, dev)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    flush = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
    scale = 1 / math.sqrt(d)
    for _ in range(args.warmup):
        fa.fattn_fwd(q, k, v, causal=True, scale=scale, out=o, lse=lse, stream=stream)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    for e0, e1 in evs:
        flush.zero_()
        e0.record(stream)
        fa.fattn_fwd(q, k, v, causal=True, scale=scale, out=o, lse=lse, stream=stream)
        e1.record(stream)
    torch.cuda.synchronize(dev)
    if fa.fattn_last_error() != 0:
        raise RuntimeError("a kernel reported a bounded-wait timeout")
    fused_ms = sum(e0.elapsed_time(e1) for e0, e1 in evs) / args.steps
    peaks, peak_src = load_peaks()
    un = measure_unfused(fa, dev, stream, P, q, k, v, fused_ms, peaks, iters=args.steps)
    if rank != 0:
        return
    fl = prefill_flops(B, H, N, d, True)
    line = {"metric": "prefill ms, fused (fattn_fwd) against standard attention in three kernels (fattn_fwd_unfused)",
            "value": un["ms"], "unit": "ms", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "higher_is_better": False, "dtype": "bf16", "data": "synthetic: seeded iid N(0,1) rounded to bf16",
            "config": {"workload": f"prefill_b{B}h{H}_n{N}_d{d} causal",
                       "l2": "a 512 MiB buffer is written before every call (outside the per-call events)"},
            "fused": {"ms": round(fused_ms, 4), "tflops": round(fl / (fused_ms * 1e-3) / 1e12, 2),
                      "algorithmic_bytes": prefill_bytes(B, H, N, d)},
            "unfused": un, "peak_source": peak_src}
    print(json.dumps(line), flush=True)


def run_e2e(fa, dev, stream, args, q, k, v, dq, dk, dv, scale_p, scale_d):
    """The same calls fed from pinned host buffers, copies included in the timing."""
    import torch
    steps = max(1, min(args.steps, args.e2e_steps))
    out = {"h2d": 0, "d2h": 0}
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
    if q is not None:
        hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
        ho = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
        hl = torch.empty(q.shape[:3], dtype=torch.float32).pin_memory()
        B, H, N, d = q.shape
        ws = torch.empty(fa.fattn_fwd_host_workspace_size(B, H, N, N, d), dtype=torch.uint8, device=dev)

        def prefill_once():
            fa.fattn_fwd_host(hq, hk, hv, causal=True, scale=scale_p, out=ho, lse=hl, workspace=ws, device=dev,
                              stream=stream)

        prefill_once()
        torch.cuda.synchronize(dev)
        ev[0].record(stream)
        for _ in range(steps):
            prefill_once()
        ev[1].record(stream)
        torch.cuda.synchronize(dev)
        out["prefill_s"] = ev[0].elapsed_time(ev[1]) * 1e-3 / steps
        out["h2d"] += sum(t.numel() * t.element_size() for t in (hq, hk, hv))
        out["d2h"] += sum(t.numel() * t.element_size() for t in (ho, hl))
        del hq, hk, hv, ws
    if dq is not None:
        hdq, hdk, hdv = (t.cpu().pin_memory() for t in (dq, dk, dv))
        hdo = torch.empty(dq.shape, dtype=torch.bfloat16).pin_memory()
        hdl = torch.empty(dq.shape[:3], dtype=torch.float32).pin_memory()
        ws = torch.empty(fa.fattn_decode_host_workspace_size(dk.shape[0], dk.shape[1], dk.shape[2], dk.shape[3]),
                         dtype=torch.uint8, device=dev)

        def decode_once():
            fa.fattn_decode_host(hdq, hdk, hdv, scale=scale_d, out=hdo, lse=hdl, workspace=ws, device=dev,
                                 stream=stream)

        decode_once()
        torch.cuda.synchronize(dev)
        ev[0].record(stream)
        for _ in range(steps):
            decode_once()
        ev[1].record(stream)
        torch.cuda.synchronize(dev)
        out["decode_s"] = ev[0].elapsed_time(ev[1]) * 1e-3 / steps
        out["h2d"] += sum(t.numel() * t.element_size() for t in (hdq, hdk, hdv))
        out["d2h"] += sum(t.numel() * t.element_size() for t in (hdo, hdl))
    return out


def run_reference(args):
    """The reference arm: the fp64 CPU oracle as it stands, on this host's cores."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    pf, _ = host_inputs_f64()
    P = PREFILL
    budget = max(1.0, args.ref_budget)
    per_step = budget / max(1, args.steps + args.warmup)
    for _ in range(args.warmup):
        oracle_prefill_sample(*pf, budget_s=per_step, seed=99)
    flops = secs = 0.0
    rows = 0
    threads = 1
    t_wall = time.perf_counter()
    for i in range(args.steps):
        f, s_, r, threads = oracle_prefill_sample(*pf, budget_s=per_step, seed=i)
        flops += f
        secs += s_
        rows += r
    t_wall = time.perf_counter() - t_wall
    value = flops / secs / 1e12
    line = {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * t_wall / max(1, args.steps), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic: seeded iid N(0,1) drawn in fp32 and rounded to bf16, computed in fp64",
        "config": {"workload": "prefill_b1h32_n8192_d64 causal (sampled rows)",
                   "prefill": {"B": P["B"], "H": P["H"], "Nq": P["N"], "Nk": P["N"], "d": P["d"],
                               "causal": True}},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
                         "sample": (f"{rows} random query rows over the run, about {per_step:.1f} s of "
                                    "oracle work per step")},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description="exact-attention hot-path benchmark")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["both", "prefill", "decode", "backward", "fp8", "unfused"],
                    default="both",
                    help="both = the benchmark step; prefill/decode time one half (profiling); backward "
                         "times fattn_bwd on the prefill shape (a line of its own); unfused times the fused "
                         "prefill and the three-kernel standard attention on that shape")
    ap.add_argument("--bwd-d", type=int, default=0, help="override d of the backward workload (64 or 128)")
    ap.add_argument("--fp8-d", type=int, default=0, help="d of the fp8 workload (64 or 128; default 128)")
    ap.add_argument("--window", type=int, default=-1,
                    help="sliding-window band (W-1, 0) for the prefill/backward workloads (FLOPs = visible pairs)")
    ap.add_argument("--prefill-heads", type=int, default=0, help="override H of the prefill (profiling)")
    ap.add_argument("--decode-batch", type=int, default=0, help="override B of the decode (profiling)")
    ap.add_argument("--cpu-budget", type=float, default=12.0,
                    help="seconds of oracle work for the cpu_baseline figure (0 = skip)")
    ap.add_argument("--ref-budget", type=float, default=60.0,
                    help="seconds of oracle work for the whole --impl reference run")
    ap.add_argument("--e2e-steps", type=int, default=5, help="steps of the host-buffer run (0 = skip)")
    ap.add_argument("--no-clocks", dest="clocks", action="store_false")
    ap.add_argument("--no-configs", dest="configs", action="store_false",
                    help="skip the smaller prefill configurations (configs_measured)")
    ap.add_argument("--no-rising", dest="rising", action="store_false",
                    help="skip the prefill on rising-score inputs (prefill_rising_scores)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "backward":
        run_backward(args)
    elif args.workload == "fp8":
        run_fp8(args)
    elif args.workload == "unfused":
        run_unfused(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
