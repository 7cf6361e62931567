"""Seeded synthetic inputs for the attention workloads.

This module only draws numbers: it holds none of the attention arithmetic, and both the CUDA
path's tests and the CPU oracle take their inputs from it.  Values are iid N(0, 1) drawn with a
seeded torch generator on the requested device, in fp32, and rounded once to bf16 (round to
nearest even).  Q, K and V are drawn in that order from one generator.

The named workloads are the sizes the library is measured and checked on:
  prefill_b1h1_n128_d64        B=1,  H=1,  Nq=Nk=128,   d=64,  non-causal
  prefill_b1h8_n1024_d64       B=1,  H=8,  Nq=Nk=1024,  d=64,  causal
  prefill_b4h16_n2048_d128     B=4,  H=16, Nq=Nk=2048,  d=128, non-causal and causal, with 1% of
                               the query rows of every head multiplied by 8
  prefill_b1h32_n8192_d64      B=1,  H=32, Nq=Nk=8192,  d=64,  causal
  decode_b32h32_nk16384_d128   B=32, H=32, Nq=1, Nk=16384, d=128, no mask

The backward pass is checked and measured on the prefill shapes; its upstream gradient dO is drawn
by make_dout from a generator of its own (seed + DOUT_SEED_OFFSET), so Q, K and V stay those of the
forward workload.
"""

from __future__ import annotations

import dataclasses

import torch

SEED_BASE = 0xFA77E000
DOUT_SEED_OFFSET = 0x100


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: tuple  # the mask settings the workload is run with
    boost_frac: float = 0.0  # fraction of query rows per head multiplied by `boost`
    boost: float = 8.0
    decode: bool = False
    config_id: int = 0

    @property
    def seed(self) -> int:
        return SEED_BASE + self.config_id

    @property
    def scale(self) -> float:
        return 1.0 / (self.d ** 0.5)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("prefill_b1h1_n128_d64", 1, 1, 128, 128, 64, (False,), config_id=1),
        Workload("prefill_b1h8_n1024_d64", 1, 8, 1024, 1024, 64, (True,), config_id=2),
        Workload("prefill_b4h16_n2048_d128", 4, 16, 2048, 2048, 128, (False, True), boost_frac=0.01,
                 config_id=3),
        Workload("prefill_b1h32_n8192_d64", 1, 32, 8192, 8192, 64, (True,), config_id=4),
        Workload("decode_b32h32_nk16384_d128", 32, 32, 1, 16384, 128, (False,), decode=True, config_id=5),
    ]
}


def _randn_bf16(shape, gen, device, chunk_rows=None):
    """N(0,1) in fp32, rounded to bf16; drawn per leading index to bound the fp32 temporary."""
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    if chunk_rows is None or shape[0] <= 1:
        out.copy_(torch.randn(shape, generator=gen, device=device, dtype=torch.float32))
        return out
    for b0 in range(0, shape[0], chunk_rows):
        sub = out[b0:b0 + chunk_rows]
        sub.copy_(torch.randn(tuple(sub.shape), generator=gen, device=device, dtype=torch.float32))
    return out


def boosted_rows(Nq: int, frac: float, gen: torch.Generator, device) -> torch.Tensor:
    """floor(frac * Nq) distinct row indices chosen by a seeded permutation."""
    n = int(frac * Nq)
    if n <= 0:
        return torch.empty(0, dtype=torch.long)
    return torch.randperm(Nq, generator=gen, device=device)[:n].cpu()


def make_qkv(B: int, H: int, Nq: int, Nk: int, d: int, seed: int, device="cpu", boost_frac: float = 0.0,
             boost: float = 8.0):
    """Seeded bf16 q [B,H,Nq,d], k [B,H,Nk,d], v [B,H,Nk,d] on `device`.

    With boost_frac > 0, floor(boost_frac * Nq) query rows of every (b, h) are multiplied by
    `boost` after rounding (a power of two, so the product is exact in bf16).  Returns
    (q, k, v, boosted) where boosted is a list of row-index tensors, one per (b, h).
    """
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    chunk = 1 if B * H * max(Nq, Nk) * d > (1 << 28) else None
    q = _randn_bf16((B, H, Nq, d), gen, device, chunk)
    k = _randn_bf16((B, H, Nk, d), gen, device, chunk)
    v = _randn_bf16((B, H, Nk, d), gen, device, chunk)
    boosted = []
    if boost_frac > 0:
        for b in range(B):
            for h in range(H):
                rows = boosted_rows(Nq, boost_frac, gen, device)
                if rows.numel():
                    q[b, h, rows.to(device)] *= boost
                boosted.append(rows)
    return q, k, v, boosted


def make_workload(w: Workload, device="cpu"):
    return make_qkv(w.B, w.H, w.Nq, w.Nk, w.d, w.seed, device, w.boost_frac, w.boost)


def make_dout(B: int, H: int, Nq: int, d: int, seed: int, device="cpu"):
    """Seeded bf16 upstream gradient dO [B,H,Nq,d], iid N(0, 1) rounded once to bf16, drawn from a
    generator seeded with seed + DOUT_SEED_OFFSET."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed) + DOUT_SEED_OFFSET)
    chunk = 1 if B * H * Nq * d > (1 << 28) else None
    return _randn_bf16((B, H, Nq, d), gen, device, chunk)


def make_rising_scores(B: int, H: int, Nq: int, Nk: int, d: int, seed: int, device="cpu", large_from=None):
    """Inputs whose scores rise sharply after the first keys (late "attention sinks"): every query
    is 30 u plus N(0, 0.01) noise for one seeded unit vector u; keys [large_from, Nk) are 30 u plus
    the same noise (scores near 900 before scaling) and the others, like the values, iid N(0, 1)
    (scores of about 30 N(0, 1)).  large_from defaults to the last 128 keys.  Drawn in fp32 on
    `device` from one seeded generator and rounded once to bf16.  Returns (q, k, v)."""
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    large_from = Nk - 128 if large_from is None else int(large_from)
    u = torch.randn(d, generator=gen, device=device, dtype=torch.float32)
    u /= u.norm()
    q = torch.empty((B, H, Nq, d), dtype=torch.bfloat16, device=device)
    k = torch.empty((B, H, Nk, d), dtype=torch.bfloat16, device=device)
    v = torch.empty((B, H, Nk, d), dtype=torch.bfloat16, device=device)
    for b in range(B):  # one batch entry at a time bounds the fp32 temporaries
        q[b] = 30 * u + 0.1 * torch.randn((H, Nq, d), generator=gen, device=device)
        kb = torch.randn((H, Nk, d), generator=gen, device=device)
        if large_from < Nk:
            kb[:, max(large_from, 0):] = 30 * u + 0.1 * torch.randn((H, Nk - max(large_from, 0), d), generator=gen,
                                                                       device=device)
        k[b] = kb
        v[b] = torch.randn((H, Nk, d), generator=gen, device=device)
    return q, k, v


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor e4m3 quantisation of a float tensor: scale so that the largest magnitude maps to
    448 (e4m3's largest finite value), round to nearest.  Returns (x_e4m3, descale) with
    x ~ x_e4m3 * descale."""
    amax = float(x.abs().max())
    descale = amax / 448.0 if amax > 0 else 1.0
    return (x.float() / descale).to(torch.float8_e4m3fn), descale


def make_qkv_fp8(B: int, H: int, Nq: int, Nk: int, d: int, seed: int, device="cpu", boost_frac: float = 0.0):
    """The bf16 inputs of make_qkv, each quantised to e4m3 with one descale factor per tensor.
    Returns ((q8, k8, v8), (q_descale, k_descale, v_descale), boosted rows as in make_qkv)."""
    q, k, v, boosted = make_qkv(B, H, Nq, Nk, d, seed, device, boost_frac)
    out = [quantize_e4m3(t) for t in (q, k, v)]
    return tuple(o[0] for o in out), tuple(o[1] for o in out), boosted
