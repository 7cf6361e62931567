"""Memory-traffic and flop counts of attention, standard and tiled, as host-side arithmetic.

"FlashAttention: attention was never compute-bound" argues the whole method from a counter: every
element that crosses between slow memory (HBM) and fast memory (SRAM), and every multiply-add, is
added up by hand, and its tables print the totals.  This module states those counting rules as
closed forms so that the printed tables can be reproduced digit for digit, and applies the same
rules to the shapes this library runs, where they give the algorithmic bytes its benchmark divides
by.  It holds no attention arithmetic and needs no GPU.

Counting rules (elements; the page's script works in float32, 4 bytes per element; its tables print
bytes / 2**20 as "MB" and flops / 1e9 as "GFLOPs"):

  standard attention, forward ("Where the time actually goes"):
      read Q and K to form S, write S, read S for the softmax, write P, read P and V, write O:
      4 n^2 + 4 n d elements; flops 4 n^2 d (the two n x n x d products, 2 flops per multiply-add);
      the largest buffer held at once is the n x n score matrix.
  tiled attention, forward ("Tiling: same answer, flat memory" and "How big should a tile be?"):
      each query tile is loaded once, each key/value tile once per query tile that visits it, and
      each output tile written once: n d + 2 n^2 d / Br + n d elements for n = Nq = Nk and no mask;
      flops are those of the standard version ("And no, it is not doing less arithmetic");
      the working set is one Q tile, one K and one V tile, one score tile and the two running
      statistics: Br d + 2 Bc d + Br Bc + 2 Br elements.
  backward ("The backward pass: pay flops, save bytes"):
      standard keeps P and the three inputs, n^2 + 3 n d elements, and spends 10 n^2 d flops; the
      tiled version keeps the inputs and two floats per row (m and l), 3 n d + 2 n, and recomputes
      the score tiles, 12 n^2 d flops (20 % more).
"""

from __future__ import annotations

import dataclasses
import math

FP32 = 4
BF16 = 2
MIB = float(1 << 20)
KIB = 1024.0


@dataclasses.dataclass(frozen=True)
class Count:
    elements: float       # elements moved between HBM and on-chip memory
    flops: float          # 2 per multiply-add of the matrix products
    peak_elements: float  # the largest working buffer held at once, in elements

    def mb(self, elem_bytes: int = FP32) -> float:
        return self.elements * elem_bytes / MIB

    def gflops(self) -> float:
        return self.flops / 1e9

    def bytes_per_flop(self, elem_bytes: int = FP32) -> float:
        return self.elements * elem_bytes / self.flops


# ------------------------------------------------------------------------------------------------
# The page's counts (one head, n = Nq = Nk, no mask)
# ------------------------------------------------------------------------------------------------
def standard_forward(n: int, d: int) -> Count:
    """Standard attention: S and P each written once and read once, Q, K, V read, O written."""
    return Count(elements=4.0 * n * n + 4.0 * n * d, flops=4.0 * n * n * d, peak_elements=float(n) * n)


def score_share(n: int, d: int) -> float:
    """Fraction of standard attention's traffic that is the n x n matrices (the "n^2 share" column)."""
    return (4.0 * n * n) / (4.0 * n * n + 4.0 * n * d)


def tile_working_set(Br: int, Bc: int, d: int) -> float:
    """Elements held on chip by one query tile's inner loop: Q_i, K_j, V_j, S_ij, m and l."""
    return float(Br * d + 2 * Bc * d + Br * Bc + 2 * Br)


def tiled_forward(n: int, d: int, Br: int = 64, Bc: int = 64) -> Count:
    """Tiled attention with Br-row query tiles and Bc-key tiles over n queries and n keys, no mask."""
    return tiled_forward_general(n, n, d, Br, Bc)


def standard_backward_stored(n: int, d: int) -> float:
    """Elements the standard backward keeps from the forward: P (n x n) and Q, K, V."""
    return float(n) * n + 3.0 * n * d


def tiled_backward_stored(n: int, d: int) -> float:
    """Elements the tiled backward keeps: Q, K, V and two statistics per row."""
    return 3.0 * n * d + 2.0 * n


def standard_backward_flops(n: int, d: int) -> float:
    return 10.0 * n * n * d


def tiled_backward_flops(n: int, d: int) -> float:
    """The standard backward's products plus one recomputation of the scores, 2 n^2 d."""
    return standard_backward_flops(n, d) + 2.0 * n * n * d


# ------------------------------------------------------------------------------------------------
# The same rules for any Nq, Nk, tile sizes and bottom-right-aligned band
# ------------------------------------------------------------------------------------------------
def visible_range(i: int, Nq: int, Nk: int, window_left: int = -1, window_right: int = -1):
    """Keys [lo, hi] that query row i sees under the band (window_left, window_right), bottom-right
    aligned (off = Nk - Nq); -1 leaves a side unbounded.  hi < lo when the row sees no key."""
    c = i + (Nk - Nq)
    hi = Nk - 1 if window_right < 0 else min(Nk - 1, c + window_right)
    lo = 0 if window_left < 0 else max(0, c - window_left)
    return lo, hi


def visible_pairs(Nq: int, Nk: int, window_left: int = -1, window_right: int = -1) -> int:
    """(query, key) pairs the band leaves visible."""
    total = 0
    for i in range(Nq):
        lo, hi = visible_range(i, Nq, Nk, window_left, window_right)
        if hi >= lo:
            total += hi - lo + 1
    return total


def tiled_forward_general(Nq: int, Nk: int, d: int, Br: int, Bc: int, window_left: int = -1,
                          window_right: int = -1) -> Count:
    """Elements moved by the tiled forward of one head: each query tile is loaded once and its
    output written once, each key/value tile once per query tile that has a visible key in it.
    Flops count the products of the visited (query tile, key tile) pairs, tile by tile."""
    elements = 0.0
    flops = 0.0
    for r0 in range(0, Nq, Br):
        rows = min(Br, Nq - r0)
        elements += 2.0 * rows * d  # Q_i in, O_i out
        lo = min(visible_range(i, Nq, Nk, window_left, window_right)[0] for i in range(r0, r0 + rows))
        hi = max(visible_range(i, Nq, Nk, window_left, window_right)[1] for i in range(r0, r0 + rows))
        if hi < lo:
            continue
        for c0 in range((lo // Bc) * Bc, hi + 1, Bc):
            cols = min(Bc, Nk - c0)
            elements += 2.0 * cols * d  # K_j, V_j
            flops += 4.0 * rows * cols * d
    return Count(elements=elements, flops=flops, peak_elements=tile_working_set(Br, Bc, d))


# ------------------------------------------------------------------------------------------------
# Algorithmic bytes of this library's entry points (bf16 tensors, fp32 L)
# ------------------------------------------------------------------------------------------------
def fused_forward_bytes(B: int, H: int, Nq: int, Nk: int, d: int, elem_bytes: int = BF16,
                        with_lse: bool = True) -> float:
    """Compulsory traffic of one fused forward: the tiled count with a single query tile per head
    (Br >= Nq, so K and V are read once), in `elem_bytes` per element, plus L in fp32.  Every key is
    read even under a causal mask, since the last query row sees them all."""
    per_head = tiled_forward_general(Nq, Nk, d, Br=max(Nq, 1), Bc=max(Nk, 1)).elements * elem_bytes
    return B * H * (per_head + (Nq * FP32 if with_lse else 0))


def fused_forward_reread_bytes(B: int, H: int, Nq: int, Nk: int, d: int, Br: int, Bc: int = 128,
                               window_left: int = -1, window_right: int = -1,
                               elem_bytes: int = BF16) -> float:
    """The same forward if every key/value tile came from HBM once per Br-row query block that
    visits it (no reuse through the L2 cache): the upper end of the DRAM traffic one launch can
    cause, against which a measured figure shows how much the cache absorbs."""
    c = tiled_forward_general(Nq, Nk, d, Br, Bc, window_left, window_right)
    return B * H * (c.elements * elem_bytes + Nq * FP32)


def fp8_forward_bytes(B: int, H: int, Nq: int, Nk: int, d: int) -> float:
    """The fused forward on 8-bit operands: q, k, v read once (1 byte each), O written in bf16, L."""
    return B * H * ((Nq + 2 * Nk) * d * 1 + Nq * d * BF16 + Nq * FP32)


def decode_bytes(B: int, H: int, Nk: int, d: int, elem_bytes: int = BF16) -> float:
    """One decode step: the forward with Nq = 1 (q in, K and V once, O out) plus L."""
    return fused_forward_bytes(B, H, 1, Nk, d, elem_bytes)


def decode_kv_bytes(B: int, H: int, Nk: int, d: int, elem_bytes: int = BF16) -> float:
    """The key/value part of a decode step's traffic: the cache read once."""
    return 2.0 * B * H * Nk * d * elem_bytes


def backward_bytes(B: int, H: int, Nq: int, Nk: int, d: int, elem_bytes: int = BF16) -> float:
    """Compulsory traffic of one fused backward: Q, O, dO and L read per query row, K and V read per
    key, dQ written per query row and dK, dV per key (the tiled backward's stored inputs, the
    forward's O and L in place of m and l, and the gradients)."""
    return B * H * ((Nq * d * 3 + Nk * d * 2) * elem_bytes + Nq * FP32 + (Nq + 2 * Nk) * d * elem_bytes)


def unfused_forward_bytes(B: int, H: int, Nq: int, Nk: int, d: int, s_bytes: int = FP32, p_bytes: int = BF16,
                          elem_bytes: int = BF16, with_lse: bool = True) -> float:
    """Compulsory traffic of standard attention in three kernels (the standard count of "Where the
    time actually goes", per head): the first product reads Q and K and writes S, the softmax reads S
    and writes P (and L), the second product reads P and V and writes O.  S and P take `s_bytes` and
    `p_bytes` per element, the inputs and O `elem_bytes`.  With 4 bytes everywhere, n = Nq = Nk and
    no L this is the page's 4 n^2 + 4 n d elements."""
    per_head = float((Nq + Nk) * d * elem_bytes)  # Q, K into S = Q K^T
    per_head += 2.0 * Nq * Nk * s_bytes           # S written, S read by the softmax
    per_head += 2.0 * Nq * Nk * p_bytes           # P written, P read by O = P V
    per_head += (Nk + Nq) * d * elem_bytes        # V read, O written
    return B * H * (per_head + (Nq * FP32 if with_lse else 0))


def forward_flops(B: int, H: int, Nq: int, Nk: int, d: int, causal: bool) -> float:
    """The benchmark convention: 4 B H Nq Nk d, halved under the causal mask."""
    f = 4.0 * B * H * Nq * Nk * d
    return f / 2 if causal else f


def fmt_table_value(x: float, digits: int) -> str:
    """Fixed-point text as the page's script prints it (round half to even on the binary value)."""
    if not math.isfinite(x):
        return str(x)
    return f"{x:.{digits}f}"
