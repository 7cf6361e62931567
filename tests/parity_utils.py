"""Shared helpers for the GPU parity tests: run the oracle on the same inputs and compare."""

from __future__ import annotations

import numpy as np
import torch

import oracle

# Tolerances of the contract: bf16 inputs and output, fp32 accumulation, fp64 oracle.
O_MAX_ABS = 2e-2
O_MEAN_ABS = 1e-3
LSE_MAX_ABS = 1e-3


def to64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu").to(torch.float64).numpy()


def compare(o_gpu, lse_gpu, o_ref, lse_ref, what=""):
    """Element-by-element comparison against the oracle; returns the error summary."""
    o = to64(o_gpu).reshape(o_ref.shape)
    err = np.abs(o - o_ref)
    assert np.all(np.isfinite(o)), f"{what}: non-finite output"
    s = {"o_max": float(err.max()), "o_mean": float(err.mean())}
    if lse_gpu is not None:
        lse = to64(lse_gpu).reshape(lse_ref.shape)
        assert np.all(np.isfinite(lse)), f"{what}: non-finite lse"
        s["lse_max"] = float(np.abs(lse - lse_ref).max())
    assert s["o_max"] <= O_MAX_ABS, f"{what}: O max abs err {s}"
    assert s["o_mean"] <= O_MEAN_ABS, f"{what}: O mean abs err {s}"
    if lse_gpu is not None:
        assert s["lse_max"] <= LSE_MAX_ABS, f"{what}: LSE max abs err {s}"
    return s


def oracle_full(q, k, v, causal, scale):
    return oracle.attention(to64(q), to64(k), to64(v), causal=causal, scale=scale)


def oracle_rows(q, k, v, rows, causal, scale):
    """Oracle on selected flat rows; copies only the heads those rows belong to."""
    B, H, Nq, d = q.shape
    rows = np.asarray(rows, dtype=np.int64)
    heads = np.unique(rows // Nq)
    o_out = np.empty((rows.size, d))
    lse_out = np.empty(rows.size)
    for bh in heads:
        b, h = divmod(int(bh), H)
        sel = np.nonzero(rows // Nq == bh)[0]
        qi = to64(q[b, h][torch.as_tensor(rows[sel] % Nq, device=q.device)])  # [n, d]
        kk = to64(k[b, h])
        vv = to64(v[b, h])
        # present the selected rows as one head whose row indices are the original ones
        qfull = np.zeros((1, 1, Nq, d))
        qfull[0, 0, rows[sel] % Nq] = qi
        o_r, l_r = oracle.attention_rows(qfull, kk[None, None], vv[None, None], rows[sel] % Nq,
                                         causal=causal, scale=scale)
        o_out[sel] = o_r
        lse_out[sel] = l_r
    return o_out, lse_out


def sample_rows(B, H, Nq, n_heads, per_head, seed, extra_per_head=None):
    """Flat row indices: `per_head` rows in each of `n_heads` heads, always including the first
    and last rows of the head and, when given, extra rows (e.g. the boosted ones)."""
    rng = np.random.default_rng(seed)
    heads = rng.choice(B * H, size=min(n_heads, B * H), replace=False)
    out = []
    for bh in heads:
        r = set(rng.choice(Nq, size=min(per_head, Nq), replace=False).tolist())
        r.update({0, Nq - 1, min(Nq - 1, 127), min(Nq - 1, 128)})
        if extra_per_head is not None:
            r.update(int(x) for x in extra_per_head(int(bh)))
        out.extend(int(bh) * Nq + x for x in sorted(r))
    return np.array(out, dtype=np.int64)
