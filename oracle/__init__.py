"""fp64 CPU oracle for exact attention -- TEST INFRASTRUCTURE ONLY.

This package is the parity reference for the CUDA library.  Only the test suite, the package's
``smoke()`` check and the benchmark's CPU-baseline leg may import it; the library itself never
does, and it shares no code with the library.

The arithmetic lives in ``attention_oracle.cpp`` (plain C++17, fp64, sequential sums, no FMA
contraction).  This module only compiles it with the host C++ compiler and marshals numpy
arrays through ctypes.

Pages cited by the functions below:
  "Flash Attention: The Hidden Gem" -- safe softmax, online softmax, the forward algorithm, L.
  "FlashAttention: attention was never compute-bound" -- online softmax demo 2 and its broken
  no-rescale variant.
  "Flash Attention: The Hidden Gem", Phase 2 -- the gradients dQ, dK, dV (softmax Jacobian).
  "Understanding FlashAttention" -- the online normalizer (g, s) and the attention shapes.
"""

from __future__ import annotations

import ctypes
import hashlib
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attention_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_STAMP = os.path.join(_HERE, "liboracle.stamp")
_lock = threading.Lock()
_lib = None

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.POINTER(ctypes.c_int64)
_U8 = ctypes.POINTER(ctypes.c_uint8)


def _digest(cmd) -> str:
    h = hashlib.sha256()
    with open(_SRC, "rb") as f:
        h.update(f.read())
    h.update(" ".join(cmd).encode())
    h.update(platform.machine().encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile ``attention_oracle.cpp`` into ``liboracle.so`` next to it (g++, -O2, no FMA).  The
    library is rebuilt whenever the source, the flags or the host architecture differ from those it
    was built with (recorded in a stamp file beside it)."""
    cmd = ["g++", "-std=c++17", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
           "-pthread", _SRC, "-o"]
    digest = _digest(cmd)
    if not force and os.path.exists(_LIB) and os.path.exists(_STAMP):
        with open(_STAMP) as f:
            if f.read().strip() == digest:
                return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(cmd + [tmp], check=True)
    os.replace(tmp, _LIB)
    with open(_STAMP, "w") as f:
        f.write(digest + "\n")
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        lib.oracle_softmax.argtypes = [_D, ctypes.c_int64, _D]
        lib.oracle_softmax.restype = None
        lib.oracle_online_softmax.argtypes = [_D, ctypes.c_int64, ctypes.c_int64, ctypes.c_int, _D]
        lib.oracle_online_softmax.restype = None
        lib.oracle_online_normalizer.argtypes = [_D, ctypes.c_int64, _D, _D]
        lib.oracle_online_normalizer.restype = None
        lib.oracle_attention.argtypes = [_D, _D, _D, _D, _D] + [ctypes.c_int64] * 7 + [
            _U8, ctypes.c_double, ctypes.c_int]
        lib.oracle_attention.restype = ctypes.c_int64
        lib.oracle_attention_rows.argtypes = [_D, _D, _D, _I64, ctypes.c_int64, _D, _D] + [
            ctypes.c_int64] * 7 + [_U8, ctypes.c_double, ctypes.c_int]
        lib.oracle_attention_rows.restype = ctypes.c_int64
        lib.oracle_attention_probs.argtypes = [_D, _D] + [ctypes.c_int64] * 5 + [_U8, ctypes.c_double, _D]
        lib.oracle_attention_probs.restype = None
        lib.oracle_attention_backward.argtypes = [_D] * 7 + [ctypes.c_int64] * 7 + [
            _U8, ctypes.c_double, ctypes.c_int]
        lib.oracle_attention_backward.restype = None
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_D)


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)


def softmax(x) -> np.ndarray:
    """Three-pass safe softmax of a vector ("Flash Attention: The Hidden Gem", Safe Softmax)."""
    x = _f64(x).ravel()
    y = np.empty_like(x)
    _load().oracle_softmax(_p(x), x.size, _p(y))
    return y


def online_softmax(x, block: int = 8, rescale: bool = True) -> np.ndarray:
    """Block-streamed online softmax; ``rescale=False`` drops the exp(m_old - m_new) factor
    ("FlashAttention: attention was never compute-bound", Online softmax: the whole idea)."""
    x = _f64(x).ravel()
    y = np.empty_like(x)
    _load().oracle_online_softmax(_p(x), x.size, int(block), 1 if rescale else 0, _p(y))
    return y


def online_normalizer(x) -> tuple[float, float]:
    """Final (g_N, s_N) of the per-element recurrence ("Understanding FlashAttention", Online softmax)."""
    x = _f64(x).ravel()
    g = ctypes.c_double()
    s = ctypes.c_double()
    _load().oracle_online_normalizer(_p(x), x.size, ctypes.byref(g), ctypes.byref(s))
    return g.value, s.value


def band(causal: bool = False, window=None) -> tuple[int, int]:
    """The mask as (window_left, window_right), bottom-right aligned; -1 = unbounded on that side.
    ``window`` overrides ``causal``: no mask is (-1, -1), causal is (-1, 0), a sliding window of W
    keys is (W - 1, 0)."""
    if window is not None:
        wl, wr = (int(window[0]), int(window[1]))
        if wl < -1 or wr < -1:
            raise ValueError("window sides must be >= -1")
        return wl, wr
    return (-1, 0) if causal else (-1, -1)


def _mask_u8(mask, B, H, Nq, Nk):
    """An element mask broadcastable to [B, H, Nq, Nk] (true = the key may be seen) as a contiguous
    uint8 array of that full shape, and its pointer (None, a null pointer, for no mask)."""
    if mask is None:
        return None, None
    m = np.ascontiguousarray(np.broadcast_to(np.asarray(mask).astype(bool), (B, H, Nq, Nk)), dtype=np.uint8)
    return m, m.ctypes.data_as(_U8)


def _shape4(q, k, v):
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B,H,N,d]")
    B, H, Nq, d = q.shape
    if k.shape[:2] != (B, H) or v.shape != k.shape or k.shape[3] != d:
        raise ValueError(f"shape mismatch q{q.shape} k{k.shape} v{v.shape}")
    return q, k, v, B, H, Nq, k.shape[2], d


def attention(q, k, v, causal: bool = False, scale: float | None = None, nthreads: int | None = None,
              window=None, mask=None):
    """O = softmax(scale*QK^T + mask) V and L = m + log l for every row, by definition.

    q: [B,H,Nq,d], k,v: [B,H,Nk,d] (any float dtype; computed in fp64).  Masks are bottom-right
    aligned bands (see band()); causal: row i sees key j iff j <= i + Nk - Nq.  `mask`, when given,
    is an element mask broadcastable to [B,H,Nq,Nk] (true = visible) applied on top of the band.  A
    row with no visible key gets o = 0 and lse = -inf.  Returns (o [B,H,Nq,d], lse [B,H,Nq]) as
    float64.
    """
    q, k, v, B, H, Nq, Nk, d = _shape4(q, k, v)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    wl, wr = band(causal, window)
    m, mp = _mask_u8(mask, B, H, Nq, Nk)
    o = np.empty((B, H, Nq, d), dtype=np.float64)
    lse = np.empty((B, H, Nq), dtype=np.float64)
    _load().oracle_attention(_p(q), _p(k), _p(v), _p(o), _p(lse), B, H, Nq, Nk, d, wl, wr, mp,
                             float(scale), nthreads or default_threads())
    return o, lse


def attention_rows(q, k, v, rows, causal: bool = False, scale: float | None = None,
                   nthreads: int | None = None, window=None, mask=None):
    """The same definition for selected flat row indices r = (b*H + h)*Nq + i.

    Returns (o [len(rows), d], lse [len(rows)]).
    """
    q, k, v, B, H, Nq, Nk, d = _shape4(q, k, v)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).ravel())
    if rows.size and (rows.min() < 0 or rows.max() >= B * H * Nq):
        raise IndexError("row index out of range")
    o = np.empty((rows.size, d), dtype=np.float64)
    lse = np.empty((rows.size,), dtype=np.float64)
    wl, wr = band(causal, window)
    m, mp = _mask_u8(mask, B, H, Nq, Nk)
    _load().oracle_attention_rows(_p(q), _p(k), _p(v), rows.ctypes.data_as(_I64), rows.size,
                                  _p(o), _p(lse), B, H, Nq, Nk, d, wl, wr, mp, float(scale),
                                  nthreads or default_threads())
    return o, lse


def attention_probs(q, k, causal: bool = False, scale: float | None = None, window=None,
                    mask=None) -> np.ndarray:
    """P = softmax(scale*QK^T + mask) for one head; q [Nq,d], k [Nk,d] -> [Nq,Nk]; `mask` an
    element mask broadcastable to [Nq, Nk] on top of the band."""
    q, k = _f64(q), _f64(k)
    Nq, d = q.shape
    Nk = k.shape[0]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    p = np.empty((Nq, Nk), dtype=np.float64)
    wl, wr = band(causal, window)
    m, mp = _mask_u8(mask, 1, 1, Nq, Nk)
    _load().oracle_attention_probs(_p(q), _p(k), Nq, Nk, d, wl, wr, mp, float(scale), _p(p))
    return p


def attention_backward(q, k, v, do, causal: bool = False, scale: float | None = None,
                       nthreads: int | None = None, window=None, mask=None):
    """Gradients (dq, dk, dv) of O = softmax(scale*QK^T + mask) V for an upstream gradient do,
    by definition ("Flash Attention: The Hidden Gem", Phase 2), with the factor scale on dq and dk
    from X = scale * Q K^T.  Shapes as in attention(); returns float64 arrays."""
    q, k, v, B, H, Nq, Nk, d = _shape4(q, k, v)
    do = _f64(do)
    if do.shape != q.shape:
        raise ValueError("do must have q's shape")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    wl, wr = band(causal, window)
    m, mp = _mask_u8(mask, B, H, Nq, Nk)
    _load().oracle_attention_backward(_p(q), _p(k), _p(v), _p(do), _p(dq), _p(dk), _p(dv), B, H, Nq, Nk, d,
                                      wl, wr, mp, float(scale), nthreads or default_threads())
    return dq, dk, dv
