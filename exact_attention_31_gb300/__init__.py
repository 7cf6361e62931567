"""exact_attention_31_gb300 -- exact fused attention for GB300 (sm_103a), Python binding.

The compute lives in ``libfattn.so`` (hand-written CUDA: a tcgen05/TMEM/TMA prefill kernel, its
backward, and a split-KV decode kernel with its combine kernel) behind the C ABI in
``include/fattn.h``.  This
module only marshals torch tensors into that ABI: it checks dtypes, devices and shapes, allocates
outputs with torch when the caller does not pass them, and raises on a non-OK status.  There is no
other implementation behind these names: if the library is missing, every call raises.

With FATTN_DEBUG=1 in the environment when this module is imported, the same calls go to
``libfattn_debug.so``, the build whose kernels check their TMA, tensor-memory and barrier operands
and their output stores on the device (``fattn_debug_take`` reads what they found).

``fattn_fwd_unfused`` is the standard three-kernel attention (``include/fattn_unfused.h``, in
``libfattn_unfused.so``): two cuBLAS GEMMs around a softmax kernel, with the score and probability
matrices in device memory.  It is the baseline the fused forward's memory traffic is measured
against, not a path the fused entry points take.
"""

from __future__ import annotations

import ctypes
import math
import os

__all__ = [
    "FattnError",
    "fattn_fwd",
    "fattn_bwd",
    "fattn_bwd_masked",
    "fattn_bwd_workspace_size",
    "fattn_bwd_mask_workspace_size",
    "fattn_fwd_masked",
    "fattn_mask_row_words",
    "fattn_mask_workspace_size",
    "pack_mask",
    "fattn_decode",
    "fattn_decode_masked",
    "fattn_decode_static",
    "fattn_decode_num_splits",
    "fattn_decode_workspace_size",
    "fattn_fwd_recomputed_rows",
    "fattn_last_error",
    "fattn_status_string",
    "fattn_debug_build",
    "fattn_debug_take",
    "fattn_fwd_unfused",
    "fattn_unfused_workspace_size",
    "lib",
    "unfused_lib",
    "LIB_PATH",
    "UNFUSED_LIB_PATH",
]

RELEASE_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfattn.so")
DEBUG_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfattn_debug.so")
LIB_PATH = DEBUG_LIB_PATH if os.environ.get("FATTN_DEBUG") == "1" else RELEASE_LIB_PATH
UNFUSED_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfattn_unfused.so")

FATTN_OK = 0
FATTN_ERR_INVALID_ARG = 1
FATTN_ERR_UNSUPPORTED = 2
FATTN_ERR_CUDA = 3
FATTN_ERR_TIMEOUT = 4
FATTN_ERR_DEBUG = 5

_lib = None
_unfused_lib = None


class FattnError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fattn_status_string(status)} ({status})")


def lib() -> ctypes.CDLL:
    """The loaded libfattn (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                           "g.build()'` (nvcc, sm_103a); there is no fallback implementation")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fattn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    L.fattn_fwd.restype = i
    L.fattn_debug_build.argtypes = []
    L.fattn_debug_build.restype = i
    L.fattn_debug_take.argtypes = [ctypes.POINTER(ctypes.c_uint), ctypes.POINTER(ctypes.c_ulonglong)]
    L.fattn_debug_take.restype = i
    L.fattn_fwd_masked.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    L.fattn_fwd_masked.restype = i
    ll = ctypes.c_longlong
    L.fattn_mask_row_words.argtypes = [i]
    L.fattn_mask_row_words.restype = i
    L.fattn_mask_workspace_size.argtypes = [i, i, i, i]
    L.fattn_mask_workspace_size.restype = sz
    L.fattn_fwd_mask.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, vp, ll, ll, i, i, f, vp, sz, vp]
    L.fattn_fwd_mask.restype = i
    L.fattn_bwd_mask_workspace_size.argtypes = [i, i, i, i, i]
    L.fattn_bwd_mask_workspace_size.restype = sz
    L.fattn_bwd_mask.argtypes = [vp] * 9 + [i, i, i, i, i, vp, ll, ll, i, i, f, vp, sz, vp]
    L.fattn_bwd_mask.restype = i
    L.fattn_bwd_workspace_size.argtypes = [i, i, i, i]
    L.fattn_bwd_workspace_size.restype = sz
    L.fattn_bwd.argtypes = [vp] * 9 + [i, i, i, i, i, i, f, vp, sz, vp]
    L.fattn_bwd.restype = i
    L.fattn_bwd_masked.argtypes = [vp] * 9 + [i, i, i, i, i, i, i, f, vp, sz, vp]
    L.fattn_bwd_masked.restype = i
    L.fattn_decode_num_splits.argtypes = [i, i, i, i]
    L.fattn_decode_num_splits.restype = i
    L.fattn_decode_workspace_size.argtypes = [i, i, i, i, i]
    L.fattn_decode_workspace_size.restype = sz
    L.fattn_decode.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, sz, vp]
    L.fattn_decode.restype = i
    L.fattn_decode_masked.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
    L.fattn_decode_masked.restype = i
    L.fattn_decode_static.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp]
    L.fattn_decode_static.restype = i
    L.fattn_fwd_host_workspace_size.argtypes = [i, i, i, i, i, i]
    L.fattn_fwd_host_workspace_size.restype = sz
    L.fattn_fwd_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, i, vp, sz, vp]
    L.fattn_fwd_host.restype = i
    L.fattn_decode_host_workspace_size.argtypes = [i, i, i, i, i, i]
    L.fattn_decode_host_workspace_size.restype = sz
    L.fattn_decode_host.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, vp, sz, vp]
    L.fattn_decode_host.restype = i
    L.fattn_fwd_fp8_workspace_size.argtypes = [i, i, i, i]
    L.fattn_fwd_fp8_workspace_size.restype = sz
    L.fattn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, f, f, f, vp, sz, vp]
    L.fattn_fwd_fp8.restype = i
    L.fattn_last_error.argtypes = [vp]
    L.fattn_last_error.restype = i
    L.fattn_fwd_recomputed_rows.argtypes = [ctypes.POINTER(ctypes.c_ulonglong)]
    L.fattn_fwd_recomputed_rows.restype = i
    L.fattn_status_string.argtypes = [i]
    L.fattn_status_string.restype = ctypes.c_char_p
    _lib = L
    return L


def fattn_status_string(status: int) -> str:
    try:
        return lib().fattn_status_string(int(status)).decode()
    except RuntimeError:
        return {0: "FATTN_OK", 1: "FATTN_ERR_INVALID_ARG", 2: "FATTN_ERR_UNSUPPORTED",
                3: "FATTN_ERR_CUDA", 4: "FATTN_ERR_TIMEOUT"}.get(int(status), "FATTN_UNKNOWN_STATUS")


def _stream_handle(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(t, name, dtype=None):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")


def fattn_mask_row_words(Nk: int) -> int:
    return lib().fattn_mask_row_words(int(Nk))


def fattn_mask_workspace_size(B: int, H: int, Nq: int, Nk: int) -> int:
    return lib().fattn_mask_workspace_size(int(B), int(H), int(Nq), int(Nk))


def pack_mask(mask):
    """A boolean mask [..., Nq, Nk] (true = the key may be seen) in the library's bit layout: int32
    words [..., Nq, fattn_mask_row_words(Nk)], key j in bit j & 31 of word j >> 5 (the 32-bit pattern
    is what matters; int32 is only torch's carrier for it)."""
    import torch
    Nk = mask.shape[-1]
    W = 4 * ((Nk + 127) // 128)
    m = torch.nn.functional.pad(mask.to(torch.bool), (0, W * 32 - Nk))
    m = m.reshape(*m.shape[:-1], W, 32).to(torch.int64)
    words = (m << torch.arange(32, dtype=torch.int64, device=m.device)).sum(-1)
    return torch.where(words >= 2 ** 31, words - 2 ** 32, words).to(torch.int32).contiguous()


def fattn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
              stream=None, want_lse: bool = True, window=None, mask=None, mask_workspace=None):
    """O = softmax(scale * Q K^T + mask) V and L per row, via the fused sm_103a kernel.

    q: bf16 [B,H,Nq,d]; k, v: bf16 [B,H,Nk,d]; d in {64, 128}.  Causal masking is bottom-right
    aligned.  ``window=(window_left, window_right)`` selects a banded mask instead (fattn_fwd_masked;
    -1 = unbounded side).  ``mask`` adds an element mask (fattn_fwd_mask): int32 words from pack_mask,
    shaped [Nq, W], [B or 1, H or 1, Nq, W] (a dimension of 1 is shared); ``mask_workspace`` a CUDA
    uint8 tensor of fattn_mask_workspace_size bytes (allocated here if omitted).
    Returns (out bf16 [B,H,Nq,d], lse fp32 [B,H,Nq] or None).
    """
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16)
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError(f"expected q [B,H,Nq,d], k/v [B,H,Nk,d]; got {tuple(q.shape)}, {tuple(k.shape)}, {tuple(v.shape)}")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("q and k/v disagree on B, H or d")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16)
    if want_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32)
    if mask is not None:
        sb, sh = _mask_strides(mask, B, H, Nq, Nk)
        need = fattn_mask_workspace_size(B, H, Nq, Nk)
        if mask_workspace is None:
            mask_workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
        wl, wr = (int(window[0]), int(window[1])) if window is not None else ((-1, 0) if causal else (-1, -1))
        st = lib().fattn_fwd_mask(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                  lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d, mask.data_ptr(),
                                  sb, sh, wl, wr, float(scale), mask_workspace.data_ptr(), mask_workspace.numel(),
                                  _stream_handle(stream, q.device))
        if st != FATTN_OK:
            raise FattnError(st, "fattn_fwd_mask")
        return out, lse
    if window is not None:
        st = lib().fattn_fwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                                    lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d,
                                    int(window[0]), int(window[1]), float(scale), _stream_handle(stream, q.device))
        if st != FATTN_OK:
            raise FattnError(st, "fattn_fwd_masked")
        return out, lse
    st = lib().fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                         lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d,
                         1 if causal else 0, float(scale), _stream_handle(stream, q.device))
    if st != FATTN_OK:
        raise FattnError(st, "fattn_fwd")
    return out, lse


def unfused_lib() -> ctypes.CDLL:
    """The loaded libfattn_unfused (raises if it has not been built)."""
    global _unfused_lib
    if _unfused_lib is not None:
        return _unfused_lib
    if not os.path.exists(UNFUSED_LIB_PATH):
        raise RuntimeError(f"{UNFUSED_LIB_PATH} is missing: build it with `python -c 'import __graft_entry__ as g; "
                           "g.build()'`")
    L = ctypes.CDLL(UNFUSED_LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fattn_unfused_workspace_size.argtypes = [i, i, i, i]
    L.fattn_unfused_workspace_size.restype = sz
    L.fattn_fwd_unfused.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, sz, vp]
    L.fattn_fwd_unfused.restype = i
    _unfused_lib = L
    return L


def fattn_unfused_workspace_size(B: int, H: int, Nq: int, Nk: int) -> int:
    return unfused_lib().fattn_unfused_workspace_size(int(B), int(H), int(Nq), int(Nk))


def fattn_fwd_unfused(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                      workspace=None, stream=None):
    """Standard attention in three kernels (S = scale Q K^T to device memory in fp32, a row softmax
    writing P in bf16 and L, O = P V), the baseline of the fused forward.  Same arguments and result
    as fattn_fwd without a band or element mask; ``workspace`` a CUDA uint8 tensor of
    fattn_unfused_workspace_size bytes (allocated here if omitted).  Returns (out, lse)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.bfloat16)
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError(f"expected q [B,H,Nq,d], k/v [B,H,Nk,d]; got {tuple(q.shape)}, {tuple(k.shape)}, {tuple(v.shape)}")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("q and k/v disagree on B, H or d")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16)
    if lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    _check(lse, "lse", torch.float32)
    if workspace is None:
        workspace = torch.empty(fattn_unfused_workspace_size(B, H, Nq, Nk), dtype=torch.uint8, device=q.device)
    st = unfused_lib().fattn_fwd_unfused(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                         B, H, Nq, Nk, d, 1 if causal else 0, float(scale), workspace.data_ptr(),
                                         workspace.numel(), _stream_handle(stream, q.device))
    if st != FATTN_OK:
        raise FattnError(st, "fattn_fwd_unfused")
    return out, lse


def fattn_bwd_workspace_size(B: int, H: int, Nq: int, d: int) -> int:
    return lib().fattn_bwd_workspace_size(int(B), int(H), int(Nq), int(d))


def _mask_strides(mask, B, H, Nq, Nk):
    """(sb, sh) in 32-bit words for a pack_mask tensor shaped [Nq, W] or [B|1, H|1, Nq, W]."""
    import torch
    _check(mask, "mask", torch.int32)
    W = fattn_mask_row_words(Nk)
    m4 = mask.reshape(1, 1, *mask.shape) if mask.dim() == 2 else mask
    if m4.dim() != 4 or m4.shape[2:] != (Nq, W) or m4.shape[0] not in (1, B) or m4.shape[1] not in (1, H):
        raise ValueError(f"mask must be [Nq, {W}] or [B|1, H|1, Nq, {W}] int32 words; got {tuple(mask.shape)}")
    return (m4.shape[1] * Nq * W if m4.shape[0] > 1 else 0), (Nq * W if m4.shape[1] > 1 else 0)


def fattn_bwd_mask_workspace_size(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return lib().fattn_bwd_mask_workspace_size(int(B), int(H), int(Nq), int(Nk), int(d))


def fattn_bwd(q, k, v, out, lse, dout, causal: bool = False, scale: float | None = None, dq=None, dk=None,
              dv=None, workspace=None, stream=None, window=None, mask=None):
    """Gradients (dq, dk, dv) of the attention forward for an upstream gradient ``dout``.

    q: bf16 [B,H,Nq,d]; k, v: bf16 [B,H,Nk,d]; out (bf16) and lse (fp32 [B,H,Nq]) are the forward's
    outputs for the same inputs, mask and scale.  ``workspace`` is a CUDA uint8 tensor of at least
    fattn_bwd_workspace_size(B, H, Nq, d) bytes (fattn_bwd_mask_workspace_size(B, H, Nq, Nk, d) with
    ``mask``; allocated here if omitted).  ``mask`` is the element mask given to fattn_fwd
    (fattn_bwd_mask).  Returns bf16 tensors.
    """
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _check(t, n, torch.bfloat16)
    _check(lse, "lse", torch.float32)
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape or out.shape != q.shape or dout.shape != q.shape:
        raise ValueError("expected q, out, dout [B,H,Nq,d] and k, v [B,H,Nk,d]")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("q and k/v disagree on B, H or d")
    if tuple(lse.shape) != (B, H, Nq):
        raise ValueError("lse must be [B,H,Nq]")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = fattn_bwd_workspace_size(B, H, Nq, d) if mask is None else fattn_bwd_mask_workspace_size(B, H, Nq, Nk, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for t, n in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check(t, n, torch.bfloat16)
    if mask is not None:
        sb, sh = _mask_strides(mask, B, H, Nq, Nk)
        wl, wr = _band(causal, window)
        st = lib().fattn_bwd_mask(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                  dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d,
                                  mask.data_ptr(), sb, sh, wl, wr, float(scale), workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
        if st != FATTN_OK:
            raise FattnError(st, "fattn_bwd_mask")
        return dq, dk, dv
    if window is not None:
        st = lib().fattn_bwd_masked(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                                    dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk,
                                    d, int(window[0]), int(window[1]), float(scale), workspace.data_ptr(),
                                    workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
        if st != FATTN_OK:
            raise FattnError(st, "fattn_bwd_masked")
        return dq, dk, dv
    st = lib().fattn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), lse.data_ptr(),
                         dout.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, H, Nq, Nk, d,
                         1 if causal else 0, float(scale), workspace.data_ptr(),
                         workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    if st != FATTN_OK:
        raise FattnError(st, "fattn_bwd")
    return dq, dk, dv


def fattn_decode_num_splits(B: int, H: int, Nk: int, num_splits: int = 0) -> int:
    return lib().fattn_decode_num_splits(int(B), int(H), int(Nk), int(num_splits))


def fattn_decode_workspace_size(B: int, H: int, Nk: int, d: int, num_splits: int = 0) -> int:
    return lib().fattn_decode_workspace_size(int(B), int(H), int(Nk), int(d), int(num_splits))


def fattn_decode(q, k_cache, v_cache, scale: float | None = None, num_splits: int = 0, workspace=None,
                 out=None, lse=None, stream=None, want_lse: bool = True, window=None):
    """One query token per (b, h) against a KV cache, split-KV + combine on the GPU.

    q: bf16 [B,H,1,d]; k_cache, v_cache: bf16 [B,H,Nk,d].  ``workspace`` is a CUDA uint8 tensor of
    at least fattn_decode_workspace_size(...) bytes (allocated here if omitted).
    ``window=(window_left, window_right)`` restricts the query to the last window_left + 1 keys
    (fattn_decode_masked).  Returns (out bf16 [B,H,1,d], lse fp32 [B,H,1] or None).
    """
    import torch
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16)
    if q.dim() != 4 or q.shape[2] != 1 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("expected q [B,H,1,d] and k/v caches [B,H,Nk,d]")
    B, H, _, d = q.shape
    if k_cache.shape[0] != B or k_cache.shape[1] != H or k_cache.shape[3] != d:
        raise ValueError("q and the caches disagree on B, H or d")
    Nk = k_cache.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    need = fattn_decode_workspace_size(B, H, Nk, d, num_splits)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check(workspace, "workspace")
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16)
    if want_lse and lse is None:
        lse = torch.empty((B, H, 1), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32)
    if window is not None:
        st = lib().fattn_decode_masked(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                       lse.data_ptr() if lse is not None else None, B, H, Nk, d, int(window[0]),
                                       int(window[1]), float(scale), int(num_splits), workspace.data_ptr(),
                                       workspace.numel() * workspace.element_size(),
                                       _stream_handle(stream, q.device))
        if st != FATTN_OK:
            raise FattnError(st, "fattn_decode_masked")
        return out, lse
    st = lib().fattn_decode(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                            lse.data_ptr() if lse is not None else None, B, H, Nk, d, float(scale),
                            int(num_splits), workspace.data_ptr(),
                            workspace.numel() * workspace.element_size(),
                            _stream_handle(stream, q.device))
    if st != FATTN_OK:
        raise FattnError(st, "fattn_decode")
    return out, lse


def fattn_decode_static(q, k_cache, v_cache, scale: float | None = None, num_splits: int = 0, out=None,
                        lse=None, stream=None, want_lse: bool = True):
    """fattn_decode without a workspace, for callers that must not allocate device memory: the
    partial states go to a fixed array inside the library (FATTN_DECODE_STATIC_WORKSPACE_BYTES per
    device).  Calls whose GPU work overlaps race on that array.  Outputs are allocated here only when
    not passed in.  Returns (out, lse)."""
    import torch
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check(t, n, torch.bfloat16)
    if q.dim() != 4 or q.shape[2] != 1 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("expected q [B,H,1,d] and k/v caches [B,H,Nk,d]")
    B, H, _, d = q.shape
    if k_cache.shape[0] != B or k_cache.shape[1] != H or k_cache.shape[3] != d:
        raise ValueError("q and the caches disagree on B, H or d")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    _check(out, "out", torch.bfloat16)
    if want_lse and lse is None:
        lse = torch.empty((B, H, 1), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32)
    st = lib().fattn_decode_static(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                   lse.data_ptr() if lse is not None else None, B, H, k_cache.shape[2], d,
                                   float(scale), int(num_splits), _stream_handle(stream, q.device))
    if st != FATTN_OK:
        raise FattnError(st, "fattn_decode_static")
    return out, lse


def _check_host(t, name, dtype):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cpu":
        raise ValueError(f"{name} must be a host (CPU) tensor (got {t.device})")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype} (got {t.dtype})")


def _band(causal, window):
    if window is not None:
        return int(window[0]), int(window[1])
    return (-1, 0) if causal else (-1, -1)


def fattn_fwd_host_workspace_size(B, H, Nq, Nk, d, heads_per_chunk: int = 0) -> int:
    return lib().fattn_fwd_host_workspace_size(int(B), int(H), int(Nq), int(Nk), int(d), int(heads_per_chunk))


def fattn_decode_host_workspace_size(B, H, Nk, d, window_left: int = -1, heads_per_chunk: int = 0) -> int:
    return lib().fattn_decode_host_workspace_size(int(B), int(H), int(Nk), int(d), int(window_left),
                                                  int(heads_per_chunk))


def fattn_fwd_host(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
                   window=None, heads_per_chunk: int = 0, workspace=None, device=None, stream=None,
                   want_lse: bool = True):
    """fattn_fwd with q, k, v, out and lse in host memory (fattn_fwd_host): chunks of heads are copied
    in, computed and copied back with the copies overlapping the kernels.  Pinned host tensors give
    asynchronous copies.  ``workspace`` is a CUDA uint8 tensor of at least
    fattn_fwd_host_workspace_size(...) bytes (allocated here if omitted).  Synchronise ``stream``
    before reading out/lse.  Returns (out, lse)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check_host(t, n, torch.bfloat16)
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,H,Nq,d], k/v [B,H,Nk,d]")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("q and k/v disagree on B, H or d")
    Nk = k.shape[2]
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    _check_host(out, "out", torch.bfloat16)
    if want_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, pin_memory=True)
    if lse is not None:
        _check_host(lse, "lse", torch.float32)
    if workspace is None:
        need = fattn_fwd_host_workspace_size(B, H, Nq, Nk, d, heads_per_chunk)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    _check(workspace, "workspace")
    wl, wr = _band(causal, window)
    st = lib().fattn_fwd_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                              lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d, wl, wr, float(scale),
                              int(heads_per_chunk), workspace.data_ptr(),
                              workspace.numel() * workspace.element_size(), _stream_handle(stream, device))
    if st != FATTN_OK:
        raise FattnError(st, "fattn_fwd_host")
    return out, lse


def fattn_decode_host(q, k_cache, v_cache, scale: float | None = None, out=None, lse=None, window=None,
                      heads_per_chunk: int = 0, workspace=None, device=None, stream=None, want_lse: bool = True):
    """fattn_decode with q, the caches, out and lse in host memory (fattn_decode_host); with a
    window only the visible keys are copied.  Synchronise ``stream`` before reading out/lse.
    Returns (out, lse)."""
    import torch
    for t, n in ((q, "q"), (k_cache, "k_cache"), (v_cache, "v_cache")):
        _check_host(t, n, torch.bfloat16)
    if q.dim() != 4 or q.shape[2] != 1 or k_cache.dim() != 4 or v_cache.shape != k_cache.shape:
        raise ValueError("expected q [B,H,1,d] and k/v caches [B,H,Nk,d]")
    B, H, _, d = q.shape
    if k_cache.shape[0] != B or k_cache.shape[1] != H or k_cache.shape[3] != d:
        raise ValueError("q and the caches disagree on B, H or d")
    Nk = k_cache.shape[2]
    device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, pin_memory=True)
    _check_host(out, "out", torch.bfloat16)
    if want_lse and lse is None:
        lse = torch.empty((B, H, 1), dtype=torch.float32, pin_memory=True)
    if lse is not None:
        _check_host(lse, "lse", torch.float32)
    wl, wr = _band(False, window)
    if workspace is None:
        need = fattn_decode_host_workspace_size(B, H, Nk, d, wl, heads_per_chunk)
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=device)
    _check(workspace, "workspace")
    st = lib().fattn_decode_host(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                 lse.data_ptr() if lse is not None else None, B, H, Nk, d, wl, wr, float(scale),
                                 int(heads_per_chunk), workspace.data_ptr(),
                                 workspace.numel() * workspace.element_size(), _stream_handle(stream, device))
    if st != FATTN_OK:
        raise FattnError(st, "fattn_decode_host")
    return out, lse


def fattn_fwd_fp8_workspace_size(B, H, Nk, d) -> int:
    return lib().fattn_fwd_fp8_workspace_size(int(B), int(H), int(Nk), int(d))


def fattn_fwd_fp8(q, k, v, q_descale: float, k_descale: float, v_descale: float, causal: bool = False,
                  scale: float | None = None, window=None, out=None, lse=None, workspace=None, stream=None,
                  want_lse: bool = True):
    """Attention of q*q_descale, k*k_descale, v*v_descale (fattn_fwd_fp8): q, k, v are
    torch.float8_e4m3fn [B,H,N,d] CUDA tensors, d 64 or 128; out bf16, lse fp32.  ``workspace`` (a CUDA uint8
    tensor of fattn_fwd_fp8_workspace_size(...) bytes) receives V transposed; allocated here if
    omitted.  Returns (out, lse)."""
    import torch
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _check(t, n, torch.float8_e4m3fn)
    if q.dim() != 4 or k.dim() != 4 or v.shape != k.shape:
        raise ValueError("expected q [B,H,Nq,d], k/v [B,H,Nk,d]")
    B, H, Nq, d = q.shape
    if k.shape[0] != B or k.shape[1] != H or k.shape[3] != d:
        raise ValueError("q and k/v disagree on B, H or d")
    Nk = k.shape[2]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=torch.bfloat16, device=q.device)
    _check(out, "out", torch.bfloat16)
    if want_lse and lse is None:
        lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check(lse, "lse", torch.float32)
    if workspace is None:
        workspace = torch.empty(max(fattn_fwd_fp8_workspace_size(B, H, Nk, d), 256), dtype=torch.uint8,
                                device=q.device)
    _check(workspace, "workspace")
    wl, wr = _band(causal, window)
    st = lib().fattn_fwd_fp8(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                             lse.data_ptr() if lse is not None else None, B, H, Nq, Nk, d, wl, wr, float(scale),
                             float(q_descale), float(k_descale), float(v_descale), workspace.data_ptr(),
                             workspace.numel() * workspace.element_size(), _stream_handle(stream, q.device))
    if st != FATTN_OK:
        raise FattnError(st, "fattn_fwd_fp8")
    return out, lse


def fattn_fwd_recomputed_rows() -> int:
    """Rows of the forward that failed the fast path's range check (their query tiles computed again
    with a running max) on the current device so far (waits
    for the device)."""
    out = ctypes.c_ulonglong(0)
    st = lib().fattn_fwd_recomputed_rows(ctypes.byref(out))
    if st != 0:
        raise FattnError(st, "fattn_fwd_recomputed_rows")
    return int(out.value)


def fattn_last_error(stream=None) -> int:
    """Synchronise ``stream`` and read-and-clear the on-device status word (0 = OK, 4 = timeout;
    5 = a device-side check failed, debug builds only)."""
    import torch
    return lib().fattn_last_error(_stream_handle(stream, torch.device("cuda", torch.cuda.current_device())))


def fattn_debug_build() -> bool:
    """True when the loaded library is the build with device-side checks."""
    return bool(lib().fattn_debug_build())


def fattn_debug_take() -> tuple[int, int]:
    """(rules, first) of the device-side checks since the last call, then cleared (fattn_debug_take):
    rules is the OR of the broken rules' bits, first the first failure as block << 32 | thread << 8 |
    rule index + 1.  (0, 0) in release builds."""
    rules, first = ctypes.c_uint(0), ctypes.c_ulonglong(0)
    st = lib().fattn_debug_take(ctypes.byref(rules), ctypes.byref(first))
    if st != FATTN_OK:
        raise FattnError(st, "fattn_debug_take")
    return int(rules.value), int(first.value)
