"""Exact softmax-attention forward on GB300 (sm_103a).

A thin ctypes binding over ``libfattn.so`` (C ABI in ``include/fattn.h``):
argument marshalling only.  Every step of the computation runs in the CUDA
kernels of that library; there is no other implementation to fall back to, and
calling into a missing library raises.

    o, lse = forward(q, k, v, causal=True)      # torch tensors on a GB300
    o, lse = forward_kvcache(q_new, k_cache, v_cache, cache_lens)  # decoding

``q, k, v``: contiguous ``[B, H, S, D]`` fp16 or bf16 CUDA tensors, D in
{64, 128, 256}.  Returns ``o`` (same shape and dtype) and ``lse``
(``[B, H, S]`` fp32, natural log of the row's softmax normaliser over scaled
scores).  The library works on the calling thread's current device; the
torch wrappers make q's device current for the call.
"""
from __future__ import annotations

import ctypes
import math
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfattn.so")

FATTN_OK = 0
FATTN_ERR_INVALID_ARG = -1
FATTN_ERR_UNSUPPORTED = -2
FATTN_ERR_MISALIGNED = -3
FATTN_ERR_TOO_LARGE = -4
FATTN_ERR_LAUNCH = -5
FATTN_ERR_PIPELINE_TIMEOUT = -6
FATTN_ERR_CUDA = -7
FATTN_FP16 = 0
FATTN_BF16 = 1

_lib = None


class FattnError(RuntimeError):
    """A non-zero status from the library."""

    def __init__(self, status: int, what: str = "fattn_fwd"):
        self.status = status
        super().__init__(f"{what} failed: {status} ({fattn_error_string(status)})")


def lib() -> ctypes.CDLL:
    """The loaded library; raises ImportError if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(
                f"{LIB_PATH} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        l = ctypes.CDLL(LIB_PATH)
        vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
        ip = ctypes.POINTER(ctypes.c_int)
        l.fattn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp]
        l.fattn_fwd.restype = i
        l.fattn_last_error.argtypes = [vp, ip]
        l.fattn_last_error.restype = i
        l.fattn_error_string.argtypes = [i]
        l.fattn_error_string.restype = ctypes.c_char_p
        l.fattn_plan.argtypes = [i, i, i, i, i, ip, ip, ip, ip, ip, ip]
        l.fattn_plan.restype = i
        l.fattn_causal_order.argtypes = [i, i, i, i, i, i, ip, ip]
        l.fattn_causal_order.restype = i
        l.fattn_check_wait_timeout.argtypes = [i, vp]
        l.fattn_check_wait_timeout.restype = i
        u64 = ctypes.c_ulonglong
        l.fattn_fwd_kvcache.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                        i, f, i, vp, u64, vp]
        l.fattn_fwd_kvcache.restype = i
        l.fattn_kvcache_plan.argtypes = [i, i, i, i, i, ctypes.POINTER(u64),
                                         ip, ip, ip, ip]
        l.fattn_kvcache_plan.restype = i
        l.fattn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, f, f, f, i, vp]
        l.fattn_fwd_fp8.restype = i
        l.fattn_fwd_kvcache_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i, i,
                                                i, i, i, i, f, i, vp, vp]
        l.fattn_fwd_kvcache_noalloc.restype = i
        l.fattn_version.argtypes = []
        l.fattn_version.restype = i
        _lib = l
    return _lib


# ------------------------------------------------------- the C ABI, by name

def fattn_fwd(q, k, v, o, lse, B, H, S, D, causal, scale, dtype, stream) -> int:
    """``fattn_fwd`` with integer device pointers and an integer stream."""
    return lib().fattn_fwd(q, k, v, o, lse, B, H, S, D, int(causal),
                           float(scale), dtype, stream)


def fattn_last_error(stream=0):
    """(status, (where, block)) of the last kernel error on this device."""
    detail = (ctypes.c_int * 2)()
    rc = lib().fattn_last_error(stream, detail)
    return rc, (detail[0], detail[1])


def fattn_error_string(status: int) -> str:
    return lib().fattn_error_string(status).decode()


def fattn_check_wait_timeout(timeout_us: int, stream=None) -> int:
    """Enqueue the bounded-wait check (a wait that nothing completes gives up
    after ``timeout_us`` and records a pipeline timeout); read the outcome
    with ``fattn_last_error``."""
    return lib().fattn_check_wait_timeout(int(timeout_us), stream)


def fattn_plan(B, H, S, D, causal=False) -> dict:
    """The launch ``fattn_fwd`` would make (grid, block, smem, units...)."""
    vals = [ctypes.c_int() for _ in range(6)]
    rc = lib().fattn_plan(B, H, S, D, int(causal), *[ctypes.byref(x) for x in vals])
    if rc != FATTN_OK:
        raise FattnError(rc, "fattn_plan")
    keys = ("grid", "block", "smem_bytes", "units", "q_tiles_per_unit",
            "kv_stages")
    return {k_: x.value for k_, x in zip(keys, vals)}


def fattn_causal_order(B, H, S, D, elem_bytes=2, sms=152) -> dict:
    """The work order of a causal launch (heads per group, units handed out
    at run time or not) on a device with ``sms`` SMs; host only."""
    g, rt = ctypes.c_int(), ctypes.c_int()
    rc = lib().fattn_causal_order(B, H, S, D, elem_bytes, sms, ctypes.byref(g),
                                  ctypes.byref(rt))
    if rc != FATTN_OK:
        raise FattnError(rc, "fattn_causal_order")
    return {"group_heads": g.value, "run_time": bool(rt.value)}


def fattn_fwd_fp8(q, k, v, o, lse, B, H, S, D, causal, scale, q_scale, k_scale,
                  v_scale, out_dtype, stream) -> int:
    """``fattn_fwd_fp8`` with integer device pointers and an integer stream."""
    return lib().fattn_fwd_fp8(q, k, v, o, lse, B, H, S, D, int(causal), float(scale),
                               float(q_scale), float(k_scale), float(v_scale),
                               out_dtype, stream)


def fattn_fwd_kvcache(q, k_cache, v_cache, cache_lens, o, lse, B, H, Sq, Sk,
                      D, causal, scale, dtype, workspace, workspace_bytes,
                      stream) -> int:
    """``fattn_fwd_kvcache`` with integer device pointers (``cache_lens`` may
    be 0 for every length equal to ``Sk``) and an integer stream."""
    return lib().fattn_fwd_kvcache(q, k_cache, v_cache, cache_lens or None, o,
                                   lse, B, H, Sq, Sk, D, int(causal),
                                   float(scale), dtype, workspace,
                                   int(workspace_bytes), stream)


def fattn_fwd_kvcache_noalloc(q, k_cache, v_cache, cache_lens, o, lse, B, H,
                              Sq, Sk, D, causal, scale, dtype, status_words,
                              stream) -> int:
    """``fattn_fwd_kvcache_noalloc`` with integer device pointers
    (``cache_lens`` and ``status_words`` may be 0) and an integer stream."""
    return lib().fattn_fwd_kvcache_noalloc(
        q, k_cache, v_cache, cache_lens or None, o, lse, B, H, Sq, Sk, D,
        int(causal), float(scale), dtype, status_words or None, stream)


def fattn_kvcache_plan(B, H, Sq, Sk, D) -> dict:
    """The launch ``fattn_fwd_kvcache`` would make on the current device."""
    ws = ctypes.c_ulonglong()
    vals = [ctypes.c_int() for _ in range(4)]
    rc = lib().fattn_kvcache_plan(B, H, Sq, Sk, D, ctypes.byref(ws),
                                  *[ctypes.byref(x) for x in vals])
    if rc != FATTN_OK:
        raise FattnError(rc, "fattn_kvcache_plan")
    out = {"workspace_bytes": ws.value}
    out.update({k_: x.value for k_, x in
                zip(("grid", "block", "smem_bytes", "split_warps"), vals)})
    return out


def fattn_version() -> int:
    return lib().fattn_version()


# ------------------------------------------------------------ torch wrapper

def _dtype_code(t):
    import torch
    if t.dtype == torch.float16:
        return FATTN_FP16
    if t.dtype == torch.bfloat16:
        return FATTN_BF16
    raise TypeError(f"unsupported dtype {t.dtype}; expected float16 or bfloat16")


def forward(q, k, v, causal: bool = False, scale: float | None = None,
            out=None, lse=None, stream=None):
    """Attention forward on the current CUDA stream (or ``stream``).

    Allocates ``o`` and ``lse`` with torch on q's device unless given.
    Raises FattnError on any non-zero status."""
    import torch
    if q.dim() != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, S, D] shape")
    if not (q.is_contiguous() and k.is_contiguous() and v.is_contiguous()):
        raise ValueError("q, k, v must be contiguous")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share a dtype")
    if not q.is_cuda:
        raise ValueError("q, k, v must be CUDA tensors")
    B, H, S, D = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                       lse.data_ptr(), B, H, S, D, causal, scale, _dtype_code(q),
                       stream.cuda_stream)
    if rc != FATTN_OK:
        raise FattnError(rc)
    return out, lse


def forward_kvcache(q, k_cache, v_cache, cache_lens=None, causal: bool = False,
                    scale: float | None = None, out=None, lse=None,
                    workspace=None, stream=None):
    """Attention of ``Sq`` new queries against a key/value cache.

    ``q``: contiguous ``[B, H, Sq, D]`` (Sq <= 16); ``k_cache, v_cache``:
    contiguous ``[B, H, Sk, D]`` of the same dtype; ``cache_lens``: optional
    int32 CUDA tensor ``[B]`` of cached lengths (default: all ``Sk``).  Query
    ``i`` sits at position ``len_b - Sq + i``; ``causal`` keeps keys up to it.
    ``workspace``: optional uint8 CUDA tensor of at least
    ``fattn_kvcache_plan(...)["workspace_bytes"]`` bytes (allocated here if
    absent).  Returns ``(o, lse)``; raises FattnError on a non-zero status."""
    import torch
    if q.dim() != 4 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("q must be [B, H, Sq, D]; caches one [B, H, Sk, D]")
    B, H, Sq, D = q.shape
    if k_cache.shape[0] != B or k_cache.shape[1] != H or k_cache.shape[3] != D:
        raise ValueError("q and the caches disagree on B, H or D")
    Sk = k_cache.shape[2]
    for t in (q, k_cache, v_cache):
        if not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q and the caches must be contiguous CUDA tensors")
    if not (q.dtype == k_cache.dtype == v_cache.dtype):
        raise TypeError("q and the caches must share a dtype")
    lens_ptr = 0
    if cache_lens is not None:
        if (cache_lens.dtype != torch.int32 or cache_lens.shape != (B,)
                or not cache_lens.is_contiguous() or not cache_lens.is_cuda):
            raise ValueError("cache_lens must be a contiguous int32 CUDA tensor [B]")
        lens_ptr = cache_lens.data_ptr()
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if workspace is None:
        need = fattn_kvcache_plan(B, H, Sq, Sk, D)["workspace_bytes"]
        workspace = torch.empty(max(16, need), dtype=torch.uint8, device=q.device)
    if stream is None:
        stream = torch.cuda.current_stream(q.device)
    with torch.cuda.device(q.device):
        rc = fattn_fwd_kvcache(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                               lens_ptr, out.data_ptr(), lse.data_ptr(), B, H, Sq,
                               Sk, D, causal, scale, _dtype_code(q),
                               workspace.data_ptr(), workspace.numel(),
                               stream.cuda_stream)
    if rc != FATTN_OK:
        raise FattnError(rc, "fattn_fwd_kvcache")
    return out, lse


def forward_fp8(q8, k8, v8, q_scale: float, k_scale: float, v_scale: float,
                causal: bool = False, scale: float | None = None, out_dtype=None,
                out=None, lse=None, stream=None):
    """Attention with E4M3 inputs.  ``q8, k8, v8``: contiguous ``[B, H, S,
    128]`` CUDA tensors of E4M3 codes (``torch.uint8`` or
    ``torch.float8_e4m3fn``); real values are code value times the scale.
    Returns ``(o, lse)``; ``o`` in ``out_dtype`` (default bf16)."""
    import torch
    if q8.dim() != 4 or q8.shape != k8.shape or q8.shape != v8.shape:
        raise ValueError("q8, k8, v8 must share one [B, H, S, D] shape")
    for t in (q8, k8, v8):
        if t.element_size() != 1 or not t.is_contiguous() or not t.is_cuda:
            raise ValueError("q8, k8, v8 must be contiguous one-byte CUDA tensors")
    B, H, S, D = q8.shape
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if out_dtype is None:
        out_dtype = torch.bfloat16
    code = _dtype_code(torch.empty(0, dtype=out_dtype))
    if out is None:
        out = torch.empty((B, H, S, D), dtype=out_dtype, device=q8.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q8.device)
    if stream is None:
        stream = torch.cuda.current_stream(q8.device)
    with torch.cuda.device(q8.device):
        rc = fattn_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), out.data_ptr(),
                           lse.data_ptr(), B, H, S, D, causal, scale, q_scale, k_scale,
                           v_scale, code, stream.cuda_stream)
    if rc != FATTN_OK:
        raise FattnError(rc, "fattn_fwd_fp8")
    return out, lse
