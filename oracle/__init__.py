"""fp64 CPU oracle for the exact softmax-attention forward (O and LSE).

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference arm of ``bench.py`` may import this package.  The
product path (the CUDA library and its binding) never imports it, and it
imports nothing from the product path; both sides take inputs from
``attn_inputs`` only.

Three independent statements of the same definition live here:

* ``attn_fwd``        -- the C oracle (``attn_oracle.c``), fp64, a thread pool
                         over rows; materialises each score row.
* ``attn_fwd_numpy``  -- the definition again in numpy fp64, whole score matrix
                         per head (small cases; a second opinion on the C one).
* ``attn_fwd_online`` -- the tile-by-tile online-softmax recurrence in fp64,
                         written in the order of the Triton FA2 loop of
                         "FlashAttention-2 in an attention layer" and the
                         update of "FlashAttention V2" section 3; it checks the
                         algebra a tiled kernel relies on, not the kernel.

Two more for attention of a few new queries against a key/value cache
("FlashAttention V2", section 6: inference with a KV cache):

* ``attn_kvcache``       -- the C oracle (``oracle_attn_kvcache``), fp64.
* ``attn_kvcache_numpy`` -- the same definition in numpy fp64.

Parity status: pinned.  The pins (closed forms, invariants, brute force at
high precision) are in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/liboracle.so`` with gcc."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", _SRC,
           "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        dp = ctypes.POINTER(ctypes.c_double)
        lib.oracle_attn_fwd.argtypes = [
            dp, dp, dp, ctypes.c_longlong, ctypes.c_longlong,
            ctypes.c_longlong, ctypes.c_longlong, ctypes.c_int,
            ctypes.c_double, ctypes.POINTER(ctypes.c_longlong),
            ctypes.c_longlong, dp, dp, dp, ctypes.c_int]
        lib.oracle_attn_fwd.restype = ctypes.c_int
        lib.oracle_attn_kvcache.argtypes = [
            dp, dp, dp, ctypes.c_longlong, ctypes.c_longlong,
            ctypes.c_longlong, ctypes.c_longlong, ctypes.c_longlong,
            ctypes.POINTER(ctypes.c_longlong), ctypes.c_int, ctypes.c_double,
            dp, dp, ctypes.c_int]
        lib.oracle_attn_kvcache.restype = ctypes.c_int
        _lib = lib
    return _lib


def _f64(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)))


def attn_fwd(q, k, v, causal: bool, scale: float, rows=None, threads=None,
             want_p: bool = False):
    """The C oracle.  ``q, k, v``: ``[B, H, S, D]`` arrays (any float dtype,
    widened exactly to fp64).  ``rows``: optional global row indices
    ``bh * S + i``.  Returns ``(O, LSE)`` (and ``P`` if ``want_p``) in fp64;
    shapes ``[B, H, S, D]`` / ``[B, H, S]`` for all rows, else ``[n, D]`` /
    ``[n]`` in the order of ``rows``."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or q.shape != k.shape or q.shape != v.shape:
        raise ValueError("q, k, v must share one [B, H, S, D] shape")
    B, H, S, D = q.shape
    if rows is None:
        n = B * H * S
        rows_arr = None
    else:
        rows_arr = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
        n = rows_arr.shape[0]
    o = np.empty((n, D), dtype=np.float64)
    lse = np.empty(n, dtype=np.float64)
    p = np.empty((n, S), dtype=np.float64) if want_p else None
    rc = _load().oracle_attn_fwd(
        _ptr(q), _ptr(k), _ptr(v), B, H, S, D, int(bool(causal)),
        float(scale),
        None if rows_arr is None else
        rows_arr.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
        n, _ptr(o), _ptr(lse), None if p is None else _ptr(p),
        int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_fwd failed with code {rc}")
    if rows is None:
        o = o.reshape(B, H, S, D)
        lse = lse.reshape(B, H, S)
        if p is not None:
            p = p.reshape(B, H, S, S)
    return (o, lse, p) if want_p else (o, lse)


def attn_fwd_numpy(q, k, v, causal: bool, scale: float, want_p: bool = False):
    """The definition in numpy fp64 over whole score matrices (small inputs).

    ``scores = scale * Q K^T``; the causal mask removes keys after the query;
    softmax over keys; ``O = P V``; ``LSE = m + ln(sum exp(s - m))``.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    S = q.shape[-2]
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    if causal:
        allowed = np.tril(np.ones((S, S), dtype=bool))
        s = np.where(allowed, s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    p = e / l
    o = np.einsum("bhij,bhjd->bhid", p, v)
    lse = (m + np.log(l))[..., 0]
    return (o, lse, p) if want_p else (o, lse)


def attn_fwd_online(q, k, v, causal: bool, scale: float, block_m: int = 128,
                    block_n: int = 128, lazy_threshold: float = 0.0):
    """Online-softmax recurrence in fp64, tile by tile.

    For each query tile: running max ``m`` (start -inf), running sum ``l``
    (start 0) and unnormalised accumulator ``acc`` (start 0).  For each key
    tile (stopping after the diagonal tile when causal): scores times scale,
    masked (causal keeps key <= query, keys past S removed),
    ``m_new = max(m, rowmax)``, ``alpha = exp(m - m_new)``,
    ``p = exp(s - m_new)``, ``l = alpha * l + rowsum(p)``,
    ``acc = alpha * acc + p V``, ``m = m_new``.  After the last key tile
    ``O = acc / l`` (one division) and ``LSE = m + ln l``.

    ``lazy_threshold > 0`` keeps the reference maximum until a tile's maximum
    exceeds it by more than that amount (natural-log units); the algebra is
    unchanged because ``acc``, ``l`` and the exponent share the reference.
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, S, D = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((B, H, S))
    for b in range(B):
        for h in range(H):
            for i0 in range(0, S, block_m):
                i1 = min(S, i0 + block_m)
                qi = q[b, h, i0:i1]
                rows = np.arange(i0, i1)
                m = np.full(i1 - i0, -np.inf)
                l = np.zeros(i1 - i0)
                acc = np.zeros((i1 - i0, D))
                end_n = min(S, i0 + block_m) if causal else S
                for j0 in range(0, end_n, block_n):
                    j1 = min(S, j0 + block_n)
                    cols = np.arange(j0, j1)
                    s = scale * (qi @ k[b, h, j0:j1].T)
                    if causal:
                        s = np.where(rows[:, None] >= cols[None, :], s, -np.inf)
                    m_new = np.maximum(m, s.max(axis=1))
                    if lazy_threshold > 0:
                        m_new = np.where(s.max(axis=1) > m + lazy_threshold,
                                         m_new, m)
                    alpha = np.exp(m - m_new)
                    p = np.exp(s - m_new[:, None])
                    l = alpha * l + p.sum(axis=1)
                    acc = alpha[:, None] * acc + p @ v[b, h, j0:j1]
                    m = m_new
                o[b, h, i0:i1] = acc / l[:, None]
                lse[b, h, i0:i1] = m + np.log(l)
    return o, lse



def _lens_array(lens, B: int, Sk: int):
    if lens is None:
        return None
    a = np.ascontiguousarray(np.asarray(lens, dtype=np.int64))
    if a.shape != (B,):
        raise ValueError("lens must have one entry per batch")
    return a


def attn_kvcache(q, k, v, causal: bool, scale: float, lens=None, threads=None):
    """The C oracle for new queries against a cache.  ``q``: ``[B, H, Sq, D]``;
    ``k, v``: ``[B, H, Sk, D]`` caches; ``lens``: cached length per batch
    (``None``: all ``Sk``).  Query ``i`` is position ``len_b - Sq + i``; causal
    keeps keys at or before that position.  Returns fp64 ``(O, LSE)``; a query
    with no allowed key gets ``O = 0``, ``LSE = -inf``."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    if q.ndim != 4 or k.shape != v.shape or k.ndim != 4:
        raise ValueError("q must be [B, H, Sq, D]; k and v one [B, H, Sk, D]")
    B, H, Sq, D = q.shape
    if k.shape[:2] != (B, H) or k.shape[3] != D:
        raise ValueError("q and the caches disagree on B, H or D")
    Sk = k.shape[2]
    la = _lens_array(lens, B, Sk)
    o = np.empty((B, H, Sq, D), dtype=np.float64)
    lse = np.empty((B, H, Sq), dtype=np.float64)
    rc = _load().oracle_attn_kvcache(
        _ptr(q), _ptr(k), _ptr(v), B, H, Sq, Sk, D,
        None if la is None else la.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)),
        int(bool(causal)), float(scale), _ptr(o), _ptr(lse),
        int(threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"oracle_attn_kvcache failed with code {rc}")
    return o, lse


def attn_kvcache_numpy(q, k, v, causal: bool, scale: float, lens=None):
    """The cache definition in numpy fp64, one head at a time: scores of the
    Sq queries against the first ``len_b`` cached keys, the causal mask
    ``j <= len_b - Sq + i``, softmax, ``O = P V``; empty rows give 0 / -inf."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    la = _lens_array(lens, B, Sk)
    o = np.zeros((B, H, Sq, D))
    lse = np.full((B, H, Sq), -np.inf)
    for b in range(B):
        n = Sk if la is None else int(la[b])
        if n == 0:
            continue
        pos = n - Sq + np.arange(Sq)
        allowed = np.ones((Sq, n), dtype=bool)
        if causal:
            allowed = np.arange(n)[None, :] <= pos[:, None]
        for h in range(H):
            s = scale * (q[b, h] @ k[b, h, :n].T)
            s = np.where(allowed, s, -np.inf)
            rows = allowed.any(axis=1)
            m = np.where(rows, s.max(axis=1, initial=-np.inf), 0.0)
            e = np.exp(s - m[:, None])
            l = e.sum(axis=1)
            o[b, h, rows] = (e[rows] @ v[b, h, :n]) / l[rows, None]
            lse[b, h, rows] = m[rows] + np.log(l[rows])
    return o, lse
