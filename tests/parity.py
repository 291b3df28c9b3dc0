"""Shared parity helpers for the GPU tests: run the CUDA path through the C
ABI, run the oracle, compare with the stated tolerances.

Tolerances (the library's accuracy targets): fp16 max|O - O_ref| <= 2e-3,
bf16 <= 1.5e-2, |LSE - LSE_ref| <= 1e-3.  Reading adopted for the
bf16 floor: casting O to bf16 alone can miss by half a unit in the last place,
which exceeds 1.5e-2 once |O_ref| >= 4 (spacing 2^-5 there), so an element
with |O_ref| >= 4 also passes when its error is within 1.5e-2 plus half an
ulp of the dtype at O_ref.  The literal maximum error is always reported.
"""
from __future__ import annotations

import math
import warnings

import numpy as np

import attn_inputs
import oracle

TOL_O = {"fp16": 2e-3, "bf16": 1.5e-2}
TOL_LSE = 1e-3
MANT_BITS = {"fp16": 10, "bf16": 7}


def ulp(x: np.ndarray, dtype: str) -> np.ndarray:
    """Spacing of the 16-bit dtype at |x| (normal range)."""
    ax = np.maximum(np.abs(x), 2.0 ** -14)
    return np.exp2(np.floor(np.log2(ax)) - MANT_BITS[dtype])


def torch_dtype(dtype: str):
    import torch
    return torch.float16 if dtype == "fp16" else torch.bfloat16


def run_cuda(x: attn_inputs.QKV, causal: bool, scale: float | None = None,
             poison: bool = True):
    """The CUDA path through the C ABI; outputs as fp64 numpy arrays."""
    import torch

    import exact_attention_forward_10_gb300 as fattn

    dev = torch.device("cuda:0")
    tdt = torch_dtype(x.dtype)
    q, k, v = (torch.from_numpy(a).to(dev).to(tdt) for a in (x.q, x.k, x.v))
    B, H, S, D = x.q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    if poison:  # every element must be written
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
    fattn.forward(q, k, v, causal=causal, scale=scale, out=o, lse=lse)
    torch.cuda.synchronize()
    rc, where = fattn.fattn_last_error(0)
    assert rc == 0, f"kernel status {rc} ({fattn.fattn_error_string(rc)}) at {where}"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def sample_rows(B: int, H: int, S: int, seed: int, n_heads: int | None = None,
                stride: int = 64):
    """Global row indices: every row of the first and last 128-row tiles plus
    a seeded 1-in-``stride`` sample of the rest, in every (batch, head) by
    default (the persistent schedule gives each head's work units to
    different CTAs and rounds), or with ``n_heads`` in a few heads only
    (first, last, seeded others)."""
    rng = np.random.default_rng(seed)
    BH = B * H
    if n_heads is None:
        heads = list(range(BH))
    else:
        heads = sorted({0, BH - 1, *rng.integers(0, BH, size=max(0, n_heads - 2)).tolist()})
    rows = []
    for bh in heads:
        r = set(range(min(S, 128)))
        r |= set(range(max(0, S - 128 - S % 128), S))
        r |= set(rng.choice(S, size=max(1, S // stride), replace=False).tolist())
        rows += [bh * S + i for i in sorted(r)]
    return np.asarray(rows, dtype=np.int64)


def compare(o, lse, ro, rl, dtype: str, label: str = ""):
    """Assert parity; returns (max|dO|, max|dLSE|)."""
    assert np.isfinite(o).all(), f"{label}: non-finite (unwritten?) O"
    assert np.isfinite(lse).all(), f"{label}: non-finite (unwritten?) LSE"
    err = np.abs(o - ro)
    tol = TOL_O[dtype]
    ok = (err <= tol) | ((np.abs(ro) >= 4.0) & (err <= tol + 0.5 * ulp(ro, dtype)))
    e_o = float(err.max()) if err.size else 0.0
    e_l = float(np.abs(lse - rl).max()) if lse.size else 0.0
    if not ok.all():
        idx = np.unravel_index(np.argmax(np.where(ok, 0, err)), err.shape)
        raise AssertionError(
            f"{label}: O mismatch at {idx}: got {o[idx]}, want {ro[idx]} "
            f"(max|dO|={e_o:.3e}, {int((~ok).sum())} elements out of tolerance)")
    assert e_l <= TOL_LSE, f"{label}: max|dLSE|={e_l:.3e} > {TOL_LSE}"
    n_ulp = int((err > tol).sum())
    if n_ulp:
        # within the per-element reading only: say so in the run's summary
        warnings.warn(f"{label}: {n_ulp} elements exceed the flat bound {tol} and pass "
                      f"through the half-ulp allowance at |O_ref| >= 4 (max|dO|={e_o:.3e})")
    return e_o, e_l


def check_full(x: attn_inputs.QKV, causal: bool, label: str = ""):
    """Every element against the oracle (sizes the oracle finishes quickly)."""
    D = x.q.shape[-1]
    scale = 1.0 / math.sqrt(D)
    o, lse = run_cuda(x, causal)
    ro, rl = oracle.attn_fwd(x.q, x.k, x.v, causal, scale)
    return compare(o, lse, ro, rl, x.dtype, label)


def check_sampled(x: attn_inputs.QKV, causal: bool, seed: int, label: str = "",
                  stride: int = 64, n_heads: int | None = None):
    """Sampled rows against the oracle (full-size workloads)."""
    B, H, S, D = x.q.shape
    scale = 1.0 / math.sqrt(D)
    o, lse = run_cuda(x, causal)
    assert np.isfinite(o).all() and np.isfinite(lse).all(), f"{label}: unwritten output"
    rows = sample_rows(B, H, S, seed, n_heads=n_heads, stride=stride)
    ro, rl = oracle.attn_fwd(x.q, x.k, x.v, causal, scale, rows=rows)
    return compare(o.reshape(-1, D)[rows], lse.reshape(-1)[rows], ro, rl,
                   x.dtype, label)


# ------------------------------------------------ attention against a cache

def run_cuda_kvcache(x: attn_inputs.KVCache, causal: bool, scale: float,
                     lens=None, poison: bool = True, workspace=None,
                     stale_nan: bool = False):
    """The cache path through the C ABI; outputs as fp64 numpy arrays.
    ``stale_nan`` fills every cache row at or past its batch's length with
    NaN before the call (those rows must not matter)."""
    import torch

    import exact_attention_forward_10_gb300 as fattn

    dev = torch.device("cuda:0")
    tdt = torch_dtype(x.dtype)
    q, k, v = (torch.from_numpy(a).to(dev).to(tdt) for a in (x.q, x.k, x.v))
    if lens is None:
        lens = x.lens
    lt = None
    if lens is not None:
        lt = torch.as_tensor(np.asarray(lens), dtype=torch.int32, device=dev)
        if stale_nan:
            for b, n in enumerate(np.asarray(lens).tolist()):
                k[b, :, n:] = float("nan")
                v[b, :, n:] = float("nan")
    B, H, Sq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    if poison:
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
    fattn.forward_kvcache(q, k, v, lt, causal=causal, scale=scale, out=o,
                          lse=lse, workspace=workspace)
    torch.cuda.synchronize()
    rc, where = fattn.fattn_last_error(0)
    assert rc == 0, f"kernel status {rc} ({fattn.fattn_error_string(rc)}) at {where}"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()


def compare_kvcache(o, lse, ro, rl, dtype: str, label: str = ""):
    """Parity for the cache path: rows with no allowed key must be exactly
    O = 0 and LSE = -inf; every other element as in ``compare``."""
    assert not np.isnan(o).any(), f"{label}: NaN (unwritten?) O"
    assert not np.isnan(lse).any(), f"{label}: NaN (unwritten?) LSE"
    empty = np.isneginf(rl)
    np.testing.assert_array_equal(np.isneginf(lse), empty,
                                  err_msg=f"{label}: empty-row pattern")
    assert np.all(o[empty] == 0.0), f"{label}: empty rows must be zero"
    full = ~empty
    return compare(o[full], lse[full], ro[full], rl[full], dtype, label)


def check_kvcache(x: attn_inputs.KVCache, causal: bool, label: str = "",
                  stale_nan: bool = False):
    """Every element of the cache path against the fp64 cache oracle."""
    D = x.q.shape[-1]
    scale = 1.0 / math.sqrt(D)
    o, lse = run_cuda_kvcache(x, causal, scale, stale_nan=stale_nan)
    ro, rl = oracle.attn_kvcache(x.q, x.k, x.v, causal, scale, x.lens)
    return compare_kvcache(o, lse, ro, rl, x.dtype, label)


# ------------------------------------------------------ E4M3 (FP8) inputs

def fp8_bound(x: attn_inputs.QKV8, causal: bool, scale: float):
    """fp64 oracle result and a per-element error bound for the FP8 path.

    The kernel rounds every attention weight to E4M3 before P V: for weights
    normalised to the row maximum, |p~ - p| <= max(2^-4 p, 2^-10) (relative
    half-ulp in the normal range, half the subnormal quantum below it; the
    lazy reference maximum only rescales p by 2^0..2^8, which keeps both
    limits).  The kernel normalises by the sum of the rounded weights, so O =
    sum w~_j v_j with w~ = p~ / sum p~, and with e_j = max(2^-4 p_j, 2^-10),
    L = sum p_j >= 1 (the maximum contributes 1) and sum p~ >= L (1 - 2^-4):
      |O - O_ref| = |sum (w~_j - w_j)(v_j - O_ref)|
                  <= (16/15) [sum e_j |v_j - O_ref| + (sum e_j) M] / L,
    M = sum_j w_j |v_j - O_ref|; plus the 16-bit output rounding (2^-8 |O|)
    and 1e-5 for fp32 accumulation and ex2.  Returns (O_ref, LSE_ref, tol),
    numpy fp64, for inputs small enough for the whole P."""
    ro, rl, P = oracle.attn_fwd_numpy(x.q, x.k, x.v, causal, scale, want_p=True)
    return ro, rl, _fp8_tol(P, x.v, ro)


def _fp8_tol(P, v, ro):
    """The bound of fp8_bound from probabilities P [..., i, j], values v
    [..., j, d] and the reference output ro [..., i, d]."""
    pn = P / P.max(axis=-1, keepdims=True)      # weights relative to the row max
    err_w = np.maximum(2.0 ** -4 * pn, np.where(pn > 0, 2.0 ** -10, 0.0))
    L = pn.sum(axis=-1)
    dev = np.abs(v[..., None, :, :] - ro[..., :, None, :])  # [..., i, j, d]
    M = np.einsum("...ij,...ijd->...id", pn / L[..., None], dev)
    tol = (16.0 / 15.0) * (np.einsum("...ij,...ijd->...id", err_w, dev) +
                           err_w.sum(axis=-1)[..., None] * M) / L[..., None]
    return tol + 2.0 ** -8 * np.abs(ro) + 1e-5


def fp8_bound_rows(x: attn_inputs.QKV8, causal: bool, scale: float, bh: int, rows):
    """fp8_bound for some query rows of head ``bh`` (long sequences): the
    definition in fp64 numpy on those rows only."""
    B, H, S, D = x.q.shape
    b, h = divmod(bh, H)
    rows = np.asarray(rows)
    s = scale * (x.q[b, h, rows] @ x.k[b, h].T)          # [n, S]
    if causal:
        s = np.where(np.arange(S)[None, :] <= rows[:, None], s, -np.inf)
    m = s.max(axis=-1, keepdims=True)
    e = np.exp(s - m)
    l = e.sum(axis=-1, keepdims=True)
    P = e / l
    ro = P @ x.v[b, h]
    rl = (m + np.log(l))[:, 0]
    return ro, rl, _fp8_tol(P, x.v[b, h], ro)


# Workloads of the FP8 RMS check, (B, H, S, seed, Q/K multiplier), head dim
# 128: the kernel's RMS error against the oracle, relative to that of
# ``fp8_model`` with the reference at the row maximum, measured on GB300
# (both masks): 1.000 with one key tile (S = 127), 1.00-1.16 over several
# tiles (the lazy reference lags the maximum).  The same model with two
# mantissa bits per weight gives 1.89-2.01.
FP8_RMS_CASES = [(1, 2, 127, 6127, 1.0), (1, 2, 300, 6300, 1.0),
                 (1, 2, 513, 6513, 1.0), (2, 3, 1000, 6100, 1.0),
                 (1, 4, 777, 6200, 4.0)]
FP8_RMS_MAX = 1.4    # two mantissa bits double the ratio
FP8_RMS_MIN = 0.7    # no E4M3 rounding of the weights would drop it far below


def fp8_round_e4m3(x):
    """Nearest E4M3 values (ties to even, subnormals, saturating at 448)."""
    return attn_inputs.e4m3_decode(attn_inputs.e4m3_encode(x))


def fp8_model(q, k, v, causal: bool, scale: float, lag, rounding=fp8_round_e4m3,
              rounded_sum: bool = True, out_dtype: str = "bf16"):
    """The FP8 forward's arithmetic in fp64 with its roundings made explicit
    ("FlashAttention V2", section 7: FP8 attention): scores of the real
    values, scaled and masked; weights p = exp(s - m_ref) against a
    reference maximum ``lag`` (natural-log units, per row, >= 0) below the
    row's true maximum; every weight rounded (``rounding``, E4M3 by
    default); O = sum p~ v / sum p~ (``rounded_sum=False``: divided by the
    sum of the unrounded weights instead); O rounded to ``out_dtype``."""
    S = q.shape[-2]
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    if causal:
        s = np.where(np.tril(np.ones((S, S), dtype=bool)), s, -np.inf)
    m_ref = s.max(axis=-1, keepdims=True) - np.asarray(lag)[..., None]
    p = np.exp(s - m_ref)
    pr = rounding(p)
    den = pr.sum(axis=-1) if rounded_sum else p.sum(axis=-1)
    o = np.einsum("bhij,bhjd->bhid", pr, v) / den[..., None]
    return attn_inputs.round_to_dtype(o, out_dtype)


def run_cuda_fp8(x: attn_inputs.QKV8, causal: bool, scale: float, out_dtype: str = "bf16"):
    import torch

    import exact_attention_forward_10_gb300 as fattn

    dev = torch.device("cuda:0")
    q8, k8, v8 = (torch.from_numpy(a).to(dev) for a in (x.q8, x.k8, x.v8))
    B, H, S, D = q8.shape
    o = torch.full((B, H, S, D), float("nan"), dtype=torch_dtype(out_dtype), device=dev)
    lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=dev)
    fattn.forward_fp8(q8, k8, v8, *x.descale, causal=causal, scale=scale,
                      out_dtype=torch_dtype(out_dtype), out=o, lse=lse)
    torch.cuda.synchronize()
    rc, where = fattn.fattn_last_error(0)
    assert rc == 0, f"kernel status {rc} ({fattn.fattn_error_string(rc)}) at {where}"
    return o.double().cpu().numpy(), lse.double().cpu().numpy()
