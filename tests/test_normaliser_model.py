"""Why the 16-bit kernels divide O by the fp32 sum with each tile's largest
weight replaced by its 16-bit value (CPU, an fp64 model of the kernel's
roundings).

Weights are taken against a reference maximum that may lag the row's true
maximum: by up to 8 log2 units when each tile takes its maximum first (the
lazy reference), and, when the maximum is taken during the exponent pass
(bf16 at head dim 128, non-causal), by as much as a tile's maximum passed
the reference chosen after the tile before, up to the 2^64 (bf16) or 2^15
(fp16) past which the kernel redoes the tile.  So a peaked row's dominant
weight can be as large as 2^8, 2^15 or 2^64.  P is rounded to the input dtype for
the P V product ("FlashAttention-2 in an attention layer": the Triton loop
casts p to V's dtype), and O is rounded to the dtype.  If O were divided by
the plain fp32 sum of the unrounded weights, the dominant weight's rounding
would show up as (1 + d) v in a nearly one-hot row.  That breaks the fp16
and bf16 tolerances on peaked inputs (Q and K x 4, x 8).  Replacing the
largest weight in the sum by its rounded value keeps every element within
them."""
from __future__ import annotations

import math

import numpy as np
import pytest

import attn_inputs
import oracle
from parity import compare

LN2 = math.log(2.0)


def _round16(x, dtype):
    if dtype == "fp16":
        return x.astype(np.float16).astype(np.float64)
    return attn_inputs.round_fp32_to_bf16(x.astype(np.float32)).astype(np.float64)


def _model(q, k, v, scale, lag, dtype, kernel_normaliser):
    """One key tile per row (S <= 128), non-causal."""
    s = scale * np.einsum("bhid,bhjd->bhij", q, k)
    p = np.exp(s - (s.max(axis=-1, keepdims=True) - lag[..., None]))
    p16 = _round16(p, dtype)
    den = p.sum(axis=-1)
    if kernel_normaliser:
        pmax = p.max(axis=-1)
        den = den - pmax + _round16(pmax, dtype)
    o = np.einsum("bhij,bhjd->bhid", p16, v) / den[..., None]
    return attn_inputs.round_to_dtype(o, dtype).astype(np.float64)


def _cases(dtype, lag_log2=8.0):
    for mult in (4.0, 8.0):
        for seed in range(6):
            x = attn_inputs.make_qkv(1, 4, 128, 64, dtype, seed=7000 + seed, qk_mult=mult)
            lag = np.random.default_rng(seed).uniform(0.0, lag_log2 * LN2, size=(1, 4, 128))
            yield x, lag


@pytest.mark.parametrize("dtype,lag_log2", [("fp16", 8.0), ("fp16", 15.0),
                                            ("bf16", 8.0), ("bf16", 64.0)])
def test_kernel_normaliser_keeps_the_tolerance(dtype, lag_log2):
    for x, lag in _cases(dtype, lag_log2):
        ro, rl = oracle.attn_fwd_numpy(x.q, x.k, x.v, False, 0.125)
        o = _model(x.q, x.k, x.v, 0.125, lag, dtype, kernel_normaliser=True)
        compare(o, rl, ro, rl, dtype, f"kernel normaliser seed {x.seed}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_plain_fp32_sum_breaks_the_tolerance(dtype):
    broke = False
    for x, lag in _cases(dtype):
        ro, rl = oracle.attn_fwd_numpy(x.q, x.k, x.v, False, 0.125)
        o = _model(x.q, x.k, x.v, 0.125, lag, dtype, kernel_normaliser=False)
        try:
            compare(o, rl, ro, rl, dtype, "plain sum")
        except AssertionError:
            broke = True
    assert broke, "the plain fp32 sum stayed within the tolerance on every case"


def test_without_lag_both_normalisers_agree():
    """With the reference at the row maximum the dominant weight is exactly
    1 (exact in 16 bits), so the two normalisers are the same number."""
    x = attn_inputs.make_qkv(1, 4, 128, 64, "fp16", seed=7100, qk_mult=4.0)
    lag = np.zeros((1, 4, 128))
    a = _model(x.q, x.k, x.v, 0.125, lag, "fp16", True)
    b = _model(x.q, x.k, x.v, 0.125, lag, "fp16", False)
    np.testing.assert_array_equal(a, b)


def _online_reference_one_tile_late(q, k, v, causal, scale, bn, thr, cap):
    """fp64 tile recurrence with the kernel's fused-maximum reference schedule
    (natural-log units): the first key tile of a row takes its own maximum;
    tile j > 0 uses the reference chosen after tile j-1, which moved to that
    tile's maximum when it passed the reference by more than ``thr``; a tile
    whose maximum passes its reference by more than ``cap`` is redone
    against that maximum.  O and l are rescaled whenever the reference of a
    tile differs from the one before, so they always share the exponent's
    frame."""
    B, H, S, D = q.shape
    o = np.zeros((B, H, S, D))
    lse = np.zeros((B, H, S))
    rows = np.arange(S)
    for b in range(B):
        for h in range(H):
            qi, kk, vv = q[b, h], k[b, h], v[b, h]
            m = np.full(S, -np.inf)
            m_next = np.zeros(S)
            l = np.zeros(S)
            acc = np.zeros((S, D))
            for j0 in range(0, S, bn):
                cols = np.arange(j0, min(S, j0 + bn))
                s = scale * (qi @ kk[cols].T)
                if causal:
                    s = np.where(rows[:, None] >= cols[None, :], s, -np.inf)
                live = np.isfinite(s).any(axis=1)  # rows with an allowed key
                tmax = s.max(axis=1)
                m_use = np.where(j0 == 0, tmax, m_next)
                m_use = np.where(tmax > m_use + cap, tmax, m_use)  # redo
                m_use = np.where(live, m_use, m)
                alpha = np.where(np.isfinite(m), np.exp(m - m_use), 0.0)
                p = np.exp(s - m_use[:, None])
                l = np.where(live, alpha * l + p.sum(axis=1), l)
                acc = np.where(live[:, None], alpha[:, None] * acc + p @ vv[cols], acc)
                m = np.where(live, m_use, m)
                m_next = np.where(live & (tmax > m_use + thr), tmax, m)
            o[b, h] = acc / l[:, None]
            lse[b, h] = m + np.log(l)
    return o, lse


@pytest.mark.parametrize("cap_log2", [2.0, 15.0, 64.0])
def test_reference_one_tile_late_equals_definition(cap_log2):
    """A tile's P in the frame chosen after the tile before (so its weights
    may pass 2^8), the frame moving one tile late, and a redo past a cap
    (small here, so that redos happen): O and LSE are those of the
    definition.  Scores spread widely so that the reference moves often."""
    rng = np.random.default_rng(7200)
    q = 4 * rng.standard_normal((1, 2, 300, 16))
    k = 4 * rng.standard_normal((1, 2, 300, 16))
    v = rng.standard_normal((1, 2, 300, 16))
    for causal in (False, True):
        o1, l1 = _online_reference_one_tile_late(q, k, v, causal, 0.3, 32, 8 * LN2,
                                                 cap_log2 * LN2)
        o2, l2 = oracle.attn_fwd(q, k, v, causal, 0.3)
        np.testing.assert_allclose(o1, o2, atol=1e-12)
        np.testing.assert_allclose(l1, l2, atol=1e-12)
