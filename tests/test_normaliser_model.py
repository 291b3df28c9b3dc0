"""Why the 16-bit kernels divide O by the fp32 sum with each tile's largest
weight replaced by its 16-bit value (CPU, an fp64 model of the kernel's
roundings).

Weights are taken against a reference maximum that may lag the row's true
maximum by up to 8 log2 units (the lazy reference), so a peaked row's
dominant weight can be as large as 2^8.  P is rounded to the input dtype for
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

LAG_MAX = 8.0 * math.log(2.0)


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


def _cases(dtype):
    for mult in (4.0, 8.0):
        for seed in range(6):
            x = attn_inputs.make_qkv(1, 4, 128, 64, dtype, seed=7000 + seed, qk_mult=mult)
            lag = np.random.default_rng(seed).uniform(0.0, LAG_MAX, size=(1, 4, 128))
            yield x, lag


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_kernel_normaliser_keeps_the_tolerance(dtype):
    for x, lag in _cases(dtype):
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
