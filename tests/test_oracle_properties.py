"""Randomised agreement between the oracle's independent statements of the
definition (CPU): the C oracle and the numpy definition, the tile-by-tile
online recurrence (any tile shape, eager or lazy reference maximum) and the
definition, a row subset and the full evaluation, and the two statements of
attention against a cache (any cached lengths, empty rows included).  Shapes,
masks, scales, magnitudes, tiles and lengths are drawn by hypothesis; the
values from a seeded generator."""
from __future__ import annotations

import math

import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
from hypothesis import given, settings, strategies as st  # noqa: E402

import oracle  # noqa: E402

SETTINGS = settings(max_examples=150, deadline=None, derandomize=True)


def _rnd(rng, shape, mag):
    return rng.standard_normal(shape) * mag


shapes = st.tuples(st.integers(1, 2), st.integers(1, 3), st.integers(1, 70),
                   st.integers(1, 20))
scales = st.floats(1e-3, 3.0, allow_nan=False, allow_infinity=False)
mags = st.sampled_from([0.0, 1.0, 4.0, 16.0])


def _close(a, b, what):
    np.testing.assert_allclose(a, b, rtol=1e-11, atol=1e-11, err_msg=what)


@SETTINGS
@given(shape=shapes, causal=st.booleans(), scale=scales, mag=mags,
       seed=st.integers(0, 2**31 - 1))
def test_c_oracle_equals_numpy_definition(shape, causal, scale, mag, seed):
    rng = np.random.default_rng(seed)
    q, k, v = (_rnd(rng, shape, m) for m in (mag, mag, 1.0))
    o1, l1 = oracle.attn_fwd(q, k, v, causal, scale, threads=2)
    o2, l2 = oracle.attn_fwd_numpy(q, k, v, causal, scale)
    _close(o1, o2, "O")
    _close(l1, l2, "LSE")


@SETTINGS
@given(shape=shapes, causal=st.booleans(), scale=scales, mag=mags,
       bm=st.integers(4, 64), bn=st.integers(4, 64), lazy=st.booleans(),
       seed=st.integers(0, 2**31 - 1))
def test_online_recurrence_equals_definition(shape, causal, scale, mag, bm, bn,
                                             lazy, seed):
    """Any query and key tile sizes (not only equal ones), ragged last tiles,
    and the lazy reference maximum (8 log2 units)."""
    rng = np.random.default_rng(seed)
    q, k, v = (_rnd(rng, shape, m) for m in (mag, mag, 1.0))
    o1, l1 = oracle.attn_fwd_online(q, k, v, causal, scale, block_m=bm, block_n=bn,
                                    lazy_threshold=8 * math.log(2) if lazy else 0.0)
    o2, l2 = oracle.attn_fwd_numpy(q, k, v, causal, scale)
    _close(o1, o2, "O")
    _close(l1, l2, "LSE")


@SETTINGS
@given(shape=shapes, causal=st.booleans(), scale=scales,
       seed=st.integers(0, 2**31 - 1), frac=st.floats(0.05, 1.0))
def test_row_subset_equals_full(shape, causal, scale, seed, frac):
    rng = np.random.default_rng(seed)
    q, k, v = (_rnd(rng, shape, 1.0) for _ in range(3))
    B, H, S, D = shape
    n = max(1, int(frac * B * H * S))
    rows = np.sort(rng.choice(B * H * S, size=n, replace=False))
    o_full, l_full = oracle.attn_fwd(q, k, v, causal, scale, threads=2)
    o_sub, l_sub = oracle.attn_fwd(q, k, v, causal, scale, rows=rows, threads=2)
    np.testing.assert_array_equal(o_sub, o_full.reshape(-1, D)[rows])
    np.testing.assert_array_equal(l_sub, l_full.reshape(-1)[rows])


@SETTINGS
@given(B=st.integers(1, 4), H=st.integers(1, 3), Sq=st.integers(1, 16),
       Sk=st.integers(1, 60), D=st.integers(1, 16), causal=st.booleans(),
       scale=scales, mag=mags, with_lens=st.booleans(), seed=st.integers(0, 2**31 - 1))
def test_cache_oracles_agree(B, H, Sq, Sk, D, causal, scale, mag, with_lens, seed):
    """Any cached lengths in [0, Sk], including fewer than the new queries
    (empty causal rows) and zero (empty batches)."""
    rng = np.random.default_rng(seed)
    q = _rnd(rng, (B, H, Sq, D), mag)
    k = _rnd(rng, (B, H, Sk, D), mag)
    v = _rnd(rng, (B, H, Sk, D), 1.0)
    lens = rng.integers(0, Sk + 1, size=B) if with_lens else None
    o1, l1 = oracle.attn_kvcache(q, k, v, causal, scale, lens, threads=2)
    o2, l2 = oracle.attn_kvcache_numpy(q, k, v, causal, scale, lens)
    empty = np.isneginf(l2)
    np.testing.assert_array_equal(np.isneginf(l1), empty)
    assert np.all(o1[empty] == 0.0)
    _close(o1[~empty], o2[~empty], "O")
    _close(l1[~empty], l2[~empty], "LSE")
