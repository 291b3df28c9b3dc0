"""Pins for the fp64 cache oracle (``oracle.attn_kvcache``): new queries
against a key/value cache ("FlashAttention V2", section 6, inference with a
KV cache).

Reading pinned here: head (b, h) holds ``len_b`` cached positions; the ``Sq``
new queries are the last ``Sq`` positions of that sequence, so query ``i`` is
position ``len_b - Sq + i`` and the causal mask keeps keys ``j <= len_b - Sq +
i``; cache rows at or past ``len_b`` are ignored; a query with no allowed key
gets ``O = 0`` and ``LSE = -inf``.

Each ``pin_*`` takes ``impl(q, k, v, causal, scale, lens) -> (O, LSE)``.  The
pins hold for the C oracle; planted mistakes in a copy of the numpy statement
must each trip at least one of them.
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(2024)


def rnd(*shape):
    return RNG.standard_normal(shape)


def c_oracle(q, k, v, causal, scale, lens=None):
    return oracle.attn_kvcache(q, k, v, causal, scale, lens, threads=2)


def pin_kv_single_key(impl):
    """One cached key: its weight is 1, O = v_0, LSE = scale * q.k_0, for every
    query row (causal or not, the key is at position 0 <= every query)."""
    q, k, v = rnd(2, 3, 1, 8), rnd(2, 3, 5, 8), rnd(2, 3, 5, 8)
    for causal in (False, True):
        o, lse = impl(q, k, v, causal, 0.37, [1, 1])
        np.testing.assert_allclose(o, v[:, :, :1], rtol=0, atol=1e-14)
        np.testing.assert_allclose(
            lse, 0.37 * np.sum(q * k[:, :, :1], axis=-1), rtol=1e-14, atol=1e-14)


def pin_kv_constant_v(impl):
    """All cached V rows equal to c: every non-empty row of O is c."""
    q, k = rnd(2, 2, 3, 5), rnd(2, 2, 23, 5)
    c = rnd(5)
    v = np.broadcast_to(c, (2, 2, 23, 5)).copy()
    for causal in (False, True):
        o, _ = impl(q, k, v, causal, 0.5, [23, 9])
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), atol=1e-13)


def pin_kv_zero_query(impl):
    """Q = 0: O is the mean of the allowed V rows, LSE = ln(their count);
    causal query i of a length-n history has n - Sq + i + 1 of them."""
    Sq, Sk = 4, 17
    lens = [17, 6]
    q = np.zeros((2, 2, Sq, 3))
    k, v = rnd(2, 2, Sk, 3), rnd(2, 2, Sk, 3)
    for causal in (False, True):
        o, lse = impl(q, k, v, causal, 1.0, lens)
        for b, n in enumerate(lens):
            for i in range(Sq):
                cnt = n - Sq + i + 1 if causal else n
                np.testing.assert_allclose(
                    o[b, :, i], v[b, :, :cnt].mean(axis=1), atol=1e-14)
                np.testing.assert_allclose(lse[b, :, i], math.log(cnt),
                                           atol=1e-14)


def pin_kv_is_last_rows_of_self_attention(impl):
    """The queries are the last Sq positions of the sequence: with the causal
    mask, the cache result equals the last Sq rows of causal self-attention
    over the whole sequence (the pinned self-attention oracle), and without
    it, the same rows of non-causal self-attention."""
    L, Sq, D = 19, 5, 6
    qf, k, v = rnd(1, 2, L, D), rnd(1, 2, L, D), rnd(1, 2, L, D)
    cap = 24
    kc = np.concatenate([k, rnd(1, 2, cap - L, D)], axis=2)
    vc = np.concatenate([v, rnd(1, 2, cap - L, D)], axis=2)
    for causal in (False, True):
        want_o, want_l = oracle.attn_fwd(qf, k, v, causal, 0.45)
        o, lse = impl(qf[:, :, L - Sq:], kc, vc, causal, 0.45, [L])
        np.testing.assert_allclose(o, want_o[:, :, L - Sq:], atol=1e-13)
        np.testing.assert_allclose(lse, want_l[:, :, L - Sq:], atol=1e-13)


def pin_kv_stale_rows_ignored(impl):
    """Cache rows at or past len_b do not enter the result, whatever they
    hold (here huge keys that would dominate every softmax)."""
    q, k, v = rnd(2, 2, 2, 4), rnd(2, 2, 12, 4), rnd(2, 2, 12, 4)
    lens = [7, 12]
    for causal in (False, True):
        o1, l1 = impl(q, k, v, causal, 0.6, lens)
        k2, v2 = k.copy(), v.copy()
        k2[0, :, 7:] = 1e3 * q[0, :, :1]
        v2[0, :, 7:] = 1e6
        o2, l2 = impl(q, k2, v2, causal, 0.6, lens)
        np.testing.assert_array_equal(o1, o2)
        np.testing.assert_array_equal(l1, l2)


def pin_kv_empty_rows(impl):
    """No cached key (len_b = 0), or causal queries placed before the first
    key (len_b < Sq): O = 0 and LSE = -inf on exactly those rows."""
    Sq = 3
    q, k, v = rnd(3, 2, Sq, 4), rnd(3, 2, 8, 4), rnd(3, 2, 8, 4)
    lens = [0, 1, 8]
    o, lse = impl(q, k, v, False, 0.5, lens)
    assert np.all(o[0] == 0.0) and np.all(lse[0] == -np.inf)
    assert np.isfinite(lse[1:]).all()
    o, lse = impl(q, k, v, True, 0.5, lens)
    assert np.all(o[0] == 0.0) and np.all(lse[0] == -np.inf)
    # len 1, Sq 3: queries at positions -2, -1, 0; only the last sees key 0
    assert np.all(o[1, :, :2] == 0.0) and np.all(lse[1, :, :2] == -np.inf)
    np.testing.assert_allclose(o[1, :, 2], v[1, :, 0], atol=1e-14)
    assert np.isfinite(lse[2]).all()


def pin_kv_permutation(impl):
    """Without the mask the result is a sum over the cached keys: permuting
    the first len_b K and V rows together changes nothing."""
    q, k, v = rnd(1, 3, 2, 7), rnd(1, 3, 20, 7), rnd(1, 3, 20, 7)
    n = 15
    perm = np.concatenate([RNG.permutation(n), np.arange(n, 20)])
    o1, l1 = impl(q, k, v, False, 0.4, [n])
    o2, l2 = impl(q, k[:, :, perm], v[:, :, perm], False, 0.4, [n])
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def pin_kv_lengths_per_batch(impl):
    """Each batch entry uses its own length, the same for all its heads: batch
    b equals a run on that batch alone with the cache cut to len_b."""
    q, k, v = rnd(3, 2, 2, 4), rnd(3, 2, 10, 4), rnd(3, 2, 10, 4)
    lens = [10, 4, 7]
    for causal in (False, True):
        o, lse = impl(q, k, v, causal, 0.7, lens)
        for b, n in enumerate(lens):
            ob, lb = impl(q[b:b + 1], k[b:b + 1, :, :n], v[b:b + 1, :, :n],
                          causal, 0.7, None)
            np.testing.assert_allclose(o[b], ob[0], atol=1e-14)
            np.testing.assert_allclose(lse[b], lb[0], atol=1e-14)


def brute_force_kv_mp(q, k, v, causal, scale, lens, dps=40):
    """Per-element direct sums at ``dps`` decimal digits (mpmath)."""
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = dps
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    o = np.zeros((B, H, Sq, D))
    lse = np.full((B, H, Sq), -np.inf)
    for b in range(B):
        n = Sk if lens is None else lens[b]
        for h in range(H):
            for i in range(Sq):
                keys = [j for j in range(n) if not causal or j <= n - Sq + i]
                if not keys:
                    continue
                ws = []
                for j in keys:
                    s = mp.fsum(mp.mpf(q[b, h, i, d]) * mp.mpf(k[b, h, j, d])
                                for d in range(D))
                    ws.append(mp.exp(mp.mpf(scale) * s))
                tot = mp.fsum(ws)
                for d in range(D):
                    o[b, h, i, d] = float(mp.fsum(
                        w * mp.mpf(v[b, h, j, d]) for w, j in zip(ws, keys)) / tot)
                lse[b, h, i] = float(mp.log(tot))
    return o, lse


def pin_kv_brute_force(impl):
    """Tiny random inputs against a 40-digit evaluation of the definition."""
    for (Sq, Sk, D, lens) in ((1, 1, 1, None), (2, 5, 3, [5, 2]),
                              (3, 6, 4, [6, 1]), (4, 9, 2, None)):
        B = 1 if lens is None else len(lens)
        q, k, v = rnd(B, 2, Sq, D), rnd(B, 2, Sk, D), rnd(B, 2, Sk, D)
        for causal in (False, True):
            want_o, want_l = brute_force_kv_mp(q, k, v, causal, 0.7, lens)
            o, lse = impl(q, k, v, causal, 0.7, lens)
            np.testing.assert_allclose(o, want_o, rtol=0, atol=1e-12)
            np.testing.assert_array_equal(np.isinf(lse), np.isinf(want_l))
            fin = np.isfinite(want_l)
            np.testing.assert_allclose(lse[fin], want_l[fin], rtol=0, atol=1e-12)


KV_PINS = [pin_kv_single_key, pin_kv_constant_v, pin_kv_zero_query,
           pin_kv_is_last_rows_of_self_attention, pin_kv_stale_rows_ignored,
           pin_kv_empty_rows, pin_kv_permutation, pin_kv_lengths_per_batch,
           pin_kv_brute_force]


@pytest.mark.parametrize("pin", KV_PINS, ids=lambda p: p.__name__)
def test_c_cache_oracle_pinned(pin):
    pin(c_oracle)


@pytest.mark.parametrize("pin", KV_PINS, ids=lambda p: p.__name__)
def test_numpy_cache_definition_pinned(pin):
    pin(oracle.attn_kvcache_numpy)


# ------------------------------------------- planted mistakes must be caught

def _kv_mutant(kind):
    """The numpy cache definition with one plausible mistake planted."""

    def impl(q, k, v, causal, scale, lens=None):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        B, H, Sq, D = q.shape
        Sk = k.shape[2]
        o = np.zeros((B, H, Sq, D))
        lse = np.full((B, H, Sq), -np.inf)
        for b in range(B):
            for h in range(H):
                if lens is None or kind == "ignore_lens":
                    n = Sk
                elif kind == "lens_by_head":
                    n = lens[(b * H + h) % len(lens)]
                else:
                    n = lens[b]
                for i in range(Sq):
                    js = np.arange(n)
                    if causal:
                        if kind == "causal_top_left":
                            js = js[js <= i]
                        elif kind == "causal_strict":
                            js = js[js < n - Sq + i]
                        else:
                            js = js[js <= n - Sq + i]
                    if js.size == 0:
                        if kind == "empty_rows_nan":
                            o[b, h, i] = np.nan
                        continue
                    s = scale * (k[b, h, js] @ q[b, h, i])
                    if kind == "no_scale":
                        s = s / scale
                    m = s.max()
                    e = np.exp(s - m)
                    l = e.sum()
                    vv = v[b, h, js]
                    if kind == "v_from_next_row":
                        vv = v[b, h, np.minimum(js + 1, Sk - 1)]
                    o[b, h, i] = (e @ vv) / l
                    lse[b, h, i] = m + np.log(l) if kind != "lse_no_max" else np.log(l)
        return o, lse

    return impl


KV_MUTANTS = ["ignore_lens", "lens_by_head", "causal_top_left", "causal_strict",
              "empty_rows_nan", "no_scale", "v_from_next_row", "lse_no_max"]


def test_clean_cache_mutant_passes_pins():
    for pin in KV_PINS:
        pin(_kv_mutant("none"))


@pytest.mark.parametrize("kind", KV_MUTANTS)
def test_planted_cache_mistake_is_caught(kind):
    impl = _kv_mutant(kind)
    failed = []
    for pin in KV_PINS:
        try:
            pin(impl)
        except (AssertionError, IndexError):
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {kind!r}"


# ------------------------------------------------ cross-checks and plumbing

def test_c_cache_oracle_matches_numpy():
    q, k, v = rnd(3, 2, 5, 16), rnd(3, 2, 70, 16), rnd(3, 2, 70, 16)
    for lens in (None, [70, 0, 33], [1, 4, 69]):
        for causal in (False, True):
            o1, l1 = oracle.attn_kvcache(q, k, v, causal, 0.25, lens, threads=3)
            o2, l2 = oracle.attn_kvcache_numpy(q, k, v, causal, 0.25, lens)
            np.testing.assert_allclose(o1, o2, atol=1e-13)
            np.testing.assert_array_equal(np.isinf(l1), np.isinf(l2))
            fin = np.isfinite(l2)
            np.testing.assert_allclose(l1[fin], l2[fin], atol=1e-13)


def test_cache_oracle_rejects_bad_arguments():
    q, k = rnd(2, 1, 1, 2), rnd(2, 1, 4, 2)
    with pytest.raises(RuntimeError):
        oracle.attn_kvcache(q, k, k, False, 1.0, [5, 1])
    with pytest.raises(RuntimeError):
        oracle.attn_kvcache(q, k, k, False, 1.0, [-1, 1])
    with pytest.raises(RuntimeError):
        oracle.attn_kvcache(q, k, k, False, 0.0)
    with pytest.raises(ValueError):
        oracle.attn_kvcache(q, k, k, False, 1.0, [1])
