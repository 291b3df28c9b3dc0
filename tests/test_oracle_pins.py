"""Pins for the fp64 oracle: what the mathematics fixes, independent of it.

Each ``pin_*`` takes an implementation ``impl(q, k, v, causal, scale) ->
(O, LSE)`` and raises ``AssertionError`` if it disagrees with a closed form,
an invariant, a limit or a high-precision brute-force evaluation.  They run
on the C oracle (all must hold) and on planted mistakes in a copy of the
definition (each mistake must trip at least one pin), so a dropped term, a
wrong sign or index, or a transposed operand in the oracle cannot go unseen.

The definition being pinned: scores ``s = scale * q . k`` over the allowed
keys (all keys; causal: key <= query), softmax over keys, ``O = P V``,
``LSE = max + ln(sum exp(s - max))`` ("FlashAttention-2 in an attention
layer", Triton FA2 kernel; "FlashAttention V2", section 3).
"""
import math

import numpy as np
import pytest

import oracle

RNG = np.random.default_rng(12345)


def rnd(*shape):
    return RNG.standard_normal(shape)


def c_oracle(q, k, v, causal, scale):
    return oracle.attn_fwd(q, k, v, causal, scale, threads=2)


# ---------------------------------------------------------------- the pins

def pin_single_key(impl):
    """S = 1: the only weight is 1, so O = V and LSE = scale * q.k."""
    q, k, v = rnd(2, 3, 1, 8), rnd(2, 3, 1, 8), rnd(2, 3, 1, 8)
    for causal in (False, True):
        o, lse = impl(q, k, v, causal, 0.37)
        np.testing.assert_allclose(o, v, rtol=0, atol=1e-14)
        np.testing.assert_allclose(lse, 0.37 * np.sum(q * k, axis=-1),
                                   rtol=1e-14, atol=1e-14)


def pin_constant_v(impl):
    """Every V row equal to c: any convex combination of them is c."""
    q, k = rnd(1, 2, 19, 5), rnd(1, 2, 19, 5)
    c = rnd(5)
    v = np.broadcast_to(c, (1, 2, 19, 5)).copy()
    for causal in (False, True):
        o, _ = impl(q, k, v, causal, 0.5)
        np.testing.assert_allclose(o, np.broadcast_to(c, o.shape), rtol=0,
                                   atol=1e-13)


def pin_causal_row0(impl):
    """Causal row 0 sees key 0 only: O_0 = V_0, LSE_0 = scale * q_0.k_0."""
    q, k, v = rnd(2, 2, 11, 6), rnd(2, 2, 11, 6), rnd(2, 2, 11, 6)
    o, lse = impl(q, k, v, True, 0.8)
    np.testing.assert_allclose(o[:, :, 0], v[:, :, 0], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[:, :, 0],
                               0.8 * np.sum(q[:, :, 0] * k[:, :, 0], -1),
                               rtol=1e-14, atol=1e-14)


def pin_zero_query(impl):
    """Q = 0: all allowed scores are 0, so O_i is the mean of the allowed V
    rows and LSE_i = ln(number of allowed keys)."""
    S = 13
    q = np.zeros((1, 2, S, 4))
    k, v = rnd(1, 2, S, 4), rnd(1, 2, S, 4)
    o, lse = impl(q, k, v, False, 1.0)
    np.testing.assert_allclose(o, np.broadcast_to(v.mean(axis=2, keepdims=True),
                                                  o.shape), atol=1e-14)
    np.testing.assert_allclose(lse, np.full((1, 2, S), math.log(S)), atol=1e-14)
    o, lse = impl(q, k, v, True, 1.0)
    count = np.arange(1, S + 1)
    prefix_mean = np.cumsum(v, axis=2) / count[None, None, :, None]
    np.testing.assert_allclose(o, prefix_mean, atol=1e-14)
    np.testing.assert_allclose(lse, np.broadcast_to(np.log(count), lse.shape),
                               atol=1e-14)


def pin_two_keys(impl):
    """S = 2, D = 1: the softmax of two scores is the logistic function.
    Non-causal row i: O_i = sig(s_i0 - s_i1) v_0 + sig(s_i1 - s_i0) v_1,
    LSE_i = ln(e^{s_i0} + e^{s_i1}).  Causal: row 0 is v_0, row 1 as above."""
    q = np.array([0.9, -1.7]).reshape(1, 1, 2, 1)
    k = np.array([1.3, 0.4]).reshape(1, 1, 2, 1)
    v = np.array([2.0, -3.0]).reshape(1, 1, 2, 1)
    scale = 0.75

    def sig(x):
        return 1.0 / (1.0 + math.exp(-x))

    want_o, want_l = [], []
    for i in range(2):
        s0 = scale * q[0, 0, i, 0] * k[0, 0, 0, 0]
        s1 = scale * q[0, 0, i, 0] * k[0, 0, 1, 0]
        want_o.append(sig(s0 - s1) * 2.0 + sig(s1 - s0) * -3.0)
        want_l.append(np.logaddexp(s0, s1))
    o, lse = impl(q, k, v, False, scale)
    np.testing.assert_allclose(o[0, 0, :, 0], want_o, rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], want_l, rtol=1e-14, atol=1e-14)
    o, lse = impl(q, k, v, True, scale)
    np.testing.assert_allclose(o[0, 0, :, 0],
                               [2.0, want_o[1]], rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(
        lse[0, 0], [scale * q[0, 0, 0, 0] * k[0, 0, 0, 0], want_l[1]],
        rtol=1e-14, atol=1e-14)


def pin_permutation(impl):
    """Non-causal attention is a sum over keys: permuting the K and V rows
    together changes nothing."""
    q, k, v = rnd(1, 3, 17, 7), rnd(1, 3, 17, 7), rnd(1, 3, 17, 7)
    perm = RNG.permutation(17)
    o1, l1 = impl(q, k, v, False, 0.4)
    o2, l2 = impl(q, k[:, :, perm], v[:, :, perm], False, 0.4)
    np.testing.assert_allclose(o1, o2, atol=1e-13)
    np.testing.assert_allclose(l1, l2, atol=1e-13)


def pin_shift(impl):
    """Adding one vector u to every key adds scale * q_i.u to every score of
    row i: softmax is shift invariant, so O is unchanged and LSE moves by
    exactly that constant."""
    q, k, v = rnd(1, 2, 9, 4), rnd(1, 2, 9, 4), rnd(1, 2, 9, 4)
    u = rnd(4)
    for causal in (False, True):
        o1, l1 = impl(q, k, v, causal, 0.6)
        o2, l2 = impl(q, k + u, v, causal, 0.6)
        np.testing.assert_allclose(o1, o2, atol=1e-13)
        np.testing.assert_allclose(l2 - l1, 0.6 * (q @ u), atol=1e-13)


def pin_one_hot(impl):
    """Q = lambda * K with orthonormal key rows: row i scores lambda on key i
    and 0 elsewhere; for lambda = 60 the other weights are e^-60 (~1e-26), so
    in fp64 O_i = V_i and LSE_i = 60 (causal: the same, keys 0..i)."""
    S = 6
    k = np.eye(S).reshape(1, 1, S, S)
    q = 60.0 * k
    v = rnd(1, 1, S, S)
    o, lse = impl(q, k, v, False, 1.0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lse[0, 0], np.full(S, 60.0), rtol=0, atol=1e-13)
    o, _ = impl(q, k, v, True, 1.0)
    np.testing.assert_allclose(o, v, rtol=0, atol=1e-15)


def pin_causal_last_row(impl):
    """The last query row is allowed every key, so causal and non-causal agree
    on it; on row i < S-1 causal equals non-causal run on keys 0..i only."""
    q, k, v = rnd(1, 2, 10, 3), rnd(1, 2, 10, 3), rnd(1, 2, 10, 3)
    oc, lc = impl(q, k, v, True, 0.9)
    on, ln_ = impl(q, k, v, False, 0.9)
    np.testing.assert_allclose(oc[:, :, -1], on[:, :, -1], atol=1e-14)
    np.testing.assert_allclose(lc[:, :, -1], ln_[:, :, -1], atol=1e-14)
    i = 4
    op, lp = impl(q[:, :, :i + 1], k[:, :, :i + 1], v[:, :, :i + 1], False, 0.9)
    np.testing.assert_allclose(oc[:, :, i], op[:, :, i], atol=1e-14)
    np.testing.assert_allclose(lc[:, :, i], lp[:, :, i], atol=1e-14)


def pin_scale_power_of_two(impl):
    """scale * (q.k) == (scale q).k exactly when scale is a power of two."""
    q, k, v = rnd(1, 2, 12, 8), rnd(1, 2, 12, 8), rnd(1, 2, 12, 8)
    for causal in (False, True):
        o1, l1 = impl(q, k, v, causal, 0.25)
        o2, l2 = impl(0.25 * q, k, v, causal, 1.0)
        np.testing.assert_allclose(o1, o2, atol=1e-15)
        np.testing.assert_allclose(l1, l2, atol=1e-15)


def brute_force_mp(q, k, v, causal, scale, dps=40):
    """Per-element direct sums at ``dps`` decimal digits (mpmath)."""
    mpmath = pytest.importorskip("mpmath")
    mp = mpmath.mp
    mp.dps = dps
    B, H, S, D = q.shape
    o = np.zeros((B, H, S, D))
    lse = np.zeros((B, H, S))
    for b in range(B):
        for h in range(H):
            for i in range(S):
                keys = range(i + 1) if causal else range(S)
                ws = []
                for j in keys:
                    s = mp.mpf(0)
                    for d in range(D):
                        s += mp.mpf(q[b, h, i, d]) * mp.mpf(k[b, h, j, d])
                    ws.append(mp.exp(mp.mpf(scale) * s))
                tot = mp.fsum(ws)
                for d in range(D):
                    o[b, h, i, d] = float(mp.fsum(
                        w * mp.mpf(v[b, h, j, d]) for w, j in zip(ws, keys)) / tot)
                lse[b, h, i] = float(mp.log(tot))
    return o, lse


def pin_brute_force(impl):
    """Tiny random inputs against a 40-digit evaluation of the definition."""
    for (S, D) in ((1, 1), (3, 2), (5, 8), (8, 5)):
        q, k, v = rnd(1, 2, S, D), rnd(1, 2, S, D), rnd(1, 2, S, D)
        for causal in (False, True):
            want_o, want_l = brute_force_mp(q, k, v, causal, 0.7)
            o, lse = impl(q, k, v, causal, 0.7)
            np.testing.assert_allclose(o, want_o, rtol=0, atol=1e-12)
            np.testing.assert_allclose(lse, want_l, rtol=0, atol=1e-12)


PINS = [pin_single_key, pin_constant_v, pin_causal_row0, pin_zero_query,
        pin_two_keys, pin_permutation, pin_shift, pin_one_hot,
        pin_causal_last_row, pin_scale_power_of_two, pin_brute_force]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_c_oracle_pinned(pin):
    pin(c_oracle)


# ------------------------------------------- planted mistakes must be caught

def _mutant(kind):
    """The numpy definition with one plausible mistake planted."""

    def impl(q, k, v, causal, scale):
        q, k, v = (np.asarray(x, dtype=np.float64) for x in (q, k, v))
        S = q.shape[-2]
        if kind == "no_scale":
            scale = 1.0
        if kind == "transposed_scores":
            s = scale * np.einsum("bhjd,bhid->bhij", q, k)
        else:
            s = scale * np.einsum("bhid,bhjd->bhij", q, k)
        if causal:
            if kind == "mask_flipped":
                allowed = np.triu(np.ones((S, S), dtype=bool))
            elif kind == "mask_strict":
                allowed = np.tril(np.ones((S, S), dtype=bool), -1)
                allowed[0, 0] = True
            else:
                allowed = np.tril(np.ones((S, S), dtype=bool))
            s = np.where(allowed, s, -np.inf)
        m = s.max(axis=-1, keepdims=True)
        e = np.exp(s - m) if kind != "sign" else np.exp(m - s)
        if kind == "sign":
            e = np.where(np.isfinite(s), e, 0.0)
        l = e.sum(axis=-1, keepdims=True)
        p = e if kind == "no_normalise" else e / l
        if kind == "v_off_by_one":
            v = np.roll(v, 1, axis=2)
        o = np.einsum("bhij,bhjd->bhid", p, v)
        if kind == "lse_drops_max":
            lse = np.log(l)[..., 0]
        elif kind == "lse_log2":
            lse = (m + np.log2(l))[..., 0]
        else:
            lse = (m + np.log(l))[..., 0]
        return o, lse

    return impl


MUTANTS = ["no_scale", "transposed_scores", "mask_flipped", "mask_strict",
           "sign", "no_normalise", "v_off_by_one", "lse_drops_max", "lse_log2"]


def test_clean_numpy_definition_passes_pins():
    for pin in PINS:
        pin(_mutant("none"))


@pytest.mark.parametrize("kind", MUTANTS)
def test_planted_mistake_is_caught(kind):
    impl = _mutant(kind)
    failed = []
    for pin in PINS:
        try:
            pin(impl)
        except AssertionError:
            failed.append(pin.__name__)
    assert failed, f"no pin caught the planted mistake {kind!r}"


# ------------------------------------------------ cross-checks and plumbing

def test_c_matches_numpy_definition():
    q, k, v = rnd(2, 3, 67, 24), rnd(2, 3, 67, 24), rnd(2, 3, 67, 24)
    for causal in (False, True):
        o1, l1 = oracle.attn_fwd(q, k, v, causal, 0.2, threads=3)
        o2, l2 = oracle.attn_fwd_numpy(q, k, v, causal, 0.2)
        np.testing.assert_allclose(o1, o2, atol=1e-13)
        np.testing.assert_allclose(l1, l2, atol=1e-13)


def test_probabilities_rows_sum_to_one():
    q, k, v = rnd(1, 2, 33, 8), rnd(1, 2, 33, 8), rnd(1, 2, 33, 8)
    for causal in (False, True):
        _, _, p = oracle.attn_fwd(q, k, v, causal, 0.5, want_p=True)
        np.testing.assert_allclose(p.sum(axis=-1), 1.0, atol=1e-12)
        assert (p >= 0).all()
        if causal:
            assert np.all(np.triu(p[0, 0], 1) == 0.0)
        # O is P V
        o, _ = oracle.attn_fwd(q, k, v, causal, 0.5)
        np.testing.assert_allclose(o, p @ v, atol=1e-13)


@pytest.mark.parametrize("bm,bn", [(128, 128), (16, 8), (8, 16), (7, 5)])
def test_online_recurrence_equals_definition(bm, bn):
    """The tile-by-tile recurrence (running max, rescale by exp(m_old - m_new),
    one final division) reaches the plain definition, ragged tiles included."""
    q, k, v = rnd(1, 2, 300, 16), rnd(1, 2, 300, 16), rnd(1, 2, 300, 16)
    for causal in (False, True):
        o1, l1 = oracle.attn_fwd_online(q, k, v, causal, 0.3, bm, bn)
        o2, l2 = oracle.attn_fwd(q, k, v, causal, 0.3)
        np.testing.assert_allclose(o1, o2, atol=1e-13)
        np.testing.assert_allclose(l1, l2, atol=1e-13)


@pytest.mark.parametrize("thr", [0.5, 8.0 * math.log(2.0)])
def test_lazy_reference_max_equals_definition(thr):
    """Keeping a stale reference maximum (moved only when a tile's maximum
    exceeds it by more than a threshold) changes nothing: O, l and the
    exponent share the reference.  Large scores make the maximum move."""
    q, k, v = 4 * rnd(1, 2, 300, 16), 4 * rnd(1, 2, 300, 16), rnd(1, 2, 300, 16)
    for causal in (False, True):
        o1, l1 = oracle.attn_fwd_online(q, k, v, causal, 0.3, 32, 32, thr)
        o2, l2 = oracle.attn_fwd(q, k, v, causal, 0.3)
        np.testing.assert_allclose(o1, o2, atol=1e-12)
        np.testing.assert_allclose(l1, l2, atol=1e-12)


def test_row_subset_equals_full():
    q, k, v = rnd(2, 2, 50, 8), rnd(2, 2, 50, 8), rnd(2, 2, 50, 8)
    rows = np.array([0, 49, 50, 77, 199, 3])
    for causal in (False, True):
        of, lf = oracle.attn_fwd(q, k, v, causal, 0.4)
        os_, ls = oracle.attn_fwd(q, k, v, causal, 0.4, rows=rows)
        np.testing.assert_array_equal(os_, of.reshape(-1, 8)[rows])
        np.testing.assert_array_equal(ls, lf.reshape(-1)[rows])


def test_thread_count_does_not_change_results():
    q, k, v = rnd(1, 3, 40, 8), rnd(1, 3, 40, 8), rnd(1, 3, 40, 8)
    o1, l1 = oracle.attn_fwd(q, k, v, True, 0.4, threads=1)
    o2, l2 = oracle.attn_fwd(q, k, v, True, 0.4, threads=7)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


def test_oracle_rejects_bad_arguments():
    q = rnd(1, 1, 4, 2)
    with pytest.raises(RuntimeError):
        oracle.attn_fwd(q, q, q, False, 0.0)
    with pytest.raises(RuntimeError):
        oracle.attn_fwd(q, q, q, False, float("nan"))
    with pytest.raises(RuntimeError):
        oracle.attn_fwd(q, q, q, False, 1.0, rows=[4])
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q[:, :, :3], q, False, 1.0)
