"""The seeded input generator: published SplitMix64 outputs, Box-Muller
statistics, exact rounding to the 16-bit dtypes and the workload seeds."""
import math

import numpy as np
import pytest
import torch

import attn_inputs as ai


def test_splitmix64_published_vectors():
    # Reference outputs of SplitMix64 started from state 1234567 (the test
    # vector of the published C implementation by S. Vigna).
    want = [6457827717110365317, 3203168211198807973, 9817491932198370423,
            4593380528125082431, 16408922859458223821]
    assert [int(x) for x in ai.splitmix64(1234567, 0, 5)] == want


def test_stream_is_counter_based():
    a = ai.splitmix64(99, 0, 1000)
    b = ai.splitmix64(99, 600, 400)
    np.testing.assert_array_equal(a[600:], b)
    z = ai.normals(7, 0, 1001)
    np.testing.assert_array_equal(z[333:1001], ai.normals(7, 333, 668))


def test_normal_statistics():
    z = ai.normals(5, 0, 1 << 20)
    assert abs(z.mean()) < 5e-3
    assert abs(z.std() - 1.0) < 5e-3
    # fourth moment of N(0,1) is 3
    assert abs((z ** 4).mean() - 3.0) < 0.05


@pytest.mark.parametrize("dtype,tdt", [("fp16", torch.float16),
                                       ("bf16", torch.bfloat16)])
def test_rounding_matches_torch_rne(dtype, tdt):
    x = ai.normals(11, 0, 100000) * 3.0
    ours = ai.round_to_dtype(x, dtype)
    ref = torch.from_numpy(x.astype(np.float32)).to(tdt).to(torch.float32)
    np.testing.assert_array_equal(ours, ref.numpy())


def test_make_qkv_shapes_and_exactness():
    w = ai.make_qkv(1, 2, 33, 8, "bf16", 4)
    assert w.q.shape == (1, 2, 33, 8) and w.q.dtype == np.float32
    for t in (w.q, w.k, w.v):
        back = torch.from_numpy(t).to(torch.bfloat16).to(torch.float32).numpy()
        np.testing.assert_array_equal(back, t)
    n = 2 * 33 * 8
    np.testing.assert_array_equal(
        w.k.reshape(-1), ai.round_to_dtype(ai.normals(4, n, n), "bf16"))
    x4 = ai.make_qkv(1, 2, 33, 8, "bf16", 4, qk_mult=4.0)
    np.testing.assert_array_equal(x4.q, 4 * w.q)
    np.testing.assert_array_equal(x4.v, w.v)
    with pytest.raises(ValueError):
        ai.make_qkv(1, 1, 4, 4, "bf16", 0, qk_mult=3.0)


def test_sweep_seeds():
    ws = ai.sweep_workloads()
    assert len(ws) == 28
    assert [w.seed for w in ws] == list(range(4, 32))
    assert (ws[0].S, ws[0].D, ws[0].dtype) == (512, 64, "fp16")
    assert (ws[3].S, ws[3].D, ws[3].dtype) == (512, 128, "bf16")
    assert (ws[-1].S, ws[-1].D, ws[-1].dtype) == (4097, 128, "bf16")
    assert all(w.B == 2 and w.H == 16 for w in ws)


def test_cache_inputs_follow_the_stream():
    """Q, then the K cache, then the V cache are consecutive normals of the
    stream; lengths are reproducible and inside their range."""
    x = ai.make_kvcache(2, 3, 4, 40, 8, "fp16", 77, (5, 40))
    nq, nk = 2 * 3 * 4 * 8, 2 * 3 * 40 * 8
    z = ai.round_to_dtype(ai.normals(77, 0, nq + 2 * nk), "fp16")
    np.testing.assert_array_equal(x.q.reshape(-1), z[:nq])
    np.testing.assert_array_equal(x.k.reshape(-1), z[nq:nq + nk])
    np.testing.assert_array_equal(x.v.reshape(-1), z[nq + nk:])
    assert x.lens.dtype == np.int64 and x.lens.shape == (2,)
    assert ((x.lens >= 5) & (x.lens <= 40)).all()
    np.testing.assert_array_equal(x.lens, ai.cache_lengths(77, 2, 5, 40))
    many = ai.cache_lengths(1, 4000, 3, 9)
    assert set(np.unique(many).tolist()) == set(range(3, 10))
    assert ai.make_kvcache(1, 1, 1, 4, 8, "bf16", 1).lens is None
    with pytest.raises(ValueError):
        ai.make_kvcache(1, 1, 1, 4, 8, "bf16", 1, (1, 5))


def test_e4m3_codes_round_trip_and_ties():
    """Every finite E4M3 code decodes and re-encodes to itself; midpoints
    between neighbours round to the even mantissa; large values saturate."""
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], dtype=np.uint8)
    vals = ai.e4m3_decode(codes)
    back = ai.e4m3_encode(vals)
    # -0 and +0 both encode as +0
    assert np.array_equal(back[vals != 0], codes[vals != 0])
    assert ai.e4m3_decode(np.array([0x7E]))[0] == 448.0
    assert ai.e4m3_decode(np.array([0x38]))[0] == 1.0
    assert ai.e4m3_decode(np.array([0x01]))[0] == 2.0 ** -9
    pos = np.sort(ai.e4m3_decode(np.arange(0, 0x7F)))
    mid = (pos[1:] + pos[:-1]) / 2
    lo = ai.e4m3_encode(mid)
    even = np.where((ai.e4m3_encode(pos[:-1]) & 1) == 0, ai.e4m3_encode(pos[:-1]),
                    ai.e4m3_encode(pos[1:]))
    assert np.array_equal(lo, even)
    assert ai.e4m3_decode(ai.e4m3_encode(np.array([1e6, -500.0, 464.0])))[0] == 448.0
    assert ai.e4m3_decode(ai.e4m3_encode(np.array([-500.0])))[0] == -448.0


def test_e4m3_matches_torch_cast_inside_range():
    f8 = getattr(torch, "float8_e4m3fn", None)
    if f8 is None:
        pytest.skip("torch has no float8_e4m3fn")
    x = ai.normals(11, 0, 50000) * 40.0
    x = x[np.abs(x) < 440]
    got = ai.e4m3_decode(ai.e4m3_encode(x))
    want = torch.from_numpy(x).to(f8).to(torch.float64).numpy()
    np.testing.assert_array_equal(got, want)


def test_fp8_inputs_dequantise_exactly():
    x = ai.make_qkv_fp8(1, 2, 64, 128, seed=5)
    for codes, scale, real in ((x.q8, x.descale[0], x.q), (x.v8, x.descale[2], x.v)):
        assert codes.dtype == np.uint8 and codes.shape == (1, 2, 64, 128)
        np.testing.assert_array_equal(ai.e4m3_decode(codes) * scale, real)
        assert np.abs(ai.e4m3_decode(codes)).max() <= 448
        assert math.log2(scale) == int(math.log2(scale))
    # the same normals as the 16-bit generator, before rounding
    z = ai.normals(5, 0, 64 * 128 * 2)
    rel = np.abs(x.q.reshape(-1) - z) / np.maximum(np.abs(z), 2 ** -6 * x.descale[0])
    assert rel.max() <= 2 ** -4 + 1e-12
