"""CUDA path vs the fp64 oracle, element by element, through the C ABI.

Small and ragged shapes are compared on every element; the full-size
workloads (the benchmark shapes, in the launch configuration the benchmark
times) on sampled rows.  Output buffers are NaN-poisoned first, so an
unwritten element fails.
"""
import json
import os

import numpy as np
import pytest

import attn_inputs
import parity
from parity import check_full, check_sampled, run_cuda, compare

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


def test_tiny_matches_golden_fixture():
    with open(os.path.join(HERE, "golden", "tiny_fp16_noncausal_oracle.json")) as f:
        g = json.load(f)
    w = attn_inputs.WORKLOADS["tiny"]
    x = w.inputs()
    o, lse = run_cuda(x, False)
    np.testing.assert_allclose(lse.reshape(-1), g["lse"], rtol=0, atol=1e-3)
    flat = o.reshape(-1, w.D)
    for r, vals in g["o_rows"].items():
        np.testing.assert_allclose(flat[int(r)], vals, rtol=0, atol=2e-3)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 127, 128, 129, 255, 300, 513])
def test_small_and_ragged(S, D, dtype, causal):
    x = attn_inputs.make_qkv(1, 2, S, D, dtype, seed=1000 + S + D)
    check_full(x, causal, f"S{S} D{D} {dtype} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_multi_head_multi_tile(D, causal):
    x = attn_inputs.make_qkv(2, 3, 1000, D, "bf16", seed=7)
    check_full(x, causal, f"B2 H3 S1000 D{D} causal={causal}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_stress_large_scores(dtype):
    """Q, K x 4: score std ~16, so the running max moves a lot."""
    x = attn_inputs.make_qkv(1, 4, 777, 128, dtype, seed=9, qk_mult=4.0)
    for causal in (False, True):
        check_full(x, causal, f"x4 {dtype} causal={causal}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_tile_maxima_jumping_past_the_overflow_cap(dtype):
    """Q, K x 8: score std ~64 (~92 log2 units), so a key tile's maximum
    often passes the reference chosen after the tile before by more than
    2^64 (the bf16 non-causal kernel's redo of a tile) and nearly every
    tile moves the reference."""
    x = attn_inputs.make_qkv(2, 3, 1000, 128, dtype, seed=19, qk_mult=8.0)
    for causal in (False, True):
        check_full(x, causal, f"x8 {dtype} causal={causal}")


def test_config_tiny():
    w = attn_inputs.WORKLOADS["tiny"]
    check_full(w.inputs(), False, w.name)


@pytest.mark.parametrize("key", ["s2048_d64", "s2048_d128"])
def test_config_s2048_full(key):
    w = attn_inputs.WORKLOADS[key]
    x = w.inputs()
    for causal in w.causal:
        check_full(x, causal, f"{w.name} causal={causal}")


@pytest.mark.parametrize("key", ["s8192_d128", "s8192_d128_x4"])
def test_config_s8192_sampled(key):
    w = attn_inputs.WORKLOADS[key]
    x = w.inputs()
    for causal in w.causal:
        check_sampled(x, causal, seed=w.seed, label=f"{w.name} causal={causal}")


@pytest.mark.parametrize("w", attn_inputs.sweep_workloads(), ids=lambda w: w.name)
def test_sweep_sampled(w):
    x = w.inputs()
    for causal in w.causal:
        check_sampled(x, causal, seed=w.seed, label=f"{w.name} causal={causal}",
                      stride=128)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("jstar", [100, 148, 228, 300])
def test_reference_moves_inside_a_tile(jstar, dtype):
    """Every query is one vector u and key j* is u too: each row's scaled
    score jumps at key j* by ~16 log2 units, past the 8 a reference may lag,
    in the first key tile, in the first or the second half of a later one."""
    x = attn_inputs.make_qkv(1, 2, 384, 128, dtype, seed=6700)
    x.q[:] = x.q[0, 0, 0]
    x.k[:, :, jstar] = x.q[0, 0, 0]
    for causal in (False, True):
        check_full(x, causal, f"jump at key {jstar} {dtype} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_zero_queries(D, dtype, causal):
    """Q = 0: every allowed score is 0, every weight 1, so O is the mean of
    the allowed V rows (a prefix mean when causal) and LSE the log of their
    count."""
    x = attn_inputs.make_qkv(1, 2, 300, D, dtype, seed=6800 + D)
    x.q[:] = 0.0
    check_full(x, causal, f"Q=0 D{D} {dtype} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128, 256])
def test_constant_value_rows(D, dtype, causal):
    """Every V row the same vector: any convex combination of them is that
    vector, whatever the scores."""
    x = attn_inputs.make_qkv(1, 2, 300, D, dtype, seed=6900 + D)
    x.v[:] = x.v[0, 0, 0]
    check_full(x, causal, f"constant V D{D} {dtype} causal={causal}")


def test_many_heads_short_sequences():
    x = attn_inputs.make_qkv(8, 64, 256, 64, "fp16", seed=11)
    for causal in (False, True):
        check_sampled(x, causal, seed=11, label=f"B8 H64 S256 causal={causal}")


def test_scale_argument():
    x = attn_inputs.make_qkv(1, 2, 200, 64, "fp16", seed=12)
    import oracle
    for scale in (0.05, 0.3):
        o, lse = run_cuda(x, True, scale=scale)
        ro, rl = oracle.attn_fwd(x.q, x.k, x.v, True, scale)
        compare(o, lse, ro, rl, "fp16", f"scale={scale}")


def test_repeated_calls_are_deterministic():
    x = attn_inputs.make_qkv(2, 4, 640, 128, "bf16", seed=13)
    o1, l1 = run_cuda(x, True)
    o2, l2 = run_cuda(x, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("offset_bytes", [0, 16])
@pytest.mark.parametrize("D", [64, 128])
def test_output_alignment(D, offset_bytes):
    """O (and the LSE) at a 32-byte boundary and 16 bytes past one: the
    epilogue's two store widths give the same result as the oracle."""
    import math

    import torch

    import exact_attention_forward_10_gb300 as fattn
    import oracle

    x = attn_inputs.make_qkv(1, 4, 300, D, "bf16", seed=1300 + D)
    dev = torch.device("cuda:0")
    q, k, v = (torch.from_numpy(a).to(dev).to(torch.bfloat16) for a in (x.q, x.k, x.v))
    n = q.numel()
    ob = torch.full((n + 64,), float("nan"), dtype=torch.bfloat16, device=dev)
    base = ob.data_ptr()
    skip = ((-base) % 32 + offset_bytes) // 2  # elements to a 32-byte boundary, then the offset
    o = ob[skip:skip + n].view(q.shape)
    assert (o.data_ptr() % 32) == offset_bytes
    lse = torch.full((1, 4, 300), float("nan"), dtype=torch.float32, device=dev)
    for causal in (False, True):
        rc = fattn.fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             1, 4, 300, D, causal, 1.0 / math.sqrt(D), fattn.FATTN_BF16, 0)
        assert rc == 0
        torch.cuda.synchronize()
        assert fattn.fattn_last_error(0)[0] == 0
        ro, rl = oracle.attn_fwd(x.q, x.k, x.v, causal, 1.0 / math.sqrt(D))
        compare(o.double().cpu().numpy(), lse.double().cpu().numpy(), ro, rl, "bf16",
                f"D{D} offset {offset_bytes} causal={causal}")
        # the guard elements around O were not written
        assert torch.isnan(ob[:skip]).all() and torch.isnan(ob[skip + n:]).all()


def test_causal_units_handed_out_at_run_time():
    """Causal launches at D = 256, and at D = 128 when the K and V of all
    heads exceed 64 MiB (96 MiB here), take their work units from a counter
    at run time (each launch a counter of its own from a pool of 256, reset
    by the launch's last CTA), in head groups sized to L2.  The
    shapes have several times more units than CTAs (pairs) and several head
    groups, so most units are fetched from the counter.  300 launches in a
    row, more than the pool, on the shapes in turn: every output is
    bit-identical to the first (a unit's result does not depend on which CTA
    computes it) and matches the oracle on sampled rows of every head."""
    import math

    import torch

    import exact_attention_forward_10_gb300 as fattn
    import oracle

    dev = torch.device("cuda:0")
    sets = []
    # D128: 96 heads x 8 units (three groups of 32 heads); D256: 40 heads x 8
    # pair units (three groups of 14, 14 and 12 heads)
    for (B, H, S, D, seed) in ((1, 96, 2048, 128, 1401), (1, 40, 2048, 256, 1402)):
        x = attn_inputs.make_qkv(B, H, S, D, "fp16", seed=seed)
        q, k, v = (torch.from_numpy(a).to(dev).to(torch.float16) for a in (x.q, x.k, x.v))
        sets.append((x, q, k, v, B, H, S, D))
    torch.cuda.synchronize()
    first = [None] * len(sets)
    for it in range(300):
        idx = it % len(sets)
        x, q, k, v, B, H, S, D = sets[idx]
        o = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, S), float("nan"), dtype=torch.float32, device=dev)
        rc = fattn.fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                             B, H, S, D, True, 1.0 / math.sqrt(D), fattn.FATTN_FP16, 0)
        assert rc == 0
        if first[idx] is None:
            torch.cuda.synchronize()
            first[idx] = (o.clone(), lse.clone())
        elif it % 37 == 0 or it >= 296:
            torch.cuda.synchronize()
            assert torch.equal(o, first[idx][0]) and torch.equal(lse, first[idx][1]), it
    torch.cuda.synchronize()
    assert fattn.fattn_last_error(0)[0] == 0
    for idx in range(len(sets)):
        x, q, k, v, B, H, S, D = sets[idx]
        o = first[idx][0].double().cpu().numpy()
        lse = first[idx][1].double().cpu().numpy()
        assert np.isfinite(o).all() and np.isfinite(lse).all()
        rows = parity.sample_rows(B, H, S, 1500 + idx, stride=64)
        ro, rl = oracle.attn_fwd(x.q, x.k, x.v, True, 1.0 / math.sqrt(D), rows=rows)
        compare(o.reshape(-1, D)[rows], lse.reshape(-1)[rows], ro, rl, "fp16",
                f"run-time units {B}x{H}x{S}x{D}")


@pytest.mark.parametrize("B,H,S,D,dtype", [
    (3, 11, 4096, 128, "bf16"),   # 33 heads in groups of 17 and 16
    (1, 20, 4096, 256, "fp16"),   # 20 heads in groups of 7, 7 and 6
    (1, 11, 4097, 256, "bf16"),   # ragged S: 11 heads in groups of 6 and 5
])
def test_causal_head_groups_with_remainder(B, H, S, D, dtype):
    """Causal units in L2-sized head groups whose last group is smaller than
    the others, and a ragged sequence: sampled rows of every head against
    the oracle."""
    x = attn_inputs.make_qkv(B, H, S, D, dtype, seed=1600 + H + D)
    check_sampled(x, True, seed=1600 + H, label=f"B{B} H{H} S{S} D{D} {dtype} causal",
                  stride=128)
