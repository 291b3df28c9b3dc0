"""Attention against a key/value cache: the CUDA path (split kernel + merge
kernel, through the C ABI) vs the fp64 cache oracle, every element.

Covers one to sixteen new queries, both head dims and dtypes, both masks,
ragged cached lengths (0, 1, tile edges, full capacity), caches whose stale
rows hold NaN, many short heads per warp and one long head over every warp,
the decoding workloads at full size, and the error paths the host and the
kernel report.  Output buffers are NaN-poisoned first.
"""
import math

import numpy as np
import pytest

import attn_inputs
from parity import check_kvcache, run_cuda_kvcache

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


EDGE_LENS = [0, 1, 31, 32, 33, 95, 257, 300]


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Sq", [1, 2, 4, 5, 11, 16])
def test_ragged_lengths(Sq, D, dtype, causal):
    x = attn_inputs.make_kvcache(len(EDGE_LENS), 3, Sq, 300, D, dtype,
                                 seed=2000 + Sq + D)
    x.lens = np.asarray(EDGE_LENS, dtype=np.int64)
    check_kvcache(x, causal, f"Sq{Sq} D{D} {dtype} causal={causal}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Sk", [1, 32, 33, 1000])
def test_full_caches_without_lengths(Sk, D):
    x = attn_inputs.make_kvcache(2, 5, 1, Sk, D, "bf16", seed=2100 + Sk)
    assert x.lens is None
    check_kvcache(x, False, f"Sk{Sk} D{D}")
    x4 = attn_inputs.make_kvcache(2, 5, 4, Sk, D, "fp16", seed=2150 + Sk)
    check_kvcache(x4, True, f"Sk{Sk} D{D} Sq4 causal")


def test_lengths_equal_to_capacity_match_no_lengths():
    """An explicit length of Sk for every batch is the same call as none."""
    x = attn_inputs.make_kvcache(3, 4, 2, 777, 128, "bf16", seed=2200)
    s = 1 / math.sqrt(128)
    o1, l1 = run_cuda_kvcache(x, True, s)
    o2, l2 = run_cuda_kvcache(x, True, s, lens=np.full(3, 777))
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


@pytest.mark.parametrize("D", [64, 128])
def test_stale_rows_hold_nan(D):
    """Cache rows at or past a batch's length are never read into the result,
    even when they hold NaN."""
    x = attn_inputs.make_kvcache(4, 2, 3, 500, D, "fp16", seed=2300 + D,
                                 lens_range=(1, 499))
    for causal in (False, True):
        check_kvcache(x, causal, f"stale NaN D{D} causal={causal}", stale_nan=True)


def test_many_short_heads_per_warp():
    """B*H far above the number of split warps: each warp covers many heads
    (and writes a record for each)."""
    x = attn_inputs.make_kvcache(64, 32, 1, 96, 64, "bf16", seed=2400,
                                 lens_range=(0, 96))
    check_kvcache(x, False, "B64 H32 short")


@pytest.mark.parametrize("Sq,D", [(8, 128), (16, 64)])
def test_many_short_heads_per_warp_multi_query(Sq, D):
    """The same with several queries (the tensor-core split kernel): every
    head switch inside a warp writes a record and reloads the query rows."""
    x = attn_inputs.make_kvcache(48, 16, Sq, 80, D, "fp16", seed=2450 + Sq,
                                 lens_range=(0, 80))
    for causal in (False, True):
        check_kvcache(x, causal, f"B48 H16 Sq{Sq} D{D} short causal={causal}")


def test_one_long_head_over_every_warp():
    """One head, a long cache: every split warp holds a slice of it and the
    merge combines hundreds of records."""
    x = attn_inputs.make_kvcache(1, 1, 2, 65536, 128, "bf16", seed=2500)
    for causal in (False, True):
        check_kvcache(x, causal, f"B1 H1 Sk65536 causal={causal}")


def test_query_scaled_scores():
    """Large scores (Q and K times 4) make the running maximum move often."""
    x = attn_inputs.make_kvcache(2, 4, 4, 3000, 128, "bf16", seed=2600,
                                 lens_range=(1, 3000))
    x.q *= np.float32(4.0)
    x.k *= np.float32(4.0)
    for causal in (False, True):
        check_kvcache(x, causal, f"Qx4 Kx4 causal={causal}")


@pytest.mark.parametrize("name", sorted(attn_inputs.CACHE_WORKLOADS))
def test_decoding_workloads_full_size(name):
    w = attn_inputs.CACHE_WORKLOADS[name]
    x = w.inputs()
    check_kvcache(x, w.causal, w.name)


def test_deterministic():
    x = attn_inputs.make_kvcache(4, 8, 1, 5000, 128, "bf16", seed=2700,
                                 lens_range=(100, 5000))
    s = 1 / math.sqrt(128)
    o1, l1 = run_cuda_kvcache(x, False, s)
    o2, l2 = run_cuda_kvcache(x, False, s)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ---------------------------------------------------------------- error paths

def _tensors(B=2, H=2, Sq=1, Sk=64, D=64):
    import torch
    dev = torch.device("cuda:0")
    q = torch.randn(B, H, Sq, D, device=dev, dtype=torch.bfloat16)
    k = torch.randn(B, H, Sk, D, device=dev, dtype=torch.bfloat16)
    v = torch.randn(B, H, Sk, D, device=dev, dtype=torch.bfloat16)
    return q, k, v


def test_workspace_too_small_is_rejected():
    import torch

    import exact_attention_forward_10_gb300 as fattn
    q, k, v = _tensors()
    need = fattn.fattn_kvcache_plan(2, 2, 1, 64, 64)["workspace_bytes"]
    ws = torch.empty(need - 16, dtype=torch.uint8, device=q.device)
    with pytest.raises(fattn.FattnError) as e:
        fattn.forward_kvcache(q, k, v, workspace=ws)
    assert e.value.status == fattn.FATTN_ERR_INVALID_ARG


def test_output_overlapping_an_input_is_rejected():
    import exact_attention_forward_10_gb300 as fattn
    q, k, v = _tensors()
    with pytest.raises(fattn.FattnError) as e:
        fattn.forward_kvcache(q, k, v, out=q)
    assert e.value.status == fattn.FATTN_ERR_INVALID_ARG


def test_length_out_of_range_is_reported():
    """A cached length above the capacity is clamped (every access stays in
    the cache) and reported by fattn_last_error with the batch index."""
    import torch

    import exact_attention_forward_10_gb300 as fattn
    q, k, v = _tensors()
    lens = torch.tensor([64, 65], dtype=torch.int32, device=q.device)
    fattn.forward_kvcache(q, k, v, lens)
    torch.cuda.synchronize()
    rc, (where, block) = fattn.fattn_last_error(0)
    assert rc == fattn.FATTN_ERR_INVALID_ARG
    assert where >> 8 == 6 and block == 1
    assert fattn.fattn_last_error(0)[0] == fattn.FATTN_OK  # cleared


def test_plan_is_consistent():
    import exact_attention_forward_10_gb300 as fattn
    p = fattn.fattn_kvcache_plan(16, 16, 1, 16384, 128)
    assert p["smem_bytes"] <= 232448 and p["block"] % 32 == 0
    assert p["split_warps"] == p["grid"] * (p["block"] // 32)
    recs = p["split_warps"] + 16 * 16
    assert p["workspace_bytes"] == recs * 1 * (128 + 1) * 4
    small = fattn.fattn_kvcache_plan(1, 1, 1, 32, 64)
    assert small["grid"] == 1
