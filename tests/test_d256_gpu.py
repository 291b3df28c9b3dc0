"""Head dim 256 (the CTA-pair kernel: clusters of two SMs issuing M = 256
tcgen05 MMAs) vs the fp64 oracle, through the C ABI.  Small and ragged
shapes on every element; long sequences and many units (more units than
co-resident clusters) on sampled rows.  Output buffers are NaN-poisoned."""
import numpy as np
import pytest

import attn_inputs
from parity import check_full, check_sampled, run_cuda

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("S", [1, 2, 127, 128, 129, 255, 256, 257, 300, 513, 640])
def test_small_and_ragged(S, dtype, causal):
    x = attn_inputs.make_qkv(1, 2, S, 256, dtype, seed=5000 + S)
    check_full(x, causal, f"D256 S{S} {dtype} causal={causal}")


@pytest.mark.parametrize("causal", [False, True])
def test_multi_head_multi_tile(causal):
    x = attn_inputs.make_qkv(2, 3, 1000, 256, "bf16", seed=5100)
    check_full(x, causal, f"D256 B2 H3 S1000 causal={causal}")


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_stress_large_scores(dtype):
    x = attn_inputs.make_qkv(1, 4, 777, 256, dtype, seed=5200, qk_mult=4.0)
    for causal in (False, True):
        check_full(x, causal, f"D256 x4 {dtype} causal={causal}")


def test_more_units_than_clusters():
    """1024 units of 256 rows: every cluster runs many rounds."""
    x = attn_inputs.make_qkv(4, 32, 2048, 256, "fp16", seed=5300)
    for causal in (False, True):
        check_sampled(x, causal, seed=5300, label=f"D256 B4 H32 S2048 causal={causal}",
                      stride=64)


@pytest.mark.parametrize("S", [4097, 8192])
def test_long_sequences_sampled(S):
    x = attn_inputs.make_qkv(2, 16, S, 256, "bf16", seed=5400 + S)
    for causal in (False, True):
        check_sampled(x, causal, seed=S, label=f"D256 B2 H16 S{S} causal={causal}",
                      stride=128)


def test_deterministic():
    x = attn_inputs.make_qkv(2, 4, 900, 256, "bf16", seed=5500)
    o1, l1 = run_cuda(x, True)
    o2, l2 = run_cuda(x, True)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
