"""Failure detection without a GPU fault: the bounded wait every kernel uses
gives up on a barrier that nothing completes, records
FATTN_ERR_PIPELINE_TIMEOUT in the device status block, and leaves the
context usable (a forward call afterwards still matches the oracle)."""
import time

import pytest

import attn_inputs
import exact_attention_forward_10_gb300 as fattn
from parity import check_full

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("limit_us", [2000, 50000])
def test_bounded_wait_gives_up_reports_and_recovers(limit_us):
    assert fattn.fattn_last_error(0)[0] == fattn.FATTN_OK  # nothing pending
    t0 = time.perf_counter()
    assert fattn.fattn_check_wait_timeout(limit_us, 0) == fattn.FATTN_OK
    rc, (where, block) = fattn.fattn_last_error(0)  # synchronises
    waited = time.perf_counter() - t0
    assert rc == fattn.FATTN_ERR_PIPELINE_TIMEOUT
    assert where == 7 << 8 and block == 0
    assert limit_us * 1e-6 <= waited < limit_us * 1e-6 + 2.0
    # the status was cleared by reading it, and the context still works
    assert fattn.fattn_last_error(0)[0] == fattn.FATTN_OK
    x = attn_inputs.make_qkv(1, 2, 300, 64, "fp16", seed=8000)
    check_full(x, True, "after a timed-out wait")
    assert fattn.fattn_last_error(0)[0] == fattn.FATTN_OK
