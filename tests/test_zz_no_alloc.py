"""The allocation-free cache entry point (fattn_fwd_kvcache_noalloc): same
results as fattn_fwd_kvcache on two calls in a row (the static scratch is
reused), its size limit, and its caller-provided status words.  Every call
goes through the C ABI with integer device pointers.  The file name sorts
last so it also runs after the rest of the suite."""
import math

import numpy as np
import pytest

import attn_inputs
import exact_attention_forward_10_gb300 as fattn
from exact_attention_forward_10_gb300 import build as fbuild

P = 1 << 20


def _call(a):
    return fattn.fattn_fwd_kvcache_noalloc(
        a["q"], a["k"], a["v"], a["lens"], a["o"], a["lse"], a["B"], a["H"],
        a["Sq"], a["Sk"], a["D"], a["causal"], a["scale"], a["dtype"],
        a["status"], a["stream"])


@pytest.mark.parametrize("args,want", [
    (dict(q=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(o=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(Sq=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(Sq=17), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(D=32), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(dtype=3), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(k=P * 3 + 2), fattn.FATTN_ERR_MISALIGNED),
    (dict(status=P * 17 + 2), fattn.FATTN_ERR_MISALIGNED),
])
def test_noalloc_host_side_rejections(args, want):
    fbuild.build()
    a = dict(q=P, k=P * 3, v=P * 7, lens=P * 15, o=P * 9, lse=P * 11, B=2, H=4,
             Sq=1, Sk=4096, D=128, causal=0, scale=0.125, dtype=1, status=P * 17,
             stream=0)
    a.update(args)
    assert _call(a) == want


@pytest.fixture(scope="module")
def torch_cuda():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch


def _device_inputs(torch, x):
    dev = torch.device("cuda:0")
    tdt = torch.bfloat16 if x.dtype == "bf16" else torch.float16
    q, k, v = (torch.from_numpy(t).to(dev).to(tdt) for t in (x.q, x.k, x.v))
    lens = (torch.as_tensor(x.lens, dtype=torch.int32, device=dev)
            if x.lens is not None else None)
    return q, k, v, lens


def _noalloc(torch, q, k, v, lens, causal, status=None):
    B, H, Sq, D = q.shape
    Sk = k.shape[2]
    o = torch.full_like(q, float("nan"))
    lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32, device=q.device)
    code = fattn.FATTN_BF16 if q.dtype == torch.bfloat16 else fattn.FATTN_FP16
    rc = fattn.fattn_fwd_kvcache_noalloc(
        q.data_ptr(), k.data_ptr(), v.data_ptr(),
        lens.data_ptr() if lens is not None else 0, o.data_ptr(), lse.data_ptr(),
        B, H, Sq, Sk, D, causal, 1.0 / math.sqrt(D), code,
        status.data_ptr() if status is not None else 0,
        torch.cuda.current_stream().cuda_stream)
    assert rc == fattn.FATTN_OK, fattn.fattn_error_string(rc)
    return o, lse


@pytest.mark.gpu
def test_two_calls_in_a_row_match_the_workspace_entry(torch_cuda):
    torch = torch_cuda
    xa = attn_inputs.make_kvcache(6, 8, 1, 3000, 128, "bf16", seed=3100,
                                  lens_range=(0, 3000))
    xb = attn_inputs.make_kvcache(3, 4, 4, 700, 64, "fp16", seed=3101,
                                  lens_range=(1, 700))
    cases = [(xa, False), (xb, True)]
    got = []
    status = torch.zeros(4, dtype=torch.int32, device="cuda:0")
    for x, causal in cases:  # back to back on one stream: the scratch is reused
        got.append(_noalloc(torch, *_device_inputs(torch, x), causal, status))
    torch.cuda.synchronize()
    assert status.cpu().tolist() == [0, 0, 0, 0]
    for (x, causal), (o, lse) in zip(cases, got):
        q, k, v, lens = _device_inputs(torch, x)
        want_o, want_l = fattn.forward_kvcache(q, k, v, lens, causal=causal)
        torch.cuda.synchronize()
        assert fattn.fattn_last_error(0)[0] == fattn.FATTN_OK
        np.testing.assert_array_equal(o.float().cpu().numpy(), want_o.float().cpu().numpy())
        np.testing.assert_array_equal(lse.cpu().numpy(), want_l.cpu().numpy())


@pytest.mark.gpu
def test_size_limit_is_enforced(torch_cuda):
    torch = torch_cuda
    # 16 query rows, D 128, many heads: the partials exceed the static scratch
    B, H, Sq, Sk, D = 64, 64, 16, 32, 128
    need = fattn.fattn_kvcache_plan(B, H, Sq, Sk, D)["workspace_bytes"]
    assert need > 32 << 20
    dev = torch.device("cuda:0")
    q = torch.zeros(B, H, Sq, D, dtype=torch.bfloat16, device=dev)
    k = torch.zeros(B, H, Sk, D, dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(B, H, Sq, dtype=torch.float32, device=dev)
    rc = fattn.fattn_fwd_kvcache_noalloc(
        q.data_ptr(), k.data_ptr(), k.data_ptr(), 0, o.data_ptr(), lse.data_ptr(),
        B, H, Sq, Sk, D, 0, 0.088, fattn.FATTN_BF16, 0, 0)
    assert rc == fattn.FATTN_ERR_TOO_LARGE


@pytest.mark.gpu
def test_kernel_errors_reach_the_caller_status_words(torch_cuda):
    torch = torch_cuda
    x = attn_inputs.make_kvcache(2, 2, 1, 64, 64, "bf16", seed=3102)
    q, k, v, _ = _device_inputs(torch, x)
    lens = torch.tensor([64, 65], dtype=torch.int32, device=q.device)
    status = torch.zeros(4, dtype=torch.int32, device=q.device)
    _noalloc(torch, q, k, v, lens, False, status)
    torch.cuda.synchronize()
    s = status.cpu().tolist()
    assert s[0] == fattn.FATTN_ERR_INVALID_ARG and s[1] >> 8 == 6 and s[2] == 1


@pytest.mark.gpu
def test_repeated_calls_leave_device_memory_unchanged(torch_cuda):
    """After the first call on the device (which may load the kernels'
    module), further calls change nothing in the device's free memory."""
    torch = torch_cuda
    x = attn_inputs.make_kvcache(4, 8, 2, 1500, 128, "bf16", seed=3103, lens_range=(1, 1500))
    q, k, v, lens = _device_inputs(torch, x)
    B, H, Sq, D = q.shape
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)

    def call():
        rc = fattn.fattn_fwd_kvcache_noalloc(
            q.data_ptr(), k.data_ptr(), v.data_ptr(), lens.data_ptr(), o.data_ptr(),
            lse.data_ptr(), B, H, Sq, k.shape[2], D, 1, 1.0 / math.sqrt(D),
            fattn.FATTN_BF16, 0, torch.cuda.current_stream().cuda_stream)
        assert rc == fattn.FATTN_OK, fattn.fattn_error_string(rc)
        torch.cuda.synchronize()

    call()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        call()
    assert torch.cuda.mem_get_info()[0] == free0
