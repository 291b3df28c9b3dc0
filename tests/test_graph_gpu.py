"""Entry points captured into a CUDA graph: each replay gives, bit for bit,
the output of the same call made outside the graph, replays repeated back to
back stay equal (the causal kernels' run-time unit counter is returned to 0
by each launch's last CTA, so the pair a graph captured starts every replay
at 0), and a replay after the inputs are overwritten in place computes on
the new values.  Captured launches take their counters from a ring of their
own, so ordinary launches made between replays stay correct too.

Every case has more work units than the GPU has SMs.  The causal cases at
D = 256, at D = 128 with H = 20, S = 4096 and in E4M3 with S = 16384 (K and
V of all heads over 32 MiB) hand units out at run time on every replay; the
D = 128 case with S = 2048 and the E4M3 one with S = 2048 take the static
order."""
from __future__ import annotations

import math

import numpy as np
import pytest

import attn_inputs
from parity import torch_dtype

pytestmark = pytest.mark.gpu

REPLAYS = 3


@pytest.fixture(scope="module")
def torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch


def _device_inputs(torch, kind, seed):
    dev = torch.device("cuda:0")
    if isinstance(kind, str) and kind.startswith("fp8"):
        S = int(kind[3:] or 2048)
        x = attn_inputs.make_qkv_fp8(2, 16, S, 128, seed=seed)
        return x, [torch.from_numpy(a).to(dev) for a in (x.q8, x.k8, x.v8)]
    B, H, S, D, dtype = kind
    x = attn_inputs.make_qkv(B, H, S, D, dtype, seed=seed)
    tdt = torch_dtype(dtype)
    return x, [torch.from_numpy(a).to(dev).to(tdt) for a in (x.q, x.k, x.v)]


def _call(fattn, kind, x, inp, causal, o, lse):
    q, k, v = inp
    if isinstance(kind, str) and kind.startswith("fp8"):
        fattn.forward_fp8(q, k, v, *x.descale, causal=causal, out_dtype=o.dtype,
                          out=o, lse=lse)
    else:
        fattn.forward(q, k, v, causal=causal, out=o, lse=lse)


CASES = [
    ("D128 bf16 causal", (2, 20, 4096, 128, "bf16"), True),
    ("D128 fp16 causal static", (2, 16, 2048, 128, "fp16"), True),
    ("D128 fp16", (2, 16, 2048, 128, "fp16"), False),
    ("D64 fp16 causal", (2, 16, 2048, 64, "fp16"), True),
    ("D256 bf16 causal", (2, 16, 2048, 256, "bf16"), True),
    ("E4M3 D128 causal", "fp8", True),
    ("E4M3 D128 causal S16384", "fp816384", True),
]


@pytest.mark.parametrize("label,kind,causal", CASES, ids=[c[0] for c in CASES])
def test_graph_replay_equals_eager_call(torch, label, kind, causal):
    import exact_attention_forward_10_gb300 as fattn

    x, inp = _device_inputs(torch, kind, seed=9100)
    shape = inp[0].shape
    odt = torch.bfloat16 if isinstance(kind, str) else inp[0].dtype
    B, H, S, _ = shape

    def outputs():
        return (torch.full(shape, float("nan"), dtype=odt, device="cuda:0"),
                torch.full((B, H, S), float("nan"), dtype=torch.float32, device="cuda:0"))

    # the first call on the device (its one-time set-up) is made before capture
    o_ref, lse_ref = outputs()
    _call(fattn, kind, x, inp, causal, o_ref, lse_ref)
    torch.cuda.synchronize()
    assert fattn.fattn_last_error()[0] == 0, label

    o, lse = outputs()
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    with torch.cuda.graph(g, stream=side):
        _call(fattn, kind, x, inp, causal, o, lse)
    torch.cuda.synchronize()

    for rep in range(REPLAYS):
        o.fill_(float("nan"))
        lse.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), f"{label}: O of replay {rep} differs from the eager call"
        assert torch.equal(lse, lse_ref), f"{label}: LSE of replay {rep} differs"
        # an ordinary launch between replays, on its own counter
        o2, lse2 = outputs()
        _call(fattn, kind, x, inp, causal, o2, lse2)
        torch.cuda.synchronize()
        assert torch.equal(o2, o_ref) and torch.equal(lse2, lse_ref), \
            f"{label}: eager call after replay {rep} differs"

    # new values in the captured input buffers: the replay reads them
    x_new, inp_new = _device_inputs(torch, kind, seed=9200)
    for dst, src in zip(inp, inp_new):
        dst.copy_(src)
    o_new, lse_new = outputs()
    _call(fattn, kind, x_new, inp, causal, o_new, lse_new)
    g.replay()
    torch.cuda.synchronize()
    assert not torch.equal(o_new, o_ref), f"{label}: new inputs gave the old output"
    assert torch.equal(o, o_new) and torch.equal(lse, lse_new), \
        f"{label}: replay on overwritten inputs differs from the eager call"
    assert fattn.fattn_last_error()[0] == 0, label
    assert np.isfinite(lse.cpu().numpy()).all(), label


@pytest.mark.parametrize("Sq,D", [(4, 128), (1, 64), (1, 128)])
def test_graph_of_cache_attention(torch, Sq, D):
    """Cache attention captured and replayed, one and several new queries,
    with a batch that has no cached key: every replay equals the eager
    call."""
    import exact_attention_forward_10_gb300 as fattn

    dev = torch.device("cuda:0")
    x = attn_inputs.make_kvcache(4, 8, Sq, 3000, D, "bf16", seed=9300 + Sq + D,
                                 lens_range=(1, 3000))
    x.lens[1] = 0
    tdt = torch_dtype("bf16")
    q, kc, vc = (torch.from_numpy(a).to(dev).to(tdt) for a in (x.q, x.k, x.v))
    lens = torch.as_tensor(x.lens, dtype=torch.int32, device=dev)
    B, H, Sq, D = q.shape
    need = fattn.fattn_kvcache_plan(B, H, Sq, kc.shape[2], D)["workspace_bytes"]
    ws = torch.empty(max(16, need), dtype=torch.uint8, device=dev)
    scale = 1.0 / math.sqrt(D)

    o_ref, lse_ref = fattn.forward_kvcache(q, kc, vc, lens, causal=True, scale=scale,
                                           workspace=ws)
    torch.cuda.synchronize()
    o = torch.full_like(o_ref, float("nan"))
    lse = torch.full_like(lse_ref, float("nan"))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=torch.cuda.Stream()):
        fattn.forward_kvcache(q, kc, vc, lens, causal=True, scale=scale, out=o,
                              lse=lse, workspace=ws)
    for rep in range(REPLAYS):
        o.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref), f"replay {rep}"
    assert fattn.fattn_last_error()[0] == 0
