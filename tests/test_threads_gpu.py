"""Several host threads calling the library at once, each on its own CUDA
stream: every head dim of the self-attention kernels, the E4M3 kernel and
both cache-attention kernels.  Each thread repeats its call while the others
run theirs; afterwards every output matches the fp64 oracle and equals,
bit for bit, the same call made alone.  Run as the first test of a process,
the threads also take the library's one-time set-up paths (device state,
shared-memory opt-ins, the CTA-pair occupancy query) at the same time.

Every kernel of the library holds at least 148 KB of shared memory per CTA,
so CTAs of different launches never share an SM: concurrent launches only
interleave CTAs across SMs."""
from __future__ import annotations

import math
import threading

import numpy as np
import pytest

import attn_inputs
import oracle
from parity import compare, compare_kvcache, fp8_bound, torch_dtype

pytestmark = pytest.mark.gpu

REPS = 4


@pytest.fixture(scope="module")
def torch():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch


class _Job:
    """One call: device inputs and outputs allocated up front, the call
    itself, and the expected result."""

    def __init__(self, torch, kind, x, causal):
        import exact_attention_forward_10_gb300 as fattn

        self.kind, self.x, self.causal = kind, x, causal
        dev = torch.device("cuda:0")
        self.stream = torch.cuda.Stream(dev)
        if kind == "fp8":
            self.inp = [torch.from_numpy(a).to(dev) for a in (x.q8, x.k8, x.v8)]
            shape = x.q8.shape
            odt = torch_dtype("bf16")
        else:
            tdt = torch_dtype(x.dtype)
            self.inp = [torch.from_numpy(a).to(dev).to(tdt) for a in (x.q, x.k, x.v)]
            shape = x.q.shape
            odt = tdt
        B, H, Sq, D = shape
        self.o = torch.full(shape, float("nan"), dtype=odt, device=dev)
        self.lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32, device=dev)
        self.scale = 1.0 / math.sqrt(D)
        if kind == "kv":
            Sk = x.k.shape[2]
            self.lens = (None if x.lens is None else
                         torch.as_tensor(x.lens, dtype=torch.int32, device=dev))
            need = fattn.fattn_kvcache_plan(B, H, Sq, Sk, D)["workspace_bytes"]
            self.ws = torch.empty(max(16, need), dtype=torch.uint8, device=dev)

    def call(self):
        import exact_attention_forward_10_gb300 as fattn

        q, k, v = self.inp
        if self.kind == "fwd":
            fattn.forward(q, k, v, causal=self.causal, scale=self.scale,
                          out=self.o, lse=self.lse, stream=self.stream)
        elif self.kind == "fp8":
            fattn.forward_fp8(q, k, v, *self.x.descale, causal=self.causal,
                              scale=self.scale, out_dtype=self.o.dtype,
                              out=self.o, lse=self.lse, stream=self.stream)
        else:
            fattn.forward_kvcache(q, k, v, self.lens, causal=self.causal,
                                  scale=self.scale, out=self.o, lse=self.lse,
                                  workspace=self.ws, stream=self.stream)

    def result(self):
        return self.o.double().cpu().numpy(), self.lse.double().cpu().numpy()

    def check(self, o, lse, label):
        x = self.x
        if self.kind == "fwd":
            ro, rl = oracle.attn_fwd(x.q, x.k, x.v, self.causal, self.scale)
            compare(o, lse, ro, rl, x.dtype, label)
        elif self.kind == "fp8":
            ro, rl, tol = fp8_bound(x, self.causal, self.scale)
            assert np.isfinite(o).all() and np.isfinite(lse).all(), label
            assert (np.abs(o - ro) <= tol).all(), f"{label}: O outside the E4M3 bound"
            assert np.abs(lse - rl).max() <= 1e-3, f"{label}: LSE"
        else:
            ro, rl = oracle.attn_kvcache(x.q, x.k, x.v, self.causal, self.scale, x.lens)
            compare_kvcache(o, lse, ro, rl, x.dtype, label)


def _jobs(torch):
    kv4 = attn_inputs.make_kvcache(3, 4, 4, 900, 128, "bf16", seed=8003,
                                   lens_range=(1, 900))
    kv1 = attn_inputs.make_kvcache(2, 3, 1, 500, 64, "fp16", seed=8004,
                                   lens_range=(0, 500))
    return [
        ("D64 fp16 causal", _Job(torch, "fwd", attn_inputs.make_qkv(1, 3, 700, 64, "fp16", seed=8000), True)),
        ("D128 bf16", _Job(torch, "fwd", attn_inputs.make_qkv(2, 2, 513, 128, "bf16", seed=8001), False)),
        ("D256 fp16 causal", _Job(torch, "fwd", attn_inputs.make_qkv(1, 2, 300, 256, "fp16", seed=8002), True)),
        ("E4M3 D128 causal", _Job(torch, "fp8", attn_inputs.make_qkv_fp8(1, 2, 400, 128, seed=8005), True)),
        ("cache Sq4 D128 bf16 causal", _Job(torch, "kv", kv4, True)),
        ("cache Sq1 D64 fp16", _Job(torch, "kv", kv1, False)),
    ]


def test_concurrent_threads_match_oracle_and_solo_calls(torch):
    import exact_attention_forward_10_gb300 as fattn

    jobs = _jobs(torch)
    torch.cuda.synchronize()
    start = threading.Barrier(len(jobs))
    errors = []

    def worker(job):
        try:
            start.wait(timeout=60)
            for _ in range(REPS):
                job.call()
            job.stream.synchronize()
        except Exception as e:  # reported on the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(j,)) for _, j in jobs]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not any(t.is_alive() for t in threads), "a calling thread did not finish"
    assert not errors, errors
    torch.cuda.synchronize()
    rc, where = fattn.fattn_last_error(0)
    assert rc == 0, f"kernel status {rc} ({fattn.fattn_error_string(rc)}) at {where}"

    together = [j.result() for _, j in jobs]
    for (label, job), (o, lse) in zip(jobs, together):
        job.check(o, lse, label)

    # the same calls one at a time give the same bits
    for (label, job), (o, lse) in zip(jobs, together):
        job.o.fill_(float("nan"))
        job.lse.fill_(float("nan"))
        torch.cuda.synchronize()  # the fills ran on the current stream
        job.call()
        job.stream.synchronize()
        o1, l1 = job.result()
        np.testing.assert_array_equal(o1, o, err_msg=f"{label}: O differs from a solo call")
        np.testing.assert_array_equal(l1, lse, err_msg=f"{label}: LSE differs from a solo call")
