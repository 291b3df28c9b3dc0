"""Attention-forward benchmark: TFLOPS (4 B H S^2 D, halved when causal).

One step is one pass of the whole path over one batch: the non-causal and the
causal forward of the B=2, H=16, S=8192, D=128 bf16 workload (seed 3), each a
single fattn_fwd launch through the C ABI.  Inputs (192 MiB Q, K, V) and
outputs are larger than L2, so no flush is needed between steps.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

N > 1 runs under torchrun as data parallelism over the batch (weak scaling):
the global batch is N x 2 rows, each rank generates and runs its own shard of
2 rows (no collective on the data path); the timing is the max over ranks.
``--fp8`` and ``--kvcache`` run the same workload on every rank (replicas).
``--impl reference`` times the fp64 CPU oracle on a bounded row sample of the
same workload (the reference arm: this path has no other implementation).

``--kvcache [NAME]`` times attention of new queries against a key/value cache
instead ("FlashAttention V2", section 6: inference with a KV cache): one step
is one fattn_fwd_kvcache call on a cache workload of ``attn_inputs`` (default:
16 sequences, 16 heads, D=128 bf16, one new token, cached lengths 1024..16384),
reported as effective HBM GB/s against the measured copy bandwidth.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import attn_inputs  # noqa: E402

METRIC = ("attn fwd TFLOPS (4BHS²D, ½ if causal) and % of GB300 dense "
          "16-bit tensor peak")
UNIT = "TFLOP/s"
WORKLOAD = attn_inputs.WORKLOADS["s8192_d128"]
MASKS = (False, True)


def metric_flops(B, H, S, D, causal) -> float:
    f = 4.0 * B * H * S * S * D
    return f / 2 if causal else f


def row_flops(S, D, causal) -> float:
    """The metric's FLOPs per query row (causal: the halved average)."""
    return (2.0 if causal else 4.0) * S * D


def algo_bytes(B, H, S, D) -> int:
    """Algorithmic HBM bytes of one launch: Q, K, V read once, O and the
    fp32 LSE written once (16-bit tensors)."""
    return B * H * S * (8 * D + 4)


# Accuracy targets of the library: max|O - O_ref| 2e-3 (fp16) / 1.5e-2 (bf16),
# |LSE - LSE_ref| 1e-3.  An element with |O_ref| >= 4 also passes within the
# flat bound plus half a unit in the last place of the 16-bit dtype there
# (the final cast alone can miss by that much); how many elements needed that
# allowance is reported beside the flat result.
TOL_O = {"fp16": 2e-3, "bf16": 1.5e-2}
TOL_LSE = 1e-3
MANT_BITS = {"fp16": 10, "bf16": 7}


def parity_stats(o, lse, ro, rl, dtype: str) -> dict:
    """Worst errors of GPU rows (o [n, D], lse [n]) against the oracle's."""
    o, lse, ro, rl = (np.asarray(a, dtype=np.float64) for a in (o, lse, ro, rl))
    finite = bool(np.isfinite(o).all() and np.isfinite(lse).all())
    err = np.abs(o - ro)
    tol = TOL_O[dtype]
    ax = np.maximum(np.abs(ro), 2.0 ** -14)
    half_ulp = 0.5 * np.exp2(np.floor(np.log2(ax)) - MANT_BITS[dtype])
    flat_ok = err <= tol
    ok = flat_ok | ((np.abs(ro) >= 4.0) & (err <= tol + half_ulp))
    dl = np.abs(lse - rl)
    e_o = float(err.max()) if err.size else 0.0
    e_l = float(dl.max()) if dl.size else 0.0
    return {"rows": int(o.shape[0]), "max_abs_dO": e_o, "max_abs_dLSE": e_l,
            "tol_O": tol, "tol_LSE": TOL_LSE, "flat_pass": bool(flat_ok.all()) and finite,
            "n_pass_by_ulp_allowance": int((ok & ~flat_ok).sum()),
            "pass": bool(ok.all()) and e_l <= TOL_LSE and finite}


def merge_parity(parts) -> dict:
    """One block over several (mask) comparisons: worst errors, all passes."""
    parts = list(parts)
    return {"rows": sum(p["rows"] for p in parts),
            "max_abs_dO": max(p["max_abs_dO"] for p in parts),
            "max_abs_dLSE": max(p["max_abs_dLSE"] for p in parts),
            "tol_O": parts[0]["tol_O"], "tol_LSE": TOL_LSE,
            "flat_pass": all(p["flat_pass"] for p in parts),
            "n_pass_by_ulp_allowance": sum(p["n_pass_by_ulp_allowance"] for p in parts),
            "pass": all(p["pass"] for p in parts)}


def head_rows(B: int, H: int, S: int, seed: int, edge: int = 16, inner: int = 8):
    """Rows of every (batch, head): the first and last ``edge`` rows and
    ``inner`` seeded others (all rows when S is small)."""
    rng = np.random.default_rng(seed)
    out = []
    for bh in range(B * H):
        if S <= 2 * edge + inner:
            r = np.arange(S)
        else:
            mid = rng.choice(np.arange(edge, S - edge), size=inner, replace=False)
            r = np.concatenate([np.arange(edge), np.sort(mid), np.arange(S - edge, S)])
        out.append(bh * S + r)
    return np.concatenate(out).astype(np.int64)


def gather_rows(torch, o, lse, rows):
    """Rows (global indices into [B*H*S]) of device outputs, as fp64 numpy."""
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    D = o.shape[-1]
    return (o.reshape(-1, D).index_select(0, idx).double().cpu().numpy(),
            lse.reshape(-1).index_select(0, idx).double().cpu().numpy())


# GB300's L2 (126.5 MiB), rounded up.  A timed launch whose inputs are
# smaller than this runs after an L2 flush (a write of twice its size
# outside the launch's own CUDA events).
L2_BYTES = 129 * 2**20


def l2_flush_buffer(torch, dev, input_bytes: int):
    """The buffer to overwrite before each timed launch, or None when the
    launch's inputs are larger than L2."""
    if input_bytes > L2_BYTES:
        return None
    return torch.empty(2 * L2_BYTES, dtype=torch.uint8, device=dev)


def l2_label(input_bytes: int, what: str = "Q,K,V") -> str:
    if input_bytes > L2_BYTES:
        return f"inputs larger than L2 ({what} {input_bytes / 2**20:.0f} MiB); no flush"
    return (f"inputs smaller than L2 ({what} {input_bytes / 2**20:.0f} MiB): L2 flushed "
            f"(a {2 * L2_BYTES / 2**20:.0f} MiB write) before each timed launch, outside its "
            "CUDA events; the step time is the sum of the launches' event times")


def workload_config(w, extra=None, elem_bytes: int = 2) -> dict:
    c = {"workload": f"B{w.B} H{w.H} S{w.S} D{w.D} {w.dtype}, non-causal + "
                     f"causal, Q/K/V iid N(0,1) seed {w.seed}, scale 1/sqrt(D)",
         "B": w.B, "H": w.H, "S": w.S, "D": w.D, "masks": "non-causal+causal",
         "l2": l2_label(3 * elem_bytes * w.B * w.H * w.S * w.D)}
    if extra:
        c.update(extra)
    return c


def load_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"burst": float(d["bf16_tflops"]),
                "sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    return {"burst": 1900.0, "sustained": 1700.0, "source": "fallback"}


class NvmlClockSampler:
    """SM clock, power and clock-event reasons read through NVML (the
    driver's libnvidia-ml, read-only queries) every ``period_s`` while the
    timed region runs, so a region of a few tens of milliseconds still
    gives tens of samples.  ``ok`` is False when NVML cannot be used."""

    # clock-event reason bits of nvmlDeviceGetCurrentClocksEventReasons
    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, pci_bus_id: str | None, index: int, period_s: float = 0.0005):
        import ctypes
        self.period = period_s
        self.samples = []
        self.thread = None
        self.stop_flag = threading.Event()
        self.ok = False
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.handle = ctypes.c_void_p()
            rc = -1
            if pci_bus_id:
                rc = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(
                    pci_bus_id.encode(), ctypes.byref(self.handle))
            if rc != 0:
                rc = self.nvml.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.handle))
            if rc != 0:
                return
            fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None)
            self.reasons_fn = fn or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            mx = ctypes.c_uint()
            self.max_mhz = (mx.value if self.nvml.nvmlDeviceGetMaxClockInfo(
                self.handle, 1, ctypes.byref(mx)) == 0 else None)
            self.ok = True
        except (OSError, AttributeError):
            self.ok = False

    def _read(self):
        import ctypes
        mhz, reasons, mw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self.stop_flag.is_set():
            if self.nvml.nvmlDeviceGetClockInfo(self.handle, 1, ctypes.byref(mhz)) == 0:
                r = reasons.value if self.reasons_fn(self.handle, ctypes.byref(reasons)) == 0 else 0
                w = mw.value / 1000.0 if self.nvml.nvmlDeviceGetPowerUsage(
                    self.handle, ctypes.byref(mw)) == 0 else None
                self.samples.append((mhz.value, r, w))
            time.sleep(self.period)

    def start(self):
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def stop(self) -> dict:
        self.stop_flag.set()
        if self.thread:
            self.thread.join(timeout=5)
        sm = [s[0] for s in self.samples]
        reasons = set()
        for _, r, _ in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit:
                    reasons.add(name)
        power = [s[2] for s in self.samples if s[2] is not None]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_min_mhz": min(sm) if sm else None,
                "sm_max_mhz": self.max_mhz,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "source": f"NVML every {self.period * 1e3:.1f} ms",
                "reasons": sorted(reasons)}


def clock_sampler(dev):
    """The NVML sampler when NVML answers, else nvidia-smi."""
    s = NvmlClockSampler(gpu_pci_bus_id(dev), dev.index)
    return s if s.ok else ClockSampler(dev.index)


def gpu_pci_bus_id(dev) -> str | None:
    """``domain:bus:device.0`` of the GPU, from torch's device properties."""
    import torch
    p = torch.cuda.get_device_properties(dev)
    if not all(hasattr(p, a) for a in ("pci_domain_id", "pci_bus_id", "pci_device_id")):
        return None
    return f"{p.pci_domain_id:04x}:{p.pci_bus_id:02x}:{p.pci_device_id:02x}.0"


def gpu_local_cpus(dev):
    """The host CPUs on the GPU's side of the machine (the PCI device's
    ``local_cpulist`` in sysfs) and its NUMA node; (None, None) when the
    system does not say."""
    bus = gpu_pci_bus_id(dev)
    if bus is None:
        return None, None
    base = f"/sys/bus/pci/devices/{bus}"
    cpus, node = None, None
    try:
        with open(f"{base}/local_cpulist") as f:
            cpus = set()
            for part in f.read().strip().split(","):
                if "-" in part:
                    a, b = part.split("-")
                    cpus.update(range(int(a), int(b) + 1))
                elif part:
                    cpus.add(int(part))
        with open(f"{base}/numa_node") as f:
            node = int(f.read().strip())
    except (OSError, ValueError):
        pass
    return cpus, node


def pinned_near_gpu(dev, make):
    """Run ``make()`` (which allocates pinned host buffers) with this thread
    on the GPU's local CPUs, so first-touch places the pages on that side of
    the machine; the previous affinity is restored afterwards.  Returns
    (make's result, a note saying what was done)."""
    cpus, node = gpu_local_cpus(dev)
    old = os.sched_getaffinity(0)
    use = (cpus & old) if cpus else None
    if not use or use == old:
        note = (f"pinned buffers allocated from the process's CPUs "
                f"({len(old)}; GPU-local CPU list {'equal' if use else 'not available'})")
        return make(), note
    os.sched_setaffinity(0, use)
    try:
        out = make()
    finally:
        os.sched_setaffinity(0, old)
    return out, (f"pinned buffers allocated with the thread on the GPU's {len(use)} local CPUs "
                 f"(NUMA node {node}) of {len(old)}")


def copy_gbs(torch, dev, stream, src, dst, reps: int = 5) -> float:
    """GB/s of copying ``src`` into ``dst`` (one list of tensors each way),
    each copy alone on ``stream``, best of ``reps``."""
    nbytes = sum(t.numel() * t.element_size() for t in src)
    best = None
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            for d, s_ in zip(dst, src):
                d.copy_(s_, non_blocking=True)
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    return nbytes / (best * 1e-3) / 1e9


def copy_both_ms(torch, dev, h2d, d2h, reps: int = 5) -> float:
    """Milliseconds for one host-to-device copy set (``h2d``: pairs (dst,
    src)) and one device-to-host set (``d2h``) issued at the same time on
    two streams, best of ``reps``: whether the two directions overlap."""
    s1, s2 = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    best = None
    for _ in range(reps):
        torch.cuda.synchronize(dev)
        a = torch.cuda.Event(enable_timing=True)
        b1 = torch.cuda.Event()
        b = torch.cuda.Event(enable_timing=True)
        a.record(s1)
        s2.wait_event(a)
        with torch.cuda.stream(s1):
            for d, x in h2d:
                d.copy_(x, non_blocking=True)
        with torch.cuda.stream(s2):
            for d, x in d2h:
                d.copy_(x, non_blocking=True)
            b1.record(s2)
        s1.wait_event(b1)
        b.record(s1)
        torch.cuda.synchronize(dev)
        ms = a.elapsed_time(b)
        best = ms if best is None else min(best, ms)
    return best


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.thread:
            self.thread.join(timeout=5)
        sm, smax, power, reasons = [], [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap")
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                smax.append(float(parts[1]))
                power.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[4:8]):
                if val.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def pipelined_e2e_ms(torch, dev, stream, host, launch_into, new_outputs, h_outs, steps,
                     barrier) -> float:
    """Milliseconds per step of a stream of end-to-end steps: each copies its
    inputs (``host``, pinned) to the GPU, runs ``launch_into(inputs,
    outputs)`` on ``stream`` and copies the outputs to ``h_outs`` (pinned;
    mask -> (O, LSE)); step k+1's input copy and step k-1's output copy
    overlap step k's kernels (an H2D and a D2H stream, two device buffers,
    events between them)."""
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    din = [[torch.empty_like(h, device=dev) for h in host] for _ in range(2)]
    dout = [new_outputs() for _ in range(2)]
    ev_in, ev_done, ev_out = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))

    def run(n):
        for kstep in range(n):
            b = kstep % 2
            if kstep >= 2:
                h2d_s.wait_event(ev_done[b])  # step k-2's kernels have read din[b]
            with torch.cuda.stream(h2d_s):
                for dst, src in zip(din[b], host):
                    dst.copy_(src, non_blocking=True)
                ev_in[b].record(h2d_s)
            stream.wait_event(ev_in[b])
            if kstep >= 2:
                stream.wait_event(ev_out[b])  # step k-2's outputs are on the host
            with torch.cuda.stream(stream):
                launch_into(din[b], dout[b])
                ev_done[b].record(stream)
            d2h_s.wait_event(ev_done[b])
            with torch.cuda.stream(d2h_s):
                for c, (ho, hl) in h_outs.items():
                    ho.copy_(dout[b][c][0], non_blocking=True)
                    hl.copy_(dout[b][c][1], non_blocking=True)
                ev_out[b].record(d2h_s)

    run(2)
    barrier()
    p0 = torch.cuda.Event(enable_timing=True)
    p1 = torch.cuda.Event(enable_timing=True)
    p0.record(h2d_s)
    stream.wait_event(p0)
    d2h_s.wait_event(p0)
    run(steps)
    p1.record(d2h_s)
    barrier()
    return p0.elapsed_time(p1) / steps


E2E_SCHEDULE = ("steps pipelined: step k+1's H2D and step k-1's D2H overlap step k's "
                "kernels (three streams, two buffers)")


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


# ------------------------------------------------------------ reference arm

def oracle_sample_rows(w, n_rows: int, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return np.sort(rng.choice(w.B * w.H * w.S, size=n_rows, replace=False))


def cpu_oracle_run(x, w, rows_per_mask: int, seed: int, keep: bool = False):
    """Oracle on ``rows_per_mask`` sampled rows per mask; returns (seconds,
    metric FLOPs of those rows, threads, and with ``keep`` a dict mask ->
    (rows, O rows, LSE rows))."""
    import oracle
    threads = oracle.default_threads()
    flops = 0.0
    outs = {}
    t0 = time.perf_counter()
    for m, causal in enumerate(MASKS):
        rows = oracle_sample_rows(w, rows_per_mask, seed + m)
        ro, rl = oracle.attn_fwd(x.q, x.k, x.v, causal, w.scale, rows=rows, threads=threads)
        if keep:
            outs[causal] = (rows, ro, rl)
        flops += rows_per_mask * row_flops(w.S, w.D, causal)
    dt = time.perf_counter() - t0
    return (dt, flops, threads, outs) if keep else (dt, flops, threads)


def calibrate_rows(x, w, target_s: float) -> int:
    """Rows per mask so that one oracle sample takes about ``target_s``."""
    n = 64
    dt, _, _ = cpu_oracle_run(x, w, n, 999)
    while dt < 0.5 and n < (1 << 16):
        n *= 4
        dt, _, _ = cpu_oracle_run(x, w, n, 999)
    return max(16, int(n * target_s / max(dt, 1e-6)))


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    w = WORKLOAD
    x = w.inputs()
    rows = calibrate_rows(x, w, target_s=max(0.2, min(10.0, 90.0 / max(1, args.steps + args.warmup))))
    for i in range(args.warmup):
        cpu_oracle_run(x, w, rows, 100 + i)
    times, flops = [], 0.0
    threads = 1
    for i in range(args.steps):
        dt, fl, threads = cpu_oracle_run(x, w, rows, 1000 + i)
        times.append(dt)
        flops += fl
    total = sum(times)
    value = flops / total / 1e12
    sample = (f"{rows} sampled query rows per mask per step (of {w.B * w.H * w.S}); "
              f"metric FLOPs of those rows / wall time")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": 1000.0 * total / max(1, args.steps),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(w, {"parallelism": "host cores, rank 0 only"}),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------------ our arm

def run_fattn(args):
    import torch

    import exact_attention_forward_10_gb300 as fattn

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    w = WORKLOAD
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    # weak scaling: a global batch of world x B rows, each rank its own shard
    from exact_attention_forward_10_gb300 import shard
    global_b = world * w.B
    b0, b1 = shard.batch_range(global_b, world, rank)
    x = (w.inputs() if world == 1 else
         attn_inputs.make_qkv_shard(global_b, b0, b1, w.H, w.S, w.D, w.dtype, w.seed))
    host, placement = pinned_near_gpu(
        dev, lambda: [torch.from_numpy(a).to(tdt).pin_memory() for a in (x.q, x.k, x.v)])
    q, k, v = (h.to(dev) for h in host)
    B, H, S, D = b1 - b0, w.H, w.S, w.D
    outs = {c: (torch.empty_like(q), torch.empty((B, H, S), dtype=torch.float32, device=dev))
            for c in MASKS}
    stream = torch.cuda.Stream(dev)
    # the launch stream does not wait for the default stream by itself
    stream.wait_stream(torch.cuda.current_stream(dev))
    sptr = stream.cuda_stream
    code = fattn.FATTN_BF16 if w.dtype == "bf16" else fattn.FATTN_FP16

    def launch(causal, qq, kk, vv, into=None):
        o, l = (into or outs)[causal]
        rc = fattn.fattn_fwd(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), o.data_ptr(),
                             l.data_ptr(), B, H, S, D, causal, w.scale, code, sptr)
        if rc != 0:
            raise fattn.FattnError(rc)

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    # correctness gate before timing: no kernel error
    with torch.cuda.stream(stream):
        for c in MASKS:
            launch(c, q, k, v)
    rc, where = fattn.fattn_last_error(sptr)
    if rc != 0:
        raise RuntimeError(f"kernel status {rc} at {where}")

    # ---- device-timed region: inputs resident in HBM
    n_ev = args.steps * len(MASKS)
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(n_ev)]
    flush = l2_flush_buffer(torch, dev, 3 * 2 * B * H * S * D)
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for c in MASKS:
                launch(c, q, k, v)
    barrier()
    sampler = clock_sampler(dev)
    sampler.start()
    time.sleep(0.05)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t_start.record(stream)
        e = 0
        for _ in range(args.steps):
            for c in MASKS:
                if flush is not None:
                    flush.add_(1)
                ev[e][0].record(stream)
                launch(c, q, k, v)
                ev[e][1].record(stream)
                e += 1
        t_end.record(stream)
    barrier()
    clocks = sampler.stop()
    elapsed_ms = t_start.elapsed_time(t_end)
    per_launch = {c: [] for c in MASKS}
    for i, (a, b) in enumerate(ev):
        per_launch[MASKS[i % len(MASKS)]].append(a.elapsed_time(b))
    if flush is not None:  # the flushes are not part of the step
        elapsed_ms = sum(a.elapsed_time(b) for a, b in ev)
    rc, where = fattn.fattn_last_error(sptr)
    if rc != 0:
        raise RuntimeError(f"kernel status {rc} at {where}")

    # ---- end to end through the public call, host buffers: every step copies
    # its Q, K, V in from pinned host memory and reads O and the LSE back.
    # As a stream of batches runs: step k+1's input copy and step k-1's output
    # copy overlap step k's kernels (an H2D and a D2H stream beside the compute
    # stream, two device buffers).  The same steps one after another on one
    # stream are reported too (e2e "serial").
    h_outs, _ = pinned_near_gpu(
        dev, lambda: {c: (torch.empty((B, H, S, D), dtype=tdt).pin_memory(),
                          torch.empty((B, H, S), dtype=torch.float32).pin_memory())
                      for c in MASKS})
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        qq, kk, vv = (h.to(dev, non_blocking=True) for h in host)
        for c in MASKS:
            launch(c, qq, kk, vv)
        for c in MASKS:
            h_outs[c][0].copy_(outs[c][0], non_blocking=True)
            h_outs[c][1].copy_(outs[c][1], non_blocking=True)

    with torch.cuda.stream(stream):
        for _ in range(2):
            e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
    barrier()
    e2e_serial_ms = e0.elapsed_time(e1) / e2e_steps

    e2e_ms = pipelined_e2e_ms(
        torch, dev, stream, host,
        lambda din, dout: [launch(c, *din, into=dout) for c in MASKS],
        lambda: {c: (torch.empty_like(q), torch.empty((B, H, S), dtype=torch.float32, device=dev))
                 for c in MASKS},
        h_outs, e2e_steps, barrier)
    h2d = sum(h.numel() * h.element_size() for h in host)
    d2h = sum(o.numel() * o.element_size() + l.numel() * l.element_size()
              for o, l in h_outs.values())
    # each direction's copy alone, so the record shows whether a step is
    # bound by the host link rather than by the kernels
    h2d_gbs = copy_gbs(torch, dev, stream, host, [q, k, v])
    d2h_gbs = copy_gbs(torch, dev, stream,
                       [t for c in MASKS for t in outs[c]], [t for c in MASKS for t in h_outs[c]])
    both_ms = copy_both_ms(torch, dev, list(zip([q, k, v], host)),
                           [(hh, d) for c in MASKS for hh, d in zip(h_outs[c], outs[c])])
    per_config, keep = [], []
    if rank == 0 and not args.no_per_config:
        per_config, keep = run_per_config(torch, fattn, dev, stream, load_peaks(),
                                          main_x=x if world == 1 else None, main_w=w)

    # ---- max over ranks
    step_ms, e2e_ms, e2e_serial_ms = shard.max_over_ranks(
        [elapsed_ms / args.steps, e2e_ms, e2e_serial_ms], device=dev)

    flops_step = sum(metric_flops(B, H, S, D, c) for c in MASKS)
    value = world * flops_step / (step_ms * 1e-3) / 1e12
    e2e_value = world * flops_step / (e2e_ms * 1e-3) / 1e12
    peaks = load_peaks()
    per_mask = {}
    for c in MASKS:
        ms = statistics.median(per_launch[c])
        tf = metric_flops(B, H, S, D, c) / (ms * 1e-3) / 1e12
        per_mask["causal" if c else "noncausal"] = {
            "ms_median": ms, "tflops": tf, "frac_of_measured_burst": tf / peaks["burst"],
            "hbm_gbs": algo_bytes(B, H, S, D) / (ms * 1e-3) / 1e9}
    # dominant kernel: the non-causal launch (2/3 of the step's FLOPs)
    dom_ms = statistics.mean(per_launch[False])
    achieved = metric_flops(B, H, S, D, False) / (dom_ms * 1e-3) / 1e12
    traffic = load_traffic(f"fattn_fwd_noncausal_{w.dtype}_d{D}_s{S}",
                           "fattn_pair" if D == 256 else "fattn_fwd")
    plan = fattn.fattn_plan(B, H, S, D, False)

    hbm = load_hbm_peak()
    step_bytes = world * len(MASKS) * algo_bytes(B, H, S, D)
    result = None
    if rank == 0:
        cpu, parity = None, None
        if world == 1 and not args.no_cpu_baseline:
            # the oracle leg: its timed sample, then its results on the same
            # rows compared with the GPU's, and each configuration's rows
            cpu, oracle_outs = cpu_baseline(x, w, keep=True)
            parity = oracle_parity(torch, outs, oracle_outs, w.dtype)
            per_config_parity(per_config, keep)
        result = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": workload_config(w, {"parallelism": (f"data parallel x{world}: each rank "
                                                          f"{B} of {global_b} batch rows")
                                                          if world > 1 else "one GPU",
                                          "global_batch": global_b,
                                          "grid": plan["grid"], "block": plan["block"],
                                          "units_per_launch": plan["units"]}),
            "per_mask": per_mask,
            "hbm_gbs": step_bytes / (step_ms * 1e-3) / 1e9,
            "hbm": {"algorithmic_bytes_per_step": step_bytes,
                    "frac_of_measured_copy": step_bytes / (step_ms * 1e-3) / 1e9 / hbm["gbs"],
                    "peak_gbs": hbm["gbs"], "peak_kind": f"HBM copy, {hbm['source']}",
                    "note": "Q, K, V read once and O, LSE written once per launch over the "
                            "step time: far below the copy bandwidth, so the step is bound "
                            "by the tensor pipe, not by HBM"},
            "parity": parity,
            "per_config": per_config,
            "roofline": {"bound": "tensor", "achieved": achieved,
                         "peak": peaks["burst"], "unit": "TFLOP/s",
                         "frac": achieved / peaks["burst"],
                         "peak_kind": f"bf16 dense, {peaks['source']} burst",
                         "kernel": (f"fattn_fwd_pair_kernel<D=256, non-causal, {w.dtype}> "
                                    "(CTA pairs)" if w.D == 256 else
                                    f"fattn_fwd_kernel<D={w.D}, non-causal, {w.dtype}>"),
                         "traffic": traffic},
            "cpu_baseline": cpu,
            "e2e": {"value": e2e_value, "unit": UNIT, "h2d_bytes_per_step": h2d,
                    "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                    "schedule": E2E_SCHEDULE,
                    "h2d_gbs_alone": h2d_gbs, "d2h_gbs_alone": d2h_gbs,
                    "copy_floor_ms": max(h2d / h2d_gbs, d2h / d2h_gbs) / 1e6,
                    "h2d_and_d2h_together_ms": both_ms,
                    "host_placement": placement,
                    "serial": {"value": world * flops_step / (e2e_serial_ms * 1e-3) / 1e12,
                               "ms_per_step": e2e_serial_ms}},
            "gpu_launches": args.steps * len(MASKS),
            "clocks": clocks,
        }
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


# The sources each kernel is built from: a stored ncu traffic figure counts
# only while these files are unchanged.
KERNEL_SOURCES = {
    "fattn_fwd": ["fattn_kernel.cuh", "fattn_launch.cuh", "fattn_fwd_d64.cu",
                  "fattn_fwd_d128.cu", "ptx.cuh", "fattn_status.h"],
    "fattn_pair": ["fattn_kernel_pair.cuh", "fattn_kernel.cuh", "fattn_launch.cuh",
                   "fattn_fwd_d256.cu", "ptx.cuh", "fattn_status.h"],
    "fattn_fwd_fp8": ["fattn_kernel.cuh", "fattn_launch.cuh", "fattn_fwd_fp8.cu",
                      "ptx.cuh", "fattn_status.h"],
    "fattn_decode": ["fattn_decode.cuh", "fattn_decode_mma.cuh", "fattn_decode_launch.h",
                     "fattn_decode.cu", "fattn_decode_d64.cu", "fattn_decode_d128.cu",
                     "ptx.cuh", "fattn_status.h"],
}


def kernel_source_hash(kernel: str = "fattn_fwd") -> str:
    """Hash of the CUDA sources of one kernel family; ties a stored ncu
    traffic figure to the kernel it was measured on."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "exact_attention_forward_10_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(key: str = "fattn_fwd_noncausal_bf16_d128", kernel: str = "fattn_fwd"):
    """DRAM bytes (read + write) per launch of a kernel from the committed ncu
    summary; None when there is none for the current sources."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f).get(key)
    if not d or d.get("kernel_source_hash") != kernel_source_hash(kernel):
        return None
    return d.get("bytes_per_launch")


def cpu_baseline(x, w, keep: bool = False):
    """The oracle timed on a bounded row sample of the workload (about 15 s
    of host work); with ``keep`` also its results for those rows (mask ->
    (rows, O rows, LSE rows)), for the comparison with the GPU's."""
    rows = calibrate_rows(x, w, target_s=15.0)
    dt, fl, threads, outs = cpu_oracle_run(x, w, rows, 4242, keep=True)
    line = {"value": fl / dt / 1e12, "unit": UNIT, "cores": threads,
            "kind": "oracle",
            "sample": f"{rows} sampled query rows per mask of {w.name} "
                      f"({dt:.1f} s); metric FLOPs of those rows / wall time"}
    return (line, outs) if keep else line


def oracle_parity(torch, outs_dev, oracle_outs, dtype: str) -> dict:
    """The GPU's rows (device outputs per mask) against the oracle's rows:
    one parity block over both masks, and each mask's."""
    per = {}
    for causal, (rows, ro, rl) in oracle_outs.items():
        go, gl = gather_rows(torch, *outs_dev[causal], rows)
        per["causal" if causal else "noncausal"] = parity_stats(go, gl, ro, rl, dtype)
    out = merge_parity(per.values())
    out["per_mask"] = per
    out["rows_from"] = "the cpu_baseline sample (seeded rows over every batch and head)"
    return out


# The configurations reported one by one beside the step: the small and
# LLM-layer shapes, the Q,K x4 stress set of the step's shape, and head dim
# 64 at the step's sequence length (from the sweep, both 16-bit types).
PER_CONFIG = (("1", "tiny"), ("2", "s2048_d64"), ("3", "s2048_d128"),
              ("4 Q,K x4", "s8192_d128_x4"),
              ("5 S8192 D64 fp16", "sweep_S8192_D64_fp16"),
              ("5 S8192 D64 bf16", "sweep_S8192_D64_bf16"))


def per_config_workloads():
    sweep = {w.name: w for w in attn_inputs.sweep_workloads()}
    return [(label, attn_inputs.WORKLOADS.get(key) or sweep[key]) for label, key in PER_CONFIG]


def time_launches(torch, dev, stream, launch, warmup: int = 10, reps: int = 20) -> float:
    """Median milliseconds of ``launch()`` over ``reps`` calls, each timed with
    CUDA events on ``stream``, after ``warmup`` calls."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            launch()
    torch.cuda.synchronize(dev)
    ev = []
    for _ in range(reps):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            launch()
            b.record(stream)
        ev.append((a, b))
    torch.cuda.synchronize(dev)
    return statistics.median(a.elapsed_time(b) for a, b in ev)


def run_per_config(torch, fattn, dev, stream, peaks, main_x=None, main_w=None):
    """Times each configuration of PER_CONFIG (every mask it runs) on its
    seeded input set; returns the records and, per record, what the oracle
    comparison needs (the host inputs, the mask and the GPU's rows of every
    batch and head)."""
    recs, keep = [], []
    for label, w in per_config_workloads():
        if (w.qk_mult != 1.0 and main_w is not None and main_x is not None
                and (w.B, w.H, w.S, w.D, w.dtype, w.seed) ==
                (main_w.B, main_w.H, main_w.S, main_w.D, main_w.dtype, main_w.seed)):
            m = np.float32(w.qk_mult)  # a power of two: exact in 16 bits
            x = attn_inputs.QKV(q=main_x.q * m, k=main_x.k * m, v=main_x.v,
                                dtype=w.dtype, seed=w.seed, qk_mult=w.qk_mult)
        else:
            x = w.inputs()
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
        code = fattn.FATTN_BF16 if w.dtype == "bf16" else fattn.FATTN_FP16
        q, k, v = (torch.from_numpy(a).to(dev).to(tdt) for a in (x.q, x.k, x.v))
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
        rows = (np.arange(w.B * w.H * w.S, dtype=np.int64) if w.B * w.H * w.S <= 4096
                else head_rows(w.B, w.H, w.S, seed=w.seed + 7000))
        stream.wait_stream(torch.cuda.current_stream(dev))  # the inputs' conversion
        for causal in w.causal:
            def launch():
                rc = fattn.fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), w.B, w.H, w.S, w.D, causal, w.scale,
                                     code, stream.cuda_stream)
                if rc != 0:
                    raise fattn.FattnError(rc)
            ms = time_launches(torch, dev, stream, launch)
            rc, where = fattn.fattn_last_error(stream.cuda_stream)
            if rc != 0:
                raise RuntimeError(f"kernel status {rc} at {where}")
            tf = metric_flops(w.B, w.H, w.S, w.D, causal) / (ms * 1e-3) / 1e12
            recs.append({"config": label, "workload": w.name, "B": w.B, "H": w.H, "S": w.S,
                         "D": w.D, "dtype": w.dtype, "causal": causal, "seed": w.seed,
                         "qk_mult": w.qk_mult, "ms_median": ms, "tflops": tf,
                         "frac_of_measured_burst": tf / peaks["burst"],
                         "hbm_gbs": algo_bytes(w.B, w.H, w.S, w.D) / (ms * 1e-3) / 1e9,
                         "parity": None})
            go, gl = gather_rows(torch, o, lse, rows)
            keep.append((len(recs) - 1, w, x, causal, rows, go, gl))
        del q, k, v, o, lse
    return recs, keep


def per_config_parity(recs, keep) -> None:
    """The oracle on each kept row set; fills each record's parity block."""
    import oracle
    threads = oracle.default_threads()
    for i, w, x, causal, rows, go, gl in keep:
        t0 = time.perf_counter()
        ro, rl = oracle.attn_fwd(x.q, x.k, x.v, causal, w.scale, rows=rows, threads=threads)
        par = parity_stats(go, gl, ro, rl, w.dtype)
        par["oracle_s"] = time.perf_counter() - t0
        par["rows_from"] = ("every row" if len(rows) == w.B * w.H * w.S else
                            "every batch and head: first and last 16 rows and 8 seeded others")
        recs[i]["parity"] = par


SWEEP_CSV_FIELDS = ("seqlen", "headdim", "dtype", "causal", "ms_median", "tflops",
                    "frac_of_measured_peak", "hbm_gbs")


def write_sweep_csv(path: str, records) -> None:
    """The sweep as CSV, one row per (S, D, dtype, mask) point, in the
    columns of the sweep's JSON lines (S as seqlen, D as headdim)."""
    import csv
    with open(path, "w", newline="") as f:
        out = csv.writer(f)
        out.writerow(SWEEP_CSV_FIELDS)
        for r in records:
            out.writerow([r["S"], r["D"], r["dtype"], int(bool(r["causal"])),
                          f"{r['ms_median']:.6f}", f"{r['tflops']:.3f}",
                          f"{r['frac_of_measured_peak']:.4f}", f"{r.get('hbm_gbs', 0.0):.1f}"])


def run_sweep(args):
    """Attention TFLOPS over the sweep shapes (B2 H16; S 512 .. 16384 and
    4097; D 64, 128; fp16, bf16; both masks): one JSON line per point, and
    with ``--csv PATH`` the same points as CSV.
    Each point runs on its seeded input set (seed 4 + index, the sets the
    parity tests compare with the oracle); generating them on the host takes
    most of the sweep's wall time.  Points whose inputs are smaller than L2
    are timed after an L2 flush outside each launch's events."""
    import torch

    import exact_attention_forward_10_gb300 as fattn

    dev = torch.device("cuda", torch.cuda.current_device())
    peaks = load_peaks()
    stream = torch.cuda.Stream(dev)
    dims = [int(d) for d in args.dims.split(",")]
    shapes = [w for w in attn_inputs.sweep_workloads() if w.D in dims]
    if 256 in dims:
        shapes += [attn_inputs.Workload(f"B2_H16_S{S}_D256_{dt}", 2, 16, S, 256, dt,
                                        (False, True), 100)
                   for S in attn_inputs.SWEEP_S for dt in attn_inputs.DTYPES]
    records = []
    for w in shapes:
        tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
        code = fattn.FATTN_BF16 if w.dtype == "bf16" else fattn.FATTN_FP16
        x = w.inputs()
        q, k, v = (torch.from_numpy(a).to(dev).to(tdt) for a in (x.q, x.k, x.v))
        del x
        o = torch.empty_like(q)
        lse = torch.empty((w.B, w.H, w.S), dtype=torch.float32, device=dev)
        stream.wait_stream(torch.cuda.current_stream(dev))  # the inputs' conversion
        for causal in w.causal:
            def launch():
                rc = fattn.fattn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                     lse.data_ptr(), w.B, w.H, w.S, w.D, causal, w.scale,
                                     code, stream.cuda_stream)
                if rc != 0:
                    raise fattn.FattnError(rc)
            with torch.cuda.stream(stream):
                for _ in range(args.warmup):
                    launch()
            torch.cuda.synchronize(dev)
            flush = l2_flush_buffer(torch, dev, 3 * 2 * w.B * w.H * w.S * w.D)
            times = []
            for _ in range(max(20, args.steps)):
                a = torch.cuda.Event(enable_timing=True)
                b = torch.cuda.Event(enable_timing=True)
                with torch.cuda.stream(stream):
                    if flush is not None:
                        flush.add_(1)
                    a.record(stream)
                    launch()
                    b.record(stream)
                times.append((a, b))
            del flush
            torch.cuda.synchronize(dev)
            ms = statistics.median(x.elapsed_time(y) for x, y in times)
            rc, where = fattn.fattn_last_error(stream.cuda_stream)
            if rc != 0:
                raise RuntimeError(f"kernel status {rc} at {where}")
            tf = metric_flops(w.B, w.H, w.S, w.D, causal) / (ms * 1e-3) / 1e12
            rec = {"S": w.S, "D": w.D, "dtype": w.dtype, "causal": causal, "seed": w.seed,
                   "ms_median": ms, "tflops": tf,
                   "frac_of_measured_peak": tf / peaks["burst"],
                   "hbm_gbs": algo_bytes(w.B, w.H, w.S, w.D) / (ms * 1e-3) / 1e9}
            records.append(rec)
            print(json.dumps(rec), flush=True)
    if args.csv:
        write_sweep_csv(args.csv, records)
    return 0


# ------------------------------------------------------ E4M3 (FP8) inputs

def run_fp8(args):
    """One step = the non-causal and the causal FP8 forward of the benchmark
    shape (B2 H16 S8192 D128; Q, K, V the seed-3 normals quantised to E4M3
    per tensor), bf16 output, inputs resident in HBM."""
    import torch

    import exact_attention_forward_10_gb300 as fattn

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    w = WORKLOAD
    x = attn_inputs.make_qkv_fp8(w.B, w.H, w.S, w.D, w.seed)
    host = [torch.from_numpy(a).pin_memory() for a in (x.q8, x.k8, x.v8)]
    q, k, v = (h.to(dev) for h in host)
    B, H, S, D = w.B, w.H, w.S, w.D
    outs = {c: (torch.empty((B, H, S, D), dtype=torch.bfloat16, device=dev),
                torch.empty((B, H, S), dtype=torch.float32, device=dev)) for c in MASKS}
    stream = torch.cuda.Stream(dev)
    # the launch stream does not wait for the default stream by itself
    stream.wait_stream(torch.cuda.current_stream(dev))
    sptr = stream.cuda_stream
    qs, ks, vs = x.descale

    def launch(causal, qq, kk, vv, into=None):
        o, l = (into or outs)[causal]
        rc = fattn.fattn_fwd_fp8(qq.data_ptr(), kk.data_ptr(), vv.data_ptr(), o.data_ptr(),
                                 l.data_ptr(), B, H, S, D, causal, w.scale, qs, ks, vs,
                                 fattn.FATTN_BF16, sptr)
        if rc != 0:
            raise fattn.FattnError(rc, "fattn_fwd_fp8")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        for c in MASKS:
            launch(c, q, k, v)
        for _ in range(args.warmup):
            for c in MASKS:
                launch(c, q, k, v)
    rc, where = fattn.fattn_last_error(sptr)
    if rc != 0:
        raise RuntimeError(f"kernel status {rc} at {where}")
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps * len(MASKS))]
    flush = l2_flush_buffer(torch, dev, 3 * B * H * S * D)  # one-byte inputs
    sampler = clock_sampler(dev)
    sampler.start()
    time.sleep(0.05)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        e = 0
        for _ in range(args.steps):
            for c in MASKS:
                if flush is not None:
                    flush.add_(1)
                ev[e][0].record(stream)
                launch(c, q, k, v)
                ev[e][1].record(stream)
                e += 1
        t1.record(stream)
    barrier()
    clocks = sampler.stop()
    rc, where = fattn.fattn_last_error(sptr)
    if rc != 0:
        raise RuntimeError(f"kernel status {rc} at {where}")
    per_launch = {c: [] for c in MASKS}
    for i, (a, b) in enumerate(ev):
        per_launch[MASKS[i % len(MASKS)]].append(a.elapsed_time(b))
    step_ms = t0.elapsed_time(t1) / args.steps
    if flush is not None:  # the flushes are not part of the step
        step_ms = sum(a.elapsed_time(b) for a, b in ev) / args.steps

    h_outs = {c: (torch.empty((B, H, S, D), dtype=torch.bfloat16).pin_memory(),
                  torch.empty((B, H, S), dtype=torch.float32).pin_memory()) for c in MASKS}

    def e2e_step():
        qq, kk, vv = (h.to(dev, non_blocking=True) for h in host)
        for c in MASKS:
            launch(c, qq, kk, vv)
        for c in MASKS:
            h_outs[c][0].copy_(outs[c][0], non_blocking=True)
            h_outs[c][1].copy_(outs[c][1], non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
    barrier()
    n_e2e = max(3, min(args.steps, 20))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(n_e2e):
            e2e_step()
        e1.record(stream)
    barrier()
    e2e_serial_ms = e0.elapsed_time(e1) / n_e2e
    e2e_ms = pipelined_e2e_ms(
        torch, dev, stream, host,
        lambda din, dout: [launch(c, *din, into=dout) for c in MASKS],
        lambda: {c: (torch.empty((B, H, S, D), dtype=torch.bfloat16, device=dev),
                     torch.empty((B, H, S), dtype=torch.float32, device=dev)) for c in MASKS},
        h_outs, n_e2e, barrier)
    from exact_attention_forward_10_gb300 import shard
    step_ms, e2e_ms, e2e_serial_ms = shard.max_over_ranks([step_ms, e2e_ms, e2e_serial_ms],
                                                          device=dev)
    flops_step = sum(metric_flops(B, H, S, D, c) for c in MASKS)
    peaks = load_peaks()
    peak8 = 2.0 * peaks["burst"]
    per_mask = {}
    for c in MASKS:
        ms = statistics.median(per_launch[c])
        tf = metric_flops(B, H, S, D, c) / (ms * 1e-3) / 1e12
        per_mask["causal" if c else "noncausal"] = {"ms_median": ms, "tflops": tf,
                                                     "frac_of_fp8_peak": tf / peak8}
    achieved = metric_flops(B, H, S, D, False) / (statistics.mean(per_launch[False]) * 1e-3) / 1e12
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = cpu_baseline(x, w)
        print(json.dumps({
            "metric": METRIC + " (E4M3 inputs, against the FP8 peak)",
            "value": world * flops_step / (step_ms * 1e-3) / 1e12, "unit": UNIT,
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic",
            "config": workload_config(w, {"inputs": "E4M3 codes, per-tensor power-of-two "
                                                    "scales", "output": "bf16",
                                          "parallelism": f"replicas x{world}"},
                                      elem_bytes=1),
            "per_mask": per_mask,
            # E4M3 Q, K, V (1 byte each) read once, bf16 O and fp32 LSE written once
            "hbm_gbs": world * len(MASKS) * B * H * S * (5 * D + 4) / (step_ms * 1e-3) / 1e9,
            "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak8,
                         "unit": "TFLOP/s", "frac": achieved / peak8,
                         "peak_kind": (f"fp8 dense, assumed: 2 x the {peaks['source']} bf16 "
                                       "burst (the nominal fp8/bf16 ratio 4.5/2.25; no fp8 "
                                       "peak is measured)"),
                         "kernel": "fattn_fwd_kernel<D=128, non-causal, E4M3 in, bf16 out>",
                         "traffic": load_traffic(f"fattn_fwd_noncausal_e4m3_d128_s{S}",
                                                 "fattn_fwd_fp8")},
            "cpu_baseline": cpu,
            "e2e": {"value": world * flops_step / (e2e_ms * 1e-3) / 1e12, "unit": UNIT,
                    "h2d_bytes_per_step": sum(h.numel() for h in host),
                    "d2h_bytes_per_step": sum(o.numel() * 2 + l.numel() * 4
                                              for o, l in h_outs.values()),
                    "ms_per_step": e2e_ms, "schedule": E2E_SCHEDULE,
                    "serial": {"value": world * flops_step / (e2e_serial_ms * 1e-3) / 1e12,
                               "ms_per_step": e2e_serial_ms}},
            "gpu_launches": args.steps * len(MASKS),
            "clocks": clocks}), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


# ------------------------------------------- attention against a KV cache

KV_METRIC = ("decode attention against a KV cache: effective HBM GB/s "
             "(cached K/V rows read + Q + O + LSE bytes / time)")


def kv_bytes(w, lens) -> int:
    """Algorithmic bytes of one call: every cached K and V row inside a
    batch's length read once, Q read, O and the fp32 LSE written once."""
    rows = int(np.sum(lens)) if lens is not None else w.B * w.Sk
    return (rows * w.H * w.D * 2 * 2 + 2 * w.B * w.H * w.Sq * w.D * 2
            + w.B * w.H * w.Sq * 4)


def kv_config(w, cached_lens, extra=None) -> dict:
    lens = (f"cached lengths uniform in [{w.lens_range[0]}, {w.lens_range[1]}] "
            f"(seed {w.seed})" if w.lens_range else f"every length {w.Sk}")
    c = {"workload": f"{w.name}: Q/K/V iid N(0,1) seed {w.seed}, {lens}, "
                     f"{'causal' if w.causal else 'non-causal'}, scale 1/sqrt(D)",
         "B": w.B, "H": w.H, "Sq": w.Sq, "Sk": w.Sk, "D": w.D,
         "l2": l2_label(kv_bytes(w, cached_lens), "bytes read per call")}
    if extra:
        c.update(extra)
    return c


def kv_oracle_run(x, w, batches: int, seed: int):
    """The cache oracle on ``batches`` sampled batch entries (all their heads,
    their cached prefix only); returns (seconds, algorithmic bytes of those
    entries, threads)."""
    import oracle
    threads = oracle.default_threads()
    rng = np.random.default_rng(seed)
    pick = rng.choice(w.B, size=min(batches, w.B), replace=False)
    byts = 0
    t0 = time.perf_counter()
    for b in pick.tolist():
        n = int(x.lens[b]) if x.lens is not None else w.Sk
        top = max(1, n)
        oracle.attn_kvcache(x.q[b:b + 1], x.k[b:b + 1, :, :top], x.v[b:b + 1, :, :top],
                            w.causal, w.scale, [n], threads=threads)
        byts += w.H * (n * w.D * 2 * 2 + 2 * w.Sq * w.D * 2 + w.Sq * 4)
    return time.perf_counter() - t0, byts, threads


def kv_calibrate(x, w, target_s: float) -> int:
    """Batch entries per oracle sample so that it takes about ``target_s``
    (at most every entry)."""
    n = 1
    dt, _, _ = kv_oracle_run(x, w, n, 999)
    while dt < 0.5 and n < w.B:
        n = min(w.B, n * 4)
        dt, _, _ = kv_oracle_run(x, w, n, 999)
    return max(1, min(w.B, int(n * target_s / max(dt, 1e-6))))


def kv_cpu_baseline(x, w, target_s: float = 10.0) -> dict:
    nb = kv_calibrate(x, w, target_s)
    dt, byts, threads = kv_oracle_run(x, w, nb, 4242)
    return {"value": byts / dt / 1e9, "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{nb} sampled batch entries (all {w.H} heads) of {w.name} "
                      f"({dt:.1f} s); algorithmic bytes of those entries / wall time"}


def run_kvcache_reference(args, w):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    x = w.inputs()
    nb = kv_calibrate(x, w, max(0.2, min(10.0, 90.0 / max(1, args.steps + args.warmup))))
    for i in range(args.warmup):
        kv_oracle_run(x, w, nb, 100 + i)
    tot_t, tot_b, threads = 0.0, 0, 1
    for i in range(args.steps):
        dt, b, threads = kv_oracle_run(x, w, nb, 1000 + i)
        tot_t += dt
        tot_b += b
    value = tot_b / tot_t / 1e9
    sample = f"{nb} sampled batch entries (all {w.H} heads) per step of {w.B}"
    print(json.dumps({
        "impl": "reference", "metric": KV_METRIC, "value": value, "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1000.0 * tot_t / max(1, args.steps), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": kv_config(w, x.lens, {"parallelism": "host cores, rank 0 only"}),
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": threads,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)
    return 0


def load_hbm_peak() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            return {"gbs": float(json.load(f)["hbm_gbs"]), "source": "measured"}
    return {"gbs": 6800.0, "source": "fallback"}


def run_kvcache(args, w):
    """One step = one fattn_fwd_kvcache call (split kernel + merge kernel) on
    the cache workload, inputs resident in HBM."""
    import torch

    import exact_attention_forward_10_gb300 as fattn

    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", torch.cuda.current_device())
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float16
    code = fattn.FATTN_BF16 if w.dtype == "bf16" else fattn.FATTN_FP16
    x = w.inputs()
    host = [torch.from_numpy(a).to(tdt).pin_memory() for a in (x.q, x.k, x.v)]
    h_lens = (torch.from_numpy(x.lens.astype(np.int32)).pin_memory()
              if x.lens is not None else None)
    q, k, v = (h.to(dev) for h in host)
    lens = h_lens.to(dev) if h_lens is not None else None
    B, H, Sq, Sk, D = w.B, w.H, w.Sq, w.Sk, w.D
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device=dev)
    plan = fattn.fattn_kvcache_plan(B, H, Sq, Sk, D)
    ws = torch.empty(plan["workspace_bytes"], dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    # the launch stream does not wait for the default stream by itself
    stream.wait_stream(torch.cuda.current_stream(dev))
    sptr = stream.cuda_stream

    def launch(qq, kk, vv, ll):
        rc = fattn.fattn_fwd_kvcache(
            qq.data_ptr(), kk.data_ptr(), vv.data_ptr(),
            ll.data_ptr() if ll is not None else 0, o.data_ptr(), lse.data_ptr(),
            B, H, Sq, Sk, D, w.causal, w.scale, code, ws.data_ptr(), ws.numel(), sptr)
        if rc != 0:
            raise fattn.FattnError(rc, "fattn_fwd_kvcache")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize(dev)

    with torch.cuda.stream(stream):
        launch(q, k, v, lens)
    rc, where = fattn.fattn_last_error(sptr)
    if rc != 0:
        raise RuntimeError(f"kernel status {rc} at {where}")
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            launch(q, k, v, lens)
    barrier()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(args.steps)]
    flush = l2_flush_buffer(torch, dev, kv_bytes(w, x.lens))
    sampler = clock_sampler(dev)
    sampler.start()
    time.sleep(0.05)
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        t0.record(stream)
        for a, b in ev:
            if flush is not None:
                flush.add_(1)
            a.record(stream)
            launch(q, k, v, lens)
            b.record(stream)
        t1.record(stream)
    barrier()
    clocks = sampler.stop()
    rc, where = fattn.fattn_last_error(sptr)
    if rc != 0:
        raise RuntimeError(f"kernel status {rc} at {where}")
    step_ms = t0.elapsed_time(t1) / args.steps
    call_ms = statistics.mean(a.elapsed_time(b) for a, b in ev)
    if flush is not None:  # the flushes are not part of the step
        step_ms = call_ms

    # end to end: the caches are the sequences' state, resident on the GPU
    # across steps (as in decoding, where each step's new keys and values are
    # appended on the device by the projection that made them); a step's
    # inputs are its new queries and the cached lengths, copied from pinned
    # host memory, then the call, then O and the LSE copied back
    h_o = torch.empty(o.shape, dtype=tdt).pin_memory()
    h_l = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    e2e_steps = max(3, min(args.steps, 20))

    def e2e_step():
        qq = host[0].to(dev, non_blocking=True)
        ll = h_lens.to(dev, non_blocking=True) if h_lens is not None else None
        launch(qq, k, v, ll)
        h_o.copy_(o, non_blocking=True)
        h_l.copy_(lse, non_blocking=True)

    with torch.cuda.stream(stream):
        e2e_step()
    barrier()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(e2e_steps):
            e2e_step()
        e1.record(stream)
    barrier()
    e2e_ms = e0.elapsed_time(e1) / e2e_steps
    h2d = host[0].numel() * host[0].element_size() + (
        h_lens.numel() * 4 if h_lens is not None else 0)
    d2h = h_o.numel() * h_o.element_size() + h_l.numel() * 4

    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([step_ms, e2e_ms], device=dev, dtype=torch.float64)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        step_ms, e2e_ms = float(t[0]), float(t[1])
    byts = kv_bytes(w, x.lens)
    value = world * byts / (step_ms * 1e-3) / 1e9
    peak = load_hbm_peak()
    achieved = byts / (call_ms * 1e-3) / 1e9
    if rank == 0:
        cpu = None
        if world == 1 and not args.no_cpu_baseline:
            cpu = kv_cpu_baseline(x, w)
        print(json.dumps({
            "metric": KV_METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": kv_config(w, x.lens, {"parallelism": f"replicas x{world}",
                                    "grid": plan["grid"], "block": plan["block"],
                                    "split_warps": plan["split_warps"],
                                    "bytes_per_call": byts}),
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak["gbs"],
                         "unit": "GB/s", "frac": achieved / peak["gbs"],
                         "peak_kind": f"HBM copy, {peak['source']}",
                         "kernel": ("fattn_decode_kernel" if w.Sq == 1 else "fattn_decode_mma_kernel")
                                   + " + merge (one call, both launches inside the timed span)",
                         "traffic": load_traffic(f"fattn_decode_{w.dtype}_d{w.D}_sq{w.Sq}_"
                                                 f"{args.kvcache}", "fattn_decode")},
            "cpu_baseline": cpu,
            "e2e": {"value": world * byts / (e2e_ms * 1e-3) / 1e9, "unit": "GB/s",
                    "inputs": "the step's new queries and the cached lengths from the host; "
                              "the K/V caches stay resident on the GPU across steps",
                    "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "ms_per_step": e2e_ms},
            "gpu_launches": 2 * args.steps,
            "clocks": clocks}), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="fattn", choices=["fattn", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-configuration block (e.g. for a profiler run)")
    ap.add_argument("--sweep", action="store_true",
                    help="TFLOPS over the sweep shapes, one JSON line each")
    ap.add_argument("--shape", default=None,
                    help="S,D,dtype (B2 H16) to use as the step workload instead of "
                         "B2 H16 S8192 D128 bf16, e.g. 8192,64,bf16 or 8192,256,bf16 "
                         "(sweep shapes keep their seeds; others use seed 100)")
    ap.add_argument("--csv", default=None, metavar="PATH",
                    help="with --sweep: also write the points to PATH as CSV")
    ap.add_argument("--dims", default="64,128",
                    help="head dims of --sweep (64,128 are the sweep's; 256 adds the "
                         "CTA-pair kernel)")
    ap.add_argument("--fp8", action="store_true",
                    help="time the E4M3-input forward on the step workload (D=128)")
    ap.add_argument("--kvcache", nargs="?", const="decode_b16_h16_d128_ragged",
                    default=None, choices=sorted(attn_inputs.CACHE_WORKLOADS),
                    help="time attention of new queries against a KV cache "
                         "(effective HBM GB/s) on this cache workload")
    args = ap.parse_args()
    if args.kvcache:
        if args.warmup < 3:
            args.warmup = 3
        w = attn_inputs.CACHE_WORKLOADS[args.kvcache]
        if args.impl == "reference":
            return run_kvcache_reference(args, w)
        return run_kvcache(args, w)
    if args.shape:
        S, D, dt = args.shape.split(",")
        picks = [w for w in attn_inputs.sweep_workloads()
                 if (w.S, w.D, w.dtype) == (int(S), int(D), dt)]
        if not picks:
            if dt not in attn_inputs.DTYPES or int(D) not in (64, 128, 256):
                ap.error(f"bad shape {args.shape}")
            # a shape outside the sweep (e.g. head dim 256): B2 H16, seed 100
            picks = [attn_inputs.Workload(f"B2_H16_S{S}_D{D}_{dt}", 2, 16, int(S), int(D),
                                          dt, (False, True), 100)]
        global WORKLOAD
        WORKLOAD = picks[0]
    if args.warmup < 3:
        args.warmup = 3
    if args.sweep:
        return run_sweep(args)
    if args.fp8:
        if WORKLOAD.D != 128:
            ap.error("--fp8 needs head dim 128")
        return run_fp8(args)
    if args.impl == "reference":
        return run_reference(args)
    return run_fattn(args)


if __name__ == "__main__":
    sys.exit(main())
