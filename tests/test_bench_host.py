"""Host-side logic of ``bench.py``, on the CPU: the metric's FLOP count and
the cache path's algorithmic bytes, the rule that a stored ncu traffic
figure is used only for the kernel sources it was measured on, the peaks
file, the JSON line of the reference arm (the fp64 oracle on the host
cores), which prints on rank 0 only, and the sweep's CSV."""
from __future__ import annotations

import argparse
import csv
import io
import json
import os
from contextlib import redirect_stdout

import numpy as np
import pytest

import attn_inputs
import bench

MEASURED_PEAKS = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))),
                              "MEASURED_PEAKS.json")


def test_metric_flops_of_the_benchmark_workload():
    """4·B·H·S²·D, half when causal: 1.0995 / 0.5498 TFLOP at B2 H16 S8192 D128."""
    assert bench.metric_flops(2, 16, 8192, 128, False) == 4 * 2 * 16 * 8192**2 * 128
    assert bench.metric_flops(2, 16, 8192, 128, False) == pytest.approx(1.0995e12, rel=1e-4)
    assert bench.metric_flops(2, 16, 8192, 128, True) == bench.metric_flops(2, 16, 8192, 128, False) / 2


@pytest.mark.parametrize("causal", [False, True])
def test_row_flops_sum_to_the_metric(causal):
    """The reference arm counts FLOPs per sampled row; over every row of the
    workload they add up to the metric exactly."""
    B, H, S, D = 2, 16, 8192, 128
    assert B * H * S * bench.row_flops(S, D, causal) == bench.metric_flops(B, H, S, D, causal)


def test_cache_bytes():
    """Cached K and V rows inside each length read once (2 bytes per value),
    Q read and O written once, the fp32 LSE written once."""
    w = attn_inputs.CacheWorkload("t", 3, 4, 2, 100, 64, "fp16", True, 1, (1, 100))
    lens = np.array([10, 0, 100])
    kv = 110 * 4 * 64 * 2 * 2
    q_o = 2 * 3 * 4 * 2 * 64 * 2
    assert bench.kv_bytes(w, lens) == kv + q_o + 3 * 4 * 2 * 4
    # without lengths every cache is full
    assert bench.kv_bytes(w, None) == 3 * 100 * 4 * 64 * 4 + q_o + 3 * 4 * 2 * 4


def test_traffic_is_used_only_for_the_sources_it_was_measured_on(tmp_path, monkeypatch):
    (tmp_path / "profiles").mkdir()
    (tmp_path / "profiles" / "traffic.json").write_text(json.dumps({
        "current": {"bytes_per_launch": 123, "kernel_source_hash": "aaaa"},
        "stale": {"bytes_per_launch": 456, "kernel_source_hash": "bbbb"}}))
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    monkeypatch.setattr(bench, "kernel_source_hash", lambda kernel="fattn_fwd": "aaaa")
    assert bench.load_traffic("current") == 123
    assert bench.load_traffic("stale") is None
    assert bench.load_traffic("absent") is None
    (tmp_path / "profiles" / "traffic.json").unlink()
    assert bench.load_traffic("current") is None


def test_source_hash_covers_every_listed_source():
    """Each kernel family's hash reads files that exist, and differs between
    families with different sources."""
    csrc = os.path.join(bench.ROOT, "exact_attention_forward_10_gb300", "csrc")
    for kernel, names in bench.KERNEL_SOURCES.items():
        for n in names:
            assert os.path.exists(os.path.join(csrc, n)), (kernel, n)
    hashes = {k: bench.kernel_source_hash(k) for k in bench.KERNEL_SOURCES}
    assert len(set(hashes.values())) == len(hashes)


def test_peaks_come_from_the_measured_file():
    p = bench.load_peaks()
    if os.path.exists(MEASURED_PEAKS):
        with open(MEASURED_PEAKS) as f:
            d = json.load(f)
        assert p["source"] == "measured" and p["burst"] == float(d["bf16_tflops"])
        assert bench.load_hbm_peak()["gbs"] == float(d["hbm_gbs"])
    else:
        assert p["source"] == "fallback"


def _args(steps, warmup):
    return argparse.Namespace(steps=steps, warmup=warmup)


def _run(fn, *a):
    out = io.StringIO()
    with redirect_stdout(out):
        rc = fn(*a)
    return rc, out.getvalue()


def _check_reference_line(d, steps, unit):
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == steps and d["unit"] == unit
    assert d["higher_is_better"] is True and d["data"] == "synthetic"
    assert d["dtype"] == "f64" and d["vs_baseline"] is None
    assert d["value"] > 0 and d["ms_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"]
    assert cb["unit"] == unit and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == unit
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0
    assert d["config"]["workload"]


def test_reference_arm_line(monkeypatch):
    """The self-attention reference arm on the tiny workload, the sample
    size fixed (calibration only sizes it)."""
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    monkeypatch.setattr(bench, "WORKLOAD", attn_inputs.WORKLOADS["tiny"])
    monkeypatch.setattr(bench, "calibrate_rows", lambda x, w, target_s: 32)
    rc, out = _run(bench.run_reference, _args(2, 1))
    assert rc == 0
    lines = [l for l in out.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    _check_reference_line(d, 2, bench.UNIT)
    assert d["metric"] == bench.METRIC
    assert "32 sampled query rows" in d["cpu_baseline"]["sample"]


def test_cache_reference_arm_line(monkeypatch):
    monkeypatch.delenv("RANK", raising=False)
    monkeypatch.delenv("WORLD_SIZE", raising=False)
    w = attn_inputs.CacheWorkload("tiny_cache", 3, 2, 2, 96, 64, "fp16", True, 7, (0, 96))
    monkeypatch.setattr(bench, "kv_calibrate", lambda x, w, target_s: 2)
    rc, out = _run(bench.run_kvcache_reference, _args(2, 1), w)
    assert rc == 0
    d = json.loads(out.strip())
    _check_reference_line(d, 2, "GB/s")
    assert d["metric"] == bench.KV_METRIC


def test_reference_arm_prints_on_rank_zero_only(monkeypatch):
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(bench, "WORKLOAD", attn_inputs.WORKLOADS["tiny"])
    monkeypatch.setattr(bench, "calibrate_rows", lambda x, w, target_s: 32)
    rc, out = _run(bench.run_reference, _args(1, 0))
    assert rc == 0 and out == ""


def test_sweep_csv(tmp_path):
    recs = [{"S": 512, "D": 64, "dtype": "fp16", "causal": False, "ms_median": 0.0184,
             "tflops": 116.9, "frac_of_measured_peak": 0.0613},
            {"S": 4097, "D": 128, "dtype": "bf16", "causal": True, "ms_median": 0.4,
             "tflops": 1010.0, "frac_of_measured_peak": 0.53}]
    path = tmp_path / "sweep.csv"
    bench.write_sweep_csv(str(path), recs)
    with open(path, newline="") as f:
        rows = list(csv.reader(f))
    assert tuple(rows[0]) == bench.SWEEP_CSV_FIELDS
    assert rows[1][:4] == ["512", "64", "fp16", "0"]
    assert rows[2][:4] == ["4097", "128", "bf16", "1"]
    assert float(rows[2][5]) == 1010.0 and float(rows[1][4]) == pytest.approx(0.0184)


def test_algorithmic_bytes():
    # Q, K, V read once, O written once (16 bits each) and the fp32 LSE
    assert bench.algo_bytes(2, 16, 8192, 128) == 2 * 16 * 8192 * (3 * 2 * 128 + 2 * 128 + 4)
    assert bench.algo_bytes(1, 1, 1, 64) == 8 * 64 + 4


def test_parity_stats_flat_and_ulp_allowance():
    ro = np.array([[0.5, 5.0], [-6.0, 1.0]])
    rl = np.array([1.0, 2.0])
    # bf16 at |x| in [4, 8): half an ulp is 2^-6; error 0.02 passes only with it
    o = ro + np.array([[0.0, 0.02], [0.0, 0.0]])
    st = bench.parity_stats(o, rl, ro, rl, "bf16")
    assert st["pass"] and not st["flat_pass"] and st["n_pass_by_ulp_allowance"] == 1
    assert st["max_abs_dO"] == pytest.approx(0.02)
    # the same error where |O_ref| < 4 fails
    o2 = ro + np.array([[0.02, 0.0], [0.0, 0.0]])
    assert not bench.parity_stats(o2, rl, ro, rl, "bf16")["pass"]
    # LSE outside 1e-3 fails; a NaN fails
    assert not bench.parity_stats(ro, rl + 2e-3, ro, rl, "fp16")["pass"]
    bad = ro.copy()
    bad[0, 0] = np.nan
    assert not bench.parity_stats(bad, rl, ro, rl, "fp16")["pass"]
    both = bench.merge_parity([st, bench.parity_stats(ro, rl, ro, rl, "bf16")])
    assert both["pass"] and both["rows"] == 4 and both["n_pass_by_ulp_allowance"] == 1


def test_head_rows_cover_every_head():
    B, H, S = 2, 16, 8192
    rows = bench.head_rows(B, H, S, seed=1)
    heads = rows // S
    assert sorted(set(heads.tolist())) == list(range(B * H))
    assert len(rows) == B * H * (16 + 8 + 16) and len(set(rows.tolist())) == len(rows)
    r0 = rows[heads == 0] % S
    assert set(range(16)) <= set(r0.tolist()) and set(range(S - 16, S)) <= set(r0.tolist())
    small = bench.head_rows(1, 2, 20, seed=1)
    assert len(small) == 40


def test_per_config_workloads_are_the_named_sets():
    got = {label: w for label, w in bench.per_config_workloads()}
    assert (got["1"].S, got["1"].D, got["1"].dtype, got["1"].seed) == (128, 64, "fp16", 0)
    assert (got["2"].B, got["2"].H, got["2"].S, got["2"].D, got["2"].seed) == (2, 16, 2048, 64, 1)
    assert (got["3"].B, got["3"].H, got["3"].S, got["3"].D, got["3"].seed) == (1, 32, 2048, 128, 2)
    assert got["4 Q,K x4"].qk_mult == 4.0 and got["4 Q,K x4"].seed == 3
    for dt in ("fp16", "bf16"):
        w = got[f"5 S8192 D64 {dt}"]
        assert (w.S, w.D, w.dtype) == (8192, 64, dt) and w.causal == (False, True)


def test_l2_policy_flushes_working_sets_under_l2():
    """Timed launches whose inputs fit in L2 are preceded by a flush; the
    label says which, and the benchmark workload's inputs are larger."""
    small = bench.l2_label(96 * 2**20)
    big = bench.l2_label(192 * 2**20)
    assert "flushed" in small and "smaller than L2" in small
    assert "larger than L2" in big and "no flush" in big
    # the cache workload of B8 H16 Sq4 D64 reads ~126 MB a call: under L2
    w = attn_inputs.CACHE_WORKLOADS["decode_b8_h16_sq4_d64"]
    lens = attn_inputs.cache_lengths(w.seed, w.B, *w.lens_range)
    assert bench.kv_bytes(w, lens) < bench.L2_BYTES
    assert "flushed" in bench.kv_config(w, lens)["l2"]
