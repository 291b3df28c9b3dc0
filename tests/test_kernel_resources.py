"""Resource use of every kernel, from the assembler's report (nvcc -Xptxas -v)
on the CPU: each expected instantiation is built, none spills registers to
local memory, and each kernel's registers fit its launch (threads x
registers within the SM's 65,536).  A change that adds spills, or a launch
that could no longer be resident, fails here before any GPU time is spent."""
from __future__ import annotations

import concurrent.futures
import os
import re
import shutil
import subprocess

import pytest

from exact_attention_forward_10_gb300 import build as fbuild

UNITS = ["fattn_fwd_d64.cu", "fattn_fwd_d128.cu", "fattn_fwd_d256.cu", "fattn_fwd_fp8.cu",
         "fattn_decode_d64.cu", "fattn_decode_d128.cu", "fattn_api.cu"]

# threads per CTA of each kernel family (from the launch code)
THREADS = {
    "fattn_fwd_kernel": 512,          # 16 warps, two query tiles
    "fattn_fwd_pair_kernel": 384,     # 12 warps per CTA of the pair
    "fattn_decode_mma_kernel": 256,   # at most 8 warps
    "fattn_decode_kernel": 384,       # at most 12 warps
    "fattn_decode_combine_kernel": 256,
    "wait_check_kernel": 32,
}

# instantiations expected: self-attention 2 masks x 2 dtypes for D = 64,
# 128 and E4M3 (2 output dtypes); pairs for D = 256; cache kernels for
# D = 64, 128 x 2 dtypes
EXPECTED = {
    "fattn_fwd_kernel": 12,
    "fattn_fwd_pair_kernel": 4,
    "fattn_decode_mma_kernel": 4,
    "fattn_decode_kernel": 4,
    "fattn_decode_combine_kernel": 4,
    "wait_check_kernel": 1,
}



def _family(mangled: str) -> str:
    for name in sorted(THREADS, key=len, reverse=True):
        if re.search(rf"\d{name}", mangled):
            return name
    raise AssertionError(f"unknown kernel {mangled}")


def _report(src: str, out_dir: str) -> list[dict]:
    obj = os.path.join(out_dir, src + ".o")
    cmd = [fbuild.nvcc(), *fbuild.ARCH, "-O3", "-std=c++17", "-Xptxas", "-v",
           "-I", fbuild.INCLUDE, "-c", os.path.join(fbuild.CSRC, src), "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    kernels, cur = [], None
    for line in r.stderr.splitlines():
        m = re.search(r"Compiling entry function '([^']+)'", line)
        if m:
            cur = {"name": m.group(1), "unit": src}
            kernels.append(cur)
            continue
        if cur is None:
            continue
        m = re.search(r"(\d+) bytes spill stores, (\d+) bytes spill loads", line)
        if m:
            cur["spill_st"], cur["spill_ld"] = int(m.group(1)), int(m.group(2))
        m = re.search(r"Used (\d+) registers", line)
        if m:
            cur["regs"] = int(m.group(1))
    return kernels


@pytest.fixture(scope="module")
def kernels(tmp_path_factory):
    if shutil.which("nvcc") is None and not os.path.exists("/usr/local/cuda/bin/nvcc"):
        pytest.skip("nvcc not available")
    out = str(tmp_path_factory.mktemp("ptxas"))
    with concurrent.futures.ThreadPoolExecutor(len(UNITS)) as ex:
        reports = list(ex.map(lambda s: _report(s, out), UNITS))
    return [k for r in reports for k in r]


def test_every_expected_kernel_is_built(kernels):
    counts = {}
    for k in kernels:
        f = _family(k["name"])
        counts[f] = counts.get(f, 0) + 1
    assert counts == EXPECTED


def test_no_register_spills(kernels):
    for k in kernels:
        assert "spill_st" in k and "regs" in k, k
        assert k["spill_st"] == 0 and k["spill_ld"] == 0, k


def test_registers_fit_the_launch(kernels):
    for k in kernels:
        threads = THREADS[_family(k["name"])]
        assert k["regs"] * threads <= 65536, k
