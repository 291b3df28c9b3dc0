"""Build ``libfattn.so`` in-tree with nvcc for sm_103a.

The translation units compile in parallel (one per head dim and kernel
family, plus the host library) and are linked into one shared library with the CUDA runtime linked
statically, so the library loads on machines without a GPU driver.

    python -m exact_attention_forward_10_gb300.build [--verbose]

Extra nvcc flags (for experiments, e.g. -DFATTN_SPIN_ROLES=2) may be given in
the FATTN_NVCC_FLAGS environment variable; they force a rebuild.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(PKG, "libfattn.so")

SOURCES = ["fattn_api.cu", "fattn_fwd_d64.cu", "fattn_fwd_d128.cu", "fattn_fwd_d256.cu",
           "fattn_fwd_fp8.cu",
           "fattn_decode.cu", "fattn_decode_d64.cu", "fattn_decode_d128.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the CUDA 13 toolkit is required")
    return cand


def _deps() -> list:
    out = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    out.append(os.path.join(INCLUDE, "fattn.h"))
    return out


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(p) <= t for p in _deps())


def _compile(src: str, verbose: bool) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
    cmd = [nvcc(), *ARCH, "-O3", "-lineinfo", "-std=c++17",
           "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE,
           *os.environ.get("FATTN_NVCC_FLAGS", "").split(),
           "-c", os.path.join(CSRC, src), "-o", obj]
    if verbose:
        cmd[1:1] = ["-Xptxas", "-v"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
    if verbose and r.stderr:
        sys.stderr.write(r.stderr)
    return obj


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit and link ``libfattn.so``."""
    if not force and not verbose and up_to_date() and not os.environ.get("FATTN_NVCC_FLAGS"):
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    with concurrent.futures.ThreadPoolExecutor(len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(s, verbose), SOURCES))
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    build(force=True, verbose="--verbose" in sys.argv)
    print(LIB_PATH)
