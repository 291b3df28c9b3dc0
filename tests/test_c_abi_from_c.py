"""The boundary is a C ABI: ``include/fattn.h`` compiles as strict C99 (and
as C++), and a plain C program links against ``libfattn.so`` and calls it
(CPU: the entry points that need no GPU, and the host-side argument checks
of the compute entry points, which return before any CUDA call)."""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

from exact_attention_forward_10_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

PROGRAM = r"""
#include <stdio.h>
#include <string.h>
#include "fattn.h"

int main(void) {
  int fails = 0;
  if (fattn_version() < 100) { puts("version"); ++fails; }
  if (strcmp(fattn_error_string(FATTN_OK), "ok") != 0) { puts("ok string"); ++fails; }
  if (strlen(fattn_error_string(FATTN_ERR_CUDA)) == 0) { puts("cuda string"); ++fails; }
  /* host-side checks: null pointers, bad sizes, bad dtype, misalignment */
  char *p = (char *)0x10000;
  float *l = (float *)0x90000;
  if (fattn_fwd(NULL, p, p, p, l, 1, 1, 128, 64, 0, 0.125f, FATTN_FP16, NULL)
      != FATTN_ERR_INVALID_ARG) { puts("null q"); ++fails; }
  if (fattn_fwd(p, p + 0x20000, p + 0x40000, p + 0x60000, l, 1, 1, 128, 96, 0, 0.125f,
                FATTN_FP16, NULL) != FATTN_ERR_UNSUPPORTED) { puts("D 96"); ++fails; }
  if (fattn_fwd(p, p + 0x20000, p + 0x40000, p + 0x60000, l, 1, 1, 128, 64, 0, 0.125f,
                7, NULL) != FATTN_ERR_UNSUPPORTED) { puts("dtype"); ++fails; }
  if (fattn_fwd(p + 8, p + 0x20000, p + 0x40000, p + 0x60000, l, 1, 1, 128, 64, 0,
                0.125f, FATTN_BF16, NULL) != FATTN_ERR_MISALIGNED) { puts("align"); ++fails; }
  if (fattn_fwd(p, p + 0x20000, p + 0x40000, p + 0x60000, l, 1, 1, 128, 64, 0, -1.0f,
                FATTN_BF16, NULL) != FATTN_ERR_INVALID_ARG) { puts("scale"); ++fails; }
  if (fattn_fwd_kvcache(p, p, p, NULL, p, l, 1, 1, 17, 64, 64, 0, 0.125f, FATTN_FP16,
                        p, 1u << 20, NULL) != FATTN_ERR_UNSUPPORTED) { puts("Sq 17"); ++fails; }
  if (fattn_fwd_fp8(p, p, p, p, l, 1, 1, 128, 64, 0, 0.125f, 1.f, 1.f, 1.f, FATTN_BF16,
                    NULL) != FATTN_ERR_UNSUPPORTED) { puts("fp8 D 64"); ++fails; }
  if (fattn_check_wait_timeout(0, NULL) != FATTN_ERR_INVALID_ARG) { puts("wait"); ++fails; }
  printf("%d failures\n", fails);
  return fails != 0;
}
"""


def _compiler(name):
    path = shutil.which(name)
    if path is None:
        pytest.skip(f"{name} not available")
    return path


def test_header_compiles_as_c99_and_cxx(tmp_path):
    src = tmp_path / "only_header.c"
    src.write_text('#include "fattn.h"\nint main(void) { return FATTN_OK; }\n')
    inc = os.path.join(ROOT, "include")
    for cc, std, extra in (("gcc", "-std=c99", ["-x", "c"]), ("g++", "-std=c++17", ["-x", "c++"])):
        r = subprocess.run([_compiler(cc), std, "-Wall", "-Wextra", "-pedantic", "-Werror",
                            *extra, "-I", inc, "-c", str(src), "-o", str(tmp_path / f"{cc}.o")],
                           capture_output=True, text=True)
        assert r.returncode == 0, f"{cc}: {r.stderr}"


def test_plain_c_program_links_and_calls_the_library(tmp_path):
    lib = fbuild.build()
    src = tmp_path / "use_fattn.c"
    src.write_text(PROGRAM)
    exe = tmp_path / "use_fattn"
    r = subprocess.run([_compiler("gcc"), "-std=c99", "-Wall", "-Werror", "-I",
                        os.path.join(ROOT, "include"), str(src), "-o", str(exe),
                        "-L", os.path.dirname(lib), "-lfattn",
                        f"-Wl,-rpath,{os.path.dirname(lib)}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "0 failures" in r.stdout
