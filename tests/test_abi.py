"""The C-ABI library: it loads without a GPU, exports every entry point that
include/fattn.h declares, and rejects bad arguments on the host before any
CUDA call (so these run on a CPU-only machine).  Without the library nothing
computes: the binding raises, and host tensors are refused."""
import os
import re

import pytest

import exact_attention_forward_10_gb300 as fattn
from exact_attention_forward_10_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fbuild.build()
    return fattn.lib()


def declared_symbols():
    out = []
    for name in os.listdir(os.path.join(ROOT, "include")):
        if not name.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", name)).read()
        out += re.findall(r"^FATTN_API\s[^;(]*?\b(\w+)\s*\(", text, re.M)
    return sorted(set(out))


def test_header_declares_entry_points():
    syms = declared_symbols()
    assert "fattn_fwd" in syms and "fattn_last_error" in syms
    assert len(syms) >= 5


def test_every_declared_symbol_is_exported(lib):
    for s in declared_symbols():
        assert hasattr(lib, s), f"{s} declared in include/ but not exported"


def test_version_and_strings(lib):
    assert fattn.fattn_version() >= 100
    for code in range(-7, 1):
        assert fattn.fattn_error_string(code) not in ("", "unknown status")
    assert fattn.fattn_error_string(-99) == "unknown status"


# A fake, 16-byte aligned, non-null address: host checks must reject the call
# before the pointer is ever looked at.
P = 1 << 20


@pytest.mark.parametrize("args,want", [
    (dict(q=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(lse=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(B=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(S=-3), fattn.FATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fattn.FATTN_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fattn.FATTN_ERR_INVALID_ARG),
    (dict(D=96), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(D=512), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(dtype=2), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(q=P + 8), fattn.FATTN_ERR_MISALIGNED),
    (dict(o=P * 9 + 2), fattn.FATTN_ERR_MISALIGNED),
    (dict(lse=P * 11 + 2), fattn.FATTN_ERR_MISALIGNED),
    (dict(B=1 << 16, H=1 << 10, S=1 << 10), fattn.FATTN_ERR_TOO_LARGE),
    (dict(o=P), fattn.FATTN_ERR_INVALID_ARG),          # o aliases q
    (dict(lse=P * 7 + 64), fattn.FATTN_ERR_INVALID_ARG),  # lse inside v
])
def test_host_side_rejections(lib, args, want):
    a = dict(q=P, k=P * 3, v=P * 7, o=P * 9, lse=P * 11, B=1, H=2, S=128,
             D=64, causal=0, scale=0.125, dtype=0, stream=0)
    a.update(args)
    rc = fattn.fattn_fwd(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"],
                         a["H"], a["S"], a["D"], a["causal"], a["scale"],
                         a["dtype"], a["stream"])
    assert rc == want


def test_plan_without_device(lib):
    p = fattn.fattn_plan(2, 16, 8192, 128, True)
    assert p["q_tiles_per_unit"] in (1, 2)
    assert p["units"] == 2 * 16 * (8192 // (128 * p["q_tiles_per_unit"]))
    assert p["smem_bytes"] <= 232448
    assert p["block"] % 128 == 0
    assert 1 <= p["grid"] <= p["units"]
    with pytest.raises(fattn.FattnError):
        fattn.fattn_plan(1, 1, 10, 80)


def test_plan_head_dim_256_uses_cta_pairs(lib):
    p = fattn.fattn_plan(2, 16, 8192, 256, False)
    assert p["q_tiles_per_unit"] == 2 and p["units"] == 2 * 16 * (8192 // 256)
    assert p["smem_bytes"] <= 232448 and p["block"] == 384
    assert p["grid"] % 2 == 0 and 2 <= p["grid"] <= 2 * p["units"]


@pytest.mark.parametrize("args,want", [
    (dict(q=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(k=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(ws=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(lse=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(B=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(Sq=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(Sk=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(scale=-1.0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fattn.FATTN_ERR_INVALID_ARG),
    (dict(Sq=17), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(D=256), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(dtype=5), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(q=P + 4), fattn.FATTN_ERR_MISALIGNED),
    (dict(v=P * 7 + 8), fattn.FATTN_ERR_MISALIGNED),
    (dict(ws=P * 13 + 8), fattn.FATTN_ERR_MISALIGNED),
    (dict(lse=P * 11 + 1), fattn.FATTN_ERR_MISALIGNED),
    (dict(lens=P * 15 + 2), fattn.FATTN_ERR_MISALIGNED),
])
def test_kvcache_host_side_rejections(lib, args, want):
    """Argument errors of the cache entry point are found before any CUDA
    call (workspace size and overlap checks need the device's SM count and
    are covered by the GPU tests)."""
    a = dict(q=P, k=P * 3, v=P * 7, lens=P * 15, o=P * 9, lse=P * 11, B=2, H=4,
             Sq=1, Sk=4096, D=128, causal=0, scale=0.125, dtype=1, ws=P * 13,
             ws_bytes=1 << 30, stream=0)
    a.update(args)
    rc = fattn.fattn_fwd_kvcache(a["q"], a["k"], a["v"], a["lens"], a["o"],
                                 a["lse"], a["B"], a["H"], a["Sq"], a["Sk"],
                                 a["D"], a["causal"], a["scale"], a["dtype"],
                                 a["ws"], a["ws_bytes"], a["stream"])
    assert rc == want


@pytest.mark.parametrize("args,want", [
    (dict(q=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(scale=0.0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(qs=-1.0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(vs=float("inf")), fattn.FATTN_ERR_INVALID_ARG),
    (dict(S=0), fattn.FATTN_ERR_INVALID_ARG),
    (dict(D=64), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(D=256), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(out=3), fattn.FATTN_ERR_UNSUPPORTED),
    (dict(k=P * 3 + 4), fattn.FATTN_ERR_MISALIGNED),
    (dict(lse=P * 11 + 2), fattn.FATTN_ERR_MISALIGNED),
    (dict(o=P), fattn.FATTN_ERR_INVALID_ARG),      # o overlaps q
])
def test_fp8_host_side_rejections(lib, args, want):
    a = dict(q=P, k=P * 3, v=P * 7, o=P * 9, lse=P * 11, B=1, H=2, S=256, D=128,
             causal=0, scale=0.088, qs=0.5, ks=0.5, vs=0.5, out=1, stream=0)
    a.update(args)
    rc = fattn.fattn_fwd_fp8(a["q"], a["k"], a["v"], a["o"], a["lse"], a["B"], a["H"],
                             a["S"], a["D"], a["causal"], a["scale"], a["qs"], a["ks"],
                             a["vs"], a["out"], a["stream"])
    assert rc == want


def test_wait_check_rejects_out_of_range_limits(lib):
    for us in (0, -5, 1000001):
        assert fattn.fattn_check_wait_timeout(us, 0) == fattn.FATTN_ERR_INVALID_ARG


def test_missing_library_raises(monkeypatch, tmp_path):
    """No library, no computation: every entry point goes through ``lib()``,
    which raises instead of falling back to anything else."""
    monkeypatch.setattr(fattn, "LIB_PATH", str(tmp_path / "libfattn.so"))
    monkeypatch.setattr(fattn, "_lib", None)
    with pytest.raises(ImportError):
        fattn.lib()
    with pytest.raises(ImportError):
        fattn.fattn_fwd(16, 16, 16, 16, 16, 1, 1, 128, 64, 0, 0.125, 0, 0)
    with pytest.raises(ImportError):
        fattn.fattn_version()


def test_host_tensors_are_rejected():
    """The torch wrappers take CUDA tensors only; there is no host path."""
    torch = pytest.importorskip("torch")
    q = torch.zeros(1, 1, 128, 64, dtype=torch.float16)
    with pytest.raises(ValueError):
        fattn.forward(q, q, q)
    with pytest.raises(ValueError):
        fattn.forward_kvcache(q[:, :, :1], q, q)
    q8 = torch.zeros(1, 1, 128, 128, dtype=torch.uint8)
    with pytest.raises(ValueError):
        fattn.forward_fp8(q8, q8, q8, 1.0, 1.0, 1.0)
