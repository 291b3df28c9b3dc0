"""Seeded synthetic inputs for the exact attention forward.

Q, K and V are i.i.d. N(0, 1), as in the benchmark shapes of "Lecture 6 --
FlashAttention-2" (Benchmark task) and the attention-layer notebook
("FlashAttention-2 in an attention layer", Numerical equivalence), where the
inputs are plain Gaussian tensors.

Generator, named so that seeds reproduce on any machine and torch version:

* SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
  generators", OOPSLA 2014), used as a counter-based stream: output ``o`` of
  seed ``s`` is ``mix(s + (o + 1) * 0x9E3779B97F4A7C15 mod 2**64)``, which is
  the sequential generator started from state ``s``.
* A uniform double in [0, 1) from the top 53 bits of each output.
* Box-Muller (Box & Muller, 1958): outputs ``2p`` and ``2p + 1`` give the
  normal pair ``p``; ``r = sqrt(-2 ln(1 - u0))``, even index ``r cos(2 pi u1)``,
  odd index ``r sin(2 pi u1)``.
* Each normal is rounded to fp32, then to the 16-bit dtype, both
  round-to-nearest-even.  Q, K and V draw consecutive normals (Q first).

This module holds none of the attention arithmetic.  The oracle and the CUDA
path both take their inputs from here and from nowhere else.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

GAMMA = 0x9E3779B97F4A7C15
_M1 = 0xBF58476D1CE4E5B9
_M2 = 0x94D049BB133111EB
_CHUNK = 1 << 22

DTYPES = ("fp16", "bf16")
DTYPE_CODE = {"fp16": 0, "bf16": 1}


def splitmix64(seed: int, start: int, count: int) -> np.ndarray:
    """Outputs ``start .. start+count-1`` of SplitMix64 seeded with ``seed``."""
    idx = np.arange(start + 1, start + count + 1, dtype=np.uint64)
    z = np.uint64(seed & 0xFFFFFFFFFFFFFFFF) + idx * np.uint64(GAMMA)
    z = (z ^ (z >> np.uint64(30))) * np.uint64(_M1)
    z = (z ^ (z >> np.uint64(27))) * np.uint64(_M2)
    return z ^ (z >> np.uint64(31))


def uniform53(words: np.ndarray) -> np.ndarray:
    """Map 64-bit words to doubles in [0, 1) using their top 53 bits."""
    return (words >> np.uint64(11)).astype(np.float64) * (2.0 ** -53)


def normals(seed: int, start: int, count: int) -> np.ndarray:
    """Standard normals ``start .. start+count-1`` of the stream (float64)."""
    if count <= 0:
        return np.zeros(0, dtype=np.float64)
    p0 = start // 2
    p1 = (start + count - 1) // 2 + 1
    w = splitmix64(seed, 2 * p0, 2 * (p1 - p0)).reshape(-1, 2)
    u0 = uniform53(w[:, 0])
    u1 = uniform53(w[:, 1])
    r = np.sqrt(-2.0 * np.log1p(-u0))
    theta = (2.0 * math.pi) * u1
    z = np.empty((p1 - p0, 2), dtype=np.float64)
    z[:, 0] = r * np.cos(theta)
    z[:, 1] = r * np.sin(theta)
    z = z.reshape(-1)
    off = start - 2 * p0
    return z[off:off + count]


def round_fp32_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bf16 (nearest-even); returned as fp32."""
    bits = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    lsb = (bits >> np.uint32(16)) & np.uint32(1)
    r = (bits + np.uint32(0x7FFF) + lsb) & np.uint32(0xFFFF0000)
    return r.view(np.float32)


def round_to_dtype(x64: np.ndarray, dtype: str) -> np.ndarray:
    """fp64 -> fp32 -> ``dtype`` (both nearest-even); returned as fp32."""
    x32 = x64.astype(np.float32)
    if dtype == "fp16":
        return x32.astype(np.float16).astype(np.float32)
    if dtype == "bf16":
        return round_fp32_to_bf16(x32)
    raise ValueError(f"unknown dtype {dtype!r}")


def gaussian_tensor(seed: int, start: int, shape, dtype: str) -> np.ndarray:
    """A tensor of ``prod(shape)`` consecutive normals, rounded to ``dtype``.

    The result is float32 holding values exactly representable in ``dtype``.
    """
    n = int(np.prod(shape))
    out = np.empty(n, dtype=np.float32)
    for c0 in range(0, n, _CHUNK):
        c1 = min(n, c0 + _CHUNK)
        out[c0:c1] = round_to_dtype(normals(seed, start + c0, c1 - c0), dtype)
    return out.reshape(shape)


@dataclasses.dataclass
class QKV:
    """One input set: ``q, k, v`` are float32 ``[B, H, S, D]`` arrays whose
    values are exactly representable in ``dtype``."""

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    dtype: str
    seed: int
    qk_mult: float

    @property
    def shape(self):
        return self.q.shape


def make_qkv(B: int, H: int, S: int, D: int, dtype: str, seed: int,
             qk_mult: float = 1.0) -> QKV:
    """Q, K, V i.i.d. N(0,1) from ``seed`` (Q, then K, then V in the stream).

    ``qk_mult`` multiplies Q and K after rounding; it must be a power of two so
    the product is exact in the 16-bit dtype (the stress set uses 4).
    """
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    m, e = math.frexp(qk_mult)
    if qk_mult <= 0 or m != 0.5:
        raise ValueError("qk_mult must be a positive power of two")
    n = B * H * S * D
    shape = (B, H, S, D)
    q = gaussian_tensor(seed, 0, shape, dtype)
    k = gaussian_tensor(seed, n, shape, dtype)
    v = gaussian_tensor(seed, 2 * n, shape, dtype)
    if qk_mult != 1.0:
        q *= np.float32(qk_mult)
        k *= np.float32(qk_mult)
    return QKV(q=q, k=k, v=v, dtype=dtype, seed=seed, qk_mult=qk_mult)


def make_qkv_shard(B_global: int, b0: int, b1: int, H: int, S: int, D: int,
                   dtype: str, seed: int) -> QKV:
    """Batch rows ``b0 .. b1-1`` of ``make_qkv(B_global, H, S, D, dtype,
    seed)``, generated directly (the generator is counter-based: each row is
    read at its own offset of the stream), so one rank of a data-parallel
    run holds only its shard."""
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    if not 0 <= b0 <= b1 <= B_global:
        raise ValueError("shard outside the global batch")
    per = H * S * D
    n = B_global * per
    shape = (b1 - b0, H, S, D)
    q = gaussian_tensor(seed, b0 * per, shape, dtype)
    k = gaussian_tensor(seed, n + b0 * per, shape, dtype)
    v = gaussian_tensor(seed, 2 * n + b0 * per, shape, dtype)
    return QKV(q=q, k=k, v=v, dtype=dtype, seed=seed, qk_mult=1.0)


# --------------------------------------------------------------------------
# The workloads: sizes, dtypes, masks and seeds of the benchmark shapes.
# --------------------------------------------------------------------------

SWEEP_S = (512, 1024, 2048, 4096, 8192, 16384, 4097)
SWEEP_D = (64, 128)


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: str
    causal: tuple  # the mask modes run on this input set
    seed: int
    qk_mult: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def inputs(self) -> QKV:
        return make_qkv(self.B, self.H, self.S, self.D, self.dtype, self.seed,
                        self.qk_mult)


def sweep_workloads():
    """B=2, H=16 sweep; seed = 4 + index over (S, D, dtype) in that nesting."""
    out = []
    idx = 0
    for S in SWEEP_S:
        for D in SWEEP_D:
            for dt in DTYPES:
                out.append(Workload(f"sweep_S{S}_D{D}_{dt}", 2, 16, S, D, dt,
                                    (False, True), 4 + idx))
                idx += 1
    return out


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, 128, 64, "fp16", (False,), 0),
    "s2048_d64": Workload("B2_H16_S2048_D64_fp16_causal", 2, 16, 2048, 64,
                        "fp16", (True,), 1),
    "s2048_d128": Workload("B1_H32_S2048_D128_fp16_causal", 1, 32, 2048, 128,
                         "fp16", (True,), 2),
    "s8192_d128": Workload("B2_H16_S8192_D128_bf16", 2, 16, 8192, 128, "bf16",
                          (False, True), 3),
    "s8192_d128_x4": Workload("B2_H16_S8192_D128_bf16_QKx4", 2, 16, 8192, 128,
                             "bf16", (False, True), 3, 4.0),
}


# --------------------------------------------------------------------------
# New queries against a key/value cache ("FlashAttention V2", section 6:
# inference with a KV cache).  Same generator; the cached lengths come from
# the same SplitMix64 stream, far past the normals.
# --------------------------------------------------------------------------

_LENS_WORD0 = 1 << 40  # first stream word used for the cached lengths


@dataclasses.dataclass
class KVCache:
    """One cache input set: ``q`` ``[B, H, Sq, D]``, ``k, v`` ``[B, H, Sk, D]``
    (float32 holding ``dtype`` values) and ``lens`` (int64 ``[B]`` cached
    lengths, or ``None`` for every length equal to ``Sk``)."""

    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    lens: np.ndarray | None
    dtype: str
    seed: int


def cache_lengths(seed: int, B: int, lo: int, hi: int) -> np.ndarray:
    """``B`` lengths uniform in ``[lo, hi]`` from stream words 2**40 + b."""
    if not 0 <= lo <= hi:
        raise ValueError("need 0 <= lo <= hi")
    w = splitmix64(seed, _LENS_WORD0, B)
    return (np.uint64(lo) + w % np.uint64(hi - lo + 1)).astype(np.int64)


def make_kvcache(B: int, H: int, Sq: int, Sk: int, D: int, dtype: str,
                 seed: int, lens_range=None) -> KVCache:
    """Q, then the K cache, then the V cache, i.i.d. N(0,1) from ``seed``;
    ``lens_range = (lo, hi)`` draws per-batch cached lengths, else all
    lengths are ``Sk``.  Cache rows past a batch's length hold normals too."""
    if dtype not in DTYPES:
        raise ValueError(f"unknown dtype {dtype!r}")
    nq = B * H * Sq * D
    nk = B * H * Sk * D
    q = gaussian_tensor(seed, 0, (B, H, Sq, D), dtype)
    k = gaussian_tensor(seed, nq, (B, H, Sk, D), dtype)
    v = gaussian_tensor(seed, nq + nk, (B, H, Sk, D), dtype)
    lens = None
    if lens_range is not None:
        lo, hi = lens_range
        if hi > Sk:
            raise ValueError("a cached length cannot exceed the capacity Sk")
        lens = cache_lengths(seed, B, lo, hi)
    return KVCache(q=q, k=k, v=v, lens=lens, dtype=dtype, seed=seed)


@dataclasses.dataclass(frozen=True)
class CacheWorkload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    D: int
    dtype: str
    causal: bool
    seed: int
    lens_range: tuple | None = None

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def inputs(self) -> KVCache:
        return make_kvcache(self.B, self.H, self.Sq, self.Sk, self.D,
                            self.dtype, self.seed, self.lens_range)


CACHE_WORKLOADS = {
    # one new token per sequence, 16 sequences of mixed history length
    "decode_b16_h16_d128_ragged": CacheWorkload(
        "decode_B16_H16_Sq1_Sk16384_D128_bf16_lens1024-16384", 16, 16, 1,
        16384, 128, "bf16", False, 40, (1024, 16384)),
    # the long-sequence benchmark shape, one new token, full caches
    "decode_b2_h16_s8192_d128": CacheWorkload(
        "decode_B2_H16_Sq1_Sk8192_D128_bf16", 2, 16, 1, 8192, 128, "bf16",
        False, 41),
    # four new tokens per sequence under the causal mask, head dim 64, fp16
    "decode_b8_h16_sq4_d64": CacheWorkload(
        "decode_B8_H16_Sq4_Sk8192_D64_fp16_causal_lens1-8192", 8, 16, 4, 8192,
        64, "fp16", True, 42, (1, 8192)),
}


# --------------------------------------------------------------------------
# 8-bit inputs: OCP FP8 E4M3 (the "fn" variant: bias 7, three mantissa bits,
# no infinities, largest finite value 448, subnormals m/8 * 2^-6), for the
# FP8 forward ("FlashAttention V2", section 7: FP8 attention).  Each tensor
# carries one fp32 dequantisation scale: real value = code value * scale.
# --------------------------------------------------------------------------

E4M3_MAX = 448.0


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """Values of E4M3 codes (uint8) as float64; the NaN codes 0x7F, 0xFF
    decode to NaN."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 15
    m = c & 7
    val = np.where(e == 0, m / 8.0 * 2.0 ** -6, (1.0 + m / 8.0) * np.exp2(e - 7.0))
    val = np.where((c & 0x7F) == 0x7F, np.nan, val)
    return sign * val


def e4m3_encode(x: np.ndarray) -> np.ndarray:
    """Round finite values to E4M3 codes: nearest, ties to even mantissa,
    magnitudes above 448 saturate to 448 (the finite-saturating cast)."""
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    # exponent of the binade, at least the subnormal one (2^-6)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    e = np.maximum(e, -6.0)
    quantum = np.exp2(e - 3.0)
    q = np.round(a / quantum) * quantum        # numpy rounds half to even
    q = np.minimum(q, E4M3_MAX)
    q = np.where(a == 0, 0.0, q)
    # encode q (exactly representable now)
    eq = np.floor(np.log2(np.where(q > 0, q, 1.0)))
    sub = q < 2.0 ** -6
    mant_sub = np.round(q / 2.0 ** -9).astype(np.int64)              # m/8 * 2^-6
    exp_n = (eq + 7).astype(np.int64)
    mant_n = np.round((q / np.exp2(eq) - 1.0) * 8.0).astype(np.int64)
    code = np.where(sub, mant_sub, (exp_n << 3) | mant_n)
    code = np.where(q == 0, 0, code)
    return (code | np.where(x < 0, 0x80, 0)).astype(np.uint8)


@dataclasses.dataclass
class QKV8:
    """E4M3 inputs: ``q8, k8, v8`` uint8 codes [B, H, S, D]; ``descale`` the
    three per-tensor scales; ``q, k, v`` the real values (code value times
    scale, exact in float64)."""

    q8: np.ndarray
    k8: np.ndarray
    v8: np.ndarray
    descale: tuple
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    seed: int


def make_qkv_fp8(B: int, H: int, S: int, D: int, seed: int,
                 qk_mult: float = 1.0) -> QKV8:
    """Q, K, V i.i.d. N(0,1) from ``seed`` (the same stream and order as
    ``make_qkv``), each multiplied by ``qk_mult`` (Q and K only), then
    quantised per tensor: scale = a power of two putting the tensor's largest
    magnitude at or below 448, code = E4M3 rounding of value / scale."""
    n = B * H * S * D
    shape = (B, H, S, D)
    out = []
    for i, mult in enumerate((qk_mult, qk_mult, 1.0)):
        x = np.empty(n, dtype=np.float64)
        for c0 in range(0, n, _CHUNK):
            c1 = min(n, c0 + _CHUNK)
            x[c0:c1] = normals(seed, i * n + c0, c1 - c0)
        x *= mult
        amax = float(np.abs(x).max()) if n else 1.0
        scale = 2.0 ** math.ceil(math.log2(amax / E4M3_MAX)) if amax > 0 else 1.0
        codes = e4m3_encode(x / scale).reshape(shape)
        out.append((codes, scale, e4m3_decode(codes) * scale))
    (q8, qs, q), (k8, ks, k), (v8, vs, v) = out
    return QKV8(q8=q8, k8=k8, v8=v8, descale=(qs, ks, vs), q=q, k=k, v=v, seed=seed)
