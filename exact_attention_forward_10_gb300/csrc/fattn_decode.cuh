// Attention of a few new queries against a key/value cache on sm_103a (GB300):
// split-KV partials plus an LSE-weighted merge.
//
// What it computes ("FlashAttention V2", section 6: inference with a KV cache,
// served by a decoding variant; the per-row recurrence of section 3): for
// head (b, h) with len_b cached positions and Sq new queries, query i sits at
// position len_b - Sq + i and attends to every cached key j < len_b (causal:
// j <= len_b - Sq + i):
//     O_i = softmax_j(scale * q_i . k_j) V,   LSE_i = m + ln(sum_j exp(s_j - m)).
// A query with no allowed key gets O = 0 and LSE = -inf.
//
// Why this shape on GB300.  With one to a few queries per head the work is
// about one multiply-add per cached 16-bit value read: it is bound by HBM
// (7.9 TB/s nominal), not by the tensor cores, so the keys are split across
// every warp of the GPU and each warp streams its slice once:
//   * the flattened sequence of (batch, head, 32-key tile) is cut into one
//     contiguous range per warp (grid = one CTA per SM), so ragged cache
//     lengths stay balanced;
//   * each warp double-buffers its own K/V tiles: TMA 3-D loads with the
//     128-byte swizzle into shared memory, completion on a per-slot mbarrier
//     (no cross-warp synchronisation at all);
//   * scores: lane l owns key l of the tile and walks its row in 16-byte
//     chunks (the swizzle makes the eight lanes of each phase hit distinct
//     banks) against a broadcast read of the query; the multiply-adds take
//     the 16-bit operands directly and accumulate in fp32;
//   * online softmax per query row across the warp (one max reduction per
//     tile, exp2 with the scale folded in); P is rounded to the input dtype
//     for the P.V product, the row sum keeps fp32 p for the LSE and the
//     rounded p for the normaliser of O;
//   * P.V: lane l owns D/32 output columns and walks the tile's keys, reading
//     each V row once (256 contiguous bytes across the warp);
//   * at the end of each head it touches, the warp writes one partial record
//     (O normalised by its own sum, and its log2-domain LSE) to a workspace;
//     a second small kernel merges a head's records with weights
//     2^(lse_s - max lse).
// Every wait is bounded; a timeout records an error in the status block and
// the warp waits for its own copies before it exits.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "fattn_status.h"
#include "ptx.cuh"

namespace fattn {
namespace decode {

constexpr int kTileKeys = 32;     // keys per tile: one per lane
constexpr int kBoxCols = 64;      // 16-bit columns per TMA box (128 bytes)
constexpr int kBoxBytes = kTileKeys * 128;
constexpr int kMaxSq = 16;        // new queries per head handled here
constexpr int kRoleDecode = 5;    // status word 1, high byte
constexpr int kRoleLens = 6;      // a cached length outside [0, Sk]
constexpr int kSmemBudget = 232448 - 1024;  // opt-in limit minus alignment slack
constexpr float kEmptyMax = -1.0e30f;       // running max before any key

struct DecodeParams {
  const void* q;         // [BH, Sq, D] 16-bit
  const int* lens;       // [B] cached lengths, or nullptr: every length is Sk
  float* part_o;         // [R, Sq, D] partial outputs (R = warps + BH)
  float* part_lse;       // [R, Sq] partial log2-domain LSE
  void* o;               // [BH, Sq, D] 16-bit
  float* lse;            // [BH, Sq] natural-log LSE
  int* status;           // device status block
  int B, H, Sq, Sk;
  int causal;
  int n_warps;           // total decode warps (grid * warps per CTA)
  float scale_log2;      // scale * log2(e)
  unsigned long long timeout_ns;
};

// Shared-memory plan of one decode CTA: per warp two K/V slots (each a K tile
// and a V tile of 32 rows, D/64 swizzled boxes apiece), the warp's query rows
// and its rounded-P buffer, then the slot barriers.
template <int D, int SQ>
struct DecodeLayout {
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;   // one K (or V) tile
  static constexpr int kSlotBytes = 2 * kTileBytes;       // K then V
  static constexpr int kQBytes = SQ * D * 2;
  static constexpr int kPBytes = SQ * kTileKeys * 2;
  static constexpr int kPerWarp = 2 * kSlotBytes + kQBytes + kPBytes + 2 * 8;
  static constexpr int kWarpsFit = kSmemBudget / kPerWarp;
  // 12 warps leave 170 registers a thread; sixteen query rows need more.
  static constexpr int kWarpCap = SQ >= 16 ? 8 : 12;
  static constexpr int kWarps = kWarpsFit > kWarpCap ? kWarpCap : kWarpsFit;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kSlotsOff = 0;  // 1024-aligned: slots first
  static constexpr int kQOff = kWarps * 2 * kSlotBytes;
  static constexpr int kPOff = kQOff + kWarps * kQBytes;
  static constexpr int kBarOff = kPOff + kWarps * kPBytes;
  static constexpr int kSmemBytes = kBarOff + kWarps * 2 * 8 + 1024;
  static_assert(kWarps >= 4, "decode CTA too small");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// ------------------------------------------------------------ small helpers

// c + a.lo * b.lo + a.hi * b.hi with 16-bit operands and fp32 accumulation.
template <bool BF16>
__device__ __forceinline__ float fma_pair(uint32_t a, uint32_t b, float c) {
  if constexpr (BF16) {
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.bf16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.bf16 %0, a1, b1, %0;\n\t}"
        : "+f"(c) : "r"(a), "r"(b));
  } else {
    asm("{\n\t.reg .b16 a0, a1, b0, b1;\n\t"
        "mov.b32 {a0, a1}, %1;\n\tmov.b32 {b0, b1}, %2;\n\t"
        "fma.rn.f32.f16 %0, a0, b0, %0;\n\t"
        "fma.rn.f32.f16 %0, a1, b1, %0;\n\t}"
        : "+f"(c) : "r"(a), "r"(b));
  }
  return c;
}

// o0 += p * v.lo, o1 += p * v.hi, where p is the HI (or LO) half of pp.
template <bool BF16, bool HI>
__device__ __forceinline__ void fma_bcast(uint32_t pp, uint32_t v, float& o0,
                                          float& o1) {
  if constexpr (BF16) {
    if constexpr (HI)
      asm("{\n\t.reg .b16 p0, p1, v0, v1;\n\t"
          "mov.b32 {p0, p1}, %2;\n\tmov.b32 {v0, v1}, %3;\n\t"
          "fma.rn.f32.bf16 %0, p1, v0, %0;\n\t"
          "fma.rn.f32.bf16 %1, p1, v1, %1;\n\t}"
          : "+f"(o0), "+f"(o1) : "r"(pp), "r"(v));
    else
      asm("{\n\t.reg .b16 p0, p1, v0, v1;\n\t"
          "mov.b32 {p0, p1}, %2;\n\tmov.b32 {v0, v1}, %3;\n\t"
          "fma.rn.f32.bf16 %0, p0, v0, %0;\n\t"
          "fma.rn.f32.bf16 %1, p0, v1, %1;\n\t}"
          : "+f"(o0), "+f"(o1) : "r"(pp), "r"(v));
  } else {
    if constexpr (HI)
      asm("{\n\t.reg .b16 p0, p1, v0, v1;\n\t"
          "mov.b32 {p0, p1}, %2;\n\tmov.b32 {v0, v1}, %3;\n\t"
          "fma.rn.f32.f16 %0, p1, v0, %0;\n\t"
          "fma.rn.f32.f16 %1, p1, v1, %1;\n\t}"
          : "+f"(o0), "+f"(o1) : "r"(pp), "r"(v));
    else
      asm("{\n\t.reg .b16 p0, p1, v0, v1;\n\t"
          "mov.b32 {p0, p1}, %2;\n\tmov.b32 {v0, v1}, %3;\n\t"
          "fma.rn.f32.f16 %0, p0, v0, %0;\n\t"
          "fma.rn.f32.f16 %1, p0, v1, %1;\n\t}"
          : "+f"(o0), "+f"(o1) : "r"(pp), "r"(v));
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// fp32 -> 16-bit (nearest-even) bits, and those bits back to fp32 exactly.
template <bool BF16>
__device__ __forceinline__ uint16_t to16(float x) {
  if constexpr (BF16) return __bfloat16_as_ushort(__float2bfloat16_rn(x));
  else return __half_as_ushort(__float2half_rn(x));
}
template <bool BF16>
__device__ __forceinline__ float from16(uint16_t b) {
  if constexpr (BF16) return __uint_as_float((uint32_t)b << 16);
  else return __half2float(__ushort_as_half(b));
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, s));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int s = 16; s > 0; s >>= 1) x += __shfl_xor_sync(0xffffffffu, x, s);
  return x;
}

__device__ __forceinline__ void record_error(int* status, int code, int where,
                                             int block) {
  if (atomicCAS(status, 0, code) == 0) {
    status[1] = where;
    status[2] = block;
  }
}

// ------------------------------------------------------------ the partition
//
// The work is the sequence of 32-key tiles of every head, batch-major:
// batch b contributes H * n_b tiles (head-major inside the batch), n_b =
// ceil(len_b / 32).  Warp g of n_warps takes tiles [g*T/n_warps,
// (g+1)*T/n_warps).  A warp's record for head bh has index g + bh: along the
// sequence of (warp, head) overlaps both indices only grow, so these are
// distinct and below n_warps + B*H.

struct Cursor {
  int b;        // batch
  int n_b;      // tiles per head in this batch
  long long base;  // index of this batch's first tile
};

// Cached length of batch b, checked against [0, Sk] (an out-of-range value is
// recorded as an invalid argument and clamped so every access stays inside
// the cache).
__device__ __forceinline__ int cached_len(const DecodeParams& p, int b) {
  if (p.lens == nullptr) return p.Sk;
  int len = __ldg(p.lens + b);
  if (len < 0 || len > p.Sk) {
    record_error(p.status, kErrInvalidArg, (kRoleLens << 8), b);
    len = len < 0 ? 0 : p.Sk;
  }
  return len;
}

__device__ __forceinline__ int tiles_of(int len) {
  return (len + kTileKeys - 1) / kTileKeys;
}

// Total number of tiles T (all lanes get it).
__device__ __forceinline__ long long total_tiles(const DecodeParams& p) {
  if (p.lens == nullptr) return (long long)p.B * p.H * tiles_of(p.Sk);
  const int lane = threadIdx.x & 31;
  long long acc = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    int c = b < p.B ? tiles_of(cached_len(p, b)) : 0;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) c += __shfl_xor_sync(0xffffffffu, c, s);
    acc += (long long)c * p.H;
  }
  return acc;
}

// The batch holding tile t (t < T), its tile count and first tile index.
__device__ __forceinline__ Cursor find_batch(const DecodeParams& p, long long t) {
  Cursor cur;
  if (p.lens == nullptr) {
    cur.n_b = tiles_of(p.Sk);
    const long long per = (long long)p.H * cur.n_b;
    cur.b = (int)(t / per);
    cur.base = (long long)cur.b * per;
    return cur;
  }
  const int lane = threadIdx.x & 31;
  long long acc = 0;
  cur.b = p.B - 1;
  cur.n_b = 0;
  cur.base = 0;
  for (int b0 = 0; b0 < p.B; b0 += 32) {
    const int b = b0 + lane;
    const int nb = b < p.B ? tiles_of(cached_len(p, b)) : 0;
    long long incl = (long long)nb * p.H;
#pragma unroll
    for (int s = 1; s < 32; s <<= 1) {
      const long long o = __shfl_up_sync(0xffffffffu, incl, s);
      if (lane >= s) incl += o;
    }
    const unsigned hit = __ballot_sync(0xffffffffu, b < p.B && acc + incl > t);
    if (hit) {
      const int f = __ffs(hit) - 1;
      cur.b = b0 + f;
      cur.n_b = __shfl_sync(0xffffffffu, nb, f);
      cur.base = acc + __shfl_sync(0xffffffffu, incl, f) - (long long)cur.n_b * p.H;
      return cur;
    }
    acc += __shfl_sync(0xffffffffu, incl, 31);
  }
  return cur;
}

// The next batch with at least one tile after batch cur.b.
__device__ __forceinline__ void next_batch(const DecodeParams& p, Cursor& cur) {
  cur.base += (long long)cur.n_b * p.H;
  do {
    ++cur.b;
    cur.n_b = cur.b < p.B ? tiles_of(cached_len(p, cur.b)) : 1;
  } while (cur.n_b == 0);
}

// Moves the cursor forward until pos (a tile index from cur.base) lies in
// its batch.  False when the lengths read now put pos past the last batch:
// that happens only when the lengths change while the call runs (the caller
// writing them concurrently), and the kernels then stop instead of reading
// outside their buffers.
__device__ __forceinline__ bool seek(const DecodeParams& p, Cursor& cur, long long& pos) {
  while (pos >= (long long)cur.n_b * p.H) {
    if (cur.b >= p.B - 1) return false;
    pos -= (long long)cur.n_b * p.H;
    next_batch(p, cur);
  }
  return cur.b < p.B;
}

__device__ __forceinline__ long long range_start(long long g, long long T,
                                                 int n_warps) {
  return g * T / n_warps;
}

// ------------------------------------------------------------ decode kernel

template <int D, int SQ, bool BF16>
__global__ void __launch_bounds__(DecodeLayout<D, SQ>::kThreads, 1)
    fattn_decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const DecodeParams p) {
  using L = DecodeLayout<D, SQ>;
  constexpr int kCols = D / 32;          // output columns per lane (4 or 2)
  constexpr int kChunks = D / 8;         // 16-byte chunks per K row
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t s_base = ptx::smem_u32(smem);
  const uint32_t slot0 = s_base + L::kSlotsOff + warp * 2 * L::kSlotBytes;
  uint8_t* qbuf = smem + L::kQOff + warp * L::kQBytes;
  uint16_t* pbuf = reinterpret_cast<uint16_t*>(smem + L::kPOff + warp * L::kPBytes);
  const uint32_t bar0 = s_base + L::kBarOff + warp * 16;

  if (lane == 0) {
    ptx::mbar_init(bar0, 1);
    ptx::mbar_init(bar0 + 8, 1);
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tm_k);
    ptx::tma_prefetch_desc(&tm_v);
  }
  __syncwarp();

  // The merge grid may start now: it waits for this grid's completion
  // before it reads a record.
  asm volatile("griddepcontrol.launch_dependents;");

  const int Sq = p.Sq;
  const long long T = total_tiles(p);
  const long long g = (long long)blockIdx.x * L::kWarps + warp;
  const long long t0 = range_start(g, T, p.n_warps);
  const long long t1 = range_start(g + 1, T, p.n_warps);
  if (t0 >= t1) return;
  const int n_tiles = (int)(t1 - t0);

  // Cursors for the loads (up to two tiles ahead) and for the compute.
  Cursor lc = find_batch(p, t0);
  Cursor cc = lc;
  long long lpos = t0 - lc.base;  // tile index inside batch lc.b
  long long cpos = lpos;
  auto issue = [&](int r) {       // load tile t0 + r into slot r & 1
    const bool found = seek(p, lc, lpos);
    const int h = found ? (int)(lpos / lc.n_b) : 0;
    const int kt = found ? (int)(lpos % lc.n_b) : 0;
    const int bh = lc.b * p.H + h;
    if (lane == 0 && !found) ptx::mbar_arrive(bar0 + (r & 1) * 8);  // phase ends empty
    if (lane == 0 && found) {
      const uint32_t slot = slot0 + (r & 1) * L::kSlotBytes;
      const uint32_t bar = bar0 + (r & 1) * 8;
      ptx::mbar_arrive_expect_tx(bar, L::kSlotBytes);
#pragma unroll
      for (int c = 0; c < L::kBoxes; ++c) {
        ptx::tma_load_3d(slot + c * kBoxBytes, &tm_k, bar, c * kBoxCols,
                         kt * kTileKeys, bh);
        ptx::tma_load_3d(slot + L::kTileBytes + c * kBoxBytes, &tm_v, bar,
                         c * kBoxCols, kt * kTileKeys, bh);
      }
    }
    ++lpos;
  };
  issue(0);
  if (n_tiles > 1) issue(1);

  int cur_bh = -1, cur_len = 0;

  float m[SQ], l32[SQ], l16[SQ], o[SQ][kCols];
  auto reset = [&]() {
#pragma unroll
    for (int q = 0; q < SQ; ++q) {
      m[q] = kEmptyMax;
      l32[q] = 0.f;
      l16[q] = 0.f;
#pragma unroll
      for (int c = 0; c < kCols; ++c) o[q][c] = 0.f;
    }
  };
  // Partial record of the current head: O normalised by the rounded-P sum,
  // LSE in log2 units of the scaled scores (-inf: no allowed key seen).
  auto flush = [&]() {
    const long long rec = g + cur_bh;
#pragma unroll
    for (int q = 0; q < SQ; ++q) {
      if (SQ > 1 && q >= Sq) break;
      const float s32 = warp_sum(l32[q]);
      const float s16 = warp_sum(l16[q]);
      const float inv = s16 > 0.f ? 1.0f / s16 : 0.f;
      float* dst = p.part_o + (rec * Sq + q) * D + lane * kCols;
      if constexpr (kCols == 4) {
        *reinterpret_cast<float4*>(dst) =
            make_float4(o[q][0] * inv, o[q][1] * inv, o[q][2] * inv, o[q][3] * inv);
      } else {
        *reinterpret_cast<float2*>(dst) = make_float2(o[q][0] * inv, o[q][1] * inv);
      }
      if (lane == 0)
        p.part_lse[rec * Sq + q] = s32 > 0.f ? m[q] + __log2f(s32) : -INFINITY;
    }
  };

  bool ok = true;
  int fail = 0;
  for (int r = 0; r < n_tiles; ++r) {
    // ---- which head and key tile
    if (!seek(p, cc, cpos)) {
      if (lane == 0) record_error(p.status, kErrInvalidArg, (kRoleLens << 8) | 1, blockIdx.x);
      ok = false;
      fail = r;
      break;
    }
    const int h = (int)(cpos / cc.n_b);
    const int kt = (int)(cpos % cc.n_b);
    ++cpos;
    const int bh = cc.b * p.H + h;
    if (bh != cur_bh) {
      if (cur_bh >= 0) flush();
      cur_bh = bh;
      cur_len = cached_len(p, cc.b);
      reset();
      // the head's query rows -> shared memory (16-byte vectors)
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(p.q) + (size_t)bh * Sq * D * 2);
      uint4* dstq = reinterpret_cast<uint4*>(qbuf);
      for (int i = lane; i < Sq * D / 8; i += 32) dstq[i] = __ldg(src + i);
      __syncwarp();
    }
    const int key0 = kt * kTileKeys;
    const int nvalid = max(0, min(kTileKeys, cur_len - key0));

    // ---- wait for the tile
    const uint32_t slot = slot0 + (r & 1) * L::kSlotBytes;
    if (!ptx::mbar_wait_drain(bar0 + (r & 1) * 8, (r >> 1) & 1, p.timeout_ns)) {
      if (lane == 0)
        record_error(p.status, kErrPipelineTimeout, (kRoleDecode << 8) | (r & 1),
                     blockIdx.x);
      ok = false;
      fail = r;
      break;
    }

    // ---- scores: lane owns key `lane`; 16-byte chunks of its K row against
    // broadcast chunks of each query row
    float s[SQ];
#pragma unroll
    for (int q = 0; q < SQ; ++q) s[q] = 0.f;
    {
      float s2[SQ];
#pragma unroll
      for (int q = 0; q < SQ; ++q) s2[q] = 0.f;
      const uint32_t krow = slot + lane * 128;
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        const uint32_t ka = krow + (c / 8) * kBoxBytes + (((c & 7) ^ (lane & 7)) << 4);
        uint32_t k0, k1, k2, k3;
        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(k0), "=r"(k1), "=r"(k2), "=r"(k3) : "r"(ka));
#pragma unroll
        for (int q = 0; q < SQ; ++q) {
          if (SQ > 1 && q >= Sq) break;
          const uint4 qv = *reinterpret_cast<const uint4*>(qbuf + q * D * 2 + c * 16);
          s[q] = fma_pair<BF16>(k0, qv.x, s[q]);
          s2[q] = fma_pair<BF16>(k1, qv.y, s2[q]);
          s[q] = fma_pair<BF16>(k2, qv.z, s[q]);
          s2[q] = fma_pair<BF16>(k3, qv.w, s2[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < SQ; ++q) s[q] += s2[q];
    }

    // ---- online softmax across the warp, per query row
    const int key = key0 + lane;
#pragma unroll
    for (int q = 0; q < SQ; ++q) {
      if (SQ > 1 && q >= Sq) break;
      const int last = p.causal ? cur_len - Sq + q : cur_len - 1;
      const float t = (key <= last && key < cur_len) ? s[q] * p.scale_log2 : -INFINITY;
      const float m_new = fmaxf(m[q], warp_max(t));
      const float pj = ex2(t - m_new);
      const uint16_t pb = to16<BF16>(pj);
      if (m_new != m[q]) {  // the same on every lane
        const float alpha = ex2(m[q] - m_new);
        l32[q] *= alpha;
        l16[q] *= alpha;
#pragma unroll
        for (int c = 0; c < kCols; ++c) o[q][c] *= alpha;
        m[q] = m_new;
      }
      l32[q] += pj;
      l16[q] += from16<BF16>(pb);
      pbuf[q * kTileKeys + lane] = pb;
    }
    __syncwarp();

    // ---- O += P V: lane owns columns [lane*kCols, lane*kCols + kCols)
    {
      const uint32_t vtile = slot + L::kTileBytes;
      // byte offset of this lane's columns inside a 128-byte box row
      const int colb = (lane * kCols * 2) & 127;
      const uint32_t vbox = vtile + ((lane * kCols * 2) >> 7) * kBoxBytes;
      for (int j0 = 0; j0 < nvalid; j0 += 8) {
        uint4 pp[SQ];
#pragma unroll
        for (int q = 0; q < SQ; ++q) {
          if (SQ > 1 && q >= Sq) break;
          pp[q] = *reinterpret_cast<const uint4*>(pbuf + q * kTileKeys + j0);
        }
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
          const int j = j0 + jj;
          if (j >= nvalid) break;
          const uint32_t va = vbox + j * 128 +
                              ((((colb >> 4) ^ (j & 7)) << 4) | (colb & 15));
          uint32_t v0, v1 = 0;
          if constexpr (kCols == 4)
            asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v0), "=r"(v1) : "r"(va));
          else
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v0) : "r"(va));
#pragma unroll
          for (int q = 0; q < SQ; ++q) {
            if (SQ > 1 && q >= Sq) break;
            const uint32_t w = jj < 2 ? pp[q].x : jj < 4 ? pp[q].y : jj < 6 ? pp[q].z : pp[q].w;
            if (jj & 1) {
              fma_bcast<BF16, true>(w, v0, o[q][0], o[q][1]);
              if constexpr (kCols == 4) fma_bcast<BF16, true>(w, v1, o[q][2], o[q][3]);
            } else {
              fma_bcast<BF16, false>(w, v0, o[q][0], o[q][1]);
              if constexpr (kCols == 4) fma_bcast<BF16, false>(w, v1, o[q][2], o[q][3]);
            }
          }
        }
      }
    }
    __syncwarp();  // every lane is done with this slot and with pbuf

    if (r + 2 < n_tiles) issue(r + 2);
  }

  if (ok) {
    flush();
    return;
  }
  // Unwind after a timeout at tile `fail`: tiles fail and fail + 1 may still
  // have copies in flight into this warp's slots; wait for them (bounded)
  // so none lands after the CTA has exited.
  ptx::mbar_wait_drain(bar0 + (fail & 1) * 8, (fail >> 1) & 1, p.timeout_ns);
  if (fail + 1 < n_tiles)
    ptx::mbar_wait_drain(bar0 + ((fail + 1) & 1) * 8, ((fail + 1) >> 1) & 1,
                         p.timeout_ns);
}

// ------------------------------------------------------------ merge kernel
//
// One warp per (head, query row): the head's records are those of the warps
// whose tile ranges overlap the head's tiles.  Weights 2^(lse_s - max lse);
// O = sum w_s O_s / sum w_s, LSE = (max lse + log2 sum w_s) * ln 2.  It is
// launched as a programmatic dependent of the split kernel: its set-up
// overlaps the split kernel's tail, and griddepcontrol.wait orders every
// record read after the split grid has completed.

constexpr int kCombineWarps = 8;

// Index of this head's first tile and its tile count.
__device__ __forceinline__ void head_tiles(const DecodeParams& p, int b, int h,
                                           long long* first, int* n) {
  if (p.lens == nullptr) {
    const int nb = tiles_of(p.Sk);
    *first = ((long long)b * p.H + h) * nb;
    *n = nb;
    return;
  }
  const int lane = threadIdx.x & 31;
  long long acc = 0;
  for (int b0 = 0; b0 < b; b0 += 32) {
    const int bb = b0 + lane;
    int c = bb < b ? tiles_of(cached_len(p, bb)) : 0;
#pragma unroll
    for (int s = 16; s > 0; s >>= 1) c += __shfl_xor_sync(0xffffffffu, c, s);
    acc += (long long)c * p.H;
  }
  const int nb = tiles_of(cached_len(p, b));
  *first = acc + (long long)h * nb;
  *n = nb;
}

// The warp whose range holds tile x (0 <= x < T).
__device__ __forceinline__ long long owner_warp(long long x, long long T, int W) {
  long long g = x * W / T;
  if (g > W - 1) g = W - 1;
  while (g > 0 && range_start(g, T, W) > x) --g;
  while (g + 1 < W && range_start(g + 1, T, W) <= x) ++g;
  return g;
}

template <int D, bool BF16>
__global__ void __launch_bounds__(kCombineWarps * 32)
    fattn_decode_combine_kernel(const DecodeParams p) {
  constexpr int kCols = D / 32;
  constexpr int kBatch = 4;  // records loaded together
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
  const bool live = row < (long long)p.B * p.H * p.Sq;
  int bh = 0, q = 0, n = 0;
  long long first = 0, g0 = 0, g1 = -1, T = 0;
  const int W = p.n_warps;
  if (live) {
    bh = (int)(row / p.Sq);
    q = (int)(row % p.Sq);
    head_tiles(p, bh / p.H, bh % p.H, &first, &n);
    if (n > 0) {
      T = total_tiles(p);
      g0 = owner_warp(first, T, W);
      g1 = owner_warp(first + n - 1, T, W);
    }
  }
  // Everything above only reads the inputs; the records come from the split
  // kernel, which may still be running when this grid starts early.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!live) return;
  // With at least one tile per warp every range is non-empty; otherwise a
  // warp between the head's first and last owner may hold no tile.
  const bool dense = T >= W;
  auto has_record = [&](long long g) {
    return dense || range_start(g, T, W) < range_start(g + 1, T, W);
  };

  float M = -INFINITY;
  for (long long g = g0 + lane; g <= g1; g += 32)
    if (has_record(g)) M = fmaxf(M, p.part_lse[(g + bh) * p.Sq + q]);
  M = warp_max(M);

  float acc[kCols];
#pragma unroll
  for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
  float wsum = 0.f;
  if (M != -INFINITY) {
    for (long long gb = g0; gb <= g1; gb += kBatch) {
      float ls[kBatch];
      float v[kBatch][kCols];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const long long g = gb + u;
        ls[u] = -INFINITY;
#pragma unroll
        for (int c = 0; c < kCols; ++c) v[u][c] = 0.f;
        if (g <= g1 && has_record(g)) {
          const long long rec = (g + bh) * p.Sq + q;
          ls[u] = p.part_lse[rec];
          const float* src = p.part_o + rec * D + lane * kCols;
          if constexpr (kCols == 4) {
            const float4 t = *reinterpret_cast<const float4*>(src);
            v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
          } else {
            const float2 t = *reinterpret_cast<const float2*>(src);
            v[u][0] = t.x; v[u][1] = t.y;
          }
        }
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float w = ls[u] == -INFINITY ? 0.f : ex2(ls[u] - M);
        wsum += w;
#pragma unroll
        for (int c = 0; c < kCols; ++c) acc[c] = fmaf(w, v[u][c], acc[c]);
      }
    }
  }
  const float inv = wsum > 0.f ? 1.0f / wsum : 0.f;
  uint16_t* dst = static_cast<uint16_t*>(p.o) + row * D + lane * kCols;
  if constexpr (kCols == 4) {
    const uint32_t lo = (uint32_t)to16<BF16>(acc[0] * inv) |
                        ((uint32_t)to16<BF16>(acc[1] * inv) << 16);
    const uint32_t hi = (uint32_t)to16<BF16>(acc[2] * inv) |
                        ((uint32_t)to16<BF16>(acc[3] * inv) << 16);
    *reinterpret_cast<uint2*>(dst) = make_uint2(lo, hi);
  } else {
    *reinterpret_cast<uint32_t*>(dst) = (uint32_t)to16<BF16>(acc[0] * inv) |
                                        ((uint32_t)to16<BF16>(acc[1] * inv) << 16);
  }
  if (lane == 0)
    p.lse[row] = wsum > 0.f ? (M + log2f(wsum)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace decode
}  // namespace fattn
