// Attention of up to 16 new queries per head against a key/value cache, with
// the score and P.V products on warp-level tensor-core MMAs (m16n8k16, fp32
// accumulation).  Same operation, partition, K/V tiles, records and merge
// kernel as fattn_decode_kernel (fattn_decode.cuh); only the per-tile
// arithmetic differs.
//
// Why warp-level MMAs here.  With Sq queries per head every cached K or V
// value takes part in 2 Sq multiply-adds, so beyond a few queries the CUDA
// cores, not HBM, set the pace (4 D Sq FMAs per cached key).  The smallest
// tcgen05 MMA has M = 64 rows, four times the 16 query rows at most served
// here, and its accumulator would sit in TMEM between the score product and
// the softmax; the m16n8k16 MMA has exactly 16 rows and leaves S, P and O in
// registers.  The path stays bound by HBM: at Sq = 16 it needs about 16 FLOP
// per byte read, ~0.1 PFLOP/s at full bandwidth.
//
// Per warp and 32-key tile (queries padded to 16 rows with zeros):
//   * S[16 x 32] = Q K^T: Q as A fragments (built once per head from shared
//     memory), K as B fragments straight from the swizzled TMA tile with
//     ldmatrix (a key row is a matrix row, so no transpose);
//   * online softmax per query row: a thread holds two rows (g, g + 8) and
//     eight keys of each; row maxima and sums combine across the four
//     threads of a quad;
//   * P is rounded to the input type and reused in registers as the A
//     fragments of O += P V (the accumulator layout of S is the A layout of
//     the next product); V as B fragments with ldmatrix.trans;
//   * cache rows at or past the cached length may hold anything (even NaN):
//     their scores are replaced by -inf, and in a tile that ends inside the
//     cache the V rows past the length are zeroed before P V, so 0 * NaN
//     never reaches O.
#pragma once

#include "fattn_decode.cuh"

namespace fattn {
namespace decode {

// Shared-memory plan of one CTA of the MMA variant: per warp two K/V slots,
// its 16 query rows, the slot barriers.
template <int D>
struct DecodeMmaLayout {
  static constexpr int kBoxes = D / kBoxCols;
  static constexpr int kTileBytes = kBoxes * kBoxBytes;
  static constexpr int kSlotBytes = 2 * kTileBytes;
  static constexpr int kQBytes = kMaxSq * D * 2;
  static constexpr int kPerWarp = 2 * kSlotBytes + kQBytes + 2 * 8;
  static constexpr int kWarpsFit = kSmemBudget / kPerWarp;
  static constexpr int kWarps = kWarpsFit > 8 ? 8 : kWarpsFit;
  static constexpr int kThreads = kWarps * 32;
  static constexpr int kSlotsOff = 0;  // 1024-aligned: slots first
  static constexpr int kQOff = kWarps * 2 * kSlotBytes;
  static constexpr int kBarOff = kQOff + kWarps * kQBytes;
  static constexpr int kSmemBytes = kBarOff + kWarps * 2 * 8 + 1024;
  static_assert(kWarps >= 4, "decode CTA too small");
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
};

// Four 8x8 16-bit matrices from shared memory; lane l gives the address of
// row l % 8 of matrix l / 8, and receives row l / 4, elements 2 (l % 4) and
// 2 (l % 4) + 1 of each (transposed with TRANS).
template <bool TRANS>
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1,
                                        uint32_t& r2, uint32_t& r3) {
  if constexpr (TRANS)
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
  else
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

// d += a (16 x 16, row-major fragments) * b (16 x 8, column-major fragments).
template <bool BF16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (BF16)
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  else
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Two fp32 values as a 16-bit pair (low half first), nearest-even.
template <bool BF16>
__device__ __forceinline__ uint32_t pack16x2(float lo, float hi) {
  return (uint32_t)to16<BF16>(lo) | ((uint32_t)to16<BF16>(hi) << 16);
}

// Shared-memory address of 16-byte chunk `chunk` (columns 8 chunk .. +7) of
// row `row` in a tile of D/64 swizzled boxes (32 rows x 128 bytes each).
__device__ __forceinline__ uint32_t tile_chunk(uint32_t tile, int row, int chunk) {
  return tile + (uint32_t)((chunk >> 3) * kBoxBytes + row * 128 + (((chunk & 7) ^ (row & 7)) << 4));
}

template <int D, bool BF16>
__global__ void __launch_bounds__(DecodeMmaLayout<D>::kThreads, 1)
    fattn_decode_mma_kernel(const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v,
                            const DecodeParams p) {
  using L = DecodeMmaLayout<D>;
  constexpr int kKS = D / 16;  // k-steps of the score product
  constexpr int kNT = D / 8;   // 8-column tiles of O
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g4 = lane >> 2;  // quad: rows g4 and g4 + 8 of the fragments
  const int t4 = lane & 3;   // thread in the quad: columns 2 t4, 2 t4 + 1
  const uint32_t s_base = ptx::smem_u32(smem);
  const uint32_t slot0 = s_base + L::kSlotsOff + warp * 2 * L::kSlotBytes;
  uint8_t* qbuf = smem + L::kQOff + warp * L::kQBytes;
  const uint32_t qaddr = s_base + L::kQOff + warp * L::kQBytes;
  const uint32_t bar0 = s_base + L::kBarOff + warp * 16;

  if (lane == 0) {
    ptx::mbar_init(bar0, 1);
    ptx::mbar_init(bar0 + 8, 1);
    ptx::fence_mbar_init();
    ptx::tma_prefetch_desc(&tm_k);
    ptx::tma_prefetch_desc(&tm_v);
  }
  __syncwarp();
  asm volatile("griddepcontrol.launch_dependents;");

  const int Sq = p.Sq;
  const long long T = total_tiles(p);
  const long long g = (long long)blockIdx.x * L::kWarps + warp;
  const long long t0 = range_start(g, T, p.n_warps);
  const long long t1 = range_start(g + 1, T, p.n_warps);
  if (t0 >= t1) return;
  const int n_tiles = (int)(t1 - t0);

  Cursor lc = find_batch(p, t0);
  Cursor cc = lc;
  long long lpos = t0 - lc.base;
  long long cpos = lpos;
  auto issue = [&](int r) {  // load tile t0 + r into slot r & 1
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
        ptx::tma_load_3d(slot + c * kBoxBytes, &tm_k, bar, c * kBoxCols, kt * kTileKeys, bh);
        ptx::tma_load_3d(slot + L::kTileBytes + c * kBoxBytes, &tm_v, bar, c * kBoxCols,
                         kt * kTileKeys, bh);
      }
    }
    ++lpos;
  };
  issue(0);
  if (n_tiles > 1) issue(1);

  int cur_bh = -1, cur_len = 0;
  // per row of this thread (i = 0: row g4, i = 1: row g4 + 8)
  float m[2], l32[2], l16[2];
  float o[kNT][4];
  uint32_t qa[kKS][4];
  auto reset = [&]() {
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      m[i] = kEmptyMax;
      l32[i] = 0.f;
      l16[i] = 0.f;
    }
#pragma unroll
    for (int n = 0; n < kNT; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[n][e] = 0.f;
  };
  auto quad_sum = [](float x) {
    x += __shfl_xor_sync(0xffffffffu, x, 1);
    x += __shfl_xor_sync(0xffffffffu, x, 2);
    return x;
  };
  // Partial record of the current head (same format as the CUDA-core kernel).
  auto flush = [&]() {
    const long long rec = g + cur_bh;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const float s32 = quad_sum(l32[i]);
      const float s16 = quad_sum(l16[i]);
      const int q = g4 + 8 * i;
      if (q < Sq) {
        const float inv = s16 > 0.f ? 1.0f / s16 : 0.f;
        float* dst = p.part_o + (rec * Sq + q) * D + 2 * t4;
#pragma unroll
        for (int n = 0; n < kNT; ++n)
          *reinterpret_cast<float2*>(dst + n * 8) =
              make_float2(o[n][2 * i] * inv, o[n][2 * i + 1] * inv);
        if (t4 == 0) p.part_lse[rec * Sq + q] = s32 > 0.f ? m[i] + __log2f(s32) : -INFINITY;
      }
    }
  };

  bool ok = true;
  int fail = 0;
  for (int r = 0; r < n_tiles; ++r) {
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
      // the head's Sq query rows, zero rows up to 16 (16-byte vectors)
      const uint4* src = reinterpret_cast<const uint4*>(
          static_cast<const uint8_t*>(p.q) + (size_t)bh * Sq * D * 2);
      uint4* dstq = reinterpret_cast<uint4*>(qbuf);
      for (int i = lane; i < kMaxSq * D / 8; i += 32)
        dstq[i] = i < Sq * D / 8 ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
      __syncwarp();
      // A fragments of Q: rows g4 / g4 + 8, columns 16 ks + 2 t4 (+ 8)
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
        const uint32_t r0 = qaddr + (uint32_t)(g4 * D * 2 + (ks * 16 + 2 * t4) * 2);
        const uint32_t r1 = r0 + 8 * D * 2;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(qa[ks][0]) : "r"(r0));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(qa[ks][1]) : "r"(r1));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(qa[ks][2]) : "r"(r0 + 16));
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(qa[ks][3]) : "r"(r1 + 16));
      }
    }
    const int key0 = kt * kTileKeys;
    const int nvalid = max(0, min(kTileKeys, cur_len - key0));

    const uint32_t slot = slot0 + (r & 1) * L::kSlotBytes;
    if (!ptx::mbar_wait_drain(bar0 + (r & 1) * 8, (r >> 1) & 1, p.timeout_ns)) {
      if (lane == 0)
        record_error(p.status, kErrPipelineTimeout, (kRoleDecode << 8) | (r & 1), blockIdx.x);
      ok = false;
      fail = r;
      break;
    }
    const uint32_t vtile = slot + L::kTileBytes;
    const bool zeroed = nvalid < kTileKeys;
    if (zeroed) {
      // V rows past the cached length may hold anything: zero them
      for (int i = lane; i < (kTileKeys - nvalid) * (D / 8); i += 32) {
        const int row = nvalid + i / (D / 8);
        const int chunk = i % (D / 8);
        asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};"
                     :: "r"(tile_chunk(vtile, row, chunk)), "r"(0u) : "memory");
      }
      __syncwarp();
    }

    // ---- S = Q K^T: four 8-key n-tiles
    float sc[4][4];
#pragma unroll
    for (int n = 0; n < 4; ++n)
#pragma unroll
      for (int e = 0; e < 4; ++e) sc[n][e] = 0.f;
    {
      // ldmatrix lane roles: matrix j = lane / 8 (bit 0: upper 8 columns of
      // the k-step, bit 1: second n-tile of the pair), row lane % 8
      const int jrow = lane & 7, jk = (lane >> 3) & 1, jn = lane >> 4;
#pragma unroll
      for (int ks = 0; ks < kKS; ++ks) {
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int key = (2 * np + jn) * 8 + jrow;
          uint32_t b0, b1, b2, b3;
          ldsm_x4<false>(tile_chunk(slot, key, 2 * ks + jk), b0, b1, b2, b3);
          mma16816<BF16>(sc[2 * np], qa[ks], b0, b1);
          mma16816<BF16>(sc[2 * np + 1], qa[ks], b2, b3);
        }
      }
    }

    // ---- online softmax per row; P rounded and packed as A fragments
    uint32_t pa[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const int q = g4 + 8 * i;
      const int last = p.causal ? cur_len - Sq + q : cur_len - 1;
      float t[8];
      float tmax = -INFINITY;
#pragma unroll
      for (int n = 0; n < 4; ++n)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int key = key0 + n * 8 + 2 * t4 + e;
          const bool valid = q < Sq && key <= last && key < cur_len;
          t[2 * n + e] = valid ? sc[n][2 * i + e] * p.scale_log2 : -INFINITY;
          tmax = fmaxf(tmax, t[2 * n + e]);
        }
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 1));
      tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 2));
      const float m_new = fmaxf(m[i], tmax);
      if (m_new != m[i]) {  // the same on the four threads of the quad
        const float alpha = ex2(m[i] - m_new);
        l32[i] *= alpha;
        l16[i] *= alpha;
#pragma unroll
        for (int n = 0; n < kNT; ++n) {
          o[n][2 * i] *= alpha;
          o[n][2 * i + 1] *= alpha;
        }
        m[i] = m_new;
      }
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const float p0 = ex2(t[2 * n] - m_new), p1 = ex2(t[2 * n + 1] - m_new);
        const uint32_t pk = pack16x2<BF16>(p0, p1);
        l32[i] += p0 + p1;
        l16[i] += from16<BF16>((uint16_t)(pk & 0xFFFFu)) + from16<BF16>((uint16_t)(pk >> 16));
        // A fragment of P V k-step n / 2: a0 / a1 rows g4 / g4 + 8, keys
        // 2 t4 (+1); a2 / a3 the same 8 keys further
        pa[n >> 1][(n & 1) * 2 + i] = pk;
      }
    }

    // ---- O += P V: two 16-key k-steps, D / 8 column tiles
    {
      const int jrow = lane & 7, jk = (lane >> 3) & 1, jn = lane >> 4;
#pragma unroll
      for (int ks = 0; ks < 2; ++ks) {
        const int key = ks * 16 + jk * 8 + jrow;
#pragma unroll
        for (int np = 0; np < kNT / 2; ++np) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4<true>(tile_chunk(vtile, key, 2 * np + jn), b0, b1, b2, b3);
          mma16816<BF16>(o[2 * np], pa[ks], b0, b1);
          mma16816<BF16>(o[2 * np + 1], pa[ks], b2, b3);
        }
      }
    }
    __syncwarp();  // every lane is done with this slot
    if (r + 2 < n_tiles) {
      // the zeroing wrote this slot through the generic proxy; order it
      // before the next TMA write into the slot
      if (zeroed && lane == 0) ptx::fence_proxy_async_smem();
      issue(r + 2);
    }
  }

  if (ok) {
    flush();
    return;
  }
  ptx::mbar_wait_drain(bar0 + (fail & 1) * 8, (fail >> 1) & 1, p.timeout_ns);
  if (fail + 1 < n_tiles)
    ptx::mbar_wait_drain(bar0 + ((fail + 1) & 1) * 8, ((fail + 1) >> 1) & 1, p.timeout_ns);
}

}  // namespace decode
}  // namespace fattn
