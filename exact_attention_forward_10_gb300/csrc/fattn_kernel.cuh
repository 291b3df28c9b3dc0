// Exact softmax-attention forward for sm_103a (GB300): O and the per-row LSE.
//
// What it computes (the plain definition, reached tile by tile):
//   O = softmax(scale * Q K^T [+ causal mask]) V,  LSE = m + ln(sum exp(s - m))
// with the online-softmax recurrence of "FlashAttention V2", section 3 (the
// unnormalised accumulator is rescaled by exp(m_old - m_new) per key tile and
// divided by the row sum once at the end) and the loop order of section 2
// (query tile outer, key/value tiles inner, O written once).  Causal masking
// keeps key <= query and stops at the diagonal tile; keys past S are removed
// ("FlashAttention-2 in an attention layer", Triton FA2 kernel).
//
// GB300 structure (one persistent CTA per SM):
//   * QT query tiles of 128 rows per work unit share every K/V tile.
//   * load warp:   TMA (128-byte swizzle) Q once per unit; K_j, V_j through an
//                  NS-stage mbarrier ring, in the order the MMAs use them.
//   * MMA warps:   one thread of a warp issues tcgen05.mma: S_i = Q_i K_j^T
//                  into TMEM (fp32, 128 lanes x 128 columns), then
//                  O_i += P_i V_j with P_i read from TMEM and O_i kept in TMEM
//                  for the whole unit.  One score buffer that the two query
//                  tiles fill in turn and P_i in columns of its own (TMEM:
//                  S 128, P 2 x 64 (16-bit) or 2 x 32 (E4M3), O 2 x D), so
//                  scores never wait for a P V; two warps issue, one the
//                  score MMAs and one the P V MMAs: a thread that issues MMAs
//                  stalls until the pipe has nearly run the ones before, so
//                  one warp's barrier waits would leave the pipe idle.  8-bit
//                  inputs: kind::f8f6f4 MMAs and P in E4M3.
//   * softmax warpgroup per query tile: thread r owns row r (TMEM lane r):
//                  tcgen05.ld of its score row, mask, exp2 against a lazily
//                  moved reference maximum with the scale folded into one
//                  FFMA, row sums, P to TMEM; when a row's reference moves,
//                  the same warp rescales that row of O_i in TMEM.
//                  (m, l) live in registers; no shuffles are needed because a
//                  row never leaves its thread.
//   * epilogue warpgroup: one 1/l per row, cast to 16-bit, vector stores of
//                  O and the LSE, while the next unit's tiles run.
// Every wait is bounded; a timeout records an error in the device status
// block and the CTA unwinds (frees TMEM, waits for its own copies) instead of
// hanging.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>
#include <type_traits>

#include "fattn_status.h"
#include "ptx.cuh"

// Optional timeline hook: FATTN_TRACE_EV(round, kv_tile, event) records one
// event of the pipeline when an instrumented build defines it; the product
// build compiles it to nothing.  Events of a whole unit use the key-tile
// slot kTraceUnit.
#ifndef FATTN_TRACE_EV
#define FATTN_TRACE_INIT ((void)0)
#define FATTN_TRACE_EV(round, kv_tile, event) ((void)0)
#endif

// P V issued in two halves of the keys (the first half while the softmax
// still works on the second) when P overwrites S (FATTN_SHARED_S 0) with
// 8-bit inputs; a build-time choice (1: on).  Measured in that layout on the
// B2 H16 S8192 D128 workloads: E4M3 1436 / 1367 TF against 1292 / 1247 in
// whole rows; bf16 1335 / 1278 against 1491 / 1412, so 16-bit inputs keep
// whole rows.
#ifndef FATTN_HALF_PV
#define FATTN_HALF_PV 1
#endif

// Head dim 128: both query tiles take turns in one TMEM score buffer and
// each keeps its P in columns of its own (1: on), so the scores of the next
// key tile never wait for the P V of this one; otherwise (0) P overwrites S
// in a score buffer per query tile and one warp issues all MMAs.  A
// build-time choice; measured on one GB300, B2 H16 S8192: bf16 1622-1625 /
// 1545-1550 TF (maximum first) and 1766-1777 / 1550-1608 (fused) against
// 1525 / 1419-1428, E4M3 1850 / 1780-1790 against 1429 / 1355.
#ifndef FATTN_SHARED_S
#define FATTN_SHARED_S 1
#endif

// Head dim 64: a score buffer per query tile (1) or the shared buffer of
// head dim 128 (0, default: the tiles' softmax warpgroups then alternate
// instead of running side by side, and one's waits overlap the other's
// exponents; B2 H16 S8192 bf16 1110 / 1072 TF against 1002 / 958); a
// build-time choice.
#ifndef FATTN_D64_SCORE_PER_TILE
#define FATTN_D64_SCORE_PER_TILE 0
#endif

// 16-bit inputs, shared score buffer: a row's later key tiles exponentiate
// against the reference chosen after the tile before, taking the tile's
// maximum in the same pass; a tile whose maximum passed that reference by
// more than kRescaleLog2 moves it for the next tile (its own P, in the old
// frame, stays below 2^kOverflowLog2), and only a tile whose 16-bit P could
// overflow is redone.  Otherwise each tile takes its maximum first.  Bits:
// 0 head dim 64, 1 head dim 128 non-causal, 2 head dim 128 causal, 3 fp16
// inputs too (else bf16 only).  A build-time choice; the default, bf16 head
// dim 128 non-causal, is where it measured faster (B2 H16 S8192 bf16 at
// 2070 MHz: 1797-1813 TF against 1611-1639 on N(0,1) inputs; 1521-1538
// against 1703-1711 with Q, K x 4; causal 1420-1477 against 1543-1553; head
// dim 64 945-1020 against 1050-1124; fp16 with Q, K x 4, where 2^15 bounds
// the lag, 1267-1274 against 1687-1690).
#ifndef FATTN_FUSED_MAX
#define FATTN_FUSED_MAX 2
#endif

// Roles whose barrier waits spin instead of suspending (bit 0: load warp,
// bit 1: MMA warp, bit 2: softmax warps waiting for scores); a build-time
// choice.
#ifndef FATTN_SPIN_ROLES
#define FATTN_SPIN_ROLES 0
#endif

namespace fattn {

constexpr int kTraceUnit = 71;
constexpr int kUnitRing = 4;  // unit indices the load warp may publish ahead
constexpr bool kSpinLoad = (FATTN_SPIN_ROLES & 1) != 0;
constexpr bool kSpinMma = (FATTN_SPIN_ROLES & 2) != 0;
constexpr bool kSpinSoftmax = (FATTN_SPIN_ROLES & 4) != 0;
constexpr int kBM = 128;  // query rows per tile (one TMEM lane each)
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kSwizzleChunkCols = 64;           // 128 bytes of 16-bit values
constexpr int kChunkBytes = kBM * 128;          // one [128 rows, 64 cols] chunk
constexpr uint32_t kTmemCols = 512;
// A row's reference maximum moves only when the new maximum exceeds it by
// more than this (log2 units), so every p = exp2(s*c - m) stays <= 2^8.
constexpr float kRescaleLog2 = 8.0f;
// With the maximum taken during the exponent pass (FATTN_FUSED_MAX) a tile's
// P is computed against the previous tile's reference; it is redone only
// when a weight could pass 2^kOverflowLog2: 2^15 < 65504 for fp16 P; bf16
// P, whose range is that of fp32, is redone past 2^64 (O and l, fp32, stay
// far from overflow: 128 keys x 2^64 x |v|).
template <bool BF16>
constexpr float kOverflowLog2 = BF16 ? 64.0f : 15.0f;

struct FwdParams {
  void* o;            // [BH, S, D] 16-bit
  float* lse;         // [BH, S] fp32
  int* status;        // device status block (kStatusWords ints)
  int S;
  int BH;
  int n_kv_tiles;     // ceil(S / kBN)
  int n_units;        // work units per head: ceil(S / (kBM * QT))
  int total_units;    // BH * n_units
  float scale_log2;   // scale * log2(e) (FP8: times the Q and K scales)
  float o_scale;      // multiplies O in the epilogue (FP8: the V scale; else 1)
  unsigned long long timeout_ns;
  // Causal masks: work units are handed out at run time from sched[0] (the
  // next unit; sched[1] counts the CTAs done, and the last one resets both
  // to 0), in groups of group_heads heads (longest units first within a
  // group) so the K/V of the heads in flight stay in L2.  With sched null
  // each CTA takes the units of its own slots of the snake order instead
  // (group_heads then equal to BH: longest first over every head).
  int* sched;
  int group_heads;
};

// EB: bytes per input element (2: fp16/bf16; 1: E4M3).  A swizzle chunk is
// 128 bytes of a row: 64 16-bit or 128 8-bit columns.
template <int D, int QT, int NS, int EB = 2>
struct FwdLayout {
  static_assert(D == 64 || D == 128, "head dim");
  static_assert(EB == 2 || (EB == 1 && D == 128), "8-bit inputs: head dim 128");
  static constexpr int kTileBytes = kBM * D * EB;
  static constexpr int kChunkCols = 128 / EB;
  static constexpr int kChunks = D / kChunkCols;
  static constexpr int kK = 32 / EB;  // K elements per MMA (32 bytes of a row)
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + QT * kTileBytes;
  static constexpr int kBars = kKV + NS * kTileBytes;
  // barrier slots (8 bytes each)
  static constexpr int bQFull = 0;
  static constexpr int bQEmpty = bQFull + QT;
  static constexpr int bKVFull = bQEmpty + QT;
  static constexpr int bKVEmpty = bKVFull + NS;
  static constexpr int bSFull = bKVEmpty + NS;
  static constexpr int bPFull = bSFull + QT;
  static constexpr int bSFree = bPFull + QT;
  static constexpr int bStats = bSFree + QT;
  static constexpr int bPVDone = bStats + QT;
  static constexpr int bOEmpty = bPVDone + QT;
  static constexpr int bDrain = bOEmpty + QT;
  static constexpr int bP1Full = bDrain + 1;         // first half of P_i ready
  static constexpr int bPV1Done = bP1Full + QT;      // its P V done
  static constexpr int bUnitFull = bPV1Done + QT;    // [kUnitRing] unit index published
  static constexpr int bUnitEmpty = bUnitFull + kUnitRing;  // [kUnitRing] read by all
  static constexpr int kNumBars = bUnitEmpty + kUnitRing;
  static constexpr int kMisc = kBars + kNumBars * 8;   // tmem base, abort flag
  static constexpr int kRowL = kMisc + 16;             // float [QT][128]
  static constexpr int kRowM = kRowL + QT * kBM * 4;   // float [QT][128]: LSE
  static constexpr int kUnitSlots = kRowM + QT * kBM * 4;  // int [kUnitRing]
  static constexpr int kEnd = kUnitSlots + kUnitRing * 4;
  // The dynamic shared memory base must be 1024-byte aligned (128-byte
  // swizzle atoms); the kernel checks it instead of reserving slack.
  static constexpr int kSmemBytes = kEnd;
  // TMEM columns.  When they fit (D = 64), P_i gets its own 64 columns, so
  // S_i(j+1) can be computed while the softmax of tile j still runs; else P_i
  // overwrites the first 64 columns of S_i.
  static constexpr bool kSepP = FATTN_D64_SCORE_PER_TILE != 0 &&
                                QT * (128 + 64) + QT * D <= (int)kTmemCols;
  // TMEM columns of one query tile's P: 128 keys, two 16-bit or four 8-bit
  // weights per column.
  static constexpr int kPCols = 128 * EB / 4;
  // Otherwise: one score buffer (columns 0-127) that the query tiles fill in
  // turn, P_i in columns of its own, then the O_i.
  static constexpr bool kShareS = !kSepP && FATTN_SHARED_S != 0 &&
                                  128 + QT * kPCols + QT * D <= (int)kTmemCols;
  // With P in columns of its own, scores and P V depend on each other only
  // through the softmax: one warp issues the score MMAs, another the P V
  // MMAs, and each one's waits overlap the other's MMAs in the pipe.
  static constexpr bool kDualMma = kSepP || kShareS;

  // P over S with 8-bit inputs: P V in two halves of the keys (FATTN_HALF_PV)
  static constexpr bool kHalfPV = FATTN_HALF_PV != 0 && !kSepP && !kShareS && EB == 1;
  __host__ __device__ static constexpr uint32_t colS(int i) {
    return kShareS ? 0u : 128u * i;
  }
  __host__ __device__ static constexpr uint32_t colP(int i) {
    return kSepP ? 128u * QT + 64u * i : kShareS ? 128u + (uint32_t)kPCols * i : colS(i);
  }
  __host__ __device__ static constexpr uint32_t colO(int i) {
    return kShareS ? 128u + (uint32_t)kPCols * QT + D * i
                   : 128u * QT + (kSepP ? 64u * QT : 0u) + D * i;
  }
  static_assert(colO(QT) <= kTmemCols, "TMEM budget");
};

template <int QT>
struct FwdWarps {
  static constexpr int kSoftmax0 = 0;          // warps [0, 4 QT)
  static constexpr int kCorrection0 = 4 * QT;  // 4 warps
  static constexpr int kMma = 4 * QT + 4;
  static constexpr int kLoad = 4 * QT + 5;
  static constexpr int kMma2 = 4 * QT + 6;  // P V issuer when S and P V issue apart
  static constexpr int kNumWarps = 4 * QT + 8;  // whole warpgroups
  static constexpr int kThreads = 32 * kNumWarps;
  // Registers per thread after the per-warpgroup split (QT == 2 only): the
  // softmax warpgroups hold a 128-float score row; the shares add up to the
  // 128 per thread the 512-thread block is launched with.
  static constexpr int kRegSoftmax = 176;
  static constexpr int kRegCorrection = 80;
  static constexpr int kRegOther = 80;
  static_assert(QT != 2 || 2 * kRegSoftmax + kRegCorrection + kRegOther ==
                               4 * (65536 / kThreads),
                "register split must equal the launch allocation");
};

// Keys [kFirst, kFirst + kCount) of a score row (an exponent pass over them).
template <int FIRST, int COUNT>
struct KeyRange {
  static constexpr int kFirst = FIRST;
  static constexpr int kCount = COUNT;
};

struct Unit {
  int bh;
  int q_row0;
  int n_max;
};

// Causal order over head groups: ng = ceil(BH / G) groups, the first
// BH - ng (G - 1) of them of G heads and the rest of G - 1 (the host passes
// G = ceil(BH / groups), so no group is more than one head smaller than
// another; a small last group would hand its longest units out last).
// Unit t of the order -> its rank within its head (longest first) and head.
struct GroupPos {
  int rank;
  int bh;
};
__device__ __forceinline__ GroupPos group_position(int t, int BH, int G, int nu) {
  const int ng = (BH + G - 1) / G;
  const int big = BH - ng * (G - 1);      // groups of G heads (all of them when G == 1)
  const int big_units = big * G * nu;
  GroupPos gp;
  if (t < big_units) {
    const int g = t / (G * nu);
    const int r = t - g * G * nu;
    gp.rank = r / G;
    gp.bh = g * G + r % G;
  } else {
    const int t2 = t - big_units;         // here G >= 2
    const int g = t2 / ((G - 1) * nu);
    const int r = t2 - g * (G - 1) * nu;
    gp.rank = r / (G - 1);
    gp.bh = big * G + g * (G - 1) + r % (G - 1);
  }
  return gp;
}

// Work unit t -> (head, first query row, key-tile counts per query tile).
// Causal units go longest first (the last query tiles need the most keys):
// GROUPED, within groups of group_heads heads; else over every head.
// Non-causal units of one head are adjacent, so CTAs running together share
// that head's K/V in L2.
template <int QT, bool CAUSAL, bool GROUPED>
__device__ __forceinline__ Unit decode_unit(int t, const FwdParams& p,
                                            int (&n)[QT]) {
  Unit w;
  int u;
  if (CAUSAL && !GROUPED) {
    u = p.n_units - 1 - t / p.BH;
    w.bh = t % p.BH;
  } else if (CAUSAL) {
    const GroupPos gp = group_position(t, p.BH, p.group_heads, p.n_units);
    u = p.n_units - 1 - gp.rank;
    w.bh = gp.bh;
  } else {
    u = t % p.n_units;
    w.bh = t / p.n_units;
  }
  w.q_row0 = u * kBM * QT;
  w.n_max = 0;
#pragma unroll
  for (int i = 0; i < QT; ++i) {
    const int q0 = w.q_row0 + kBM * i;
    int ni;
    if (q0 >= p.S)
      ni = 0;
    else if (CAUSAL)
      ni = q0 / kBN + 1;  // tiles up to and including the diagonal
    else
      ni = p.n_kv_tiles;
    n[i] = ni;
    w.n_max = ni > w.n_max ? ni : w.n_max;
  }
  return w;
}

// Round k of the persistent loop: CTA g takes unit k*G + g in even rounds and
// k*G + (G-1-g) in odd rounds (a snake over the longest-first order), which
// evens out the causal work per CTA.  Returns a value >= total when this CTA
// has nothing in round k.
__device__ __forceinline__ int unit_of_round(int k) {
  const int G = (int)gridDim.x;
  const int g = (int)blockIdx.x;
  return k * G + ((k & 1) ? (G - 1 - g) : g);
}

__device__ __forceinline__ void raise_error(const FwdParams& p,
                                            volatile int* abort_flag, int code,
                                            int role, int bar) {
  if (atomicCAS(p.status, 0, code) == 0) {
    p.status[1] = (role << 8) | bar;
    p.status[2] = (int)blockIdx.x;
  }
  *abort_flag = 1;
}

// max of three floats in one instruction
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (BF16) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// The two fp32 values of a packed 16-bit pair (low half first).
template <bool BF16>
__device__ __forceinline__ float2 unpack2(uint32_t v) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(v << 16), __uint_as_float(v & 0xFFFF0000u));
  } else {
    __half2 h = *reinterpret_cast<__half2*>(&v);
    return __half22float2(h);
  }
}

// Four fp32 values to E4M3 (nearest-even, saturating at 448), packed so that
// byte j holds value j (the order a kind::f8f6f4 MMA reads K from TMEM).
__device__ __forceinline__ uint32_t pack4_e4m3(float p0, float p1, float p2, float p3) {
  uint16_t lo, hi;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(p1), "f"(p0));
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(p3), "f"(p2));
  return (uint32_t)lo | ((uint32_t)hi << 16);
}

// The four E4M3 values of a packed word (as pack4_e4m3 makes it), summed
// into two fp32 accumulators: two f16 pairs, one packed add, two
// mixed-precision FMAs.
__device__ __forceinline__ void add4_e4m3(uint32_t w, float& acc0, float& acc1) {
  uint32_t h01, h23, h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h01) : "h"((uint16_t)(w & 0xFFFFu)));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h23) : "h"((uint16_t)(w >> 16)));
  asm("add.rn.f16x2 %0, %1, %2;" : "=r"(h) : "r"(h01), "r"(h23));
  asm("{\n\t.reg .b16 lo, hi, one;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "mov.b16 one, 0x3C00;\n\t"
      "fma.rn.f32.f16 %0, lo, one, %0;\n\t"
      "fma.rn.f32.f16 %1, hi, one, %1;\n\t}"
      : "+f"(acc0), "+f"(acc1) : "r"(h));
}

// BF16: the output type (and, for 16-bit inputs, the input type).  FP8:
// E4M3 inputs with per-tensor scales (folded into scale_log2 and o_scale),
// scores and P V on kind::f8f6f4 MMAs, P rounded to E4M3.
template <int D, int QT, int NS, bool CAUSAL, bool BF16, bool FP8 = false>
__global__ void __launch_bounds__(FwdWarps<QT>::kThreads, 1)
    fattn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q,
                     const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_v,
                     const FwdParams p) {
  using L = FwdLayout<D, QT, NS, FP8 ? 1 : 2>;
  using W = FwdWarps<QT>;
  // Causal units at D = 128 (16-bit and E4M3) may be handed out at run time
  // from the launch's counter (p.sched, set by the host when the K and V of
  // all heads exceed what L2 keeps), in head groups; otherwise, and in the
  // other kernels, each CTA takes a static snake over a fixed order.
  constexpr bool kRunTimeCapable = CAUSAL && D == 128;
  const bool run_time_units = kRunTimeCapable && p.sched != nullptr;
  constexpr bool kFusedMax =
      !FP8 && (L::kSepP || L::kShareS) && (BF16 || (FATTN_FUSED_MAX & 8) != 0) &&
      (FATTN_FUSED_MAX & (D == 64 ? 1 : D != 128 ? 0 : CAUSAL ? 4 : 2)) != 0;
  // warps that read the unit sequence: MMA issuers, softmax, epilogue
  constexpr int kUnitReaders = 4 * QT + 4 + (L::kDualMma ? 2 : 1);
  constexpr int kUnitEnd = -2;
  static_assert(!FP8 || !L::kSepP, "8-bit inputs use the layout where P overwrites S");
  extern __shared__ uint8_t smem_raw[];

  const uint32_t base = ptx::smem_u32(smem_raw);
  if (base & 1023u) {
    // Not 1024-byte aligned: report instead of touching shared memory.
    if (threadIdx.x == 0 && atomicCAS(p.status, 0, kErrLaunch) == 0) {
      p.status[1] = 0;
      p.status[2] = (int)blockIdx.x;
    }
    // this CTA still counts as done, so the launch's unit counter is reset
    if (run_time_units && threadIdx.x == 0 &&
        atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
    return;
  }
  uint8_t* const smem = smem_raw;
  const uint32_t sQ = base + L::kQ;
  const uint32_t sKV = base + L::kKV;
  const uint32_t bars = base + L::kBars;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  float* const sRowL = reinterpret_cast<float*>(smem + L::kRowL);
  float* const sRowM = reinterpret_cast<float*>(smem + L::kRowM);

  auto bar = [&](int slot) -> uint32_t { return bars + 8u * slot; };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = p.timeout_ns;
  FATTN_TRACE_INIT;

  if (threadIdx.x == 0) {
    for (int i = 0; i < QT; ++i) {
      ptx::mbar_init(bar(L::bQFull + i), 1);
      ptx::mbar_init(bar(L::bQEmpty + i), 1);
      ptx::mbar_init(bar(L::bSFull + i), 1);
      ptx::mbar_init(bar(L::bPFull + i), kBM);
      ptx::mbar_init(bar(L::bSFree + i), kBM);
      ptx::mbar_init(bar(L::bStats + i), kBM);
      ptx::mbar_init(bar(L::bPVDone + i), 1);
      ptx::mbar_init(bar(L::bOEmpty + i), kBM);
      ptx::mbar_init(bar(L::bP1Full + i), kBM);
      ptx::mbar_init(bar(L::bPV1Done + i), 1);
    }
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(bar(L::bKVFull + s), 1);
      ptx::mbar_init(bar(L::bKVEmpty + s), 1);
    }
    ptx::mbar_init(bar(L::bDrain), L::kDualMma ? 2 : 1);
    for (int r = 0; r < kUnitRing; ++r) {
      ptx::mbar_init(bar(L::bUnitFull + r), 1);
      ptx::mbar_init(bar(L::bUnitEmpty + r), kUnitReaders);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == W::kMma) {
    ptx::tmem_alloc(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // The unit of this CTA's k-th round.  Run-time units (causal masks with a
  // counter): the load warp takes units from the launch's counter and
  // publishes them through a small ring (a value >= total_units ends the
  // sequence).  Otherwise the static snake, where a round may have no unit
  // for this CTA (a value >= total_units).  kUnitEnd ends the sequence; -1
  // is an error.
  int* const unit_slots = reinterpret_cast<int*>(smem + L::kUnitSlots);
  auto next_unit = [&](int k, int role) -> int {
    if (run_time_units) {
      const int slot = k % kUnitRing;
      bool w_ok = ptx::mbar_wait(bar(L::bUnitFull + slot), (k / kUnitRing) & 1, abort_flag, tmo);
      w_ok = __all_sync(0xffffffffu, w_ok);
      if (!w_ok) {
        if (lane == 0) raise_error(p, abort_flag, kErrPipelineTimeout, role, L::bUnitFull + slot);
        return -1;
      }
      const int t = *reinterpret_cast<volatile int*>(unit_slots + slot);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(L::bUnitEmpty + slot));
      return t >= p.total_units ? kUnitEnd : t;
    } else {
      if (k * (int)gridDim.x >= p.total_units) return kUnitEnd;
      return unit_of_round(k);
    }
  };

  // The register split is stated at the top of each role's branch so it
  // dominates that role's code.
  if (warp >= W::kMma) {
    if constexpr (QT == 2) ptx::setmaxnreg_dec<W::kRegOther>();
  }

  if (warp == W::kLoad) {
    // ------------------------------------------------------------ load warp
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_q);
      ptx::tma_prefetch_desc(&tm_k);
      ptx::tma_prefetch_desc(&tm_v);
      uint32_t kv_idx = 0, kv_ph = 0;
      int q_uses[QT];
      for (int i = 0; i < QT; ++i) q_uses[i] = 0;
      uint32_t kv_filled = 0, kv_fill_ph = 0;  // per stage: ever filled, parity
      bool ok = true;
      // Run-time units: a CTA's first unit is its own index (the first
      // gridDim.x units of the order), later ones come from the launch's
      // counter.
      int t_next = (int)blockIdx.x < p.total_units ? (int)blockIdx.x : p.total_units;
      for (int k = 0; ok; ++k) {
        int t;
        if (run_time_units) {
          // publish this unit to the other roles
          t = t_next;
          const int slot = k % kUnitRing;
          if (k >= kUnitRing &&
              !ptx::mbar_wait<kSpinLoad>(bar(L::bUnitEmpty + slot), ((k / kUnitRing) - 1) & 1,
                                         abort_flag, tmo)) {
            raise_error(p, abort_flag, kErrPipelineTimeout, kRoleLoad, L::bUnitEmpty + slot);
            ok = false;
            break;
          }
          *reinterpret_cast<volatile int*>(unit_slots + slot) = t;
          ptx::mbar_arrive(bar(L::bUnitFull + slot));
          if (t >= p.total_units) break;
        } else {
          if (k * (int)gridDim.x >= p.total_units) break;
          t = unit_of_round(k);
          if (t >= p.total_units) continue;
        }
        int n[QT];
        const Unit w = decode_unit<QT, CAUSAL, kRunTimeCapable>(t, p, n);
        for (int i = 0; ok && i < QT; ++i) {
          if (n[i] == 0) continue;
          if (q_uses[i] > 0 &&
              !ptx::mbar_wait<kSpinLoad>(bar(L::bQEmpty + i), (q_uses[i] - 1) & 1, abort_flag, tmo)) {
            raise_error(p, abort_flag, kErrPipelineTimeout, kRoleLoad, L::bQEmpty + i);
            ok = false;
            break;
          }
          const uint32_t qb = bar(L::bQFull + i);
          FATTN_TRACE_EV(k, kTraceUnit, 13 + i);
          ptx::mbar_arrive_expect_tx(qb, L::kTileBytes);
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c)
            ptx::tma_load_3d(sQ + i * L::kTileBytes + c * kChunkBytes, &tm_q, qb,
                             c * L::kChunkCols, w.q_row0 + kBM * i, w.bh);
          ++q_uses[i];
        }
        // Items in the order the MMA warps consume them: K_j, V_j; when
        // scores and P V issue apart, K_0, then K_{j+1} before V_j (the next
        // tile's scores are issued while this tile's softmax runs), so the
        // slots are released about in load order.
        int taken = 0;  // causal: the counter's value for the next unit
        for (int it = 0; ok && it < 2 * w.n_max; ++it) {
          // The next unit is taken as this unit's last key tile is loaded:
          // the CTAs that will be free first take the longest units left;
          // the atomic's result is first used after the loop, so its latency
          // passes under the last copies.
          if (run_time_units && it == 2 * w.n_max - 2) taken = atomicAdd(p.sched, 1);
          int j, kv;
          if constexpr (L::kDualMma) {
            if (it == 0) {
              j = 0;
              kv = 0;
            } else if (it == 2 * w.n_max - 1) {
              j = w.n_max - 1;
              kv = 1;
            } else {
              j = (it - 1) / 2 + ((it & 1) ? 1 : 0);
              kv = (it & 1) ? 0 : 1;
            }
          } else {
            j = it / 2;
            kv = it & 1;
          }
          {
            if (kv == 1) FATTN_TRACE_EV(k, j, 7);
            if (!ptx::mbar_wait<kSpinLoad>(bar(L::bKVEmpty + kv_idx), kv_ph ^ 1u, abort_flag, tmo)) {
              raise_error(p, abort_flag, kErrPipelineTimeout, kRoleLoad, L::bKVEmpty + kv_idx);
              ok = false;
              break;
            }
            const uint32_t fb = bar(L::bKVFull + kv_idx);
            ptx::mbar_arrive_expect_tx(fb, L::kTileBytes);
#pragma unroll
            for (int c = 0; c < L::kChunks; ++c)
              ptx::tma_load_3d(sKV + kv_idx * L::kTileBytes + c * kChunkBytes,
                               kv == 0 ? &tm_k : &tm_v, fb, c * L::kChunkCols,
                               j * kBN, w.bh);
            FATTN_TRACE_EV(k, j, 5 + kv);
            kv_filled |= 1u << kv_idx;
            kv_fill_ph = (kv_fill_ph & ~(1u << kv_idx)) | (kv_ph << kv_idx);
            if (++kv_idx == NS) {
              kv_idx = 0;
              kv_ph ^= 1u;
            }
          }
        }
        if (run_time_units) {
          t_next = (int)gridDim.x + taken;
          if (t_next > p.total_units) t_next = p.total_units;
        }
      }
      // Never leave with copies in flight into this CTA's shared memory.
      for (int s = 0; s < NS; ++s)
        if (kv_filled & (1u << s))
          ptx::mbar_wait_drain(bar(L::bKVFull + s), (kv_fill_ph >> s) & 1u, tmo);
      for (int i = 0; i < QT; ++i)
        if (q_uses[i] > 0)
          ptx::mbar_wait_drain(bar(L::bQFull + i), (q_uses[i] - 1) & 1, tmo);
    }
  } else if (warp == W::kMma || (L::kDualMma && warp == W::kMma2)) {
    // ------------------------------------------------------------ MMA warps
    // Each MMA warp runs its role converged, so its counters and descriptors
    // stay warp-uniform; one elected lane issues each tcgen05 instruction.
    // The issuing thread stalls until the tensor pipe has nearly finished
    // the MMAs before, so what one warp does between two MMA groups (barrier
    // waits, commits) is tensor idle time unless another warp's MMAs are
    // queued meanwhile: with P in columns of its own, warp kMma issues the
    // score MMAs and warp kMma2 the P V MMAs.
    const bool s_role = warp == W::kMma;  // dual issue: this warp's share
    {
      constexpr uint32_t kIdS = FP8 ? ptx::idesc_e4m3(kBM, kBN, 0, 0)
                                    : ptx::idesc_f16(BF16 ? 1 : 0, kBM, kBN, 0, 0);
      constexpr uint32_t kIdPV = FP8 ? ptx::idesc_e4m3(kBM, D, 0, 1)
                                     : ptx::idesc_f16(BF16 ? 1 : 0, kBM, D, 0, 1);
      uint32_t kv_idx = 0, kv_ph = 0;
      uint32_t kv_item = 0;  // separate-P layouts: ring index of the next unit's K_0
      uint32_t s_total = 0;  // shared score buffer: S MMAs issued into it so far
      int q_uses[QT], p_cnt[QT], oe_cnt[QT], used[QT], s_issued[QT];
      for (int i = 0; i < QT; ++i) q_uses[i] = p_cnt[i] = oe_cnt[i] = used[i] = s_issued[i] = 0;
      bool ok = true;

      auto wait_or_fail = [&](int slot, uint32_t parity) -> bool {
        bool w_ok = ptx::mbar_wait<kSpinMma>(bar(slot), parity, abort_flag, tmo);
        w_ok = __all_sync(0xffffffffu, w_ok);
        if (!w_ok && lane == 0) raise_error(p, abort_flag, kErrPipelineTimeout, kRoleMma, slot);
        return w_ok;
      };
      auto commit = [&](int slot) {
        if (ptx::elect_one()) ptx::mma_commit(bar(slot));
      };
      auto next_kv = [&](uint32_t& slot) -> bool {
        if (!wait_or_fail(L::bKVFull + kv_idx, kv_ph)) return false;
        slot = kv_idx;
        if (++kv_idx == NS) {
          kv_idx = 0;
          kv_ph ^= 1u;
        }
        ptx::tc_fence_after();
        return true;
      };
      // Descriptors: one constant high word (SBO = 1024: eight 128-byte rows
      // per swizzle atom) and low words stepped by immediates.
      constexpr uint32_t kHi = ptx::desc_sw128_hi(1024);
      constexpr uint32_t kTileLo = L::kTileBytes >> 4;  // one K/V stage
      const uint32_t q_lo = ptx::desc_sw128_lo(sQ, 16);
      const uint32_t k_lo = ptx::desc_sw128_lo(sKV, 16);
      const uint32_t v_lo = ptx::desc_sw128_lo(sKV, kChunkBytes);  // LBO: next 64 columns
      // S_i = Q_i K^T: M = 128, N = 128, K = D in steps of kK (32 bytes of a
      // 128-byte swizzled row; the next 128 bytes of the row are one chunk
      // further).
      auto issue_s = [&](int i, uint32_t k_slot) {
        const uint32_t d = tmem + L::colS(i);
        const uint32_t qa = q_lo + i * kTileLo;
        const uint32_t kb = k_lo + k_slot * kTileLo;
        if (!ptx::elect_one()) return;
#pragma unroll
        for (int kk = 0; kk < D / L::kK; ++kk) {
          const uint32_t off = ((kk / 4) * kChunkBytes + (kk % 4) * 32) >> 4;
          if (kk == 0)
            ptx::mma_ss_lohi<0, FP8>(d, qa + off, kb + off, kHi, kIdS, 0u);
          else
            ptx::mma_ss_lohi<1, FP8>(d, qa + off, kb + off, kHi, kIdS, 1u);
        }
      };
      // O_i += P_i V: M = 128, N = D, K = 128 keys in steps of kK.  P_i is
      // read from TMEM (two 16-bit or four 8-bit values per column: 8
      // columns per step); V is MN-major, each step kK key rows further.
      // part: 0 all keys, 1 the first half, 2 the second half (accumulating).
      auto issue_pv = [&](int i, uint32_t v_slot, bool acc, int part = 0) {
        constexpr int kSteps = kBN / L::kK;
        const uint32_t d = tmem + L::colO(i);
        const uint32_t a = tmem + L::colP(i);
        const uint32_t vb = v_lo + v_slot * kTileLo;
        if (!ptx::elect_one()) return;
        const int k0 = part == 2 ? kSteps / 2 : 0;
        const int k1 = part == 1 ? kSteps / 2 : kSteps;
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
          if (kk < k0 || kk >= k1) continue;
          if (kk == 0)
            ptx::mma_ts_lohi<0, FP8>(d, a, vb, kHi, kIdPV, acc ? 1u : 0u);
          else
            ptx::mma_ts_lohi<1, FP8>(d, a + kk * 8, vb + kk * ((L::kK * 128) >> 4), kHi,
                                     kIdPV, 1u);
        }
      };

      for (int k = 0; ok; ++k) {
        const int t = next_unit(k, kRoleMma);
        if (t == kUnitEnd) break;
        if (t < 0) {
          ok = false;
          break;
        }
        if (t >= p.total_units) continue;
        int n[QT];
        const Unit w = decode_unit<QT, CAUSAL, kRunTimeCapable>(t, p, n);
        if (!L::kDualMma || s_role)
          for (int i = 0; ok && i < QT; ++i)
            if (n[i] > 0) {
              ok = wait_or_fail(L::bQFull + i, q_uses[i] & 1);
              ++q_uses[i];
              FATTN_TRACE_EV(k, kTraceUnit, 15 + i);
            }
        if (!ok) break;
        if constexpr (L::kDualMma) {
          // K/V items in the load warp's order K_0, K_1, V_0, K_2, V_1, ...,
          // V_{n-1} (K_{j+1} before V_j: scores run ahead of P V), addressed
          // by their index in the ring.
          const uint32_t base = kv_item;  // ring index of this unit's K_0
          kv_item += 2u * (uint32_t)w.n_max;
          auto wait_item = [&](uint32_t idx) -> bool {
            const uint32_t g = base + idx;
            if (!wait_or_fail(L::bKVFull + (int)(g % NS), (g / NS) & 1u)) return false;
            ptx::tc_fence_after();
            return true;
          };
          auto item_slot = [&](uint32_t idx) -> int { return (int)((base + idx) % NS); };
          auto k_item = [&](int jj) -> uint32_t { return jj == 0 ? 0u : 2u * jj - 1u; };
          auto v_item = [&](int jj) -> uint32_t {
            return jj < w.n_max - 1 ? 2u * jj + 2u : 2u * jj + 1u;
          };
          auto last_user = [&](int jj) -> int {
            int u = -1;
            for (int i = 0; i < QT; ++i)
              if (jj < n[i]) u = i;
            return u;
          };
          if (s_role) {
            // S_0(j), S_1(j), S_0(j+1), ...: each waits until its score
            // buffer's previous contents are in the softmax's registers
            // (per tile, or for the shared buffer the other tile's).
            for (int j = 0; ok && j < w.n_max; ++j) {
              if (!wait_item(k_item(j))) {
                ok = false;
                break;
              }
              for (int i = 0; ok && i < QT; ++i) {
                if (j >= n[i]) continue;
                if constexpr (L::kShareS) {
                  if (s_total > 0) ok = wait_or_fail(L::bSFree, (s_total - 1) & 1u);
                  ++s_total;
                } else {
                  if (s_issued[i] > 0) ok = wait_or_fail(L::bSFree + i, (s_issued[i] - 1) & 1);
                  ++s_issued[i];
                }
                if (!ok) break;
                ptx::tc_fence_after();
                FATTN_TRACE_EV(k, j, 26 + 2 * i);
                issue_s(i, (uint32_t)item_slot(k_item(j)));
                FATTN_TRACE_EV(k, j, 13 + i);
                commit(L::bSFull + i);
                if (j == n[i] - 1) commit(L::bQEmpty + i);
                if (i == last_user(j)) commit(L::bKVEmpty + item_slot(k_item(j)));
              }
            }
          } else {
            // PV_0(j), PV_1(j), ...: each waits for its P (and, first in a
            // unit, for the epilogue to have read the previous unit's O).
            for (int j = 0; ok && j < w.n_max; ++j) {
              if (!wait_item(v_item(j))) {
                ok = false;
                break;
              }
              FATTN_TRACE_EV(k, j, 24);
              for (int i = 0; ok && i < QT; ++i) {
                if (j >= n[i]) continue;
                ok = wait_or_fail(L::bPFull + i, p_cnt[i] & 1);
                ++p_cnt[i];
                if (ok && j == 0 && used[i] > 0) {
                  ok = wait_or_fail(L::bOEmpty + i, oe_cnt[i] & 1);
                  ++oe_cnt[i];
                  FATTN_TRACE_EV(k, kTraceUnit, 21 + i);
                }
                if (!ok) break;
                FATTN_TRACE_EV(k, j, 25 + 2 * i);
                ptx::tc_fence_after();
                issue_pv(i, (uint32_t)item_slot(v_item(j)), j > 0);
                FATTN_TRACE_EV(k, j, 15 + i);
                commit(L::bPVDone + i);
                if (i == last_user(j)) commit(L::bKVEmpty + item_slot(v_item(j)));
              }
            }
          }
        } else {
          uint32_t k_slot = 0;
          if (!next_kv(k_slot)) {
            ok = false;
            break;
          }
          for (int i = 0; i < QT; ++i)
            if (n[i] > 0) {
              issue_s(i, k_slot);
              commit(L::bSFull + i);
              if (n[i] == 1) commit(L::bQEmpty + i);
            }
          commit(L::bKVEmpty + k_slot);

          for (int j = 0; ok && j < w.n_max; ++j) {
            uint32_t v_slot = 0, kn_slot = 0;
            bool have_kn = false;
            if (!next_kv(v_slot)) {
              ok = false;
              break;
            }
            FATTN_TRACE_EV(k, j, 24);
            int last_pv = -1;
            for (int i = 0; i < QT; ++i)
              if (j < n[i]) last_pv = i;
            for (int i = 0; ok && i < QT; ++i) {
              if (j < n[i]) {
                if (i == QT - 1) FATTN_TRACE_EV(k, j, 29);
                if constexpr (L::kHalfPV) {
                  // the first half of P is ready while the softmax still
                  // works on the second: its P V goes first
                  ok = wait_or_fail(L::bP1Full + i, p_cnt[i] & 1);
                  if (ok && j == 0 && used[i] > 0) {
                    ok = wait_or_fail(L::bOEmpty + i, oe_cnt[i] & 1);
                    ++oe_cnt[i];
                  }
                  if (!ok) break;
                  ptx::tc_fence_after();
                  issue_pv(i, v_slot, j > 0, 1);
                  commit(L::bPV1Done + i);
                }
                ok = wait_or_fail(L::bPFull + i, p_cnt[i] & 1);
                ++p_cnt[i];
                if (i == QT - 1) FATTN_TRACE_EV(k, j, 30);
                if (!L::kHalfPV && ok && j == 0 && used[i] > 0) {
                  ok = wait_or_fail(L::bOEmpty + i, oe_cnt[i] & 1);
                  ++oe_cnt[i];
                }
                if (!ok) break;
                if (i == QT - 1) FATTN_TRACE_EV(k, j, 31);
                FATTN_TRACE_EV(k, j, 25 + 2 * i);
                ptx::tc_fence_after();
                if constexpr (L::kHalfPV)
                  issue_pv(i, v_slot, true, 2);
                else
                  issue_pv(i, v_slot, j > 0);
                commit(L::bPVDone + i);
                if (i == last_pv) commit(L::bKVEmpty + v_slot);
              }
              if (j + 1 < n[i]) {
                if (!have_kn) {
                  if (!next_kv(kn_slot)) {
                    ok = false;
                    break;
                  }
                  have_kn = true;
                }
                FATTN_TRACE_EV(k, j, 26 + 2 * i);
                issue_s(i, kn_slot);
                commit(L::bSFull + i);
                if (j + 2 == n[i]) commit(L::bQEmpty + i);
              }
            }
            if (have_kn) commit(L::bKVEmpty + kn_slot);
          }
        }
        for (int i = 0; i < QT; ++i)
          if (n[i] > 0) ++used[i];
      }
      // Drain: every MMA these warps issued completes before TMEM is freed.
      commit(L::bDrain);
      ptx::mbar_wait_drain(bar(L::bDrain), 0, tmo);
    }
  } else if (warp < W::kCorrection0) {
    // ---------------------------------------------------- softmax warpgroups
    if constexpr (QT == 2) ptx::setmaxnreg_inc<W::kRegSoftmax>();
    const int i = warp / 4;          // query tile of this warpgroup
    const int quarter = warp % 4;    // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const uint32_t s_addr = tmem + ((uint32_t)(quarter * 32) << 16) + L::colS(i);
    const uint32_t p_addr = tmem + ((uint32_t)(quarter * 32) << 16) + L::colP(i);
    const float c = p.scale_log2;
    int sf_cnt = 0;
    int units_done = 0;  // units of this tile whose row statistics were published
    int p_writes = 0;    // P_i buffer fills so far (separate-P layout)
    int h1_published = 0;  // first halves of P_i published (half-P V layout)
    // O_i rows of this warp's lane quarter times a (per row).  In the
    // half-P V layout it may run while half a score row is still in
    // registers: 16 columns at a time there.
    auto rescale_o = [&](float a) {
      const uint32_t o_addr = tmem + ((uint32_t)(quarter * 32) << 16) + L::colO(i);
      if constexpr (L::kHalfPV) {
#pragma unroll 1
        for (int ch = 0; ch < D / 16; ++ch) {
          uint32_t u[16];
          ptx::tmem_ld16(o_addr + ch * 16, u);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 16; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * a);
          ptx::tmem_st16(o_addr + ch * 16, u);
        }
      } else {
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t u[32];
          ptx::tmem_ld32(o_addr + ch * 32, u);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * a);
          ptx::tmem_st32(o_addr + ch * 32, u);
        }
      }
    };
    // p = exp2(s*c - mref) for the row, with the scale folded into one packed
    // FFMA per pair; 16-bit P goes to TMEM over the S columns (the whole row
    // is in registers), the row sum runs in four packed partial sums, and
    // with TRACK the row maximum of s is taken on the side.
    // With FP8 also the sum of the weights as rounded to E4M3 (rsum): the
    // normaliser of O, so that O is exactly a convex combination of V rows.
    // range_c: the keys (KeyRange); P of key kFirst goes to column addr.
    auto exp_pass = [&](const float (&s)[kBN], float mref, uint32_t addr, auto track_c,
                        float& tmax, float& rsum, auto range_c) -> float {
      constexpr bool kTrack = decltype(track_c)::value;
      constexpr int kFirst = decltype(range_c)::kFirst;
      constexpr int kN = decltype(range_c)::kCount;
      const float2 c2 = make_float2(c, c);
      const float2 neg2 = make_float2(-mref, -mref);
      float2 sum2[4];
      float acc[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) sum2[a] = make_float2(0.f, 0.f);
#pragma unroll
      for (int a = 0; a < 4; ++a) acc[a] = -INFINITY;
      [[maybe_unused]] float r0 = 0.f, r1 = 0.f;
#pragma unroll
      for (int ch = 0; ch < kN / 32; ++ch) {
        uint32_t pk[16];
        float2 prev = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float s0 = s[kFirst + ch * 32 + 2 * e], s1 = s[kFirst + ch * 32 + 2 * e + 1];
          if (kTrack) acc[e & 3] = fmax3(acc[e & 3], s0, s1);
          const float2 x = __ffma2_rn(make_float2(s0, s1), c2, neg2);
          const float2 pp = make_float2(ex2(x.x), ex2(x.y));
          sum2[e & 3] = __fadd2_rn(sum2[e & 3], pp);
          if constexpr (FP8) {
            if (e & 1) {
              pk[e / 2] = pack4_e4m3(prev.x, prev.y, pp.x, pp.y);
              add4_e4m3(pk[e / 2], r0, r1);
            }
            prev = pp;
          } else {
            pk[e] = pack2<BF16>(pp.x, pp.y);
          }
        }
        if constexpr (FP8) {
          uint32_t p8[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) p8[e] = pk[e];
          ptx::tmem_st8(addr + ch * 8, p8);
        } else {
          ptx::tmem_st16(addr + ch * 16, pk);
        }
      }
      if (kTrack) tmax = fmaxf(fmax3(acc[0], acc[1], acc[2]), acc[3]);
      if constexpr (FP8) rsum = r0 + r1;
      const float2 s4 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
      return s4.x + s4.y;
    };
    // The same exponent pass keeping the packed P in registers (stored once
    // the PV that last read this P buffer has completed).
    auto exp_pack = [&](const float (&s)[kBN], float mref, uint32_t (&pk)[kBN / 2]) -> float {
      const float2 c2 = make_float2(c, c);
      const float2 neg2 = make_float2(-mref, -mref);
      float2 sum2[4];
#pragma unroll
      for (int a = 0; a < 4; ++a) sum2[a] = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < kBN / 2; ++e) {
        const float2 x = __ffma2_rn(make_float2(s[2 * e], s[2 * e + 1]), c2, neg2);
        const float2 pp = make_float2(ex2(x.x), ex2(x.y));
        sum2[e & 3] = __fadd2_rn(sum2[e & 3], pp);
        pk[e] = pack2<BF16>(pp.x, pp.y);
      }
      const float2 s4 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
      return s4.x + s4.y;
    };
    // The 8-bit form: four E4M3 weights per word (byte j = key 4e + j), and
    // the sum of the weights as rounded (rsum), the normaliser of O.
    auto exp_pack8 = [&](const float (&s)[kBN], float mref, uint32_t (&pk)[kBN / 4],
                         float& rsum) -> float {
      const float2 c2 = make_float2(c, c);
      const float2 neg2 = make_float2(-mref, -mref);
      float2 sum2[4];
      float r0 = 0.f, r1 = 0.f;
#pragma unroll
      for (int a = 0; a < 4; ++a) sum2[a] = make_float2(0.f, 0.f);
#pragma unroll
      for (int e = 0; e < kBN / 4; ++e) {
        const float2 x0 = __ffma2_rn(make_float2(s[4 * e], s[4 * e + 1]), c2, neg2);
        const float2 x1 = __ffma2_rn(make_float2(s[4 * e + 2], s[4 * e + 3]), c2, neg2);
        const float2 p0 = make_float2(ex2(x0.x), ex2(x0.y));
        const float2 p1 = make_float2(ex2(x1.x), ex2(x1.y));
        sum2[(2 * e) & 3] = __fadd2_rn(sum2[(2 * e) & 3], p0);
        sum2[(2 * e + 1) & 3] = __fadd2_rn(sum2[(2 * e + 1) & 3], p1);
        pk[e] = pack4_e4m3(p0.x, p0.y, p1.x, p1.y);
        add4_e4m3(pk[e], r0, r1);
      }
      rsum = r0 + r1;
      const float2 s4 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
      return s4.x + s4.y;
    };
    for (int k = 0;; ++k) {
      const int t = next_unit(k, kRoleSoftmax);
      if (t == kUnitEnd || t < 0) break;
      if (t >= p.total_units) continue;
      int n[QT];
      const Unit w = decode_unit<QT, CAUSAL, kRunTimeCapable>(t, p, n);
      const int nk = n[i];
      if (nk == 0) continue;
      // m: the row's reference maximum of scaled scores (log2 domain), moved
      // only when a new maximum exceeds it by more than kRescaleLog2; l: the
      // running sum of exp2(s*c - m) with that same reference.
      float m = -INFINITY;
      float m_next = 0.f;  // fused maximum: the reference for the next tile
      float l = 0.f;   // sum of fp32 p (log-sum-exp)
      float lr = 0.f;  // the same with each tile's largest p rounded as the
                       // MMA multiplies it (normaliser of O)
      bool ok = true;
      for (int j = 0; j < nk; ++j) {
        FATTN_TRACE_EV(k, j, 8 * i + 0);
        ok = ptx::mbar_wait<kSpinSoftmax>(bar(L::bSFull + i), sf_cnt & 1, abort_flag, tmo);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) raise_error(p, abort_flag, kErrPipelineTimeout, kRoleSoftmax, L::bSFull + i);
          break;
        }
        ++sf_cnt;
        FATTN_TRACE_EV(k, j, 8 * i + 1);
        ptx::tc_fence_after();
        float s[kBN];
#pragma unroll
        for (int ch = 0; ch < kBN / 32; ++ch) {
          uint32_t u[32];
          ptx::tmem_ld32(s_addr + ch * 32, u);
#pragma unroll
          for (int e = 0; e < 32; ++e) s[ch * 32 + e] = __uint_as_float(u[e]);
        }
        ptx::tmem_wait_ld();
        if constexpr (L::kSepP || L::kShareS) {
          // S_i is in registers: the MMA may compute the next scores into
          // this buffer now (S_i(j+1); in the shared buffer, the other tile's).
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(L::bSFree + (L::kShareS ? 0 : i)));
        }
        FATTN_TRACE_EV(k, j, 8 * i + 2);
        // masks: causal diagonal tile keeps key <= query; keys >= S removed
        const int kv0 = j * kBN;
        const bool diag = CAUSAL && (j == nk - 1);
        const bool ragged = kv0 + kBN > p.S;
        if (diag || ragged) {
          int limit = kBN;
          if (diag) limit = r + 1;
          if (ragged && p.S - kv0 < limit) limit = p.S - kv0;
#pragma unroll
          for (int e = 0; e < kBN; ++e) s[e] = e < limit ? s[e] : -INFINITY;
        }
        float m_use = m, alpha = 1.0f, sum, tmax, rsum = 0.f;
        if constexpr (kFusedMax) {
          // Maximum fused into the exponent pass.  The first tile of a row
          // takes its maximum first; a later one uses the reference chosen
          // after the tile before (m_next), so its weights may pass 2^8 (by
          // as much as that tile's maximum passed the reference) and the
          // reference, when it moves, moves one tile late: O and l stay in
          // one frame with each tile's P.  Only a tile whose weights could
          // overflow the 16-bit P is redone, against its own maximum.
          if (j == 0) {
            float acc[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) acc[a] = fmax3(s[2 * a], s[2 * a + 1], -INFINITY);
#pragma unroll
            for (int e = 16; e < kBN; e += 16) {
#pragma unroll
              for (int a = 0; a < 8; ++a) acc[a] = fmax3(acc[a], s[e + 2 * a], s[e + 2 * a + 1]);
            }
            m_use = c * fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]),
                              fmaxf(acc[6], acc[7]));
            if (m_use == -INFINITY) m_use = 0.f;  // no allowed key in this row
          } else {
            m_use = m_next;
          }
          FATTN_TRACE_EV(k, j, 8 * i + 3);
          // P_i's columns are free, and O_i complete through tile j-1, once
          // the P V that read the previous P has landed.
          if (p_writes > 0) {
            bool w_ok = ptx::mbar_wait(bar(L::bPVDone + i), (p_writes - 1) & 1, abort_flag, tmo);
            w_ok = __all_sync(0xffffffffu, w_ok);
            if (!w_ok) {
              if (lane == 0) raise_error(p, abort_flag, kErrPipelineTimeout, kRoleSoftmax, L::bPVDone + i);
              ok = false;
              break;
            }
            ptx::tc_fence_after();
          }
          ++p_writes;
          sum = exp_pass(s, m_use, p_addr, std::true_type{}, tmax, rsum, KeyRange<0, kBN>{});
          {
            const bool ovf = tmax * c > m_use + kOverflowLog2<BF16>;
            if (__any_sync(0xffffffffu, ovf)) {
              if (ovf) m_use = tmax * c;
              sum = exp_pass(s, m_use, p_addr, std::false_type{}, tmax, rsum, KeyRange<0, kBN>{});
            }
          }
          if (j > 0 && m_use != m) alpha = ex2(m - m_use);
          m_next = tmax * c > m_use + kRescaleLog2 ? tmax * c : m_use;
        } else if constexpr (L::kSepP || L::kShareS) {
          // Separate P, maximum first: the exponents go to registers at once
          // and P to TMEM once the previous P V has landed (no redo is
          // possible once packed P waits in registers for its buffer).  The
          // fused form above saves the maximum pass but waits for that P V
          // before its exponents; it measured faster only for bf16
          // non-causal at head dim 128 (FATTN_FUSED_MAX).
          float acc[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) acc[a] = fmax3(s[2 * a], s[2 * a + 1], -INFINITY);
#pragma unroll
          for (int e = 16; e < kBN; e += 16) {
#pragma unroll
            for (int a = 0; a < 8; ++a) acc[a] = fmax3(acc[a], s[e + 2 * a], s[e + 2 * a + 1]);
          }
          tmax = fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]),
                       fmaxf(acc[6], acc[7]));
          const float mxc = tmax * c;
          const bool move = mxc > m + kRescaleLog2;
          if (move) m_use = mxc;
          if (m_use == -INFINITY) m_use = 0.f;  // no allowed key in this row yet
          if (move && j > 0) alpha = ex2(m - m_use);
          FATTN_TRACE_EV(k, j, 8 * i + 3);
          uint32_t pk[FP8 ? kBN / 4 : kBN / 2];
          if constexpr (FP8)
            sum = exp_pack8(s, m_use, pk, rsum);
          else
            sum = exp_pack(s, m_use, pk);
          // P_i is free once the PV that read its previous contents is done
          // (that PV also ends the last update of O_i before a rescale).
          if (p_writes > 0) {
            bool w_ok = ptx::mbar_wait(bar(L::bPVDone + i), (p_writes - 1) & 1, abort_flag, tmo);
            w_ok = __all_sync(0xffffffffu, w_ok);
            if (!w_ok) {
              if (lane == 0) raise_error(p, abort_flag, kErrPipelineTimeout, kRoleSoftmax, L::bPVDone + i);
              ok = false;
              break;
            }
          }
          ++p_writes;
#pragma unroll
          for (int ch = 0; ch < (FP8 ? kBN / 64 : kBN / 32); ++ch) {
            uint32_t part[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) part[e] = pk[ch * 16 + e];
            ptx::tmem_st16(p_addr + ch * 16, part);
          }
        } else if constexpr (L::kHalfPV) {
          // P V in two halves of the keys.  The first tile of a row takes
          // its maximum first; later tiles exponentiate each half against
          // the current reference with the maximum on the side, and a half
          // whose maximum passed the reference by more than kRescaleLog2
          // moves it and is redone (warp-uniformly).  The first half's P is
          // published before the second is computed; if the second half
          // moves the reference, O (which then holds the first half's P V)
          // is rescaled once that P V has landed, with l and lr: the same
          // result, since alpha * p_old = p_new.
          if (j == 0) {
            float acc[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) acc[a] = fmax3(s[2 * a], s[2 * a + 1], -INFINITY);
#pragma unroll
            for (int e = 16; e < kBN; e += 16) {
#pragma unroll
              for (int a = 0; a < 8; ++a) acc[a] = fmax3(acc[a], s[e + 2 * a], s[e + 2 * a + 1]);
            }
            m_use = c * fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]),
                              fmaxf(acc[6], acc[7]));
            if (m_use == -INFINITY) m_use = 0.f;  // no allowed key in this row
          }
          FATTN_TRACE_EV(k, j, 8 * i + 3);
          constexpr int kHalf = kBN / 2;
          constexpr uint32_t kPHalfCols = FP8 ? kHalf / 4 : kHalf / 2;
          // the largest weight of a half as the MMA sees it, minus its fp32 value
          auto round_corr = [&](float tm, float mr) -> float {
            if constexpr (FP8) {
              return 0.f;
            } else {
              const float pt = ex2(fmaf(tm, c, -mr));
              return unpack2<BF16>(pack2<BF16>(pt, 0.f)).x - pt;
            }
          };
          // ---- first half
          float tmax0 = -INFINITY, rsum0 = 0.f;
          float sum0 = exp_pass(s, m_use, s_addr, std::true_type{}, tmax0, rsum0,
                                KeyRange<0, kHalf>{});
          if (j > 0) {
            const float mxc = tmax0 * c;
            const bool move = mxc > m + kRescaleLog2;
            if (__any_sync(0xffffffffu, move)) {
              if (move) {
                m_use = mxc;
                alpha = ex2(m - m_use);
              }
              sum0 = exp_pass(s, m_use, s_addr, std::false_type{}, tmax0, rsum0,
                              KeyRange<0, kHalf>{});
            }
          }
          // PV_i(j-1) has landed (S_i(j) was issued after it): O may change
          if (__any_sync(0xffffffffu, alpha != 1.f)) rescale_o(alpha);
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(L::bP1Full + i));
          ++h1_published;
          l = alpha * l + sum0;
          lr = alpha * lr + (FP8 ? rsum0 : sum0 + round_corr(tmax0, m_use));
          m = m_use;
          // ---- second half
          float tmax1 = -INFINITY, rsum1 = 0.f;
          float sum1 = exp_pass(s, m, s_addr + kPHalfCols, std::true_type{}, tmax1, rsum1,
                                KeyRange<kHalf, kHalf>{});
          {
            const float mxc = tmax1 * c;
            const bool move = mxc > m + kRescaleLog2;
            if (__any_sync(0xffffffffu, move)) {
              float m_new = m, alpha1 = 1.f;
              if (move) {
                m_new = mxc;
                alpha1 = ex2(m - m_new);
              }
              sum1 = exp_pass(s, m_new, s_addr + kPHalfCols, std::false_type{}, tmax1, rsum1,
                              KeyRange<kHalf, kHalf>{});
              // the first half's P V must have landed before O is rescaled
              bool w_ok = ptx::mbar_wait(bar(L::bPV1Done + i), (uint32_t)(h1_published - 1) & 1u,
                                         abort_flag, tmo);
              w_ok = __all_sync(0xffffffffu, w_ok);
              if (!w_ok) {
                if (lane == 0) raise_error(p, abort_flag, kErrPipelineTimeout, kRoleSoftmax, L::bPV1Done + i);
                ok = false;
                break;
              }
              ptx::tc_fence_after();
              if (__any_sync(0xffffffffu, alpha1 != 1.f)) rescale_o(alpha1);
              l *= alpha1;
              lr *= alpha1;
              m = m_new;
            }
          }
          ptx::tmem_wait_st();
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(L::bPFull + i));
          FATTN_TRACE_EV(k, j, 8 * i + 4);
          l += sum1;
          lr += FP8 ? rsum1 : sum1 + round_corr(tmax1, m);
        } else {
          // P over S.  Reference maximum m (log2 domain).  The first tile of
          // a row has none yet: take its maximum first.  Later tiles
          // exponentiate against the current reference at once and track
          // their maximum on the side; the rare tile whose maximum passes the
          // reference by more than kRescaleLog2 is redone against the new
          // maximum (warp-uniformly, since P goes back to TMEM with warp-wide
          // stores).  O, l and the exponent share the reference, so any
          // choice is exact; p <= 2^8.
          if (j == 0) {
            float acc[8];
#pragma unroll
            for (int a = 0; a < 8; ++a) acc[a] = fmax3(s[2 * a], s[2 * a + 1], -INFINITY);
#pragma unroll
            for (int e = 16; e < kBN; e += 16) {
#pragma unroll
              for (int a = 0; a < 8; ++a) acc[a] = fmax3(acc[a], s[e + 2 * a], s[e + 2 * a + 1]);
            }
            m_use = c * fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]),
                              fmaxf(acc[6], acc[7]));
            if (m_use == -INFINITY) m_use = 0.f;  // no allowed key in this row
          }
          FATTN_TRACE_EV(k, j, 8 * i + 3);
          tmax = -INFINITY;
          sum = exp_pass(s, m_use, s_addr, std::true_type{}, tmax, rsum, KeyRange<0, kBN>{});
          if (j > 0) {
            const float mxc = tmax * c;
            const bool move = mxc > m + kRescaleLog2;
            if (__any_sync(0xffffffffu, move)) {
              if (move) {
                m_use = mxc;
                alpha = ex2(m - m_use);
              }
              sum = exp_pass(s, m_use, s_addr, std::false_type{}, tmax, rsum, KeyRange<0, kBN>{});
            }
          }
        }
        if constexpr (!L::kHalfPV) {
        // A row that moved its reference scales its O by exp2(m_old - m_new).
        // This warp owns these O rows (its TMEM lane quarter) and may touch
        // them now: PV_i(j-1) has landed (with P aliasing S, S_i(j) was
        // issued after it; with separate P, its completion was awaited
        // above), and no MMA writes O_i until this warp reports P ready.
        if (__any_sync(0xffffffffu, alpha != 1.f)) rescale_o(alpha);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(L::bPFull + i));
        FATTN_TRACE_EV(k, j, 8 * i + 4);
        // The tile's largest weight, as the MMA sees it (rounded to 16 bits):
        // normalising O by the fp32 sum with that one term replaced keeps a
        // peaked row's dominant weight exact, as p = 1 would be under an
        // exact running maximum.  (fmaf gives the same value as a lane of
        // the packed FFMA above.)
        l = alpha * l + sum;
        if constexpr (FP8) {
          lr = alpha * lr + rsum;
        } else {
          const float pt = ex2(fmaf(tmax, c, -m_use));
          const float pt16 = unpack2<BF16>(pack2<BF16>(pt, 0.f)).x;
          lr = alpha * lr + (sum + (pt16 - pt));
        }
        m = m_use;
        }
      }
      if (!ok) break;
      // The previous unit's epilogue must have read its statistics before
      // they are overwritten; it releases O_i (o_empty) after reading them.
      if (units_done > 0) {
        ok = ptx::mbar_wait(bar(L::bOEmpty + i), (units_done - 1) & 1, abort_flag, tmo);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) {
          if (lane == 0) raise_error(p, abort_flag, kErrPipelineTimeout, kRoleSoftmax, L::bOEmpty + i);
          break;
        }
      }
      ++units_done;
      sRowL[i * kBM + r] = lr;
      sRowM[i * kBM + r] = (m + log2f(l)) * 0.69314718055994531f;  // natural-log LSE
      ptx::mbar_arrive(bar(L::bStats + i));
    }
  } else if (warp < W::kMma) {
    // -------------------------------------------------- correction warpgroup
    if constexpr (QT == 2) ptx::setmaxnreg_dec<W::kRegCorrection>();
    const int quarter = warp % 4;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    // st_cnt: units whose final row statistics were read; pv_base: PV MMAs
    // of earlier units, so the phase of "last PV_i of this unit done" is
    // known without waiting on every PV.
    int st_cnt[QT], pv_base[QT];
    for (int i = 0; i < QT; ++i) st_cnt[i] = pv_base[i] = 0;
    bool ok = true;
    auto wait_all = [&](int slot, uint32_t parity) -> bool {
      bool w_ok = ptx::mbar_wait(bar(slot), parity, abort_flag, tmo);
      w_ok = __all_sync(0xffffffffu, w_ok);
      if (!w_ok && lane == 0)
        raise_error(p, abort_flag, kErrPipelineTimeout, kRoleCorrection, slot);
      return w_ok;
    };
    for (int k = 0; ok; ++k) {
      const int t = next_unit(k, kRoleCorrection);
      if (t == kUnitEnd) break;
      if (t < 0) {
        ok = false;
        break;
      }
      if (t >= p.total_units) continue;
      int n[QT];
      const Unit w = decode_unit<QT, CAUSAL, kRunTimeCapable>(t, p, n);
      // epilogue: O = acc / l (one reciprocal per row), LSE = ln2 (m + log2 l)
      for (int i = 0; i < QT; ++i) {
        if (n[i] == 0) continue;
        if (!wait_all(L::bStats + i, st_cnt[i] & 1)) { ok = false; break; }
        ++st_cnt[i];
        const float l = sRowL[i * kBM + r];    // normaliser of O
        const float lse = sRowM[i * kBM + r];  // log-sum-exp of the row
        if (!wait_all(L::bPVDone + i, (uint32_t)(pv_base[i] + n[i] - 1) & 1u)) { ok = false; break; }
        pv_base[i] += n[i];
        FATTN_TRACE_EV(k, kTraceUnit, 17 + i);
        ptx::tc_fence_after();
        const float inv_l = p.o_scale / l;
        const int row = w.q_row0 + kBM * i + r;
        const bool valid = row < p.S;
        const size_t grow = (size_t)w.bh * (size_t)p.S + (size_t)row;
        uint4* const orow = reinterpret_cast<uint4*>(
            reinterpret_cast<uint8_t*>(p.o) + grow * (size_t)(D * 2));
        const uint32_t o_addr = tmem + lane_off + L::colO(i);
        const bool o_aligned32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
        // The next chunk's TMEM load is in flight while this one is scaled,
        // packed and stored.
        uint32_t u[32];
        ptx::tmem_ld32(o_addr, u);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          ptx::tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            pk[e] = pack2<BF16>(__uint_as_float(u[2 * e]) * inv_l,
                                __uint_as_float(u[2 * e + 1]) * inv_l);
          if (ch + 1 < D / 32) {
            ptx::tmem_ld32(o_addr + (ch + 1) * 32, u);
          } else {
            // O_i (and the row statistics, read above) are in registers: the
            // next unit's P V may overwrite them while the stores below run.
            ptx::tc_fence_before();
            ptx::mbar_arrive(bar(L::bOEmpty + i));
            FATTN_TRACE_EV(k, kTraceUnit, 19 + i);
          }
          if (valid) {
            // a thread writes its own row: 32-byte stores when the output is
            // 32-byte aligned (rows are 128 or 256 bytes), else 16-byte ones
            if (o_aligned32) {
#pragma unroll
              for (int v8 = 0; v8 < 2; ++v8) {
                uint32_t w8[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) w8[e] = pk[8 * v8 + e];
                ptx::st_global_v8(orow + ch * 4 + 2 * v8, w8);
              }
            } else {
#pragma unroll
              for (int v4 = 0; v4 < 4; ++v4)
                orow[ch * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2], pk[4 * v4 + 3]);
            }
          }
        }
        if (valid) p.lse[grow] = lse;
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == W::kMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTmemCols);
  }
  if constexpr (CAUSAL) {
    // Every unit this CTA will ever take has been taken; the last CTA to
    // get here returns the launch's counter to 0 for the next launch.
    if (run_time_units && threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
        atomicExch(p.sched, 0);
        atomicExch(p.sched + 1, 0);
      }
    }
  }
}

}  // namespace fattn
