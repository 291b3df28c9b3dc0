// Exact softmax-attention forward for head dim 256 on sm_103a (GB300), one
// 256-row query block per pair of SMs.
//
// What it computes is the same as fattn_kernel.cuh (O = softmax(scale Q K^T
// [+ causal]) V and the per-row LSE, by the online-softmax recurrence of
// "FlashAttention V2", section 3).  Head dim 256 is a size the pages list as
// supported ("FlashAttention V2", section 6, the table of when V2 is used).
//
// Why a CTA pair.  At D = 256 one query tile's O takes 256 TMEM columns, so a
// CTA holds a single 128-row query tile, and every K/V byte it loads serves
// half the rows it serves at D = 128: L2-to-SM traffic per FLOP doubles and
// the 64 KB K/V tiles leave no room for a deep ring.  Two SMs of a cluster
// instead issue one tcgen05 MMA with M = 256 (cta_group::2): each SM holds
// its own 128 query rows, and each SM loads only HALF of every K tile (64 of
// its 128 keys) and half of every V tile (128 of its 256 columns); the MMA
// reads the peer's half through the cluster.  Per SM this is the traffic and
// shared-memory footprint of the D = 128 kernel.
//
// Per CTA (both ranks run every role; rank 0, the even CTA, issues the MMAs):
//   * load warp:   TMA Q (its 128 rows) once per unit; its K and V halves
//                  through a 5-item ring of 32 KB.  Completion is counted on
//                  rank 0's barriers (a pair MMA needs both halves), which
//                  rank 0's load warp arms with the pair's byte count.
//   * MMA warp:    (rank 0) S = Q K^T, M = 256, N = 128, into two TMEM score
//                  buffers in turn; O += P V, M = 256, N = 256, P read from
//                  TMEM where it overwrote its scores.  Order per key tile j:
//                  PV(j), then S(j+2) into the buffer PV(j) just read (the
//                  pair's tensor pipe keeps issue order).  Commits are
//                  multicast to both CTAs' barriers.
//   * softmax warpgroup: thread r owns row r (TMEM lane r): scores, masks,
//                  lazy reference maximum, exp2, 16-bit P back to TMEM; it
//                  rescales its own O rows in the rare tile that moves the
//                  reference (after the previous P V has landed).
//   * epilogue warpgroup: O / l, cast, store O and the LSE.
// Cross-CTA hand-offs: P ready and O free are counted on rank 0's barriers by
// one arrival per warp of either CTA.  Every wait is bounded; a timeout
// records an error and the CTA unwinds; both CTAs meet at a final cluster
// barrier before TMEM is freed.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "fattn_kernel.cuh"
#include "fattn_status.h"
#include "ptx.cuh"

namespace fattn {
namespace pair {

constexpr int kRows = 2 * kBM;          // query rows per unit (the pair)
constexpr int kQChunk = kBM * 128;      // [128 rows, 64 cols]
constexpr int kKChunk = 64 * 128;       // [64 keys, 64 cols]
constexpr int kVChunk = kBN * 128;      // [128 keys, 64 cols]
constexpr uint16_t kBoth = 3;           // multicast mask: both CTAs

// D: head dim (128 or 256).  NSB: TMEM score buffers (P overwrites the
// first 64 columns of one); O takes D columns after them.  NS: K/V ring items.
template <int D, int NSB, int NS>
struct PairLayout {
  static_assert(D == 128 || D == 256, "head dim");
  static_assert(128 * NSB + D <= (int)kTmemCols, "TMEM budget");
  static constexpr int kQBytes = kBM * D * 2;      // this CTA's Q tile
  static constexpr int kItemBytes = 128 * D;       // one K half or one V half
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + kQBytes;
  static constexpr int kBars = kKV + NS * kItemBytes;
  static constexpr int bQFull = 0;          // rank 0: 1 arrival + both Q tiles
  static constexpr int bQEmpty = 1;         // each CTA: pair commit
  static constexpr int bKVFull = 2;         // rank 0: 1 arrival + both halves
  static constexpr int bKVEmpty = bKVFull + NS;   // each CTA: pair commit
  static constexpr int bSFull = bKVEmpty + NS;    // [NSB] each CTA: pair commit
  static constexpr int bPFull = bSFull + NSB;     // [NSB] rank 0: 8 warp arrivals
  static constexpr int bPVDone = bPFull + NSB;    // [NSB] each CTA: pair commit per PV
                                                  // reading that buffer
  static constexpr int bODone = bPVDone + NSB;    // each CTA: pair commit per unit
  static constexpr int bOEmpty = bODone + 1;      // rank 0: 8 warp arrivals
  static constexpr int bStats = bOEmpty + 1;      // each CTA: 128 arrivals
  static constexpr int bStatsFree = bStats + 1;   // each CTA: 4 warp arrivals
  static constexpr int bDrain = bStatsFree + 1;   // rank 0: MMA drain
  static constexpr int bUnitFull = bDrain + 1;    // [kUnitRing] each CTA: rank 0's load warp
  static constexpr int bUnitEmpty = bUnitFull + kUnitRing;  // [kUnitRing] rank 0: every reader
  static constexpr int kNumBars = bUnitEmpty + kUnitRing;
  static constexpr int kMisc = kBars + kNumBars * 8;
  static constexpr int kRowL = kMisc + 16;
  static constexpr int kRowM = kRowL + kBM * 4;
  static constexpr int kUnitSlots = kRowM + kBM * 4;  // int [kUnitRing]
  static constexpr int kSmemBytes = kUnitSlots + kUnitRing * 4;
  static_assert(kSmemBytes <= 232448, "shared memory per CTA");
  __host__ __device__ static constexpr uint32_t colS(int b) { return 128u * b; }
  static constexpr uint32_t kColO = 128u * NSB;
};

struct PairWarps {
  static constexpr int kSoftmax0 = 0;     // warps 0-3
  static constexpr int kEpilogue0 = 4;    // warps 4-7
  static constexpr int kMma = 8;
  static constexpr int kLoad = 9;
  static constexpr int kNumWarps = 12;    // whole warpgroups
  static constexpr int kThreads = 32 * kNumWarps;
  // 384 threads launch with 168 registers each; the per-warpgroup split
  // adds up to the same total.
  static constexpr int kRegSoftmax = 200;
  static constexpr int kRegEpilogue = 152;
  static constexpr int kRegOther = 152;
  static_assert(kRegSoftmax + kRegEpilogue + kRegOther == 3 * 168,
                "register split must equal the launch allocation");
};

struct PairUnit {
  int bh;
  int row0;  // first query row of the pair's 256-row block
  int n;     // key tiles the pair processes
};

// Unit t: causal units longest first (the last query blocks need the most
// keys) within groups of group_heads heads, so the K/V of the heads in flight
// stay in L2; non-causal units of one head adjacent (they share its K/V).
// The last group takes the remaining heads.  (Near-equal groups, as the
// single-SM kernel decodes them, measured 5% faster at B2 H16 S4097 causal,
// whose 32 heads then run as 7, 7, 6, 6 and 6 instead of 7, 7, 7, 7 and 4,
// but ~2% slower at S = 4096, 8192 and 12288, where the groups are the same.)
template <bool CAUSAL>
__device__ __forceinline__ PairUnit pair_unit(int t, const FwdParams& p) {
  PairUnit w;
  int u;
  if (CAUSAL) {
    const int G = p.group_heads;
    const int g = t / (G * p.n_units);
    const int r = t - g * G * p.n_units;
    const int gh = p.BH - g * G < G ? p.BH - g * G : G;
    u = p.n_units - 1 - r / gh;
    w.bh = g * G + r % gh;
  } else {
    u = t % p.n_units;
    w.bh = t / p.n_units;
  }
  w.row0 = u * kRows;
  if (CAUSAL) {
    // through the diagonal tile of the pair's last valid query tile
    const int last_q0 = (w.row0 + kBM < p.S) ? w.row0 + kBM : w.row0;
    w.n = last_q0 / kBN + 1;
  } else {
    w.n = p.n_kv_tiles;
  }
  return w;
}

// Round k of the persistent loop over clusters: a snake, as in the one-SM
// kernel.
__device__ __forceinline__ int pair_unit_of_round(int k) {
  const int G = (int)gridDim.x / 2;
  const int g = (int)blockIdx.x / 2;
  return k * G + ((k & 1) ? (G - 1 - g) : g);
}

template <int D, int NSB, int NS, bool CAUSAL, bool BF16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(PairWarps::kThreads, 1)
    fattn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q,
                          const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v,
                          const FwdParams p) {
  using L = PairLayout<D, NSB, NS>;
  constexpr int kQBytes = L::kQBytes;
  constexpr int kItemBytes = L::kItemBytes;
  using W = PairWarps;
  // every warp that reads the unit sequence, in both CTAs: softmax (4) and
  // epilogue (4) in each, rank 0's MMA warp and rank 1's load warp
  constexpr int kUnitReaders = 18;
  constexpr int kUnitEnd = -2;
  extern __shared__ uint8_t smem_raw[];

  // A causal launch without its unit counter reports a launch error and
  // does nothing (every CTA of every cluster returns here).
  if (CAUSAL && p.sched == nullptr) {
    if (threadIdx.x == 0 && atomicCAS(p.status, 0, kErrLaunch) == 0) {
      p.status[1] = 0;
      p.status[2] = (int)blockIdx.x;
    }
    return;
  }
  const uint32_t base = ptx::smem_u32(smem_raw);
  // Both CTAs of a cluster get the same layout; a misaligned base would be
  // the same in both, so both return here and neither waits for the other.
  if (base & 1023u) {
    if (threadIdx.x == 0 && atomicCAS(p.status, 0, kErrLaunch) == 0) {
      p.status[1] = 0;
      p.status[2] = (int)blockIdx.x;
    }
    // this CTA still counts as done, so the launch's unit counter is reset
    if (CAUSAL && threadIdx.x == 0 && atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(p.sched, 0);
      atomicExch(p.sched + 1, 0);
    }
    return;
  }
  uint8_t* const smem = smem_raw;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool leader = rank == 0;
  const uint32_t sQ = base + L::kQ;
  const uint32_t sKV = base + L::kKV;
  const uint32_t bars = base + L::kBars;
  uint32_t* const tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMisc);
  volatile int* const abort_flag = reinterpret_cast<volatile int*>(smem + L::kMisc + 4);
  float* const sRowL = reinterpret_cast<float*>(smem + L::kRowL);
  float* const sRowM = reinterpret_cast<float*>(smem + L::kRowM);
  auto bar = [&](int slot) -> uint32_t { return bars + 8u * slot; };
  // The same barrier in rank 0 (shared::cluster address).
  auto bar0 = [&](int slot) -> uint32_t { return ptx::mapa_shared(bar(slot), 0); };

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t tmo = p.timeout_ns;

  if (threadIdx.x == 0) {
    ptx::mbar_init(bar(L::bQFull), 1);
    ptx::mbar_init(bar(L::bQEmpty), 1);
    for (int s = 0; s < NS; ++s) {
      ptx::mbar_init(bar(L::bKVFull + s), 1);
      ptx::mbar_init(bar(L::bKVEmpty + s), 1);
    }
    for (int b = 0; b < NSB; ++b) {
      ptx::mbar_init(bar(L::bSFull + b), 1);
      ptx::mbar_init(bar(L::bPFull + b), 8);
      ptx::mbar_init(bar(L::bPVDone + b), 1);
    }
    ptx::mbar_init(bar(L::bODone), 1);
    ptx::mbar_init(bar(L::bOEmpty), 8);
    ptx::mbar_init(bar(L::bStats), kBM);
    ptx::mbar_init(bar(L::bStatsFree), 4);
    ptx::mbar_init(bar(L::bDrain), 1);
    for (int r = 0; r < kUnitRing; ++r) {
      ptx::mbar_init(bar(L::bUnitFull + r), 1);
      ptx::mbar_init(bar(L::bUnitEmpty + r), kUnitReaders);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == W::kMma) {
    ptx::tmem_alloc_pair(ptx::smem_u32(tmem_slot), kTmemCols);
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  // Barriers of both CTAs initialised and TMEM allocated before any CTA
  // signals the other.
  ptx::cluster_sync();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&](int role, int slot) {
    if (atomicCAS(p.status, 0, kErrPipelineTimeout) == 0) {
      p.status[1] = (role << 8) | slot;
      p.status[2] = (int)blockIdx.x;
    }
    *abort_flag = 1;
  };
  // The unit of this CTA pair's k-th round.  Causal: rank 0's load warp
  // takes units at run time (its cluster's index first, then the launch's
  // counter) and writes each into a small ring in both CTAs; every reader
  // hands its slot back to rank 0.  A value >= total_units ends the
  // sequence.  Non-causal: the static snake, where a round may have no unit
  // for this pair (a value >= total_units).  kUnitEnd ends the sequence; -1
  // is an error.
  const int n_clusters = (int)gridDim.x / 2;
  volatile int* const unit_slots = reinterpret_cast<volatile int*>(smem + L::kUnitSlots);
  // one lane's read of unit k (the load warp of rank 1 runs in one lane)
  auto read_unit = [&](int k, int role) -> int {
    const int slot = k % kUnitRing;
    if (!ptx::mbar_wait_cluster(bar(L::bUnitFull + slot), (k / kUnitRing) & 1, abort_flag, tmo)) {
      fail(role, L::bUnitFull + slot);
      return -1;
    }
    const int t = unit_slots[slot];
    ptx::mbar_arrive_cluster(bar0(L::bUnitEmpty + slot));
    return t >= p.total_units ? kUnitEnd : t;
  };
  auto next_unit = [&](int k, int role) -> int {
    if constexpr (CAUSAL) {
      const int slot = k % kUnitRing;
      bool w_ok = ptx::mbar_wait_cluster(bar(L::bUnitFull + slot), (k / kUnitRing) & 1,
                                         abort_flag, tmo);
      w_ok = __all_sync(0xffffffffu, w_ok);
      if (!w_ok) {
        if (lane == 0) fail(role, L::bUnitFull + slot);
        return -1;
      }
      const int t = unit_slots[slot];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive_cluster(bar0(L::bUnitEmpty + slot));
      return t >= p.total_units ? kUnitEnd : t;
    } else {
      if (k * n_clusters >= p.total_units) return kUnitEnd;
      return pair_unit_of_round(k);
    }
  };

  if (warp >= W::kMma) ptx::setmaxnreg_dec<W::kRegOther>();

  if (warp == W::kLoad) {
    // ------------------------------------------------------------ load warp
    if (lane == 0) {
      ptx::tma_prefetch_desc(&tm_q);
      ptx::tma_prefetch_desc(&tm_k);
      ptx::tma_prefetch_desc(&tm_v);
      uint32_t idx = 0, ph = 0;  // ring position
      int q_uses = 0;
      uint32_t filled = 0, fill_ph = 0;
      bool ok = true;
      int t_next = (int)blockIdx.x / 2 < p.total_units ? (int)blockIdx.x / 2 : p.total_units;
      for (int k = 0; ok; ++k) {
        int t;
        if constexpr (CAUSAL) {
          if (leader) {
            // publish unit k in both CTAs' rings
            t = t_next;
            const int slot = k % kUnitRing;
            if (k >= kUnitRing &&
                !ptx::mbar_wait_cluster(bar(L::bUnitEmpty + slot), ((k / kUnitRing) - 1) & 1,
                                        abort_flag, tmo)) {
              fail(kRoleLoad, L::bUnitEmpty + slot);
              ok = false;
              break;
            }
            unit_slots[slot] = t;
            ptx::st_shared_cluster_u32(ptx::mapa_shared(base + L::kUnitSlots + 4u * slot, 1),
                                       (uint32_t)t);
            ptx::mbar_arrive(bar(L::bUnitFull + slot));
            ptx::mbar_arrive_cluster(ptx::mapa_shared(bar(L::bUnitFull + slot), 1));
            if (t >= p.total_units) break;
          } else {
            t = read_unit(k, kRoleLoad);
            if (t == kUnitEnd) break;
            if (t < 0) {
              ok = false;
              break;
            }
          }
        } else {
          if (k * n_clusters >= p.total_units) break;
          t = pair_unit_of_round(k);
          if (t >= p.total_units) continue;
        }
        const PairUnit w = pair_unit<CAUSAL>(t, p);
        int taken = 0;  // causal, rank 0: the counter's value for the next unit
        if (q_uses > 0 &&
            !ptx::mbar_wait_cluster(bar(L::bQEmpty), (q_uses - 1) & 1, abort_flag, tmo)) {
          fail(kRoleLoad, L::bQEmpty);
          ok = false;
          break;
        }
        FATTN_TRACE_EV(k, kTraceUnit, 0);
        if (leader) ptx::mbar_arrive_expect_tx(bar(L::bQFull), 2 * kQBytes);
#pragma unroll
        for (int c = 0; c < D / kSwizzleChunkCols; ++c)
          ptx::tma_load_3d_pair(sQ + c * kQChunk, &tm_q, bar0(L::bQFull),
                                c * kSwizzleChunkCols, w.row0 + kBM * (int)rank, w.bh);
        ++q_uses;
        for (int j = 0; ok && j < w.n; ++j) {
          // The next unit is taken as this unit's last key tile is loaded:
          // the pairs that will be free first take the longest units left.
          if (CAUSAL && leader && j == w.n - 1) taken = atomicAdd(p.sched, 1);
#pragma unroll
          for (int kv = 0; kv < 2; ++kv) {
            if (!ptx::mbar_wait_cluster(bar(L::bKVEmpty + idx), ph ^ 1u, abort_flag, tmo)) {
              fail(kRoleLoad, L::bKVEmpty + idx);
              ok = false;
              break;
            }
            if (leader) ptx::mbar_arrive_expect_tx(bar(L::bKVFull + idx), 2 * kItemBytes);
            const uint32_t dst = sKV + idx * kItemBytes;
            const uint32_t fb = bar0(L::bKVFull + idx);
            if (kv == 0) {
              // K half: keys [128 j + 64 rank, +64), all 256 columns
#pragma unroll
              for (int c = 0; c < D / kSwizzleChunkCols; ++c)
                ptx::tma_load_3d_pair(dst + c * kKChunk, &tm_k, fb, c * kSwizzleChunkCols,
                                      j * kBN + 64 * (int)rank, w.bh);
            } else {
              // V half: keys [128 j, +128), columns [D/2 rank, +D/2)
#pragma unroll
              for (int c = 0; c < D / 128; ++c)
                ptx::tma_load_3d_pair(dst + c * kVChunk, &tm_v, fb,
                                      (D / 2) * (int)rank + c * kSwizzleChunkCols, j * kBN,
                                      w.bh);
            }
            FATTN_TRACE_EV(k, j, 1 + kv);
            filled |= 1u << idx;
            fill_ph = (fill_ph & ~(1u << idx)) | (ph << idx);
            if (++idx == NS) {
              idx = 0;
              ph ^= 1u;
            }
          }
        }
        if constexpr (CAUSAL) {
          if (leader) {
            t_next = n_clusters + taken;
            if (t_next > p.total_units) t_next = p.total_units;
          }
        }
      }
      // Never leave copies in flight: both halves land on rank 0's barriers,
      // so rank 0 waits for them; rank 1 is held by the final cluster barrier
      // until rank 0 is through.
      if (leader) {
        for (int s = 0; s < NS; ++s)
          if (filled & (1u << s))
            ptx::mbar_wait_cluster_drain(bar(L::bKVFull + s), (fill_ph >> s) & 1u, tmo);
        if (q_uses > 0)
          ptx::mbar_wait_cluster_drain(bar(L::bQFull), (q_uses - 1) & 1, tmo);
      }
    }
  } else if (warp == W::kMma) {
    // ------------------------------------------------------ MMA warp (rank 0)
    if (leader) {
      constexpr uint32_t kIdS = ptx::idesc_f16(BF16 ? 1 : 0, kRows, kBN, 0, 0);
      constexpr uint32_t kIdPV = ptx::idesc_f16(BF16 ? 1 : 0, kRows, D, 0, 1);
      constexpr uint32_t kHi = ptx::desc_sw128_hi(1024);
      constexpr uint32_t kItemLo = kItemBytes >> 4;
      const uint32_t q_lo = ptx::desc_sw128_lo(sQ, 16);
      const uint32_t k_lo = ptx::desc_sw128_lo(sKV, 16);
      const uint32_t v_lo = ptx::desc_sw128_lo(sKV, kVChunk);  // LBO: next 64 columns
      uint32_t item = 0;  // ring index of the next unit's K_0
      int q_uses = 0, oe_cnt = 0, used = 0;
      uint32_t pf_par = 0;  // bit b: parity of buffer b's P-full completions seen
      bool ok = true;
      auto wait_or_fail = [&](int slot, uint32_t parity) -> bool {
        bool w_ok = ptx::mbar_wait_cluster(bar(slot), parity, abort_flag, tmo);
        w_ok = __all_sync(0xffffffffu, w_ok);
        if (!w_ok && lane == 0) fail(kRoleMma, slot);
        return w_ok;
      };
      auto commit = [&](int slot) {
        if (ptx::elect_one()) ptx::mma_commit_pair(bar(slot), kBoth);
      };
      // S = Q K^T: K = 256 in steps of 16 (32 bytes of a 128-byte swizzled
      // row; the next 64 columns are one chunk further: 16 KB in Q, 8 KB in
      // the K half).
      auto issue_s = [&](int b, uint32_t slot) {
        const uint32_t d = tmem + L::colS(b);
        const uint32_t kb = k_lo + slot * kItemLo;
        if (!ptx::elect_one()) return;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t qa = q_lo + (((kk / 4) * kQChunk + (kk % 4) * 32) >> 4);
          const uint32_t ka = kb + (((kk / 4) * kKChunk + (kk % 4) * 32) >> 4);
          if (kk == 0)
            ptx::mma_ss_pair<0>(d, qa, ka, kHi, kIdS, 0u);
          else
            ptx::mma_ss_pair<1>(d, qa, ka, kHi, kIdS, 1u);
        }
      };
      // O += P V: K = 128 keys in steps of 16 (P: 8 TMEM columns of packed
      // pairs; V, MN-major: 16 rows = 2048 bytes further).
      auto issue_pv = [&](int b, uint32_t slot, bool acc) {
        const uint32_t d = tmem + L::kColO;
        const uint32_t a = tmem + L::colS(b);
        const uint32_t vb = v_lo + slot * kItemLo;
        if (!ptx::elect_one()) return;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          if (kk == 0)
            ptx::mma_ts_pair<0>(d, a, vb, kHi, kIdPV, acc ? 1u : 0u);
          else
            ptx::mma_ts_pair<1>(d, a + kk * 8, vb + kk * (2048 >> 4), kHi, kIdPV, 1u);
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
        const PairUnit w = pair_unit<CAUSAL>(t, p);
        const uint32_t ubase = item;
        item += 2u * (uint32_t)w.n;
        auto wait_item = [&](uint32_t i) -> bool {
          const uint32_t g = ubase + i;
          if (!wait_or_fail(L::bKVFull + (int)(g % NS), (g / NS) & 1u)) return false;
          ptx::tc_fence_after();
          return true;
        };
        auto slot_of = [&](uint32_t i) -> uint32_t { return (ubase + i) % NS; };
        if (!wait_or_fail(L::bQFull, q_uses & 1)) break;
        FATTN_TRACE_EV(k, kTraceUnit, 4);
        ++q_uses;
        ptx::tc_fence_after();
        // prologue: S(0) .. S(NSB-1)
        for (int j = 0; ok && j < NSB && j < w.n; ++j) {
          ok = wait_item(2u * j);
          if (!ok) break;
          issue_s(j, slot_of(2u * j));
          FATTN_TRACE_EV(k, j, 5);
          commit(L::bSFull + j);
          commit(L::bKVEmpty + (int)slot_of(2u * j));
          if (j == w.n - 1) commit(L::bQEmpty);
        }
        for (int j = 0; ok && j < w.n; ++j) {
          const int b = j % NSB;
          if (!wait_item(2u * j + 1u)) { ok = false; break; }
          if (!wait_or_fail(L::bPFull + b, (pf_par >> b) & 1u)) { ok = false; break; }
          FATTN_TRACE_EV(k, j, 7);
          pf_par ^= 1u << b;
          if (j == 0 && used > 0) {
            if (!wait_or_fail(L::bOEmpty, oe_cnt & 1)) { ok = false; break; }
            FATTN_TRACE_EV(k, kTraceUnit, 8);
            ++oe_cnt;
          }
          ptx::tc_fence_after();
          issue_pv(b, slot_of(2u * j + 1u), j > 0);
          FATTN_TRACE_EV(k, j, 6);
          commit(L::bPVDone + b);
          commit(L::bKVEmpty + (int)slot_of(2u * j + 1u));
          if (j == w.n - 1) commit(L::bODone);
          // S(j+NSB) overwrites the buffer PV(j) reads P from; the pair's
          // tensor pipe runs MMAs in issue order, so it may follow at once.
          if (j + NSB < w.n) {
            if (!wait_item(2u * (j + NSB))) { ok = false; break; }
            issue_s(b, slot_of(2u * (j + NSB)));
            FATTN_TRACE_EV(k, j + NSB, 5);
            commit(L::bSFull + b);
            commit(L::bKVEmpty + (int)slot_of(2u * (j + NSB)));
            if (j + NSB == w.n - 1) commit(L::bQEmpty);
          }
        }
        ++used;
      }
      // Drain: every pair MMA completes before TMEM is freed.
      if (ptx::elect_one()) ptx::mma_commit_pair(bar(L::bDrain), 1);
      __syncwarp();
      ptx::mbar_wait_drain(bar(L::bDrain), 0, tmo);
    }
  } else if (warp < W::kEpilogue0) {
    // ---------------------------------------------------- softmax warpgroup
    ptx::setmaxnreg_inc<W::kRegSoftmax>();
    const int quarter = warp;  // TMEM lanes 32*quarter .. +31
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const float c = p.scale_log2;
    // Per score buffer, the parity of its S-full completions seen so far and
    // of the P V MMAs reading it issued so far (bit b: buffer b).  Bit masks,
    // not arrays: a buffer index that varies at run time would put an array
    // in local memory.
    uint32_t sf_par = 0, pv_par = 0;
    int units_done = 0;
    bool ok = true;
    auto wait_all = [&](int slot, uint32_t parity) -> bool {
      bool w_ok = ptx::mbar_wait_cluster(bar(slot), parity, abort_flag, tmo);
      w_ok = __all_sync(0xffffffffu, w_ok);
      if (!w_ok && lane == 0) fail(kRoleSoftmax, slot);
      return w_ok;
    };
    // exp2(s*c - mref) for the row into packed 16-bit P in TMEM (over the
    // score columns), returning the fp32 sum; with TRACK also the row max.
    auto exp_pass = [&](const float (&s)[kBN], float mref, uint32_t addr, auto track_c,
                        float& tmax) -> float {
      constexpr bool kTrack = decltype(track_c)::value;
      const float2 c2 = make_float2(c, c);
      const float2 neg2 = make_float2(-mref, -mref);
      float2 sum2[4];
      float acc[8];
#pragma unroll
      for (int a = 0; a < 4; ++a) sum2[a] = make_float2(0.f, 0.f);
#pragma unroll
      for (int a = 0; a < 8; ++a) acc[a] = -INFINITY;
#pragma unroll
      for (int ch = 0; ch < kBN / 32; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 16; ++e) {
          const float s0 = s[ch * 32 + 2 * e], s1 = s[ch * 32 + 2 * e + 1];
          if (kTrack) acc[e & 7] = fmax3(acc[e & 7], s0, s1);
          const float2 x = __ffma2_rn(make_float2(s0, s1), c2, neg2);
          const float2 pp = make_float2(ex2(x.x), ex2(x.y));
          sum2[e & 3] = __fadd2_rn(sum2[e & 3], pp);
          pk[e] = pack2<BF16>(pp.x, pp.y);
        }
        ptx::tmem_st16(addr + ch * 16, pk);
      }
      if (kTrack)
        tmax = fmax3(fmax3(acc[0], acc[1], acc[2]), fmax3(acc[3], acc[4], acc[5]),
                     fmaxf(acc[6], acc[7]));
      const float2 s4 = __fadd2_rn(__fadd2_rn(sum2[0], sum2[1]), __fadd2_rn(sum2[2], sum2[3]));
      return s4.x + s4.y;
    };
    for (int k = 0; ok; ++k) {
      const int t = next_unit(k, kRoleSoftmax);
      if (t == kUnitEnd) break;
      if (t < 0) {
        ok = false;
        break;
      }
      if (t >= p.total_units) continue;
      const PairUnit w = pair_unit<CAUSAL>(t, p);
      const int row = w.row0 + kBM * (int)rank + r;  // this thread's query row
      float m = -INFINITY, l = 0.f, lr = 0.f;
      for (int j = 0; j < w.n; ++j) {
        const int b = j % NSB;
        if (!wait_all(L::bSFull + b, (sf_par >> b) & 1u)) { ok = false; break; }
        if (quarter == 0) FATTN_TRACE_EV(k, j, 10);
        sf_par ^= 1u << b;
        ptx::tc_fence_after();
        const uint32_t s_addr = tmem + lane_off + L::colS(b);
        float s[kBN];
#pragma unroll
        for (int ch = 0; ch < kBN / 32; ++ch) {
          uint32_t u[32];
          ptx::tmem_ld32(s_addr + ch * 32, u);
#pragma unroll
          for (int e = 0; e < 32; ++e) s[ch * 32 + e] = __uint_as_float(u[e]);
        }
        ptx::tmem_wait_ld();
        // masks: causal keeps key <= row; keys >= S removed
        const int kv0 = j * kBN;
        int limit = kBN;
        if (CAUSAL && row - kv0 + 1 < limit) limit = row - kv0 + 1;
        if (p.S - kv0 < limit) limit = p.S - kv0;
        if (__any_sync(0xffffffffu, limit < kBN)) {
#pragma unroll
          for (int e = 0; e < kBN; ++e) s[e] = e < limit ? s[e] : -INFINITY;
        }
        // Lazy reference maximum, as in the one-SM kernel: the first tile
        // takes its maximum; later tiles exponentiate against the reference
        // and redo (warp-uniformly) the rare tile whose maximum passes it by
        // more than kRescaleLog2.
        float m_use = m, alpha = 1.0f, sum, tmax;
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
          if (m_use == -INFINITY) m_use = 0.f;  // no allowed key in this row yet
        }
        tmax = -INFINITY;
        sum = exp_pass(s, m_use, s_addr, std::true_type{}, tmax);
        if (j > 0) {
          const float mxc = tmax * c;
          const bool move = mxc > m + kRescaleLog2;
          if (__any_sync(0xffffffffu, move)) {
            if (move) {
              m_use = mxc;
              alpha = ex2(m - m_use);
            }
            sum = exp_pass(s, m_use, s_addr, std::false_type{}, tmax);
            if (quarter == 0) FATTN_TRACE_EV(k, j, 13);
          }
        }
        // A row that moved its reference scales its O rows, once the P V of
        // the previous tile (the last writer of O) has landed; no later P V
        // runs before this warp reports P ready.  That PV's buffer barrier
        // has at most it outstanding (the one before it on the buffer is
        // older than S(j)), so its parity is unambiguous.
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
          const int pb = (j - 1) % NSB;
          if (!wait_all(L::bPVDone + pb, ((pv_par >> pb) & 1u) ^ 1u)) { ok = false; break; }
          ptx::tc_fence_after();
          if (quarter == 0) FATTN_TRACE_EV(k, j, 14);
          const uint32_t o_addr = tmem + lane_off + L::kColO;
#pragma unroll 1
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t u[32];
            ptx::tmem_ld32(o_addr + ch * 32, u);
            ptx::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) u[e] = __float_as_uint(__uint_as_float(u[e]) * alpha);
            ptx::tmem_st32(o_addr + ch * 32, u);
          }
        }
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        // rank 0 arrives on its own barrier (CTA scope); the peer's warps
        // release across the cluster.
        if (quarter == 0) FATTN_TRACE_EV(k, j, 11);
        if (lane == 0) {
          if (leader)
            ptx::mbar_arrive(bar(L::bPFull + b));
          else
            ptx::mbar_arrive_cluster(bar0(L::bPFull + b));
        }
        pv_par ^= 1u << b;  // PV(j) may be issued from here on
        const float pt = ex2(fmaf(tmax, c, -m_use));
        const float pt16 = unpack2<BF16>(pack2<BF16>(pt, 0.f)).x;
        l = alpha * l + sum;
        lr = alpha * lr + (sum + (pt16 - pt));
        m = m_use;
      }
      if (!ok) break;
      // The epilogue must have read the previous unit's statistics.
      if (units_done > 0 && !wait_all(L::bStatsFree, (units_done - 1) & 1)) break;
      ++units_done;
      if (quarter == 0) FATTN_TRACE_EV(k, kTraceUnit, 12);
      sRowL[r] = lr;
      sRowM[r] = (m + log2f(l)) * 0.69314718055994531f;  // natural-log LSE
      ptx::mbar_arrive(bar(L::bStats));
    }
  } else if (warp < W::kMma) {
    // --------------------------------------------------- epilogue warpgroup
    ptx::setmaxnreg_dec<W::kRegEpilogue>();
    const int quarter = warp - W::kEpilogue0;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    int st_cnt = 0, od_cnt = 0;
    bool ok = true;
    auto wait_all = [&](int slot, uint32_t parity) -> bool {
      bool w_ok = ptx::mbar_wait_cluster(bar(slot), parity, abort_flag, tmo);
      w_ok = __all_sync(0xffffffffu, w_ok);
      if (!w_ok && lane == 0) fail(kRoleCorrection, slot);
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
      const PairUnit w = pair_unit<CAUSAL>(t, p);
      if (!wait_all(L::bStats, st_cnt & 1)) break;
      if (quarter == 0) FATTN_TRACE_EV(k, kTraceUnit, 15);
      ++st_cnt;
      const float l = sRowL[r];
      const float lse = sRowM[r];
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(bar(L::bStatsFree));
      // The unit's last P V, by its own once-per-unit barrier: a wait on the
      // per-PV barrier could meet it two phases early (the softmax may
      // publish the statistics while the last two P V MMAs still run) and
      // pass on the parity of an older phase.
      if (!wait_all(L::bODone, od_cnt & 1)) break;
      if (quarter == 0) FATTN_TRACE_EV(k, kTraceUnit, 16);
      ++od_cnt;
      ptx::tc_fence_after();
      const float inv_l = 1.0f / l;
      const int row = w.row0 + kBM * (int)rank + r;
      const bool valid = row < p.S;
      const size_t grow = (size_t)w.bh * (size_t)p.S + (size_t)row;
      uint4* const orow = reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.o) +
                                                   grow * (size_t)(D * 2));
      const uint32_t o_addr = tmem + lane_off + L::kColO;
      const bool o_aligned32 = (reinterpret_cast<uintptr_t>(p.o) & 31u) == 0;
      // The next chunk's TMEM load is in flight while this one is scaled,
      // packed and stored.
      uint32_t u[32];
      ptx::tmem_ld32(o_addr, u);
#pragma unroll 4
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
          // all of O is read: the next unit's first P V may overwrite it
          // while the stores below run
          ptx::tc_fence_before();
          __syncwarp();
          if (quarter == 0) FATTN_TRACE_EV(k, kTraceUnit, 17);
          if (lane == 0) ptx::mbar_arrive_cluster(bar0(L::bOEmpty));
        }
        if (valid) {
          // a thread writes its own 512-byte row: 32-byte stores when the
          // output is 32-byte aligned, else 16-byte ones
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
              orow[ch * 4 + v4] = make_uint4(pk[4 * v4], pk[4 * v4 + 1], pk[4 * v4 + 2],
                                             pk[4 * v4 + 3]);
          }
        }
      }
      if (valid) p.lse[grow] = lse;
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // Neither CTA frees TMEM or exits while the other may still use its shared
  // memory, its barriers or the pair's MMAs.
  ptx::cluster_sync();
  if (warp == W::kMma) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, kTmemCols);
  }
  if constexpr (CAUSAL) {
    // Every unit this pair will take has been taken; the last CTA to get
    // here returns the launch's counter to 0 for the next launch.
    if (threadIdx.x == 0) {
      __threadfence();
      if (atomicAdd(p.sched + 1, 1) == (int)gridDim.x - 1) {
        atomicExch(p.sched, 0);
        atomicExch(p.sched + 1, 0);
      }
    }
  }
}

}  // namespace pair
}  // namespace fattn
