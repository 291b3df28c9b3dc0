// Per-head-dim kernel configuration and the launcher shared by the
// instantiation units (fattn_fwd_d64.cu, fattn_fwd_d128.cu).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fattn_kernel.cuh"
#include "fattn_kernel_pair.cuh"
#include "fattn_smem_opt_in.h"

namespace fattn {

// Query tiles per work unit and K/V ring depth: as many stages as fit in the
// 227 KB a CTA may use (one CTA per SM).  A K/V copy from L2 takes about
// 1.8 us under full load, so the ring depth sets how early it can start.
template <int D>
struct FwdConfig;
template <>
struct FwdConfig<64> {
  static constexpr int QT = 2;
  static constexpr int NS = 12;
};
template <>
struct FwdConfig<128> {
  static constexpr int QT = 2;
  static constexpr int NS = 5;
};

struct LaunchArgs {
  const CUtensorMap* tm_q;
  const CUtensorMap* tm_k;
  const CUtensorMap* tm_v;
  FwdParams params;
  int grid;
  cudaStream_t stream;
};

template <int D>
struct FwdShape {
  using C = FwdConfig<D>;
  using L = FwdLayout<D, C::QT, C::NS>;
  static constexpr int kSmem = L::kSmemBytes;
  static constexpr int kThreads = FwdWarps<C::QT>::kThreads;
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_fwd(const LaunchArgs& a) {
  using C = FwdConfig<D>;
  auto kern = &fattn_fwd_kernel<D, C::QT, C::NS, CAUSAL, BF16>;
  constexpr int smem = FwdShape<D>::kSmem;
  static std::atomic<bool> attr_set[64];
  cudaError_t e = smem_opt_in(kern, smem, attr_set);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, FwdShape<D>::kThreads, smem, a.stream>>>(*a.tm_q, *a.tm_k,
                                                          *a.tm_v, a.params);
  return cudaGetLastError();
}

// E4M3 inputs, head dim 128: 16 KB tiles leave room for a 12-stage ring.
constexpr int kFp8Stages = 12;
struct Fp8Shape {
  using L = FwdLayout<128, 2, kFp8Stages, 1>;
  static constexpr int kSmem = L::kSmemBytes;
  static constexpr int kThreads = FwdWarps<2>::kThreads;
  static_assert(kSmem <= 232448, "shared memory per CTA");
};

template <bool CAUSAL, bool BF16>
cudaError_t launch_fwd_fp8(const LaunchArgs& a) {
  auto kern = &fattn_fwd_kernel<128, 2, kFp8Stages, CAUSAL, BF16, true>;
  static std::atomic<bool> attr_set[64];
  cudaError_t e = smem_opt_in(kern, Fp8Shape::kSmem, attr_set);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, Fp8Shape::kThreads, Fp8Shape::kSmem, a.stream>>>(*a.tm_q, *a.tm_k,
                                                                  *a.tm_v, a.params);
  return cudaGetLastError();
}

// The CTA-pair kernel (clusters of two CTAs, one per SM) for head dim 256:
// two TMEM score buffers and a 5-item ring of 32 KB halves.
template <int D>
struct PairConfig;
template <>
struct PairConfig<256> {
  static constexpr int NSB = 2;
  static constexpr int NS = 5;
};
template <int D>
struct PairShape {
  using C = PairConfig<D>;
  static constexpr int kSmem = pair::PairLayout<D, C::NSB, C::NS>::kSmemBytes;
  static constexpr int kThreads = pair::PairWarps::kThreads;
};

template <int D, bool CAUSAL, bool BF16>
cudaError_t set_pair_attr() {
  using C = PairConfig<D>;
  auto kern = &pair::fattn_fwd_pair_kernel<D, C::NSB, C::NS, CAUSAL, BF16>;
  static std::atomic<bool> attr_set[64];
  return smem_opt_in(kern, PairShape<D>::kSmem, attr_set);
}

// a.grid counts CTAs (twice the clusters).
template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_fwd_pair(const LaunchArgs& a) {
  using C = PairConfig<D>;
  cudaError_t e = set_pair_attr<D, CAUSAL, BF16>();
  if (e != cudaSuccess) return e;
  pair::fattn_fwd_pair_kernel<D, C::NSB, C::NS, CAUSAL, BF16>
      <<<a.grid, PairShape<D>::kThreads, PairShape<D>::kSmem, a.stream>>>(
          *a.tm_q, *a.tm_k, *a.tm_v, a.params);
  return cudaGetLastError();
}

// Clusters of the pair kernel that fit on the current device at once (the
// persistent grid must not exceed it: work is assigned to clusters
// statically).  0 on error.
template <int D, bool CAUSAL, bool BF16>
int pair_clusters_fit() {
  using C = PairConfig<D>;
  if (set_pair_attr<D, CAUSAL, BF16>() != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(PairShape<D>::kThreads);
  cfg.dynamicSmemBytes = PairShape<D>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(
          &n, &pair::fattn_fwd_pair_kernel<D, C::NSB, C::NS, CAUSAL, BF16>, &cfg) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

// Defined in the instantiation units.
cudaError_t launch_fwd_d64(bool causal, bool bf16, const LaunchArgs& a);
cudaError_t launch_fwd_d128(bool causal, bool bf16, const LaunchArgs& a);
cudaError_t launch_fwd_d256(bool causal, bool bf16, const LaunchArgs& a);
cudaError_t launch_fwd_fp8_d128(bool causal, bool bf16_out, const LaunchArgs& a);
int pair_clusters_d256(bool causal, bool bf16);

}  // namespace fattn
