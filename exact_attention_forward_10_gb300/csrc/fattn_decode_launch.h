// Host-side interface of the cache-attention kernels (fattn_decode.cu), used by
// the C ABI in fattn_api.cu.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "fattn_decode.cuh"
#include "fattn_decode_mma.cuh"
#include "fattn_smem_opt_in.h"

namespace fattn {
namespace decode {

struct DecodeLaunch {
  const CUtensorMap* tm_k;  // K cache, [BH, Sk, D], boxes of 64 cols x 32 rows
  const CUtensorMap* tm_v;  // V cache, same geometry
  DecodeParams params;
  int grid;                 // CTAs of the split kernel (one per SM)
  cudaStream_t stream;
};

// The query-count bucket that serves Sq new queries: 1 (the CUDA-core split
// kernel) or kMaxSq (2 to 16 queries: the warp-level tensor-core MMA kernel).
int sq_bucket(int Sq);
// Warps per split CTA and its dynamic shared memory, for head dim D.
int warps_per_cta(int D, int Sq);
int smem_bytes(int D, int Sq);
// Enqueue the split kernel and then the merge kernel on a.stream.
cudaError_t launch(int D, bool bf16, const DecodeLaunch& a);
// Per head dim, defined in fattn_decode_d64.cu / fattn_decode_d128.cu.
cudaError_t launch_d64(bool bf16, const DecodeLaunch& a);
cudaError_t launch_d128(bool bf16, const DecodeLaunch& a);

// The merge kernel as a programmatic dependent launch: it may begin while
// the split kernel finishes and waits (griddepcontrol.wait) for its results.
template <int D, bool BF16>
cudaError_t launch_merge(const DecodeLaunch& a) {
  const long long rows = (long long)a.params.B * a.params.H * a.params.Sq;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + kCombineWarps - 1) / kCombineWarps));
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, &fattn_decode_combine_kernel<D, BF16>, a.params);
}

// Split kernel with warp-level tensor-core MMAs (up to 16 queries), then the
// merge.
template <int D, bool BF16>
cudaError_t launch_split_mma(const DecodeLaunch& a) {
  using L = DecodeMmaLayout<D>;
  auto kern = &fattn_decode_mma_kernel<D, BF16>;
  static std::atomic<bool> attr_set[64];
  cudaError_t e = smem_opt_in(kern, L::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, L::kThreads, L::kSmemBytes, a.stream>>>(*a.tm_k, *a.tm_v, a.params);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_merge<D, BF16>(a);
}

template <int D, int SQ, bool BF16>
cudaError_t launch_split(const DecodeLaunch& a) {
  using L = DecodeLayout<D, SQ>;
  auto kern = &fattn_decode_kernel<D, SQ, BF16>;
  static std::atomic<bool> attr_set[64];
  cudaError_t e = smem_opt_in(kern, L::kSmemBytes, attr_set);
  if (e != cudaSuccess) return e;
  kern<<<a.grid, L::kThreads, L::kSmemBytes, a.stream>>>(*a.tm_k, *a.tm_v, a.params);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_merge<D, BF16>(a);
}

template <int D, bool BF16>
cudaError_t launch_d(const DecodeLaunch& a) {
  return sq_bucket(a.params.Sq) == 1 ? launch_split<D, 1, BF16>(a) : launch_split_mma<D, BF16>(a);
}


}  // namespace decode
}  // namespace fattn
