// Host-side planning for attention against a key/value cache: the query-count
// buckets (one query: the CUDA-core split kernel; 2 to 16: the warp-level MMA
// split kernel), warps and shared memory of the split kernel, and the
// dispatch to the per-head-dim instantiation units.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fattn_decode.cuh"
#include "fattn_decode_launch.h"

namespace fattn {
namespace decode {
int sq_bucket(int Sq) { return Sq <= 1 ? 1 : kMaxSq; }

int warps_per_cta(int D, int Sq) {
  if (sq_bucket(Sq) == 1) return D == 64 ? DecodeLayout<64, 1>::kWarps : DecodeLayout<128, 1>::kWarps;
  return D == 64 ? DecodeMmaLayout<64>::kWarps : DecodeMmaLayout<128>::kWarps;
}

int smem_bytes(int D, int Sq) {
  if (sq_bucket(Sq) == 1)
    return D == 64 ? DecodeLayout<64, 1>::kSmemBytes : DecodeLayout<128, 1>::kSmemBytes;
  return D == 64 ? DecodeMmaLayout<64>::kSmemBytes : DecodeMmaLayout<128>::kSmemBytes;
}

cudaError_t launch(int D, bool bf16, const DecodeLaunch& a) {
  return D == 64 ? launch_d64(bf16, a) : launch_d128(bf16, a);
}

}  // namespace decode
}  // namespace fattn
