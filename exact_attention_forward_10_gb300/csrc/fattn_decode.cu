// Host-side planning for attention against a key/value cache: the query-count
// buckets, warps and shared memory of the split kernel, and the dispatch to
// the per-head-dim instantiation units.
#include <cuda.h>
#include <cuda_runtime.h>

#include "fattn_decode.cuh"
#include "fattn_decode_launch.h"

namespace fattn {
namespace decode {
int sq_bucket(int Sq) { return Sq <= 1 ? 1 : Sq <= 4 ? 4 : 16; }

int warps_per_cta(int D, int Sq) {
  const int b = sq_bucket(Sq);
  if (D == 64) return b == 1 ? DecodeLayout<64, 1>::kWarps
                     : b == 4 ? DecodeLayout<64, 4>::kWarps
                              : DecodeLayout<64, 16>::kWarps;
  return b == 1 ? DecodeLayout<128, 1>::kWarps
       : b == 4 ? DecodeLayout<128, 4>::kWarps
                : DecodeLayout<128, 16>::kWarps;
}

int smem_bytes(int D, int Sq) {
  const int b = sq_bucket(Sq);
  if (D == 64) return b == 1 ? DecodeLayout<64, 1>::kSmemBytes
                     : b == 4 ? DecodeLayout<64, 4>::kSmemBytes
                              : DecodeLayout<64, 16>::kSmemBytes;
  return b == 1 ? DecodeLayout<128, 1>::kSmemBytes
       : b == 4 ? DecodeLayout<128, 4>::kSmemBytes
                : DecodeLayout<128, 16>::kSmemBytes;
}

cudaError_t launch(int D, bool bf16, const DecodeLaunch& a) {
  return D == 64 ? launch_d64(bf16, a) : launch_d128(bf16, a);
}

}  // namespace decode
}  // namespace fattn
