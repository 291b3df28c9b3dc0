// Instantiations of the cache-attention kernels for head dim 64.
#include "fattn_decode_launch.h"

namespace fattn {
namespace decode {

cudaError_t launch_d64(bool bf16, const DecodeLaunch& a) {
  return bf16 ? launch_d<64, true>(a) : launch_d<64, false>(a);
}

}  // namespace decode
}  // namespace fattn
