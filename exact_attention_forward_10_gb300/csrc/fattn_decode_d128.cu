// Instantiations of the cache-attention kernels for head dim 128.
#include "fattn_decode_launch.h"

namespace fattn {
namespace decode {

cudaError_t launch_d128(bool bf16, const DecodeLaunch& a) {
  return bf16 ? launch_d<128, true>(a) : launch_d<128, false>(a);
}

}  // namespace decode
}  // namespace fattn
