// Kernel instantiations for head dim 128: fp16 / bf16 x non-causal / causal.
#include "fattn_launch.cuh"

namespace fattn {

cudaError_t launch_fwd_d128(bool causal, bool bf16, const LaunchArgs& a) {
  if (causal)
    return bf16 ? launch_fwd<128, true, true>(a) : launch_fwd<128, true, false>(a);
  return bf16 ? launch_fwd<128, false, true>(a) : launch_fwd<128, false, false>(a);
}

}  // namespace fattn
