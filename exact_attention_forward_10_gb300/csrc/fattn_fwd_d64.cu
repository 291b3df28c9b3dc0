// Kernel instantiations for head dim 64: fp16 / bf16 x non-causal / causal.
#include "fattn_launch.cuh"

namespace fattn {

cudaError_t launch_fwd_d64(bool causal, bool bf16, const LaunchArgs& a) {
  if (causal)
    return bf16 ? launch_fwd<64, true, true>(a) : launch_fwd<64, true, false>(a);
  return bf16 ? launch_fwd<64, false, true>(a) : launch_fwd<64, false, false>(a);
}

}  // namespace fattn
