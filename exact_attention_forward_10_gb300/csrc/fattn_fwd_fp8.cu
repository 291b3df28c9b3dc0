// Kernel instantiations for E4M3 inputs, head dim 128: fp16 / bf16 output x
// non-causal / causal.
#include "fattn_launch.cuh"

namespace fattn {

cudaError_t launch_fwd_fp8_d128(bool causal, bool bf16_out, const LaunchArgs& a) {
  if (causal)
    return bf16_out ? launch_fwd_fp8<true, true>(a) : launch_fwd_fp8<true, false>(a);
  return bf16_out ? launch_fwd_fp8<false, true>(a) : launch_fwd_fp8<false, false>(a);
}

}  // namespace fattn
