// Kernel instantiations for head dim 256 (the CTA-pair kernel): fp16 / bf16 x
// non-causal / causal.
#include "fattn_launch.cuh"

namespace fattn {

cudaError_t launch_fwd_d256(bool causal, bool bf16, const LaunchArgs& a) {
  if (causal)
    return bf16 ? launch_fwd_pair<256, true, true>(a) : launch_fwd_pair<256, true, false>(a);
  return bf16 ? launch_fwd_pair<256, false, true>(a) : launch_fwd_pair<256, false, false>(a);
}

int pair_clusters_d256(bool causal, bool bf16) {
  if (causal) return bf16 ? pair_clusters_fit<256, true, true>() : pair_clusters_fit<256, true, false>();
  return bf16 ? pair_clusters_fit<256, false, true>() : pair_clusters_fit<256, false, false>();
}

}  // namespace fattn
