// bf16 instantiations of the 2-CTA (SM pair) GEMM kernel, 256 x 256 tiles, all four operand
// layouts.
#include "sk_pair_launch.cuh"

namespace sk {

cudaError_t setup_bf16_pair(int layout, int* max_clusters) {
  switch (layout) {
    case 1: return setup_pair_kernel<false, true, false>(max_clusters);
    case 2: return setup_pair_kernel<false, false, true>(max_clusters);
    case 3: return setup_pair_kernel<false, true, true>(max_clusters);
    default: return setup_pair_kernel<false, false, false>(max_clusters);
  }
}

cudaError_t launch_bf16_pair(int layout, const Launch& l) {
  switch (layout) {
    case 1: return launch_pair_kernel<false, true, false>(l);
    case 2: return launch_pair_kernel<false, false, true>(l);
    case 3: return launch_pair_kernel<false, true, true>(l);
    default: return launch_pair_kernel<false, false, false>(l);
  }
}

}  // namespace sk
