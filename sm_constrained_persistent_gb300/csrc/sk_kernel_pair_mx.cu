// MXFP4 instantiation of the 2-CTA (SM pair) GEMM kernel, 256 x 256 x 256 tiles.
#include "sk_pair_launch.cuh"

namespace sk {

cudaError_t setup_mx_pair(int* max_clusters) { return setup_pair_kernel<true, false, false>(max_clusters); }
cudaError_t launch_mx_pair(const Launch& l) { return launch_pair_kernel<true, false, false>(l); }

}  // namespace sk
