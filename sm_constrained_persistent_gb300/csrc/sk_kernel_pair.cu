// Instantiations of the 2-CTA (SM pair) GEMM kernel: bf16 and MXFP4, 256 x 256 tiles.
#include "sk_kernel_pair.cuh"
#include "sk_launch.h"

namespace sk {

template <bool kMx>
static cudaError_t launch_pair(const Launch& l) {
  using Cf = PairCfg<kMx>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(l.grid), 1, 1);
  cfg.blockDim = dim3(pair_threads<kMx>(), 1, 1);
  cfg.dynamicSmemBytes = Cf::kSmemBytes;
  cfg.stream = l.stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<kMx>, *l.tmA, *l.tmB, *l.tmSfa, *l.tmSfb,
                            l.args);
}

template <bool kMx>
static cudaError_t setup_pair(int* max_clusters) {
  using Cf = PairCfg<kMx>;
  cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<kMx>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cf::kSmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(pair_threads<kMx>(), 1, 1);
  cfg.dynamicSmemBytes = Cf::kSmemBytes;
  e = cudaOccupancyMaxActiveClusters(max_clusters, gemm_pair_kernel<kMx>, &cfg);
  if (e == cudaSuccess && *max_clusters > 0) return e;
  // Some runtimes want the cluster shape in the query even when the kernel declares it.
  cudaGetLastError();
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(max_clusters, gemm_pair_kernel<kMx>, &cfg);
}

cudaError_t pair_variant_setup(int variant, int* max_clusters) {
  return variant == kVariantMxPair ? setup_pair<true>(max_clusters) : setup_pair<false>(max_clusters);
}

cudaError_t pair_variant_launch(int variant, const Launch& l) {
  return variant == kVariantMxPair ? launch_pair<true>(l) : launch_pair<false>(l);
}

size_t pair_variant_smem_bytes(int variant) {
  return variant == kVariantMxPair ? PairCfg<true>::kSmemBytes : PairCfg<false>::kSmemBytes;
}

}  // namespace sk
