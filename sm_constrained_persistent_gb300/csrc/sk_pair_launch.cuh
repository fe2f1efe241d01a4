// Launch and set-up of one instantiation of the 2-CTA (SM pair) GEMM kernel.
#pragma once

#include "sk_kernel_pair.cuh"
#include "sk_launch.h"

namespace sk {

template <bool kMx, bool kAT, bool kBT, bool kF8 = false>
cudaError_t launch_pair_kernel(const Launch& l) {
  using Cf = PairCfg<kMx, kAT, kBT, kF8>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(l.grid), 1, 1);
  cfg.blockDim = dim3(pair_threads<kMx>(), 1, 1);
  cfg.dynamicSmemBytes = Cf::kSmemBytes;
  cfg.stream = l.stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, gemm_pair_kernel<kMx, kAT, kBT, kF8>, *l.tmA, *l.tmB, *l.tmSfa,
                            *l.tmSfb, l.tmC != nullptr ? *l.tmC : *l.tmA, l.args);
}

template <bool kMx, bool kAT, bool kBT, bool kF8 = false>
cudaError_t setup_pair_kernel(int* max_clusters) {
  using Cf = PairCfg<kMx, kAT, kBT, kF8>;
  cudaError_t e = cudaFuncSetAttribute(gemm_pair_kernel<kMx, kAT, kBT, kF8>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cf::kSmemBytes));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(pair_threads<kMx>(), 1, 1);
  cfg.dynamicSmemBytes = Cf::kSmemBytes;
  e = cudaOccupancyMaxActiveClusters(max_clusters, gemm_pair_kernel<kMx, kAT, kBT, kF8>, &cfg);
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
  return cudaOccupancyMaxActiveClusters(max_clusters, gemm_pair_kernel<kMx, kAT, kBT, kF8>, &cfg);
}

}  // namespace sk
