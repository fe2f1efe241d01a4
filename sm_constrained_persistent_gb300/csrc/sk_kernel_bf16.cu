// bf16 instantiations of the GEMM kernel (CTA tiles 128 x 128 and 128 x 256).
#include "sk_kernel.cuh"
#include "sk_launch.h"

namespace sk {

template <bool kMx, int kBN>
cudaError_t launch_variant(const Launch& l) {
  using Cf = Cfg<kMx, kBN>;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(l.grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Cf::kSmemBytes;
  cfg.stream = l.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = l.cooperative ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_kernel<kMx, kBN>, *l.tmA, *l.tmB, l.args);
}

template <bool kMx, int kBN>
cudaError_t setup_variant(int* ctas_per_sm) {
  using Cf = Cfg<kMx, kBN>;
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<kMx, kBN>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cf::kSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, gemm_kernel<kMx, kBN>,
                                                       kThreads, Cf::kSmemBytes);
}

cudaError_t launch_bf16(int tile_n, const Launch& l) {
  return tile_n == 256 ? launch_variant<false, 256>(l) : launch_variant<false, 128>(l);
}

cudaError_t setup_bf16(int tile_n, int* ctas_per_sm) {
  return tile_n == 256 ? setup_variant<false, 256>(ctas_per_sm)
                       : setup_variant<false, 128>(ctas_per_sm);
}

size_t smem_bf16(int tile_n) {
  return tile_n == 256 ? Cfg<false, 256>::kSmemBytes : Cfg<false, 128>::kSmemBytes;
}

}  // namespace sk
