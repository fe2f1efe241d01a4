// bf16 instantiations of the one-CTA-per-tile GEMM kernel with tall stages (128 K per stage,
// 64 rows of A): 128 x 128 and 128 x 96 tiles in the plain layout, for problems of at most 64
// rows that stream B.
#include "sk_kernel.cuh"
#include "sk_launch.h"

namespace sk {

template <int kBN>
static cudaError_t launch_tall(const Launch& l) {
  using Cf = Cfg<false, kBN, false, false, false, true>;
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
  return cudaLaunchKernelEx(&cfg, gemm_kernel<false, kBN, false, false, false, true>, *l.tmA,
                            *l.tmB, l.tmC != nullptr ? *l.tmC : *l.tmA, l.args);
}

template <int kBN>
static cudaError_t setup_tall(int* ctas_per_sm) {
  using Cf = Cfg<false, kBN, false, false, false, true>;
  const auto kernel = gemm_kernel<false, kBN, false, false, false, true>;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cf::kSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, kernel, kThreads,
                                                       Cf::kSmemBytes);
}

cudaError_t setup_bf16_tall(int bn, int* ctas_per_sm) {
  return bn == 96 ? setup_tall<96>(ctas_per_sm) : setup_tall<128>(ctas_per_sm);
}

cudaError_t launch_bf16_tall(int bn, const Launch& l) {
  return bn == 96 ? launch_tall<96>(l) : launch_tall<128>(l);
}

size_t tall_smem_bytes(int bn) {
  return bn == 96 ? Cfg<false, 96, false, false, false, true>::kSmemBytes
                  : Cfg<false, 128, false, false, false, true>::kSmemBytes;
}

}  // namespace sk
