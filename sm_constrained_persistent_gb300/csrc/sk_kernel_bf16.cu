// bf16 instantiations of the one-CTA-per-tile GEMM kernel: 128 x 128 tiles in all four operand
// layouts, and 128 x 96 tiles in the plain layout.
#include "sk_kernel.cuh"
#include "sk_launch.h"

namespace sk {

template <bool kAT, bool kBT, int kBN = 128>
static cudaError_t launch_one(const Launch& l) {
  using Cf = Cfg<false, kBN, kAT, kBT>;
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
  return cudaLaunchKernelEx(&cfg, gemm_kernel<false, kBN, kAT, kBT>, *l.tmA, *l.tmB,
                            l.tmC != nullptr ? *l.tmC : *l.tmA, l.args);
}

template <bool kAT, bool kBT, int kBN = 128>
static cudaError_t setup_one(int* ctas_per_sm) {
  using Cf = Cfg<false, kBN, kAT, kBT>;
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<false, kBN, kAT, kBT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cf::kSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, gemm_kernel<false, kBN, kAT, kBT>,
                                                       kThreads, Cf::kSmemBytes);
}

cudaError_t setup_bf16_n96(int* ctas_per_sm) { return setup_one<false, false, 96>(ctas_per_sm); }
cudaError_t launch_bf16_n96(const Launch& l) { return launch_one<false, false, 96>(l); }

cudaError_t setup_bf16_n128(int layout, int* ctas_per_sm) {
  switch (layout) {
    case 1: return setup_one<true, false>(ctas_per_sm);
    case 2: return setup_one<false, true>(ctas_per_sm);
    case 3: return setup_one<true, true>(ctas_per_sm);
    default: return setup_one<false, false>(ctas_per_sm);
  }
}

cudaError_t launch_bf16_n128(int layout, const Launch& l) {
  switch (layout) {
    case 1: return launch_one<true, false>(l);
    case 2: return launch_one<false, true>(l);
    case 3: return launch_one<true, true>(l);
    default: return launch_one<false, false>(l);
  }
}

}  // namespace sk
