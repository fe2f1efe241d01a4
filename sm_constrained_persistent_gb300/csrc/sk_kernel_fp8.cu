// fp8 (E4M3) instantiations of the GEMM kernels: one CTA per 128 x 128 or 128 x 256 tile, and
// SM pairs on 256 x 256 tiles.  Same layouts as bf16 (A K-major, B MN-major), 1-byte elements.
#include "sk_kernel.cuh"
#include "sk_pair_launch.cuh"

namespace sk {

template <int kBN>
static cudaError_t launch_f8_one(const Launch& l) {
  using Cf = Cfg<false, kBN, false, false, true>;
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
  return cudaLaunchKernelEx(&cfg, gemm_kernel<false, kBN, false, false, true>, *l.tmA, *l.tmB,
                            l.tmC != nullptr ? *l.tmC : *l.tmA, l.args);
}

template <int kBN>
static cudaError_t setup_f8_one(int* ctas_per_sm) {
  using Cf = Cfg<false, kBN, false, false, true>;
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<false, kBN, false, false, true>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cf::kSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(
      ctas_per_sm, gemm_kernel<false, kBN, false, false, true>, kThreads, Cf::kSmemBytes);
}

cudaError_t setup_f8(int kind, int* n) {
  switch (kind) {
    case kKindF8N128: return setup_f8_one<128>(n);
    case kKindF8N256: return setup_f8_one<256>(n);
    default: return setup_pair_kernel<false, false, false, true>(n);
  }
}

cudaError_t launch_f8(int kind, const Launch& l) {
  switch (kind) {
    case kKindF8N128: return launch_f8_one<128>(l);
    case kKindF8N256: return launch_f8_one<256>(l);
    default: return launch_pair_kernel<false, false, false, true>(l);
  }
}

}  // namespace sk
