// MXFP4 instantiation of the GEMM kernel, the scale-layout kernel, and the variant dispatch.
#include "sk_kernel.cuh"
#include "sk_launch.h"

namespace sk {

cudaError_t launch_bf16(int tile_n, const Launch& l);
cudaError_t setup_bf16(int tile_n, int* ctas_per_sm);
size_t smem_bf16(int tile_n);

__global__ void __launch_bounds__(256) mx_scale_prep_kernel(const uint8_t* __restrict__ scales,
                                                            int64_t rows, int64_t kblocks,
                                                            int64_t row_blocks, int64_t kgroups,
                                                            uint32_t* __restrict__ out) {
  const int64_t total = row_blocks * kgroups * 128;   // 32-bit words
  for (int64_t w = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; w < total;
       w += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t within = w % 128;
    const int64_t group = w / 128;
    const int64_t g = group % kgroups;
    const int64_t rb = group / kgroups;
    const int64_t i = within / 4;
    const int64_t c = within % 4;
    const int64_t r = rb * 128 + c * 32 + i;
    uint32_t word = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int64_t kb = g * 4 + j;
      const uint32_t byte = (r < rows && kb < kblocks) ? scales[r * kblocks + kb] : 127u;
      word |= byte << (8 * j);
    }
    out[w] = word;
  }
}

cudaError_t mx_scale_prep(const uint8_t* scales, int64_t rows, int64_t kblocks,
                          int64_t row_blocks, int64_t kgroups, uint8_t* out, int sm_count,
                          cudaStream_t stream) {
  const int64_t total = row_blocks * kgroups * 128;
  int64_t blocks = (total + 255) / 256;
  const int64_t cap = static_cast<int64_t>(sm_count) * 8;
  if (blocks > cap) blocks = cap;
  if (blocks < 1) blocks = 1;
  mx_scale_prep_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      scales, rows, kblocks, row_blocks, kgroups, reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

size_t variant_smem_bytes(int variant) {
  switch (variant) {
    case kVariantBf16N128: return smem_bf16(128);
    case kVariantBf16N256: return smem_bf16(256);
    default: return Cfg<true, 128>::kSmemBytes;
  }
}

cudaError_t variant_setup(int variant, int* ctas_per_sm) {
  if (variant == kVariantBf16N128) return setup_bf16(128, ctas_per_sm);
  if (variant == kVariantBf16N256) return setup_bf16(256, ctas_per_sm);
  using Cf = Cfg<true, 128>;
  cudaError_t e = cudaFuncSetAttribute(gemm_kernel<true, 128>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(Cf::kSmemBytes));
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, gemm_kernel<true, 128>,
                                                       kThreads, Cf::kSmemBytes);
}

cudaError_t variant_launch(int variant, const Launch& l) {
  if (variant == kVariantBf16N128) return launch_bf16(128, l);
  if (variant == kVariantBf16N256) return launch_bf16(256, l);
  using Cf = Cfg<true, 128>;
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
  return cudaLaunchKernelEx(&cfg, gemm_kernel<true, 128>, *l.tmA, *l.tmB, l.args);
}

}  // namespace sk
