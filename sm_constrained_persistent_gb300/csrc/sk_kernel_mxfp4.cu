// MXFP4 instantiation of the GEMM kernel, the scale-layout kernel, and the variant dispatch.
#include "sk_kernel.cuh"
#include "sk_kernel_pair.cuh"
#include "sk_launch.h"

namespace sk {

// Word of output group (row block, k group g) for row r: scales of blocks 4g .. 4g+3, padding
// (127, scale 1.0) outside the matrix.
__device__ __forceinline__ uint32_t scale_word(const uint8_t* __restrict__ s, int32_t r, int32_t rows,
                                               int32_t kblocks, int32_t g) {
  const int32_t kb0 = g * 4;
  if (r < rows && kb0 + 4 <= kblocks && (kblocks & 3) == 0)
    return __ldg(reinterpret_cast<const uint32_t*>(s + static_cast<int64_t>(r) * kblocks + kb0));
  uint32_t word = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int32_t kb = kb0 + j;
    const uint32_t byte = (r < rows && kb < kblocks) ? s[static_cast<int64_t>(r) * kblocks + kb] : 127u;
    word |= byte << (8 * j);
  }
  return word;
}

// One 128-thread block per row block rb and span of kPrepGroups 512-byte output groups: in
// group g, thread t writes word t, i.e. the scales of row rb*128 + 32*(t%4) + t/4, blocks 4g ..
// 4g+3.  Where the span's 32 scale bytes of a row are whole and 16-byte aligned, the thread reads
// them with two 16-byte loads.  blockIdx.y < a_blocks covers A, the rest B.
constexpr int kPrepGroups = 8;

__global__ void __launch_bounds__(128) mx_scale_prep_kernel(
    const uint8_t* __restrict__ sa, int32_t a_rows, int32_t a_blocks, const uint8_t* __restrict__ sb,
    int32_t b_rows, int32_t kblocks, int32_t kgroups, uint32_t* __restrict__ out) {
  const int32_t g0 = blockIdx.x * kPrepGroups;
  int32_t rb = blockIdx.y;
  const bool is_a = rb < a_blocks;
  const uint8_t* s = is_a ? sa : sb;
  const int32_t rows = is_a ? a_rows : b_rows;
  const int32_t t = threadIdx.x;
  const int32_t r = (is_a ? rb : rb - a_blocks) * 128 + (t & 3) * 32 + (t >> 2);
  uint32_t* dst = out + (static_cast<int64_t>(rb) * kgroups + g0) * 128 + t;
  const uint8_t* src = s + static_cast<int64_t>(r) * kblocks + g0 * 4;
  const bool whole = r < rows && (kblocks & 15) == 0 && g0 * 4 + 4 * kPrepGroups <= kblocks &&
                     g0 + kPrepGroups <= kgroups && (reinterpret_cast<uintptr_t>(s) & 15) == 0;
  if (whole) {
    const uint4 lo = __ldg(reinterpret_cast<const uint4*>(src));
    const uint4 hi = __ldg(reinterpret_cast<const uint4*>(src) + 1);
    const uint32_t w[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int j = 0; j < kPrepGroups; ++j) dst[j * 128] = w[j];
  } else {
    for (int j = 0; j < kPrepGroups && g0 + j < kgroups; ++j)
      dst[j * 128] = scale_word(s, r, rows, kblocks, g0 + j);
  }
}

cudaError_t mx_scale_prep(const uint8_t* a_scales, int64_t a_rows, int64_t a_row_blocks,
                          const uint8_t* b_scales, int64_t b_rows, int64_t b_row_blocks,
                          int64_t kblocks, int64_t kgroups, uint8_t* out, cudaStream_t stream) {
  const dim3 grid(static_cast<unsigned>((kgroups + kPrepGroups - 1) / kPrepGroups),
                  static_cast<unsigned>(a_row_blocks + b_row_blocks));
  mx_scale_prep_kernel<<<grid, 128, 0, stream>>>(
      a_scales, static_cast<int32_t>(a_rows), static_cast<int32_t>(a_row_blocks), b_scales,
      static_cast<int32_t>(b_rows), static_cast<int32_t>(kblocks), static_cast<int32_t>(kgroups),
      reinterpret_cast<uint32_t*>(out));
  return cudaGetLastError();
}

size_t variant_smem_bytes(int variant) {
  switch (variant_kind(variant)) {
    case kKindBf16N128: return Cfg<false, 128>::kSmemBytes;
    case kKindBf16N256: return Cfg<false, 256>::kSmemBytes;
    case kKindMxN128: return Cfg<true, 128>::kSmemBytes;
    case kKindBf16Pair: return PairCfg<false>::kSmemBytes;
    case kKindF8N128: return Cfg<false, 128, false, false, true>::kSmemBytes;
    case kKindF8N256: return Cfg<false, 256, false, false, true>::kSmemBytes;
    case kKindF8Pair: return PairCfg<false, false, false, true>::kSmemBytes;
    case kKindBf16N96: return Cfg<false, 96>::kSmemBytes;
    case kKindBf16N128Tall: return tall_smem_bytes(128);
    case kKindBf16N96Tall: return tall_smem_bytes(96);
    default: return PairCfg<true>::kSmemBytes;
  }
}

cudaError_t variant_setup(int variant, int* ctas_per_sm) {
  const int layout = variant_layout(variant);
  switch (variant_kind(variant)) {
    case kKindBf16N128: return setup_bf16_n128(layout, ctas_per_sm);
    case kKindBf16N256: return setup_bf16_n256(layout, ctas_per_sm);
    case kKindMxN128: {
      using Cf = Cfg<true, 128>;
      cudaError_t e = cudaFuncSetAttribute(gemm_kernel<true, 128>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           static_cast<int>(Cf::kSmemBytes));
      if (e != cudaSuccess) return e;
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, gemm_kernel<true, 128>,
                                                           kThreads, Cf::kSmemBytes);
    }
    case kKindF8N128:
    case kKindF8N256: return setup_f8(variant_kind(variant), ctas_per_sm);
    case kKindBf16N96: return setup_bf16_n96(ctas_per_sm);
    case kKindBf16N128Tall: return setup_bf16_tall(128, ctas_per_sm);
    case kKindBf16N96Tall: return setup_bf16_tall(96, ctas_per_sm);
    default: return cudaErrorInvalidValue;   // pair kinds: pair_variant_setup
  }
}

cudaError_t variant_launch(int variant, const Launch& l) {
  const int layout = variant_layout(variant);
  switch (variant_kind(variant)) {
    case kKindBf16N128: return launch_bf16_n128(layout, l);
    case kKindBf16N256: return launch_bf16_n256(layout, l);
    case kKindMxN128: {
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
      return cudaLaunchKernelEx(&cfg, gemm_kernel<true, 128>, *l.tmA, *l.tmB,
                            l.tmC != nullptr ? *l.tmC : *l.tmA, l.args);
    }
    case kKindF8N128:
    case kKindF8N256: return launch_f8(variant_kind(variant), l);
    case kKindBf16N96: return launch_bf16_n96(l);
    case kKindBf16N128Tall: return launch_bf16_tall(128, l);
    case kKindBf16N96Tall: return launch_bf16_tall(96, l);
    default: return cudaErrorInvalidValue;   // pair kinds: pair_variant_launch
  }
}

cudaError_t pair_variant_setup(int variant, int* max_clusters) {
  if (variant_kind(variant) == kKindF8Pair) return setup_f8(kKindF8Pair, max_clusters);
  return variant_kind(variant) == kKindMxPair ? setup_mx_pair(max_clusters)
                                              : setup_bf16_pair(variant_layout(variant), max_clusters);
}

cudaError_t pair_variant_launch(int variant, const Launch& l) {
  if (variant_kind(variant) == kKindF8Pair) return launch_f8(kKindF8Pair, l);
  return variant_kind(variant) == kKindMxPair ? launch_mx_pair(l)
                                              : launch_bf16_pair(variant_layout(variant), l);
}

size_t pair_variant_smem_bytes(int variant) { return variant_smem_bytes(variant); }

}  // namespace sk
