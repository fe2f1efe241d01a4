// Host-side interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include "sk_kernel_args.h"

namespace sk {

// A named NVTX range around one C-ABI call, so a profiler's timeline attributes the kernels to
// the call that queued them (nearly free when no profiler is attached).
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

// Kernel variants: kernel kind (operand format x CTA tile) x operand layout.  The pair kinds
// run 2-CTA clusters on 256 x 256 tiles (one CTA per 128 rows); `Launch::grid` always counts
// CTAs.  Layout bit 0: A stored transposed (K x M); bit 1: B stored transposed (N x K); the
// transposed layouts exist for bf16 only.
enum Kind : int {
  kKindBf16N128 = 0,
  kKindBf16N256 = 1,
  kKindMxN128 = 2,
  kKindBf16Pair = 3,
  kKindMxPair = 4,
  kKindF8N128 = 5,     // fp8 (E4M3) kinds: plain layout only
  kKindF8N256 = 6,
  kKindF8Pair = 7,
  kKindBf16N96 = 8,    // 96-wide bf16 tiles (one row of tiles streaming B): plain layout only
  kKindBf16N128Tall = 9,   // bf16, at most 64 rows of A: 128 K per stage (plain layout only)
  kKindBf16N96Tall = 10,
  kNumKinds = 11
};
constexpr int kNumLayouts = 4;
constexpr int kNumVariants = kNumKinds * kNumLayouts;
constexpr int variant_of(int kind, int layout) { return kind * kNumLayouts + layout; }
inline int variant_kind(int v) { return v / kNumLayouts; }
inline int variant_layout(int v) { return v % kNumLayouts; }
inline bool variant_is_pair(int v) {
  return variant_kind(v) == kKindBf16Pair || variant_kind(v) == kKindMxPair ||
         variant_kind(v) == kKindF8Pair;
}
// the plain (untransposed) layout of each kind
enum : int {
  kVariantBf16N128 = variant_of(kKindBf16N128, 0),
  kVariantBf16N256 = variant_of(kKindBf16N256, 0),
  kVariantMxN128 = variant_of(kKindMxN128, 0),
  kVariantBf16Pair = variant_of(kKindBf16Pair, 0),
  kVariantMxPair = variant_of(kKindMxPair, 0)
};

struct Launch {
  const CUtensorMap* tmA;
  const CUtensorMap* tmB;
  const CUtensorMap* tmSfa;   // pair MXFP4 only: rearranged scales as rows of 1 KB
  const CUtensorMap* tmSfb;
  const CUtensorMap* tmC;     // C as boxes of 32 rows x 64 bytes (null: no TMA stores; the
                              // one-CTA kernels then store directly, args.c_tma = 0)
  Args args;
  int grid;
  bool cooperative;   // ask the driver to guarantee that every CTA is resident at once
  cudaStream_t stream;
};

// Per translation unit: set-up (shared-memory limit + occupancy) and launch of one kind.
cudaError_t setup_bf16_n128(int layout, int* ctas_per_sm);
cudaError_t launch_bf16_n128(int layout, const Launch& l);
cudaError_t setup_bf16_n256(int layout, int* ctas_per_sm);
cudaError_t launch_bf16_n256(int layout, const Launch& l);
cudaError_t setup_bf16_n96(int* ctas_per_sm);
cudaError_t launch_bf16_n96(const Launch& l);
// Tall stages (128 K per stage, 64 rows of A) for 128- or 96-wide tiles (`bn`).
cudaError_t setup_bf16_tall(int bn, int* ctas_per_sm);
cudaError_t launch_bf16_tall(int bn, const Launch& l);
size_t tall_smem_bytes(int bn);
cudaError_t setup_bf16_pair(int layout, int* max_clusters);
cudaError_t launch_bf16_pair(int layout, const Launch& l);
cudaError_t setup_mx_pair(int* max_clusters);
cudaError_t launch_mx_pair(const Launch& l);
cudaError_t setup_f8(int kind, int* ctas_or_clusters);
cudaError_t launch_f8(int kind, const Launch& l);

// Frees the device copies, streams and events of the host-buffer entry points.
void release_host_stages();
// The same for the host-buffer staging of one (device, stream) only; the device must be
// current.  Frees are queued on `stream`.
cudaError_t release_host_stage(int device, cudaStream_t stream);
// Device bytes the host-buffer staging of (device, stream) holds.
int64_t host_stage_bytes(int device, cudaStream_t stream);

// Dynamic shared memory of a variant, in bytes.
size_t variant_smem_bytes(int variant);
// Raises the variant's dynamic shared-memory limit on the current device and reports how many
// of its CTAs fit on one SM.
cudaError_t variant_setup(int variant, int* ctas_per_sm);
cudaError_t variant_launch(int variant, const Launch& l);
// Pair variants: raises the shared-memory limit and reports how many 2-CTA clusters of the
// variant can be resident at once on the current device.
cudaError_t pair_variant_setup(int variant, int* max_clusters);
cudaError_t pair_variant_launch(int variant, const Launch& l);
size_t pair_variant_smem_bytes(int variant);

// Rearranges the row-major [rows][kblocks] E8M0 scales of A and of B into one buffer of
// [row_blocks][kgroups][512]: A's row blocks first, then B's.  In group (rb, g), byte
// 16*i + 4*c + j holds scale (row rb*128 + 32*c + i, block 4*g + j); positions outside the
// matrix hold 127 (scale 1.0, so the zero-filled operand padding stays 0).  One launch.
cudaError_t mx_scale_prep(const uint8_t* a_scales, int64_t a_rows, int64_t a_row_blocks,
                          const uint8_t* b_scales, int64_t b_rows, int64_t b_row_blocks,
                          int64_t kblocks, int64_t kgroups, uint8_t* out, cudaStream_t stream);

// Column sums of a row-major M x N bf16 matrix (N even) into N values of fp32 (out_bf16 = 0)
// or bf16; `scratch` holds colsum_scratch_bytes(M, N) bytes.
int64_t colsum_scratch_bytes(int64_t M, int64_t N);
cudaError_t colsum_bf16(const void* x, int64_t M, int64_t N, void* out, int out_bf16,
                        float* scratch, cudaStream_t stream);

}  // namespace sk
