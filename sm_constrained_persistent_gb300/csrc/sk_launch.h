// Host-side interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "sk_kernel_args.h"

namespace sk {

// Kernel variants: operand format x CTA tile.  The pair variants run 2-CTA clusters on
// 256 x 256 tiles (one CTA per 128 rows); `Launch::grid` always counts CTAs.
enum Variant : int {
  kVariantBf16N128 = 0,
  kVariantBf16N256 = 1,
  kVariantMxN128 = 2,
  kVariantBf16Pair = 3,
  kVariantMxPair = 4,
  kNumVariants = 5
};

inline bool variant_is_pair(int v) { return v == kVariantBf16Pair || v == kVariantMxPair; }

struct Launch {
  const CUtensorMap* tmA;
  const CUtensorMap* tmB;
  const CUtensorMap* tmSfa;   // pair MXFP4 only: rearranged scales as rows of 1 KB
  const CUtensorMap* tmSfb;
  Args args;
  int grid;
  bool cooperative;   // ask the driver to guarantee that every CTA is resident at once
  cudaStream_t stream;
};

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

}  // namespace sk
