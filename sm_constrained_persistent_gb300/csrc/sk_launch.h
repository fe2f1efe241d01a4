// Host-side interface between the C-ABI layer and the kernel translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "sk_kernel_args.h"

namespace sk {

// Kernel variants: operand format x CTA tile width.
enum Variant : int { kVariantBf16N128 = 0, kVariantBf16N256 = 1, kVariantMxN128 = 2, kNumVariants = 3 };

struct Launch {
  const CUtensorMap* tmA;
  const CUtensorMap* tmB;
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

// Rearranges row-major [rows][kblocks] E8M0 scales into [row_blocks][kgroups][512]: in group
// (rb, g), byte 16*i + 4*c + j holds scale (row rb*128 + 32*c + i, block 4*g + j); positions
// outside the matrix hold 127 (scale 1.0, so the zero-filled operand padding stays 0).
cudaError_t mx_scale_prep(const uint8_t* scales, int64_t rows, int64_t kblocks,
                          int64_t row_blocks, int64_t kgroups, uint8_t* out, int sm_count,
                          cudaStream_t stream);

}  // namespace sk
