// Kernel argument block of the GEMM kernels (plain data, shared by host and device code).
#pragma once

#include <cstdint>

#include "sk_schedule.cuh"

namespace sk {

struct Args {
  const void* bias;      // null or N values of C's dtype
  void* C;
  int64_t M, N, K;
  int32_t out_bf16;      // C (and bias) dtype: 1 = bf16, 0 = fp32
  int32_t inject_drop;   // fault injection: CTA drop_cta never releases its partial
  int32_t drop_cta;
  uint32_t epoch;        // value a contributor publishes in its flag for this launch
  Plan plan;
  float* P;              // grid slots of kBM * BN fp32 partials
  uint32_t* flags;       // grid flags
  uint32_t* err;         // [0] status, [1] site, [2] cta, [3] linear tile
  uint64_t timeout_ns;
  const uint8_t* sfa;    // MXFP4 scales, rearranged: [row block][k group][512 bytes]
  const uint8_t* sfb;
  int64_t sf_kgroups;    // k groups (4 scale blocks = 128 K elements each) per row block
  int32_t c_tma;         // one-CTA kernels: 1 = C is written through the tmC tensor map
  int32_t replay;        // 1: the launch is captured into a CUDA graph, so every replay sees the
                         // same epoch; each flag is then cleared by its one reader
  uint32_t* sm_record;   // null, or one entry per CTA: the SM it ran on
};

}  // namespace sk
