// Streaming a K x N row-major bf16 matrix (the B operand of a one-row-of-tiles GEMM, 64 x 14336
// x 4096) through TMA with nothing else running: the read rate each access pattern reaches.
//
// CTA (strip, part) reads columns [strip * W, (strip + 1) * W) of rows [part * K / P, (part +
// 1) * K / P), H rows per stage, as W / box_cols boxes of box_cols x H, through a ring of S
// stages in shared memory.  One thread issues the copies, another waits for each stage and hands
// it back at once (or, where a hold is given, that many nanoseconds after it lands, as an MMA
// reading the stage would), so the only limit is how fast the bytes arrive.  Three copies of the matrix
// (351 MB, well over the 129 MB L2) are read in turn by launches timed back to back, so every
// launch reads from DRAM and the event timer's ~2 us resolution is spread over six launches.
// Each line of output is one pattern: its parameters, the CTAs it runs, the time per launch and
// the GB/s of the matrix bytes.
//
// Every wait is bounded: a stage that does not arrive within ~2 s sets an error word, and the
// CTA waits (bounded again) for the copies it issued before it exits.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <vector>

#define CHECK(x)                                                                  \
  do {                                                                            \
    cudaError_t e_ = (x);                                                         \
    if (e_ != cudaSuccess) {                                                      \
      std::printf("{\"error\": \"%s at line %d\"}\n", cudaGetErrorString(e_), __LINE__); \
      return 1;                                                                   \
    }                                                                             \
  } while (0)

namespace {

constexpr int kK = 4096, kN = 14336;

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ bool bar_try(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` for at most ~2 s.
__device__ __forceinline__ bool bar_wait(uint64_t* bar, uint32_t parity) {
  const uint64_t t0 = now_ns();
  while (!bar_try(bar, parity))
    if (now_ns() - t0 > 2000000000ull) return false;
  return true;
}

__global__ void __launch_bounds__(64, 1)
    stream_kernel(const __grid_constant__ CUtensorMap tm, int strip_cols, int box_cols, int box_h,
                  int stages, int parts, int hold_ns, uint32_t* err) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const int stage_bytes = strip_cols * 2 * box_h;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + stages * stage_bytes);
  uint64_t* empty = full + stages;
  const int strip = blockIdx.x / parts, part = blockIdx.x % parts;
  const int rows = kK / parts;
  const int row0 = part * rows;
  const int iters = rows / box_h;
  if (threadIdx.x == 0) {
    for (int s = 0; s < stages; ++s) {
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&full[s])));
      asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(&empty[s])));
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int issued = 0;
    bool ok = true;
    for (int i = 0; i < iters; ++i) {
      const int s = i % stages;
      const uint32_t par = static_cast<uint32_t>(i / stages) & 1u;
      if (!bar_wait(&empty[s], par ^ 1u)) {
        ok = false;
        break;
      }
      asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(
                       smem_u32(&full[s])),
                   "r"(stage_bytes)
                   : "memory");
      for (int b = 0; b < strip_cols / box_cols; ++b) {
        uint8_t* dst = ring + s * stage_bytes + b * box_cols * 2 * box_h;
        asm volatile(
            "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
            " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
            "l"(reinterpret_cast<uint64_t>(&tm)), "r"(smem_u32(&full[s])),
            "r"(strip * strip_cols + b * box_cols), "r"(row0 + i * box_h)
            : "memory");
      }
      ++issued;
    }
    if (!ok) {
      atomicExch(err, 1u);
      // let the copies already issued land before shared memory goes away
      for (int j = issued - stages < 0 ? 0 : issued - stages; j < issued; ++j)
        bar_wait(&full[j % stages], static_cast<uint32_t>(j / stages) & 1u);
    }
  } else if (threadIdx.x == 32) {
    for (int i = 0; i < iters; ++i) {
      const int s = i % stages;
      if (!bar_wait(&full[s], static_cast<uint32_t>(i / stages) & 1u)) {
        atomicExch(err, 2u);
        break;
      }
      if (hold_ns > 0) {   // bounded: hold_ns is at most a few microseconds
        const uint64_t h0 = now_ns();
        while (now_ns() - h0 < static_cast<uint64_t>(hold_ns)) {
        }
      }
      asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(&empty[s]))
                   : "memory");
    }
  }
  __syncthreads();
}

__global__ void read_kernel(const uint4* p, size_t n, uint32_t* sink) {
  uint32_t acc = 0;
  for (size_t i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    acc ^= p[i].x;
  if (acc == 0x12345678u) *sink = acc;
}

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct Pattern {
  int strip_cols, box_cols, box_h, stages, parts;
  CUtensorMapL2promotion promo;
  int hold_ns;   // the consumer's hold per stage (0: handed back at once)
};

}  // namespace

int main() {
  void* fnp = nullptr;
  cudaDriverEntryPointQueryResult q;
  CHECK(cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fnp, 12000, cudaEnableDefault,
                                         &q));
  if (fnp == nullptr || q != cudaDriverEntryPointSuccess) {
    std::printf("{\"error\": \"no tensor-map encoder\"}\n");
    return 1;
  }
  const EncodeFn encode = reinterpret_cast<EncodeFn>(fnp);
  int sms = 0;
  CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  constexpr int kCopies = 3, kLaunches = 6;
  void* B[kCopies] = {};
  const size_t b_bytes = static_cast<size_t>(kK) * kN * 2;
  for (int c = 0; c < kCopies; ++c) {
    CHECK(cudaMalloc(&B[c], b_bytes));
    CHECK(cudaMemset(B[c], 0, b_bytes));
  }
  const size_t flush_bytes = 256ull << 20;
  void* flush = nullptr;
  CHECK(cudaMalloc(&flush, flush_bytes));
  uint32_t* err = nullptr;
  CHECK(cudaMalloc(&err, 8));
  CHECK(cudaMemset(err, 0, 8));
  CHECK(cudaFuncSetAttribute(stream_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024));

  const CUtensorMapL2promotion P0 = CU_TENSOR_MAP_L2_PROMOTION_NONE,
                               P256 = CU_TENSOR_MAP_L2_PROMOTION_L2_256B;
  std::vector<Pattern> pats = {
      // the skinny GEMM's own patterns: 128-wide strips (2 boxes of 64 x 64), 96-wide (3 of
      // 32 x 64), with and without 256-byte L2 promotion
      {128, 64, 64, 6, 1, P256}, {96, 32, 64, 7, 1, P256}, {128, 64, 64, 6, 1, P0},
      {96, 32, 64, 7, 1, P0},
      // the same strips with taller boxes (more K rows per stage) and fewer stages
      {128, 64, 32, 12, 1, P256}, {128, 64, 128, 2, 1, P256}, {128, 64, 128, 3, 1, P256},
      {128, 64, 128, 4, 1, P256}, {128, 64, 128, 6, 1, P256}, {128, 64, 256, 2, 1, P256},
      {128, 64, 256, 3, 1, P256}, {96, 32, 128, 3, 1, P256},  {96, 32, 128, 6, 1, P256},
      {96, 32, 256, 3, 1, P256},
      // the strips split in K over two or more CTAs per SM
      {128, 64, 64, 3, 2, P256},  {128, 64, 64, 6, 2, P256},  {128, 64, 128, 3, 2, P256},
      {256, 64, 64, 3, 3, P256},  {512, 256, 16, 6, 6, P256}, {512, 256, 32, 3, 6, P256},
      // narrow strips, many CTAs
      {64, 64, 64, 6, 1, P256},   {64, 64, 128, 3, 1, P256},  {64, 64, 256, 2, 1, P256},
      {32, 32, 64, 6, 1, P256},
      // 96-wide strips in 128-row boxes with a 200 ns hold per stage, as the tall-stage kernel's
      // MMAs take: how many stages hide it
      {96, 32, 128, 5, 1, P256, 200}, {96, 32, 128, 6, 1, P256, 200}, {96, 32, 128, 7, 1, P256, 200},
      {96, 32, 128, 8, 1, P256, 200}, {96, 32, 128, 5, 1, P256, 0},   {96, 32, 128, 7, 1, P256, 0},
      {128, 64, 128, 4, 1, P256, 260}, {128, 64, 128, 6, 1, P256, 260},
  };

  cudaEvent_t e0, e1;
  CHECK(cudaEventCreate(&e0));
  CHECK(cudaEventCreate(&e1));
  for (const Pattern& p : pats) {
    CUtensorMap tm[kCopies];
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kN), static_cast<cuuint64_t>(kK)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kN) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(p.box_cols), static_cast<cuuint32_t>(p.box_h)};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = p.box_cols * 2 == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : p.box_cols * 2 == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                         : CU_TENSOR_MAP_SWIZZLE_NONE;
    bool encoded = true;
    for (int c = 0; c < kCopies; ++c)
      encoded = encoded &&
                encode(&tm[c], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B[c], dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, sw, p.promo,
                       CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
    if (!encoded) {
      std::printf("{\"strip\": %d, \"box\": [%d, %d], \"error\": \"encode\"}\n", p.strip_cols,
                  p.box_cols, p.box_h);
      continue;
    }
    const int strips = (kN + p.strip_cols - 1) / p.strip_cols;
    const int ctas = strips * p.parts;
    // bytes of the matrix the launch reads (a ragged last strip or K split reads a little less)
    const double bytes = static_cast<double>(std::min(strips * p.strip_cols, kN)) * 2.0 *
                         p.parts * ((kK / p.parts) / p.box_h) * p.box_h;
    const size_t smem = 1024 + static_cast<size_t>(p.stages) * p.strip_cols * 2 * p.box_h +
                        16 * p.stages;
    if (smem > 227 * 1024) continue;
    int per_sm = 0;
    CHECK(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, stream_kernel, 64, smem));
    float best = 1e30f;
    std::vector<float> ts;
    for (int rep = 0; rep < 7; ++rep) {
      CHECK(cudaMemsetAsync(flush, rep, flush_bytes));
      read_kernel<<<4 * sms, 512>>>(static_cast<const uint4*>(flush), flush_bytes / 16, err + 1);
      CHECK(cudaEventRecord(e0));
      for (int l = 0; l < kLaunches; ++l)
        stream_kernel<<<ctas, 64, smem>>>(tm[l % kCopies], p.strip_cols, p.box_cols, p.box_h,
                                          p.stages, p.parts, p.hold_ns, err);
      CHECK(cudaEventRecord(e1));
      CHECK(cudaEventSynchronize(e1));
      float ms = 0;
      CHECK(cudaEventElapsedTime(&ms, e0, e1));
      if (rep >= 1) ts.push_back(ms / kLaunches);
    }
    uint32_t h_err = 0;
    CHECK(cudaMemcpy(&h_err, err, 4, cudaMemcpyDeviceToHost));
    std::sort(ts.begin(), ts.end());
    best = ts[ts.size() / 2];
    std::printf(
        "{\"strip_cols\": %d, \"box\": [%d, %d], \"stages\": %d, \"k_parts\": %d, \"l2_promo\": %d, "
        "\"hold_ns\": %d, \"ctas\": %d, \"ctas_per_sm\": %d, \"us\": %.2f, \"GBs\": %.0f, \"err\": %u}\n",
        p.strip_cols, p.box_cols, p.box_h, p.stages, p.parts, p.promo == P256 ? 256 : 0, p.hold_ns, ctas,
        per_sm, best * 1000.0f, bytes / (best * 1e-3) / 1e9, h_err);
    std::fflush(stdout);
    if (h_err != 0) return 2;
  }
  return 0;
}
