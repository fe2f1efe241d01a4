// Column sums of a bf16 matrix (the bias gradient of addmm: dbias[n] = sum over m of
// dC[m][n]).  Two deterministic passes: partial sums over row chunks, then a sum over the
// chunks in chunk order; fp32 accumulation.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "sk_launch.h"

namespace sk {

constexpr int kColsumThreads = 256;
constexpr int64_t kColsumRowsPerChunk = 128;

// Block (x, y): columns [2 * (x * 256 + t), +2), rows [y * 128, +128).  N is even.
__global__ void __launch_bounds__(kColsumThreads) colsum_partial_kernel(
    const __nv_bfloat16* __restrict__ x, int64_t M, int64_t N, float* __restrict__ partial) {
  const int64_t col = 2 * (static_cast<int64_t>(blockIdx.x) * kColsumThreads + threadIdx.x);
  const int64_t r0 = static_cast<int64_t>(blockIdx.y) * kColsumRowsPerChunk;
  const int64_t r1 = (r0 + kColsumRowsPerChunk < M) ? r0 + kColsumRowsPerChunk : M;
  if (col >= N) return;
  float s0 = 0.0f, s1 = 0.0f;
  for (int64_t r = r0; r < r1; ++r) {
    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(x + r * N + col));
    s0 += v.x;
    s1 += v.y;
  }
  float* out = partial + static_cast<int64_t>(blockIdx.y) * N + col;
  out[0] = s0;
  out[1] = s1;
}

__global__ void __launch_bounds__(kColsumThreads) colsum_final_kernel(
    const float* __restrict__ partial, int64_t chunks, int64_t N, void* out, int out_bf16) {
  const int64_t col = static_cast<int64_t>(blockIdx.x) * kColsumThreads + threadIdx.x;
  if (col >= N) return;
  float s = 0.0f;
  for (int64_t c = 0; c < chunks; ++c) s += partial[c * N + col];
  if (out_bf16) {
    static_cast<__nv_bfloat16*>(out)[col] = __float2bfloat16_rn(s);
  } else {
    static_cast<float*>(out)[col] = s;
  }
}

int64_t colsum_scratch_bytes(int64_t M, int64_t N) {
  const int64_t chunks = (M + kColsumRowsPerChunk - 1) / kColsumRowsPerChunk;
  return chunks * N * static_cast<int64_t>(sizeof(float));
}

cudaError_t colsum_bf16(const void* x, int64_t M, int64_t N, void* out, int out_bf16,
                        float* scratch, cudaStream_t stream) {
  const int64_t chunks = (M + kColsumRowsPerChunk - 1) / kColsumRowsPerChunk;
  const int64_t col_pairs = N / 2;
  const dim3 grid1(static_cast<unsigned>((col_pairs + kColsumThreads - 1) / kColsumThreads),
                   static_cast<unsigned>(chunks));
  colsum_partial_kernel<<<grid1, kColsumThreads, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), M, N, scratch);
  const dim3 grid2(static_cast<unsigned>((N + kColsumThreads - 1) / kColsumThreads));
  colsum_final_kernel<<<grid2, kColsumThreads, 0, stream>>>(scratch, chunks, N, out, out_bf16);
  return cudaGetLastError();
}

}  // namespace sk
