// Tensor-pipe instruction rate on sm_103a: back-to-back tcgen05.mma of one kind and shape per
// CTA (one CTA per SM, or one 2-CTA cluster per SM pair), timed by clock64 in the issuing thread
// and by %globaltimer (their ratio is the SM clock while the pipe is busy).  Operands are one
// shared-memory stage (A 16 KB at 0, B up to 32 KB at 16 KB), all zero or random bits; the
// accumulator is tensor-memory columns [0, 256) and the scale factors columns [384, 448) of one
// 512-column allocation.  Prints clocks per MMA and FLOP per clock per SM for each variant.
//
// This measures the ceiling a GEMM kernel's main loop can reach with each MMA kind: on GB300 the
// documented kinds all issue at a fixed number of clocks per MMA, and the FP4 kinds at four
// times the bf16 rate per clock.
#include <cstdint>
#include <cstdio>
#include <algorithm>
#include <vector>

#include <cuda_runtime.h>

namespace {

__device__ __forceinline__ uint32_t saddr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t sdesc(uint32_t a, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((a & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}

__device__ __forceinline__ uint64_t gtimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Waits for phase 0 of `bar`, at most 2 s; returns whether it completed.
__device__ __forceinline__ uint32_t wait_bounded(uint64_t* bar) {
  const uint64_t t0 = gtimer();
  uint32_t done = 0;
  while (!done && gtimer() - t0 < 2000000000ull) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(saddr(bar)), "r"(0)
        : "memory");
  }
  return done;
}

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

enum Kind { kF16, kF8, kMxf4, kMxf4Nvf4x2, kMxf4Nvf4x4 };

// Instruction descriptor: fp32 D; bf16 A/B (kind::f16), E4M3 A/B (kind::f8f6f4) or E2M1 A/B
// with E8M0 scales (block-scaled kinds); both K-major; N >> 3 at bit 17, M >> 4 at bit 24.
template <int kKind, int M, int N>
__host__ __device__ constexpr uint32_t idesc() {
  return kKind == kF16 ? ((1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(N >> 3) << 17) |
                          (uint32_t(M >> 4) << 24))
         : kKind == kF8 ? ((1u << 4) | (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24))
                        : ((1u << 7) | (1u << 10) | (1u << 23) | (uint32_t(N >> 3) << 17) |
                           (uint32_t(M >> 4) << 24));
}

template <int kKind, bool kPair>
__device__ __forceinline__ void mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t id,
                                    uint32_t sfa, uint32_t sfb, uint32_t acc) {
#define SK_MMA(CG, KIND)                                                                        \
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"                                \
               "tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], %1, %2, %3, p;\n\t}" ::"r"(d), \
               "l"(ad), "l"(bd), "r"(id), "r"(acc)                                              \
               : "memory")
#define SK_MMA_BS(CG, KIND)                                                                     \
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"                                \
               "tcgen05.mma.cta_group::" CG ".kind::" KIND " [%0], %1, %2, %3, [%5], [%6], p;\n\t}" \
               ::"r"(d), "l"(ad), "l"(bd), "r"(id), "r"(acc), "r"(sfa), "r"(sfb)               \
               : "memory")
  if constexpr (kPair) {
    if constexpr (kKind == kF16) SK_MMA("2", "f16");
    else if constexpr (kKind == kF8) SK_MMA("2", "f8f6f4");
    else if constexpr (kKind == kMxf4) SK_MMA_BS("2", "mxf4.block_scale.scale_vec::2X");
    else if constexpr (kKind == kMxf4Nvf4x2) SK_MMA_BS("2", "mxf4nvf4.block_scale.scale_vec::2X");
    else SK_MMA_BS("2", "mxf4nvf4.block_scale.scale_vec::4X");
  } else {
    if constexpr (kKind == kF16) SK_MMA("1", "f16");
    else if constexpr (kKind == kF8) SK_MMA("1", "f8f6f4");
    else if constexpr (kKind == kMxf4) SK_MMA_BS("1", "mxf4.block_scale.scale_vec::2X");
    else if constexpr (kKind == kMxf4Nvf4x2) SK_MMA_BS("1", "mxf4nvf4.block_scale.scale_vec::2X");
    else SK_MMA_BS("1", "mxf4nvf4.block_scale.scale_vec::4X");
  }
#undef SK_MMA
#undef SK_MMA_BS
}

// out[cta] = clocks, out[256 + cta] = nanoseconds of `iters` x 4 MMAs (issuing CTAs only).
template <int kKind, bool kPair, int N, int M>
__device__ void body(int iters, int random, unsigned long long* out) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + 65536);
  uint32_t* slot = reinterpret_cast<uint32_t*>(sm + 65536 + 64);
  for (int i = threadIdx.x; i < 65536 / 4; i += blockDim.x) {
    uint32_t x = (i + 1) * 2654435761u ^ (blockIdx.x * 40503u);
    x ^= x >> 15; x *= 2246822519u; x ^= x >> 13; x *= 3266489917u; x ^= x >> 16;
    // bf16 values stay finite (exponent <= 0x7E); E4M3 codes avoid NaN
    const uint32_t v = kKind == kF16 ? (x & 0xBF7FBF7Fu) : (kKind == kF8 ? (x & 0xF7F7F7F7u) : x);
    reinterpret_cast<uint32_t*>(sm)[i] = random ? v : 0u;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = kPair ? cluster_rank() : 0;
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(1) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 1) {
    if constexpr (kPair) {
      asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(slot)), "r"(512) : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
    } else {
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(slot)), "r"(512) : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if constexpr (kPair) cluster_sync();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tb = *slot;
  if (warp == 1 && lane == 0 && rank == 0) {
    const uint32_t a0 = saddr(sm), b0 = saddr(sm + 16384);
    const long long t0 = clock64();
    const uint64_t g0 = gtimer();
    for (int i = 0; i < iters; ++i) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {   // four MMAs of 32 bytes of K: one 128-byte swizzle row
        const uint32_t sf_id = kKind == kMxf4Nvf4x4 ? 0u : static_cast<uint32_t>((j & 1) * 2);
        const uint32_t id = idesc<kKind, M, N>() |
                            ((kKind == kF16 || kKind == kF8) ? 0u : ((sf_id << 29) | (sf_id << 4)));
        mma<kKind, kPair>(tb, sdesc(a0 + 32 * j, 16, 1024, 2), sdesc(b0 + 32 * j, 16, 1024, 2), id,
                          tb + 384, tb + 416, (i > 0 || j > 0) ? 1u : 0u);
      }
    }
    if constexpr (kPair) {
      asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
                   ::"r"(saddr(bar)), "h"(static_cast<uint16_t>(3)) : "memory");
    } else {
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar)) : "memory");
    }
    const uint32_t done = wait_bounded(bar);
    const long long t1 = clock64();
    const uint64_t g1 = gtimer();
    out[blockIdx.x] = done ? static_cast<unsigned long long>(t1 - t0) : 0ull;
    out[256 + blockIdx.x] = done ? (g1 - g0) : 0ull;
  } else if (kPair && warp == 1 && lane == 0) {
    wait_bounded(bar);   // the peer leaves only after the last MMA
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if constexpr (kPair) cluster_sync();
  if (warp == 1) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    if constexpr (kPair)
      asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(512) : "memory");
    else
      asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(512) : "memory");
  }
}

template <int kKind, int N, int M>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1)
    rate_pair(int iters, int random, unsigned long long* out) {
  body<kKind, true, N, M>(iters, random, out);
}

template <int kKind, int N, int M>
__global__ void __launch_bounds__(128, 1) rate_single(int iters, int random, unsigned long long* out) {
  body<kKind, false, N, M>(iters, random, out);
}

// M: rows of one MMA (256 or 128 for a pair, 128 or 64 for one CTA); the operands are read
// from the same 64 KB of shared memory whatever the shape.
template <int kKind, bool kPair, int N, int M = (kPair ? 256 : 128)>
bool run(const char* name, int sms, unsigned long long* d_out, int iters, int random) {
  constexpr int K = kKind == kF16 ? 16 : (kKind == kF8 ? 32 : 64);
  const size_t smem = 200 * 1024;   // one CTA per SM
  auto* fn = kPair ? rate_pair<kKind, N, M> : rate_single<kKind, N, M>;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
      cudaSuccess)
    return false;
  const int grid = sms & ~1;
  std::vector<unsigned long long> h(512);
  for (int rep = 0; rep < 2; ++rep) {   // the first launch warms up
    cudaMemset(d_out, 0, 512 * sizeof(unsigned long long));
    fn<<<grid, 128, smem>>>(iters, random, d_out);
    if (cudaDeviceSynchronize() != cudaSuccess) return false;
  }
  cudaMemcpy(h.data(), d_out, 512 * sizeof(unsigned long long), cudaMemcpyDeviceToHost);
  std::vector<double> clk, mhz;
  for (int i = 0; i < grid; ++i)
    if (h[i] && h[256 + i]) {
      clk.push_back(static_cast<double>(h[i]));
      mhz.push_back(1e3 * h[i] / h[256 + i]);
    }
  if (clk.empty()) return false;
  std::sort(clk.begin(), clk.end());
  std::sort(mhz.begin(), mhz.end());
  const double per_mma = clk[clk.size() / 2] / (4.0 * iters);
  const double flop_per_clk_sm = 2.0 * M * N * K / (kPair ? 2.0 : 1.0) / per_mma;
  printf("{\"variant\": \"%s\", \"cta_group\": %d, \"M\": %d, \"N\": %d, \"K\": %d, \"operands\": \"%s\", "
         "\"clk_per_mma\": %.1f, \"flop_per_clk_per_sm\": %.0f, \"x_bf16_rate\": %.3f, \"sm_mhz\": %.0f}\n",
         name, kPair ? 2 : 1, M, N, K, random ? "random" : "zero", per_mma, flop_per_clk_sm,
         flop_per_clk_sm / 8192.0, mhz[mhz.size() / 2]);
  return true;
}

}  // namespace

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long* d_out = nullptr;
  if (cudaMalloc(&d_out, 512 * sizeof(unsigned long long)) != cudaSuccess) return 1;
  const int iters = 16384;
  bool ok = true;
  for (int random = 0; random < 2; ++random) {
    ok &= run<kF16, true, 256>("kind::f16", sms, d_out, iters, random);
    ok &= run<kF8, true, 256>("kind::f8f6f4 (E4M3)", sms, d_out, iters, random);
    ok &= run<kMxf4, true, 256>("kind::mxf4.block_scale.scale_vec::2X", sms, d_out, iters, random);
    ok &= run<kMxf4Nvf4x2, true, 256>("kind::mxf4nvf4.block_scale.scale_vec::2X", sms, d_out, iters, random);
    ok &= run<kMxf4Nvf4x4, true, 256>("kind::mxf4nvf4.block_scale.scale_vec::4X", sms, d_out, iters, random);
  }
  ok &= run<kMxf4, true, 128>("kind::mxf4.block_scale.scale_vec::2X", sms, d_out, iters, 0);
  ok &= run<kF16, false, 256>("kind::f16", sms, d_out, iters, 0);
  ok &= run<kMxf4, false, 256>("kind::mxf4.block_scale.scale_vec::2X", sms, d_out, iters, 0);
  // smaller bf16 shapes, as a ragged edge tile could issue them
  ok &= run<kF16, true, 128>("kind::f16", sms, d_out, iters, 0);
  ok &= run<kF16, true, 256, 128>("kind::f16", sms, d_out, iters, 0);
  ok &= run<kF16, true, 128, 128>("kind::f16", sms, d_out, iters, 0);
  ok &= run<kF16, false, 128>("kind::f16", sms, d_out, iters, 0);
  ok &= run<kF16, false, 256, 64>("kind::f16", sms, d_out, iters, 0);
  cudaFree(d_out);
  return ok ? 0 : 1;
}
