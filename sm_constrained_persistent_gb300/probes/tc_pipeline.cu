// The per-stage structure of the MXFP4 SM-pair GEMM kernel, measured without operand loads: a
// 6-slot ring of tensor-memory scale-factor slots, a commit per stage, a producer handshake
// (full / empty mbarriers) and the scale-factor copies into tensor memory, added one at a time
// to back-to-back cta_group::2 kind::mxf4 MMAs (256 x 256 x 64, four per stage).  Operands are
// random bits in shared memory (A 16 KB at 0, B 16 KB at 16 KB, copy sources 12 KB at 32 KB,
// barriers at 48 KB); tensor memory holds the accumulator in columns [0, 256) and slot s in
// [256 + 24 s, 280 + 24 s).  Prints clocks per stage against the 512 the MMAs alone take.
//
// The copies of one stage's scales are either six 32x128b.warpx4 copies of the compact 512-byte
// groups or three 128x256b copies of the same scales laid out per lane; both fill the same
// tensor-memory columns.
#include <cstdio>
#include <cstdint>
#include <vector>
#include <algorithm>
#include <cuda_runtime.h>

__device__ __forceinline__ uint32_t saddr(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }
__device__ __forceinline__ uint64_t sdesc(uint32_t a, uint32_t lbo, uint32_t sbo, uint32_t layout) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((a & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo & 0x3FFFFu) >> 4) << 16;
  d |= static_cast<uint64_t>((sbo & 0x3FFFFu) >> 4) << 32;
  d |= 1ull << 46;
  d |= static_cast<uint64_t>(layout & 7u) << 61;
  return d;
}
__device__ __forceinline__ uint64_t gtimer() { uint64_t t; asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t)); return t; }
__device__ __forceinline__ bool try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
               : "=r"(done) : "r"(saddr(bar)), "r"(parity) : "memory");
  return done != 0;
}
// bounded wait (2 s)
__device__ __forceinline__ bool wait_b(uint64_t* bar, uint32_t parity) {
  if (try_wait(bar, parity)) return true;
  const uint64_t t0 = gtimer();
  while (!try_wait(bar, parity)) if (gtimer() - t0 > 2000000000ull) return false;
  return true;
}
__device__ __forceinline__ void arrive(uint64_t* bar) { asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(bar)) : "memory"); }
__device__ __forceinline__ void fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void commit_mc(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;"
               ::"r"(saddr(bar)), "h"(static_cast<uint16_t>(3)) : "memory");
}
__device__ __forceinline__ void commit_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar)) : "memory");
}
__device__ __forceinline__ void mma(uint32_t d, uint64_t ad, uint64_t bd, uint32_t id, uint32_t sfa, uint32_t sfb, uint32_t acc) {
  asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
               "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], [%6], p;\n\t}"
               ::"r"(d), "l"(ad), "l"(bd), "r"(id), "r"(acc), "r"(sfa), "r"(sfb) : "memory");
}
__device__ __forceinline__ void cp_x4(uint32_t taddr, uint64_t d) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}
__device__ __forceinline__ void cp_128x256(uint32_t taddr, uint64_t d) {
  asm volatile("tcgen05.cp.cta_group::2.128x256b [%0], %1;" ::"r"(taddr), "l"(d) : "memory");
}
__device__ __forceinline__ uint32_t cl_rank() { uint32_t r; asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r)); return r; }
__device__ __forceinline__ void cl_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

constexpr int S = 6;
constexpr uint32_t kIdesc = (1u << 7) | (1u << 10) | (1u << 23) | (uint32_t(256 >> 3) << 17) | (uint32_t(256 >> 4) << 24);

// copies of stage slot s: kind 0 = 6 x 32x128b.warpx4, kind 1 = 3 x 128x256b
__device__ __forceinline__ void copies(int kind, uint32_t tb, int s, uint32_t sf_s) {
  const uint32_t slot = tb + 256 + 24 * s;
  if (kind == 0) {
    for (int i = 0; i < 6; ++i) cp_x4(slot + 4 * i, sdesc(sf_s + 512 * i, 0, 128, 0));
  } else {
    for (int i = 0; i < 3; ++i) cp_128x256(slot + 8 * i, sdesc(sf_s + 4096 * i, 128, 256, 0));
  }
}

// V: 6 MMAs only; 0 + a commit per stage; 5 + producer handshake (full/empty), no copies;
// 1 + copy warp (warpx4) waited on through per-stage barriers; 2 the same with 128x256b copies;
// 4 warpx4 copies issued by the MMA thread itself; 7 handshake + copy warp (warpx4), as the
// kernel; 8 the same with 128x256b copies.
template <int V>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(128, 1) kpipe(int iters, unsigned long long* out) {
  extern __shared__ uint8_t raw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(sm + 49152);
  uint64_t* full = bars;          // S
  uint64_t* empty = bars + S;     // S
  uint64_t* sfr = bars + 2 * S;   // S
  uint64_t* done = bars + 3 * S;
  uint64_t* cpd = done + 1;
  uint32_t* slot = reinterpret_cast<uint32_t*>(cpd + 1);
  for (int i = threadIdx.x; i < 49152 / 4; i += blockDim.x) {
    uint32_t x = (i + 1) * 2654435761u ^ (blockIdx.x * 40503u);
    x ^= x >> 15; x *= 2246822519u; x ^= x >> 13; x *= 3266489917u; x ^= x >> 16;
    // scale bytes: keep them finite (E8M0 255 is NaN) by clearing bit 7 of every byte there
    reinterpret_cast<uint32_t*>(sm)[i] = (i >= 32768 / 4) ? (x & 0x7F7F7F7Fu) : x;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cl_rank();
  if (threadIdx.x == 0) {
    for (int i = 0; i < 3 * S + 2; ++i) asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bars + i)), "r"(1) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(saddr(slot)), "r"(512) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  }
  fence_before();
  __syncthreads();
  cl_sync();
  fence_after();
  const uint32_t tb = *slot;
  const uint32_t a0 = saddr(sm), b0 = saddr(sm + 16384), sf0 = saddr(sm + 32768);
  constexpr bool kCopyWarp = (V == 1 || V == 2 || V == 7 || V == 8);
  constexpr int kCopyKind = (V == 2 || V == 8) ? 1 : 0;
  constexpr bool kProducer = (V == 5 || V == 7 || V == 8);
  if (rank == 0 && lane == 0 && warp == 1) {
    bool ok = true;
    const long long c0 = clock64();
    const uint64_t g0 = gtimer();
    for (int it = 0; it < iters && ok; ++it) {
      const int s = it % S;
      const uint32_t ph = (it / S) & 1;
      if (kCopyWarp) ok = wait_b(&sfr[s], ph);
      else if (kProducer) ok = wait_b(&full[s], ph);
      if (!ok) break;
      if (V == 4) copies(0, tb, s, sf0);
      fence_after();
      const uint32_t sl = tb + 256 + 24 * s;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t g = j >> 1, id = (j & 1) * 2;
        mma(tb, sdesc(a0 + 32 * j, 16, 1024, 2), sdesc(b0 + 32 * j, 16, 1024, 2), kIdesc | (id << 29) | (id << 4),
            sl + 4 * g, sl + 8 + 8 * g, (it > 0 || j > 0) ? 1u : 0u);
      }
      if (V != 6) commit_mc(&empty[s]);
    }
    commit_mc(done);
    const bool fin = wait_b(done, 0);
    const long long c1 = clock64();
    const uint64_t g1 = gtimer();
    out[blockIdx.x] = (ok && fin) ? static_cast<unsigned long long>(c1 - c0) : 0ull;
    out[256 + blockIdx.x] = (ok && fin) ? (g1 - g0) : 0ull;
  } else if (rank == 1 && lane == 0 && warp == 1) {
    wait_b(done, 0);   // the peer leaves after the last MMA too
  } else if (kCopyWarp && rank == 0 && lane == 0 && warp == 2) {
    bool ok = true;
    for (int it = 0; it < iters && ok; ++it) {
      const int s = it % S;
      const uint32_t ph = (it / S) & 1;
      ok = wait_b(&empty[s], ph ^ 1u);     // the slot's previous MMAs are done
      if (ok && kProducer) ok = wait_b(&full[s], ph);
      if (!ok) break;
      fence_after();
      copies(kCopyKind, tb, s, sf0);
      commit_local(&sfr[s]);
    }
    commit_local(cpd);
    wait_b(cpd, 0);
  } else if (kProducer && rank == 0 && lane == 0 && warp == 0) {
    for (int it = 0; it < iters; ++it) {
      const int s = it % S;
      const uint32_t ph = (it / S) & 1;
      if (!wait_b(&empty[s], ph ^ 1u)) break;
      arrive(&full[s]);
    }
  }
  fence_before();
  __syncthreads();
  cl_sync();
  if (warp == 1) {
    fence_after();
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(tb), "r"(512) : "memory");
  }
}

template <int V>
void run(const char* name, int sms, unsigned long long* d_out, int iters) {
  const size_t smem = 200 * 1024;
  if (cudaFuncSetAttribute(kpipe<V>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess) {
    printf("%s: attr failed\n", name);
    return;
  }
  const int grid = sms & ~1;
  cudaMemset(d_out, 0, 512 * 8);
  for (int rep = 0; rep < 2; ++rep) {
    kpipe<V><<<grid, 128, smem>>>(iters, d_out);
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) { printf("%s: %s\n", name, cudaGetErrorString(e)); return; }
  }
  std::vector<unsigned long long> h(512);
  cudaMemcpy(h.data(), d_out, 512 * 8, cudaMemcpyDeviceToHost);
  std::vector<double> cyc, mhz;
  for (int i = 0; i < grid; i += 2)
    if (h[i] && h[256 + i]) { cyc.push_back((double)h[i]); mhz.push_back(1e3 * h[i] / h[256 + i]); }
  if (cyc.empty()) { printf("%s: no result\n", name); return; }
  std::sort(cyc.begin(), cyc.end());
  std::sort(mhz.begin(), mhz.end());
  const double per_stage = cyc[cyc.size() / 2] / iters;
  printf("{\"variant\": \"%s\", \"clk_per_stage\": %.0f, \"pct_of_512\": %.1f, \"sm_mhz\": %.0f, \"pairs\": %zu}\n", name,
         per_stage, 100.0 * 512 / per_stage, mhz[mhz.size() / 2], cyc.size());
}

int main() {
  int sms = 0;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0);
  unsigned long long* d_out;
  cudaMalloc(&d_out, 512 * 8);
  const int iters = 24000;   // 4000 rounds of the 6-stage ring
  run<6>("MMAs only", sms, d_out, iters);
  run<0>("MMAs + a commit per stage", sms, d_out, iters);
  run<5>("+ producer handshake (full/empty)", sms, d_out, iters);
  run<1>("+ copy warp, 6 x 32x128b.warpx4 per stage", sms, d_out, iters);
  run<2>("+ copy warp, 3 x 128x256b per stage", sms, d_out, iters);
  run<4>("copies issued by the MMA thread, 6 x warpx4", sms, d_out, iters);
  run<7>("handshake + copy warp, 6 x warpx4 (as the kernel)", sms, d_out, iters);
  run<8>("handshake + copy warp, 3 x 128x256b (as the kernel)", sms, d_out, iters);
  cudaError_t e = cudaDeviceSynchronize();
  cudaFree(d_out);
  return e == cudaSuccess ? 0 : 1;
}
