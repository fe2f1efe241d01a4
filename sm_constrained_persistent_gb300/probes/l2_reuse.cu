// How much of a working set the L2 keeps between two reads of it, and whether data read by the SMs
// of one half of the GPU is found in L2 by the SMs of the other half.
//
// For each size S: L2 is scrubbed (a 512 MB write, then a 512 MB read of another buffer), a first
// pass reads the S-byte buffer once, then a second pass reads it again and is timed.  A pass is run
// by the CTAs that land on a chosen set of SMs (by %smid: the lower half, the upper half, or all),
// which take 64 KB chunks from a shared counter until the buffer is covered, so every byte is read
// once per pass whatever the CTAs' placement.  Loads bypass L1 (ld.global.cg).  The second pass's
// rate tells where it read from: at the copy bandwidth (~6.7 TB/s) from DRAM, well above it from L2.
//   same:  both passes on the lower half of the SMs;
//   cross: the first pass on the lower half, the second on the upper half;
//   all:   both passes on every SM.
// Each line of output is one (pattern, S): the second pass's time and rate, from the first
// participating CTA's start to the last one's end (%globaltimer; the events around a launch add
// ~4.5 us and tick in ~2 us steps).
//
// Nothing waits on anything: every CTA reads chunks until the counter passes the end, then exits.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdio>
#include <vector>

#define CHECK(x)                                                                         \
  do {                                                                                   \
    cudaError_t e_ = (x);                                                                \
    if (e_ != cudaSuccess) {                                                             \
      std::printf("{\"error\": \"%s at line %d\"}\n", cudaGetErrorString(e_), __LINE__); \
      return 1;                                                                          \
    }                                                                                    \
  } while (0)

namespace {

constexpr size_t kChunk = 64 << 10;   // bytes per work item
constexpr int kThreads = 256;

__device__ __forceinline__ uint32_t smid() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}

__device__ __forceinline__ unsigned long long now_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint4 ld_cg(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// sm_lo <= smid < sm_hi take part; the others exit at once.
__global__ void __launch_bounds__(kThreads) read_pass(const uint4* buf, uint32_t n_chunks,
                                                      uint32_t sm_lo, uint32_t sm_hi,
                                                      uint32_t* counter, uint32_t* sink,
                                                      unsigned long long* span) {
  const uint32_t s = smid();
  if (s < sm_lo || s >= sm_hi) return;
  if (threadIdx.x == 0) atomicMin(&span[0], now_ns());
  __shared__ uint32_t chunk;
  uint32_t acc = 0;
  while (true) {
    if (threadIdx.x == 0) chunk = atomicAdd(counter, 1u);
    __syncthreads();
    const uint32_t c = chunk;
    __syncthreads();
    if (c >= n_chunks) break;
    const uint4* p = buf + static_cast<size_t>(c) * (kChunk / 16);
#pragma unroll 4
    for (uint32_t i = threadIdx.x; i < kChunk / 16; i += kThreads) {
      const uint4 v = ld_cg(p + i);
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
  }
  if (acc == 0x9E3779B9u) *sink = acc;   // keeps the loads; the buffers never hold this
  __syncthreads();
  if (threadIdx.x == 0) atomicMax(&span[1], now_ns());
}

__global__ void scrub_read(const uint4* p, size_t n, uint32_t* sink) {
  uint32_t acc = 0;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    acc ^= ld_cg(p + i).x;
  if (acc == 0x9E3779B9u) *sink = acc;
}

}  // namespace

int main() {
  int sms = 0;
  CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  const size_t max_bytes = 192ull << 20, scrub_bytes = 512ull << 20;
  void *buf = nullptr, *scrub = nullptr;
  uint32_t* ctl = nullptr;   // [0] counter, [1] sink
  unsigned long long* span = nullptr;   // [0] first start, [1] last end (ns)
  CHECK(cudaMalloc(&span, 2 * sizeof(unsigned long long)));
  CHECK(cudaMalloc(&buf, max_bytes));
  CHECK(cudaMalloc(&scrub, scrub_bytes));
  CHECK(cudaMalloc(&ctl, 8));
  CHECK(cudaMemset(buf, 1, max_bytes));
  CHECK(cudaMemset(ctl, 0, 8));
  cudaEvent_t e0, e1;
  CHECK(cudaEventCreate(&e0));
  CHECK(cudaEventCreate(&e1));
  const uint32_t half = static_cast<uint32_t>(sms) / 2;
  struct Pattern {
    const char* name;
    uint32_t lo1, hi1, lo2, hi2;
  };
  const Pattern pats[] = {{"same", 0, half, 0, half},
                          {"cross", 0, half, half, static_cast<uint32_t>(sms)},
                          {"all", 0, static_cast<uint32_t>(sms), 0, static_cast<uint32_t>(sms)}};
  const int grid = 8 * sms;   // enough CTAs that every SM of either half gets several
  for (const Pattern& pat : pats) {
    for (size_t mb = 16; mb <= 192; mb += 16) {
      const size_t bytes = mb << 20;
      const uint32_t n_chunks = static_cast<uint32_t>(bytes / kChunk);
      std::vector<float> ts;
      for (int rep = 0; rep < 5; ++rep) {
        CHECK(cudaMemsetAsync(scrub, rep, scrub_bytes));
        scrub_read<<<4 * sms, 512>>>(static_cast<const uint4*>(scrub), scrub_bytes / 16, ctl + 1);
        CHECK(cudaMemsetAsync(ctl, 0, 4));
        read_pass<<<grid, kThreads>>>(static_cast<const uint4*>(buf), n_chunks, pat.lo1, pat.hi1, ctl,
                                      ctl + 1, span);
        CHECK(cudaMemsetAsync(ctl, 0, 4));
        const unsigned long long init[2] = {~0ull, 0ull};
        CHECK(cudaMemcpyAsync(span, init, sizeof(init), cudaMemcpyHostToDevice));
        CHECK(cudaEventRecord(e0));
        read_pass<<<grid, kThreads>>>(static_cast<const uint4*>(buf), n_chunks, pat.lo2, pat.hi2, ctl,
                                      ctl + 1, span);
        CHECK(cudaEventRecord(e1));
        CHECK(cudaEventSynchronize(e1));
        unsigned long long h[2];
        CHECK(cudaMemcpy(h, span, sizeof(h), cudaMemcpyDeviceToHost));
        ts.push_back(static_cast<float>(h[1] - h[0]) * 1e-6f);   // ms
      }
      std::sort(ts.begin(), ts.end());
      const float ms = ts[ts.size() / 2];
      std::printf("{\"pattern\": \"%s\", \"MB\": %zu, \"second_pass_in_kernel_us\": %.2f, \"GBs\": %.0f}\n",
                  pat.name, mb, ms * 1000.0f, static_cast<double>(bytes) / (ms * 1e-3) / 1e9);
      std::fflush(stdout);
    }
  }
  return 0;
}
