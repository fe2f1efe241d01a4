// Host <-> device transfer rates over the host link, for the host-buffer GEMM entry points:
// 268 MB in (the A and B of a bf16 8192^3 addmm) and 134 MB out (its C), between pinned host
// memory and device memory.
//
//  * copy engines: cudaMemcpyAsync, in one piece or split over 2 or 4 streams, each direction
//    alone and both at once;
//  * kernels: a grid of CTAs that loads 16-byte words from pinned host memory (through its
//    device pointer) and stores them to device memory, or the reverse, per grid size, each
//    direction alone and both at once (the two kernels on two streams).
//
// Each line of output is one case with its GB/s per direction.  Times are CUDA events around 5
// repetitions after one untimed.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>

#define CHECK(x)                                                                           \
  do {                                                                                     \
    cudaError_t e_ = (x);                                                                  \
    if (e_ != cudaSuccess) {                                                               \
      std::printf("{\"error\": \"%s at line %d\"}\n", cudaGetErrorString(e_), __LINE__);   \
      return 1;                                                                            \
    }                                                                                      \
  } while (0)

namespace {

// Copies n 16-byte words from src to dst, grid-stride, four words in flight per thread.
__global__ void __launch_bounds__(512) copy_words(const uint4* __restrict__ src,
                                                  uint4* __restrict__ dst, size_t n) {
  const size_t stride = static_cast<size_t>(gridDim.x) * blockDim.x;
  size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < n; i += 4 * stride) {
    const uint4 a = src[i], b = src[i + stride], c = src[i + 2 * stride], d = src[i + 3 * stride];
    dst[i] = a;
    dst[i + stride] = b;
    dst[i + 2 * stride] = c;
    dst[i + 3 * stride] = d;
  }
  for (; i < n; i += stride) dst[i] = src[i];
}

constexpr size_t kIn = 268ull << 20, kOut = 134ull << 20;
constexpr int kReps = 5;

}  // namespace

int main() {
  int sms = 0;
  CHECK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, 0));
  uint8_t *h_in = nullptr, *h_out = nullptr, *d_in = nullptr, *d_out = nullptr;
  CHECK(cudaMallocHost(&h_in, kIn));
  CHECK(cudaMallocHost(&h_out, kOut));
  CHECK(cudaMalloc(&d_in, kIn));
  CHECK(cudaMalloc(&d_out, kOut));
  for (size_t i = 0; i < kIn; i += 4096) h_in[i] = static_cast<uint8_t>(i >> 12);
  CHECK(cudaMemset(d_out, 1, kOut));
  uint8_t *hd_in = nullptr, *hd_out = nullptr;   // device pointers of the pinned buffers
  CHECK(cudaHostGetDevicePointer(reinterpret_cast<void**>(&hd_in), h_in, 0));
  CHECK(cudaHostGetDevicePointer(reinterpret_cast<void**>(&hd_out), h_out, 0));
  cudaStream_t st[4];
  for (auto& s : st) CHECK(cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking));
  cudaEvent_t e0, e1, f[4];
  CHECK(cudaEventCreate(&e0));
  CHECK(cudaEventCreate(&e1));
  for (auto& e : f) CHECK(cudaEventCreateWithFlags(&e, cudaEventDisableTiming));

  // Runs `issue` (which enqueues one repetition on the given streams) kReps times after one
  // warm-up; returns ms per repetition.
  auto timed = [&](auto issue, int nstreams, float* ms) -> cudaError_t {
    for (int rep = 0; rep <= kReps; ++rep) {
      cudaError_t e;
      if (rep == 1 && (e = cudaEventRecord(e0, st[0])) != cudaSuccess) return e;
      if (rep >= 1)
        for (int s = 1; s < nstreams; ++s)
          if ((e = cudaStreamWaitEvent(st[s], e0, 0)) != cudaSuccess) return e;
      if ((e = issue()) != cudaSuccess) return e;
      for (int s = 1; s < nstreams; ++s) {
        if ((e = cudaEventRecord(f[s], st[s])) != cudaSuccess) return e;
        if ((e = cudaStreamWaitEvent(st[0], f[s], 0)) != cudaSuccess) return e;
      }
      if (rep == 0 && (e = cudaStreamSynchronize(st[0])) != cudaSuccess) return e;
    }
    cudaError_t e = cudaEventRecord(e1, st[0]);
    if (e != cudaSuccess) return e;
    if ((e = cudaEventSynchronize(e1)) != cudaSuccess) return e;
    e = cudaEventElapsedTime(ms, e0, e1);
    *ms /= kReps;
    return e;
  };
  auto report = [](const char* what, int n, float ms, double in_bytes, double out_bytes) {
    std::printf("{\"case\": \"%s\", \"n\": %d, \"ms\": %.3f, \"h2d_GBs\": %.0f, \"d2h_GBs\": %.0f}\n",
                what, n, ms, in_bytes / (ms * 1e-3) / 1e9, out_bytes / (ms * 1e-3) / 1e9);
    std::fflush(stdout);
  };

  for (int ns : {1, 2, 4}) {
    for (int dir = 0; dir < 3; ++dir) {   // 0: in, 1: out, 2: both
      // both directions: each piece out goes on another stream than the piece in beside it
      const int nst = (dir == 2 && ns == 1) ? 2 : ns;
      float ms = 0;
      CHECK(timed(
          [&]() -> cudaError_t {
            for (int s = 0; s < ns; ++s) {
              cudaError_t e = cudaSuccess;
              if (dir != 1)
                e = cudaMemcpyAsync(d_in + s * (kIn / ns), h_in + s * (kIn / ns), kIn / ns,
                                    cudaMemcpyHostToDevice, st[s]);
              if (e == cudaSuccess && dir != 0)
                e = cudaMemcpyAsync(h_out + s * (kOut / ns), d_out + s * (kOut / ns), kOut / ns,
                                    cudaMemcpyDeviceToHost, dir == 2 ? st[(s + 1) % nst] : st[s]);
              if (e != cudaSuccess) return e;
            }
            return cudaSuccess;
          },
          nst, &ms));
      const char* what[3] = {"memcpy_in", "memcpy_out", "memcpy_both"};
      report(what[dir], ns, ms, dir != 1 ? kIn : 0, dir != 0 ? kOut : 0);
    }
  }
  for (int ctas : {sms / 4, sms / 2, sms, 2 * sms, 4 * sms}) {
    for (int dir = 0; dir < 3; ++dir) {
      float ms = 0;
      CHECK(timed(
          [&]() -> cudaError_t {
            if (dir != 1)
              copy_words<<<ctas, 512, 0, st[0]>>>(reinterpret_cast<const uint4*>(hd_in),
                                                  reinterpret_cast<uint4*>(d_in), kIn / 16);
            if (dir != 0)
              copy_words<<<ctas, 512, 0, dir == 2 ? st[1] : st[0]>>>(
                  reinterpret_cast<const uint4*>(d_out), reinterpret_cast<uint4*>(hd_out),
                  kOut / 16);
            return cudaGetLastError();
          },
          dir == 2 ? 2 : 1, &ms));
      const char* what[3] = {"kernel_in", "kernel_out", "kernel_both"};
      report(what[dir], ctas, ms, dir != 1 ? kIn : 0, dir != 0 ? kOut : 0);
    }
  }
  // the kernel's copy in must equal the host bytes
  CHECK(cudaDeviceSynchronize());
  uint8_t probe = 0;
  CHECK(cudaMemcpy(&probe, d_in + 4096 * 7, 1, cudaMemcpyDeviceToHost));
  if (probe != 7) {
    std::printf("{\"error\": \"copied bytes differ\"}\n");
    return 2;
  }
  return 0;
}
