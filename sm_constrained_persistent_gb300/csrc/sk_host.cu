// Host-buffer entry points: the same addmm with A, B, bias and C in host memory.  The library
// copies the operands in, runs the GEMM and copies C out, overlapping the three: B (and the
// bias) goes first, then A in row blocks; the GEMM of a block starts once its rows have
// arrived, and its rows of C leave while later blocks are still computing.  Declared in
// include/sk_gemm.h.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <map>
#include <mutex>
#include <utility>

#include "sk_gemm.h"
#include "sk_launch.h"

namespace {

constexpr int kMaxBlocks = 8;           // row blocks per call
constexpr int64_t kMinBlockRows = 256;  // a block keeps at least one row of pair tiles

// Device copies of one call's operands, plus the copy streams and events, per (device, stream).
struct Stage {
  void* A = nullptr;
  size_t A_bytes = 0;
  void* B = nullptr;
  size_t B_bytes = 0;
  void* bias = nullptr;
  size_t bias_bytes = 0;
  void* C = nullptr;
  size_t C_bytes = 0;
  void* A_scale = nullptr;
  size_t A_scale_bytes = 0;
  void* B_scale = nullptr;
  size_t B_scale_bytes = 0;
  cudaStream_t h2d = nullptr;
  cudaStream_t d2h = nullptr;
  cudaEvent_t start = nullptr;
  cudaEvent_t b_ready = nullptr;
  cudaEvent_t a_ready[kMaxBlocks] = {};
  cudaEvent_t c_ready[kMaxBlocks] = {};
  cudaEvent_t done = nullptr;
};

std::mutex g_host_mutex;
std::map<std::pair<int, cudaStream_t>, Stage> g_stages;

bool grow(void** ptr, size_t* have, size_t need, cudaStream_t st) {
  if (need == 0 || (*have >= need && *ptr != nullptr)) return true;
  if (*ptr != nullptr) {
    if (cudaFreeAsync(*ptr, st) != cudaSuccess) return false;
    *ptr = nullptr;
    *have = 0;
  }
  if (cudaMallocAsync(ptr, need, st) != cudaSuccess) {
    cudaGetLastError();   // an allocation failure must not surface as a later call's launch error
    *ptr = nullptr;
    return false;
  }
  *have = need;
  return true;
}

bool make_stream_objects(Stage& s) {
  if (s.h2d != nullptr) return true;
  if (cudaStreamCreateWithFlags(&s.h2d, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&s.d2h, cudaStreamNonBlocking) != cudaSuccess)
    return false;
  cudaEvent_t* all[] = {&s.start, &s.b_ready, &s.done};
  for (cudaEvent_t* e : all)
    if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return false;
  for (int i = 0; i < kMaxBlocks; ++i)
    if (cudaEventCreateWithFlags(&s.a_ready[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.c_ready[i], cudaEventDisableTiming) != cudaSuccess)
      return false;
  return true;
}

struct HostProblem {
  int format;                  // 0 bf16, 1 MXFP4, 2 fp8
  const void* A;
  const void* A_scale;
  const void* B;
  const void* B_scale;
  const void* bias;
  void* C;
  sk_dtype_t out_dtype;
  int64_t M, N, K;
  int num_sms;
  sk_mode_t mode;
  const sk_options_t* options;
};

// Bytes of one row of A (and of its scales), of B, and of C.
size_t a_row_bytes(const HostProblem& p) {
  return p.format == 0 ? p.K * 2 : (p.format == 1 ? p.K / 2 : p.K);
}
size_t b_bytes(const HostProblem& p) {
  return p.format == 0 ? p.K * p.N * 2 : (p.format == 1 ? p.N * (p.K / 2) : p.K * p.N);
}
size_t c_elem(const HostProblem& p) { return p.out_dtype == SK_BF16 ? 2 : 4; }

sk_status_t gemm_block(const HostProblem& p, const Stage& s, int64_t m0, int64_t rows,
                       cudaStream_t st) {
  const uint8_t* A = static_cast<const uint8_t*>(s.A) + m0 * a_row_bytes(p);
  uint8_t* C = static_cast<uint8_t*>(s.C) + m0 * p.N * c_elem(p);
  const void* bias = p.bias != nullptr ? s.bias : nullptr;
  switch (p.format) {
    case 0:
      return sk_gemm_bf16_ex(A, s.B, bias, C, p.out_dtype, rows, p.N, p.K, p.num_sms, p.mode,
                             p.options, st);
    case 2:
      return sk_gemm_fp8_ex(A, s.B, bias, C, p.out_dtype, rows, p.N, p.K, p.num_sms, p.mode,
                            p.options, st);
    default: {
      const uint8_t* As = static_cast<const uint8_t*>(s.A_scale) + m0 * (p.K / 32);
      return sk_gemm_mxfp4_ex(A, As, s.B, s.B_scale, bias, C, p.out_dtype, rows, p.N, p.K,
                              p.num_sms, p.mode, p.options, st);
    }
  }
}

sk_status_t run_host(const HostProblem& p, void* stream) {
  if (p.A == nullptr || p.B == nullptr || p.C == nullptr) return SK_ERR_INVALID_ARG;
  if (p.format == 1 && (p.A_scale == nullptr || p.B_scale == nullptr)) return SK_ERR_INVALID_ARG;
  if (p.M < 1 || p.N < 1 || p.K < 1 || (p.format == 1 && p.K % 32 != 0))
    return SK_ERR_INVALID_ARG;
  if (p.out_dtype != SK_F32 && p.out_dtype != SK_BF16) return SK_ERR_INVALID_ARG;
  // The same shape rules as the device-buffer calls, checked before anything is copied.
  const int64_t row_align = p.format == 0 ? 8 : (p.format == 2 ? 16 : 32);
  if (p.K % row_align != 0 || (p.format != 1 && p.N % row_align != 0)) return SK_ERR_INVALID_ARG;
  int dev = 0, sm_count = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SK_ERR_UNSUPPORTED;
  sk_plan_t plan;
  const sk_status_t planned =
      sk_plan(p.format, p.M, p.N, p.K, p.num_sms, p.mode, sm_count, p.options, &plan);
  if (planned != SK_OK) return planned;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return SK_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return SK_ERR_UNSUPPORTED;

  // Row blocks: at most kMaxBlocks, each a multiple of 256 rows (the last one ragged).
  int64_t block_rows = std::max<int64_t>(kMinBlockRows, (p.M + kMaxBlocks - 1) / kMaxBlocks);
  block_rows = (block_rows + kMinBlockRows - 1) / kMinBlockRows * kMinBlockRows;
  const int blocks = static_cast<int>((p.M + block_rows - 1) / block_rows);

  std::lock_guard<std::mutex> lock(g_host_mutex);
  Stage& s = g_stages[{dev, st}];
  if (!make_stream_objects(s)) return SK_ERR_CUDA;
  const size_t bias_bytes = p.bias != nullptr ? p.N * c_elem(p) : 0;
  const size_t a_scale_bytes = p.format == 1 ? p.M * (p.K / 32) : 0;
  const size_t b_scale_bytes = p.format == 1 ? p.N * (p.K / 32) : 0;
  // Grown on the caller's stream, so a buffer still used by an earlier call is freed only
  // after that call's work on this stream.
  if (!grow(&s.A, &s.A_bytes, p.M * a_row_bytes(p), st) ||
      !grow(&s.B, &s.B_bytes, b_bytes(p), st) || !grow(&s.bias, &s.bias_bytes, bias_bytes, st) ||
      !grow(&s.C, &s.C_bytes, p.M * p.N * c_elem(p), st) ||
      !grow(&s.A_scale, &s.A_scale_bytes, a_scale_bytes, st) ||
      !grow(&s.B_scale, &s.B_scale_bytes, b_scale_bytes, st))
    return SK_ERR_OOM;

  // Everything earlier on the caller's stream (including the previous call's copies out and
  // any buffer growth) happens before this call's copies in.
  if (cudaEventRecord(s.start, st) != cudaSuccess ||
      cudaStreamWaitEvent(s.h2d, s.start, 0) != cudaSuccess ||
      cudaStreamWaitEvent(s.d2h, s.start, 0) != cudaSuccess)
    return SK_ERR_CUDA;
  const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
  if (cudaMemcpyAsync(s.B, p.B, b_bytes(p), h2d, s.h2d) != cudaSuccess) return SK_ERR_CUDA;
  if (bias_bytes && cudaMemcpyAsync(s.bias, p.bias, bias_bytes, h2d, s.h2d) != cudaSuccess)
    return SK_ERR_CUDA;
  if (b_scale_bytes &&
      cudaMemcpyAsync(s.B_scale, p.B_scale, b_scale_bytes, h2d, s.h2d) != cudaSuccess)
    return SK_ERR_CUDA;
  if (cudaEventRecord(s.b_ready, s.h2d) != cudaSuccess) return SK_ERR_CUDA;
  for (int i = 0; i < blocks; ++i) {
    const int64_t m0 = i * block_rows, rows = std::min(block_rows, p.M - m0);
    const size_t ra = a_row_bytes(p);
    if (cudaMemcpyAsync(static_cast<uint8_t*>(s.A) + m0 * ra,
                        static_cast<const uint8_t*>(p.A) + m0 * ra, rows * ra, h2d,
                        s.h2d) != cudaSuccess)
      return SK_ERR_CUDA;
    if (a_scale_bytes) {
      const size_t rs = p.K / 32;
      if (cudaMemcpyAsync(static_cast<uint8_t*>(s.A_scale) + m0 * rs,
                          static_cast<const uint8_t*>(p.A_scale) + m0 * rs, rows * rs, h2d,
                          s.h2d) != cudaSuccess)
        return SK_ERR_CUDA;
    }
    if (cudaEventRecord(s.a_ready[i], s.h2d) != cudaSuccess) return SK_ERR_CUDA;
  }

  // GEMMs on the caller's stream, one per row block; copies out on their own stream.
  sk_status_t status = SK_OK;
  if (cudaStreamWaitEvent(st, s.b_ready, 0) != cudaSuccess) return SK_ERR_CUDA;
  for (int i = 0; i < blocks; ++i) {
    const int64_t m0 = i * block_rows, rows = std::min(block_rows, p.M - m0);
    if (cudaStreamWaitEvent(st, s.a_ready[i], 0) != cudaSuccess) return SK_ERR_CUDA;
    if (status == SK_OK) status = gemm_block(p, s, m0, rows, st);
    if (cudaEventRecord(s.c_ready[i], st) != cudaSuccess) return SK_ERR_CUDA;
    if (cudaStreamWaitEvent(s.d2h, s.c_ready[i], 0) != cudaSuccess) return SK_ERR_CUDA;
    if (status == SK_OK) {
      const size_t rc = p.N * c_elem(p);
      if (cudaMemcpyAsync(static_cast<uint8_t*>(p.C) + m0 * rc,
                          static_cast<const uint8_t*>(s.C) + m0 * rc, rows * rc, d2h,
                          s.d2h) != cudaSuccess)
        return SK_ERR_CUDA;
    }
  }
  // The caller's stream resumes once C is back in host memory.
  if (cudaEventRecord(s.done, s.d2h) != cudaSuccess ||
      cudaStreamWaitEvent(st, s.done, 0) != cudaSuccess)
    return SK_ERR_CUDA;
  return status;
}

}  // namespace

namespace sk {

int64_t host_stage_bytes(int device, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_host_mutex);
  const auto it = g_stages.find({device, stream});
  if (it == g_stages.end()) return 0;
  const Stage& s = it->second;
  return static_cast<int64_t>(s.A_bytes + s.B_bytes + s.bias_bytes + s.C_bytes +
                              s.A_scale_bytes + s.B_scale_bytes);
}

cudaError_t release_host_stage(int device, cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_host_mutex);
  const auto it = g_stages.find({device, stream});
  if (it == g_stages.end()) return cudaSuccess;
  Stage& s = it->second;
  cudaError_t result = cudaSuccess;
  // The buffers were grown on `stream`, and every later use of them (the copies on the two copy
  // streams included) is ordered before the caller's stream resumes, so a free queued on
  // `stream` runs after all of them.  Streams and events with work pending are destroyed once
  // that work completes.
  void* bufs[] = {s.A, s.B, s.bias, s.C, s.A_scale, s.B_scale};
  for (void* b : bufs)
    if (b != nullptr && cudaFreeAsync(b, stream) != cudaSuccess) result = cudaErrorUnknown;
  if (s.h2d != nullptr) {
    cudaStreamDestroy(s.h2d);
    cudaStreamDestroy(s.d2h);
    cudaEventDestroy(s.start);
    cudaEventDestroy(s.b_ready);
    cudaEventDestroy(s.done);
    for (int i = 0; i < kMaxBlocks; ++i) {
      cudaEventDestroy(s.a_ready[i]);
      cudaEventDestroy(s.c_ready[i]);
    }
  }
  g_stages.erase(it);
  return result;
}

void release_host_stages() {
  std::lock_guard<std::mutex> lock(g_host_mutex);
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return;
  for (auto& kv : g_stages) {
    if (cudaSetDevice(kv.first.first) != cudaSuccess) continue;
    cudaDeviceSynchronize();
    Stage& s = kv.second;
    void* bufs[] = {s.A, s.B, s.bias, s.C, s.A_scale, s.B_scale};
    for (void* b : bufs)
      if (b != nullptr) cudaFree(b);
    if (s.h2d != nullptr) {
      cudaStreamDestroy(s.h2d);
      cudaStreamDestroy(s.d2h);
      cudaEventDestroy(s.start);
      cudaEventDestroy(s.b_ready);
      cudaEventDestroy(s.done);
      for (int i = 0; i < kMaxBlocks; ++i) {
        cudaEventDestroy(s.a_ready[i]);
        cudaEventDestroy(s.c_ready[i]);
      }
    }
  }
  g_stages.clear();
  cudaSetDevice(prev);
}

}  // namespace sk

extern "C" {

sk_status_t sk_gemm_bf16_host(const void* A, const void* B, const void* bias, void* C,
                              sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                              sk_mode_t mode, const sk_options_t* options, void* stream) {
  const sk::NvtxRange range("sk_gemm_bf16_host");
  const HostProblem p = {0, A, nullptr, B, nullptr, bias, C, out_dtype, M, N, K, num_sms, mode,
                         options};
  return run_host(p, stream);
}

sk_status_t sk_gemm_fp8_host(const void* A, const void* B, const void* bias, void* C,
                             sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                             sk_mode_t mode, const sk_options_t* options, void* stream) {
  const sk::NvtxRange range("sk_gemm_fp8_host");
  const HostProblem p = {2, A, nullptr, B, nullptr, bias, C, out_dtype, M, N, K, num_sms, mode,
                         options};
  return run_host(p, stream);
}

sk_status_t sk_gemm_mxfp4_host(const void* A, const void* A_scale, const void* B,
                               const void* B_scale, const void* bias, void* C,
                               sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K,
                               int num_sms, sk_mode_t mode, const sk_options_t* options,
                               void* stream) {
  const sk::NvtxRange range("sk_gemm_mxfp4_host");
  const HostProblem p = {1, A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms, mode,
                         options};
  return run_host(p, stream);
}

}  // extern "C"
