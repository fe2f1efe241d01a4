// sk_gemm_bf16_static: the bf16 addmm for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc (or anything that allocates) at the point where they
// run the GEMM: code that runs under an allocator it does not own (a framework whose caching
// allocator must see every byte, a memory pool reserved up front), code on a latency-critical
// path where an allocation could synchronise the device, or code that must not fail for lack
// of memory after start-up.  The regular entry points keep their scratch (the Stream-K partial
// tiles, their flags and the error words) in a per-(device, stream) workspace that they grow
// on demand; this entry point instead takes that scratch from one fixed array compiled into
// the library, so it never allocates.
//
// Limits and behaviour:
//  * The array holds kStaticMaxGrid partial slots of 128 x 128 fp32 (10 MiB plus flags); every
//    GPU that loads the library keeps it until the process exits.  The entry point always uses
//    128 x 128 CTA tiles and returns SK_ERR_UNSUPPORTED when a schedule would need more than
//    kStaticMaxGrid Stream-K slots.
//  * On its first call on a device it looks up the array's device address (once per device,
//    with that device current) and raises the kernel's shared-memory limit; make that first
//    call before any stream capture on that device.  That set-up is kept for the life of the
//    process: after a cudaDeviceReset the cached address and limit are stale, so this entry
//    point must not be used on a device that has been reset.
//  * Every call on every stream shares the one array, which keeps what the last call left.
//    Each call clears the error words and the flags (which must start at zero) on its stream
//    before the GEMM.  Calls that overlap on the GPU (other streams, other host threads) race
//    on the array and give wrong results: serialise them.
//  * A kernel-side timeout is recorded in the array's error words, which each call clears
//    first; sk_stream_status (which reads the regular workspaces) does not see it, and
//    sk_gemm_bf16_static_status reads it back.  The owner concerned leaves its tile unwritten.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <mutex>

#include "sk_gemm.h"
#include "sk_launch.h"

namespace {

constexpr int kStaticMaxGrid = 160;
constexpr size_t kStaticTile = 128;
constexpr size_t kErrBytes = 256;                                  // 4 error words, padded
constexpr size_t kFlagBytes = 1024;                                // kStaticMaxGrid flags, padded
constexpr size_t kSlotBytes = 128 * kStaticTile * sizeof(float);  // one partial tile
constexpr size_t kScratchBytes = kErrBytes + kFlagBytes + kStaticMaxGrid * kSlotBytes;
static_assert(kStaticMaxGrid * sizeof(uint32_t) <= kFlagBytes, "flag area");

// The scratch.  In host code this name only stands for the array: its device address comes
// from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

struct StaticDevice {
  bool ready = false;
  unsigned char* base = nullptr;   // device address of g_static_scratch on this device
  int sm_count = 0;
  int ctas_per_sm = 0;
};

constexpr int kMaxDevices = 64;
std::mutex g_static_mutex;
StaticDevice g_static_devices[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool encode_bf16_2d(CUtensorMap* map, const void* base, int64_t rows, int64_t cols,
                    uint32_t box_cols, uint32_t box_rows) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One-time set-up for the current device: the array's device address, the SM count and the
// kernel's shared-memory limit.  Caller holds g_static_mutex.
sk_status_t static_device(int dev, StaticDevice** out) {
  if (dev < 0 || dev >= kMaxDevices) return SK_ERR_UNSUPPORTED;
  StaticDevice& d = g_static_devices[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return SK_ERR_CUDA;
    if (major != 10 || minor != 3) return SK_ERR_UNSUPPORTED;
    void* base = nullptr;
    if (cudaGetSymbolAddress(&base, g_static_scratch) != cudaSuccess || base == nullptr)
      return SK_ERR_CUDA;
    // the 128 x 128 kernel, and its tall-stage form for problems of at most 64 rows (both one
    // CTA per SM)
    int tall_ctas = 0;
    if (sk::variant_setup(sk::kVariantBf16N128, &d.ctas_per_sm) != cudaSuccess ||
        sk::variant_setup(sk::variant_of(sk::kKindBf16N128Tall, 0), &tall_ctas) != cudaSuccess)
      return SK_ERR_CUDA;
    d.ctas_per_sm = std::min(d.ctas_per_sm, tall_ctas);
    d.base = static_cast<unsigned char*>(base);
    d.ready = true;
  }
  *out = &d;
  return SK_OK;
}

}  // namespace

extern "C" sk_status_t sk_gemm_bf16_static(const void* A, const void* B, const void* bias,
                                           void* C, sk_dtype_t out_dtype, int64_t M, int64_t N,
                                           int64_t K, int num_sms, sk_mode_t mode,
                                           void* stream_ptr) {
  // Argument checks (the same rules as sk_gemm_bf16), before any CUDA call.
  const auto misaligned = [](const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) != 0; };
  if (A == nullptr || B == nullptr || C == nullptr) return SK_ERR_INVALID_ARG;
  if (misaligned(A) || misaligned(B) || misaligned(C) || (bias != nullptr && misaligned(bias)))
    return SK_ERR_INVALID_ARG;
  if (out_dtype != SK_F32 && out_dtype != SK_BF16) return SK_ERR_INVALID_ARG;
  if (mode < SK_MODE_DP || mode > SK_MODE_AUTO) return SK_ERR_INVALID_ARG;
  const int64_t max_dim = (int64_t(1) << 31) - 1;
  if (M < 1 || N < 1 || K < 1 || M > max_dim || N > max_dim || K > max_dim)
    return SK_ERR_INVALID_ARG;
  if (K % 8 != 0 || N % 8 != 0) return SK_ERR_INVALID_ARG;

  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SK_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_static_mutex);
  StaticDevice* d = nullptr;
  sk_status_t st = static_device(dev, &d);
  if (st != SK_OK) return st;

  sk_options_t opt = {};
  opt.tile_m = static_cast<int32_t>(kStaticTile);   // SK_MODE_AUTO then picks the schedule only
  opt.tile_n = static_cast<int32_t>(kStaticTile);
  opt.drop_release_cta = -1;
  sk_plan_t plan;
  st = sk_plan(0, M, N, K, num_sms, mode, d->sm_count, &opt, &plan);
  if (st != SK_OK) return st;
  const bool streamk = plan.sk_tiles > 0;
  if (streamk && plan.grid > kStaticMaxGrid) return SK_ERR_UNSUPPORTED;   // beyond the array
  if (streamk && static_cast<int64_t>(plan.grid) > static_cast<int64_t>(d->ctas_per_sm) * d->sm_count)
    return SK_ERR_NOT_CORESIDENT;

  // The error words and the flags must start at zero; the partial slots need no clearing.
  if (cudaMemsetAsync(d->base, 0, kErrBytes + kFlagBytes, stream) != cudaSuccess) return SK_ERR_CUDA;

  // The planner gives problems of at most 64 rows tall stages (128 K: A boxes of 64 rows, B
  // boxes of 128 k-rows).
  const bool tall = plan.tile_k == 128;
  CUtensorMap tmA, tmB;
  if (!encode_bf16_2d(&tmA, A, M, K, 64, tall ? 64 : 128) ||
      !encode_bf16_2d(&tmB, B, K, N, 64, tall ? 128 : 64))
    return SK_ERR_CUDA;

  sk::Launch l = {};
  l.tmA = &tmA;
  l.tmB = &tmB;
  l.grid = plan.grid;
  l.cooperative = streamk;
  l.stream = stream;
  sk::Args& a = l.args;
  a.bias = bias;
  a.C = C;
  a.M = M;
  a.N = N;
  a.K = K;
  a.out_bf16 = out_dtype == SK_BF16 ? 1 : 0;
  a.inject_drop = 0;
  a.drop_cta = -1;
  a.epoch = 1;   // flags were just cleared, so a fixed value identifies this call's releases
  a.plan.tiles_m = plan.tiles_m;
  a.plan.tiles_n = plan.tiles_n;
  a.plan.iters = plan.iters;
  a.plan.grid = plan.grid;
  a.plan.group_m = plan.raster_group;
  a.plan.tiles = plan.tiles;
  a.plan.whole_tiles = plan.whole_tiles;
  a.plan.sk_base = plan.sk_base;
  a.plan.sk_extra = plan.sk_extra;
  a.err = reinterpret_cast<uint32_t*>(d->base);
  a.flags = reinterpret_cast<uint32_t*>(d->base + kErrBytes);
  a.P = reinterpret_cast<float*>(d->base + kErrBytes + kFlagBytes);
  a.timeout_ns = 2000000000ull;
  const cudaError_t e =
      sk::variant_launch(tall ? sk::variant_of(sk::kKindBf16N128Tall, 0) : sk::kVariantBf16N128, l);
  if (e == cudaErrorCooperativeLaunchTooLarge) return SK_ERR_NOT_CORESIDENT;
  return e == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}

extern "C" sk_status_t sk_gemm_bf16_static_status(void* stream_ptr) {
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SK_ERR_UNSUPPORTED;
  unsigned char* base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (dev < 0 || dev >= kMaxDevices) return SK_ERR_UNSUPPORTED;
    if (!g_static_devices[dev].ready) return SK_OK;   // no call has run on this device
    base = g_static_devices[dev].base;
  }
  // Ordered after the calls queued on `stream`; the words land in a host variable (no
  // allocation).
  uint32_t words[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(words, base, sizeof(words), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return SK_ERR_CUDA;
  return words[0] == 0 ? SK_OK : static_cast<sk_status_t>(words[0]);
}
