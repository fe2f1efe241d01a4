// The addmm GEMM kernel for sm_103a: C = A * B (+ bias[n]), fp32 accumulation in tensor
// memory, for bf16 operands (tcgen05 kind::f16), fp8 E4M3 operands (kind::f8f6f4) and MXFP4
// operands (kind::mxf4 with E8M0 block scales), under the data-parallel, SM-constrained
// persistent, Stream-K and hybrid schedules of sk_schedule.cuh.
//
// One CTA of 192 threads per SM, warp-specialised:
//   warp 0      TMA producer: streams the A and B tiles of every k-iteration (and the MXFP4
//               scale blocks) into a ring of shared-memory stages, each guarded by a "full"
//               mbarrier (transaction bytes) and an "empty" mbarrier (released by the MMAs).
//   warp 1      allocates tensor memory, then one lane issues the tcgen05 MMAs of each piece
//               into one of two fp32 accumulators (128 lanes x BN columns each), so the
//               epilogue of one tile overlaps the main loop of the next.
//   warps 2..5  epilogue, thread = tile row: tensor memory -> registers, then by role
//                 whole tile / owner:  (+ partials of the contributors) + bias[n] -> cast ->
//                                      store C (TMA stores from shared memory where C's
//                                      rows are 16-byte aligned);
//                 contribution:        fp32 partial -> this CTA's scratch slot P[cta] with
//                                      coalesced 16-byte stores, then a release of
//                                      flags[cta].
// The bias is added only where a tile is finished (whole tile or owner, after all partials),
// never by a contributor (tritonBLAS PR #67 "Fix StreamK Kernel Bias", Motivation).
//
// Every wait is bounded (global timer); when one runs out the kernel records SK_ERR_TIMEOUT
// in the workspace error words, skips the stores that depend on it, waits (bounded) for its
// own copies and MMAs in flight, frees its tensor memory and returns.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sk_kernel_args.h"
#include "sk_ptx.cuh"
#include "sk_schedule.cuh"

namespace sk {

constexpr int kBM = 128;          // rows per CTA tile (tcgen05 M = 128, one row per TMEM lane)
constexpr int kThreads = 192;
constexpr int kEpilogueThreads = 128;
constexpr uint32_t kErrTimeout = 5;   // numeric value of SK_ERR_TIMEOUT

// outcome of one piece, as decided by the epilogue's first thread
enum : uint32_t { kUnitStore = 0, kUnitSkip = 1, kUnitAbort = 2 };

// where a wait ran out (second error word)
enum : uint32_t {
  kSiteFlag = 1,
  kSiteProducer = 2,
  kSiteMma = 3,
  kSiteEpilogue = 4,
  kSiteDrain = 5
};



// kAT: A is stored transposed (K x M row-major) and read M-major; kBT: B is stored transposed
// (N x K row-major) and read K-major.  kF8: 1-byte E4M3 operands instead of bf16 (same layouts).
// kTall: bf16 with at most 64 rows of A (one row of tiles streaming B): 128 K per stage, so
// that every B box is 128 k-rows tall, and only A's 64 real rows are loaded.  Streamed alone
// through TMA, a 4096 x 14336 bf16 B is read at 5.4 TB/s in 64 x 128 boxes against 4.0 TB/s
// in 64 x 64 ones; inside the GEMM, whose stages wait for their MMAs before they refill, the
// gain shrinks to 0-4 %.
template <bool kMx, int kBN, bool kAT = false, bool kBT = false, bool kF8 = false,
          bool kTall = false>
struct Cfg {
  static_assert(kBN == 96 || kBN == 128 || kBN == 256, "tile width");
  static_assert(kBN != 96 || (!kMx && !kF8 && !kAT && !kBT), "96-wide tiles: bf16, plain layouts");
  static_assert(!kMx || (!kAT && !kBT && !kF8), "MXFP4 operands are K-major");
  static_assert(!kMx || kBN == 128, "MXFP4 tiles are 128 wide");
  static_assert(!kTall || (!kMx && !kF8 && !kAT && !kBT && kBN != 256),
                "tall stages: bf16, plain layouts, 96- or 128-wide tiles");
  // One k-iteration is one 128-byte swizzle row of K: 64 bf16, 128 fp8 or 256 fp4 elements
  // (two rows, 128 bf16, for tall stages).
  static constexpr int kKHalves = kTall ? 2 : 1;   // 128-byte K atoms of A per stage
  static constexpr int kTileK = kMx ? 256 : (kF8 ? 128 : 64 * kKHalves);
  static constexpr int kMmaK = kMx ? 64 : (kF8 ? 32 : 16);   // K per tcgen05.mma (32 bytes)
  static constexpr int kMmasPerStage = kTileK / kMmaK;        // 4 (8 for tall stages)
  // Rows of A a stage holds per K atom.  Tall stages load only 64: the M = 128 MMA then reads
  // its rows 64-127 from the next 8 KB of the ring (still inside shared memory), and those
  // accumulator rows lie at m >= M, which is never stored.
  static constexpr int kARows = kTall ? 64 : kBM;
  // MMA rows: tall stages run M = 64 MMAs over exactly those rows (half the tensor-pipe time of
  // M = 128 ones, which matters where few SMs stream B).  An M = 64 accumulator holds row r in
  // tensor-memory lane 32 * (r / 16) + r % 16: the first 16 lanes of each warp's quarter.
  static constexpr int kMmaM = kTall ? 64 : kBM;
  // MN-major tiles are blocks of 128 bytes (kAtom elements) x kTileK k-rows, kBoxBytes each;
  // one MMA's K advances kMnAdvance bytes through a block.
  static constexpr int kAtom = kF8 ? 128 : 64;
  static constexpr int kBoxBytes = kTileK * 128;
  static constexpr int kMnAdvance = kMmaK * 128;
  // B (MN-major) is read in blocks of kAtomB columns with kRowB-byte rows: the 128-byte
  // blocks above, or for 96-wide tiles three blocks of 32 bf16 (64-byte rows, 64-byte swizzle).
  static constexpr int kAtomB = kBN == 96 ? 32 : kAtom;
  static constexpr int kRowB = kBN == 96 ? 64 : 128;
  static constexpr int kBoxBytesB = kTileK * kRowB;
  static constexpr uint32_t kLayoutB = kBN == 96 ? kLayoutSwizzle64B : kLayoutSwizzle128B;
  static constexpr int kStageA = kARows * 128 * kKHalves;
  static constexpr int kStageB = kBN * 128 * kKHalves;
  static constexpr int kStageSfa = kMx ? 1024 : 0;               // 2 k groups x 512 B
  static constexpr int kStageSfb = kMx ? (kBN / 128) * 1024 : 0;
  // 96-wide tiles stream B for one row of tiles: a deeper ring keeps more of it in flight.
  static constexpr int kStages = ((kBN == 96 ? 200 : 192) * 1024) / (kStageA + kStageB);
  static constexpr int kStageBytes = kStageA + kStageB + kStageSfa + kStageSfb;
  static constexpr uint32_t kAccCols = kBN == 96 ? 128 : kBN;   // tensor-memory columns per accumulator
  static constexpr uint32_t kSfaCols = 8;              // per stage: 2 groups x 4 columns
  static constexpr uint32_t kSfbCols = 2 * (kBN / 32); // per stage: 2 groups x BN/32 columns
  static constexpr uint32_t kTmemCols = 512;
  static_assert(2 * kAccCols + (kMx ? kStages * (kSfaCols + kSfbCols) : 0) <= kTmemCols,
                "tensor memory budget");
  static constexpr int kBarrierBytes = 256;
  static_assert((2 * kStages + 5) * 8 + 24 <= kBarrierBytes, "barrier area");
  // C leaves through TMA stores when its rows are 16-byte aligned: each epilogue warp stages
  // 32 rows x 64 bytes in one of its two 2 KB buffers.
  static constexpr int kEpiBytes = 4 * 2 * 2048;
  static constexpr size_t kSmemBytes =
      1024 + static_cast<size_t>(kStages) * kStageBytes + kEpiBytes + kBarrierBytes;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  // Instruction descriptor: fp32 D; bf16: bf16 A/B, A K-major (M-major when kAT, bit 15),
  // B MN-major (K-major when kBT, bit 16 clear); MXFP4: E2M1 A/B, E8M0 scales, both K-major.
  // N >> 3 at bit 17, M >> 4 at bit 24.
  static constexpr uint32_t kIdesc =
      kMx ? ((1u << 7) | (1u << 10) | (1u << 23) | (uint32_t(kBN >> 3) << 17) |
             (uint32_t(kBM >> 4) << 24))
          : ((1u << 4) | (kF8 ? 0u : ((1u << 7) | (1u << 10))) | (kAT ? (1u << 15) : 0u) |
             (kBT ? 0u : (1u << 16)) | (uint32_t(kBN >> 3) << 17) | (uint32_t(kMmaM >> 4) << 24));
  // (A/B format fields: bf16 = 1 for kind::f16, E4M3 = 0 for kind::f8f6f4)
};

__device__ __forceinline__ void record_error(const Args& a, uint32_t site, int64_t tile) {
  if (atomicCAS(&a.err[0], 0u, kErrTimeout) == 0u) {
    a.err[1] = site;
    a.err[2] = blockIdx.x;
    a.err[3] = static_cast<uint32_t>(tile);
  }
}

// Bounded mbarrier wait.  Gives up when the CTA has aborted or the time limit runs out (then
// it records the error and aborts the CTA).
__device__ __forceinline__ bool wait_bar(uint64_t* bar, uint32_t parity,
                                         volatile uint32_t* abort_flag, const Args& a,
                                         uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((++n & 255u) == 0) {
      if (*abort_flag) return false;
      if (global_timer_ns() - t0 > a.timeout_ns) {
        *abort_flag = 1;
        record_error(a, site, -1);
        return false;
      }
    }
  }
}

// Bounded wait used while tearing down: no abort check.
__device__ __forceinline__ bool wait_bar_drain(uint64_t* bar, uint32_t parity, uint64_t limit) {
  const uint64_t t0 = global_timer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (global_timer_ns() - t0 > limit) return false;
  }
  return true;
}

__device__ __forceinline__ bool wait_flag(const uint32_t* flag, uint32_t epoch,
                                          uint64_t timeout_ns) {
  if (flag_acquire(flag) == epoch) return true;
  const uint64_t t0 = global_timer_ns();
  // Back off to at most ~128 ns between polls: one thread per CTA polls one word, and a
  // longer sleep would be added to the fix-up of a tile whose contributor finishes last.
  uint32_t ns = 32;
  while (true) {
    __nanosleep(ns);
    if (ns < 128) ns <<= 1;
    if (flag_acquire(flag) == epoch) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// Thread 0 of an owner's epilogue while its piece's k-loop may still run: waits for the flag of
// one contributor, unless the k-loop finishes first (the accumulator's full barrier `full`
// completes phase `parity`) or the CTA is aborting.  kPollFlag: the flag was seen (and, with
// `consume`, cleared), so the partial can be summed into the idle accumulator now.
// kPollLoopDone: the partial is left to the drain, which reads it while it stores C.
// kPollTimeout: no flag within the limit.  (A flag holds the launch's epoch, so one left set
// is never mistaken for a later launch's; clearing it is optional.  The pair kernels, whose
// flags several CTAs may read, leave them set.)
enum : uint32_t { kPollFlag = 0, kPollLoopDone = 1, kPollTimeout = 2 };
__device__ __forceinline__ uint32_t poll_flag_or_full(uint32_t* flag, uint32_t epoch, uint64_t* full,
                                                      uint32_t parity,
                                                      volatile uint32_t* abort_flag,
                                                      uint64_t timeout_ns, bool consume = true) {
  const uint64_t t0 = global_timer_ns();
  uint32_t ns = 32;
  while (true) {
    if (mbar_test_wait(full, parity) || *abort_flag) return kPollLoopDone;
    if (flag_acquire(flag) == epoch) {
      if (consume) *reinterpret_cast<volatile uint32_t*>(flag) = 0u;
      return kPollFlag;
    }
    if (global_timer_ns() - t0 > timeout_ns) return kPollTimeout;
    __nanosleep(ns);
    if (ns < 128) ns <<= 1;
  }
}

// Eight float4 of one Stream-K partial (one 32-column chunk of a row), `stride` float4 apart.
__device__ __forceinline__ void load_partial8(float4 (&b)[8], const float4* src, int stride) {
  const uint64_t policy = l2_policy_evict_first();
#pragma unroll
  for (int q = 0; q < 8; ++q) b[q] = ld_cg_policy(src + q * stride, policy);
}

// sum = b (first) or sum += b, for one 32-column chunk.
__device__ __forceinline__ void add_partial8(float (&sum)[32], const float4 (&b)[8], bool first) {
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    sum[4 * q] = first ? b[q].x : sum[4 * q] + b[q].x;
    sum[4 * q + 1] = first ? b[q].y : sum[4 * q + 1] + b[q].y;
    sum[4 * q + 2] = first ? b[q].z : sum[4 * q + 2] + b[q].z;
    sum[4 * q + 3] = first ? b[q].w : sum[4 * q + 3] + b[q].w;
  }
}

// Adds one contributor's partial (its P slot from `src`, fragment order, stride kBM float4s per
// 4 columns) to this thread's row of kChunks 32-column chunks held in tensor memory at
// `t_stage`; the first contributor is copied.  The loads of kGroup chunks are issued together,
// so a partial costs one round trip to L2 per kGroup chunks rather than one per chunk (kGroup
// is what the kernel's register budget allows).  The whole warp takes the same `first`.
template <int kChunks, int kGroup>
__device__ __forceinline__ void stage_partial(const float4* src, uint32_t t_stage, bool first) {
  static_assert(kChunks % kGroup == 0, "chunks are loaded kGroup at a time");
#pragma unroll 1
  for (int g = 0; g < kChunks; g += kGroup) {
    float4 pp[kGroup][8];
#pragma unroll
    for (int j = 0; j < kGroup; ++j)
      load_partial8(pp[j], src + static_cast<int64_t>(g + j) * 8 * kBM, kBM);
#pragma unroll
    for (int j = 0; j < kGroup; ++j) {
      float sum[32];
      if (first) {
        add_partial8(sum, pp[j], true);
      } else {
        uint32_t prev[32];
        __syncwarp();
        tmem_load_32cols(t_stage + (g + j) * 32, prev);
        tmem_load_wait();
#pragma unroll
        for (int k = 0; k < 32; ++k) sum[k] = __uint_as_float(prev[k]);
        add_partial8(sum, pp[j], false);
      }
      __syncwarp();
      tmem_store_32cols(t_stage + (g + j) * 32, sum);
    }
  }
  tmem_store_wait();
}

// Adds bias[n0 .. n0+32) (those below N) to v.
__device__ __forceinline__ void add_bias_chunk(const Args& a, int64_t n0, float (&v)[32]) {
  if (a.bias == nullptr) return;
  const bool full_chunk = n0 + 32 <= a.N;
  if (a.out_bf16) {
    const __nv_bfloat16* bias = static_cast<const __nv_bfloat16*>(a.bias);
    if (full_chunk) {
      const uint4* bp = reinterpret_cast<const uint4*>(bias + n0);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w = __ldg(bp + q);
        const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float2 f = __bfloat1622float2(h[e]);
          v[8 * q + 2 * e] += f.x;
          v[8 * q + 2 * e + 1] += f.y;
        }
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < a.N) v[j] += __bfloat162float(bias[n0 + j]);
    }
  } else {
    const float* bias = static_cast<const float*>(a.bias);
    if (full_chunk) {
      const float4* bp = reinterpret_cast<const float4*>(bias + n0);
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        float4 f = __ldg(bp + q);
        v[4 * q] += f.x;
        v[4 * q + 1] += f.y;
        v[4 * q + 2] += f.z;
        v[4 * q + 3] += f.w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < a.N) v[j] += bias[n0 + j];
    }
  }
}

// The bias of this lane's column in each of kChunks 32-column chunks from n0 (0 past N), read
// when a piece starts so that no chunk's store waits for it.
template <int kChunks>
__device__ __forceinline__ void load_bias_lanes(const Args& a, int64_t n0, int lane,
                                                float (&b)[kChunks]) {
#pragma unroll
  for (int ch = 0; ch < kChunks; ++ch) {
    const int64_t n = n0 + ch * 32 + lane;
    b[ch] = 0.0f;
    if (a.bias != nullptr && n < a.N)
      b[ch] = a.out_bf16 ? __bfloat162float(static_cast<const __nv_bfloat16*>(a.bias)[n])
                         : static_cast<const float*>(a.bias)[n];
  }
}

// b[i] for a loop index i, without indexing the array in local memory.
template <int kChunks>
__device__ __forceinline__ float pick_chunk(const float (&b)[kChunks], int i) {
  float r = b[kChunks - 1];
#pragma unroll
  for (int k = kChunks - 2; k >= 0; --k) r = i == k ? b[k] : r;
  return r;
}

// v[j] += the bias of column j of the chunk, held by lane j.  (Nothing is added without a
// bias, so that a zero keeps its sign.)
__device__ __forceinline__ void add_bias_lanes(const Args& a, float (&v)[32], float b) {
  if (a.bias == nullptr) return;
#pragma unroll
  for (int j = 0; j < 32; ++j) v[j] += __shfl_sync(0xffffffffu, b, j);
}

// Stages one piece of C -- 32 rows (one per lane) x 64 bytes -- in `buf` and writes it with a
// TMA store at column x, row y.  The tensor map clips rows and columns past the matrix edge;
// a piece that starts past the edge is skipped (returns false).  The caller alternates between
// two buffers after every issued store, so the most recent pending store used the other one,
// and a wait for at most one pending group means this buffer's last store has read it.
__device__ __forceinline__ bool tma_store_piece(const Args& a, const CUtensorMap* tmC,
                                                uint8_t* buf, int lane, const uint4 (&q)[4],
                                                int64_t x, int64_t y) {
  if (x >= a.N || y >= a.M) return false;
  if (lane == 0) bulk_wait_read<1>();
  __syncwarp();
  // C's tensor map uses the 64-byte swizzle: 16-byte chunk i of row r sits at chunk
  // i ^ ((r >> 1) & 3), so the eight rows of each quarter-warp write eight different banks.
  uint4* dst = reinterpret_cast<uint4*>(buf + lane * 64);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i ^ sw] = q[i];
  fence_async_shared();
  __syncwarp();
  if (lane == 0) {
    tma_store_2d(tmC, buf, static_cast<int32_t>(x), static_cast<int32_t>(y));
    bulk_commit();
  }
  return true;
}

// Adds the bias to columns [n0, n0+32) of this warp's 32 rows (rows y .. y+31, one per lane),
// casts, and stores them through the warp's two 2 KB staging buffers (`stage`, alternating by
// `buf`): one bf16 piece of 32 columns, or two fp32 pieces of 16.
// (kAddBias = false: the caller has added the bias.)
template <bool kAddBias = true>
__device__ __forceinline__ void store_chunk_tma(const Args& a, const CUtensorMap* tmC,
                                                uint8_t* stage, int& buf, int lane, int64_t n0,
                                                int64_t y, float (&v)[32]) {
  if constexpr (kAddBias) add_bias_chunk(a, n0, v);
  if (a.out_bf16) {
    uint4 q[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q[i]);
#pragma unroll
      for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(v[8 * i + 2 * e], v[8 * i + 2 * e + 1]);
    }
    if (tma_store_piece(a, tmC, stage + buf * 2048, lane, q, n0, y)) buf ^= 1;
  } else {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint4 q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i)
        q[i] = make_uint4(__float_as_uint(v[16 * hf + 4 * i]), __float_as_uint(v[16 * hf + 4 * i + 1]),
                          __float_as_uint(v[16 * hf + 4 * i + 2]), __float_as_uint(v[16 * hf + 4 * i + 3]));
      if (tma_store_piece(a, tmC, stage + buf * 2048, lane, q, n0 + 16 * hf, y)) buf ^= 1;
    }
  }
}

// The same through one 1 KB staging buffer per warp (the MXFP4 pair kernel's shared memory has
// room for no more): pieces of 32 bytes of each of the warp's 32 rows -- 16 bf16 or 8 fp32
// columns, two or four per 32-column chunk -- each stored by TMA (C's tensor map then has
// 32 x 32-byte boxes, no swizzle) once the previous piece has been read out of the buffer.
template <bool kAddBias = true>
__device__ __forceinline__ void store_chunk_tma_1k(const Args& a, const CUtensorMap* tmC,
                                                   uint8_t* buf, int lane, int64_t n0, int64_t y,
                                                   float (&v)[32]) {
  if constexpr (kAddBias) add_bias_chunk(a, n0, v);
  const int cols = a.out_bf16 ? 16 : 8;   // columns per 32-byte piece
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    if (a.out_bf16 && p >= 2) break;
    const int64_t x = n0 + cols * p;
    if (x >= a.N || y >= a.M) break;
    uint4 q[2];
    if (a.out_bf16) {
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q[i]);
#pragma unroll
        for (int e = 0; e < 4; ++e)
          h[e] = __floats2bfloat162_rn(v[16 * p + 8 * i + 2 * e], v[16 * p + 8 * i + 2 * e + 1]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 2; ++i)
        q[i] = make_uint4(__float_as_uint(v[8 * p + 4 * i]), __float_as_uint(v[8 * p + 4 * i + 1]),
                          __float_as_uint(v[8 * p + 4 * i + 2]), __float_as_uint(v[8 * p + 4 * i + 3]));
    }
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
    uint4* dst = reinterpret_cast<uint4*>(buf + lane * 32);
    dst[0] = q[0];
    dst[1] = q[1];
    fence_async_shared();
    __syncwarp();
    if (lane == 0) {
      tma_store_2d(tmC, buf, static_cast<int32_t>(x), static_cast<int32_t>(y));
      bulk_commit();
    }
  }
}

// Adds the bias (unless kAddBias is false), casts and stores 32 consecutive columns [n0, n0+32)
// of row m.
template <bool kAddBias = true>
__device__ __forceinline__ void store_row_chunk(const Args& a, int64_t m, int64_t n0,
                                                float (&v)[32]) {
  if (m >= a.M) return;
  const bool full_chunk = (n0 + 32 <= a.N) && ((a.N & 7) == 0);
  if (a.out_bf16) {
    const __nv_bfloat16* bias = kAddBias ? static_cast<const __nv_bfloat16*>(a.bias) : nullptr;
    __nv_bfloat16* c = static_cast<__nv_bfloat16*>(a.C) + m * a.N + n0;
    if (full_chunk) {
      if (bias != nullptr) {
        const uint4* bp = reinterpret_cast<const uint4*>(bias + n0);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 w = __ldg(bp + q);
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&w);
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float2 f = __bfloat1622float2(h[e]);
            v[8 * q + 2 * e] += f.x;
            v[8 * q + 2 * e + 1] += f.y;
          }
        }
      }
      uint4* cp = reinterpret_cast<uint4*>(c);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) h[e] = __floats2bfloat162_rn(v[8 * q + 2 * e], v[8 * q + 2 * e + 1]);
        cp[q] = w;
      }
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (n0 + j < a.N) {
          float y = v[j];
          if (bias != nullptr) y += __bfloat162float(bias[n0 + j]);
          c[j] = __float2bfloat16_rn(y);
        }
      }
    }
  } else {
    const float* bias = kAddBias ? static_cast<const float*>(a.bias) : nullptr;
    float* c = static_cast<float*>(a.C) + m * a.N + n0;
    if (full_chunk) {
      if (bias != nullptr) {
        const float4* bp = reinterpret_cast<const float4*>(bias + n0);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          float4 f = __ldg(bp + q);
          v[4 * q] += f.x;
          v[4 * q + 1] += f.y;
          v[4 * q + 2] += f.z;
          v[4 * q + 3] += f.w;
        }
      }
      float4* cp = reinterpret_cast<float4*>(c);
#pragma unroll
      for (int q = 0; q < 8; ++q) cp[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        if (n0 + j < a.N) c[j] = v[j] + (bias != nullptr ? bias[n0 + j] : 0.0f);
      }
    }
  }
}

template <bool kMx, int kBN, bool kAT = false, bool kBT = false, bool kF8 = false,
          bool kTall = false>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmC, const __grid_constant__ Args args) {
  using Cf = Cfg<kMx, kBN, kAT, kBT, kF8, kTall>;
  constexpr int S = Cf::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring_a = smem;
  uint8_t* ring_b = ring_a + S * Cf::kStageA;
  uint8_t* ring_sfa = ring_b + S * Cf::kStageB;
  uint8_t* ring_sfb = ring_sfa + S * Cf::kStageSfa;
  uint8_t* epi_stage = ring_sfb + S * Cf::kStageSfb;   // 1 KB aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + Cf::kEpiBytes);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + 2;
  uint64_t* mma_done = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* unit_status = tmem_slot + 2;   // two slots, indexed by accumulator
  volatile uint32_t* staged_status = tmem_slot + 4; // two slots: partials staged in tensor memory

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int64_t cta = blockIdx.x;
  const Plan& plan = args.plan;
  record_sm(args.sm_record);

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], kEpilogueThreads / 32);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    unit_status[0] = 0;
    unit_status[1] = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, Cf::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      Cursor cur(plan, cta);
      Unit u;
      while (ok && cur.next(plan, u)) {
        int32_t tm, tn;
        tile_coords(plan, u.tile, tm, tn);
        for (int32_t i = 0; i < u.k1 - u.k0; ++i) {
          const int32_t k = unit_k(u, i);
          if (!wait_bar(&empty[stage], phase ^ 1u, abort_flag, args, kSiteProducer)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&full[stage], Cf::kStageBytes);
          uint8_t* sa = ring_a + stage * Cf::kStageA;
          uint8_t* sb = ring_b + stage * Cf::kStageB;
          if constexpr (kMx) {
            tma_load_2d(sa, &tmA, &full[stage], k * 128, tm * kBM);
            tma_load_2d(sb, &tmB, &full[stage], k * 128, tn * kBN);
            bulk_load(ring_sfa + stage * Cf::kStageSfa,
                      args.sfa + (static_cast<int64_t>(tm) * args.sf_kgroups + 2 * k) * 512, 1024,
                      &full[stage]);
#pragma unroll
            for (int j = 0; j < kBN / 128; ++j) {
              const int64_t nb = static_cast<int64_t>(tn) * (kBN / 128) + j;
              bulk_load(ring_sfb + stage * Cf::kStageSfb + j * 1024,
                        args.sfb + (nb * args.sf_kgroups + 2 * k) * 512, 1024, &full[stage]);
            }
          } else {
            constexpr int TK = Cf::kTileK, AT = Cf::kAtom, BX = Cf::kBoxBytes;
            // A: K-major tile (128 rows x TK), or M-major (TK k-rows x 128 m, AT-wide boxes).
            if constexpr (kAT) {
#pragma unroll
              for (int j = 0; j < kBM / AT; ++j)
                tma_load_2d(sa + j * BX, &tmA, &full[stage], tm * kBM + j * AT, k * TK);
            } else {
              // one box of kARows rows x 64 k per 128-byte K atom (two for tall stages)
#pragma unroll
              for (int h = 0; h < Cf::kKHalves; ++h)
                tma_load_2d(sa + h * (Cf::kARows * 128), &tmA, &full[stage], k * TK + h * 64,
                            tm * kBM);
            }
            // B: MN-major (TK k-rows x BN n, kAtomB-wide boxes), or K-major (BN rows x TK k).
            if constexpr (kBT) {
              tma_load_2d(sb, &tmB, &full[stage], k * TK, tn * kBN);
            } else {
              constexpr int ATB = Cf::kAtomB, BXB = Cf::kBoxBytesB;
#pragma unroll
              for (int j = 0; j < kBN / ATB; ++j)
                tma_load_2d(sb + j * BXB, &tmB, &full[stage], tn * kBN + j * ATB, k * TK);
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok) {
        // Let the copies already issued land before the CTA's shared memory goes away.
        const int64_t outstanding = issued < S ? issued : S;
        for (int64_t i = 1; i <= outstanding; ++i) {
          const int s = static_cast<int>((stage - i + S) % S);
          const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
          if (!wait_bar_drain(&full[s], par, 100000000ull)) record_error(args, kSiteDrain, -1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      Cursor cur(plan, cta);
      Unit u;
      while (ok && cur.next(plan, u)) {
        if (!wait_bar(&tempty[acc], acc_phase ^ 1u, abort_flag, args, kSiteMma)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc) * Cf::kAccCols;
        for (int32_t i = 0; i < u.k1 - u.k0; ++i) {
          const int32_t k = unit_k(u, i);
          if (!wait_bar(&full[stage], phase, abort_flag, args, kSiteMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_addr(ring_a + stage * Cf::kStageA);
          const uint32_t b0 = smem_addr(ring_b + stage * Cf::kStageB);
          if constexpr (kMx) {
            // Scale blocks of this stage -> tensor memory slot `stage` (each 512-byte group
            // holds 128 rows x 4 scale bytes, rows r, r+32, r+64, r+96 in one 16-byte line).
            const uint32_t sfa_t = tmem_base + 2 * Cf::kAccCols + stage * Cf::kSfaCols;
            const uint32_t sfb_t = tmem_base + 2 * Cf::kAccCols + S * Cf::kSfaCols + stage * Cf::kSfbCols;
            const uint32_t sfa_s = smem_addr(ring_sfa + stage * Cf::kStageSfa);
            const uint32_t sfb_s = smem_addr(ring_sfb + stage * Cf::kStageSfb);
#pragma unroll
            for (int g = 0; g < 2; ++g)
              tmem_copy_32x128b_x4(sfa_t + g * 4, smem_desc(sfa_s + g * 512, 0, 128, kLayoutSwizzleNone));
#pragma unroll
            for (int j = 0; j < kBN / 128; ++j)
#pragma unroll
              for (int g = 0; g < 2; ++g)
                tmem_copy_32x128b_x4(sfb_t + g * (kBN / 32) + j * 4,
                                     smem_desc(sfb_s + j * 1024 + g * 512, 0, 128, kLayoutSwizzleNone));
#pragma unroll
            for (int j = 0; j < Cf::kMmasPerStage; ++j) {
              const uint32_t g = j >> 1;
              const uint32_t sf_id = (j & 1) * 2;
              const uint32_t idesc = Cf::kIdesc | (sf_id << 29) | (sf_id << 4);
              const uint64_t ad = smem_desc(a0 + j * 32, 16, 1024, kLayoutSwizzle128B);
              const uint64_t bd = smem_desc(b0 + j * 32, 16, 1024, kLayoutSwizzle128B);
              mma_mxf4(d_tmem, ad, bd, idesc, sfa_t + g * 4, sfb_t + g * (kBN / 32),
                       (i > 0 || j > 0) ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < Cf::kMmasPerStage; ++j) {
              // A: K-major, 128-byte swizzle, 8-row groups 1024 B apart; K advances 32 B.
              // B: MN-major, 128-byte swizzle; 64-column blocks 8 KB apart (leading offset),
              //    8-row K groups 1024 B apart (stride offset); K advances 16 rows = 2 KB.
              // K-major: K advances 32 bytes along the swizzled row.  M-major A / MN-major B:
              // blocks of 128-byte rows kBoxBytes apart, K advances kMmaK rows.
              // (Tall stages: MMAs 4-7 read the second K atom, kARows * 128 bytes on.)
              constexpr uint32_t BX = Cf::kBoxBytes, ADV = Cf::kMnAdvance;
              const uint64_t ad =
                  kAT ? smem_desc(a0 + j * ADV, BX, 1024, kLayoutSwizzle128B)
                      : smem_desc(a0 + (j / 4) * (Cf::kARows * 128) + (j % 4) * 32, 16, 1024,
                                  kLayoutSwizzle128B);
              // MN-major B: blocks kBoxBytesB apart, 8-row K groups 8 * kRowB apart, K advances
              // kMmaK rows.
              constexpr uint32_t BXB = Cf::kBoxBytesB, RB = Cf::kRowB;
              const uint64_t bd = kBT ? smem_desc(b0 + j * 32, 16, 1024, kLayoutSwizzle128B)
                                      : smem_desc(b0 + j * Cf::kMmaK * RB, BXB, 8 * RB, Cf::kLayoutB);
              if constexpr (kF8) {
                mma_f8(d_tmem, ad, bd, Cf::kIdesc, (i > 0 || j > 0) ? 1u : 0u);
              } else {
                mma_f16(d_tmem, ad, bd, Cf::kIdesc, (i > 0 || j > 0) ? 1u : 0u);
              }
            }
          }
          mma_commit(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // Every MMA this thread issued has completed once mma_done flips.
      mma_commit(mma_done);
      if (!wait_bar_drain(mma_done, 0, 100000000ull)) record_error(args, kSiteDrain, -1);
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    // Thread 0 of the epilogue does the waits of a piece (accumulator ready; for an owner,
    // the contributors' flags) and publishes the outcome in unit_status[acc]; a named barrier
    // then makes the decision uniform, so no epilogue thread can be left at a barrier.
    const int quarter = warp & 3;               // TMEM lanes this warp may read
    const int row = quarter * 32 + lane;        // tile row of this thread
    const int et = threadIdx.x - 64;            // 0..127
    int acc = 0;
    uint32_t acc_phase = 0;
    uint8_t* my_stage = epi_stage + (warp - 2) * 4096;   // this warp's two C staging buffers
    int sbuf = 0;
    Cursor cur(plan, cta);
    Unit u;
    while (cur.next(plan, u)) {
      // where this piece's rows and columns lie (worked out before the waits below)
      int32_t tm, tn;
      tile_coords(plan, u.tile, tm, tn);
      const int64_t y_warp = static_cast<int64_t>(tm) * kBM + quarter * 32;
      // (tall stages: this lane's accumulator row, or past the matrix for lanes 16-31)
      const int64_t m = Cf::kMmaM == 64
                            ? (lane < 16 ? static_cast<int64_t>(tm) * kBM + quarter * 16 + lane : args.M)
                            : y_warp + lane;
      const int64_t n_tile = static_cast<int64_t>(tn) * kBN;
      float bias_l[kBN / 32];
      load_bias_lanes(args, n_tile, lane, bias_l);
      bool has_next;
      {
        Cursor peek = cur;
        Unit later;
        has_next = peek.next(plan, later);
      }
      // Contributions to an owned tile come from CTAs cta+1, cta+2, ... until k is covered.
      int n_contrib = 0;
      if (u.role == kRoleOwner) {
        int64_t covered = u.k1;
        for (int64_t c = cta + 1; covered < plan.iters; ++c, ++n_contrib) {
          const int64_t len = sk_range_len(plan, c);
          covered += (len < plan.iters - covered) ? len : (plan.iters - covered);
        }
      }
      // A shared tile that is this CTA's last piece: while its k-loop still runs, the
      // contributors' partials that are already complete are summed into the idle accumulator
      // (which held the previous piece, already drained; no later piece uses it); the drain
      // after the loop reads the rest.
      const bool staged = u.role == kRoleOwner && !has_next && n_contrib > 0;
      const uint32_t t_stage = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                               static_cast<uint32_t>(acc ^ 1) * Cf::kAccCols;
      uint32_t flag_status = kUnitStore;
      int n_staged = 0;   // contributors summed into the idle accumulator (the farthest ones)
      if (staged) {
        // The farthest contributor first: it worked on this tile at the start of its range and
        // is long done, while the nearest may still be on it.  Each partial is added as soon as
        // its flag is seen, for as long as the k-loop runs; the rest are read by the drain.
        // (The status word alternates between two slots, so thread 0 never overwrites one
        // that a slower thread has yet to read.)
#pragma unroll 1
        for (int i = 0; i < n_contrib; ++i) {
          const int c = n_contrib - 1 - i;
          if (et == 0) {
            const uint32_t r = poll_flag_or_full(args.flags + cta + 1 + c, args.epoch, &tfull[acc],
                                                 acc_phase, abort_flag, args.timeout_ns);
            if (r == kPollTimeout) record_error(args, kSiteFlag, u.tile);
            staged_status[i & 1] = r;
          }
          named_barrier_sync(1, kEpilogueThreads);
          const uint32_t r = staged_status[i & 1];
          if (r == kPollLoopDone) break;
          if (r == kPollTimeout) {
            flag_status = kUnitSkip;
            break;
          }
          stage_partial<kBN / 32, (kBN / 32) % 2 == 0 ? 2 : 1>(
              reinterpret_cast<const float4*>(args.P + (cta + 1 + c) * (kBM * kBN)) + row, t_stage,
              i == 0);
          n_staged = i + 1;
        }
      }
      // contributors 0 .. n_rem-1 (the nearest) are read by the drain
      const int n_rem = flag_status == kUnitStore ? n_contrib - n_staged : 0;
      if (et < 32) {
        // Lane 0 of the first epilogue warp waits for the accumulator; an owner then waits for
        // its remaining contributors' flags, lane l for contributors l, l + 32, ... side by side.
        uint32_t status = kUnitStore;
        if (et == 0 && !wait_bar(&tfull[acc], acc_phase, abort_flag, args, kSiteEpilogue))
          status = kUnitAbort;
        status = __shfl_sync(0xffffffffu, status, 0);
        if (status == kUnitStore && u.role == kRoleOwner) {
          bool ok = true;
          for (int c = et; c < n_rem && ok; c += 32) {
            uint32_t* f = args.flags + cta + 1 + c;
            ok = wait_flag(f, args.epoch, args.timeout_ns);
            if (ok) *reinterpret_cast<volatile uint32_t*>(f) = 0u;  // consumed: ready for the next launch
          }
          if (!__all_sync(0xffffffffu, ok)) {
            if (et == 0) record_error(args, kSiteFlag, u.tile);
            status = kUnitSkip;
          }
        }
        if (et == 0) unit_status[acc] = status;
      }
      named_barrier_sync(1, kEpilogueThreads);
      const uint32_t status = unit_status[acc];
      if (status == kUnitAbort) break;
      tc_fence_after();
      const bool do_store = status == kUnitStore && flag_status == kUnitStore;

      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc) * Cf::kAccCols;
      float4* my_slot = reinterpret_cast<float4*>(args.P + cta * (kBM * kBN));
      // Partials not summed during the k-loop are read here: two contributors' chunks in
      // flight at a time, the next chunk's requested before this one is stored, so the round
      // trips to L2 overlap the drain's other work.
      constexpr int64_t kSlot4 = kBM * kBN / 4;   // float4s between consecutive CTAs' slots
      const float4* rem0 = reinterpret_cast<const float4*>(args.P + (cta + 1) * (kBM * kBN)) + row;
      float4 pp[8], pq[8];
      if (do_store && n_rem > 0) load_partial8(pp, rem0, kBM);
      if (do_store && n_rem > 1) load_partial8(pq, rem0 + kSlot4, kBM);
#pragma unroll 1
      for (int ch = 0; ch < kBN / 32; ++ch) {
        const float4* rem = rem0 + static_cast<int64_t>(ch) * 8 * kBM;
        uint32_t r[32];
        __syncwarp();
        tmem_load_32cols(t_row + ch * 32, r);
        float v[32];
        if (n_staged > 0) {
          uint32_t part[32];
          tmem_load_32cols(t_stage + ch * 32, part);
          tmem_load_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]) + __uint_as_float(part[j]);
        } else {
          tmem_load_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
        }
        if (u.role == kRoleContrib) {
          // Slot layout [chunk][column quad][row]: one warp store covers 512 contiguous bytes.
          float4* dst = my_slot + static_cast<int64_t>(ch) * 8 * kBM + row;
          const uint64_t policy = l2_policy_evict_last();
#pragma unroll
          for (int q = 0; q < 8; ++q)
            st_cg_policy(dst + q * kBM, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]),
                         policy);
        } else if (do_store) {
          if (n_rem > 0) {
            add_partial8(v, pp, false);
            if (n_rem > 1) add_partial8(v, pq, false);
#pragma unroll 1
            for (int c = 2; c < n_rem; c += 2) {
              load_partial8(pp, rem + c * kSlot4, kBM);
              if (c + 1 < n_rem) load_partial8(pq, rem + (c + 1) * kSlot4, kBM);
              add_partial8(v, pp, false);
              if (c + 1 < n_rem) add_partial8(v, pq, false);
            }
            if (ch + 1 < kBN / 32) {
              load_partial8(pp, rem + 8 * kBM, kBM);
              if (n_rem > 1) load_partial8(pq, rem + 8 * kBM + kSlot4, kBM);
            }
          }
          add_bias_lanes(args, v, pick_chunk(bias_l, ch));
          if (args.c_tma && Cf::kMmaM == kBM) {   // (M = 64 accumulators: direct stores)
            store_chunk_tma<false>(args, &tmC, my_stage, sbuf, lane, n_tile + ch * 32, y_warp, v);
          } else {
            store_row_chunk<false>(args, m, n_tile + ch * 32, v);
          }
        }
      }
      // Accumulator drained: hand it back to the MMA warp.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (u.role == kRoleContrib) {
        // Publish the partial: every thread's stores, then one release at GPU scope.
        __threadfence();
        named_barrier_sync(1, kEpilogueThreads);
        if (et == 0 && !(args.inject_drop && cta == args.drop_cta))
          flag_release(args.flags + cta, args.epoch);
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (lane == 0) bulk_wait_all();   // staged pieces of C are read and written before exit
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Cf::kTmemCols);
  }
}

}  // namespace sk
