// The addmm GEMM kernel on SM pairs: a cluster of two CTAs computes one 256 x 256 output tile
// with tcgen05 cta_group::2 MMAs (M = 256), each CTA holding 128 rows x 256 fp32 columns of
// the accumulator in its own tensor memory.  Same schedules, roles and results as
// sk_kernel.cuh; what changes is the data each SM moves per FLOP: a CTA loads its 128 rows of A
// and half (128 columns) of the B tile, and the pair's MMA reads the other half of B from the
// peer CTA, so operand traffic per SM per MMA drops by a third (bf16) to a half (MXFP4).
//
// Roles (320 threads per CTA, one CTA per SM, clusters of 2):
//   warp 0      TMA producer of this CTA's halves.  Both CTAs' loads complete on the leader
//               CTA's (cluster rank 0) "full" barrier, which expects the bytes of both.
//   warp 1      both CTAs allocate tensor memory together; in the leader one lane issues the
//               cta_group::2 MMAs and commits them to the "empty" and "accumulator full"
//               barriers of both CTAs at once (multicast).
//   warps 2..9  epilogue, two warps per 32-lane quarter: warp w reads lanes 32*(w%4).. and
//               columns [128*h, 128*h+128), h = (w-2)/4.  Each thread drains its row 32
//               columns at a time (bf16, fp8) or all 128 into registers at once (MXFP4), spills
//               them (contribution) or adds partials + bias, casts and stores them, and then
//               releases the accumulator to the leader.
//   warp 10     (MXFP4 only) in the leader, one lane copies each stage's scale factors from
//               shared to tensor memory (tcgen05.cp) and commits them to that stage's
//               "scales ready" barrier, which the MMA thread waits on; keeping the copies off
//               the MMA thread lets them overlap the previous stage's MMAs.
// MXFP4 keeps one accumulator (256 columns) so that the per-stage scale-factor slots fit in
// the 512 tensor-memory columns; the fast drain keeps the MMA's wait for it short.  bf16 keeps
// two accumulators.
//
// Shared finish (bf16, fp8): where a split tile's owner ends its range on that tile and at
// least two of its contributors hold nothing but their piece of it, the owner and those
// contributors each finish a share of the tile's 32-column chunks.  Each writes the other
// parties' chunks of its accumulator to scratch (the owner to a second slot) and releases a
// flag, then waits for the others' flags and adds their partials, the bias, and stores its
// own chunks.  Every element still gets every partial and the bias exactly once.  Without it
// the owner alone reads all the partials after its k-loop, while the contributors, done at
// the same moment, sit idle: 1.5x faster Stream-K on 512 x 512 x 16384, 1.1x on 1024^2 x 16384.
// A flag may then have several readers, so flags are not cleared once read: each launch
// releases them with a new epoch.  A launch captured into a CUDA graph keeps one epoch for all
// its replays; it finishes every tile by its owner alone, which clears each flag it reads.
#pragma once

#include "sk_kernel.cuh"

namespace sk {

constexpr int kPairEpilogueThreads = 256;
// 2 issuing warps + 8 epilogue warps; MXFP4 adds a warp that copies scale factors to TMEM.
template <bool kMx>
constexpr int pair_threads() { return kMx ? 352 : 320; }

__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// Address of the same shared-memory location in cluster CTA `rank`.
__device__ __forceinline__ uint32_t cluster_addr(const void* p, uint32_t rank) {
  uint32_t out;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(p)), "r"(rank));
  return out;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}

__device__ __forceinline__ void remote_arrive(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_addr(dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void mma_f16_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                             uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_mxf4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                              uint32_t idesc, uint32_t sfa_tmem,
                                              uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%5], "
      "[%6], p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "r"(sfa_tmem), "r"(sfb_tmem)
      : "memory");
}

__device__ __forceinline__ void tmem_copy_32x128b_x4_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc)
               : "memory");
}

// Arrive once on `bar` (same offset) in both CTAs of the pair when this thread's tcgen05
// operations have completed.
__device__ __forceinline__ void mma_commit_pair(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
      " [%0], %1;" ::"r"(smem_addr(bar)),
      "h"(static_cast<uint16_t>(3))
      : "memory");
}

// Arrive once on this CTA's `bar` when this thread's tcgen05 operations have completed.
__device__ __forceinline__ void mma_commit_pair_local(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_addr(bar))
               : "memory");
}

// TMA 2-D load into this CTA's shared memory, completing on a barrier of either CTA of the
// pair (cluster address).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* map,
                                                 uint32_t cluster_bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(cluster_bar), "r"(x), "r"(y)
      : "memory");
}

template <bool kMx, bool kAT = false, bool kBT = false, bool kF8 = false>
struct PairCfg {
  static_assert(!kMx || (!kAT && !kBT && !kF8), "MXFP4 operands are K-major");
  static constexpr int kBN = 256;                        // pair tile: 256 x 256
  static constexpr int kHalfN = kBN / 2;                 // B columns loaded by each CTA
  static constexpr int kTileK = kMx ? 256 : (kF8 ? 128 : 64);   // one 128-byte row of K
  static constexpr int kMmaK = kMx ? 64 : (kF8 ? 32 : 16);
  static constexpr int kMmasPerStage = kTileK / kMmaK;   // 4
  static constexpr int kAtom = kF8 ? 128 : 64;           // MN-major block width (128 bytes)
  static constexpr int kBoxBytes = kTileK * 128;
  static constexpr int kMnAdvance = kMmaK * 128;
  static constexpr int kStageA = kBM * 128;              // 16 KB
  static constexpr int kStageB = kHalfN * 128;           // 16 KB
  static constexpr int kStageSfa = kMx ? 1024 : 0;       // own 128 rows, 2 k groups
  static constexpr int kStageSfb = kMx ? 2048 : 0;       // all 256 columns, 2 k groups
  static constexpr int kStageBytes = kStageA + kStageB + kStageSfa + kStageSfb;
  static constexpr int kStages = (212 * 1024) / kStageBytes;
  // bf16 / fp8 results leave through TMA stores: each epilogue warp stages 32 rows x 64 bytes
  // of C in one of its two 2 KB buffers.  MXFP4, whose scale-factor slots take the room, has
  // one 1 KB buffer per warp: its C leaves through 32 x 32-byte TMA stores when C's rows are
  // 16-byte aligned (args.c_tma), else through direct stores.
  static constexpr bool kTmaStore = !kMx;
  static constexpr int kEpiBytes = kTmaStore ? 8 * 2 * 2048 : 8 * 1024;
  static constexpr int kAccBufs = kMx ? 1 : 2;
  static constexpr uint32_t kAccCols = kBN;
  static constexpr uint32_t kSfaCols = 8;
  static constexpr uint32_t kSfbCols = 16;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kAccBufs * kAccCols + (kMx ? kStages * (kSfaCols + kSfbCols) : 0) <= kTmemCols,
                "tensor memory budget");
  static constexpr int kBarrierBytes = 512;
  static_assert((3 * kStages + 6) * 8 + 24 <= kBarrierBytes, "barrier area");
  static constexpr size_t kSmemBytes =
      1024 + static_cast<size_t>(kStages) * kStageBytes + kEpiBytes + kBarrierBytes;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
  static constexpr uint32_t kIdesc =
      kMx ? ((1u << 7) | (1u << 10) | (1u << 23) | (uint32_t(kBN >> 3) << 17) |
             (uint32_t(256 >> 4) << 24))
          : ((1u << 4) | (kF8 ? 0u : ((1u << 7) | (1u << 10))) | (kAT ? (1u << 15) : 0u) |
             (kBT ? 0u : (1u << 16)) | (uint32_t(kBN >> 3) << 17) | (uint32_t(256 >> 4) << 24));
};

// Registers are granted per 128-thread warpgroup, so 320 or 352 threads are charged as 384:
// the launch bound caps the kernel at 65536 / 384 -> 168 registers per thread.
template <bool kMx, bool kAT = false, bool kBT = false, bool kF8 = false>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(pair_threads<kMx>(), 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmSfa,
                     const __grid_constant__ CUtensorMap tmSfb,
                     const __grid_constant__ CUtensorMap tmC, const __grid_constant__ Args args) {
  using Cf = PairCfg<kMx, kAT, kBT, kF8>;
  constexpr int S = Cf::kStages;
  constexpr int kBN = Cf::kBN;
  constexpr bool kShare = Cf::kAccBufs == 2;   // shared tiles may be finished by several CTAs
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* ring_a = smem;
  uint8_t* ring_b = ring_a + S * Cf::kStageA;
  uint8_t* ring_sfa = ring_b + S * Cf::kStageB;
  uint8_t* ring_sfb = ring_sfa + S * Cf::kStageSfa;
  uint8_t* epi_stage = ring_sfb + S * Cf::kStageSfb;   // 1 KB aligned
  uint64_t* bars = reinterpret_cast<uint64_t*>(epi_stage + Cf::kEpiBytes);
  uint64_t* full = bars;                 // leader: both CTAs' bytes of a stage
  uint64_t* empty = bars + S;            // each CTA: its stage may be refilled
  uint64_t* tfull = bars + 2 * S;        // each CTA: accumulator b is ready
  uint64_t* tempty = tfull + 2;          // leader: both CTAs have drained accumulator b
  uint64_t* mma_done = tempty + 2;
  uint64_t* sf_ready = mma_done + 1;     // leader, MXFP4: stage's scales are in TMEM
  uint64_t* cp_done = sf_ready + S;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(cp_done + 1);
  volatile uint32_t* abort_flag = tmem_slot + 1;
  volatile uint32_t* unit_status = tmem_slot + 2;   // two slots, indexed by unit parity
  volatile uint32_t* staged_status = tmem_slot + 4; // two slots: partials staged in tensor memory

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_rank();
  const bool leader = rank == 0;
  const int64_t pair = blockIdx.x >> 1;
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
      mbar_init(&tempty[b], 2 * (kPairEpilogueThreads / 32));
    }
    mbar_init(mma_done, 1);
    for (int st = 0; st < S; ++st) mbar_init(&sf_ready[st], 1);
    mbar_init(cp_done, 1);
    *abort_flag = 0;
    unit_status[0] = 0;
    unit_status[1] = 0;
    fence_mbar_init();
    prefetch_tensormap(&tmA);
    prefetch_tensormap(&tmB);
    if constexpr (kMx) {
      prefetch_tensormap(&tmSfa);
      prefetch_tensormap(&tmSfb);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, Cf::kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();   // both CTAs' barriers exist before any cross-CTA signal
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint32_t full_leader0 = cluster_addr(&full[0], 0);
      int stage = 0;
      uint32_t phase = 0;
      int64_t issued = 0;
      bool ok = true;
      Cursor cur(plan, pair);
      Unit u;
      while (ok && cur.next(plan, u)) {
        int32_t tm, tn;
        tile_coords(plan, u.tile, tm, tn);
        const int32_t row0 = tm * 256 + static_cast<int32_t>(rank) * 128;
        const int32_t col0 = tn * kBN + static_cast<int32_t>(rank) * Cf::kHalfN;
        for (int32_t i = 0; i < u.k1 - u.k0; ++i) {
          const int32_t k = unit_k(u, i);
          if (!wait_bar(&empty[stage], phase ^ 1u, abort_flag, args, kSiteProducer)) {
            ok = false;
            break;
          }
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * Cf::kStageBytes);
          const uint32_t fb = full_leader0 + stage * 8;
          uint8_t* sa = ring_a + stage * Cf::kStageA;
          uint8_t* sb = ring_b + stage * Cf::kStageB;
          if constexpr (kMx) {
            tma_load_2d_pair(sa, &tmA, fb, k * 128, row0);
            tma_load_2d_pair(sb, &tmB, fb, k * 128, col0);
            // scale blocks: rows of 1 KB = (row block, k-iteration); A: this CTA's 128 rows,
            // B: both 128-column blocks of the pair's tile.
            tma_load_2d_pair(ring_sfa + stage * Cf::kStageSfa, &tmSfa, fb, 0,
                             (tm * 2 + static_cast<int32_t>(rank)) * plan.iters + k);
            tma_load_2d_pair(ring_sfb + stage * Cf::kStageSfb, &tmSfb, fb, 0,
                             (tn * 2) * plan.iters + k);
            tma_load_2d_pair(ring_sfb + stage * Cf::kStageSfb + 1024, &tmSfb, fb, 0,
                             (tn * 2 + 1) * plan.iters + k);
          } else {
            constexpr int TK = Cf::kTileK, AT = Cf::kAtom, BX = Cf::kBoxBytes;
            if constexpr (kAT) {   // M-major A: AT-wide boxes of TK k-rows
#pragma unroll
              for (int j = 0; j < 128 / AT; ++j)
                tma_load_2d_pair(sa + j * BX, &tmA, fb, row0 + j * AT, k * TK);
            } else {
              tma_load_2d_pair(sa, &tmA, fb, k * TK, row0);
            }
            if constexpr (kBT) {   // K-major B: this CTA's 128 columns as rows of TK k
              tma_load_2d_pair(sb, &tmB, fb, k * TK, col0);
            } else {
#pragma unroll
              for (int j = 0; j < Cf::kHalfN / AT; ++j)
                tma_load_2d_pair(sb + j * BX, &tmB, fb, col0 + j * AT, k * TK);
            }
          }
          ++issued;
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      if (!ok && leader) {
        const int64_t outstanding = issued < S ? issued : S;
        for (int64_t i = 1; i <= outstanding; ++i) {
          const int s = static_cast<int>((stage - i + S) % S);
          const uint32_t par = (s < stage) ? phase : (phase ^ 1u);
          if (!wait_bar_drain(&full[s], par, 100000000ull)) record_error(args, kSiteDrain, -1);
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------------ MMA issuer (leader)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      Cursor cur(plan, pair);
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
          // MXFP4: the scales-ready barrier also implies the stage's data has landed.
          if (!wait_bar(kMx ? &sf_ready[stage] : &full[stage], phase, abort_flag, args,
                        kSiteMma)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = smem_addr(ring_a + stage * Cf::kStageA);
          const uint32_t b0 = smem_addr(ring_b + stage * Cf::kStageB);
          if constexpr (kMx) {
            const uint32_t sf_base = tmem_base + Cf::kAccBufs * Cf::kAccCols;
            const uint32_t sfa_t = sf_base + stage * Cf::kSfaCols;
            const uint32_t sfb_t = sf_base + S * Cf::kSfaCols + stage * Cf::kSfbCols;
#pragma unroll
            for (int j = 0; j < Cf::kMmasPerStage; ++j) {
              const uint32_t g = j >> 1;
              const uint32_t sf_id = (j & 1) * 2;
              const uint32_t idesc = Cf::kIdesc | (sf_id << 29) | (sf_id << 4);
              const uint64_t ad = smem_desc(a0 + j * 32, 16, 1024, kLayoutSwizzle128B);
              const uint64_t bd = smem_desc(b0 + j * 32, 16, 1024, kLayoutSwizzle128B);
              mma_mxf4_pair(d_tmem, ad, bd, idesc, sfa_t + g * 4, sfb_t + g * 8,
                            (i > 0 || j > 0) ? 1u : 0u);
            }
          } else {
#pragma unroll
            for (int j = 0; j < Cf::kMmasPerStage; ++j) {
              constexpr uint32_t BX = Cf::kBoxBytes, ADV = Cf::kMnAdvance;
              const uint64_t ad = kAT ? smem_desc(a0 + j * ADV, BX, 1024, kLayoutSwizzle128B)
                                      : smem_desc(a0 + j * 32, 16, 1024, kLayoutSwizzle128B);
              const uint64_t bd = kBT ? smem_desc(b0 + j * 32, 16, 1024, kLayoutSwizzle128B)
                                      : smem_desc(b0 + j * ADV, BX, 1024, kLayoutSwizzle128B);
              if constexpr (kF8) {
                mma_f8_pair(d_tmem, ad, bd, Cf::kIdesc, (i > 0 || j > 0) ? 1u : 0u);
              } else {
                mma_f16_pair(d_tmem, ad, bd, Cf::kIdesc, (i > 0 || j > 0) ? 1u : 0u);
              }
            }
          }
          mma_commit_pair(&empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        mma_commit_pair(&tfull[acc]);
        if (++acc == Cf::kAccBufs) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      mma_commit_pair_local(mma_done);
      if (!wait_bar_drain(mma_done, 0, 100000000ull)) record_error(args, kSiteDrain, -1);
    }
  } else if (warp == 10) {
    // ------------------------------------------------------------------ scale copies (MXFP4)
    if constexpr (kMx) {
      if (leader && lane == 0) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        Cursor cur(plan, pair);
        Unit u;
        while (ok && cur.next(plan, u)) {
          for (int32_t i = 0; i < u.k1 - u.k0; ++i) {
          const int32_t k = unit_k(u, i);
            if (!wait_bar(&full[stage], phase, abort_flag, args, kSiteMma)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t sf_base = tmem_base + Cf::kAccBufs * Cf::kAccCols;
            const uint32_t sfa_t = sf_base + stage * Cf::kSfaCols;
            const uint32_t sfb_t = sf_base + S * Cf::kSfaCols + stage * Cf::kSfbCols;
            const uint32_t sfa_s = smem_addr(ring_sfa + stage * Cf::kStageSfa);
            const uint32_t sfb_s = smem_addr(ring_sfb + stage * Cf::kStageSfb);
#pragma unroll
            for (int g = 0; g < 2; ++g)
              tmem_copy_32x128b_x4_pair(sfa_t + g * 4,
                                        smem_desc(sfa_s + g * 512, 0, 128, kLayoutSwizzleNone));
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
              for (int g = 0; g < 2; ++g)
                tmem_copy_32x128b_x4_pair(
                    sfb_t + g * 8 + j * 4,
                    smem_desc(sfb_s + j * 1024 + g * 512, 0, 128, kLayoutSwizzleNone));
            mma_commit_pair_local(&sf_ready[stage]);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        mma_commit_pair_local(cp_done);
        if (!wait_bar_drain(cp_done, 0, 100000000ull)) record_error(args, kSiteDrain, -1);
      }
    }
  } else {
    // ------------------------------------------------------------------ epilogue
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;            // which 128 accumulator columns
    const int row = quarter * 32 + lane;         // tile row within this CTA's 128
    const int et = threadIdx.x - 64;             // 0..255
    const uint32_t tempty_leader0 = cluster_addr(&tempty[0], 0);
    int acc = 0;
    uint32_t acc_phase = 0;
    int parity = 0;
    // this warp's staging: two 2 KB buffers (bf16 / fp8), one 1 KB buffer (MXFP4)
    uint8_t* my_stage = epi_stage + (warp - 2) * (Cf::kEpiBytes / 8);
    int sbuf = 0;
    Cursor cur(plan, pair);
    Unit u;
    while (cur.next(plan, u)) {
      // where this piece's rows and columns lie (worked out before the waits below)
      int32_t tm, tn;
      tile_coords(plan, u.tile, tm, tn);
      const int64_t y_warp = static_cast<int64_t>(tm) * 256 + rank * 128 + quarter * 32;
      const int64_t m = y_warp + lane;
      const int64_t n_half = static_cast<int64_t>(tn) * kBN + half * 128;
      float bias_l[4];   // read here, or after the staging below (whose registers it would take)
      bool has_next;
      {
        Cursor peek = cur;
        Unit later;
        has_next = peek.next(plan, later);
      }
      // The tile's contributors, and which CTAs finish its columns.  Columns go in 32-column
      // chunks, chunk j = 4 * half + ch to party j % parties; the owner is party 0.  Mostly the
      // owner finishes the whole tile (parties = 1).  In the bf16 and fp8 pairs, when the
      // owner's shared tile is its last piece and at least two contributors hold nothing else
      // (finishers: contributor i is party i + 1), the finishers finish a share of the chunks
      // each: they reach the end of their ranges with the owner, and sharing the tile spreads the
      // partials' reads and the stores of C over all of them instead of queueing them on the
      // owner.  With one finisher the owner keeps the tile: handing out half of it costs the
      // owner about what the drain it saves does.
      int n_contrib = 0;
      int parties = 1;
      int party = 0;
      int64_t owner = pair;
      if (u.role == kRoleOwner) {
        const TileShare s = tile_contributors(plan, pair, u.k1);
        n_contrib = s.n_contrib;
        if (kShare && !args.replay && pair >= plan.whole_tiles && s.finishers >= 2)
          parties = 1 + s.finishers;
      } else if (kShare && !args.replay && u.role == kRoleContrib) {
        const int64_t first = (u.tile - plan.whole_tiles) * plan.iters;   // the tile's k = 0
        const int64_t o = sk_range_cta(plan, first);
        if (sk_range_begin(plan, pair) + sk_range_len(plan, pair) <= first + plan.iters &&
            o >= plan.whole_tiles) {
          const TileShare s =
              tile_contributors(plan, o, sk_range_begin(plan, o) + sk_range_len(plan, o) - first);
          if (s.finishers >= 2) {
            owner = o;
            n_contrib = s.n_contrib;
            parties = 1 + s.finishers;
            party = static_cast<int>(pair - o);
          }
        }
      }
      const bool shared_finish = parties > 1;
      // The shared tile an owner finishes with: no later piece waits for its accumulator, so it
      // is drained from tensor memory 32 columns at a time with the partials added (below).
      // With two accumulators, partials that are complete while its k-loop still runs are
      // summed into the idle one meanwhile (it held the previous piece, already drained; no
      // later piece uses it), so the fix-up after the loop reads tensor memory.
      const bool last_shared = u.role == kRoleOwner && !has_next && n_contrib > 0;
      // (An owner that shares its tile's finish does not stage: it needs only its own chunks of
      // each partial, and its share, which the finishers wait for, goes out first.)
      const bool staged = Cf::kAccBufs == 2 && last_shared && !shared_finish;
      if (!staged) load_bias_lanes(args, n_half, lane, bias_l);
      uint32_t flag_status = kUnitStore;
      int n_staged = 0;   // contributors summed into the idle accumulator (the farthest ones)
      if (staged) {
        // The farthest contributor first (it is long done; the nearest may still be on this
        // tile), each partial added as soon as its flag is seen, for as long as the k-loop
        // runs; the rest are read by the drain.  The status word alternates between two slots
        // so thread 0 never overwrites one not yet read.
        const uint32_t t_stage = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 static_cast<uint32_t>(acc ^ 1) * Cf::kAccCols + half * 128;
#pragma unroll 1
        for (int i = 0; i < n_contrib; ++i) {
          const int c = n_contrib - 1 - i;
          if (et == 0) {
            const uint32_t r =
                poll_flag_or_full(args.flags + 2 * (pair + 1 + c) + rank, args.epoch, &tfull[acc],
                                  acc_phase, abort_flag, args.timeout_ns, args.replay != 0);
            if (r == kPollTimeout) record_error(args, kSiteFlag, u.tile);
            staged_status[i & 1] = r;
          }
          named_barrier_sync(1, kPairEpilogueThreads);
          const uint32_t r = staged_status[i & 1];
          if (r == kPollLoopDone) break;
          if (r == kPollTimeout) {
            flag_status = kUnitSkip;
            break;
          }
          stage_partial<4, 2>(reinterpret_cast<const float4*>(args.P + (2 * (pair + 1 + c) + rank) * (kBM * kBN)) +
                               static_cast<int64_t>(half * 4) * 8 * kBM + row,
                           t_stage, i == 0);
          n_staged = i + 1;
        }
      }
      if (staged) load_bias_lanes(args, n_half, lane, bias_l);
      // contributors 0 .. n_rem-1 (the nearest) are read by the drain
      const int n_rem = flag_status == kUnitStore ? n_contrib - n_staged : 0;
      if (et < 32) {
        // Lane 0 of the first epilogue warp waits for the accumulator; an owner finishing its
        // tile alone then waits for its remaining contributors' flags, lane l for contributors
        // l, l + 32, ... side by side.
        uint32_t status = kUnitStore;
        if (et == 0 && !wait_bar(&tfull[acc], acc_phase, abort_flag, args, kSiteEpilogue))
          status = kUnitAbort;
        status = __shfl_sync(0xffffffffu, status, 0);
        if (status == kUnitStore && u.role == kRoleOwner && !shared_finish) {
          bool ok = true;
          for (int c = et; c < n_rem && ok; c += 32) {
            uint32_t* f = args.flags + 2 * (pair + 1 + c) + rank;
            ok = wait_flag(f, args.epoch, args.timeout_ns);
            // A captured launch keeps its epoch across replays, so its one reader clears the
            // flag; otherwise every launch has a new epoch and the flag may stay set.
            if (ok && args.replay) *reinterpret_cast<volatile uint32_t*>(f) = 0u;
          }
          if (!__all_sync(0xffffffffu, ok)) {
            if (et == 0) record_error(args, kSiteFlag, u.tile);
            status = kUnitSkip;
          }
        }
        if (et == 0) unit_status[parity] = status;
      }
      named_barrier_sync(1, kPairEpilogueThreads);
      const uint32_t status = unit_status[parity];
      if (status == kUnitAbort) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                             static_cast<uint32_t>(acc) * Cf::kAccCols + half * 128;

      if (shared_finish) {
        // 1. Hand out: the owner writes the other parties' chunks of its own accumulator (not
        //    the partials staged beside it) to its second slot, 2 * grid + cta; a finisher
        //    writes every chunk but its own to its slot, as any contributor does.  Then the flag.
        const bool is_owner = u.role == kRoleOwner;
        const int64_t out_slot = is_owner ? 2 * static_cast<int64_t>(plan.grid) + cta : cta;
        {
          float4* out = reinterpret_cast<float4*>(args.P + out_slot * (kBM * kBN)) +
                        static_cast<int64_t>(half * 4) * 8 * kBM + row;
          const uint64_t policy = l2_policy_evict_last();
#pragma unroll 1
          for (int ch = 0; ch < 4; ++ch) {
            if ((4 * half + ch) % parties == party) continue;
            uint32_t r[32];
            __syncwarp();
            tmem_load_32cols(t_row + ch * 32, r);
            tmem_load_wait();
            float4* dst = out + static_cast<int64_t>(ch) * 8 * kBM;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_cg_policy(dst + q * kBM,
                           make_float4(__uint_as_float(r[4 * q]), __uint_as_float(r[4 * q + 1]),
                                       __uint_as_float(r[4 * q + 2]), __uint_as_float(r[4 * q + 3])),
                           policy);
          }
        }
        // 2. Wait for the other parties' partials of this CTA's chunks: for the owner, the
        //    contributors not staged; for a finisher, the owner's second slot and every other
        //    contributor.  (unit_status[parity ^ 1] is free: every thread read it before the
        //    barrier above, and no piece follows this one.)
        // (With more than 8 parties, those past the eighth finish no chunk and wait for nothing.)
        const int n_src = party >= kBN / 32 ? 0 : (is_owner ? n_rem : n_contrib);
        // Source s of this thread's row: s = 0 is `first` (the owner's second slot for a
        // finisher, the nearest contributor for the owner); s >= 1 the next contributors, from
        // `rest` on, one slot pair apart, skipping this CTA's own.
        constexpr int64_t kSlot = kBM * kBN / 4;   // float4s per slot
        const int64_t c0 = 2 * (owner + 1) + rank;  // slot of the tile's first contributor
        const float4* first =
            reinterpret_cast<const float4*>(args.P) + static_cast<int64_t>(half * 4) * 8 * kBM + row +
            (is_owner ? c0 : 2 * static_cast<int64_t>(plan.grid) + 2 * owner + rank) * kSlot;
        const float4* rest = reinterpret_cast<const float4*>(args.P) +
                             static_cast<int64_t>(half * 4) * 8 * kBM + row +
                             (is_owner ? c0 + 2 : c0) * kSlot;
        const int skip = is_owner ? 1 << 30 : party - 1;
        __threadfence();
        named_barrier_sync(1, kPairEpilogueThreads);
        if (et < 32) {
          // The first epilogue warp: lane 0 releases this CTA's flag, then lane l waits for
          // sources l, l + 32, ..., so the flags are polled side by side rather than one
          // round trip to L2 after another.
          if (et == 0 && !(args.inject_drop && cta == args.drop_cta))
            flag_release(args.flags + out_slot, args.epoch);
          bool ok = true;
          for (int s = et; s < n_src && ok; s += 32) {
            const int64_t slot =
                s == 0 ? (is_owner ? c0 : 2 * static_cast<int64_t>(plan.grid) + 2 * owner + rank)
                       : (is_owner ? c0 + 2 * s : c0 + 2 * (s - 1 < skip ? s - 1 : s));
            ok = wait_flag(args.flags + slot, args.epoch, args.timeout_ns);
          }
          ok = __all_sync(0xffffffffu, ok);
          if (et == 0) {
            if (!ok) record_error(args, kSiteFlag, u.tile);
            unit_status[parity ^ 1] = ok ? kUnitStore : kUnitSkip;
          }
        }
        named_barrier_sync(1, kPairEpilogueThreads);
        const bool store = unit_status[parity ^ 1] == kUnitStore && flag_status == kUnitStore;
        // 3. Finish this CTA's chunks: its accumulator (+ the staged partials, owner) + the
        //    partials read here + bias, cast and stored.
        //    The first source of the next chunk is requested before this one is stored (one
        //    more would not fit in the registers).
        const uint32_t t_stage = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 static_cast<uint32_t>(acc ^ 1) * Cf::kAccCols + half * 128;
        auto mine = [&](int c) { return (4 * half + c) % parties == party; };
        auto src = [&](int s, int c) {
          const float4* b = s == 0 ? first : rest + (s - 1 < skip ? s - 1 : s) * 2 * kSlot;
          return b + static_cast<int64_t>(c) * 8 * kBM;
        };
        int ch = 0;
        while (ch < 4 && !mine(ch)) ++ch;
        float4 pp[8];
        if (store && ch < 4 && n_src > 0) load_partial8(pp, src(0, ch), kBM);
#pragma unroll 1
        while (ch < 4) {
          int next = ch + 1;
          while (next < 4 && !mine(next)) ++next;
          uint32_t own[32];
          float w[32];
          __syncwarp();
          tmem_load_32cols(t_row + ch * 32, own);
          if (is_owner && n_staged > 0) {
            uint32_t part[32];
            tmem_load_32cols(t_stage + ch * 32, part);
            tmem_load_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = __uint_as_float(own[j]) + __uint_as_float(part[j]);
          } else {
            tmem_load_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = __uint_as_float(own[j]);
          }
          if (store) {
            if (n_src > 0) add_partial8(w, pp, false);
#pragma unroll 1
            for (int s = 1; s < n_src; s += 2) {
              float4 pq[8];
              load_partial8(pp, src(s, ch), kBM);
              if (s + 1 < n_src) load_partial8(pq, src(s + 1, ch), kBM);
              add_partial8(w, pp, false);
              if (s + 1 < n_src) add_partial8(w, pq, false);
            }
            if (next < 4 && n_src > 0) load_partial8(pp, src(0, next), kBM);
            add_bias_lanes(args, w, pick_chunk(bias_l, ch));
            if constexpr (Cf::kTmaStore) {
              store_chunk_tma<false>(args, &tmC, my_stage, sbuf, lane, n_half + ch * 32, y_warp, w);
            } else if (args.c_tma) {
              store_chunk_tma_1k<false>(args, &tmC, my_stage, lane, n_half + ch * 32, y_warp, w);
            } else {
              store_row_chunk<false>(args, m, n_half + ch * 32, w);
            }
          }
          ch = next;
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) remote_arrive(tempty_leader0 + acc * 8);
        break;   // the last piece
      }

      if (last_shared) {
        // Last piece: no later piece waits for this accumulator, so add and store it 32
        // columns at a time, then release it as usual.  The partials not summed during the
        // k-loop are read here.
        const bool store = status == kUnitStore && flag_status == kUnitStore;
        const uint32_t t_stage = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16) +
                                 static_cast<uint32_t>(acc ^ 1) * Cf::kAccCols + half * 128;
        const float4* rem0 =
            reinterpret_cast<const float4*>(args.P + (2 * (pair + 1) + rank) * (kBM * kBN)) +
            static_cast<int64_t>(half * 4) * 8 * kBM + row;
        constexpr int64_t kSlot4 = 2 * (kBM * kBN / 4);   // float4s between consecutive pairs' slots
        // Two contributors' chunks are in flight at a time, and the next chunk's are requested
        // before this chunk is stored, so the round trips to L2 overlap the drain's other work.
        float4 pp[8], pq[8];
        if (store && n_rem > 0) load_partial8(pp, rem0, kBM);
        if (store && n_rem > 1) load_partial8(pq, rem0 + kSlot4, kBM);
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          const float4* rem = rem0 + static_cast<int64_t>(ch) * 8 * kBM;
          uint32_t own[32];
          __syncwarp();
          tmem_load_32cols(t_row + ch * 32, own);
          float w[32];
          if (n_staged > 0) {
            uint32_t part[32];
            tmem_load_32cols(t_stage + ch * 32, part);
            tmem_load_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = __uint_as_float(own[j]) + __uint_as_float(part[j]);
          } else {
            tmem_load_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) w[j] = __uint_as_float(own[j]);
          }
          if (store && n_rem > 0) {
            add_partial8(w, pp, false);
            if (n_rem > 1) add_partial8(w, pq, false);
#pragma unroll 1
            for (int c = 2; c < n_rem; c += 2) {
              load_partial8(pp, rem + c * kSlot4, kBM);
              if (c + 1 < n_rem) load_partial8(pq, rem + (c + 1) * kSlot4, kBM);
              add_partial8(w, pp, false);
              if (c + 1 < n_rem) add_partial8(w, pq, false);
            }
            if (ch + 1 < 4) {
              load_partial8(pp, rem + 8 * kBM, kBM);
              if (n_rem > 1) load_partial8(pq, rem + 8 * kBM + kSlot4, kBM);
            }
          }
          if (store) {
            // bf16 and fp8 pairs always have 16-byte aligned rows of C (N is a multiple of 8);
            // MXFP4 ones when N allows
            add_bias_lanes(args, w, pick_chunk(bias_l, ch));
            if constexpr (Cf::kTmaStore) {
              store_chunk_tma<false>(args, &tmC, my_stage, sbuf, lane, n_half + ch * 32, y_warp, w);
            } else if (args.c_tma) {
              store_chunk_tma_1k<false>(args, &tmC, my_stage, lane, n_half + ch * 32, y_warp, w);
            } else {
              store_row_chunk<false>(args, m, n_half + ch * 32, w);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) remote_arrive(tempty_leader0 + acc * 8);
        break;   // the last piece
      }

      if constexpr (Cf::kAccBufs == 2) {
        // Two accumulators: the MMA works on the other one meanwhile, so this one is drained
        // and stored 32 columns at a time and handed back at the end.
        float4* my_slot = reinterpret_cast<float4*>(args.P + cta * (kBM * kBN)) +
                          static_cast<int64_t>(half * 4) * 8 * kBM + row;
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t r[32];
          __syncwarp();
          tmem_load_32cols(t_row + ch * 32, r);
          tmem_load_wait();
          float w[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) w[j] = __uint_as_float(r[j]);
          if (u.role == kRoleContrib) {
            float4* dst = my_slot + static_cast<int64_t>(ch) * 8 * kBM;
            const uint64_t policy = l2_policy_evict_last();
#pragma unroll
            for (int q = 0; q < 8; ++q)
              st_cg_policy(dst + q * kBM, make_float4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]),
                           policy);
          } else if (status == kUnitStore) {
            for (int c = 0; c < n_contrib; ++c) {
              const float4* src =
                  reinterpret_cast<const float4*>(args.P + (2 * (pair + 1 + c) + rank) * (kBM * kBN)) +
                  static_cast<int64_t>(half * 4 + ch) * 8 * kBM + row;
              float4 pp[8];
              load_partial8(pp, src, kBM);
              add_partial8(w, pp, false);
            }
            // bf16 and fp8 pairs always have 16-byte aligned rows of C (N is a multiple of 8);
            // MXFP4 ones when N allows
            add_bias_lanes(args, w, pick_chunk(bias_l, ch));
            if constexpr (Cf::kTmaStore) {
              store_chunk_tma<false>(args, &tmC, my_stage, sbuf, lane, n_half + ch * 32, y_warp, w);
            } else if (args.c_tma) {
              store_chunk_tma_1k<false>(args, &tmC, my_stage, lane, n_half + ch * 32, y_warp, w);
            } else {
              store_row_chunk<false>(args, m, n_half + ch * 32, w);
            }
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) remote_arrive(tempty_leader0 + acc * 8);
        if (u.role == kRoleContrib) {
          __threadfence();
          named_barrier_sync(1, kPairEpilogueThreads);
          if (et == 0 && !(args.inject_drop && cta == args.drop_cta))
            flag_release(args.flags + cta, args.epoch);
        }
      } else {
        // Drain this thread's 128 columns, then hand the accumulator back.
        float v[128];
        __syncwarp();
        tmem_load_64cols(t_row, reinterpret_cast<uint32_t*>(v));
        tmem_load_64cols(t_row + 64, reinterpret_cast<uint32_t*>(v) + 64);
        tmem_load_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) remote_arrive(tempty_leader0 + acc * 8);

        if (u.role == kRoleContrib) {
          float4* dst = reinterpret_cast<float4*>(args.P + cta * (kBM * kBN)) +
                        static_cast<int64_t>(half * 4) * 8 * kBM + row;
          const uint64_t policy = l2_policy_evict_last();
  #pragma unroll
          for (int q = 0; q < 32; ++q)
            st_cg_policy(dst + q * kBM, make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]),
                         policy);
          __threadfence();
          named_barrier_sync(1, kPairEpilogueThreads);
          if (et == 0 && !(args.inject_drop && cta == args.drop_cta))
            flag_release(args.flags + cta, args.epoch);
        } else if (status == kUnitStore) {
          const uint64_t policy = l2_policy_evict_first();
          for (int c = 0; c < n_contrib; ++c) {
            const float4* src =
                reinterpret_cast<const float4*>(args.P + (2 * (pair + 1 + c) + rank) * (kBM * kBN)) +
                static_cast<int64_t>(half * 4) * 8 * kBM + row;
  #pragma unroll
            for (int ch = 0; ch < 4; ++ch) {
              float4 p[8];
  #pragma unroll
              for (int q = 0; q < 8; ++q) p[q] = ld_cg_policy(src + (ch * 8 + q) * kBM, policy);
  #pragma unroll
              for (int q = 0; q < 8; ++q) {
                v[ch * 32 + 4 * q] += p[q].x;
                v[ch * 32 + 4 * q + 1] += p[q].y;
                v[ch * 32 + 4 * q + 2] += p[q].z;
                v[ch * 32 + 4 * q + 3] += p[q].w;
              }
              asm volatile("" ::: "memory");   // keep the chunks' loads apart (register pressure)
            }
          }
  #pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            float(&w)[32] = *reinterpret_cast<float(*)[32]>(&v[ch * 32]);
            // bf16 and fp8 pairs always have 16-byte aligned rows of C (N is a multiple of 8);
            // MXFP4 ones when N allows
            add_bias_lanes(args, w, pick_chunk(bias_l, ch));
            if constexpr (Cf::kTmaStore) {
              store_chunk_tma<false>(args, &tmC, my_stage, sbuf, lane, n_half + ch * 32, y_warp, w);
            } else if (args.c_tma) {
              store_chunk_tma_1k<false>(args, &tmC, my_stage, lane, n_half + ch * 32, y_warp, w);
            } else {
              store_row_chunk<false>(args, m, n_half + ch * 32, w);
            }
          }
        }
      }
      parity ^= 1;
      if (++acc == Cf::kAccBufs) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (Cf::kTmaStore || args.c_tma) {
      if (lane == 0) bulk_wait_all();   // staged pieces are read and written before exit
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();   // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, Cf::kTmemCols);
  }
}

}  // namespace sk
