// Tile scheduler shared by the host planner and the kernels (__host__ __device__).
//
// A plan fixes, for a problem of tiles_m x tiles_n output tiles with `iters` k-iterations
// each and a grid of g CTAs, which (tile, k-range) pieces every CTA runs and in which order:
//   * linear tiles [0, whole_tiles) run whole, CTA c taking c, c+g, c+2g, ... (this covers the
//     data-parallel schedule, where g = tiles, and the SM-constrained persistent schedule of
//     flashinfer PR #982 "SM-constraint-GEMM by triton persistent kernel");
//   * linear tiles [whole_tiles, tiles) form the Stream-K region: its tiles x iters
//     iterations, in tile-major order, are cut into g contiguous ranges, CTA c's range holding
//     sk_base iterations plus one if c < sk_extra.
// A piece holding k = 0 makes its CTA the tile's owner; a piece starting past k = 0 is a
// partial that the owner adds in before the bias (tritonBLAS PR #67 "Fix StreamK Kernel
// Bias", Technical Details).  Because ranges are contiguous, only the start of a range can lie
// inside a tile, so a CTA spills at most once (one scratch slot per CTA, as in tritonBLAS PR
// #74 "Stream-k mxfp4 kernel"), and the tile a CTA owns but shares is the one its range ends
// in, continued by CTAs c+1, c+2, ...  The order in which a CTA runs its pieces is given by
// Cursor below.  (The SM-pair kernels may split the owner's fix-up of a tile among the owner
// and contributors that have no other piece; see tile_contributors.)
//
// Linear tile index -> (tile row, tile column) goes through two bijections:
//  1. In the Stream-K region, the tau-th tile owned by CTA c is given raster position
//     whole_tiles + tau * g + c (the CTAs holding one more tile than the others come last, in
//     CTA order).  CTAs advance through their owned tiles in step, so the tiles they work on at
//     the same time take consecutive raster positions -- one compact block, as in a wave of the
//     persistent schedule -- instead of being spread over the whole matrix.  The whole-tile
//     region keeps its linear order.
//  2. A grouped raster: groups of `group_m` tile rows, column-major inside a group, so tiles
//     at consecutive raster positions share A and B panels in L2.
// Both only decide which output tile a piece works on; every tile is still summed over k in
// ascending order.
#pragma once

#include <cstdint>

namespace sk {

enum : int32_t { kRoleFull = 0, kRoleOwner = 1, kRoleContrib = 2 };

struct Plan {
  int32_t tiles_m, tiles_n;
  int32_t iters;        // k-iterations per tile
  int32_t grid;         // CTAs launched
  int32_t group_m;      // raster group height in tiles
  int32_t pad_;
  int64_t tiles;        // tiles_m * tiles_n
  int64_t whole_tiles;  // linear tiles [0, whole_tiles) run whole
  int64_t sk_base;      // Stream-K iterations per CTA
  int64_t sk_extra;     // CTAs [0, sk_extra) take one more
};

struct Unit {
  int64_t tile;   // linear tile index
  int32_t k0, k1; // k-iteration range [k0, k1)
  int32_t role;
};

// a / b and a % b for the values of a plan, all non-negative and below 2^31 (the planner refuses
// larger Stream-K regions, and tiles are fewer).  On the GPU a 64-bit division is a long
// software sequence; the 32-bit one is several times cheaper, which matters for the set-up of
// every piece (a piece's first loads wait for it).
__host__ __device__ __forceinline__ int64_t sk_div(int64_t a, int64_t b) {
#ifdef __CUDA_ARCH__
  return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
#else
  return a / b;
#endif
}

__host__ __device__ __forceinline__ int64_t sk_mod(int64_t a, int64_t b) {
#ifdef __CUDA_ARCH__
  return static_cast<int64_t>(static_cast<uint32_t>(a) % static_cast<uint32_t>(b));
#else
  return a % b;
#endif
}

__host__ __device__ __forceinline__ int64_t sk_range_begin(const Plan& p, int64_t cta) {
  return cta * p.sk_base + (cta < p.sk_extra ? cta : p.sk_extra);
}

__host__ __device__ __forceinline__ int64_t sk_range_len(const Plan& p, int64_t cta) {
  return p.sk_base + (cta < p.sk_extra ? 1 : 0);
}

// The CTA whose range holds Stream-K region iteration x.
__host__ __device__ __forceinline__ int64_t sk_range_cta(const Plan& p, int64_t x) {
  const int64_t long_span = p.sk_extra * (p.sk_base + 1);  // iterations of the longer ranges
  if (x < long_span) return sk_div(x, p.sk_base + 1);
  return p.sk_base > 0 ? p.sk_extra + sk_div(x - long_span, p.sk_base) : p.sk_extra;
}

// The CTAs that continue the shared tile CTA `owner` owns, whose own piece is the tile's first
// `owned` k-iterations: CTAs owner+1, owner+2, ..., `n_contrib` of them.  The first
// `finishers` of them hold nothing but their piece of this tile: their ranges begin inside it
// and end inside it or at its end.  (Every contributor but the last lies inside the tile; the
// last one is a finisher when its range ends at the tile's end.)
struct TileShare {
  int32_t n_contrib;
  int32_t finishers;
};

__host__ __device__ __forceinline__ TileShare tile_contributors(const Plan& p, int64_t owner,
                                                                int64_t owned) {
  TileShare s = {0, 0};
  int64_t covered = owned;
  for (int64_t c = owner + 1; covered < p.iters; ++c) {
    const int64_t len = sk_range_len(p, c);
    const int64_t room = p.iters - covered;
    if (len <= room) ++s.finishers;
    covered += len < room ? len : room;
    ++s.n_contrib;
  }
  return s;
}

// Walks one CTA's pieces in execution order:
//   1. the Stream-K tiles it owns entirely, in linear order,
//   2. its contribution (the piece of its range that starts inside a tile), spilled to P,
//   3. the tile it owns but shares (the piece of its range that ends inside a tile),
//   4. its tiles of the whole-tile region (c, c+g, ...).
// Contributions never wait, and every CTA reaches its contribution before its own shared
// tile, so an owner's wait is short and there is no cycle.  Step 1 starts every tile at k = 0
// on every CTA at the same time, so CTAs working on neighbouring tiles read the same k-slices
// of A and B together; step 4 after the shared tile lets the owner's fix-up epilogue overlap
// the next tile's main loop.
struct Cursor {
  int64_t begin, end;      // this CTA's Stream-K iterations [begin, end), region-relative
  int64_t full_next, full_end;   // whole owned Stream-K tiles still to run (region tiles)
  int64_t next_whole;      // next tile of the whole-tile region
  int32_t step;            // 0: owned Stream-K tiles, 1: contribution, 2: shared owned
                           // tile, 3: whole-tile region

  __host__ __device__ __forceinline__ Cursor(const Plan& p, int64_t cta) {
    begin = sk_range_begin(p, cta);
    end = begin + sk_range_len(p, cta);
    const int64_t first_full = sk_div(begin + p.iters - 1, p.iters);   // first tile starting in range
    const int64_t last_full = sk_div(end, p.iters);                    // tiles ending in range
    full_next = first_full;
    full_end = last_full > first_full ? last_full : first_full;
    next_whole = cta;
    step = 0;
  }

  __host__ __device__ __forceinline__ bool next(const Plan& p, Unit& u) {
    if (step == 0) {
      if (full_next < full_end) {
        u.tile = p.whole_tiles + full_next;
        u.k0 = 0;
        u.k1 = p.iters;
        u.role = kRoleFull;
        ++full_next;
        return true;
      }
      step = 1;
    }
    if (step == 1) {
      step = 2;
      if (begin < end && sk_mod(begin, p.iters) != 0) {   // starts inside a tile: a contribution
        const int64_t t = sk_div(begin, p.iters);
        const int64_t tile_end = (t + 1) * p.iters;
        u.tile = p.whole_tiles + t;
        u.k0 = static_cast<int32_t>(begin - t * p.iters);
        u.k1 = static_cast<int32_t>((end < tile_end ? end : tile_end) - t * p.iters);
        u.role = kRoleContrib;
        return true;
      }
    }
    if (step == 2) {
      step = 3;
      // ends inside a tile whose k = 0 lies in this range: the shared tile this CTA owns
      const int64_t t = sk_div(end, p.iters);
      if (begin < end && sk_mod(end, p.iters) != 0 && t * p.iters >= begin) {
        u.tile = p.whole_tiles + t;
        u.k0 = 0;
        u.k1 = static_cast<int32_t>(end - t * p.iters);
        u.role = kRoleOwner;
        return true;
      }
    }
    if (next_whole < p.whole_tiles) {
      u.tile = next_whole;
      u.k0 = 0;
      u.k1 = p.iters;
      u.role = kRoleFull;
      next_whole += p.grid;
      return true;
    }
    return false;
  }
};

// The i-th k-iteration a piece runs.  Whole tiles ascend from k = 0; the two split pieces
// (contribution and shared owned tile) descend from their last iteration.  CTAs reach their
// split pieces at different times, and descending keeps them on neighbouring k-slices of A
// and B at the same time: every contribution ends at the tile's last iteration, so they all
// start there, and an owned piece picks up where the CTA's range ends.  Only the order of the
// fp32 additions inside a piece changes.
__host__ __device__ __forceinline__ int32_t unit_k(const Unit& u, int32_t i) {
  return u.role == kRoleFull ? u.k0 + i : u.k1 - 1 - i;
}

// Raster position of a linear tile (bijection 1 above).
__host__ __device__ __forceinline__ int64_t raster_position(const Plan& p, int64_t t) {
  if (t < p.whole_tiles) return t;
  const int64_t local = t - p.whole_tiles;
  const int64_t c = sk_range_cta(p, local * p.iters);      // owner: holds the tile's k = 0
  const int64_t start = sk_range_begin(p, c);
  const int64_t first_owned = sk_div(start + p.iters - 1, p.iters);   // first tile whose k = 0 is c's
  const int64_t tau = local - first_owned;
  const int64_t f = sk_div(p.sk_base, p.iters);   // every CTA owns f or f + 1 tiles
  const int64_t pos = (tau < f) ? tau * p.grid + c : f * p.grid + (first_owned - c * f);
  return p.whole_tiles + pos;
}

__host__ __device__ __forceinline__ void tile_coords(const Plan& p, int64_t t, int32_t& tm,
                                                     int32_t& tn) {
  const int64_t r_pos = raster_position(p, t);
  const int64_t per_group = static_cast<int64_t>(p.group_m) * p.tiles_n;
  const int64_t group = sk_div(r_pos, per_group);
  const int64_t first_m = group * p.group_m;
  const int64_t rows_here =
      (p.tiles_m - first_m < p.group_m) ? (p.tiles_m - first_m) : p.group_m;
  const int64_t r = r_pos - group * per_group;
  tm = static_cast<int32_t>(first_m + sk_mod(r, rows_here));
  tn = static_cast<int32_t>(sk_div(r, rows_here));
}

}  // namespace sk
