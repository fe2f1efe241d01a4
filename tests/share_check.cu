// Host-only check program for the Stream-K range bookkeeping the SM-pair kernels use to share a
// split tile's fix-up (sk_range_cta, tile_contributors in sk_schedule.cuh).  Compiled by
// tests/test_share_check.py with nvcc; no device code runs.
//
// stdin: lines "tiles_m tiles_n iters grid whole_tiles sk_base sk_extra".
// stdout, per plan, one line per split tile of the Stream-K region (region index t):
//   "t owner n_contrib finishers"
// where owner = sk_range_cta(plan, t * iters) and (n_contrib, finishers) =
// tile_contributors(plan, owner, owned) with owned = the owner's iterations in the tile, then
// a line "end".
#include <cstdio>

#include "sk_schedule.cuh"

int main() {
  long long tm, tn, it, g, whole, base, extra;
  while (std::scanf("%lld %lld %lld %lld %lld %lld %lld", &tm, &tn, &it, &g, &whole, &base,
                    &extra) == 7) {
    sk::Plan p = {};
    p.tiles_m = static_cast<int32_t>(tm);
    p.tiles_n = static_cast<int32_t>(tn);
    p.iters = static_cast<int32_t>(it);
    p.grid = static_cast<int32_t>(g);
    p.group_m = 1;
    p.tiles = tm * tn;
    p.whole_tiles = whole;
    p.sk_base = base;
    p.sk_extra = extra;
    const int64_t sk_tiles = p.tiles - p.whole_tiles;
    for (int64_t t = 0; t < sk_tiles; ++t) {
      const int64_t first = t * p.iters;
      const int64_t owner = sk::sk_range_cta(p, first);
      const int64_t owned = sk::sk_range_begin(p, owner) + sk::sk_range_len(p, owner) - first;
      if (owned >= p.iters) continue;   // the owner holds the whole tile
      const sk::TileShare s = sk::tile_contributors(p, owner, owned);
      std::printf("%lld %lld %d %d\n", static_cast<long long>(t), static_cast<long long>(owner),
                  s.n_contrib, s.finishers);
    }
    std::printf("end\n");
  }
  return 0;
}
