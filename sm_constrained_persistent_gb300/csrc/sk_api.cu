// C-ABI layer: argument checks, schedule planning, per-(device, stream) workspaces, TMA
// descriptor encoding and kernel launches.  Declared in include/sk_gemm.h.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "sk_gemm.h"
#include "sk_launch.h"
#include "sk_schedule.cuh"

namespace {

constexpr int kTileM = 128;
constexpr int kBf16TileK = 64;
constexpr int64_t kTallMaxRows = 64;   // rows of A a tall-stage tile loads
constexpr int kMxTileK = 256;
constexpr int kF8TileK = 128;
constexpr int kDefaultRasterGroup = 16;
constexpr int64_t kDefaultTimeoutNs = 2000000000LL;   // 2 s
constexpr int64_t kMaxDim = (int64_t(1) << 31) - 1;

// ---------------------------------------------------------------------------------------
// planning (pure host arithmetic)
// ---------------------------------------------------------------------------------------

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

sk_status_t auto_plan(int format, int64_t M, int64_t N, int64_t K, int num_sms, int sm_count,
                      int max_pairs, const sk_options_t* opt, sk_plan_t* p, int layout);

// max_pairs: how many 2-CTA clusters the device can hold at once (the planner's caller passes
// sm_count / 2 when it cannot ask the device).  layout: the bf16 operand layout (bit 0 A stored
// transposed, bit 1 B stored transposed); 96-wide tiles exist for the plain layout only.
sk_status_t make_plan(int format, int64_t M, int64_t N, int64_t K, int num_sms, int mode,
                      int sm_count, int max_pairs, const sk_options_t* opt, sk_plan_t* p,
                      int layout = 0) {
  if (mode == SK_MODE_AUTO && p != nullptr)
    return auto_plan(format, M, N, K, num_sms, sm_count, max_pairs, opt, p, layout);
  if (p == nullptr || format < 0 || format > 2 || mode < 0 || mode > 3 || sm_count < 1)
    return SK_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return SK_ERR_INVALID_ARG;
  int tile_n = opt ? opt->tile_n : 0;
  int tile_m = opt ? opt->tile_m : 0;
  if (tile_n != 0 && tile_n != 96 && tile_n != 128 && tile_n != 256) return SK_ERR_INVALID_ARG;
  if (tile_m != 0 && tile_m != 128 && tile_m != 256) return SK_ERR_INVALID_ARG;
  if (tile_m == 256 && (tile_n == 128 || tile_n == 96)) return SK_ERR_INVALID_ARG;
  if (tile_n == 96 && format != 0) return SK_ERR_INVALID_ARG;   // 96-wide tiles: bf16 only
  if (format == 1 && tile_m != 256 && tile_n == 256) return SK_ERR_INVALID_ARG;
  const int64_t sms = (num_sms <= 0 || num_sms > sm_count) ? sm_count : num_sms;
  const int64_t pairs_avail = std::min<int64_t>(sms / 2, max_pairs);
  const int64_t pair_tiles = ceil_div(M, 256) * ceil_div(N, 256);
  bool pair;
  if (tile_m == 256) {
    if (pairs_avail < 1) return SK_ERR_INVALID_ARG;
    pair = true;
  } else if (tile_m == 128 || tile_n == 128 || tile_n == 96) {
    pair = false;
  } else {
    // SM pairs halve the operand bytes per FLOP; use them when the tile still has more than
    // 128 real rows, there are at least two tiles, and at least two pairs to run them.
    pair = M > 128 && pair_tiles >= 2 && pairs_avail >= 2;
  }
  if (pair) {
    tile_m = 256;
    tile_n = 256;
  } else {
    tile_m = kTileM;
    if (tile_n == 0) {
      if (format == 1) {
        tile_n = 128;
      } else {
        // Wide tiles halve the B traffic per FLOP; use them while they still fill every SM.
        const int64_t wide_tiles = ceil_div(M, kTileM) * ceil_div(N, 256);
        tile_n = (N >= 256 && wide_tiles >= sm_count) ? 256 : 128;
        // One row of tiles (M <= 128) streams B: 96-wide tiles put more SMs on it, but each SM
        // streams a 96-wide tile's columns ~24 % slower (64-byte rows).  Take them when they need
        // no more waves than 128-wide tiles, so the extra tiles only add SMs: 64 x 14336 on 152
        // SMs runs 150 tiles in one wave instead of 112 (31.0 vs 33.1 us); on 32 SMs, 5 waves of
        // 96-wide tiles took 96 us against 78 us for 4 waves of 128-wide ones.
        if (format == 0 && layout == 0 && tile_n == 128 && M <= kTileM && N > 96 &&
            (mode == SK_MODE_DP || mode == SK_MODE_PERSISTENT)) {
          const int64_t workers = mode == SK_MODE_DP ? sm_count : sms;
          const int64_t t128 = ceil_div(N, 128), t96 = ceil_div(N, 96);
          if (ceil_div(t96, workers) <= ceil_div(t128, workers)) tile_n = 96;
        }
      }
    }
  }
  std::memset(p, 0, sizeof(*p));
  p->format = format;
  p->mode = mode;
  p->tile_m = tile_m;
  p->tile_n = tile_n;
  p->tile_k = format == 1 ? kMxTileK : (format == 2 ? kF8TileK : kBf16TileK);
  // bf16 with at most 64 rows of A on one-CTA 96- or 128-wide tiles (plain layout): tall stages
  // of 128 K, whose 128-row B boxes TMA streams faster than 64-row ones.
  const bool tall_ok =
      format == 0 && layout == 0 && !pair && M <= kTallMaxRows && tile_n != 256;
  const int tile_k = opt ? opt->tile_k : 0;
  if (tile_k == 0) {
    if (tall_ok) p->tile_k = 2 * kBf16TileK;
  } else if (tile_k != p->tile_k) {
    if (!(tall_ok && tile_k == 2 * kBf16TileK)) return SK_ERR_INVALID_ARG;
    p->tile_k = tile_k;
  }
  p->ctas_per_tile = pair ? 2 : 1;
  const int64_t tiles_m = ceil_div(M, tile_m), tiles_n = ceil_div(N, tile_n);
  const int64_t tiles = tiles_m * tiles_n;
  const int64_t iters = ceil_div(K, p->tile_k);
  if (tiles > kMaxDim / 2) return SK_ERR_UNSUPPORTED;
  p->tiles_m = static_cast<int32_t>(tiles_m);
  p->tiles_n = static_cast<int32_t>(tiles_n);
  p->tiles = tiles;
  p->iters = static_cast<int32_t>(iters);
  const int64_t units = pair ? pairs_avail : sms;   // schedulable workers
  int64_t grid = 0, sk_tiles = 0;
  switch (mode) {
    case SK_MODE_DP: grid = tiles; sk_tiles = 0; break;
    case SK_MODE_PERSISTENT: grid = std::min(units, tiles); sk_tiles = 0; break;
    case SK_MODE_STREAMK: grid = std::min(units, tiles * iters); sk_tiles = tiles; break;
    default: {
      grid = std::min(units, tiles * iters);
      const int64_t waves = opt != nullptr ? std::max<int32_t>(opt->hybrid_sk_waves, 0) : 0;
      sk_tiles = std::min(tiles, tiles % grid + waves * grid);
      break;
    }
  }
  // The kernels' schedule arithmetic runs in 32 bits: a Stream-K region of 2^31 or more
  // k-iterations (a product of 2^51 multiply-adds and up on 128 x 128 tiles) is refused.
  if (sk_tiles * iters > kMaxDim) return SK_ERR_UNSUPPORTED;
  p->grid = static_cast<int32_t>(grid);
  p->whole_tiles = tiles - sk_tiles;
  p->sk_tiles = sk_tiles;
  p->sk_base = sk_tiles * iters / grid;
  p->sk_extra = sk_tiles * iters % grid;
  int group = opt && opt->raster_group > 0 ? opt->raster_group : kDefaultRasterGroup;
  if (pair && !(opt && opt->raster_group > 0)) group = kDefaultRasterGroup / 2;
  p->raster_group = static_cast<int32_t>(std::min<int64_t>(group, tiles_m));
  return SK_OK;
}

// ---- automatic schedule and tile choice ---------------------------------------------------
//
// Estimated time of a plan, in microseconds.  The constants were fitted (least squares on the
// relative error, non-negative) to the measured times of 40 bf16 shapes (from 64x14336x4096
// to 8192^3, square, skinny, long-K, few-tile and wave-boundary cases) under every schedule
// and tile kind on a 152-SM GB300; on those shapes the cheapest estimate picks a
// configuration within 0.6 % of the fastest on average, 4.3 % at most.
struct CostModel {
  double t_iter[3];   // one k-iteration of a bf16 tile: SM pair 256x256x64, 128x256x64, 128x128x64
  double t_piece;     // each piece of work a CTA runs (tile hand-over, pipeline refill)
  double t_split;     // a Stream-K region whose tiles are split between CTAs (spill + fix-up)
  double t_part;      // each CTA that shares one split tile
  double t_launch;    // launch and first loads
  double t_split_shared;   // t_split and t_part where SM pairs share the finish of their split
  double t_part_shared;    // tiles (shared_finish below)
};
constexpr CostModel kCost = {{0.2836, 0.3321, 0.2501}, 1.021, 4.248, 2.0208, 10.6876,
                             9.9955, 0.3779};

// Whether the SM-pair kernels (bf16, fp8) finish most split tiles of a plan together with the
// contributors that hold nothing else: a Stream-K region over the whole grid's work whose
// ranges are at most a third of a tile, so that tiles have two such contributors or more.
bool shared_finish(const sk_plan_t& p, int format) {
  if (p.ctas_per_tile != 2 || format == 1 || p.sk_tiles == 0 || p.whole_tiles != 0) return false;
  const int64_t per = ceil_div(p.sk_tiles * p.iters, std::max<int64_t>(p.grid, 1));
  return ceil_div(static_cast<int64_t>(p.iters), std::max<int64_t>(per, 1)) >= 3;
}
// A k-iteration carries the same operand bytes in every format; an MXFP4 one (plus its scale
// copies) takes ~1.45 times a bf16 one (8192^3 persistent: 0.44 vs 0.30 us), fp8 the same.
constexpr double kMxIterScale = 1.45;
// Per 64 K, a tall stage's time against a 64-K stage's on the same tile (64 x 14336 x 4096 on
// one GB300: 128-wide tiles 28.9 against 30.2 us, 96-wide 28.9 against 28.9 us).
constexpr double kTallIterScale = 0.97;

double plan_cost(const sk_plan_t& p, int format) {
  const int kind = p.ctas_per_tile == 2 ? 0 : (p.tile_n == 256 ? 1 : 2);
  // A 96-wide k-iteration takes about as long as a 128-wide one on a busy SM (three quarters of
  // the B bytes at ~76 % of the rate); in one wave on more SMs the whole call ran ~6 % faster.
  // A tall stage (128 K) carries two 64-K iterations' bytes, streamed faster (kTallIterScale).
  const double t_iter = kCost.t_iter[kind] * (format == 1 ? kMxIterScale : 1.0) *
                        (p.tile_n == 96 ? 0.94 : 1.0) *
                        (format == 0 && p.tile_k == 2 * kBf16TileK ? 2.0 * kTallIterScale : 1.0);
  const int64_t g = std::max<int64_t>(p.grid, 1), T = p.tiles, I = p.iters;
  double iters = 0.0, pieces = 0.0, fixup = 0.0;
  if (p.mode == SK_MODE_DP || p.mode == SK_MODE_PERSISTENT) {
    const int64_t waves = ceil_div(T, g);
    iters = static_cast<double>(waves * I);
    pieces = static_cast<double>(waves);
  } else {
    const int64_t skT = p.sk_tiles, whole = p.whole_tiles;
    const int64_t per = skT > 0 ? ceil_div(skT * I, g) : 0;   // Stream-K iterations of a CTA
    iters = static_cast<double>(per + ceil_div(whole, g) * I);
    pieces = static_cast<double>(ceil_div(whole, g) + (skT > 0 ? ceil_div(per, I) + 1 : 0));
    if (skT > 0) {
      const bool split = per % I != 0 || (skT * I) % g != 0;
      const bool shared = shared_finish(p, format);
      fixup = (split ? (shared ? kCost.t_split_shared : kCost.t_split) : 0.0) +
              (shared ? kCost.t_part_shared : kCost.t_part) *
                  static_cast<double>(ceil_div(I, std::max<int64_t>(per, 1)));
    }
  }
  return kCost.t_launch + iters * t_iter + pieces * kCost.t_piece + fixup;
}

sk_status_t auto_plan(int format, int64_t M, int64_t N, int64_t K, int num_sms, int sm_count,
                      int max_pairs, const sk_options_t* opt, sk_plan_t* p, int layout) {
  struct Tile { int m, n; };
  const Tile tiles[4] = {{256, 256}, {128, 256}, {128, 128}, {128, 96}};
  const int modes[3] = {SK_MODE_PERSISTENT, SK_MODE_STREAMK, SK_MODE_HYBRID};
  sk_options_t base = {};
  base.drop_release_cta = -1;
  if (opt != nullptr) base = *opt;
  double best = 0.0;
  bool found = false;
  sk_status_t first_error = SK_ERR_INVALID_ARG;
  for (const Tile& t : tiles) {
    // tiles the options force stay forced
    if (base.tile_m != 0 && base.tile_m != t.m) continue;
    if (base.tile_n != 0 && base.tile_n != t.n) continue;
    // One row of tiles (M <= 128) is bound by streaming B, which 128-column tiles do faster on
    // GB300 than 256-column ones whatever the k-iteration count says: 64x14336x4096 31 vs
    // 38 us, 128x4096x11008 37 vs 55 us, 96x8192x8192 40 vs 49 us (best schedule of each).
    if (base.tile_n == 0 && M <= 128 && t.m == 128 && t.n == 256) continue;
    // ... and no SM-pair tile, half of whose 256 rows would be empty.
    if (base.tile_m == 0 && M <= 128 && t.m == 256) continue;
    // 96-wide tiles: one row of tiles, bf16 in the plain layout
    if (t.n == 96 && (format != 0 || layout != 0 || M > 128) && base.tile_n != 96) continue;
    for (int mode : modes) {
      sk_options_t o = base;
      o.tile_m = t.m;
      o.tile_n = t.n;
      sk_plan_t cand;
      const sk_status_t st = make_plan(format, M, N, K, num_sms, mode, sm_count, max_pairs, &o,
                                       &cand, layout);
      if (st != SK_OK) {
        if (!found) first_error = st;
        continue;
      }
      const double c = plan_cost(cand, format);
      if (!found || c < best) {
        best = c;
        *p = cand;
        found = true;
      }
    }
  }
  return found ? SK_OK : first_error;
}

sk::Plan kernel_plan(const sk_plan_t& p) {
  sk::Plan k = {};
  k.tiles_m = p.tiles_m;
  k.tiles_n = p.tiles_n;
  k.iters = p.iters;
  k.grid = p.grid;
  k.group_m = p.raster_group;
  k.tiles = p.tiles;
  k.whole_tiles = p.whole_tiles;
  k.sk_base = p.sk_base;
  k.sk_extra = p.sk_extra;
  return k;
}

bool aligned16(const void* ptr) { return (reinterpret_cast<uintptr_t>(ptr) & 15u) == 0; }

// ---------------------------------------------------------------------------------------
// devices, workspaces, tensor maps
// ---------------------------------------------------------------------------------------

struct DeviceInfo {
  bool known = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  bool variant_ready[sk::kNumVariants] = {};
  int ctas_per_sm[sk::kNumVariants] = {};   // 1-CTA variants: resident CTAs per SM
  int max_pairs[sk::kNumVariants] = {};     // pair variants: resident 2-CTA clusters
  int setup_error[sk::kNumVariants] = {};   // cudaError_t of the variant's last set-up
};

struct Workspace {
  float* P = nullptr;
  size_t P_bytes = 0;
  uint32_t* flags = nullptr;
  size_t flag_count = 0;
  uint32_t* err = nullptr;     // 4 words
  uint8_t* sf = nullptr;
  size_t sf_bytes = 0;
  float* red = nullptr;        // column-sum partials (bias gradient)
  size_t red_bytes = 0;
  uint32_t epoch = 0;
};

std::mutex g_mutex;
std::map<int, DeviceInfo> g_devices;
std::map<std::pair<int, cudaStream_t>, Workspace> g_workspaces;

// Choices measured by sk_autotune, per device and problem; SK_MODE_AUTO uses them first.
struct TuneKey {
  int dev, format, layout, out_dtype, num_sms;
  int64_t M, N, K;
  bool operator<(const TuneKey& o) const {
    if (dev != o.dev) return dev < o.dev;
    if (format != o.format) return format < o.format;
    if (layout != o.layout) return layout < o.layout;
    if (out_dtype != o.out_dtype) return out_dtype < o.out_dtype;
    if (num_sms != o.num_sms) return num_sms < o.num_sms;
    if (M != o.M) return M < o.M;
    if (N != o.N) return N < o.N;
    return K < o.K;
  }
};
struct TuneChoice {
  int mode, tile_m, tile_n, hybrid_sk_waves;
};
std::map<TuneKey, TuneChoice> g_tuned;   // guarded by g_mutex

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
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
  return fn;
}

// 2-D tensor map over a row-major matrix [rows][cols] of `elem` bytes per element, boxes of
// box_cols x box_rows elements, `swizzle` (128-byte unless given), zero fill outside the matrix.
bool encode_2d(CUtensorMap* map, CUtensorMapDataType type, size_t elem, const void* base,
               int64_t rows, int64_t cols, uint32_t box_cols, uint32_t box_rows,
               CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
  const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * elem};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, type, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Caller holds g_mutex.
sk_status_t device_info(int dev, DeviceInfo** out) {
  DeviceInfo& d = g_devices[dev];
  if (!d.known) {
    if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return SK_ERR_CUDA;
    d.known = true;
  }
  *out = &d;
  return SK_OK;
}

sk_status_t ensure_variant(DeviceInfo& d, int variant) {
  if (!d.variant_ready[variant]) {
    int n = 0;
    const cudaError_t e = sk::variant_is_pair(variant) ? sk::pair_variant_setup(variant, &n)
                                                       : sk::variant_setup(variant, &n);
    d.setup_error[variant] = static_cast<int>(e);
    if (e != cudaSuccess) {
      cudaGetLastError();   // clear the sticky-free launch error so later calls can run
      return SK_ERR_CUDA;
    }
    if (sk::variant_is_pair(variant)) {
      d.max_pairs[variant] = n;
    } else {
      d.ctas_per_sm[variant] = n;
    }
    d.variant_ready[variant] = true;
  }
  return SK_OK;
}

template <class T>
cudaError_t regrow(T** ptr, size_t* have, size_t need, cudaStream_t st) {
  if (*have >= need && *ptr != nullptr) return cudaSuccess;
  if (*ptr != nullptr) {
    cudaError_t e = cudaFreeAsync(*ptr, st);
    if (e != cudaSuccess) return e;
    *ptr = nullptr;
    *have = 0;
  }
  void* p = nullptr;
  cudaError_t e = cudaMallocAsync(&p, need, st);
  if (e != cudaSuccess) {
    cudaGetLastError();   // an allocation failure must not surface as a later call's launch error
    return e;
  }
  *ptr = static_cast<T*>(p);
  *have = need;
  return cudaSuccess;
}

// Caller holds g_mutex.  Grows the workspace of (dev, st) to at least the given sizes.
sk_status_t ensure_workspace(int dev, cudaStream_t st, size_t P_bytes, size_t flag_count,
                             size_t sf_bytes, Workspace** out, size_t red_bytes = 0) {
  Workspace& w = g_workspaces[{dev, st}];
  const bool fits = w.err != nullptr && w.P_bytes >= P_bytes && w.flags != nullptr &&
                    w.flag_count >= flag_count && w.sf_bytes >= sf_bytes &&
                    w.red_bytes >= red_bytes;
  if (!fits) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return SK_ERR_CUDA;
    if (cs != cudaStreamCaptureStatusNone) return SK_ERR_UNSUPPORTED;
    if (w.err == nullptr) {
      size_t have = 0;
      if (regrow(&w.err, &have, 16, st) != cudaSuccess) return SK_ERR_OOM;
      if (cudaMemsetAsync(w.err, 0, 16, st) != cudaSuccess) return SK_ERR_CUDA;
    }
    if (P_bytes > 0 && regrow(&w.P, &w.P_bytes, P_bytes, st) != cudaSuccess) return SK_ERR_OOM;
    if (w.flag_count < flag_count || w.flags == nullptr) {
      size_t bytes = w.flag_count * sizeof(uint32_t);
      const size_t need = std::max<size_t>(flag_count, 1) * sizeof(uint32_t);
      if (regrow(&w.flags, &bytes, need, st) != cudaSuccess) {
        w.flag_count = 0;   // the old flags are gone too
        return SK_ERR_OOM;
      }
      w.flag_count = bytes / sizeof(uint32_t);
      if (cudaMemsetAsync(w.flags, 0, bytes, st) != cudaSuccess) return SK_ERR_CUDA;
    }
    if (sf_bytes > 0 && regrow(&w.sf, &w.sf_bytes, sf_bytes, st) != cudaSuccess) return SK_ERR_OOM;
    if (red_bytes > 0 && regrow(&w.red, &w.red_bytes, red_bytes, st) != cudaSuccess) return SK_ERR_OOM;
  }
  *out = &w;
  return SK_OK;
}

struct MxLayout {
  int64_t kgroups, a_row_blocks, b_row_blocks;
  size_t bytes() const { return static_cast<size_t>((a_row_blocks + b_row_blocks) * kgroups * 512); }
};

MxLayout mx_layout(const sk_plan_t& p) {
  MxLayout l;
  l.kgroups = 2 * static_cast<int64_t>(p.iters);
  l.a_row_blocks = static_cast<int64_t>(p.tiles_m) * (p.tile_m / 128);
  l.b_row_blocks = static_cast<int64_t>(p.tiles_n) * (p.tile_n / 128);
  return l;
}

// The rearranged scales as a 2-D uint32 tensor of 1 KB rows: row (row block, k-iteration)
// holds the two 512-byte k groups one stage of the pair kernel reads.
bool encode_scale_rows(CUtensorMap* map, const void* base, int64_t row_blocks, int64_t iters) {
  EncodeTiledFn fn = encode_fn();
  if (fn == nullptr) return false;
  const cuuint64_t dims[2] = {256, static_cast<cuuint64_t>(row_blocks * iters)};
  const cuuint64_t strides[1] = {1024};
  const cuuint32_t box[2] = {256, 1};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT32, 2, const_cast<void*>(base), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------------------
// the GEMM call
// ---------------------------------------------------------------------------------------

sk_status_t validate(int format, const void* A, const void* A_scale, const void* B,
                     const void* B_scale, const void* bias, const void* C, int out_dtype,
                     int64_t M, int64_t N, int64_t K, int mode, const sk_options_t* opt,
                     int layout = 0) {
  if (A == nullptr || B == nullptr || C == nullptr) return SK_ERR_INVALID_ARG;
  if (!aligned16(A) || !aligned16(B) || !aligned16(C) || (bias && !aligned16(bias)))
    return SK_ERR_INVALID_ARG;
  if (out_dtype != SK_F32 && out_dtype != SK_BF16) return SK_ERR_INVALID_ARG;
  if (mode < SK_MODE_DP || mode > SK_MODE_AUTO) return SK_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim)
    return SK_ERR_INVALID_ARG;
  if (format == 0) {
    // 16-byte row pitches: A rows hold K (or M when stored transposed), B rows N (or K)
    const int64_t a_pitch = (layout & 1) ? M : K;
    const int64_t b_pitch = (layout & 2) ? K : N;
    if (a_pitch % 8 != 0 || b_pitch % 8 != 0 || N % 8 != 0) return SK_ERR_INVALID_ARG;
  } else if (format == 2) {
    if (layout != 0) return SK_ERR_INVALID_ARG;
    if (K % 16 != 0 || N % 16 != 0) return SK_ERR_INVALID_ARG;   // 16-byte row pitches
  } else {
    if (layout != 0) return SK_ERR_INVALID_ARG;
    if (A_scale == nullptr || B_scale == nullptr) return SK_ERR_INVALID_ARG;
    if (K % 32 != 0) return SK_ERR_INVALID_ARG;
  }
  if (opt != nullptr) {
    if (opt->tile_n != 0 && opt->tile_n != 96 && opt->tile_n != 128 && opt->tile_n != 256)
      return SK_ERR_INVALID_ARG;
    if (opt->tile_m != 0 && opt->tile_m != 128 && opt->tile_m != 256) return SK_ERR_INVALID_ARG;
    if (opt->tile_m == 256 && (opt->tile_n == 128 || opt->tile_n == 96)) return SK_ERR_INVALID_ARG;
    // 96-wide tiles: bf16 in the plain layout only
    if (opt->tile_n == 96 && (format != 0 || layout != 0)) return SK_ERR_INVALID_ARG;
    if (format == 1 && opt->tile_n == 256 && opt->tile_m != 256) return SK_ERR_INVALID_ARG;
    if (opt->spin_timeout_ns < 0 || opt->raster_group < 0 || opt->hybrid_sk_waves < 0)
      return SK_ERR_INVALID_ARG;
    if (opt->resident_limit < 0 || opt->sm_record_len < 0) return SK_ERR_INVALID_ARG;
    if ((opt->tile_k != 0 && opt->tile_k != 64 && opt->tile_k != 128 && opt->tile_k != 256) ||
        opt->reserved != 0)
      return SK_ERR_INVALID_ARG;
    if (opt->sm_record != nullptr &&
        (opt->sm_record_len == 0 || (reinterpret_cast<uintptr_t>(opt->sm_record) & 3u) != 0))
      return SK_ERR_INVALID_ARG;
  }
  return SK_OK;
}

// layout: bit 0 = A stored transposed (K x M), bit 1 = B stored transposed (N x K); bf16 only.
sk_status_t run_gemm(int format, const void* A, const void* A_scale, const void* B,
                     const void* B_scale, const void* bias, void* C, sk_dtype_t out_dtype,
                     int64_t M, int64_t N, int64_t K, int num_sms, sk_mode_t mode,
                     const sk_options_t* opt, void* stream_ptr, int layout = 0) {
  sk_status_t st =
      validate(format, A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, mode, opt, layout);
  if (st != SK_OK) return st;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SK_ERR_UNSUPPORTED;

  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo* di = nullptr;
  if ((st = device_info(dev, &di)) != SK_OK) return st;
  if (di->cc_major != 10 || di->cc_minor != 3) return SK_ERR_UNSUPPORTED;   // built for sm_103a

  // SK_MODE_AUTO: a choice measured by sk_autotune for this problem wins over the cost model
  // (when the options force no tile).
  sk_options_t tuned_opt = {};
  if (mode == SK_MODE_AUTO && (opt == nullptr || (opt->tile_m == 0 && opt->tile_n == 0))) {
    const auto it = g_tuned.find(TuneKey{dev, format, layout, static_cast<int>(out_dtype),
                                         num_sms <= 0 ? 0 : num_sms, M, N, K});
    if (it != g_tuned.end()) {
      if (opt != nullptr) {
        tuned_opt = *opt;
      } else {
        tuned_opt.drop_release_cta = -1;
      }
      tuned_opt.tile_m = it->second.tile_m;
      tuned_opt.tile_n = it->second.tile_n;
      tuned_opt.hybrid_sk_waves = it->second.hybrid_sk_waves;
      opt = &tuned_opt;
      mode = static_cast<sk_mode_t>(it->second.mode);
    }
  }

  // The pair variants' cluster capacity is needed to plan; set both candidates up first.
  const int pair_variant = format == 1   ? sk::kVariantMxPair
                           : format == 2 ? sk::variant_of(sk::kKindF8Pair, 0)
                                         : sk::variant_of(sk::kKindBf16Pair, layout);
  if ((st = ensure_variant(*di, pair_variant)) != SK_OK) return st;
  sk_plan_t plan;
  if ((st = make_plan(format, M, N, K, num_sms, mode, di->sm_count, di->max_pairs[pair_variant],
                      opt, &plan, layout)) != SK_OK)
    return st;
  const bool pair = plan.ctas_per_tile == 2;
  const int variant =
      pair ? pair_variant
      : format == 1 ? sk::kVariantMxN128
      : format == 2 ? sk::variant_of(plan.tile_n == 256 ? sk::kKindF8N256 : sk::kKindF8N128, 0)
      : plan.tile_k == 2 * kBf16TileK
          ? sk::variant_of(plan.tile_n == 96 ? sk::kKindBf16N96Tall : sk::kKindBf16N128Tall, 0)
      : plan.tile_n == 96 ? sk::variant_of(sk::kKindBf16N96, 0)
                    : sk::variant_of(plan.tile_n == 256 ? sk::kKindBf16N256 : sk::kKindBf16N128,
                                     layout);
  if ((st = ensure_variant(*di, variant)) != SK_OK) return st;
  const bool streamk = plan.sk_tiles > 0;
  if (streamk) {
    int64_t capacity = pair ? di->max_pairs[variant]
                            : static_cast<int64_t>(di->ctas_per_sm[variant]) * di->sm_count;
    if (opt != nullptr && opt->resident_limit > 0)
      capacity = std::min<int64_t>(capacity, opt->resident_limit);
    if (plan.grid > capacity) return SK_ERR_NOT_CORESIDENT;
  }
  const int64_t ctas = static_cast<int64_t>(plan.grid) * plan.ctas_per_tile;
  if (opt != nullptr && opt->sm_record != nullptr && ctas > opt->sm_record_len)
    return SK_ERR_INVALID_ARG;

  // Flags and partial slots are needed only where tiles are split: one per CTA, and in the bf16
  // and fp8 pairs a second one, for an owner's share of a tile that several CTAs finish.
  const size_t slots = streamk ? static_cast<size_t>(ctas) * (pair && format != 1 ? 2 : 1) : 0;
  const size_t P_bytes = slots * kTileM * plan.tile_n * sizeof(float);
  const MxLayout mx = mx_layout(plan);
  Workspace* ws = nullptr;
  if ((st = ensure_workspace(dev, stream, P_bytes, slots, format == 1 ? mx.bytes() : 0, &ws)) !=
      SK_OK)
    return st;
  if (++ws->epoch == 0) ws->epoch = 1;

  CUtensorMap tmA, tmB, tmSfa, tmSfb, tmC;
  std::memset(&tmSfa, 0, sizeof(tmSfa));
  std::memset(&tmSfb, 0, sizeof(tmSfb));
  std::memset(&tmC, 0, sizeof(tmC));
  const uint32_t b_box = pair ? 128u : static_cast<uint32_t>(plan.tile_n);   // B rows per CTA (MXFP4)
  bool ok;
  if (format == 0) {
    // A: M x K (box 64 k x 128 rows), or stored K x M (box 64 m x 64 k-rows).
    // B: K x N (box 64 n x 64 k-rows), or stored N x K (box 64 k x one CTA's columns).
    // Tall stages: A in boxes of 64 k x 64 rows, B in boxes 128 k-rows tall.
    const uint32_t bt_rows = pair ? 128u : static_cast<uint32_t>(plan.tile_n);
    const bool tall = plan.tile_k == 2 * kBf16TileK;
    const uint32_t b_rows = tall ? 128u : 64u;
    ok = ((layout & 1) ? encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, K, M, 64, 64)
                       : encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, A, M, K, 64,
                                   tall ? 64u : static_cast<uint32_t>(kTileM))) &&
         ((layout & 2) ? encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, N, K, 64, bt_rows)
          : plan.tile_n == 96
              // 96-wide tiles: boxes of 32 columns (64-byte rows, 64-byte swizzle)
              ? encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, K, N, 32, b_rows,
                          CU_TENSOR_MAP_SWIZZLE_64B)
              : encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, B, K, N, 64, b_rows));
  } else if (format == 2) {
    // fp8 as bytes: A M x K (box 128 k x 128 rows), B K x N (box 128 n x 128 k-rows).
    ok = encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, M, K, 128, kTileM) &&
         encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, K, N, 128, 128);
  } else {
    ok = encode_2d(&tmA, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, A, M, K / 2, 128, kTileM) &&
         encode_2d(&tmB, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, B, N, K / 2, 128, b_box);
  }
  // C leaves through TMA stores when its row pitch is a multiple of 16 bytes: always for bf16
  // and fp8 operands (N % 8 == 0), and for MXFP4 when N allows.  Boxes of 32 rows x 64 bytes
  // (64-byte swizzle); the MXFP4 pair kernel, with room for a 1 KB buffer per warp only, stores
  // 32 rows x 32 bytes at a time (no swizzle).
  const bool c_tma = out_dtype == SK_BF16 ? N % 8 == 0 : N % 4 == 0;
  const bool c_small = pair && format == 1;
  if (ok && c_tma) {
    const uint32_t box_bytes = c_small ? 32u : 64u;
    const CUtensorMapSwizzle sw = c_small ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_64B;
    ok = out_dtype == SK_BF16
             ? encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, C, M, N, box_bytes / 2, 32, sw)
             : encode_2d(&tmC, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, C, M, N, box_bytes / 4, 32, sw);
  }
  if (!ok) return SK_ERR_CUDA;

  sk::Launch l = {};
  l.tmA = &tmA;
  l.tmB = &tmB;
  l.tmSfa = &tmSfa;
  l.tmSfb = &tmSfb;
  l.tmC = c_tma ? &tmC : nullptr;
  l.grid = static_cast<int>(ctas);
  l.cooperative = streamk && !pair;
  l.stream = stream;
  sk::Args& a = l.args;
  a.bias = bias;
  a.C = C;
  a.M = M;
  a.N = N;
  a.K = K;
  a.out_bf16 = out_dtype == SK_BF16 ? 1 : 0;
  a.inject_drop = (opt != nullptr && opt->inject_faults) ? 1 : 0;
  a.drop_cta = opt != nullptr ? opt->drop_release_cta : -1;
  a.epoch = ws->epoch;
  a.plan = kernel_plan(plan);
  a.P = ws->P;
  a.flags = ws->flags;
  a.err = ws->err;
  a.c_tma = c_tma ? 1 : 0;
  if (streamk) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return SK_ERR_CUDA;
    a.replay = cs != cudaStreamCaptureStatusNone ? 1 : 0;
  }
  a.sm_record = opt != nullptr ? static_cast<uint32_t*>(opt->sm_record) : nullptr;
  a.timeout_ns = static_cast<uint64_t>(
      opt != nullptr && opt->spin_timeout_ns > 0 ? opt->spin_timeout_ns : kDefaultTimeoutNs);
  if (format == 1) {
    uint8_t* sfa = ws->sf;
    uint8_t* sfb = ws->sf + mx.a_row_blocks * mx.kgroups * 512;
    if (sk::mx_scale_prep(static_cast<const uint8_t*>(A_scale), M, mx.a_row_blocks,
                          static_cast<const uint8_t*>(B_scale), N, mx.b_row_blocks, K / 32,
                          mx.kgroups, ws->sf, stream) != cudaSuccess)
      return SK_ERR_CUDA;
    a.sfa = sfa;
    a.sfb = sfb;
    a.sf_kgroups = mx.kgroups;
    if (pair && !(encode_scale_rows(&tmSfa, sfa, mx.a_row_blocks, plan.iters) &&
                  encode_scale_rows(&tmSfb, sfb, mx.b_row_blocks, plan.iters)))
      return SK_ERR_CUDA;
  }
  cudaError_t e = pair ? sk::pair_variant_launch(variant, l) : sk::variant_launch(variant, l);
  if (e == cudaErrorCooperativeLaunchTooLarge) return SK_ERR_NOT_CORESIDENT;
  return e == cudaSuccess ? SK_OK : SK_ERR_CUDA;
}

}  // namespace

extern "C" {

sk_status_t sk_gemm_bf16(const void* A, const void* B, const void* bias, void* C,
                         sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                         sk_mode_t mode, void* stream) {
  const sk::NvtxRange range("sk_gemm_bf16");
  return run_gemm(0, A, nullptr, B, nullptr, bias, C, out_dtype, M, N, K, num_sms, mode, nullptr,
                  stream);
}

sk_status_t sk_gemm_bf16_ex(const void* A, const void* B, const void* bias, void* C,
                            sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                            sk_mode_t mode, const sk_options_t* options, void* stream) {
  const sk::NvtxRange range("sk_gemm_bf16_ex");
  return run_gemm(0, A, nullptr, B, nullptr, bias, C, out_dtype, M, N, K, num_sms, mode, options,
                  stream);
}

sk_status_t sk_gemm_mxfp4(const void* A, const void* A_scale, const void* B,
                          const void* B_scale, const void* bias, void* C, sk_dtype_t out_dtype,
                          int64_t M, int64_t N, int64_t K, int num_sms, sk_mode_t mode,
                          void* stream) {
  const sk::NvtxRange range("sk_gemm_mxfp4");
  return run_gemm(1, A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms, mode, nullptr,
                  stream);
}

sk_status_t sk_gemm_mxfp4_ex(const void* A, const void* A_scale, const void* B,
                             const void* B_scale, const void* bias, void* C,
                             sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                             sk_mode_t mode, const sk_options_t* options, void* stream) {
  const sk::NvtxRange range("sk_gemm_mxfp4_ex");
  return run_gemm(1, A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms, mode, options,
                  stream);
}

sk_status_t sk_gemm_fp8(const void* A, const void* B, const void* bias, void* C,
                        sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                        sk_mode_t mode, void* stream) {
  const sk::NvtxRange range("sk_gemm_fp8");
  return run_gemm(2, A, nullptr, B, nullptr, bias, C, out_dtype, M, N, K, num_sms, mode, nullptr,
                  stream);
}

sk_status_t sk_gemm_fp8_ex(const void* A, const void* B, const void* bias, void* C,
                           sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                           sk_mode_t mode, const sk_options_t* options, void* stream) {
  const sk::NvtxRange range("sk_gemm_fp8_ex");
  return run_gemm(2, A, nullptr, B, nullptr, bias, C, out_dtype, M, N, K, num_sms, mode, options,
                  stream);
}

sk_status_t sk_gemm_bf16_t(const void* A, int trans_a, const void* B, int trans_b,
                           const void* bias, void* C, sk_dtype_t out_dtype, int64_t M, int64_t N,
                           int64_t K, int num_sms, sk_mode_t mode, const sk_options_t* options,
                           void* stream) {
  const sk::NvtxRange range("sk_gemm_bf16_t");
  if ((trans_a != 0 && trans_a != 1) || (trans_b != 0 && trans_b != 1)) return SK_ERR_INVALID_ARG;
  return run_gemm(0, A, nullptr, B, nullptr, bias, C, out_dtype, M, N, K, num_sms, mode, options,
                  stream, trans_a | (trans_b << 1));
}

sk_status_t sk_addmm_backward_bf16(const void* dC, const void* A, const void* B, void* dA,
                                   void* dB, void* dbias, sk_dtype_t grad_dtype, int64_t M,
                                   int64_t N, int64_t K, int num_sms, sk_mode_t mode,
                                   void* stream) {
  const sk::NvtxRange range("sk_addmm_backward_bf16");
  if (dC == nullptr || (dA == nullptr && dB == nullptr && dbias == nullptr))
    return SK_ERR_INVALID_ARG;
  if ((dA != nullptr && B == nullptr) || (dB != nullptr && A == nullptr)) return SK_ERR_INVALID_ARG;
  if (grad_dtype != SK_F32 && grad_dtype != SK_BF16) return SK_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1 || M > kMaxDim || N > kMaxDim || K > kMaxDim) return SK_ERR_INVALID_ARG;
  if (!aligned16(dC) || (dA && !aligned16(dA)) || (dB && !aligned16(dB)) ||
      (dbias && !aligned16(dbias)) || (A && !aligned16(A)) || (B && !aligned16(B)))
    return SK_ERR_INVALID_ARG;
  if (N % 8 != 0 || K % 8 != 0) return SK_ERR_INVALID_ARG;
  if (dB != nullptr && M % 8 != 0) return SK_ERR_INVALID_ARG;   // A read M-major
  sk_status_t st = SK_OK;
  // dA (M x K) = dC (M x N) * B^T: B is stored K x N, i.e. transposed for this product.
  if (dA != nullptr &&
      (st = run_gemm(0, dC, nullptr, B, nullptr, nullptr, dA, grad_dtype, M, K, N, num_sms, mode,
                     nullptr, stream, 2)) != SK_OK)
    return st;
  // dB (K x N) = A^T * dC: A is stored M x K, i.e. transposed for this product.
  if (dB != nullptr &&
      (st = run_gemm(0, A, nullptr, dC, nullptr, nullptr, dB, grad_dtype, K, N, M, num_sms, mode,
                     nullptr, stream, 1)) != SK_OK)
    return st;
  if (dbias != nullptr) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return SK_ERR_UNSUPPORTED;
    Workspace* ws = nullptr;
    {
      std::lock_guard<std::mutex> lock(g_mutex);
      DeviceInfo* di = nullptr;
      if ((st = device_info(dev, &di)) != SK_OK) return st;
      if (di->cc_major != 10 || di->cc_minor != 3) return SK_ERR_UNSUPPORTED;
      if ((st = ensure_workspace(dev, s, 0, 1, 0, &ws,
                                 static_cast<size_t>(sk::colsum_scratch_bytes(M, N)))) != SK_OK)
        return st;
    }
    if (sk::colsum_bf16(dC, M, N, dbias, grad_dtype == SK_BF16 ? 1 : 0, ws->red, s) != cudaSuccess)
      return SK_ERR_CUDA;
  }
  return SK_OK;
}

sk_status_t sk_stream_status(void* stream_ptr) {
  const sk::NvtxRange range("sk_stream_status");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return SK_ERR_CUDA;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SK_ERR_CUDA;
  uint32_t* err = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    auto it = g_workspaces.find({dev, stream});
    if (it == g_workspaces.end() || it->second.err == nullptr) return SK_OK;
    err = it->second.err;
  }
  uint32_t words[4] = {0, 0, 0, 0};
  if (cudaMemcpyAsync(words, err, sizeof(words), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return SK_ERR_CUDA;
  if (words[0] == 0) return SK_OK;
  if (cudaMemsetAsync(err, 0, sizeof(words), stream) != cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return SK_ERR_CUDA;
  return static_cast<sk_status_t>(words[0]);
}

sk_status_t sk_workspace_reserve(int device, void* stream_ptr, int max_grid, int64_t max_mx_m,
                                 int64_t max_mx_n, int64_t max_mx_k) {
  const sk::NvtxRange range("sk_workspace_reserve");
  if (max_grid < 1 || max_mx_m < 0 || max_mx_n < 0 || max_mx_k < 0 || (max_mx_k % 32) != 0)
    return SK_ERR_INVALID_ARG;
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return SK_ERR_CUDA;
  if (cudaSetDevice(device) != cudaSuccess) return SK_ERR_INVALID_ARG;
  sk_status_t st = SK_OK;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    size_t sf_bytes = 0;
    if (max_mx_m > 0 && max_mx_n > 0 && max_mx_k > 0) {
      sk_plan_t p;
      // the larger of the two tile layouts
      sk_options_t o = {};
      o.tile_m = 128;
      st = make_plan(1, max_mx_m, max_mx_n, max_mx_k, 0, SK_MODE_DP, 1, 0, &o, &p);
      if (st == SK_OK) sf_bytes = mx_layout(p).bytes();
      o.tile_m = 256;
      if (st == SK_OK && make_plan(1, max_mx_m, max_mx_n, max_mx_k, 0, SK_MODE_DP, 2, 1, &o, &p) == SK_OK)
        sf_bytes = std::max(sf_bytes, mx_layout(p).bytes());
    }
    Workspace* ws = nullptr;
    if (st == SK_OK)
      // two slots and flags per CTA: the most any grid uses (bf16 and fp8 SM pairs)
      st = ensure_workspace(device, static_cast<cudaStream_t>(stream_ptr),
                            2 * static_cast<size_t>(max_grid) * kTileM * 256 * sizeof(float),
                            2 * static_cast<size_t>(max_grid), sf_bytes, &ws);
  }
  cudaSetDevice(prev);
  return st;
}

sk_status_t sk_workspace_release(int device, void* stream_ptr) {
  const sk::NvtxRange range("sk_workspace_release");
  cudaStream_t st = static_cast<cudaStream_t>(stream_ptr);
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return SK_ERR_UNSUPPORTED;   // no usable device
  // The capture state first: while a stream is captured, no call that could invalidate the
  // capture (such as changing the current device) is made.
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return SK_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return SK_ERR_UNSUPPORTED;
  if (device != prev && cudaSetDevice(device) != cudaSuccess) {
    cudaGetLastError();
    return SK_ERR_INVALID_ARG;
  }
  sk_status_t result = SK_OK;
  {
    {
      std::lock_guard<std::mutex> lock(g_mutex);
      const auto it = g_workspaces.find({device, st});
      if (it != g_workspaces.end()) {
        // Stream-ordered frees: the buffers go once the work already queued on `st` (the only
        // stream that uses them) has run, with no host synchronisation.
        Workspace& w = it->second;
        void* bufs[] = {w.P, w.flags, w.err, w.sf, w.red};
        for (void* b : bufs)
          if (b != nullptr && cudaFreeAsync(b, st) != cudaSuccess) result = SK_ERR_CUDA;
        g_workspaces.erase(it);
      }
    }
    if (sk::release_host_stage(device, st) != cudaSuccess) result = SK_ERR_CUDA;
  }
  if (device != prev) cudaSetDevice(prev);
  return result;
}

int64_t sk_workspace_bytes(int device, void* stream_ptr) {
  if (device < 0) return -1;
  const cudaStream_t st = static_cast<cudaStream_t>(stream_ptr);
  int64_t bytes = 0;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    const auto it = g_workspaces.find({device, st});
    if (it != g_workspaces.end()) {
      const Workspace& w = it->second;
      bytes += static_cast<int64_t>(w.P_bytes + w.flag_count * sizeof(uint32_t) + w.sf_bytes +
                                    w.red_bytes) +
               (w.err != nullptr ? 16 : 0);
    }
  }
  return bytes + sk::host_stage_bytes(device, st);
}

void sk_workspace_release_all(void) {
  std::lock_guard<std::mutex> lock(g_mutex);
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return;
  for (auto& kv : g_workspaces) {
    if (cudaSetDevice(kv.first.first) != cudaSuccess) continue;
    cudaDeviceSynchronize();
    Workspace& w = kv.second;
    if (w.P) cudaFree(w.P);
    if (w.flags) cudaFree(w.flags);
    if (w.err) cudaFree(w.err);
    if (w.sf) cudaFree(w.sf);
    if (w.red) cudaFree(w.red);
  }
  g_workspaces.clear();
  g_tuned.clear();
  cudaSetDevice(prev);
  sk::release_host_stages();
}

const char* sk_status_string(sk_status_t s) {
  switch (s) {
    case SK_OK: return "ok";
    case SK_ERR_INVALID_ARG: return "invalid argument";
    case SK_ERR_UNSUPPORTED: return "unsupported request (device or capture state)";
    case SK_ERR_OOM: return "workspace allocation failed";
    case SK_ERR_CUDA: return "CUDA call failed";
    case SK_ERR_TIMEOUT: return "a bounded wait inside the kernel ran out";
    case SK_ERR_NOT_CORESIDENT: return "Stream-K grid cannot be resident all at once";
  }
  return "unknown status";
}

sk_status_t sk_device_caps(int device, sk_device_caps_t* caps) {
  if (caps == nullptr) return SK_ERR_INVALID_ARG;
  std::memset(caps, 0, sizeof(*caps));
  int prev = 0;
  if (cudaGetDevice(&prev) != cudaSuccess) return SK_ERR_UNSUPPORTED;
  if (cudaSetDevice(device) != cudaSuccess) return SK_ERR_INVALID_ARG;
  sk_status_t st = SK_OK;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    DeviceInfo* d = nullptr;
    st = device_info(device, &d);
    if (st == SK_OK) {
      caps->sm_count = d->sm_count;
      caps->cc_major = d->cc_major;
      caps->cc_minor = d->cc_minor;
      if (d->cc_major == 10 && d->cc_minor == 3) {
        // the five reported variants, in the order of sk_device_caps_t's arrays
        const int reported[5] = {sk::kVariantBf16N128, sk::kVariantBf16N256, sk::kVariantMxN128,
                                 sk::kVariantBf16Pair, sk::kVariantMxPair};
        for (int i = 0; i < 5; ++i) ensure_variant(*d, reported[i]);
        caps->ctas_per_sm[0] = d->ctas_per_sm[sk::kVariantBf16N128];
        caps->ctas_per_sm[1] = d->ctas_per_sm[sk::kVariantBf16N256];
        caps->ctas_per_sm[2] = d->ctas_per_sm[sk::kVariantMxN128];
        caps->max_pair_clusters[0] = d->max_pairs[sk::kVariantBf16Pair];
        caps->max_pair_clusters[1] = d->max_pairs[sk::kVariantMxPair];
        for (int i = 0; i < 5; ++i) caps->setup_error[i] = d->setup_error[reported[i]];
        const int fp8[3] = {sk::variant_of(sk::kKindF8N128, 0), sk::variant_of(sk::kKindF8N256, 0),
                            sk::variant_of(sk::kKindF8Pair, 0)};
        for (int i = 0; i < 3; ++i) ensure_variant(*d, fp8[i]);
        caps->fp8_ctas_per_sm[0] = d->ctas_per_sm[fp8[0]];
        caps->fp8_ctas_per_sm[1] = d->ctas_per_sm[fp8[1]];
        caps->fp8_max_pair_clusters = d->max_pairs[fp8[2]];
        for (int i = 0; i < 3; ++i) caps->fp8_setup_error[i] = d->setup_error[fp8[i]];
      } else {
        st = SK_ERR_UNSUPPORTED;
      }
    }
  }
  cudaSetDevice(prev);
  return st;
}

sk_status_t sk_autotune(int format, const void* A, const void* A_scale, const void* B,
                        const void* B_scale, const void* bias, void* C, sk_dtype_t out_dtype,
                        int64_t M, int64_t N, int64_t K, int num_sms, int reps, sk_plan_t* chosen,
                        float* best_ms, void* stream_ptr) {
  const sk::NvtxRange range("sk_autotune");
  if (format < 0 || format > 2 || reps < 1 || reps > 1000) return SK_ERR_INVALID_ARG;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_ptr);
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return SK_ERR_CUDA;
  if (cs != cudaStreamCaptureStatusNone) return SK_ERR_UNSUPPORTED;   // timing synchronises
  int dev = 0, sm_count = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return SK_ERR_UNSUPPORTED;
  struct Cand {
    int tile_m, tile_n, mode, waves;
  };
  const Cand cands[] = {
      {256, 256, SK_MODE_PERSISTENT, 0}, {256, 256, SK_MODE_STREAMK, 0},
      {256, 256, SK_MODE_HYBRID, 0},     {256, 256, SK_MODE_HYBRID, 1},
      {128, 256, SK_MODE_PERSISTENT, 0}, {128, 256, SK_MODE_STREAMK, 0},
      {128, 256, SK_MODE_HYBRID, 0},     {128, 128, SK_MODE_PERSISTENT, 0},
      {128, 128, SK_MODE_STREAMK, 0},    {128, 128, SK_MODE_HYBRID, 0},
      {128, 128, SK_MODE_HYBRID, 1},     {128, 96, SK_MODE_PERSISTENT, 0},
      {128, 96, SK_MODE_STREAMK, 0}};
  auto run = [&](const Cand& c) -> sk_status_t {
    sk_options_t o = {};
    o.drop_release_cta = -1;
    o.tile_m = c.tile_m;
    o.tile_n = c.tile_n;
    o.hybrid_sk_waves = c.waves;
    const sk_mode_t m = static_cast<sk_mode_t>(c.mode);
    switch (format) {
      case 0: return sk_gemm_bf16_ex(A, B, bias, C, out_dtype, M, N, K, num_sms, m, &o, stream);
      case 2: return sk_gemm_fp8_ex(A, B, bias, C, out_dtype, M, N, K, num_sms, m, &o, stream);
      default:
        return sk_gemm_mxfp4_ex(A, A_scale, B, B_scale, bias, C, out_dtype, M, N, K, num_sms, m,
                                &o, stream);
    }
  };
  cudaEvent_t ev[2];
  if (cudaEventCreate(&ev[0]) != cudaSuccess) return SK_ERR_CUDA;
  if (cudaEventCreate(&ev[1]) != cudaSuccess) {
    cudaEventDestroy(ev[0]);
    return SK_ERR_CUDA;
  }
  sk_status_t result = SK_ERR_INVALID_ARG;   // no candidate ran
  float best = 0.0f;
  const Cand* pick = nullptr;
  for (const Cand& c : cands) {
    sk_status_t st = run(c);                       // warm-up; refuses invalid combinations
    if (st == SK_ERR_INVALID_ARG || st == SK_ERR_NOT_CORESIDENT) continue;
    if (st == SK_ERR_UNSUPPORTED) {   // e.g. a Stream-K region too large: other candidates may run
      if (pick == nullptr) result = st;
      continue;
    }
    if (st != SK_OK) {
      result = st;
      pick = nullptr;
      break;
    }
    cudaEventRecord(ev[0], stream);
    for (int r = 0; r < reps && st == SK_OK; ++r) st = run(c);
    cudaEventRecord(ev[1], stream);
    if (st == SK_OK) st = sk_stream_status(stream);   // synchronises; reports kernel errors
    if (st != SK_OK) {
      result = st;
      pick = nullptr;
      break;
    }
    float ms = 0.0f;
    if (cudaEventElapsedTime(&ms, ev[0], ev[1]) != cudaSuccess) {
      result = SK_ERR_CUDA;
      pick = nullptr;
      break;
    }
    ms /= static_cast<float>(reps);
    if (pick == nullptr || ms < best) {
      best = ms;
      pick = &c;
    }
    result = SK_OK;
  }
  cudaEventDestroy(ev[0]);
  cudaEventDestroy(ev[1]);
  if (result != SK_OK || pick == nullptr) return result;
  {
    std::lock_guard<std::mutex> lock(g_mutex);
    g_tuned[TuneKey{dev, format, 0, static_cast<int>(out_dtype), num_sms <= 0 ? 0 : num_sms, M,
                    N, K}] = TuneChoice{pick->mode, pick->tile_m, pick->tile_n, pick->waves};
  }
  if (best_ms != nullptr) *best_ms = best;
  if (chosen != nullptr) {
    sk_options_t o = {};
    o.drop_release_cta = -1;
    o.tile_m = pick->tile_m;
    o.tile_n = pick->tile_n;
    o.hybrid_sk_waves = pick->waves;
    return sk_plan(format, M, N, K, num_sms, static_cast<sk_mode_t>(pick->mode), sm_count, &o,
                   chosen);
  }
  return SK_OK;
}

sk_status_t sk_plan(int format, int64_t M, int64_t N, int64_t K, int num_sms, sk_mode_t mode,
                    int sm_count, const sk_options_t* options, sk_plan_t* plan) {
  return make_plan(format, M, N, K, num_sms, mode, sm_count, sm_count / 2, options, plan);
}

int64_t sk_plan_segments(const sk_plan_t* plan, int64_t* rows, int64_t cap) {
  if (plan == nullptr || plan->grid < 1 || plan->iters < 1 || plan->tiles < 1) return -1;
  const sk::Plan p = kernel_plan(*plan);
  int64_t n = 0;
  for (int64_t cta = 0; cta < p.grid; ++cta) {
    sk::Cursor cur(p, cta);
    sk::Unit u;
    while (cur.next(p, u)) {
      if (n < cap && rows != nullptr) {
        int32_t tm, tn;
        sk::tile_coords(p, u.tile, tm, tn);
        int64_t* r = rows + 7 * n;
        r[0] = cta;
        r[1] = u.tile;
        r[2] = u.k0;
        r[3] = u.k1;
        r[4] = u.role;
        r[5] = tm;
        r[6] = tn;
      }
      ++n;
    }
  }
  return n;
}

}  // extern "C"
