/*
 * sk_gemm.h — C ABI of the GB300 (sm_103a) persistent / SM-constrained / Stream-K addmm GEMM.
 *
 * The library computes   C = A * B (+ bias[n] broadcast over every row m)
 * with fp32 accumulation, for bf16 operands and for MXFP4 operands (E2M1 codes with one E8M0
 * scale per 32 consecutive K elements), under four work schedules:
 *
 *   SK_MODE_DP          data-parallel: one CTA per BM x BN output tile (the non-persistent
 *                       "naive" GEMM of flashinfer PR #982 "SM-constraint-GEMM by triton
 *                       persistent kernel", overview).
 *   SK_MODE_PERSISTENT  SM-constrained persistent grid: g = min(num_sms, SM count, tiles)
 *                       CTAs, CTA c takes tiles c, c+g, ... (same page: the grid is capped at
 *                       num_sms, and at the device's SM count — its nsys block shows a request
 *                       of 133 launched as 132 CTAs).
 *   SK_MODE_STREAMK     Stream-K: the tiles x k-iterations are split evenly over g CTAs; a CTA
 *                       whose range starts inside a tile spills its fp32 partial tile to a
 *                       scratch slot P[cta] and releases a flag; the tile's owner (the CTA
 *                       holding k = 0) acquires the flags, adds the partials, and only then
 *                       adds the bias along N and stores (tritonBLAS PR #67 "Fix StreamK Kernel
 *                       Bias", Motivation and Technical Details; tritonBLAS PR #74 "Stream-k
 *                       mxfp4 kernel": one P slot and one lock per CTA).  In the bf16 and
 *                       fp8 SM-pair kernels, where at least two CTAs have nothing to do but
 *                       their piece of a tile the owner ends on, they and the owner each
 *                       finish a share of its columns (the owner spills the others' share to
 *                       a second slot); every element still gets each partial and the bias
 *                       once.  (Not in calls captured into a CUDA graph, whose replays share
 *                       one flag epoch: there the owner finishes every tile.)
 *   SK_MODE_HYBRID      the last (tiles mod g) tiles run Stream-K over all g CTAs (each CTA does
 *                       its Stream-K share first), the other tiles run whole, round-robin.
 *   SK_MODE_AUTO        the library picks the schedule (persistent, Stream-K or hybrid) and the
 *                       CTA tile (256 x 256 SM pairs, 128 x 256 or 128 x 128, within any tile
 *                       the options force) with the lowest estimated time.  The estimate is a
 *                       cost model fitted to GB300 timings: launch + per-k-iteration time of
 *                       the tile kind x the iterations of the busiest CTA + a cost per piece of
 *                       work + a Stream-K fix-up cost per split tile and per CTA sharing it.
 *                       A problem with one row of tiles (M <= 128), bound by streaming B,
 *                       does not get 128 x 256 tiles unless the options force them.
 *                       This is the tuning step the SM-constraint GEMM page lists as optional
 *                       (flashinfer PR #982, "tune: get best config for gemm").  sk_plan()
 *                       reports the choice (its `mode` field holds the schedule picked).
 *
 * Conventions shared by every entry point
 *   - Pointers A, B, bias, C, A_scale, B_scale are DEVICE pointers owned by the caller, on the
 *     current CUDA device; they must stay valid until the work queued on `stream` has run.
 *     Each must be 16-byte aligned.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *   - Calls are asynchronous: the return value reports argument checks and enqueue errors
 *     only.  Errors found by the kernel (a Stream-K wait that timed out) are recorded in the
 *     stream's workspace and returned by sk_stream_status().
 *   - No exception crosses this boundary; every failure is a status code.
 *   - Scratch (the Stream-K partial slots P, their flags, the error words and the MXFP4
 *     scale-layout buffers) belongs to the library: one workspace per (device, stream), created
 *     on first use and grown on demand, never at load time and never on a default device.
 *     While `stream` is being captured into a CUDA graph no allocation is made; a workspace too
 *     small for the call then yields SK_ERR_UNSUPPORTED (reserve it beforehand with
 *     sk_workspace_reserve()).
 *   - Calls on one stream are ordered.  Calls on different streams use different workspaces
 *     and may run concurrently.
 */
#ifndef SK_GEMM_H
#define SK_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SK_MODE_DP = 0,
  SK_MODE_PERSISTENT = 1,
  SK_MODE_STREAMK = 2,
  SK_MODE_HYBRID = 3,
  SK_MODE_AUTO = 4
} sk_mode_t;

/* dtype of C, and of bias (the bias always has C's dtype) */
typedef enum { SK_F32 = 0, SK_BF16 = 1 } sk_dtype_t;

typedef enum {
  SK_OK = 0,
  SK_ERR_INVALID_ARG = 1,     /* bad size, null or misaligned pointer, bad enum value      */
  SK_ERR_UNSUPPORTED = 2,     /* valid request the library cannot run (e.g. no sm_103 GPU, */
                              /* a workspace too small while the stream is capturing, or a */
                              /* Stream-K region of 2^31 tile k-iterations or more)        */
  SK_ERR_OOM = 3,             /* workspace allocation failed                               */
  SK_ERR_CUDA = 4,            /* a CUDA runtime/driver call failed                         */
  SK_ERR_TIMEOUT = 5,         /* kernel-side: a bounded wait ran out (see sk_stream_status) */
  SK_ERR_NOT_CORESIDENT = 6   /* Stream-K/hybrid grid cannot be fully resident at once     */
} sk_status_t;

/*
 * sk_gemm_bf16 — C[M x N] = A[M x K] * B[K x N] (+ bias[N]).
 *   A: bf16, row-major M x K (row pitch K elements).  K must be a multiple of 8.
 *   B: bf16, row-major K x N (the torch `mm(a, b)` layout; row pitch N).  N must be a
 *      multiple of 8 (16-byte row pitch for the tensor-memory-accelerator loads).
 *   bias: NULL, or N values of out_dtype.  Added once per output element, after all partial
 *      tiles are summed, broadcast over rows (tritonBLAS PR #67, Technical Details).
 *   C: row-major M x N of out_dtype (SK_BF16: rounded to nearest-even from fp32; SK_F32).
 *   M, N, K >= 1 and < 2^31.  Stream-K and hybrid calls whose Stream-K region holds 2^31 or
 *      more tile k-iterations (products of 2^51 multiply-adds and up, on 128 x 128 tiles) are
 *      refused with SK_ERR_UNSUPPORTED; persistent and data-parallel calls are not.
 *   num_sms: <= 0 means every SM; larger than the SM count is capped to it.  Ignored by
 *      SK_MODE_DP (grid = number of tiles).
 * Returns SK_OK once the kernel is queued on `stream`.
 */
sk_status_t sk_gemm_bf16(const void* A, const void* B, const void* bias, void* C,
                         sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                         sk_mode_t mode, void* stream);

/*
 * sk_gemm_mxfp4 — the same product for MXFP4 operands (tritonBLAS PR #74 "Stream-k mxfp4
 * kernel"; encoding per OCP MX v1.0).
 *   A:       uint8, M x K/2 bytes, two E2M1 codes per byte packed along K, the even-k element
 *            in the low nibble.
 *   A_scale: uint8 E8M0, M x K/32, row-major; byte (m, j) scales A[m][32j .. 32j+31] by
 *            2^(E-127) (E = 255 is NaN and propagates).
 *   B:       uint8, N x K/2 bytes (B stored transposed: row n holds column n of the K x N
 *            operand, packed along K like A).
 *   B_scale: uint8 E8M0, N x K/32.
 *   K must be a multiple of 32.  M, N >= 1 (any value).  Other arguments as sk_gemm_bf16.
 * The call also runs a small kernel that rearranges the two scale arrays into the order the
 * tensor cores read them (into the stream's workspace); it is part of every call.
 */
sk_status_t sk_gemm_mxfp4(const void* A, const void* A_scale, const void* B,
                          const void* B_scale, const void* bias, void* C, sk_dtype_t out_dtype,
                          int64_t M, int64_t N, int64_t K, int num_sms, sk_mode_t mode,
                          void* stream);

/*
 * Optional tuning and test controls for the *_ex entry points.  Zero-initialise, then set
 * fields; a NULL options pointer means all defaults.
 *   tile_n:               0 = automatic, else 128 or 256 (columns per CTA tile; MXFP4 only 128).
 *   raster_group:         0 = automatic, else rows of tiles per group in the tile order.
 *   spin_timeout_ns:      0 = default (2 s).  Bound on every wait inside the kernel; when it
 *                         runs out the kernel records SK_ERR_TIMEOUT, skips the affected
 *                         stores and returns normally.
 *   drop_release_cta:     fault injection for tests, -1 (or any value when zeroed options are
 *                         passed with inject_faults = 0) = off.  When inject_faults != 0, the
 *                         CTA with this index never releases its Stream-K partial, so its
 *                         tile's owner times out.
 *   tile_m:               0 = automatic, 128 = one CTA per tile, 256 = a 2-CTA cluster (an SM
 *                         pair) per 256 x 256 tile.  Pair tiles need tile_n 0 or 256 and at
 *                         least two SMs; num_sms then counts both SMs of every pair (an odd
 *                         num_sms leaves one SM unused).
 *   hybrid_sk_waves:      SK_MODE_HYBRID only: full waves of g tiles added to the Stream-K
 *                         region on top of the (tiles mod g) remainder (0 = the remainder only;
 *                         1 = the "two-tile" variant, in which each CTA's Stream-K share is at
 *                         least one whole tile).  Capped at the tiles there are.
 *   resident_limit:       test control, 0 = off.  Otherwise the co-residency check of Stream-K
 *                         and hybrid grids takes this as the number of CTAs (one-CTA tiles) or
 *                         SM pairs (pair tiles) the device can hold at once, in place of the
 *                         occupancy the device reports; a grid above it is refused with
 *                         SK_ERR_NOT_CORESIDENT before anything is launched.  It stands in for
 *                         a device with less room than the planner assumed (the plan itself is
 *                         not changed), so the refusal can be tested.
 *   sm_record_len, sm_record:
 *                         SM-usage record, NULL = off.  Otherwise sm_record is a device buffer
 *                         of sm_record_len uint32 values (4-byte aligned) and CTA i of the launch
 *                         writes the index of the SM it runs on (%smid) to sm_record[i] when it
 *                         starts: one 4-byte store per CTA.  The launch has
 *                         plan.grid * plan.ctas_per_tile CTAs (sk_plan); a call whose launch
 *                         has more CTAs than sm_record_len is refused with SK_ERR_INVALID_ARG.
 *                         The distinct values show how many SMs an SM-constrained call used
 *                         (flashinfer PR #982 "SM-constraint-GEMM by triton persistent kernel"
 *                         checks the SMs a capped call occupies in its nsys profile).  Calls
 *                         that launch several GEMMs (the host-buffer and backward calls) each
 *                         overwrite the record.
 *   tile_k:               0 = automatic, else the K a pipeline stage carries: bf16 64 or 128,
 *                         fp8 128, MXFP4 256.  bf16 128 ("tall" stages) exists for one CTA per
 *                         96- or 128-wide tile, the plain layout and M <= 64; the automatic
 *                         choice takes it there (TMA streams B faster in 128-row boxes).  Any
 *                         other value is SK_ERR_INVALID_ARG.
 *   reserved:             0.
 */
typedef struct {
  int32_t tile_n;
  int32_t raster_group;
  int64_t spin_timeout_ns;
  int32_t inject_faults;
  int32_t drop_release_cta;
  int32_t tile_m;
  int32_t hybrid_sk_waves;
  int32_t resident_limit;
  int32_t sm_record_len;
  void* sm_record;
  int32_t tile_k;
  int32_t reserved;   /* 0 */
} sk_options_t;

sk_status_t sk_gemm_bf16_ex(const void* A, const void* B, const void* bias, void* C,
                            sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                            sk_mode_t mode, const sk_options_t* options, void* stream);

sk_status_t sk_gemm_mxfp4_ex(const void* A, const void* A_scale, const void* B,
                             const void* B_scale, const void* bias, void* C,
                             sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                             sk_mode_t mode, const sk_options_t* options, void* stream);

/*
 * sk_gemm_fp8 / sk_gemm_fp8_ex — the same product for 8-bit float operands (OCP FP8 E4M3: 1 sign
 * bit, 4 exponent bits with bias 7, 3 mantissa bits, largest finite 448, S.1111.111 = NaN, no
 * infinities), as taken by the SM-constraint GEMM of flashinfer PR #982 ("float8_e4m3fn",
 * review comments on the 16-byte minimum chunk).  Products accumulate in fp32.
 *   A: M x K bytes row-major; B: K x N bytes row-major (the torch `mm(a, b)` layout).
 *   K and N must be multiples of 16 (16-byte row pitches).  bias, C, out_dtype and the
 *   schedule arguments as sk_gemm_bf16 / sk_gemm_bf16_ex.  No scaling is applied (a per-tensor
 *   scale, if any, belongs to the caller).  Errors as sk_gemm_bf16.
 */
sk_status_t sk_gemm_fp8(const void* A, const void* B, const void* bias, void* C,
                        sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                        sk_mode_t mode, void* stream);

sk_status_t sk_gemm_fp8_ex(const void* A, const void* B, const void* bias, void* C,
                           sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                           sk_mode_t mode, const sk_options_t* options, void* stream);

/*
 * sk_gemm_bf16_host / sk_gemm_fp8_host / sk_gemm_mxfp4_host — the same addmm for operands and
 * result in HOST memory (the pages' calls take device tensors; this is the path for a caller
 * whose data lives on the host).  Arguments as the _ex calls, except that A, A_scale, B,
 * B_scale, bias and C are host pointers.  Page-locked (pinned) host memory lets the copies
 * overlap the computation; pageable memory works but copies synchronously.
 *   - The library keeps device copies of the operands and two copy streams per (device,
 *     stream), grown on demand and freed by sk_workspace_release_all.
 *   - B, its scales and the bias are copied first; A (and its scales) follows in up to 8
 *     row blocks of a multiple of 256 rows.  Each block's GEMM starts on `stream` when its
 *     rows have arrived, and its rows of C are copied back while later blocks compute.
 *   - Asynchronous like the other calls: C is complete once `stream` reaches the point after
 *     this call (synchronise it before reading C).  The host buffers must stay valid until then.
 *   - Shape, option and dtype errors are reported before anything is copied.  Refused
 *     (SK_ERR_UNSUPPORTED) while `stream` is being captured.
 */
sk_status_t sk_gemm_bf16_host(const void* A, const void* B, const void* bias, void* C,
                              sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                              sk_mode_t mode, const sk_options_t* options, void* stream);

sk_status_t sk_gemm_fp8_host(const void* A, const void* B, const void* bias, void* C,
                             sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K, int num_sms,
                             sk_mode_t mode, const sk_options_t* options, void* stream);

sk_status_t sk_gemm_mxfp4_host(const void* A, const void* A_scale, const void* B,
                               const void* B_scale, const void* bias, void* C,
                               sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K,
                               int num_sms, sk_mode_t mode, const sk_options_t* options,
                               void* stream);

/*
 * sk_gemm_bf16_t — C[M x N] = op(A) * op(B) (+ bias[N]) with either bf16 operand stored
 * transposed, through the same schedules and kernels (operands read M-major / K-major by the
 * tensor cores, no copy).
 *   trans_a = 0: A is M x K row-major;  trans_a = 1: A is stored K x M row-major (op(A) = A^T).
 *   trans_b = 0: B is K x N row-major;  trans_b = 1: B is stored N x K row-major (op(B) = B^T).
 *   Row pitches of the stored A and B (and N) must be multiples of 8 elements.  Other
 *   arguments as sk_gemm_bf16_ex.
 */
sk_status_t sk_gemm_bf16_t(const void* A, int trans_a, const void* B, int trans_b,
                           const void* bias, void* C, sk_dtype_t out_dtype, int64_t M, int64_t N,
                           int64_t K, int num_sms, sk_mode_t mode, const sk_options_t* options,
                           void* stream);

/*
 * sk_addmm_backward_bf16 — gradients of C = A * B + bias for an incoming gradient dC
 * (the backward of the addmm the correctness tests of tritonBLAS PR #67 "Fix StreamK Kernel
 * Bias" check through a.grad, b.grad and bias.grad):
 *   dA = dC * B^T   (M x K),   dB = A^T * dC   (K x N),   dbias[n] = sum_m dC[m][n]   (N).
 *   dC: M x N bf16; A: M x K bf16; B: K x N bf16 (the forward operands, as sk_gemm_bf16 takes
 *   them).  dA, dB, dbias: outputs of grad_dtype (SK_BF16 or SK_F32); each may be NULL to skip
 *   it (A may then be NULL when dB is skipped, B when dA is skipped).
 *   The two GEMMs run with `mode` and `num_sms` like the forward; dbias is a column sum with
 *   fp32 accumulation (deterministic, partial sums in the stream's workspace).
 *   N and K must be multiples of 8, and M too when dB is requested.
 */
sk_status_t sk_addmm_backward_bf16(const void* dC, const void* A, const void* B, void* dA,
                                   void* dB, void* dbias, sk_dtype_t grad_dtype, int64_t M,
                                   int64_t N, int64_t K, int num_sms, sk_mode_t mode,
                                   void* stream);

/*
 * sk_gemm_bf16_static — sk_gemm_bf16 for callers that cannot allocate device memory.
 * The pages this library follows have no counterpart to this entry point.
 * Some callers may not allocate at the point where they run the GEMM (they live under an
 * allocator they do not own, sit on a path where an allocation could synchronise the device,
 * or must not fail for lack of memory after start-up).  This entry point allocates nothing:
 * its scratch (error words, Stream-K flags and up to 160 partial tiles of 128 x 128 fp32,
 * about 10 MiB) is one fixed array inside the library that every GPU loading the library
 * keeps until the process exits.  Arguments and results are those of sk_gemm_bf16; it
 * always uses 128 x 128 CTA tiles (SK_MODE_AUTO picks the schedule among those tiles only).
 *   - Returns SK_ERR_UNSUPPORTED when the schedule would need more than 160 Stream-K slots.
 *   - The first call on a device looks up the array's device address and prepares the kernel
 *     on that device; make that first call before any stream capture on the device.  The
 *     set-up lasts for the life of the process: do not use this entry point on a device after
 *     cudaDeviceReset.
 *   - All calls share the one array (it keeps the last call's contents; each call clears the
 *     parts that must start at zero on its stream).  Calls that overlap on the GPU race and
 *     give wrong results: serialise them.
 *   - Kernel-side timeouts of this entry point are not reported by sk_stream_status; read them
 *     with sk_gemm_bf16_static_status.
 */
sk_status_t sk_gemm_bf16_static(const void* A, const void* B, const void* bias, void* C,
                                sk_dtype_t out_dtype, int64_t M, int64_t N, int64_t K,
                                int num_sms, sk_mode_t mode, void* stream);

/*
 * sk_gemm_bf16_static_status — waits for `stream`, then returns the error the last
 * sk_gemm_bf16_static call on the current device recorded (SK_OK, or SK_ERR_TIMEOUT when a
 * Stream-K wait ran out and its owner left that tile unwritten), or SK_ERR_CUDA if the copy or
 * the wait fails.  Allocates nothing.  The words are cleared by the next static call, so read
 * them before it.
 */
sk_status_t sk_gemm_bf16_static_status(void* stream);

/*
 * sk_stream_status — waits for `stream`, then returns (and clears) the first error the kernels
 * recorded in that stream's workspace on the current device: SK_OK, SK_ERR_TIMEOUT, or
 * SK_ERR_CUDA if the stream itself reports a CUDA error.
 */
sk_status_t sk_stream_status(void* stream);

/*
 * sk_workspace_reserve — size the workspace of (device, stream) for Stream-K and hybrid grids
 * of up to max_grid CTAs and MXFP4 problems of up to max_mx_m x max_mx_n x max_mx_k (0 = none),
 * so that later calls (e.g. while the stream is captured into a CUDA graph) need no allocation.
 * Data-parallel and persistent grids split no tile and use no per-CTA scratch, whatever their
 * size; MXFP4 calls of every schedule use the scale scratch.
 */
sk_status_t sk_workspace_reserve(int device, void* stream, int max_grid, int64_t max_mx_m,
                                 int64_t max_mx_n, int64_t max_mx_k);

/*
 * sk_workspace_release — frees the workspace of one (device, stream): its Stream-K slots,
 * flags, error words and MXFP4 scale scratch, and the device copies, copy streams and events
 * of the host-buffer calls on that stream.  For callers that create a stream per request, so
 * that workspaces do not accumulate until sk_workspace_release_all.
 *   - The frees are queued on `stream` (stream-ordered, no host synchronisation): work already
 *     queued there still runs with the old buffers.  A later call on the stream creates a new
 *     workspace.
 *   - A kernel error recorded in the workspace and not yet read by sk_stream_status is lost.
 *   - Refused (SK_ERR_UNSUPPORTED) while `stream` is being captured, and when no CUDA device
 *     is usable.  A (device, stream) with no workspace is not an error.  SK_ERR_INVALID_ARG for
 *     a device index that does not exist.
 */
sk_status_t sk_workspace_release(int device, void* stream);

/*
 * sk_workspace_bytes — device memory the library holds for (device, stream): the workspace
 * (Stream-K slots, flags, error words, MXFP4 scale scratch, column-sum partials) plus the
 * host-buffer calls' device copies.  0 when the stream has none; -1 for a negative device.
 * Host-only bookkeeping (no CUDA call).
 */
int64_t sk_workspace_bytes(int device, void* stream);

/* Frees every workspace (synchronises each device that has one first). */
void sk_workspace_release_all(void);

/* Static English description of a status code. */
const char* sk_status_string(sk_status_t status);

/*
 * sk_device_caps — what the library can launch on `device` (prepares every kernel variant of
 * the plain operand layouts on it): SM count, compute capability, resident CTAs per SM of the
 * one-CTA-per-tile variants (bf16 128x128, bf16 128x256, MXFP4 128x128; fp8 128x128 and
 * 128x256) and resident 2-CTA clusters of the SM-pair variants (bf16, MXFP4 and fp8 256x256),
 * with the CUDA error (0 = none) of each variant's set-up.
 */
typedef struct {
  int32_t sm_count;
  int32_t cc_major, cc_minor;
  int32_t ctas_per_sm[3];        /* bf16 128x128, bf16 128x256, MXFP4 128x128   */
  int32_t max_pair_clusters[2];  /* bf16 256x256 pairs, MXFP4 256x256 pairs      */
  int32_t setup_error[5];        /* cudaError_t of each variant's set-up, in the order above */
  int32_t fp8_ctas_per_sm[2];    /* fp8 128x128, fp8 128x256                     */
  int32_t fp8_max_pair_clusters; /* fp8 256x256 pairs                            */
  int32_t fp8_setup_error[3];    /* fp8 128x128, 128x256, 256x256 pairs          */
} sk_device_caps_t;

sk_status_t sk_device_caps(int device, sk_device_caps_t* caps);

/*
 * Planning (host only, makes no CUDA call).  Fills *plan with the schedule the library would
 * launch for this problem on a device with `sm_count` SMs.  format: 0 = bf16, 1 = MXFP4,
 * 2 = fp8 (E4M3).
 */
typedef struct {
  int32_t format;
  int32_t mode;
  int32_t tile_m, tile_n, tile_k;   /* CTA tile; tile_k in elements per k-iteration       */
  int32_t tiles_m, tiles_n;
  int64_t tiles;                    /* tiles_m * tiles_n                                  */
  int32_t iters;                    /* k-iterations per tile                              */
  int32_t grid;                     /* scheduling units: CTAs, or CTA pairs (see below)   */
  int32_t raster_group;
  int32_t ctas_per_tile;            /* 1, or 2 for SM-pair tiles (2 * grid CTAs launched) */
  int64_t whole_tiles;              /* linear tiles [0, whole_tiles) run whole            */
  int64_t sk_tiles;                 /* linear tiles [whole_tiles, tiles) run Stream-K     */
  int64_t sk_base;                  /* Stream-K iterations per CTA ...                    */
  int64_t sk_extra;                 /* ... plus one for CTAs [0, sk_extra)                */
} sk_plan_t;

sk_status_t sk_plan(int format, int64_t M, int64_t N, int64_t K, int num_sms, sk_mode_t mode,
                    int sm_count, const sk_options_t* options, sk_plan_t* plan);

/*
 * sk_autotune — measure every schedule x tile candidate for one problem on `stream` and keep
 * the fastest: later SK_MODE_AUTO calls with the same device, format, output dtype, M, N, K
 * and num_sms (and no forced tile in their options) use it instead of the cost model.  This is
 * the measured form of the optional tuning step of the SM-constraint GEMM page (flashinfer PR
 * #982, "tune: get best config for gemm").
 *   Operands, C and the other arguments as the format's _ex call (format 0 bf16, 1 MXFP4,
 *   2 fp8; plain layouts).  Each candidate runs once to warm up, then `reps` times (1..1000)
 *   between two events; C holds the product afterwards (from the last candidate run).
 *   chosen (may be NULL) receives the winning plan (its `mode` field is the schedule);
 *   best_ms (may be NULL) its mean time per call in milliseconds.
 *   Synchronises `stream`; refused (SK_ERR_UNSUPPORTED) while `stream` is being captured.
 *   Kernel errors during the runs are returned as by sk_stream_status.  The measured choices
 *   are kept until sk_workspace_release_all.
 */
sk_status_t sk_autotune(int format, const void* A, const void* A_scale, const void* B,
                        const void* B_scale, const void* bias, void* C, sk_dtype_t out_dtype,
                        int64_t M, int64_t N, int64_t K, int num_sms, int reps, sk_plan_t* chosen,
                        float* best_ms, void* stream);

/*
 * Enumerates the work the kernel's CTAs (or CTA pairs) perform for `plan`, in each one's
 * execution order: rows of 7 int64 (unit, linear tile, k_begin, k_end, role, tile_m index,
 * tile_n index), role
 * 0 = whole tile, 1 = owner of a split tile, 2 = partial contribution.  Writes at most `cap`
 * rows and returns the total count (call with cap = 0 to size the buffer), or -1 on bad input.
 * This runs the same scheduling code the kernel runs.
 */
int64_t sk_plan_segments(const sk_plan_t* plan, int64_t* rows, int64_t cap);

#ifdef __cplusplus
}
#endif

#endif /* SK_GEMM_H */
