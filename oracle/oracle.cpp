// CPU oracle for the addmm GEMM path: C = A*B (+ bias[n] broadcast over rows).
//
// TEST INFRASTRUCTURE ONLY.  This file is the slow, plain statement of what the GPU
// path must compute.  It shares no code, header, table or helper with the CUDA library,
// and the CUDA library never calls it: only the test suite, the smoke check and the
// CPU-baseline leg of the benchmark load it.
//
// Sources followed (cited by page title and section):
//  * flashinfer PR #982 "SM-constraint-GEMM by triton persistent kernel", overview:
//    the persistent kernel computes the ordinary GEMM; only the grid (number of CTAs)
//    is capped, so the result is the plain product.
//  * tritonBLAS PR #67 "Fix StreamK Kernel Bias", Motivation / Technical Details: the
//    bias is a vector along N broadcast over M, added once to each output element after
//    the Stream-K partial tiles of a tile have been aggregated ("quantized" mode converts
//    the bias to fp32 before the add).
//  * tritonBLAS PR #74 "Stream-k mxfp4 kernel", Changes: the same GEMM with MXFP4
//    operands.  The operand encoding is the OCP Microscaling (MX) v1.0 definition:
//    E2M1 elements (1 sign, 2 exponent bits with bias 1, 1 mantissa bit, no Inf/NaN)
//    and one E8M0 scale 2^(E-127) per 32 consecutive K elements (E = 255 is NaN).
//
// Arithmetic: every product a*b of two bf16 values, or of two decoded MX values, is exact
// in binary64; sums are accumulated in binary64 in ascending k; the bias is added once;
// the single final rounding to the output type is round-to-nearest-even.  Build with
// -ffp-contract=off so no multiply-add is fused (results are then identical on every
// host architecture).
//
// Readings where the pages are silent (each one also listed in the design notes):
//  * packed FP4 byte: the element with the even k index sits in the low nibble;
//  * MXFP4 B operand is stored N rows x K/2 bytes (packed along K);
//  * scales are row-major [rows][K/32] bytes, block j covering k in [32j, 32j+32);
//  * bias has the output's dtype (fp32 or bf16); a null bias means no bias.
//  * Stream-K split: see oracle_schedule below.
//  * addmm backward (the tests of tritonBLAS PR #67 compare a.grad, b.grad and bias.grad of
//    addmm against torch): for C = A*B + bias and an incoming gradient dC,
//    dA = dC * B^T, dB = A^T * dC, dbias[n] = sum over m of dC[m][n].

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

// ---------------------------------------------------------------------------------------
// Scalar encodings
// ---------------------------------------------------------------------------------------

// bf16 is the upper half of an IEEE binary32 word.
double bf16_value(uint16_t bits) {
  uint32_t word = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &word, sizeof f);
  return static_cast<double>(f);
}

// OCP MX E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
// Exponent field 0 is subnormal: value = m * 2^(1-1) * 0.5.
double e2m1_value(uint8_t code) {
  const int sign = (code >> 3) & 1;
  const int expo = (code >> 1) & 3;
  const int mant = code & 1;
  double magnitude;
  if (expo == 0) {
    magnitude = 0.5 * mant;
  } else {
    magnitude = std::ldexp(1.0 + 0.5 * mant, expo - 1);
  }
  return sign ? -magnitude : magnitude;
}

// OCP FP8 E4M3: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa; exponent 0 is
// subnormal (m * 2^-9); S.1111.111 is NaN; there are no infinities (largest finite 448).
double e4m3_value(uint8_t code) {
  const int sign = (code >> 7) & 1;
  const int expo = (code >> 3) & 15;
  const int mant = code & 7;
  if (expo == 15 && mant == 7) return std::nan("");
  const double magnitude =
      expo == 0 ? std::ldexp(static_cast<double>(mant), -9) : std::ldexp(1.0 + mant / 8.0, expo - 7);
  return sign ? -magnitude : magnitude;
}

// OCP MX E8M0: 2^(E-127); E = 255 encodes NaN.
double e8m0_value(uint8_t e) {
  if (e == 255) return std::nan("");
  return std::ldexp(1.0, static_cast<int>(e) - 127);
}

// Round a binary64 value to bf16 (8 exponent bits, 7 fraction bits), nearest-even,
// overflow to +-Inf, NaN to the canonical quiet NaN.
uint16_t round_to_bf16(double x) {
  if (std::isnan(x)) return 0x7FC0;
  const uint16_t sign = std::signbit(x) ? 0x8000 : 0x0000;
  if (std::isinf(x)) return sign | 0x7F80;
  if (x == 0.0) return sign;
  const double a = std::fabs(x);
  int e2;
  std::frexp(a, &e2);              // a in [2^(e2-1), 2^e2)
  const int unbiased = e2 - 1;
  // Spacing of bf16 values around a: 2^(E-7) for normals, 2^(-126-7) for subnormals.
  const int quantum_exp = std::max(unbiased, -126) - 7;
  const double steps = std::ldexp(a, -quantum_exp);   // exact power-of-two scaling
  const double rounded = std::nearbyint(steps);        // default mode: ties to even
  const double v = std::ldexp(rounded, quantum_exp);
  if (v >= std::ldexp(1.0, 128)) return sign | 0x7F80;
  const float f = static_cast<float>(v);               // exact: v is a bf16 value
  uint32_t word;
  std::memcpy(&word, &f, sizeof word);
  return sign | static_cast<uint16_t>((word >> 16) & 0x7FFF);
}

int worker_count(int requested) {
  if (requested > 0) return requested;
  unsigned hw = std::thread::hardware_concurrency();
  return hw == 0 ? 1 : static_cast<int>(hw);
}

// Run body(row) for row in [r0, r1) over `threads` workers (contiguous row blocks).
template <class F>
void parallel_rows(int64_t r0, int64_t r1, int threads, F body) {
  const int64_t n = r1 - r0;
  if (n <= 0) return;
  const int64_t workers = std::min<int64_t>(worker_count(threads), n);
  std::vector<std::thread> pool;
  for (int64_t w = 0; w < workers; ++w) {
    const int64_t lo = r0 + n * w / workers;
    const int64_t hi = r0 + n * (w + 1) / workers;
    pool.emplace_back([=] {
      for (int64_t r = lo; r < hi; ++r) body(r);
    });
  }
  for (auto& t : pool) t.join();
}

double bias_value(const void* bias, int bias_dtype, int64_t n) {
  if (bias == nullptr) return 0.0;
  if (bias_dtype == 0) return static_cast<double>(static_cast<const float*>(bias)[n]);
  return bf16_value(static_cast<const uint16_t*>(bias)[n]);
}

// Element (m, k) of an MXFP4 operand stored as rows x K/2 code bytes with rows x K/32 scales.
double mx_element(const uint8_t* codes, const uint8_t* scales, int64_t K, int64_t row,
                  int64_t k) {
  const uint8_t byte = codes[row * (K / 2) + k / 2];
  const uint8_t code = (k % 2 == 0) ? (byte & 0x0F) : (byte >> 4);
  return e2m1_value(code) * e8m0_value(scales[row * (K / 32) + k / 32]);
}

// ---------------------------------------------------------------------------------------
// Schedule restatement (Stream-K / persistent / data-parallel / hybrid)
// ---------------------------------------------------------------------------------------

enum { MODE_DP = 0, MODE_PERSISTENT = 1, MODE_STREAMK = 2, MODE_HYBRID = 3 };
enum { ROLE_FULL = 0, ROLE_OWNER = 1, ROLE_CONTRIB = 2 };

struct Segment {
  int64_t cta, tile, k0, k1, role;
};

// Segments of every CTA, each CTA's list in execution order.
//  * data-parallel: one CTA per tile (grid = tiles).
//  * persistent (SM-constrained): CTA c takes tiles c, c+g, c+2g, ...
//  * Stream-K: the tiles x k-iterations of the Stream-K region, taken in linear order
//    (tile-major, then k), are split into g contiguous ranges whose lengths differ by at
//    most one (the first (total mod g) ranges are one longer).  A range piece that holds
//    k = 0 of its tile makes that CTA the tile's owner; a piece that starts past k = 0 is a
//    partial contribution that the owner adds in before the bias.
//  * hybrid: the last (tiles mod g) tiles form the Stream-K region, the others are run
//    whole, round-robin.
// A CTA runs, in order: the Stream-K tiles lying entirely in its range; its contribution
// (the start of its range, if that is inside a tile); the tile its range ends in, if it owns
// that tile but does not finish it; then its whole tiles outside the Stream-K region.
// hybrid_waves: full waves of `grid` tiles added to the hybrid schedule's Stream-K region on
// top of the (tiles mod grid) remainder -- the "two-tile" form of the hybrid, in which every
// CTA's Stream-K share is at least one whole tile (0 = the remainder only).
std::vector<Segment> schedule(int mode, int64_t tiles, int64_t iters, int64_t grid,
                              int64_t hybrid_waves = 0) {
  std::vector<Segment> out;
  if (mode == MODE_DP) {
    for (int64_t t = 0; t < tiles; ++t) out.push_back({t, t, 0, iters, ROLE_FULL});
    return out;
  }
  if (mode == MODE_PERSISTENT) {
    for (int64_t c = 0; c < grid; ++c)
      for (int64_t t = c; t < tiles; t += grid) out.push_back({c, t, 0, iters, ROLE_FULL});
    return out;
  }
  const int64_t sk_tiles = (mode == MODE_STREAMK)
                               ? tiles
                               : std::min(tiles, tiles % grid + hybrid_waves * grid);
  const int64_t whole_tiles = tiles - sk_tiles;
  const int64_t total = sk_tiles * iters;
  const int64_t base = total / grid;
  const int64_t extra = total % grid;
  for (int64_t c = 0; c < grid; ++c) {
    // cut this CTA's range at tile boundaries
    const int64_t begin = c * base + std::min(c, extra);
    const int64_t end = begin + base + (c < extra ? 1 : 0);
    std::vector<Segment> pieces;
    for (int64_t it = begin; it < end;) {
      const int64_t t = it / iters;
      const int64_t k0 = it % iters;
      const int64_t k1 = std::min(iters, k0 + (end - it));
      int64_t role;
      if (k0 > 0) role = ROLE_CONTRIB;
      else if (k1 == iters) role = ROLE_FULL;
      else role = ROLE_OWNER;
      pieces.push_back({c, whole_tiles + t, k0, k1, role});
      it += k1 - k0;
    }
    for (const Segment& s : pieces) if (s.role == ROLE_FULL) out.push_back(s);
    for (const Segment& s : pieces) if (s.role == ROLE_CONTRIB) out.push_back(s);
    for (const Segment& s : pieces) if (s.role == ROLE_OWNER) out.push_back(s);
    for (int64_t t = c; t < whole_tiles; t += grid) out.push_back({c, t, 0, iters, ROLE_FULL});
  }
  return out;
}

}  // namespace

extern "C" {

// ---- scalar helpers exposed for the pins -------------------------------------------------

double oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }
double oracle_e2m1_value(uint8_t code) { return e2m1_value(code); }
double oracle_e8m0_value(uint8_t e) { return e8m0_value(e); }
double oracle_e4m3_value(uint8_t code) { return e4m3_value(code); }
uint16_t oracle_round_bf16(double x) { return round_to_bf16(x); }

// Round n binary64 values to the output type: out_dtype 0 = fp32 (float*), 1 = bf16 (uint16_t*).
void oracle_round_output(const double* x, void* y, int64_t n, int out_dtype) {
  for (int64_t i = 0; i < n; ++i) {
    if (out_dtype == 0) {
      static_cast<float*>(y)[i] = static_cast<float>(x[i]);  // IEEE conversion, nearest-even
    } else {
      static_cast<uint16_t*>(y)[i] = round_to_bf16(x[i]);
    }
  }
}

// ---- bf16 addmm ---------------------------------------------------------------------------
// A: M x K bf16 row-major.  B: K x N bf16 row-major.  bias: N values (bias_dtype 0 = fp32,
// 1 = bf16) or null.  out: rows [m0, m1) of the exact-product, binary64-accumulated result,
// written as out[(m - m0) * N + n].
int oracle_addmm_bf16_rows(const uint16_t* A, const uint16_t* B, const void* bias,
                           int bias_dtype, int64_t M, int64_t N, int64_t K, int64_t m0,
                           int64_t m1, double* out, int threads) {
  if (M < 0 || N < 0 || K < 0 || m0 < 0 || m1 > M || m0 > m1) return 1;
  std::vector<double> Bv(static_cast<size_t>(K * N));
  for (int64_t i = 0; i < K * N; ++i) Bv[i] = bf16_value(B[i]);
  parallel_rows(m0, m1, threads, [&](int64_t m) {
    double* row = out + (m - m0) * N;
    for (int64_t n = 0; n < N; ++n) row[n] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = bf16_value(A[m * K + k]);
      const double* brow = Bv.data() + k * N;
      for (int64_t n = 0; n < N; ++n) row[n] = row[n] + a * brow[n];
    }
    for (int64_t n = 0; n < N; ++n) row[n] = row[n] + bias_value(bias, bias_dtype, n);
  });
  return 0;
}

// Selected elements only: out[i] = C(ms[i], ns[i]) in binary64, same summation order.
int oracle_addmm_bf16_at(const uint16_t* A, const uint16_t* B, const void* bias,
                         int bias_dtype, int64_t M, int64_t N, int64_t K, const int64_t* ms,
                         const int64_t* ns, int64_t count, double* out, int threads) {
  for (int64_t i = 0; i < count; ++i)
    if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return 1;
  parallel_rows(0, count, threads, [&](int64_t i) {
    const int64_t m = ms[i], n = ns[i];
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) s = s + bf16_value(A[m * K + k]) * bf16_value(B[k * N + n]);
    out[i] = s + bias_value(bias, bias_dtype, n);
  });
  return 0;
}

// ---- general bf16 GEMM with stored-transposed operands ---------------------------------
// C[m][n] = sum_k opA(m, k) * opB(k, n) (+ bias[n]), where opA(m, k) = A[m*K + k] (A stored
// M x K) or A[k*M + m] when trans_a (A stored K x M), and opB(k, n) = B[k*N + n] (B stored
// K x N) or B[n*K + k] when trans_b (B stored N x K).  Rows [m0, m1) into out.
int oracle_gemm_bf16_t_rows(const uint16_t* A, int trans_a, const uint16_t* B, int trans_b,
                            const void* bias, int bias_dtype, int64_t M, int64_t N, int64_t K,
                            int64_t m0, int64_t m1, double* out, int threads) {
  if (M < 0 || N < 0 || K < 0 || m0 < 0 || m1 > M || m0 > m1) return 1;
  std::vector<double> Bv(static_cast<size_t>(K * N));   // opB(k, n) at k * N + n
  for (int64_t k = 0; k < K; ++k)
    for (int64_t n = 0; n < N; ++n)
      Bv[k * N + n] = bf16_value(trans_b ? B[n * K + k] : B[k * N + n]);
  parallel_rows(m0, m1, threads, [&](int64_t m) {
    double* row = out + (m - m0) * N;
    for (int64_t n = 0; n < N; ++n) row[n] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = bf16_value(trans_a ? A[k * M + m] : A[m * K + k]);
      const double* brow = Bv.data() + k * N;
      for (int64_t n = 0; n < N; ++n) row[n] = row[n] + a * brow[n];
    }
    for (int64_t n = 0; n < N; ++n) row[n] = row[n] + bias_value(bias, bias_dtype, n);
  });
  return 0;
}

int oracle_gemm_bf16_t_at(const uint16_t* A, int trans_a, const uint16_t* B, int trans_b,
                          int64_t M, int64_t N, int64_t K, const int64_t* ms, const int64_t* ns,
                          int64_t count, double* out, int threads) {
  for (int64_t i = 0; i < count; ++i)
    if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return 1;
  parallel_rows(0, count, threads, [&](int64_t i) {
    const int64_t m = ms[i], n = ns[i];
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
      s = s + bf16_value(trans_a ? A[k * M + m] : A[m * K + k]) *
                  bf16_value(trans_b ? B[n * K + k] : B[k * N + n]);
    out[i] = s;
  });
  return 0;
}

// ---- addmm backward -------------------------------------------------------------------------
// For C = A * B + bias (A: M x K, B: K x N, bf16) and dC (M x N, bf16):
//   dA[m][k] = sum_n dC[m][n] * B[k][n]        (M x K)
//   dB[k][n] = sum_m A[m][k] * dC[m][n]        (K x N)
//   dbias[n] = sum_m dC[m][n]                  (N)
// in binary64, sums in ascending index.  Any output pointer may be null.
int oracle_addmm_backward_bf16(const uint16_t* dC, const uint16_t* A, const uint16_t* B,
                               int64_t M, int64_t N, int64_t K, double* dA, double* dB,
                               double* dbias, int threads) {
  if (M < 1 || N < 1 || K < 1) return 1;
  if (dA != nullptr) {
    parallel_rows(0, M, threads, [&](int64_t m) {
      for (int64_t k = 0; k < K; ++k) {
        double s = 0.0;
        for (int64_t n = 0; n < N; ++n) s = s + bf16_value(dC[m * N + n]) * bf16_value(B[k * N + n]);
        dA[m * K + k] = s;
      }
    });
  }
  if (dB != nullptr) {
    parallel_rows(0, K, threads, [&](int64_t k) {
      for (int64_t n = 0; n < N; ++n) dB[k * N + n] = 0.0;
      for (int64_t m = 0; m < M; ++m) {
        const double a = bf16_value(A[m * K + k]);
        for (int64_t n = 0; n < N; ++n) dB[k * N + n] = dB[k * N + n] + a * bf16_value(dC[m * N + n]);
      }
    });
  }
  if (dbias != nullptr) {
    for (int64_t n = 0; n < N; ++n) {
      double s = 0.0;
      for (int64_t m = 0; m < M; ++m) s = s + bf16_value(dC[m * N + n]);
      dbias[n] = s;
    }
  }
  return 0;
}

// ---- fp8 (E4M3) addmm -----------------------------------------------------------------------
// A: M x K bytes, B: K x N bytes, both E4M3, row-major.  Output as for the bf16 form.
int oracle_addmm_fp8_rows(const uint8_t* A, const uint8_t* B, const void* bias, int bias_dtype,
                          int64_t M, int64_t N, int64_t K, int64_t m0, int64_t m1, double* out,
                          int threads) {
  if (M < 0 || N < 0 || K < 0 || m0 < 0 || m1 > M || m0 > m1) return 1;
  std::vector<double> Bv(static_cast<size_t>(K * N));
  for (int64_t i = 0; i < K * N; ++i) Bv[i] = e4m3_value(B[i]);
  parallel_rows(m0, m1, threads, [&](int64_t m) {
    double* row = out + (m - m0) * N;
    for (int64_t n = 0; n < N; ++n) row[n] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = e4m3_value(A[m * K + k]);
      const double* brow = Bv.data() + k * N;
      for (int64_t n = 0; n < N; ++n) row[n] = row[n] + a * brow[n];
    }
    for (int64_t n = 0; n < N; ++n) row[n] = row[n] + bias_value(bias, bias_dtype, n);
  });
  return 0;
}

int oracle_addmm_fp8_at(const uint8_t* A, const uint8_t* B, const void* bias, int bias_dtype,
                        int64_t M, int64_t N, int64_t K, const int64_t* ms, const int64_t* ns,
                        int64_t count, double* out, int threads) {
  for (int64_t i = 0; i < count; ++i)
    if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return 1;
  double value[256];
  for (int c = 0; c < 256; ++c) value[c] = e4m3_value(static_cast<uint8_t>(c));
  parallel_rows(0, count, threads, [&](int64_t i) {
    const int64_t m = ms[i], n = ns[i];
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) s = s + value[A[m * K + k]] * value[B[k * N + n]];
    out[i] = s + bias_value(bias, bias_dtype, n);
  });
  return 0;
}

// ---- MXFP4 addmm --------------------------------------------------------------------------
// A: M x K/2 code bytes, A_scale: M x K/32 E8M0 bytes.  B: N x K/2 code bytes, B_scale:
// N x K/32.  K must be a multiple of 32.  Output as for the bf16 form.
int oracle_addmm_mxfp4_rows(const uint8_t* A, const uint8_t* A_scale, const uint8_t* B,
                            const uint8_t* B_scale, const void* bias, int bias_dtype, int64_t M,
                            int64_t N, int64_t K, int64_t m0, int64_t m1, double* out,
                            int threads) {
  if (M < 0 || N < 0 || K < 0 || K % 32 != 0 || m0 < 0 || m1 > M || m0 > m1) return 1;
  // b(k, n), decoded once, stored k-major so the inner loop runs over n.
  std::vector<double> Bv(static_cast<size_t>(K * N));
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k) Bv[k * N + n] = mx_element(B, B_scale, K, n, k);
  parallel_rows(m0, m1, threads, [&](int64_t m) {
    double* row = out + (m - m0) * N;
    for (int64_t n = 0; n < N; ++n) row[n] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = mx_element(A, A_scale, K, m, k);
      const double* brow = Bv.data() + k * N;
      for (int64_t n = 0; n < N; ++n) row[n] = row[n] + a * brow[n];
    }
    for (int64_t n = 0; n < N; ++n) row[n] = row[n] + bias_value(bias, bias_dtype, n);
  });
  return 0;
}

int oracle_addmm_mxfp4_at(const uint8_t* A, const uint8_t* A_scale, const uint8_t* B,
                          const uint8_t* B_scale, const void* bias, int bias_dtype, int64_t M,
                          int64_t N, int64_t K, const int64_t* ms, const int64_t* ns,
                          int64_t count, double* out, int threads) {
  if (K % 32 != 0) return 1;
  for (int64_t i = 0; i < count; ++i)
    if (ms[i] < 0 || ms[i] >= M || ns[i] < 0 || ns[i] >= N) return 1;
  parallel_rows(0, count, threads, [&](int64_t i) {
    const int64_t m = ms[i], n = ns[i];
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k)
      s = s + mx_element(A, A_scale, K, m, k) * mx_element(B, B_scale, K, n, k);
    out[i] = s + bias_value(bias, bias_dtype, n);
  });
  return 0;
}

// ---- schedule ------------------------------------------------------------------------------
// Writes up to `cap` rows of 5 int64 (cta, tile, k_begin, k_end, role) and returns the total
// number of segments (call with cap = 0 to size the buffer).  role: 0 whole tile,
// 1 owner of a split tile, 2 partial contribution.  Tiles are linear indices.
int64_t oracle_schedule_hybrid(int mode, int64_t tiles, int64_t iters, int64_t grid,
                               int64_t hybrid_waves, int64_t* rows, int64_t cap) {
  if (tiles < 1 || iters < 1 || grid < 1 || mode < 0 || mode > 3 || hybrid_waves < 0) return -1;
  const std::vector<Segment> segs = schedule(mode, tiles, iters, grid, hybrid_waves);
  const int64_t n = static_cast<int64_t>(segs.size());
  for (int64_t i = 0; i < std::min(n, cap); ++i) {
    rows[5 * i + 0] = segs[i].cta;
    rows[5 * i + 1] = segs[i].tile;
    rows[5 * i + 2] = segs[i].k0;
    rows[5 * i + 3] = segs[i].k1;
    rows[5 * i + 4] = segs[i].role;
  }
  return n;
}

int64_t oracle_schedule(int mode, int64_t tiles, int64_t iters, int64_t grid, int64_t* rows,
                        int64_t cap) {
  return oracle_schedule_hybrid(mode, tiles, iters, grid, 0, rows, cap);
}

// Schedule-emulating bf16 addmm: for every tile, the partial sums of its segments (each a
// binary64 sum over the segment's k range, k ascending) are added in the order owner
// first, then contributors by increasing CTA, and the bias is added once at the end.
// Tiles are BM x BN (linear tile index row-major over the tile grid), one k-iteration is
// BK elements.  Output: the full M x N result in binary64.
int oracle_addmm_bf16_scheduled(const uint16_t* A, const uint16_t* B, const void* bias,
                                int bias_dtype, int64_t M, int64_t N, int64_t K, int mode,
                                int64_t BM, int64_t BN, int64_t BK, int64_t grid,
                                double* out) {
  if (M < 1 || N < 1 || K < 1 || BM < 1 || BN < 1 || BK < 1) return 1;
  const int64_t tiles_m = (M + BM - 1) / BM, tiles_n = (N + BN - 1) / BN;
  const int64_t tiles = tiles_m * tiles_n, iters = (K + BK - 1) / BK;
  if (mode == MODE_DP) grid = tiles;
  if (grid < 1) return 1;
  std::vector<Segment> segs = schedule(mode, tiles, iters, grid);
  // Order: by tile, then owner/whole before contributions, contributions by CTA.
  std::stable_sort(segs.begin(), segs.end(), [](const Segment& x, const Segment& y) {
    if (x.tile != y.tile) return x.tile < y.tile;
    if ((x.role == ROLE_CONTRIB) != (y.role == ROLE_CONTRIB)) return x.role != ROLE_CONTRIB;
    return x.cta < y.cta;
  });
  std::vector<char> covered(static_cast<size_t>(tiles * iters), 0);
  for (const Segment& s : segs)
    for (int64_t k = s.k0; k < s.k1; ++k) {
      if (covered[s.tile * iters + k]) return 2;
      covered[s.tile * iters + k] = 1;
    }
  for (char c : covered)
    if (!c) return 3;
  for (int64_t i = 0; i < M * N; ++i) out[i] = 0.0;
  for (const Segment& s : segs) {
    const int64_t tm = s.tile / tiles_n, tn = s.tile % tiles_n;
    const int64_t kb = s.k0 * BK, ke = std::min(K, s.k1 * BK);
    for (int64_t m = tm * BM; m < std::min(M, (tm + 1) * BM); ++m)
      for (int64_t n = tn * BN; n < std::min(N, (tn + 1) * BN); ++n) {
        double partial = 0.0;
        for (int64_t k = kb; k < ke; ++k)
          partial = partial + bf16_value(A[m * K + k]) * bf16_value(B[k * N + n]);
        out[m * N + n] = out[m * N + n] + partial;
      }
  }
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) out[m * N + n] = out[m * N + n] + bias_value(bias, bias_dtype, n);
  return 0;
}

int oracle_hardware_threads(void) { return worker_count(0); }

}  // extern "C"
