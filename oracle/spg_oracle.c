/*
 * Plain CPU oracle for the scaled low-precision linear-layer GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library product calls this file:
 * only the test suite, the smoke check and the CPU-baseline leg of the bench
 * load it.  It shares no code, header, table or constant with the CUDA path.
 *
 * What it computes, and where each step is defined:
 *
 *  - E4M3FN and E2M1 code decode, written from the format definitions
 *    (sign / exponent / mantissa fields; E4M3FN has no infinity, 0x7F and
 *    0xFF are NaN, the largest finite value is 448; E2M1 magnitudes are
 *    {0, 0.5, 1, 1.5, 2, 3, 4, 6}).  The pages only name the formats: "FP8
 *    E4M3 row-scaled A8 GEMM" (ninfer PR #167, opening paragraph) and "E2M1
 *    codes with an E4M3 scale per 16 elements" (ninfer PR #160, body).
 *  - Encoders: round-to-nearest-even onto the finite grid with saturation,
 *    found by searching the exact decode table (nearest value, ties to the
 *    code whose mantissa LSB is 0).
 *  - FP8 row quantizer: per row, amax, s = amax/448 in IEEE fp32, codes of
 *    x/s (ninfer PR #167, "What actually changes": one scale per activation
 *    row and per weight row).
 *  - FP8 per-tensor quantizer: the same with one amax over the tensor
 *    (AstrAI fp8 gemm.cuh commit log, quantize bullets).
 *  - NVFP4 quantizer: global g = amax/(448*6), one E4M3 scale per 16
 *    K-elements encoding (amax_b/6)/g, E2M1 codes of x/(dec(sf)*g)
 *    (ninfer PR #160, body: E2M1 codes with an E4M3 scale per 16 elements).
 *  - GEMMs: Y = dequant(A) . dequant(W)^T with the dot product accumulated
 *    EXACTLY in 64-bit integer fixed point (every decoded product is an
 *    integer multiple of 2^-18 for E4M3 and 2^-20 for scaled E2M1), converted
 *    to fp64 once, then the fp32 scales and the epilogue applied in fp64.
 *    Epilogues: linear, linear_add (bf16 residual), linear_swiglu over
 *    interleaved gate/up columns (ninfer PR #167, opening paragraph: the five
 *    call sites linear, linear_add, linear_swiglu ...).
 *  - Per-tensor FP8 GEMM in NT / NN / TN layouts with batch strides (AstrAI
 *    fp8 gemm.cuh commit log, first bullet: 3D operands, batch strides,
 *    size-1 batches broadcast with stride 0, .t() views as layout tags).
 *  - Optional fused bias per output column, added after the scales and
 *    before the epilogue (AstrAI fp8 gemm.cuh commit log, bias bullets).
 *
 * fp32 steps are written as C float operations; the file must be compiled
 * without fast-math and with -ffp-contract=off so every fp32 operation is a
 * single IEEE-rounded operation.
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define SPG_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------ */
/* bf16 -> float (exact: bf16 is the top half of an fp32)              */
/* ------------------------------------------------------------------ */
static float bf16_to_float(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ------------------------------------------------------------------ */
/* Code decode, from the format definitions                            */
/* ------------------------------------------------------------------ */

/* E4M3FN: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa.
 * Exponent field 0 is subnormal: (m/8) * 2^-6.  No infinities; the codes
 * with all exponent and mantissa bits set (0x7F, 0xFF) are NaN. */
SPG_EXPORT double spg_oracle_e4m3_value(uint32_t code) {
  code &= 0xFFu;
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  if (e == 0xF && m == 0x7) return NAN;
  double mag;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6);
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -mag : mag;
}

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent 0 is subnormal: m * 0.5.  Every code is finite. */
SPG_EXPORT double spg_oracle_e2m1_value(uint32_t code) {
  code &= 0xFu;
  int sign = (code >> 3) & 1;
  int e = (code >> 1) & 0x3;
  int m = code & 0x1;
  double mag;
  if (e == 0)
    mag = 0.5 * (double)m;
  else
    mag = ldexp(1.0 + 0.5 * (double)m, e - 1);
  return sign ? -mag : mag;
}

/* ------------------------------------------------------------------ */
/* Encoders: nearest finite value of the decode table, ties to even    */
/* ------------------------------------------------------------------ */

/* Round |x| to the nearest of the non-negative finite magnitudes held by
 * codes 0..max_code (ascending by code, as both formats are), ties to the
 * even code.  Values at or above the largest magnitude saturate to it.
 * A binary search finds the neighbours c, c+1 with mags[c] <= |x| <
 * mags[c+1]; the nearer one wins. */
static uint32_t nearest_magnitude_code(double ax, const double* mags,
                                       uint32_t max_code) {
  if (ax >= mags[max_code]) return max_code;
  if (ax <= mags[0]) return 0;
  uint32_t lo = 0, hi = max_code; /* mags[lo] <= ax < mags[hi] */
  while (hi - lo > 1) {
    uint32_t mid = (lo + hi) / 2;
    if (mags[mid] <= ax)
      lo = mid;
    else
      hi = mid;
  }
  double d_lo = ax - mags[lo], d_hi = mags[hi] - ax;
  if (d_lo < d_hi) return lo;
  if (d_hi < d_lo) return hi;
  return (lo & 1u) == 0 ? lo : hi;
}

static double g_e4m3_mag[127];
static double g_e2m1_mag[8];
static int g_tables_ready = 0;

static void ensure_tables(void) {
  if (g_tables_ready) return;
  for (uint32_t c = 0; c < 127; ++c) g_e4m3_mag[c] = spg_oracle_e4m3_value(c);
  for (uint32_t c = 0; c < 8; ++c) g_e2m1_mag[c] = spg_oracle_e2m1_value(c);
  g_tables_ready = 1;
}

/* E4M3FN, round-to-nearest-even, saturating to +-448.  The sign bit is
 * copied from x, so a negative value that rounds to zero gives 0x80.
 * NaN input is outside the contract. */
SPG_EXPORT uint32_t spg_oracle_e4m3_encode(double x) {
  ensure_tables();
  uint32_t mag = nearest_magnitude_code(fabs(x), g_e4m3_mag, 126);
  return (signbit(x) ? 0x80u : 0u) | mag;
}

/* E2M1, round-to-nearest-even, saturating to +-6; sign copied from x. */
SPG_EXPORT uint32_t spg_oracle_e2m1_encode(double x) {
  ensure_tables();
  uint32_t mag = nearest_magnitude_code(fabs(x), g_e2m1_mag, 7);
  return (signbit(x) ? 0x8u : 0u) | mag;
}

/* ------------------------------------------------------------------ */
/* Quantizers                                                          */
/* ------------------------------------------------------------------ */

static float amax_bf16(const uint16_t* x, int64_t n) {
  float a = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float v = fabsf(bf16_to_float(x[i]));
    if (v > a) a = v;
  }
  return a;
}

/* One row (or a whole tensor) to E4M3 codes with the scale s = amax/448.
 * An all-zero input stores s = 1 (its codes are then the signed zeros of
 * x / 1). */
static void fp8_encode_with_scale(const uint16_t* x, int64_t n, float amax,
                                  uint8_t* codes, float* s_out) {
  float s = (amax == 0.0f) ? 1.0f : amax / 448.0f;
  *s_out = s;
  for (int64_t i = 0; i < n; ++i) {
    float q = bf16_to_float(x[i]) / s;
    codes[i] = (uint8_t)spg_oracle_e4m3_encode((double)q);
  }
}

/* FP8 row quantizer: x [rows, K] bf16 row-major -> codes [rows, K],
 * scales [rows] fp32. */
SPG_EXPORT void spg_oracle_quantize_fp8_rows(const uint16_t* x, int64_t rows,
                                             int64_t K, uint8_t* codes,
                                             float* scales) {
  ensure_tables();
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const uint16_t* xr = x + r * K;
    fp8_encode_with_scale(xr, K, amax_bf16(xr, K), codes + r * K, scales + r);
  }
}

/* FP8 per-tensor quantizer: one scale for all numel values. */
SPG_EXPORT void spg_oracle_quantize_fp8_tensor(const uint16_t* x, int64_t numel,
                                               uint8_t* codes, float* scale) {
  ensure_tables();
  fp8_encode_with_scale(x, numel, amax_bf16(x, numel), codes, scale);
}

/* Delayed scaling with an amax history ring (AstrAI fp8 gemm.cuh commit log,
 * scale-ring bullets: the quantizer folds this call's amax into hist[idx],
 * reduces the window and publishes the next scale).  One call:
 *   scale_used = *scale                      (the scale published last time)
 *   codes      = E4M3(x / scale_used)         (IEEE fp32 division, RNE, satfinite)
 *   hist[*idx] = amax(x);  *idx = (*idx + 1) % history
 *   *scale     = max(hist) / 448, or 1 when max(hist) == 0   (next call's scale)
 * hist starts all zero, *idx at 0 and *scale at the caller's initial scale. */
SPG_EXPORT void spg_oracle_fp8_delayed_step(const uint16_t* x, int64_t numel, uint8_t* codes,
                                            float* hist, int history, int32_t* idx,
                                            float* scale, float* scale_used) {
  ensure_tables();
  const float s = *scale;
  *scale_used = s;
  for (int64_t i = 0; i < numel; ++i) {
    float q = bf16_to_float(x[i]) / s;
    codes[i] = (uint8_t)spg_oracle_e4m3_encode((double)q);
  }
  hist[*idx] = amax_bf16(x, numel);
  *idx = (*idx + 1) % history;
  float m = 0.0f;
  for (int h = 0; h < history; ++h)
    if (hist[h] > m) m = hist[h];
  *scale = (m == 0.0f) ? 1.0f : m / 448.0f;
}

/* NVFP4 global scale g = amax(tensor) / (448 * 6); 1 for an all-zero tensor. */
SPG_EXPORT float spg_oracle_nvfp4_global_scale(const uint16_t* x, int64_t numel) {
  float amax = amax_bf16(x, numel);
  if (amax == 0.0f) return 1.0f;
  return amax / 2688.0f;
}

/* NVFP4 block quantizer.  x [rows, K] bf16 (K a multiple of 16), global
 * scale g.  Per 16-element block along K:
 *   sf   = E4M3((amax_b / 6) / g)            (two IEEE fp32 divisions)
 *   d    = dec(sf) * g                       (IEEE fp32 multiply)
 *   code = E2M1(x / d), or 0 when d == 0
 * codes [rows, K/2]: element 2i in the low nibble, 2i+1 in the high nibble.
 * sf [rows, K/16] row-major. */
SPG_EXPORT void spg_oracle_quantize_nvfp4(const uint16_t* x, int64_t rows,
                                          int64_t K, float g, uint8_t* codes,
                                          uint8_t* sf) {
  ensure_tables();
  const int64_t nb = K / 16;
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint16_t* xb = x + r * K + b * 16;
      float amax_b = amax_bf16(xb, 16);
      float t = (amax_b / 6.0f) / g;
      uint32_t sfc = spg_oracle_e4m3_encode((double)t);
      sf[r * nb + b] = (uint8_t)sfc;
      float d = (float)spg_oracle_e4m3_value(sfc) * g;
      uint8_t nib[16];
      for (int i = 0; i < 16; ++i) {
        if (d == 0.0f) {
          nib[i] = 0;
        } else {
          float q = bf16_to_float(xb[i]) / d;
          nib[i] = (uint8_t)spg_oracle_e2m1_encode((double)q);
        }
      }
      for (int i = 0; i < 8; ++i)
        codes[r * (K / 2) + b * 8 + i] = (uint8_t)(nib[2 * i] | (nib[2 * i + 1] << 4));
    }
  }
}

/* ------------------------------------------------------------------ */
/* Exact integer images of decoded values                              */
/* ------------------------------------------------------------------ */

static int is_e4m3_nan(uint32_t code) { return (code & 0x7Fu) == 0x7Fu; }

/* dec(E4M3 code) * 2^9 is an integer for every finite code (the smallest
 * step, the subnormal 2^-9, sets the unit). */
static int64_t e4m3_units(uint32_t code) {
  return (int64_t)ldexp(spg_oracle_e4m3_value(code), 9);
}
/* dec(E2M1 code) * 2 is an integer. */
static int64_t e2m1_units(uint32_t code) {
  return (int64_t)ldexp(spg_oracle_e2m1_value(code), 1);
}

enum { EPI_LINEAR = 0, EPI_ADD = 1, EPI_SWIGLU = 2 };

/* Bias of output column n (fused bias, AstrAI fp8 gemm.cuh commit log: bf16
 * bias, or E4M3 bias storage dequantized with bias_scale after the operand
 * scaling): bias_kind 0 none, 1 bf16 values, 2 E4M3 codes times bias_scale
 * (the product rounded to fp32). */
static double bias_value(const void* bias, int bias_kind, float bias_scale, int64_t n) {
  if (bias_kind == 1) return (double)bf16_to_float(((const uint16_t*)bias)[n]);
  if (bias_kind == 2) {
    float d = (float)spg_oracle_e4m3_value(((const uint8_t*)bias)[n]) * bias_scale;
    return (double)d;
  }
  return 0.0;
}

/* Apply the epilogue to one output row.  y [N] holds the scaled fp64
 * linear output of that row; out gets N values (linear / add) or N/2
 * (SwiGLU: gate = column 2j, up = column 2j+1). */
static void epilogue_row(const double* y, int64_t N, int epi,
                         const uint16_t* residual_row, double* out) {
  if (epi == EPI_SWIGLU) {
    for (int64_t j = 0; j < N / 2; ++j) {
      double gate = y[2 * j], up = y[2 * j + 1];
      out[j] = gate / (1.0 + exp(-gate)) * up;
    }
  } else if (epi == EPI_ADD) {
    for (int64_t n = 0; n < N; ++n) out[n] = y[n] + (double)bf16_to_float(residual_row[n]);
  } else {
    for (int64_t n = 0; n < N; ++n) out[n] = y[n];
  }
}

/* ------------------------------------------------------------------ */
/* FP8 row-scaled GEMM                                                 */
/* ------------------------------------------------------------------ */

/* Y[t, :] for the nrows row indices in rows[] (all rows when rows is NULL,
 * nrows = T).  A [T,K] codes, sa [T], W [N,K] codes, sw [N], residual
 * [T,N] bf16 (linear_add only).  out is [nrows, N_out] fp64 with N_out = N
 * or N/2 for SwiGLU.  acc_out, when not NULL, receives the exact unscaled
 * dot products [nrows, N]. */
SPG_EXPORT void spg_oracle_fp8_rowscaled_gemm_bias(
    const uint8_t* A, const float* sa, const uint8_t* W, const float* sw,
    const void* bias, int bias_kind, float bias_scale,
    const uint16_t* residual, int64_t T, int64_t N, int64_t K, int epi,
    const int64_t* rows, int64_t nrows, double* out, double* acc_out) {
  ensure_tables();
  (void)T;
  int64_t lut[256];
  for (int c = 0; c < 256; ++c) lut[c] = is_e4m3_nan((uint32_t)c) ? 0 : e4m3_units((uint32_t)c);
  const int64_t n_out = (epi == EPI_SWIGLU) ? N / 2 : N;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t t = rows ? rows[i] : i;
    const uint8_t* a = A + t * K;
    double* y = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int64_t n = 0; n < N; ++n) {
      const uint8_t* w = W + n * K;
      int64_t acc = 0;
      int nan = 0;
      for (int64_t k = 0; k < K; ++k) {
        acc += lut[a[k]] * lut[w[k]];
        nan |= is_e4m3_nan(a[k]) | is_e4m3_nan(w[k]);
      }
      double dot = nan ? NAN : ldexp((double)acc, -18);
      if (acc_out) acc_out[i * N + n] = dot;
      y[n] = dot * (double)sa[t] * (double)sw[n] + bias_value(bias, bias_kind, bias_scale, n);
    }
    epilogue_row(y, N, epi, residual ? residual + t * N : NULL, out + i * n_out);
    free(y);
  }
}

SPG_EXPORT void spg_oracle_fp8_rowscaled_gemm(
    const uint8_t* A, const float* sa, const uint8_t* W, const float* sw,
    const uint16_t* residual, int64_t T, int64_t N, int64_t K, int epi,
    const int64_t* rows, int64_t nrows, double* out, double* acc_out) {
  spg_oracle_fp8_rowscaled_gemm_bias(A, sa, W, sw, NULL, 0, 0.0f, residual, T, N, K, epi, rows,
                                     nrows, out, acc_out);
}

/* ------------------------------------------------------------------ */
/* NVFP4 block-scaled GEMM                                             */
/* ------------------------------------------------------------------ */

/* A codes [T, K/2] packed E2M1, sfA [T, K/16] row-major E4M3, gA scalar;
 * W codes [N, K/2], sfW [N, K/16], gW.  Y = (sum_k dec(A)dec(sfA)dec(W)
 * dec(sfW)) * gA * gW, then the epilogue.  The sum is exact in units of
 * 2^-20.  Same row selection and outputs as the FP8 function. */
SPG_EXPORT void spg_oracle_nvfp4_gemm_bias(
    const uint8_t* A, const uint8_t* sfA, float gA, const uint8_t* W,
    const uint8_t* sfW, float gW, const void* bias, int bias_kind, float bias_scale,
    const uint16_t* residual, int64_t T,
    int64_t N, int64_t K, int epi, const int64_t* rows, int64_t nrows,
    double* out, double* acc_out) {
  ensure_tables();
  (void)T;
  int64_t sf_lut[256], v_lut[16];
  for (int c = 0; c < 256; ++c) sf_lut[c] = is_e4m3_nan((uint32_t)c) ? 0 : e4m3_units((uint32_t)c);
  for (int c = 0; c < 16; ++c) v_lut[c] = e2m1_units((uint32_t)c);
  const int64_t nb = K / 16;
  const int64_t n_out = (epi == EPI_SWIGLU) ? N / 2 : N;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < nrows; ++i) {
    int64_t t = rows ? rows[i] : i;
    double* y = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
    for (int64_t n = 0; n < N; ++n) {
      int64_t acc = 0;
      int nan = 0;
      for (int64_t k = 0; k < K; ++k) {
        uint32_t ca = (A[t * (K / 2) + k / 2] >> ((k & 1) * 4)) & 0xF;
        uint32_t cw = (W[n * (K / 2) + k / 2] >> ((k & 1) * 4)) & 0xF;
        uint32_t sa_c = sfA[t * nb + k / 16], sw_c = sfW[n * nb + k / 16];
        int64_t av = v_lut[ca] * sf_lut[sa_c];
        int64_t wv = v_lut[cw] * sf_lut[sw_c];
        acc += av * wv;
        nan |= is_e4m3_nan(sa_c) | is_e4m3_nan(sw_c);
      }
      double dot = nan ? NAN : ldexp((double)acc, -20);
      if (acc_out) acc_out[i * N + n] = dot;
      y[n] = dot * (double)gA * (double)gW + bias_value(bias, bias_kind, bias_scale, n);
    }
    epilogue_row(y, N, epi, residual ? residual + t * N : NULL, out + i * n_out);
    free(y);
  }
}

SPG_EXPORT void spg_oracle_nvfp4_gemm(
    const uint8_t* A, const uint8_t* sfA, float gA, const uint8_t* W,
    const uint8_t* sfW, float gW, const uint16_t* residual, int64_t T,
    int64_t N, int64_t K, int epi, const int64_t* rows, int64_t nrows,
    double* out, double* acc_out) {
  spg_oracle_nvfp4_gemm_bias(A, sfA, gA, W, sfW, gW, NULL, 0, 0.0f, residual, T, N, K, epi, rows,
                             nrows, out, acc_out);
}

/* ------------------------------------------------------------------ */
/* Per-tensor FP8 GEMM, NT / NN / TN, batched                          */
/* ------------------------------------------------------------------ */

/* C[b] (M x N) = sA * sB * opA(A[b]) * opB(B[b]) with
 *   layout "NT": A[b] is [M,K], B[b] is [N,K]   (C = A . B^T)
 *   layout "NN": A[b] is [M,K], B[b] is [K,N]   (C = A . B)
 *   layout "TN": A[b] is [K,M], B[b] is [K,N]   (C = A^T . B)
 * All row-major with the natural leading dimension; batch b starts at
 * b * strideA / b * strideB elements (stride 0 broadcasts one matrix).
 * out is [batch, M, N] fp64 (only rows in rows[] when rows != NULL, then
 * out is [batch, nrows, N]). */
SPG_EXPORT void spg_oracle_fp8_tensor_gemm_bias(
    char la, char lb, int64_t batch, const uint8_t* A, int64_t strideA,
    float sA, const uint8_t* B, int64_t strideB, float sB, const void* bias,
    int bias_kind, float bias_scale, int64_t M,
    int64_t N, int64_t K, const int64_t* rows, int64_t nrows, double* out) {
  ensure_tables();
  int64_t lut[256];
  for (int c = 0; c < 256; ++c) lut[c] = is_e4m3_nan((uint32_t)c) ? 0 : e4m3_units((uint32_t)c);
  const int64_t nr = rows ? nrows : M;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t b = 0; b < batch; ++b) {
    for (int64_t i = 0; i < nr; ++i) {
      int64_t m = rows ? rows[i] : i;
      const uint8_t* Ab = A + b * strideA;
      const uint8_t* Bb = B + b * strideB;
      for (int64_t n = 0; n < N; ++n) {
        int64_t acc = 0;
        int nan = 0;
        for (int64_t k = 0; k < K; ++k) {
          uint8_t a = (la == 'T') ? Ab[k * M + m] : Ab[m * K + k];
          uint8_t w = (lb == 'N') ? Bb[k * N + n] : Bb[n * K + k];
          acc += lut[a] * lut[w];
          nan |= is_e4m3_nan(a) | is_e4m3_nan(w);
        }
        out[(b * nr + i) * N + n] =
            nan ? NAN
                : ldexp((double)acc, -18) * (double)sA * (double)sB +
                      bias_value(bias, bias_kind, bias_scale, n);
      }
    }
  }
}

SPG_EXPORT void spg_oracle_fp8_tensor_gemm(
    char la, char lb, int64_t batch, const uint8_t* A, int64_t strideA,
    float sA, const uint8_t* B, int64_t strideB, float sB, int64_t M,
    int64_t N, int64_t K, const int64_t* rows, int64_t nrows, double* out) {
  spg_oracle_fp8_tensor_gemm_bias(la, lb, batch, A, strideA, sA, B, strideB, sB, NULL, 0, 0.0f,
                                  M, N, K, rows, nrows, out);
}
