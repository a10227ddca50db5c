/*
 * qk_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * The plain, slow, obviously correct CPU oracle for the quantized GEMM
 *
 *     C[m,n] = bf16( epilogue( sum_k A[m,k] * B[n,k] ) )
 *
 * with A [M,K] and B [N,K] both K-major.  Only the test suite, the smoke
 * check and the benchmark's CPU-baseline / reference arm may load this
 * library.  It shares no code, header, table or constant with the CUDA path
 * under block_scaled_precision_tcgen05_gb300/csrc, and neither side includes
 * the other.
 *
 * Sources (web pages; cited by title and section):
 *  [CK174]  comfy-kitchen PR #174 "Optimize HIP WMMA INT8 GEMM staging,
 *           epilogue, and deep-K tiling": Summary (rowwise epilogue with
 *           cached scales and bias; signed zero without bias), Validation
 *           (the results match the reference bit for bit, zero error), and
 *           the update "Keep the cached INT8 epilogue scale order exact"
 *           ((acc*sa)*sb, never acc*(sa*sb)); the update "rebased onto
 *           v0.2.38" (the INT8 kernel specialization serves bf16, fp16 and
 *           fp32 outputs; read as the same x rounded per IEEE binary16 or
 *           kept).
 *  [MORI806] ROCm/mori PR #806 "perf(gemm-ar): mxfp8 with row-major scales
 *           staged through LDS", section "What": 32-wide ue8m0 scales held
 *           raw, row-major, one byte per 32 K-elements.
 *  [FLY990] ROCm/FlyDSL PR #990 "[fp4_gemm_4wave] MXFP4 GEMM perf optimize":
 *           MXFP4 = e2m1 elements with per-1x32 ue8m0 scales, checked
 *           against an MXFP4-dequant reference.
 *  [AITER6262] ROCm/aiter PR #6262, "Technical Details": FP8 A8W8 GEMM with
 *           per-token x per-channel scales; its gemm_a4w4 signature takes
 *           optional per-tensor global A and B scales for NVFP4.
 *  [MORI806-RAW] ROCm/mori PR #806, section "What" and the review thread's
 *           scale reader (B_scale read with rows_per 32): the mxfp8_raw form
 *           takes B's scales as [N/32, K/32], one byte per 32 rows x 32 K.
 *  [MORI806-BS] ROCm/mori PR #806, the pipeline-drain fix's measurements:
 *           a "blockscale" FP8 GEMM kind (16384x7168x2048) beside ptpc and
 *           mxfp8.  The block sizes are not stated on the page.
 * The element formats (E4M3FN, E2M1, UE8M0) are not defined on the pages;
 * they are restated here from the OCP Microscaling (MX) v1.0 format
 * definitions: sign/exponent/mantissa bit fields with the stated biases.
 * NVFP4 is not defined on the pages either; it is restated from NVIDIA's
 * published format: E2M1 elements, one unsigned E4M3 (UE4M3) scale per 16
 * consecutive K-elements, and one fp32 scale per tensor.  "Blockscale" FP8
 * is read as the DeepSeek-V3 layout: fp32 scales per 1x128 (row, K-block)
 * of A and per 128x128 (N-block, K-block) of B.
 *
 * Arithmetic rules of this file:
 *  - INT8 accumulates in int64 and asserts the int32 range.
 *  - E4M3 / E2M1 / UE8M0 are decoded by lookup tables built once from the
 *    bit-field definitions.
 *  - MX and FP8 accumulate the exact products in fp64 (every product of
 *    decoded elements and power-of-two scales is exact in fp64).
 *  - The INT8 epilogue is evaluated in IEEE fp32 with round-to-nearest-even
 *    at every operation, in the order the pages fix.  The bf16 and binary16
 *    output conversions are written from the formats' definitions.  Build with
 *    -ffp-contract=off and without -ffast-math so no multiply-add is fused.
 *  - Parallelism (OpenMP) is over independent output elements only; each
 *    element's sum runs k = 0..K-1 in order.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QKO_OK 0
#define QKO_ERR_ARG 1
#define QKO_ERR_INT32 2

#define QKO_FMT_MXFP8_E4M3 1
#define QKO_FMT_MXFP4_E2M1 2

#define QKO_OUT_BF16 0
#define QKO_OUT_FP16 1
#define QKO_OUT_FP32 2

/* ------------------------------------------------------------------ */
/* Format decode tables (OCP MX v1.0 element and scale formats)        */
/* ------------------------------------------------------------------ */

static double g_e4m3[256];
static double g_e2m1[16];
static double g_ue8m0[256];
static double g_ue4m3[256];
static int g_tables_ready = 0;

/* E4M3FN: bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0 mantissa.
 * Exponent field 0 is subnormal: (m/8) * 2^(1-7).  The all-ones pattern
 * S.1111.111 is NaN; there is no infinity, so S.1111.110 = 448 is the
 * largest magnitude. */
static double e4m3_from_fields(unsigned code) {
  unsigned s = (code >> 7) & 1u, e = (code >> 3) & 15u, m = code & 7u;
  double mag;
  if (e == 15u && m == 7u) return NAN;
  if (e == 0u)
    mag = ldexp((double)m / 8.0, 1 - 7);
  else
    mag = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
  return s ? -mag : mag;
}

/* E2M1: bit 3 sign, bits 2..1 exponent (bias 1), bit 0 mantissa.
 * Exponent field 0 is subnormal: (m/2) * 2^(1-1).  No NaN, no infinity. */
static double e2m1_from_fields(unsigned code) {
  unsigned s = (code >> 3) & 1u, e = (code >> 1) & 3u, m = code & 1u;
  double mag;
  if (e == 0u)
    mag = ldexp((double)m / 2.0, 1 - 1);
  else
    mag = ldexp(1.0 + (double)m / 2.0, (int)e - 1);
  return s ? -mag : mag;
}

/* UE8M0: unsigned, 8-bit exponent, bias 127, no mantissa.  0xFF is NaN. */
static double ue8m0_from_fields(unsigned code) {
  if (code == 255u) return NAN;
  return ldexp(1.0, (int)code - 127);
}

/* UE4M3 (NVFP4 block scale): E4M3FN without the sign, so bit 7 is not part
 * of the format.  Bits 6..3 exponent (bias 7), bits 2..0 mantissa, exponent
 * field 0 subnormal, 0x7F NaN, 0x7E = 448 the largest.  Codes with bit 7
 * set are outside the format and decode to NaN here. */
static double ue4m3_from_fields(unsigned code) {
  unsigned e = (code >> 3) & 15u, m = code & 7u;
  if (code > 0x7Eu) return NAN;
  if (e == 0u) return ldexp((double)m / 8.0, 1 - 7);
  return ldexp(1.0 + (double)m / 8.0, (int)e - 7);
}

static void build_tables(void) {
  if (g_tables_ready) return;
  for (unsigned c = 0; c < 256u; ++c) g_e4m3[c] = e4m3_from_fields(c);
  for (unsigned c = 0; c < 16u; ++c) g_e2m1[c] = e2m1_from_fields(c);
  for (unsigned c = 0; c < 256u; ++c) g_ue8m0[c] = ue8m0_from_fields(c);
  for (unsigned c = 0; c < 256u; ++c) g_ue4m3[c] = ue4m3_from_fields(c);
  g_tables_ready = 1;
}

void qko_init(void) { build_tables(); }

double qko_decode_e4m3(uint8_t code) { build_tables(); return g_e4m3[code]; }
double qko_decode_e2m1(uint8_t nibble) { build_tables(); return g_e2m1[nibble & 15u]; }
double qko_decode_ue8m0(uint8_t code) { build_tables(); return g_ue8m0[code]; }
double qko_decode_ue4m3(uint8_t code) { build_tables(); return g_ue4m3[code]; }

/* ------------------------------------------------------------------ */
/* bf16                                                                */
/* ------------------------------------------------------------------ */

/* fp32 -> bf16 with round-to-nearest, ties to even, on the bit pattern.
 * Overflow rounds to +-Inf; NaN stays NaN (quiet bit set, sign kept). */
uint16_t qko_f32_to_bf16_rne(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  if ((u & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lsb = (u >> 16) & 1u;
  u += 0x7fffu + lsb;
  return (uint16_t)(u >> 16);
}

/* fp32 -> IEEE binary16 with round-to-nearest, ties to even, from the value:
 * the result is the multiple of the binary16 spacing of x's binade (2^(e-10)
 * for |x| in [2^e, 2^(e+1)), e >= -14; 2^-24 below 2^-14, the subnormals)
 * nearest to |x|, ties to the even multiple.  A result above 65504 is +-Inf
 * (from |x| >= 65520, the midpoint to 2^16).  The sign is kept (-0 stays
 * -0); NaN stays NaN (quiet).  The division by the spacing and the product
 * back are exact in double. */
uint16_t qko_f32_to_f16_rne(float x) {
  uint32_t u;
  memcpy(&u, &x, sizeof u);
  const uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  if (x != x) return (uint16_t)(sign | 0x7e00u);
  double v = fabs((double)x);
  if (isinf(v)) return (uint16_t)(sign | 0x7c00u);
  if (v == 0.0) return sign;
  int e2;
  (void)frexp(v, &e2);                 /* v = f * 2^e2, f in [0.5, 1): binade e2 - 1 */
  int e = e2 - 1;
  if (e < -14) e = -14;                /* subnormals share the spacing 2^-24 */
  const double spacing = ldexp(1.0, e - 10);
  const double r = nearbyint(v / spacing) * spacing;  /* ties to even (default rounding mode) */
  if (r > 65504.0) return (uint16_t)(sign | 0x7c00u);
  if (r < ldexp(1.0, -14)) return (uint16_t)(sign | (uint16_t)(r / ldexp(1.0, -24)));
  int re2;
  const double f = frexp(r, &re2);     /* r = f * 2^re2, f in [0.5, 1) */
  const uint32_t biased = (uint32_t)(re2 - 1 + 15);
  const uint32_t mant = (uint32_t)((2.0 * f - 1.0) * 1024.0);
  return (uint16_t)(sign | (biased << 10) | mant);
}

float qko_bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float x;
  memcpy(&x, &u, sizeof x);
  return x;
}

/* ------------------------------------------------------------------ */
/* Encoders (used only by tests that pin the OCP encode rules)         */
/* ------------------------------------------------------------------ */

/* Nearest finite code by exhaustive search over the decode table; ties go
 * to the code whose mantissa LSB is 0 (round half to even).  Magnitudes
 * above the largest finite value saturate to it. */
static unsigned nearest_code(const double* table, unsigned ncodes_pos, double mag) {
  unsigned best = 0;
  double best_err = INFINITY;
  for (unsigned c = 0; c < ncodes_pos; ++c) {
    double v = table[c];
    if (isnan(v)) continue;
    double err = fabs(v - mag);
    if (err < best_err || (err == best_err && (c & 1u) == 0u)) {
      best = c;
      best_err = err;
    }
  }
  return best;
}

uint8_t qko_encode_e4m3(double x) {
  build_tables();
  if (isnan(x)) return 0x7f;
  unsigned s = signbit(x) ? 0x80u : 0u;
  double mag = fabs(x);
  if (mag >= 448.0) return (uint8_t)(s | 0x7eu);
  return (uint8_t)(s | nearest_code(g_e4m3, 128u, mag));
}

uint8_t qko_encode_e2m1(double x) {
  build_tables();
  unsigned s = signbit(x) ? 0x8u : 0u;
  double mag = fabs(x);
  if (isnan(x)) mag = 6.0;
  if (mag >= 6.0) return (uint8_t)(s | 0x7u);
  return (uint8_t)(s | nearest_code(g_e2m1, 8u, mag));
}

/* One MX block of 32 values: shared exponent floor(log2(amax)) - emax_elem
 * (emax 8 for E4M3, 2 for E2M1), clamped to [-127, 127] and stored biased
 * by 127; an all-zero block takes exponent code 0.  Elements are v / 2^s,
 * rounded to nearest even and saturated.  E2M1 codes are returned one per
 * byte (not packed). */
void qko_mx_quantize_block(int fmt, const float* v, uint8_t* codes, uint8_t* scale_code) {
  build_tables();
  double amax = 0.0;
  for (int i = 0; i < 32; ++i) {
    double a = fabs((double)v[i]);
    if (a > amax) amax = a;
  }
  int emax = (fmt == QKO_FMT_MXFP8_E4M3) ? 8 : 2;
  int sexp;
  if (amax == 0.0) {
    sexp = -127;
  } else {
    int e;
    (void)frexp(amax, &e); /* amax = f * 2^e, f in [0.5, 1) => floor(log2) = e-1 */
    sexp = (e - 1) - emax;
    if (sexp < -127) sexp = -127;
    if (sexp > 127) sexp = 127;
  }
  *scale_code = (uint8_t)(sexp + 127);
  for (int i = 0; i < 32; ++i) {
    double q = ldexp((double)v[i], -sexp);
    codes[i] = (fmt == QKO_FMT_MXFP8_E4M3) ? qko_encode_e4m3(q) : qko_encode_e2m1(q);
  }
}

/* One row of per-token FP8 quantization (the step that feeds the FP8
 * per-token x per-channel GEMM; ROCm/aiter PR #6262 "Technical Details",
 * ROCm/mori PR #806 "ptpc"): amax over the row, scale s = amax / 448 in fp32
 * (1 for an all-zero row), codes = E4M3(x / s) with the fp32 division
 * rounded to nearest even, then rounded to nearest even E4M3, saturated. */
void qko_ptpc_quantize_row(const float* x, int64_t K, uint8_t* codes, float* scale) {
  build_tables();
  float amax = 0.0f;
  for (int64_t k = 0; k < K; ++k) {
    float a = fabsf(x[k]);
    if (a > amax) amax = a;
  }
  float s = amax / 448.0f;
  if (amax == 0.0f) s = 1.0f;
  *scale = s;
  for (int64_t k = 0; k < K; ++k) {
    float q = x[k] / s;
    codes[k] = qko_encode_e4m3((double)q);
  }
}

/* ------------------------------------------------------------------ */
/* INT8 row/column-scaled GEMM  [CK174]                                */
/* ------------------------------------------------------------------ */

/* Fills out[(m-m0)*ldo + (n-n0)] for m in [m0,m1), n in [n0,n1).
 *  1. acc = sum_k (int64)A[m,k] * (int64)B[n,k]; must fit in int32.
 *  2. x   = (float)acc                      (fp32, round to nearest even)
 *  3. x   = x * sa[m];  x = x * sb[n]       (two fp32 roundings, that order)
 *  4. if bias: x = x + (float)bias[n]       (bf16 widened exactly; one add)
 *     without bias no add happens, so a -0 from step 3 survives.
 *  5. out = x in the output type: QKO_OUT_BF16 (uint16 bits, bf16 round to
 *     nearest even), QKO_OUT_FP16 (uint16 bits, binary16 round to nearest
 *     even) or QKO_OUT_FP32 (x itself).  The page's INT8 kernel
 *     specialization serves all three output types (update "rebased onto
 *     v0.2.38", its resources paragraph); bf16 is the one its numbers use.
 * acc_out (nullable) receives the int64 sums with the same indexing. */
int qko_gemm_int8_rowwise_out(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                              const uint16_t* bias, void* out, int out_type, int64_t ldo, int64_t M, int64_t N,
                              int64_t K, int64_t m0, int64_t m1, int64_t n0, int64_t n1,
                              int64_t* acc_out) {
  if (!A || !B || !sa || !sb || !out || M < 0 || N < 0 || K < 0) return QKO_ERR_ARG;
  if (m0 < 0 || n0 < 0 || m1 > M || n1 > N || m0 > m1 || n0 > n1 || ldo < n1 - n0) return QKO_ERR_ARG;
  if (out_type != QKO_OUT_BF16 && out_type != QKO_OUT_FP16 && out_type != QKO_OUT_FP32) return QKO_ERR_ARG;
  int bad = 0;
#pragma omp parallel for collapse(2) schedule(static) reduction(| : bad)
  for (int64_t m = m0; m < m1; ++m) {
    for (int64_t n = n0; n < n1; ++n) {
      const int8_t* a = A + m * K;
      const int8_t* b = B + n * K;
      int64_t acc = 0;
      for (int64_t k = 0; k < K; ++k) acc += (int64_t)a[k] * (int64_t)b[k];
      if (acc > INT32_MAX || acc < INT32_MIN) bad = 1;
      float x = (float)(int32_t)acc;
      x = x * sa[m];
      x = x * sb[n];
      if (bias) x = x + qko_bf16_to_f32(bias[n]);
      const int64_t o = (m - m0) * ldo + (n - n0);
      if (out_type == QKO_OUT_FP32)
        ((float*)out)[o] = x;
      else if (out_type == QKO_OUT_FP16)
        ((uint16_t*)out)[o] = qko_f32_to_f16_rne(x);
      else
        ((uint16_t*)out)[o] = qko_f32_to_bf16_rne(x);
      if (acc_out) acc_out[o] = acc;
    }
  }
  return bad ? QKO_ERR_INT32 : QKO_OK;
}

/* The bf16 output of qko_gemm_int8_rowwise_out. */
int qko_gemm_int8_rowwise(const int8_t* A, const int8_t* B, const float* sa, const float* sb,
                          const uint16_t* bias, uint16_t* out, int64_t ldo, int64_t M, int64_t N,
                          int64_t K, int64_t m0, int64_t m1, int64_t n0, int64_t n1,
                          int64_t* acc_out) {
  return qko_gemm_int8_rowwise_out(A, B, sa, sb, bias, out, QKO_OUT_BF16, ldo, M, N, K, m0, m1, n0, n1, acc_out);
}

/* ------------------------------------------------------------------ */
/* FP8 E4M3 per-token x per-channel GEMM  [AITER6262], [MORI806]       */
/* ------------------------------------------------------------------ */

/* ref[(m-m0)*ldr + (n-n0)] = (acc * sa[m]) * sb[n] (+ bias[n]) in fp64, where
 * acc = sum_k e4m3(A[m,k]) * e4m3(B[n,k]) accumulated in fp64.  This is the
 * value before the bf16 output rounding. */
int qko_gemm_fp8_rowwise(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                         const uint16_t* bias, double* ref, int64_t ldr, int64_t M, int64_t N,
                         int64_t K, int64_t m0, int64_t m1, int64_t n0, int64_t n1) {
  if (!A || !B || !sa || !sb || !ref || M < 0 || N < 0 || K < 0) return QKO_ERR_ARG;
  if (m0 < 0 || n0 < 0 || m1 > M || n1 > N || m0 > m1 || n0 > n1 || ldr < n1 - n0) return QKO_ERR_ARG;
  build_tables();
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = m0; m < m1; ++m) {
    for (int64_t n = n0; n < n1; ++n) {
      const uint8_t* a = A + m * K;
      const uint8_t* b = B + n * K;
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += g_e4m3[a[k]] * g_e4m3[b[k]];
      double x = acc * (double)sa[m] * (double)sb[n];
      if (bias) x += (double)qko_bf16_to_f32(bias[n]);
      ref[(m - m0) * ldr + (n - n0)] = x;
    }
  }
  return QKO_OK;
}

/* ------------------------------------------------------------------ */
/* MX block-scaled GEMM (MXFP8 E4M3, MXFP4 E2M1)  [MORI806], [FLY990]  */
/* ------------------------------------------------------------------ */

/* Element k of row r of an operand.  MXFP8: one E4M3 code per byte.
 * MXFP4: two E2M1 codes per byte, element 2i in the low nibble and 2i+1 in
 * the high nibble; a row holds K/2 bytes. */
static double mx_elem(int fmt, const uint8_t* rowp, int64_t k) {
  if (fmt == QKO_FMT_MXFP8_E4M3) return g_e4m3[rowp[k]];
  uint8_t byte = rowp[k >> 1];
  uint8_t nib = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15u);
  return g_e2m1[nib];
}

/* ref[(m-m0)*ldr + (n-n0)] = sum_b 2^(sA[m,b]-127) * 2^(sB[n,b]-127)
 *                                * sum_{j<32} dec(A[m,32b+j]) * dec(B[n,32b+j])
 *                            (+ bias[n])
 * in fp64.  Scales are raw row-major bytes: sA [M, K/32], sB [N, K/32].
 * K must be a multiple of 32.  This is the value before bf16 rounding. */
int qko_gemm_mx(int fmt, const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB,
                const uint16_t* bias, double* ref, int64_t ldr, int64_t M, int64_t N, int64_t K,
                int64_t m0, int64_t m1, int64_t n0, int64_t n1) {
  if (fmt != QKO_FMT_MXFP8_E4M3 && fmt != QKO_FMT_MXFP4_E2M1) return QKO_ERR_ARG;
  if (!A || !sA || !B || !sB || !ref || M < 0 || N < 0 || K < 0 || (K % 32) != 0) return QKO_ERR_ARG;
  if (m0 < 0 || n0 < 0 || m1 > M || n1 > N || m0 > m1 || n0 > n1 || ldr < n1 - n0) return QKO_ERR_ARG;
  build_tables();
  const int64_t kb = K / 32;
  const int64_t row_bytes = (fmt == QKO_FMT_MXFP8_E4M3) ? K : K / 2;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = m0; m < m1; ++m) {
    for (int64_t n = n0; n < n1; ++n) {
      const uint8_t* a = A + m * row_bytes;
      const uint8_t* b = B + n * row_bytes;
      double acc = 0.0;
      for (int64_t blk = 0; blk < kb; ++blk) {
        double inner = 0.0;
        for (int64_t j = 0; j < 32; ++j) {
          int64_t k = blk * 32 + j;
          inner += mx_elem(fmt, a, k) * mx_elem(fmt, b, k);
        }
        acc += g_ue8m0[sA[m * kb + blk]] * g_ue8m0[sB[n * kb + blk]] * inner;
      }
      if (bias) acc += (double)qko_bf16_to_f32(bias[n]);
      ref[(m - m0) * ldr + (n - n0)] = acc;
    }
  }
  return QKO_OK;
}

/* MX block-scaled GEMM with 32x32 scale blocks for B  [MORI806-RAW]
 *
 * ref[(m-m0)*ldr + (n-n0)] = sum_b 2^(sA[m,b]-127) * 2^(sB32[n/32,b]-127)
 *                                * sum_{j<32} dec(A[m,32b+j]) * dec(B[n,32b+j])
 *                            (+ bias[n])
 * in fp64.  A's scales as in qko_gemm_mx, one per (row, 32 K): sA [M, K/32];
 * B's one per 32 rows and 32 K: sB32 [ceil(N/32), K/32], row n of B taking
 * scale row n / 32 (integer division; the last group may hold fewer than 32
 * rows).  K must be a multiple of 32.  This is the value before bf16
 * rounding. */
int qko_gemm_mx_b32(int fmt, const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB32,
                    const uint16_t* bias, double* ref, int64_t ldr, int64_t M, int64_t N, int64_t K,
                    int64_t m0, int64_t m1, int64_t n0, int64_t n1) {
  if (fmt != QKO_FMT_MXFP8_E4M3 && fmt != QKO_FMT_MXFP4_E2M1) return QKO_ERR_ARG;
  if (!A || !sA || !B || !sB32 || !ref || M < 0 || N < 0 || K < 0 || (K % 32) != 0) return QKO_ERR_ARG;
  if (m0 < 0 || n0 < 0 || m1 > M || n1 > N || m0 > m1 || n0 > n1 || ldr < n1 - n0) return QKO_ERR_ARG;
  build_tables();
  const int64_t kb = K / 32;
  const int64_t row_bytes = (fmt == QKO_FMT_MXFP8_E4M3) ? K : K / 2;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = m0; m < m1; ++m) {
    for (int64_t n = n0; n < n1; ++n) {
      const uint8_t* a = A + m * row_bytes;
      const uint8_t* b = B + n * row_bytes;
      const int64_t g = n / 32;  /* B's 32-row scale group */
      double acc = 0.0;
      for (int64_t blk = 0; blk < kb; ++blk) {
        double inner = 0.0;
        for (int64_t j = 0; j < 32; ++j) {
          int64_t k = blk * 32 + j;
          inner += mx_elem(fmt, a, k) * mx_elem(fmt, b, k);
        }
        acc += g_ue8m0[sA[m * kb + blk]] * g_ue8m0[sB32[g * kb + blk]] * inner;
      }
      if (bias) acc += (double)qko_bf16_to_f32(bias[n]);
      ref[(m - m0) * ldr + (n - n0)] = acc;
    }
  }
  return QKO_OK;
}

/* ------------------------------------------------------------------ */
/* NVFP4 block-scaled GEMM  [AITER6262] global scales                  */
/* ------------------------------------------------------------------ */

/* ref[(m-m0)*ldr + (n-n0)] =
 *     ga * gb * sum_b ue4m3(sA[m,b]) * ue4m3(sB[n,b])
 *                     * sum_{j<16} e2m1(A[m,16b+j]) * e2m1(B[n,16b+j])
 *     (+ bias[n])
 * in fp64.  A and B hold two E2M1 codes per byte (element 2i in the low
 * nibble), K/2 bytes per row; sA [M, K/16] and sB [N, K/16] are raw
 * row-major UE4M3 bytes; ga, gb are the per-tensor fp32 scales.  K must be a
 * multiple of 16.  This is the value before bf16 rounding. */
int qko_gemm_nvfp4(const uint8_t* A, const uint8_t* sA, const uint8_t* B, const uint8_t* sB, float ga,
                   float gb, const uint16_t* bias, double* ref, int64_t ldr, int64_t M, int64_t N, int64_t K,
                   int64_t m0, int64_t m1, int64_t n0, int64_t n1) {
  if (!A || !sA || !B || !sB || !ref || M < 0 || N < 0 || K < 0 || (K % 16) != 0) return QKO_ERR_ARG;
  if (m0 < 0 || n0 < 0 || m1 > M || n1 > N || m0 > m1 || n0 > n1 || ldr < n1 - n0) return QKO_ERR_ARG;
  build_tables();
  const int64_t kb = K / 16;
  const int64_t row_bytes = K / 2;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = m0; m < m1; ++m) {
    for (int64_t n = n0; n < n1; ++n) {
      const uint8_t* a = A + m * row_bytes;
      const uint8_t* b = B + n * row_bytes;
      double acc = 0.0;
      for (int64_t blk = 0; blk < kb; ++blk) {
        double inner = 0.0;
        for (int64_t j = 0; j < 16; ++j) {
          int64_t k = blk * 16 + j;
          inner += mx_elem(QKO_FMT_MXFP4_E2M1, a, k) * mx_elem(QKO_FMT_MXFP4_E2M1, b, k);
        }
        acc += g_ue4m3[sA[m * kb + blk]] * g_ue4m3[sB[n * kb + blk]] * inner;
      }
      acc *= (double)ga * (double)gb;
      if (bias) acc += (double)qko_bf16_to_f32(bias[n]);
      ref[(m - m0) * ldr + (n - n0)] = acc;
    }
  }
  return QKO_OK;
}

/* ------------------------------------------------------------------ */
/* FP8 blockscale GEMM  [MORI806-BS]                                   */
/* ------------------------------------------------------------------ */

/* ref[(m-m0)*ldr + (n-n0)] =
 *     sum_g sa[m, g] * sb[n / 128, g] * sum_{k in K-block g} e4m3(A[m,k]) * e4m3(B[n,k])
 *     (+ bias[n])
 * in fp64, where K-block g covers k in [128 g, min(128 g + 128, K)).
 * sa is [M, KB] and sb is [NB, KB] fp32, row-major, with KB = ceil(K/128)
 * and NB = ceil(N/128).  This is the value before bf16 rounding. */
int qko_gemm_fp8_blockscale(const uint8_t* A, const uint8_t* B, const float* sa, const float* sb,
                            const uint16_t* bias, double* ref, int64_t ldr, int64_t M, int64_t N, int64_t K,
                            int64_t m0, int64_t m1, int64_t n0, int64_t n1) {
  if (!A || !B || !sa || !sb || !ref || M < 0 || N < 0 || K < 0) return QKO_ERR_ARG;
  if (m0 < 0 || n0 < 0 || m1 > M || n1 > N || m0 > m1 || n0 > n1 || ldr < n1 - n0) return QKO_ERR_ARG;
  build_tables();
  const int64_t KB = (K + 127) / 128;
#pragma omp parallel for collapse(2) schedule(static)
  for (int64_t m = m0; m < m1; ++m) {
    for (int64_t n = n0; n < n1; ++n) {
      const uint8_t* a = A + m * K;
      const uint8_t* b = B + n * K;
      double acc = 0.0;
      for (int64_t g = 0; g < KB; ++g) {
        double inner = 0.0;
        const int64_t k1 = (g + 1) * 128 < K ? (g + 1) * 128 : K;
        for (int64_t k = g * 128; k < k1; ++k) inner += g_e4m3[a[k]] * g_e4m3[b[k]];
        acc += (double)sa[m * KB + g] * (double)sb[(n / 128) * KB + g] * inner;
      }
      if (bias) acc += (double)qko_bf16_to_f32(bias[n]);
      ref[(m - m0) * ldr + (n - n0)] = acc;
    }
  }
  return QKO_OK;
}

/* Number of OpenMP threads a parallel region of this library uses. */
int qko_num_threads(void) {
#ifdef _OPENMP
  int n = 1;
#pragma omp parallel
  {
#pragma omp single
    n = omp_get_num_threads();
  }
  return n;
#else
  return 1;
#endif
}
