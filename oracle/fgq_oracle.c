/*
 * Oracle for fine-grained FP8 quantization and the block-scaled FP8 GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, host-only
 * restatement of what the method computes.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline / reference arm may load it; the
 * library's product path never calls it and shares no code, header, table
 * or constant with it.
 *
 * Source: "Fine-Grained FP8/FP4 Quantization" (KernelWiki technique page):
 *   - §Scaling Granularities: 1x128 tile-wise scales for activations,
 *     128x128 block-wise scales for weights.
 *   - §DeepGEMM: Tile-wise and Block-wise Scaling: scale_A[M, K/128],
 *     scale_B[K/128, N/128]; per 128-wide K chunk the MMA partial is
 *     multiplied by scale_A * scale_B and added to an fp32 accumulator.
 *   - §UE8M0 vs E4M3 Scale Formats (table): E4M3 spans about 0..448; a UE8M0
 *     scale is a pure power of two.
 *   - §Blackwell: Native Block Scaling: UE8M0 value = 2^(e - 127), four
 *     codes per 32-bit word, byte i = block i.
 *   - §UE8M0 vs E4M3 Scale Formats and §NVFP4 Two-Level Scaling: E2M1
 *     values 0, .5, 1, 1.5, 2, 3, 4, 6; MXFP4 = a UE8M0 scale per 32;
 *     NVFP4 = an E4M3 scale per 16 times an fp32 per-tensor scale.
 *
 * Readings where the page is silent (each is listed with its reason in the
 * design notes of this repository):
 *   scale       s = fl32(amax / 448) in fp32 mode; in UE8M0 mode the
 *               smallest power of two 2^e >= fl32(amax / 448), e in
 *               [-127, 127];
 *   zero group  amax == 0 gives s = 1 (codes are all +-0, no NaN);
 *   encode      q = E4M3(fl32(x / s)), round to nearest, ties to even,
 *               values beyond 448 saturate to +-448, sign kept on zero;
 *   inputs      finite bf16 values (a non-finite input is reported, -1).
 *
 * Every floating-point step is written out in the order above.  Build with
 * -ffp-contract=off so no multiply-add is fused on any host.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define FGQO_MODE_FP32 0
#define FGQO_MODE_UE8M0 1

/* ---- element formats ------------------------------------------------- */

/* bf16 bit pattern -> float: bf16 is the top half of an IEEE binary32, so
 * the widening is exact (Half-Precision Math, bf16 row of the precision
 * table: 8 exponent bits, 7 mantissa bits, fp32's range). */
float fgqo_bf16_to_float(uint16_t bits) {
  uint32_t u = (uint32_t)bits << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* Exact value of an E4M3 code (1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits; no infinities; S.1111.111 is NaN).  Normal codes are
 * (1 + m/8) * 2^(e-7) = (8 + m) * 2^(e-10); subnormals (e == 0) are
 * m * 2^-9.  Largest finite value: code 0x7E = 1.75 * 2^8 = 448. */
double fgqo_e4m3_decode(uint8_t code) {
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    mag = ldexp((double)m, -9);
  else
    mag = ldexp((double)(8 + m), e - 10);
  return (code & 0x80) ? -mag : mag;
}

/* Non-negative finite E4M3 values in code order 0x00 .. 0x7E; the format is
 * monotone in its code, so this table is sorted. */
static double g_e4m3_pos[127];
static int g_e4m3_ready = 0;

static void e4m3_table_init(void) {
  if (g_e4m3_ready) return;
  for (int c = 0; c <= 0x7E; ++c) g_e4m3_pos[c] = fgqo_e4m3_decode((uint8_t)c);
  g_e4m3_ready = 1;
}

/* Round a finite fp32 value to E4M3: nearest representable value, ties to
 * the even code (even mantissa), magnitudes above 448 saturate to 448, and
 * the sign bit is kept (a negative value that rounds to zero gives 0x80).
 * Comparisons are done in double, where every quantity involved is exact. */
uint8_t fgqo_e4m3_encode(float v) {
  uint8_t sign = signbit(v) ? 0x80 : 0x00;
  double a = fabs((double)v);
  e4m3_table_init();
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  /* largest code lo with value(lo) <= a; then a < value(lo + 1) */
  int lo = 0, hi = 0x7E; /* invariant: value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (g_e4m3_pos[mid] <= a)
      lo = mid;
    else
      hi = mid;
  }
  double d_lo = a - g_e4m3_pos[lo];
  double d_hi = g_e4m3_pos[lo + 1] - a;
  int c;
  if (d_lo < d_hi)
    c = lo;
  else if (d_hi < d_lo)
    c = lo + 1;
  else
    c = (lo % 2 == 0) ? lo : lo + 1; /* tie: even mantissa */
  return (uint8_t)(sign | c);
}

/* ---- scales ---------------------------------------------------------- */

/* Smallest power of two 2^e >= t (t > 0), with e clamped to [-127, 127]
 * (the UE8M0 code e + 127 then lies in 0..254; 255 is not produced). */
float fgqo_pow2_ceil(float t) {
  int e = ilogb(t); /* 2^e <= t < 2^(e+1) */
  if (ldexp(1.0, e) < (double)t) e += 1;
  if (e < -127) e = -127;
  if (e > 127) e = 127;
  return (float)ldexp(1.0, e);
}

/* The dequantisation multiplier of one group from its absolute maximum.
 * fp32 mode: amax / 448 rounded once in fp32.  UE8M0 mode: that quotient
 * rounded up to a power of two.  amax == 0 gives 1 in both modes. */
float fgqo_scale_from_amax(float amax, int mode) {
  if (amax == 0.0f) return 1.0f;
  float t = amax / 448.0f;
  if (mode == FGQO_MODE_UE8M0) return fgqo_pow2_ceil(t);
  return t;
}

/* UE8M0 code of a power-of-two scale: the biased exponent e + 127, so that
 * the value is 2^(code - 127).  Returns -1 if s is not such a power. */
int fgqo_ue8m0_code(float s) {
  if (!(s > 0.0f) || isinf(s)) return -1;
  int e;
  double f = frexp((double)s, &e); /* s = f * 2^e, f in [0.5, 1) */
  if (f != 0.5) return -1;
  e -= 1;
  if (e < -127 || e > 127) return -1;
  return e + 127;
}

/* ---- quantizers ------------------------------------------------------ */

/* Absolute maximum of a rows x cols group of bf16 values starting at x,
 * rows `ld` elements apart.  bf16 widens exactly to fp32, so the maximum is
 * exact.  Returns -1 on a non-finite element. */
static int group_amax(const uint16_t *x, int64_t ld, int64_t rows, int64_t cols,
                      float *amax_out) {
  float amax = 0.0f;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      float v = fgqo_bf16_to_float(x[r * ld + c]);
      if (!isfinite(v)) return -1;
      float a = fabsf(v);
      if (a > amax) amax = a;
    }
  *amax_out = amax;
  return 0;
}

static void group_encode(const uint16_t *x, int64_t ld, int64_t rows, int64_t cols,
                         float s, uint8_t *q, int64_t ldq) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      float v = fgqo_bf16_to_float(x[r * ld + c]);
      float y = v / s; /* one fp32 division, rounded to nearest even */
      q[r * ldq + c] = fgqo_e4m3_encode(y);
    }
}

/* 1x128 tile-wise activation quantization (§Scaling Granularities,
 * "per-tile 1x128"): X is bf16 [M, K] row-major, K % 128 == 0.
 * Outputs Xq [M, K] E4M3 codes row-major and sX [M, K/128] row-major. */
int fgqo_quant_act_1x128(const uint16_t *x, int64_t M, int64_t K, uint8_t *xq,
                         float *sx, int mode) {
  if (K % 128 != 0) return -2;
  int64_t kc = K / 128;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t g = 0; g < kc; ++g) {
      const uint16_t *src = x + m * K + g * 128;
      float amax;
      if (group_amax(src, K, 1, 128, &amax) != 0) return -1;
      float s = fgqo_scale_from_amax(amax, mode);
      sx[m * kc + g] = s;
      group_encode(src, K, 1, 128, s, xq + m * K + g * 128, K);
    }
  return 0;
}

/* 128x1 activation quantization, the transposed variant a weight-gradient
 * GEMM (reducing over the rows M of X) needs: the plainest extension of the
 * 1x128 tiles of §Scaling Granularities to groups of 128 consecutive rows
 * of one column.  X is bf16 [M, K] row-major, M and K multiples of 128.
 * Group (k, mb) is rows 128 mb .. 128 mb + 127 of column k.  Outputs, in
 * the layout the GEMM takes for its A operand (rows = k, reduction = m):
 * XqT [K, M] E4M3 codes row-major, XqT[k, m] = code of X[m, k], and
 * sXT [K, M/128] row-major, sXT[k, mb] = scale of group (k, mb). */
int fgqo_quant_act_128x1(const uint16_t *x, int64_t M, int64_t K, uint8_t *xqt,
                         float *sxt, int mode) {
  if (M % 128 != 0 || K % 128 != 0) return -2;
  int64_t mc = M / 128;
  for (int64_t k = 0; k < K; ++k)
    for (int64_t g = 0; g < mc; ++g) {
      const uint16_t *src = x + (g * 128) * K + k; /* 128 rows, stride K */
      float amax;
      if (group_amax(src, K, 128, 1, &amax) != 0) return -1;
      float s = fgqo_scale_from_amax(amax, mode);
      sxt[k * mc + g] = s;
      /* row r of the group (element X[128 g + r, k]) -> XqT[k, 128 g + r] */
      group_encode(src, K, 128, 1, s, xqt + k * M + g * 128, 1);
    }
  return 0;
}

/* 128x128 block-wise weight quantization (§Scaling Granularities,
 * "per-block 128x128"): W is bf16 [K, N] row-major, K and N multiples of
 * 128.  Outputs Wq [K, N] E4M3 codes row-major (logical layout) and
 * sW [K/128, N/128] row-major. */
int fgqo_quant_w_128x128(const uint16_t *w, int64_t K, int64_t N, uint8_t *wq,
                         float *sw, int mode) {
  if (K % 128 != 0 || N % 128 != 0) return -2;
  int64_t kb = K / 128, nb = N / 128;
  for (int64_t i = 0; i < kb; ++i)
    for (int64_t j = 0; j < nb; ++j) {
      const uint16_t *src = w + (i * 128) * N + j * 128;
      float amax;
      if (group_amax(src, N, 128, 128, &amax) != 0) return -1;
      float s = fgqo_scale_from_amax(amax, mode);
      sw[i * nb + j] = s;
      group_encode(src, N, 128, 128, s, wq + (i * 128) * N + j * 128, N);
    }
  return 0;
}

/* ---- GEMM references --------------------------------------------------- */

/* Dequantised operands in fp64: A_hat[m,k] = e4m3(Aq[m,k]) * sA[m, k/128],
 * B_hat[k,n] = e4m3(Bq[k,n]) * sB[k/128, n/128]; both products are exact in
 * fp64 (a 4-bit by 24-bit significand product). */
static double a_hat(const uint8_t *aq, const float *sa, int64_t K, int64_t m, int64_t k) {
  return fgqo_e4m3_decode(aq[m * K + k]) * (double)sa[m * (K / 128) + k / 128];
}
static double b_hat(const uint8_t *bq, const float *sb, int64_t N, int64_t k, int64_t n) {
  return fgqo_e4m3_decode(bq[k * N + n]) * (double)sb[(k / 128) * (N / 128) + n / 128];
}

/* The plain definition: C[m,n] = sum_k A_hat[m,k] * B_hat[k,n] in fp64,
 * k ascending, and the error scale T[m,n] = sum_k |A_hat[m,k]| |B_hat[k,n]|.
 * Aq [M,K], Bq [K,N] (logical layouts), C and T [M,N] row-major.
 * B_hat is dequantised once into a K x N fp64 buffer; the loop then runs
 * m, k, n so that each C[m,n] still sums in k order.  Returns -3 if the
 * buffer cannot be allocated. */
int fgqo_gemm_dequant(const uint8_t *aq, const float *sa, const uint8_t *bq,
                      const float *sb, int64_t M, int64_t N, int64_t K, double *c,
                      double *t) {
  double *bh = (double *)malloc((size_t)(K * N) * sizeof(double));
  if (!bh) return -3;
  for (int64_t k = 0; k < K; ++k)
    for (int64_t n = 0; n < N; ++n) bh[k * N + n] = b_hat(bq, sb, N, k, n);
  for (int64_t m = 0; m < M; ++m) {
    double *crow = c + m * N, *trow = t + m * N;
    for (int64_t n = 0; n < N; ++n) crow[n] = 0.0, trow[n] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double a = a_hat(aq, sa, K, m, k);
      const double *brow = bh + k * N;
      for (int64_t n = 0; n < N; ++n) {
        crow[n] += a * brow[n];
        trow[n] += fabs(a) * fabs(brow[n]);
      }
    }
  }
  free(bh);
  return 0;
}

/* Same definition at listed output positions only (rows[i], cols[i]). */
void fgqo_gemm_dequant_at(const uint8_t *aq, const float *sa, const uint8_t *bq,
                          const float *sb, int64_t N, int64_t K, const int64_t *rows,
                          const int64_t *cols, int64_t count, double *c, double *t) {
  for (int64_t i = 0; i < count; ++i) {
    int64_t m = rows[i], n = cols[i];
    double acc = 0.0, mag = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double a = a_hat(aq, sa, K, m, k), b = b_hat(bq, sb, N, k, n);
      acc += a * b;
      mag += fabs(a) * fabs(b);
    }
    c[i] = acc;
    t[i] = mag;
  }
}

/* The page's chunked form (§DeepGEMM): for each 128-wide K chunk kc,
 * partial = sum_{k in chunk} e4m3(Aq[m,k]) * e4m3(Bq[k,n]) (exact in fp64:
 * at most 128 terms, each a multiple of 2^-18 below 2^18), then
 * C[m,n] += partial * (sA[m,kc] * sB[kc, n/128]).  Real-number identical to
 * fgqo_gemm_dequant; kept as a cross-check of the regrouping. */
void fgqo_gemm_chunked(const uint8_t *aq, const float *sa, const uint8_t *bq,
                       const float *sb, int64_t M, int64_t N, int64_t K, double *c) {
  int64_t kc_n = K / 128, nb = N / 128;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t kc = 0; kc < kc_n; ++kc) {
        double partial = 0.0;
        for (int64_t k = kc * 128; k < kc * 128 + 128; ++k)
          partial += fgqo_e4m3_decode(aq[m * K + k]) * fgqo_e4m3_decode(bq[k * N + n]);
        double combined = (double)sa[m * kc_n + kc] * (double)sb[kc * nb + n / 128];
        acc += partial * combined;
      }
      c[m * N + n] = acc;
    }
}

/* Brute force over the plain definition, for tiny inputs: recomputes every
 * dequantised value from scratch for every (m, n, k) with no reuse. */
void fgqo_gemm_bruteforce(const uint8_t *aq, const float *sa, const uint8_t *bq,
                          const float *sb, int64_t M, int64_t N, int64_t K, double *c) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += a_hat(aq, sa, K, m, k) * b_hat(bq, sb, N, k, n);
      c[m * N + n] = acc;
    }
}

/* UE8M0 packing (§Blackwell: Native Block Scaling, BlockScaleDescriptor):
 * four codes per 32-bit word, block i in bits 8i..8i+7, so that
 * scale_i = 2^(((packed >> (8 i)) & 0xFF) - 127). */
uint32_t fgqo_ue8m0_pack4(const uint8_t *codes) {
  uint32_t packed = 0;
  for (int i = 0; i < 4; ++i) packed |= (uint32_t)codes[i] << (8 * i);
  return packed;
}

double fgqo_ue8m0_unpack(uint32_t packed, int i) {
  int code = (int)((packed >> (8 * i)) & 0xFFu);
  return ldexp(1.0, code - 127);
}

/* ---- MXFP4: E2M1 elements, one UE8M0 scale per 32 ------------------------
 *
 * "Fine-Grained FP8/FP4 Quantization", §UE8M0 vs E4M3 Scale Formats (UE8M0
 * scales, block size 32, the MXFP standard), §NVFP4 Two-Level Scaling (the
 * E2M1 value list 0, 0.5, 1, 1.5, 2, 3, 4, 6) and §When to Use (MXFP4 with
 * UE8M0 scales for native hardware acceleration).  Readings: the scale of a
 * group is the smallest power of two >= amax / 6 (6 = largest E2M1 value),
 * the rounding-up rule the page gives for UE8M0 scales, so no element
 * saturates; a zero group gets scale 1; codes are E2M1(x / s) rounded to
 * nearest, ties to even. */

/* E2M1: bit 3 sign, bits 2-1 exponent (bias 1), bit 0 mantissa; codes 0..7
 * are 0, 0.5, 1, 1.5, 2, 3, 4, 6. */
double fgqo_e2m1_decode(uint8_t code) {
  static const double mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};
  double v = mag[code & 7];
  return (code & 8) ? -v : v;
}

/* Nearest E2M1 code to v, ties to the code with mantissa bit 0, magnitudes
 * beyond 6 saturate to 6, the sign kept (a negative value rounding to 0
 * gives 8). */
uint8_t fgqo_e2m1_encode(double v) {
  const double a = fabs(v);
  int best = 0;
  for (int c = 1; c < 8; ++c) {
    const double dc = fabs(fgqo_e2m1_decode((uint8_t)c) - a);
    const double db = fabs(fgqo_e2m1_decode((uint8_t)best) - a);
    if (dc < db || (dc == db && (c & 1) == 0)) best = c;
  }
  if (a > 6.0) best = 7;
  return (uint8_t)(best | (signbit(v) ? 8 : 0));
}

/* MXFP4 quantization of the rows of X bf16 [R, K] row-major, K % 32 == 0.
 * Outputs Xq [R, K/2] bytes (element 2j in the low nibble of byte j,
 * element 2j+1 in the high nibble) and sX [R, K/32] UE8M0 codes
 * (scale 2^(code - 127)). */
int fgqo_quant_mxfp4_1x32(const uint16_t *x, int64_t R, int64_t K, uint8_t *xq, uint8_t *sx) {
  if (K % 32 != 0) return -2;
  const int64_t kg = K / 32;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t g = 0; g < kg; ++g) {
      const uint16_t *src = x + r * K + g * 32;
      float amax;
      if (group_amax(src, K, 1, 32, &amax) != 0) return -1;
      const float s = amax == 0.0f ? 1.0f : fgqo_pow2_ceil(amax / 6.0f);
      sx[r * kg + g] = (uint8_t)fgqo_ue8m0_code(s);
      for (int64_t j = 0; j < 32; j += 2) {
        const uint8_t lo = fgqo_e2m1_encode((double)fgqo_bf16_to_float(src[j]) / s);
        const uint8_t hi = fgqo_e2m1_encode((double)fgqo_bf16_to_float(src[j + 1]) / s);
        xq[r * (K / 2) + (g * 32 + j) / 2] = (uint8_t)(lo | (hi << 4));
      }
    }
  return 0;
}

static double mx_hat(const uint8_t *q, const uint8_t *s, int64_t K, int64_t r, int64_t k) {
  const uint8_t byte = q[r * (K / 2) + k / 2];
  const uint8_t code = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
  return fgqo_e2m1_decode(code) * ldexp(1.0, (int)s[r * (K / 32) + k / 32] - 127);
}

/* Dequantised MXFP4 rows in fp64: out[r * K + k] = A_hat[r, k] (exact). */
static double *mx_dequant(const uint8_t *q, const uint8_t *s, int64_t R, int64_t K) {
  double *h = (double *)malloc((size_t)(R * K) * sizeof(double));
  if (!h) return NULL;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k) h[r * K + k] = mx_hat(q, s, K, r, k);
  return h;
}

/* MXFP4 GEMM reference: both operands as rows along K (A [M, K], B given as
 * its transpose [N, K], each quantized by fgqo_quant_mxfp4_1x32):
 * C[m,n] = sum_k A_hat[m,k] B_hat[n,k] in fp64, k ascending, and
 * T[m,n] = sum_k |A_hat| |B_hat| (each product is exact in fp64).  Both
 * operands are dequantised once; returns -3 if that memory is not there. */
int fgqo_gemm_mxfp4(const uint8_t *aq, const uint8_t *sa, const uint8_t *bq, const uint8_t *sb,
                    int64_t M, int64_t N, int64_t K, double *c, double *t) {
  if (K % 32 != 0) return -2;
  double *ah = mx_dequant(aq, sa, M, K), *bh = mx_dequant(bq, sb, N, K);
  if (!ah || !bh) {
    free(ah);
    free(bh);
    return -3;
  }
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, tt = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double p = ah[m * K + k] * bh[n * K + k];
        acc += p;
        tt += fabs(p);
      }
      c[m * N + n] = acc;
      t[m * N + n] = tt;
    }
  free(ah);
  free(bh);
  return 0;
}

/* The same at listed outputs (rows[i], cols[i]), i < count. */
int fgqo_gemm_mxfp4_at(const uint8_t *aq, const uint8_t *sa, const uint8_t *bq,
                       const uint8_t *sb, int64_t M, int64_t N, int64_t K, const int64_t *rows,
                       const int64_t *cols, int64_t count, double *c, double *t) {
  if (K % 32 != 0) return -2;
  for (int64_t i = 0; i < count; ++i) {
    const int64_t m = rows[i], n = cols[i];
    if (m < 0 || m >= M || n < 0 || n >= N) return -4;
    double acc = 0.0, tt = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double p = mx_hat(aq, sa, K, m, k) * mx_hat(bq, sb, K, n, k);
      acc += p;
      tt += fabs(p);
    }
    c[i] = acc;
    t[i] = tt;
  }
  return 0;
}

/* ---- NVFP4 (§NVFP4 Two-Level Scaling) ------------------------------- */

/* The page defines NVFP4 by its dequantization: a value is
 *   global_scale * block_scale * e2m1
 * with one E4M3 block scale per 16 consecutive elements of a row
 * (scale_A [M, K/16]) and one fp32 global scale per tensor.  It gives no
 * encoder; the readings here (the FP8 rule amax / 448 applied at both
 * levels, with 6 = the largest E2M1 value):
 *   global   g = fl32(amax / 2688) over the whole tensor (2688 = 6 * 448),
 *            1 for an all-zero tensor;
 *   block    s_b = E4M3(fl32(amax_b / fl32(6 g))): nearest, ties to even,
 *            saturating at 448 (fgqo_e4m3_encode);
 *   element  q = E2M1(fl32(x / D)) with D = fl32(g * s_b): nearest, ties
 *            to even, saturating at 6 (s_b may have rounded down);
 *            a block whose D is 0 gets signed zeros. */
float fgqo_nvfp4_global_scale(const uint16_t *x, int64_t R, int64_t K) {
  float amax;
  if (group_amax(x, K, R, K, &amax) != 0) return NAN;
  if (amax == 0.0f) return 1.0f;
  return amax / 2688.0f; /* one fp32 division */
}

/* X bf16 [R, K] row-major, K % 16 == 0, global scale g (> 0) ->
 * Xq [R, K/2] E2M1 pairs (element 2j in the low nibble of byte j) and
 * sX [R, K/16] E4M3 codes. */
int fgqo_quant_nvfp4_1x16(const uint16_t *x, int64_t R, int64_t K, float g, uint8_t *xq,
                          uint8_t *sx) {
  if (K % 16 != 0) return -2;
  if (!(g > 0.0f) || !isfinite(g)) return -5;
  const int64_t kb = K / 16;
  const float d6 = 6.0f * g;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t b = 0; b < kb; ++b) {
      const uint16_t *src = x + r * K + b * 16;
      float amax;
      if (group_amax(src, K, 1, 16, &amax) != 0) return -1;
      const float t = amax / d6;
      const uint8_t sc = fgqo_e4m3_encode(t);
      sx[r * kb + b] = sc;
      const float d = g * (float)fgqo_e4m3_decode(sc);
      for (int64_t j = 0; j < 16; j += 2) {
        uint8_t code[2];
        for (int h = 0; h < 2; ++h) {
          const float v = fgqo_bf16_to_float(src[j + h]);
          code[h] = d == 0.0f ? (uint8_t)(signbit(v) ? 8 : 0) : fgqo_e2m1_encode((double)(v / d));
        }
        xq[r * (K / 2) + (b * 16 + j) / 2] = (uint8_t)(code[0] | (code[1] << 4));
      }
    }
  return 0;
}

/* The page's dequantization, global * block * e2m1, in fp64 (exact). */
static double nv_hat(const uint8_t *q, const uint8_t *s, float g, int64_t K, int64_t r,
                     int64_t k) {
  const uint8_t byte = q[r * (K / 2) + k / 2];
  const uint8_t code = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
  return (double)g * fgqo_e4m3_decode(s[r * (K / 16) + k / 16]) * fgqo_e2m1_decode(code);
}

static double *nv_dequant(const uint8_t *q, const uint8_t *s, float g, int64_t R, int64_t K) {
  double *h = (double *)malloc((size_t)(R * K) * sizeof(double));
  if (!h) return NULL;
  for (int64_t r = 0; r < R; ++r)
    for (int64_t k = 0; k < K; ++k) h[r * K + k] = nv_hat(q, s, g, K, r, k);
  return h;
}

/* NVFP4 GEMM reference: A [M, K] and B as its transpose [N, K], each
 * quantized by fgqo_quant_nvfp4_1x16 with its own global scale:
 * C[m,n] = sum_k A_hat[m,k] B_hat[n,k] in fp64, k ascending, and
 * T[m,n] = sum_k |A_hat| |B_hat|. */
int fgqo_gemm_nvfp4(const uint8_t *aq, const uint8_t *sa, float ga, const uint8_t *bq,
                    const uint8_t *sb, float gb, int64_t M, int64_t N, int64_t K, double *c,
                    double *t) {
  if (K % 16 != 0) return -2;
  double *ah = nv_dequant(aq, sa, ga, M, K), *bh = nv_dequant(bq, sb, gb, N, K);
  if (!ah || !bh) {
    free(ah);
    free(bh);
    return -3;
  }
  for (int64_t m = 0; m < M; ++m)
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, tt = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        const double p = ah[m * K + k] * bh[n * K + k];
        acc += p;
        tt += fabs(p);
      }
      c[m * N + n] = acc;
      t[m * N + n] = tt;
    }
  free(ah);
  free(bh);
  return 0;
}

/* The same at listed outputs (rows[i], cols[i]), i < count. */
int fgqo_gemm_nvfp4_at(const uint8_t *aq, const uint8_t *sa, float ga, const uint8_t *bq,
                       const uint8_t *sb, float gb, int64_t M, int64_t N, int64_t K,
                       const int64_t *rows, const int64_t *cols, int64_t count, double *c,
                       double *t) {
  if (K % 16 != 0) return -2;
  for (int64_t i = 0; i < count; ++i) {
    const int64_t m = rows[i], n = cols[i];
    if (m < 0 || m >= M || n < 0 || n >= N) return -4;
    double acc = 0.0, tt = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double p = nv_hat(aq, sa, ga, K, m, k) * nv_hat(bq, sb, gb, K, n, k);
      acc += p;
      tt += fabs(p);
    }
    c[i] = acc;
    t[i] = tt;
  }
  return 0;
}
