/*
 * qg_oracle.c -- slow, plain CPU oracle for the quantized decode GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file: it is used by tests/, by __graft_entry__.smoke() and by the
 * cpu_baseline leg of bench.py, and by nothing else.  It shares no code,
 * header, table or constant generator with the CUDA library.
 *
 * Source of the method: "Building a High-Performance and Portable vLLM Linear
 * Backend with Helion" (discuss.pytorch.kr, PyTorch blog re-post), referred to
 * below as [HLB].  [HLB] "Helion Linear Backend > Scope" names the three
 * formats:
 *   FP8_Dynamic  FP8, per-token activation scale, per-channel weight scale
 *   W8A8_INT8    INT8, per-token activation scale, per-channel weight scale
 *   Block_FP8    FP8, 1x128 activation groups, 128x128 weight blocks
 * and [HLB] "Kernel Implementation" gives the GEMM (acc = A.B, fp32 or wider
 * accumulation, then scaling and the cast to the output dtype).
 *
 * The page states no scale formula, rounding mode, FP8 flavour or output dtype.
 * The readings taken here (each one plain and consistent with the rest):
 *   - FP8 is OCP E4M3FN (max 448, no infinities, 0x7F/0xFF are NaN).
 *   - scale s = amax / QMAX in IEEE fp32 (QMAX = 448 for FP8, 127 for INT8);
 *     an all-zero row/group/block (amax == 0) takes s = 1.0f.
 *   - the quantized value is encode(x / s) with one IEEE fp32 division;
 *     encode is round-to-nearest-even, saturating to the finite range
 *     (+-448 for E4M3, [-127, 127] for INT8 -- symmetric, never -128).
 *   - the output is bf16, rounded once, to nearest even, from the exact
 *     (fp64) scaled accumulator; no bias.
 *
 * Every function below is the plain definition, element by element.  The
 * accumulations are exact: int64 for INT8 and fp64 for E4M3 (an E4M3 x E4M3
 * product has at most 8 significant bits and lies in [2^-18, 2^17.6], so a
 * sum of up to 2^15 of them fits the 53-bit fp64 significand exactly).
 *
 * Build: gcc -O2 -std=c11 -fPIC -shared -ffp-contract=off (never -ffast-math).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define ORC_E4M3_MAX 448.0f
#define ORC_INT8_MAX 127.0f

static uint32_t f32_bits(float x) { uint32_t u; memcpy(&u, &x, 4); return u; }
static uint64_t f64_bits(double x) { uint64_t u; memcpy(&u, &x, 8); return u; }

/* ---------------------------------------------------------------- E4M3 ---- */

/* Decode one E4M3FN code: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa
 * bits; exponent field 0 is subnormal (m * 2^-9); S.1111.111 is NaN. */
double orc_e4m3_decode(uint8_t code) {
  int sign = code >> 7, e = (code >> 3) & 15, m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp(1.0 + (double)m / 8.0, e - 7);
  return sign ? -v : v;
}

/* Encode an fp32 value to E4M3FN: round to nearest, ties to even mantissa,
 * then saturate to +-448 (any |x| > 448, infinities included).  Computed from
 * the fp32 bit fields with integer arithmetic only.  NaN maps to 0x7F. */
uint8_t orc_e4m3_encode(float x) {
  uint32_t u = f32_bits(x);
  uint8_t sign = (uint8_t)((u >> 31) << 7);
  uint32_t E = (u >> 23) & 0xFF, F = u & 0x7FFFFF;
  if (E == 0xFF && F != 0) return 0x7F;            /* NaN */
  if (E == 0xFF) return (uint8_t)(sign | 0x7E);      /* +-inf saturate */
  if (E == 0) return sign;                           /* fp32 zero/subnormal: far below 2^-10 */
  int e = (int)E - 127;                              /* |x| = S * 2^(e-23) */
  uint32_t S = F | 0x800000u;
  if (e >= -6) {                                     /* E4M3 normal range */
    uint32_t q = S >> 20, rem = S & 0xFFFFFu, half = 0x80000u;
    if (rem > half || (rem == half && (q & 1))) ++q;
    if (q == 16) { q = 8; ++e; }
    if (e > 8 || (e == 8 && q > 14)) return (uint8_t)(sign | 0x7E); /* > 448 */
    return (uint8_t)(sign | ((uint32_t)(e + 7) << 3) | (q & 7));
  }
  /* E4M3 subnormal: count units of 2^-9.  |x| / 2^-9 = S * 2^(e-14). */
  int shift = 14 - e;                                /* >= 21 */
  if (shift > 31) return sign;
  uint32_t q = S >> shift, rem = S & ((1u << shift) - 1), half = 1u << (shift - 1);
  if (rem > half || (rem == half && (q & 1))) ++q;
  return (uint8_t)(sign | q);                        /* q == 8 is 2^-6, the min normal */
}

/* -------------------------------------------------------------- INT8 ---- */

/* Symmetric INT8 encode: round to nearest even, clamp to [-127, 127]. */
int8_t orc_int8_encode(float x) {
  if (x != x) return 0;
  if (x >= ORC_INT8_MAX) return 127;
  if (x <= -ORC_INT8_MAX) return -127;
  float r = rintf(x);                                /* default mode: ties to even */
  return (int8_t)(int)r;
}

/* -------------------------------------------------------------- BF16 ---- */

/* Round an fp64 value once to bf16 (8 significant bits), ties to even,
 * overflow to infinity; returns the bf16 bit pattern. */
uint16_t orc_bf16_from_double(double y) {
  uint64_t u = f64_bits(y);
  uint16_t sign = (uint16_t)((u >> 63) << 15);
  uint32_t E = (uint32_t)((u >> 52) & 0x7FF);
  uint64_t F = u & 0xFFFFFFFFFFFFFull;
  if (E == 0x7FF) return F ? (uint16_t)0x7FC0 : (uint16_t)(sign | 0x7F80);
  if (E == 0) return sign;                           /* fp64 zero/subnormal */
  int e = (int)E - 1023;
  uint64_t S = F | (1ull << 52);                     /* |y| = S * 2^(e-52) */
  if (e >= -126) {
    uint64_t q = S >> 45, rem = S & ((1ull << 45) - 1), half = 1ull << 44;
    if (rem > half || (rem == half && (q & 1))) ++q;
    if (q == 256) { q = 128; ++e; }
    if (e > 127) return (uint16_t)(sign | 0x7F80);
    return (uint16_t)(sign | ((uint32_t)(e + 127) << 7) | (uint32_t)(q & 0x7F));
  }
  /* bf16 subnormal: units of 2^-133.  |y| / 2^-133 = S * 2^(e+81). */
  int shift = -81 - e;                               /* >= 46 */
  if (shift > 63) return sign;
  uint64_t q = S >> shift, rem = S & ((1ull << shift) - 1), half = 1ull << (shift - 1);
  if (rem > half || (rem == half && (q & 1))) ++q;
  return (uint16_t)(sign | (uint16_t)q);
}

/* ------------------------------------------------------- quantization ---- */

static float scale_of(float amax, float qmax) { return amax > 0.0f ? amax / qmax : 1.0f; }

/* Per-row FP8 (per-token activation, FP8_Dynamic; per-channel weight):
 * s[r] = amax_c |X[r,c]| / 448, Xq[r,c] = E4M3(X[r,c] / s[r]). */
void orc_quant_rows_fp8(const float* X, int64_t rows, int64_t cols, uint8_t* Xq, float* s) {
  for (int64_t r = 0; r < rows; ++r) {
    float amax = 0.0f;
    for (int64_t c = 0; c < cols; ++c) { float a = fabsf(X[r * cols + c]); if (a > amax) amax = a; }
    float sc = scale_of(amax, ORC_E4M3_MAX);
    s[r] = sc;
    for (int64_t c = 0; c < cols; ++c) Xq[r * cols + c] = orc_e4m3_encode(X[r * cols + c] / sc);
  }
}

/* Per-row INT8 (W8A8_INT8): s[r] = amax / 127, Xq = clamp(RNE(X / s)). */
void orc_quant_rows_int8(const float* X, int64_t rows, int64_t cols, int8_t* Xq, float* s) {
  for (int64_t r = 0; r < rows; ++r) {
    float amax = 0.0f;
    for (int64_t c = 0; c < cols; ++c) { float a = fabsf(X[r * cols + c]); if (a > amax) amax = a; }
    float sc = scale_of(amax, ORC_INT8_MAX);
    s[r] = sc;
    for (int64_t c = 0; c < cols; ++c) Xq[r * cols + c] = orc_int8_encode(X[r * cols + c] / sc);
  }
}

/* 1x128 activation groups (Block_FP8): one scale per row r and group g of
 * 128 consecutive columns, s laid out [rows][ceil(cols/128)]. */
void orc_quant_groups_fp8(const float* X, int64_t rows, int64_t cols, uint8_t* Xq, float* s) {
  int64_t ng = (cols + 127) / 128;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t g = 0; g < ng; ++g) {
      int64_t c0 = g * 128, c1 = c0 + 128 < cols ? c0 + 128 : cols;
      float amax = 0.0f;
      for (int64_t c = c0; c < c1; ++c) { float a = fabsf(X[r * cols + c]); if (a > amax) amax = a; }
      float sc = scale_of(amax, ORC_E4M3_MAX);
      s[r * ng + g] = sc;
      for (int64_t c = c0; c < c1; ++c) Xq[r * cols + c] = orc_e4m3_encode(X[r * cols + c] / sc);
    }
}

/* 128x128 weight blocks (Block_FP8): one scale per block (nb, kb) of W[N,K],
 * s laid out [ceil(N/128)][ceil(K/128)]; edge blocks cover what remains. */
void orc_quant_blocks_fp8(const float* W, int64_t N, int64_t K, uint8_t* Wq, float* s) {
  int64_t nbn = (N + 127) / 128, nbk = (K + 127) / 128;
  for (int64_t bn = 0; bn < nbn; ++bn)
    for (int64_t bk = 0; bk < nbk; ++bk) {
      int64_t n0 = bn * 128, n1 = n0 + 128 < N ? n0 + 128 : N;
      int64_t k0 = bk * 128, k1 = k0 + 128 < K ? k0 + 128 : K;
      float amax = 0.0f;
      for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = k0; k < k1; ++k) { float a = fabsf(W[n * K + k]); if (a > amax) amax = a; }
      float sc = scale_of(amax, ORC_E4M3_MAX);
      s[bn * nbk + bk] = sc;
      for (int64_t n = n0; n < n1; ++n)
        for (int64_t k = k0; k < k1; ++k) Wq[n * K + k] = orc_e4m3_encode(W[n * K + k] / sc);
    }
}

/* -------------------------------------------------------------- GEMMs ---- */
/* Each GEMM computes, for every token row m in [0, M) and every output column
 * n listed in ns[0..nn), the exact accumulator and the bf16 output
 *   acc[m, j] = sum_k A_q[m,k] * W_q[ns[j],k]     (A_q [M,K], W_q [N,K])
 * stored at acc_out[m * nn + j] and y_out[m * nn + j].  The listed columns let
 * a caller sample a large output or split the work across threads. */

/* W8A8_INT8: int64 accumulation; Y = bf16(acc * (s_a[m] * s_w[n])). */
void orc_gemm_int8(const int8_t* Aq, const float* sa, const int8_t* Wq, const float* sw,
                   int64_t M, int64_t K, const int64_t* ns, int64_t nn,
                   int64_t* acc_out, uint16_t* y_out) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t j = 0; j < nn; ++j) {
      int64_t n = ns[j], acc = 0;
      for (int64_t k = 0; k < K; ++k) acc += (int64_t)Aq[m * K + k] * (int64_t)Wq[n * K + k];
      double scale = (double)sa[m] * (double)sw[n];  /* exact: 24 + 24 bits */
      acc_out[m * nn + j] = acc;
      y_out[m * nn + j] = orc_bf16_from_double((double)acc * scale);
    }
}

/* FP8_Dynamic: exact fp64 accumulation of decoded E4M3 products. */
void orc_gemm_fp8(const uint8_t* Aq, const float* sa, const uint8_t* Wq, const float* sw,
                  int64_t M, int64_t K, const int64_t* ns, int64_t nn,
                  double* acc_out, uint16_t* y_out) {
  for (int64_t m = 0; m < M; ++m)
    for (int64_t j = 0; j < nn; ++j) {
      int64_t n = ns[j];
      double acc = 0.0;
      for (int64_t k = 0; k < K; ++k) acc += orc_e4m3_decode(Aq[m * K + k]) * orc_e4m3_decode(Wq[n * K + k]);
      double scale = (double)sa[m] * (double)sw[n];
      acc_out[m * nn + j] = acc;
      y_out[m * nn + j] = orc_bf16_from_double(acc * scale);
    }
}

/* Block_FP8: per 128-wide K group kb, the exact partial sum is scaled by the
 * activation group scale s_a[m, kb] and the weight block scale
 * s_w[n / 128, kb], and the scaled partials are summed in fp64.
 * acc_out holds the scaled fp64 sum (the value rounded to bf16). */
void orc_gemm_blockfp8(const uint8_t* Aq, const float* sa, const uint8_t* Wq, const float* sw,
                       int64_t M, int64_t K, const int64_t* ns, int64_t nn,
                       double* acc_out, uint16_t* y_out) {
  int64_t nbk = (K + 127) / 128;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t j = 0; j < nn; ++j) {
      int64_t n = ns[j], bn = n / 128;
      double y = 0.0;
      for (int64_t kb = 0; kb < nbk; ++kb) {
        int64_t k0 = kb * 128, k1 = k0 + 128 < K ? k0 + 128 : K;
        double part = 0.0;
        for (int64_t k = k0; k < k1; ++k) part += orc_e4m3_decode(Aq[m * K + k]) * orc_e4m3_decode(Wq[n * K + k]);
        y += ((double)sa[m * nbk + kb] * (double)sw[bn * nbk + kb]) * part;
      }
      acc_out[m * nn + j] = y;
      y_out[m * nn + j] = orc_bf16_from_double(y);
    }
}

/* Per-element magnitude used by the FP8 accuracy bound:
 * mag[m, j] = sum_k |A_q[m,k] * W_q[n,k]| (decoded), times the scales of the
 * format: s_a[m] * s_w[n] for FP8_Dynamic, per 128-K group for Block_FP8. */
void orc_abs_mag_fp8(const uint8_t* Aq, const float* sa, const uint8_t* Wq, const float* sw,
                     int64_t M, int64_t K, const int64_t* ns, int64_t nn, int blocked,
                     double* mag_out) {
  int64_t nbk = (K + 127) / 128;
  for (int64_t m = 0; m < M; ++m)
    for (int64_t j = 0; j < nn; ++j) {
      int64_t n = ns[j];
      double tot = 0.0;
      for (int64_t kb = 0; kb < nbk; ++kb) {
        int64_t k0 = kb * 128, k1 = k0 + 128 < K ? k0 + 128 : K;
        double part = 0.0;
        for (int64_t k = k0; k < k1; ++k) part += fabs(orc_e4m3_decode(Aq[m * K + k]) * orc_e4m3_decode(Wq[n * K + k]));
        tot += blocked ? ((double)sa[m * nbk + kb] * (double)sw[(n / 128) * nbk + kb]) * part : part;
      }
      mag_out[m * nn + j] = blocked ? tot : tot * ((double)sa[m] * (double)sw[n]);
    }
}
