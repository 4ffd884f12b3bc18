// quant.cuh -- dynamic activation quantization and static weight
// quantization for the three formats of "Building a High-Performance and
// Portable vLLM Linear Backend with Helion", section "Helion Linear Backend >
// Scope":
//   FP8_Dynamic  per-token (row) E4M3, s = amax/448
//   W8A8_INT8    per-token (row) symmetric int8, s = amax/127
//   Block_FP8    E4M3 with one scale per 1x128 activation group and one per
//                128x128 weight block
// The page gives no formula; this code takes s = amax/QMAX in IEEE fp32
// (s = 1 when amax == 0) and q = RNE-saturate(x / s) with one IEEE fp32
// division, the same reading as the CPU oracle, so both agree bit for bit.
#pragma once
#include "common.cuh"
#include <cuda_fp8.h>

namespace qg {

enum : int { kFmtFP8 = 0, kFmtINT8 = 1, kFmtBlock = 2 };

// s = amax / qmax, correctly rounded, for the two format maxima (448 for
// E4M3, 127 for INT8), by Markstein's method (see Divider below) with the
// correctly rounded reciprocals of the constants written out: RN(1/448) has
// the bits 0x3b124925 and RN(1/127) 0x3c010204.  The quotient of a positive
// amax >= 2^-100 is normal, so two residual steps return it correctly
// rounded; smaller amax (and any other qmax) divide with __fdiv_rn.  A
// per-group or per-row scale costs a few fma, not a division routine.
__device__ __forceinline__ float scale_from_amax(float amax, float qmax) {
  if (!(amax > 0.0f)) return 1.0f;
  const bool known = qmax == 448.0f || qmax == 127.0f;
  if (!known || amax < 0x1p-100f) return __fdiv_rn(amax, qmax);
  const float r = __uint_as_float(qmax == 448.0f ? 0x3b124925u : 0x3c010204u);
  const float q1 = __fmul_rn(amax, r);
  const float q2 = __fmaf_rn(__fmaf_rn(-q1, qmax, amax), r, q1);
  return __fmaf_rn(__fmaf_rn(-q2, qmax, amax), r, q2);
}

// Two fp32 -> two E4M3 codes (round to nearest even, saturate to +-448);
// `lo` lands in the low byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  return static_cast<uint16_t>(__nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}
__device__ __forceinline__ uint8_t int8_sym(float x) {
  int v = __float2int_rn(x);  // round to nearest even
  v = v > 127 ? 127 : (v < -127 ? -127 : v);
  return static_cast<uint8_t>(static_cast<int8_t>(v));
}

// 8 consecutive inputs as fp32 (16-byte load for bf16, 2 x 16 bytes for f32).
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&x)[8]) {
  uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}
__device__ __forceinline__ void load8(const float* p, float (&x)[8]) {
  float4 a = *reinterpret_cast<const float4*>(p);
  float4 b = *reinterpret_cast<const float4*>(p + 4);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w; x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

template <int OUT>  // kFmtFP8 or kFmtINT8
__device__ __forceinline__ uint2 encode8(const float (&x)[8], float s) {
  uint32_t w[2];
  if constexpr (OUT == kFmtFP8) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint16_t lo = e4m3x2(__fdiv_rn(x[4 * h + 0], s), __fdiv_rn(x[4 * h + 1], s));
      uint16_t hi = e4m3x2(__fdiv_rn(x[4 * h + 2], s), __fdiv_rn(x[4 * h + 3], s));
      w[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t b0 = int8_sym(__fdiv_rn(x[4 * h + 0], s)), b1 = int8_sym(__fdiv_rn(x[4 * h + 1], s));
      uint32_t b2 = int8_sym(__fdiv_rn(x[4 * h + 2], s)), b3 = int8_sym(__fdiv_rn(x[4 * h + 3], s));
      w[h] = b0 | (b1 << 8) | (b2 << 16) | (b3 << 24);
    }
  }
  return make_uint2(w[0], w[1]);
}

// Quotient x / s rounded to nearest even, for many x and one s, without a
// division per element: Markstein's method (P. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", 1990).  With r
// the correctly rounded reciprocal of s, q1 = RN(x*r) is within two ulps of
// x/s; one residual step q2 = q1 + r*(x - s*q1) makes it faithful, and a
// second one returns the correctly rounded quotient, because each residual
// x - s*q of a faithful q is exact in one fma.  A zero x is returned as is,
// with its sign.  Valid when s, x/s and the
// residuals are normal numbers: Divider::exact is false for rows whose scale
// lies outside [2^-100, 2^100] (those divide with __fdiv_rn), and x/s below
// 2^-100 only matters up to its sign once encoded (it rounds to zero).
struct Divider {
  float s, r;
  bool exact;
  __device__ __forceinline__ explicit Divider(float scale) : s(scale) {
    r = __frcp_rn(scale);
    exact = scale >= 0x1p-100f && scale <= 0x1p100f;
  }
  // x / s when `exact` (no branch, no division routine)
  __device__ __forceinline__ float fast(float x) const {
    const float q1 = __fmul_rn(x, r);
    const float q2 = __fmaf_rn(__fmaf_rn(-q1, s, x), r, q1);
    const float q3 = __fmaf_rn(__fmaf_rn(-q2, s, x), r, q2);
    // the residual steps turn -0 into +0; the quotient of +-0 is +-0 (E4M3
    // keeps the sign of zero)
    return x == 0.0f ? x : q3;
  }
  __device__ __forceinline__ float operator()(float x) const { return exact ? fast(x) : __fdiv_rn(x, s); }
  // q[i] = x[i] / s for a whole piece with one branch: a branch per value,
  // each with a division routine on its other side, made the quantizers
  // several times slower than the arithmetic itself
  template <int N>
  __device__ __forceinline__ void divide(const float (&x)[N], float (&q)[N]) const {
    if (exact) {
#pragma unroll
      for (int i = 0; i < N; ++i) q[i] = fast(x[i]);
    } else {
#pragma unroll
      for (int i = 0; i < N; ++i) q[i] = __fdiv_rn(x[i], s);
    }
  }
};

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// One CTA per row: per-row absmax over K (16-byte vector loads, warp-shuffle
// then shared-memory reduction), one scale per row, then encode the row.
// Rows: X[r * ldx + k], k < K (K % 8 == 0); Q[r * K + k]; s[r].
template <typename InT, int OUT, int THREADS>
__global__ void __launch_bounds__(THREADS) quant_rows_kernel(const InT* __restrict__ X, int64_t ldx, int K,
                                                            uint8_t* __restrict__ Q, float* __restrict__ S,
                                                            float qmax, unsigned long long* ts) {
  stamp_start(ts);
  const int64_t r = blockIdx.x;
  const InT* x = X + r * ldx;
  // the row requested into L2 before the wait (see prefetch_l2_bulk)
  if (threadIdx.x == 0) prefetch_l2_bulk(x, static_cast<uint32_t>(K) * static_cast<uint32_t>(sizeof(InT)));
  // Let the next kernel (a GEMM that first streams its static weights) be
  // scheduled now; this kernel's own inputs are read only after the wait.
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float red[THREADS / 32];
  float amax = 0.0f;
  for (int k = threadIdx.x * 8; k < K; k += THREADS * 8) {
    float v[8];
    load8(x + k, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < THREADS / 32 ? red[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float s = scale_from_amax(red[0], qmax);
  if (threadIdx.x == 0) S[r] = s;
  uint8_t* q = Q + r * static_cast<int64_t>(K);
  for (int k = threadIdx.x * 8; k < K; k += THREADS * 8) {
    float v[8];
    load8(x + k, v);
    *reinterpret_cast<uint2*>(q + k) = encode8<OUT>(v, s);
  }
  stamp_end(ts);
}

// Activation rows (bf16) up to 512 x 8 x CH elements: one CTA per row, each
// thread keeps its CH chunks of 8 values in registers, so the row is read
// once with all loads in flight together; a single barrier gives every
// thread the row maximum; the quotients come from Divider (correctly rounded,
// the same codes as one IEEE division each).
template <int OUT, int CH>
__global__ void __launch_bounds__(512) quant_rows_reg_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx, int K,
                                                             uint8_t* __restrict__ Q, float* __restrict__ S,
                                                             float qmax, unsigned long long* ts) {
  constexpr int kThreads = 512;
  stamp_start(ts);
  const int64_t r = blockIdx.x;
  const __nv_bfloat16* x = X + r * ldx;
  // the row's bytes requested into L2 while the kernel ahead finishes (K % 16 == 0: 32-byte multiple)
  if (threadIdx.x == 0) prefetch_l2_bulk(x, static_cast<uint32_t>(K) * 2u);
  pdl_launch_dependents();
  pdl_wait();
  __shared__ float red[kThreads / 32];
  float v[CH][8];
  float amax = 0.0f;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int k = (c * kThreads + static_cast<int>(threadIdx.x)) * 8;
    if (k < K) {
      load8(x + k, v[c]);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[c][i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[c][i]));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.0f;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) amax = fmaxf(amax, red[w]);
  const float s = scale_from_amax(amax, qmax);
  if (threadIdx.x == 0) S[r] = s;
  const Divider dv(s);
  uint8_t* q = Q + r * static_cast<int64_t>(K);
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int k = (c * kThreads + static_cast<int>(threadIdx.x)) * 8;
    if (k >= K) break;
    uint32_t w[2];
    float qv[8];
    dv.divide(v[c], qv);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if constexpr (OUT == kFmtFP8) {
        const uint16_t lo = e4m3x2(qv[4 * h + 0], qv[4 * h + 1]);
        const uint16_t hi = e4m3x2(qv[4 * h + 2], qv[4 * h + 3]);
        w[h] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
      } else {
        w[h] = static_cast<uint32_t>(int8_sym(qv[4 * h + 0])) |
               (static_cast<uint32_t>(int8_sym(qv[4 * h + 1])) << 8) |
               (static_cast<uint32_t>(int8_sym(qv[4 * h + 2])) << 16) |
               (static_cast<uint32_t>(int8_sym(qv[4 * h + 3])) << 24);
      }
    }
    *reinterpret_cast<uint2*>(q + k) = make_uint2(w[0], w[1]);
  }
  stamp_end(ts);
}

// Block_FP8 activations: one warp per 1x128 group (32 lanes x 4 values).
// S is [rows][K/128] row-major.  K % 128 == 0.
template <int WARPS>
__global__ void __launch_bounds__(WARPS * 32) quant_groups_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx,
                                                                 int rows, int K, uint8_t* __restrict__ Q,
                                                                 float* __restrict__ S, unsigned long long* ts) {
  stamp_start(ts);
  const int groups = K / 128;
  const int64_t gid = static_cast<int64_t>(blockIdx.x) * WARPS + (threadIdx.x >> 5);
  // each warp's 256-byte group requested into L2 before the wait (see prefetch_l2_bulk)
  if ((threadIdx.x & 31) == 0 && gid < static_cast<int64_t>(rows) * groups)
    prefetch_l2_bulk(X + (gid / groups) * ldx + (gid % groups) * 128, 256u);
  // Let the next kernel (a GEMM that first streams its static weights) be
  // scheduled now; this kernel's own inputs are read only after the wait.
  pdl_launch_dependents();
  pdl_wait();
  if (gid < static_cast<int64_t>(rows) * groups) {  // (no early return: the end stamp is a CTA barrier)
    const int lane = threadIdx.x & 31;
    const int64_t r = gid / groups;
    const int g = static_cast<int>(gid % groups);
    const __nv_bfloat16* x = X + r * ldx + g * 128 + lane * 4;
    uint2 u = *reinterpret_cast<const uint2*>(x);
    float v[4] = {__uint_as_float(u.x << 16), __uint_as_float(u.x & 0xFFFF0000u), __uint_as_float(u.y << 16),
                  __uint_as_float(u.y & 0xFFFF0000u)};
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    amax = warp_max(amax);
    const float s = scale_from_amax(amax, 448.0f);
    if (lane == 0) S[r * groups + g] = s;
    float qv[4];
    Divider(s).divide(v, qv);
    uint16_t lo = e4m3x2(qv[0], qv[1]);
    uint16_t hi = e4m3x2(qv[2], qv[3]);
    *reinterpret_cast<uint32_t*>(Q + r * static_cast<int64_t>(K) + g * 128 + lane * 4) =
        static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
  }
  stamp_end(ts);
}

// Block_FP8 weights: one CTA of 256 threads per 128x128 block of W[N, K]
// (fp32); the last block row may be ragged (N % 128 != 0).  K % 128 == 0.
// S is [ceil(N/128)][K/128] row-major.
__global__ void __launch_bounds__(256) quant_blocks_kernel(const float* __restrict__ W, int N, int K,
                                                          uint8_t* __restrict__ Q, float* __restrict__ S) {
  __shared__ float red[8];
  const int kb = blockIdx.x, nb = blockIdx.y, kblocks = K / 128;
  const int n0 = nb * 128, rows = min(128, N - n0);
  // thread t covers rows t/16 + 16*j, columns (t%16)*8 .. +7
  const int c = (threadIdx.x & 15) * 8;
  float amax = 0.0f;
  for (int rr = threadIdx.x >> 4; rr < rows; rr += 16) {
    float v[8];
    load8(W + static_cast<int64_t>(n0 + rr) * K + kb * 128 + c, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
  amax = warp_max(amax);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < 8 ? red[threadIdx.x] : 0.0f;
    v = warp_max(v);
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float s = scale_from_amax(red[0], 448.0f);
  if (threadIdx.x == 0) S[nb * kblocks + kb] = s;
  for (int rr = threadIdx.x >> 4; rr < rows; rr += 16) {
    float v[8];
    const int64_t off = static_cast<int64_t>(n0 + rr) * K + kb * 128 + c;
    load8(W + off, v);
    *reinterpret_cast<uint2*>(Q + off) = encode8<kFmtFP8>(v, s);
  }
}

}  // namespace qg
