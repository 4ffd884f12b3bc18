// gemm_i8.cuh -- W8A8_INT8 GEMM (Swap-AB, optional Split-K) on the sm_103a
// tensor cores.
//
// "W8A8_INT8: INT8 per-token activation and per-channel weight scaling"
// ("Building a High-Performance and Portable vLLM Linear Backend with
// Helion", section "Helion Linear Backend > Scope") needs an exact int32
// accumulator.  sm_103a has no tcgen05 int8 MMA kind and its legacy int8
// mma.sync is slow, so this kernel converts both int8 operands to fp16
// (exact for [-128, 127]) and runs tcgen05.mma kind::f16 with an fp32
// accumulator.  Every product is an integer below 2^14 and every partial sum
// over at most 1024 K stays below 2^24, so each 1024-K segment accumulates
// exactly in fp32; segments are converted to int32 and summed in registers.
//
// Pipeline per CTA (one 128-row weight tile x one K range), sized so that two
// CTAs share an SM (at most 256 TMEM columns and ~113 KB of shared memory):
//   warp 0      TMA: int8 W tile (128 x 128 B) + int8 activation tile into a
//               `stages`-deep shared-memory ring;
//   warps 2..9  weight converters: warp w owns TMEM lane quarter w % 4
//               (weight rows 32*(w%4) .. +31) and half (w-2)/4 of each
//               128-byte k-tile row; each thread widens its 64 weight bytes
//               to fp16 and writes them with tcgen05.st into a TMEM operand
//               buffer (the MMA A operand lives in TMEM, so the widened
//               weights never touch shared memory); they drain finished
//               accumulator segments into int32 (warp w takes token half
//               (w-2)/4) and run the epilogue;
//   warps 10,11 activation converters: widen the activation tile into a
//               128-byte-swizzled shared buffer (MMA B operand);
//   warp 1      one thread issues 8 MMAs (K = 16 each) per k-tile.
// Weights and activations land on separate barriers, so the weight tiles
// fetched before the activations exist (programmatic dependent launch) are
// already widened into TMEM when the activations arrive.
// Split-K reduces through distributed shared memory across the cluster of
// a tile's CTAs (up to 16 ranges) or through the caller workspace, exactly
// as the FP8 kernel does, in int32.
//
// PREW (QG_CONFIG_I8_PREWIDEN, the compute-bound regime beyond the decode
// range): the activations are widened once per launch by widen_i8_kernel
// into an fp16 copy in the workspace, and the producer loads that copy by
// TMA straight into the stage in the MMA's operand layout (two 128-byte
// swizzle atoms of 64 K).  No activation converter warps, no operand copy:
// the MMA reads the B operand from the stage and releases it with a commit.
// Each weight tile is widened once per block of up to 128 tokens (instead of
// once per 64, with the activations widened again in every CTA), so a
// widened weight byte feeds twice the MMA work.
#pragma once
#include "common.cuh"
#include "gemm_f8.cuh"

namespace qg {

constexpr int kI8ConvWarps = 8;                    // weight converters (warps 2..9)
constexpr int kI8ConvThreads = 32 * kI8ConvWarps;  // 256
constexpr int kI8AWarp = 2 + kI8ConvWarps;         // first activation converter (warp 10)
constexpr int kI8AWarps = 2;                       // activation converters (warps 10, 11)
constexpr int kI8Threads = 32 * (kI8AWarp + kI8AWarps);  // 384
constexpr int kI8OpBufs = 3;        // TMEM/shared operand buffers in flight
constexpr int kI8SegTiles = 8;      // k-tiles (of 128) per exact fp32 segment: 1024 K

struct alignas(8) CtrlI8 {
  uint64_t full[16];     // weight tile of the stage landed
  uint64_t full_a[16];   // activation tile of the stage landed
  uint64_t empty[16];
  uint64_t op_full[kI8OpBufs];
  uint64_t op_empty[kI8OpBufs];
  uint64_t d_full[2];
  uint64_t d_empty[2];
  uint64_t never;
  uint64_t done;
  uint64_t recv_bar;  // split-K: peers' partial rows have landed
  uint64_t amax_bar;  // fused quantization: peers' partial row maxima have landed
  uint32_t tmem_base;
  int last_flag;
  int abort_flag;
  float sa_s[128];  // per-token scales, staged for the epilogue
  float sw_s[128];  // per-channel scales of the tile's rows
  float amax_s[kMaxClusterSplits * 64];  // fused quantization: [source rank][token] partial row maxima
};

template <int MPAD>
struct I8Shape {
  static constexpr uint32_t kWBytes = kBN * kBK;           // 16 KB int8 weights
  static constexpr uint32_t kABytes = MPAD * kBK;          // int8 activations
  static constexpr uint32_t kStageBytes = kWBytes + kABytes;
  static constexpr uint32_t kOpBBytes = MPAD * 256;        // fp16 activations: 2 swizzle atoms of 64 K
  static constexpr uint32_t kPrewStageBytes = kWBytes + kOpBBytes;  // PREW: int8 weights + fp16 activations
  static constexpr uint32_t kACols = 64;                   // 128 fp16 per row = 64 TMEM columns
  static constexpr uint32_t kDCols = MPAD;
  static constexpr int kHalf = MPAD / 2;                   // tokens drained per converter warp
  static constexpr uint32_t kTmemCols = pow2_cols(kI8OpBufs * kACols + 2 * kDCols);
};

template <int MPAD, bool PREW = false>
__host__ __device__ constexpr size_t gemm_i8_smem_bytes(int stages, int recv_bytes = 0) {
  return PREW ? 1024 + static_cast<size_t>(stages) * I8Shape<MPAD>::kPrewStageBytes + recv_bytes + sizeof(CtrlI8)
              : 1024 + static_cast<size_t>(stages) * I8Shape<MPAD>::kStageBytes +
                    static_cast<size_t>(kI8OpBufs) * I8Shape<MPAD>::kOpBBytes + recv_bytes + sizeof(CtrlI8);
}
// CW weight converter warps (warps 2 .. 2+CW-1; 8, or 16 in the form that
// runs one CTA per SM with the deepest ring, QG_CONFIG_I8_CONV16): the
// converters of a row quarter (warp % 4, the TMEM lanes a warp may reach)
// split each k-tile into CW/4 parts of 8/(CW/4) 16-byte chunks, and drain
// the accumulator in CW/4 token parts.
template <int CW>
struct I8Conv {
  static constexpr int kWarps = CW;
  static constexpr int kThreads = 32 * CW;
  static constexpr int kAWarp = 2 + CW;     // first activation converter warp
  static constexpr int kParts = CW / 4;     // K parts / token parts of a row quarter
  static constexpr int kChunks = 8 / kParts;
};
// one CTA per SM: the PREW form beyond 32 tokens (its TMEM takes all 512
// columns) and the sixteen-converter form
__host__ __device__ constexpr bool i8_one_per_sm(int mpad, bool prew, int cw) {
  return (prew && mpad > 32) || cw > kI8ConvWarps;
}
// threads of the kernel: the PREW form has no activation converter warps
__host__ __device__ constexpr int i8_threads(bool prew, int cw = kI8ConvWarps) {
  return 32 * (2 + cw + (prew ? 0 : kI8AWarps));
}

// 4 int8 (one 32-bit word, element 0 in the low byte) -> two fp16x2 words:
// bias each byte by 128 into an unsigned byte u, form the fp16 1024 + u by
// placing u under the exponent byte 0x64, subtract 1152 = 1024 + 128.  All
// steps are exact.
__device__ __forceinline__ void int8x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t a = __byte_perm(u, 0x64646464u, 0x4140u);
  uint32_t b = __byte_perm(u, 0x64646464u, 0x4342u);
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  __half2 ha = __hsub2(*reinterpret_cast<__half2*>(&a), bias);
  __half2 hb = __hsub2(*reinterpret_cast<__half2*>(&b), bias);
  lo = *reinterpret_cast<uint32_t*>(&ha);
  hi = *reinterpret_cast<uint32_t*>(&hb);
}

// TMEM -> registers: this warp's 32 lanes x 4 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_x4(uint32_t taddr, uint32_t (&v)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3])
               : "r"(taddr));
}

// int8 activation codes -> their exact fp16 values (the B operand of the
// PREW form), 16 codes a thread per step; n16 = codes / 16.
__global__ void __launch_bounds__(256) widen_i8_kernel(const uint8_t* __restrict__ src, uint4* __restrict__ dst,
                                                       int64_t n16) {
  pdl_launch_dependents();  // the GEMM may start streaming its weights
  pdl_wait();               // the codes come from the kernel this one depends on
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * 256 + threadIdx.x; i < n16;
       i += static_cast<int64_t>(gridDim.x) * 256) {
    const uint4 v = reinterpret_cast<const uint4*>(src)[i];
    uint32_t o[8];
    int8x4_to_f16x4(v.x, o[0], o[1]);
    int8x4_to_f16x4(v.y, o[2], o[3]);
    int8x4_to_f16x4(v.z, o[4], o[5]);
    int8x4_to_f16x4(v.w, o[6], o[7]);
    dst[2 * i] = make_uint4(o[0], o[1], o[2], o[3]);
    dst[2 * i + 1] = make_uint4(o[4], o[5], o[6], o[7]);
  }
}

// FUSED: the activation warps read bf16 activations (g.A) and quantize them
// to int8 codes themselves (qg_linear_w8a8): no quantization kernel and no
// int8 activation tensor in between; tmA is unused.
template <int MPAD, bool FUSED, bool PREW = false, int CW = kI8ConvWarps>
__global__ void __launch_bounds__(i8_threads(PREW, CW), i8_one_per_sm(MPAD, PREW, CW) ? 1 : 2)
    gemm_i8_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA, GemmArgs g) {
  using S = I8Shape<MPAD>;
  using C = I8Conv<CW>;
  constexpr int kHalf = MPAD / C::kParts;  // tokens drained per converter thread
  static_assert(CW == 8 || CW == 16, "8 or 16 weight converter warps");
  static_assert(!(FUSED && CW != kI8ConvWarps), "the fused form keeps 8 converter warps");
  static_assert(kHalf % 4 == 0, "token parts of at least 4");
  static_assert(!(PREW && FUSED), "the pre-widened form takes quantized activations");
  static_assert(MPAD <= 128, "token blocks of at most 128");
  constexpr uint32_t kStage = PREW ? S::kPrewStageBytes : S::kStageBytes;
  stamp_start(g.tstamp);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stages = g.stages;
  uint8_t* opb = smem + static_cast<size_t>(stages) * kStage;                // fp16 activation buffers (not PREW)
  uint8_t* recv = opb + (PREW ? 0 : kI8OpBufs * S::kOpBBytes);               // split-K receive buffer
  CtrlI8* ctl = reinterpret_cast<CtrlI8*>(recv + g.recv_bytes);
  const bool clustered = g.reduce == kReduceCluster;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the token blocks of one weight tile are adjacent block indices (weights
  // read from HBM once, then from L2)
  const int n_tile = static_cast<int>(blockIdx.x / g.m_tiles), split = blockIdx.y;
  const int m_blk = static_cast<int>(blockIdx.x % g.m_tiles);  // token block: tokens [m_base, m_base + Mb)
  const GroupView grp = group_view(g);
  const int m_base = grp.tok0 + m_blk * MPAD;
  const int Mb = min(MPAD, grp.tok0 + grp.tokens - m_base);
  if (Mb <= 0) return;  // a token block past its group's tokens (the whole cluster alike)
  const int w_row0 = static_cast<int>(blockIdx.z) * g.N;  // the group's weight rows
  const float* s_w = g.s_w + static_cast<int64_t>(blockIdx.z) * g.sw_group_stride;
  const int kb0 = static_cast<int>(static_cast<int64_t>(split) * g.kt_total / g.splits);
  const int kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * g.kt_total / g.splits);
  const int nk = kb1 - kb0;
  const int nseg = (nk + kI8SegTiles - 1) / kI8SegTiles;

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->full_a[i], 1);
      // PREW: the MMAs read the stage's activations, so their commit releases it too
      mbar_init(&ctl->empty[i], C::kWarps + (PREW ? 1 : (FUSED ? 0 : kI8AWarps)));
    }
    for (int b = 0; b < kI8OpBufs; ++b) {
      mbar_init(&ctl->op_full[b], C::kWarps + (PREW ? 0 : kI8AWarps));
      mbar_init(&ctl->op_empty[b], 1);
    }
    for (int d = 0; d < 2; ++d) {
      mbar_init(&ctl->d_full[d], 1);
      mbar_init(&ctl->d_empty[d], C::kWarps);
    }
    mbar_init(&ctl->never, 1);
    mbar_init(&ctl->done, 1);
    mbar_init(&ctl->recv_bar, 1);
    mbar_init(&ctl->amax_bar, 1);
    ctl->last_flag = 0;
    ctl->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmA);
  }
  __syncthreads();
  if (clustered) {
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&ctl->recv_bar, static_cast<uint32_t>((g.splits - 1) * cluster_rows_of(split, g.splits) *
                                                                  cluster_mv(Mb) * 4));
      if (FUSED) mbar_arrive_expect_tx(&ctl->amax_bar, static_cast<uint32_t>((g.splits - 1) * Mb * 4));
    }
    cluster_arrive_relaxed();
  }
  pdl_launch_dependents();
  volatile int* abort_flag = &ctl->abort_flag;
  // converter threads: weight row `row` of the tile x tokens [h*kHalf, h*kHalf + kHalf)
  int32_t iacc[kHalf];
#pragma unroll
  for (int m = 0; m < kHalf; ++m) iacc[m] = 0;
  const int cw = warp - 2;        // converter warp 0..7 (negative for warps 0, 1)
  const int h = cw >> 2;          // K part of the weight row / token part of the accumulator
  const uint32_t row = (warp & 3) * 32u + lane;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      const int w_row = w_row0 + n_tile * kBN;
      const int pre = nk < stages ? nk : stages;
      // the stage's activation tile: int8 codes, or (PREW) their fp16 copy
      // as two 64-K swizzle atoms in the MMA's operand layout
      auto load_act = [&](uint8_t* st, int i, uint64_t* bar) {
        if constexpr (PREW) {
          mbar_arrive_expect_tx(bar, S::kOpBBytes);
          for (int atom = 0; atom < 2; ++atom)
            tma_load_2d(st + S::kWBytes + atom * (MPAD * 128), &tmA, (kb0 + i) * kBK + 64 * atom, m_base, bar, pol_a);
        } else {
          mbar_arrive_expect_tx(bar, S::kABytes);
          tma_load_2d(st + S::kWBytes, &tmA, (kb0 + i) * kBK, m_base, bar, pol_a);
        }
      };
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = smem + static_cast<size_t>(i) * kStage;
        mbar_arrive_expect_tx(&ctl->full[i], S::kWBytes);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[i], pol_w);
      }
      for (int i = pre; i < nk && i < pre + g.l2_prefetch; ++i) tma_prefetch_l2_2d(&tmW, (kb0 + i) * kBK, w_row);
      pdl_wait();
      if (!FUSED) {
        for (int i = 0; i < pre; ++i) load_act(smem + static_cast<size_t>(i) * kStage, i, &ctl->full_a[i]);
      }
      int issued = pre;
      for (int i = pre; i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
        if (!mbar_wait(&ctl->empty[s], ph ^ 1u, g.wait_ns) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(s) * kStage;
        mbar_arrive_expect_tx(&ctl->full[s], S::kWBytes);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[s], pol_w);
        if (g.l2_prefetch > 0 && i + g.l2_prefetch < nk) tma_prefetch_l2_2d(&tmW, (kb0 + i + g.l2_prefetch) * kBK, w_row);
        if (!FUSED) load_act(st, i, &ctl->full_a[s]);
        issued = i + 1;
      }
      // every issued copy lands before the CTA may exit or reuse the ring
      for (int j = issued > stages ? issued - stages : 0; j < issued; ++j) {
        mbar_wait(&ctl->full[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
        if (!FUSED) mbar_wait(&ctl->full_a[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
      }
    }
  } else {
    if (warp == 1) tmem_alloc(&ctl->tmem_base, S::kTmemCols);
    tc_fence_before();
    named_bar_sync(2, i8_threads(PREW, CW) - 32);
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    const uint32_t tmem_a = tmem;                                   // kI8OpBufs x 64 columns
    const uint32_t tmem_d = tmem + kI8OpBufs * S::kACols;           // 2 x MPAD columns
    if (warp == 1) {
      // -------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc = make_idesc(128, MPAD, 0, 0);  // F16 x F16 -> F32
        bool ok = true;
        if (g.force_timeout) ok = mbar_wait(&ctl->never, 0, g.wait_ns);
        for (int i = 0; ok && i < nk; ++i) {
          const int seg = i / kI8SegTiles, d = seg & 1, buf = i % kI8OpBufs;
          const bool seg_start = (i % kI8SegTiles) == 0;
          if (seg_start && seg >= 2 &&
              !mbar_wait(&ctl->d_empty[d], static_cast<uint32_t>((seg - 2) / 2) & 1u, g.wait_ns)) {
            ok = false;
            break;
          }
          if (!mbar_wait(&ctl->op_full[buf], static_cast<uint32_t>(i / kI8OpBufs) & 1u, g.wait_ns) || *abort_flag) {
            ok = false;
            break;
          }
          // PREW: the fp16 activations come straight from the stage
          const int s = i % stages;
          if (PREW && !mbar_wait(&ctl->full_a[s], static_cast<uint32_t>(i / stages) & 1u, g.wait_ns)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t b_base =
              PREW ? smem_u32(smem + static_cast<size_t>(s) * kStage + S::kWBytes) : smem_u32(opb + buf * S::kOpBBytes);
#pragma unroll
          for (int kk = 0; kk < 8; ++kk) {
            const uint32_t b_addr = b_base + (kk >> 2) * (MPAD * 128) + (kk & 3) * 32;
            mma_f16_ts(tmem_d + d * S::kDCols, tmem_a + buf * S::kACols + kk * 8, sw128_kmajor_desc(b_addr), idesc,
                       (!seg_start || kk > 0) ? 1u : 0u);
          }
          tc_commit(&ctl->op_empty[buf]);
          if (PREW) tc_commit(&ctl->empty[s]);  // the stage's activations are consumed
          if ((i % kI8SegTiles) == kI8SegTiles - 1 || i == nk - 1) tc_commit(&ctl->d_full[d]);
        }
        if (!ok) {
          *abort_flag = 1;
          mbar_arrive(&ctl->d_full[0]);
          mbar_arrive(&ctl->d_full[1]);
        }
        tc_commit(&ctl->done);  // all issued MMAs complete
      }
    } else if (FUSED && warp >= C::kAWarp) {
      // ---------------------------------------- activation quantizers (fused)
      pdl_wait();  // the activations are written by the kernel this one depends on
      const int at = threadIdx.x - 32 * C::kAWarp;  // 0..63
      const bool whole_row = !clustered && g.splits > 1;  // workspace Split-K: scale over the whole row
      const int k0 = whole_row ? 0 : kb0 * kBK, k1 = whole_row ? g.K : min(g.K, kb1 * kBK);
      fused_token_scales(g, m_base, Mb, k0, k1, clustered, clustered ? split : 0, 127.0f, ctl->amax_s, ctl->sa_s,
                         &ctl->amax_bar, at, 32 * kI8AWarps, 3, n_tile == 0 && split == 0);
      const bool write_codes = g.a_q_out != nullptr && n_tile == 0;
      bool ok = true;
      for (int i = 0; i < nk; ++i) {
        const int buf = i % kI8OpBufs;
        if (i >= kI8OpBufs &&
            !__all_sync(0xffffffffu, mbar_wait(&ctl->op_empty[buf], static_cast<uint32_t>(i / kI8OpBufs - 1) & 1u,
                                               g.wait_ns) && !*abort_flag)) {
          ok = false;
          break;
        }
        const int kt0 = (kb0 + i) * kBK;
        uint8_t* ob = opb + buf * S::kOpBBytes;
#pragma unroll
        for (int piece = at; piece < MPAD * 4; piece += 32 * kI8AWarps) {
          const int r = piece >> 2, p = piece & 3;  // token row, 32-element quarter of the 128 K
          uint32_t o[16];
          if (r < Mb) {
            float x[32];
            load_act32(g, m_base + r, kt0 + 32 * p, x);
            float qv[32];
            Divider(ctl->sa_s[r]).divide(x, qv);
            uint32_t codes[8];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int q0 = max(-127, min(127, __float2int_rn(qv[2 * j])));
              const int q1 = max(-127, min(127, __float2int_rn(qv[2 * j + 1])));
              __half2 hh = __halves2half2(__int2half_rn(q0), __int2half_rn(q1));
              o[j] = *reinterpret_cast<uint32_t*>(&hh);
              const uint32_t pair = (static_cast<uint32_t>(q0) & 0xFFu) | ((static_cast<uint32_t>(q1) & 0xFFu) << 8);
              if (j & 1) codes[j >> 1] |= pair << 16; else codes[j >> 1] = pair;
            }
            if (write_codes) {
              uint8_t* dst = g.a_q_out + static_cast<int64_t>(m_base + r) * g.K + kt0 + 32 * p;
#pragma unroll
              for (int c = 0; c < 2; ++c)
                if (kt0 + 32 * p + 16 * c < g.K)
                  *reinterpret_cast<uint4*>(dst + 16 * c) =
                      make_uint4(codes[4 * c], codes[4 * c + 1], codes[4 * c + 2], codes[4 * c + 3]);
            }
          } else {
#pragma unroll
            for (int j = 0; j < 16; ++j) o[j] = 0u;
          }
          uint8_t* atom = ob + (p >> 1) * (MPAD * 128);
          const uint32_t c0 = (p & 1) * 4;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(atom + sw128_chunk(r, c0 + j)) =
                make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->op_full[buf]);
      }
      if (!ok) *abort_flag = 1;
    } else if (warp >= C::kAWarp) {
      // -------------------------------------------- activation converters
      pdl_wait();  // s_a is written by the kernel this one depends on
      const int at = threadIdx.x - 32 * C::kAWarp;  // 0..63
      if (at < MPAD) ctl->sa_s[at] = at < Mb ? __ldg(g.s_a + m_base + at) : 0.0f;
      bool ok = true;
      for (int i = 0; i < nk; ++i) {
        const int buf = i % kI8OpBufs, s = i % stages;
        bool w = mbar_wait(&ctl->full_a[s], static_cast<uint32_t>(i / stages) & 1u, g.wait_ns);
        if (i >= kI8OpBufs)
          w = w && mbar_wait(&ctl->op_empty[buf], static_cast<uint32_t>(i / kI8OpBufs - 1) & 1u, g.wait_ns);
        if (!__all_sync(0xffffffffu, w && !*abort_flag)) {
          ok = false;
          break;
        }
        // activation tile -> fp16, swizzled K-major B operand (2 atoms of 64 K)
        const uint8_t* src = smem + static_cast<size_t>(s) * kStage + S::kWBytes;
        uint8_t* ob = opb + buf * S::kOpBBytes;
#pragma unroll
        for (int piece = at; piece < MPAD * 4; piece += 32 * kI8AWarps) {
          const uint32_t r = piece >> 2, p = piece & 3;  // row, 32-element quarter of the 128 K
          const uint4 v0 = *reinterpret_cast<const uint4*>(src + sw128_chunk(r, 2 * p));
          const uint4 v1 = *reinterpret_cast<const uint4*>(src + sw128_chunk(r, 2 * p + 1));
          uint32_t o[16];
          int8x4_to_f16x4(v0.x, o[0], o[1]);
          int8x4_to_f16x4(v0.y, o[2], o[3]);
          int8x4_to_f16x4(v0.z, o[4], o[5]);
          int8x4_to_f16x4(v0.w, o[6], o[7]);
          int8x4_to_f16x4(v1.x, o[8], o[9]);
          int8x4_to_f16x4(v1.y, o[10], o[11]);
          int8x4_to_f16x4(v1.z, o[12], o[13]);
          int8x4_to_f16x4(v1.w, o[14], o[15]);
          uint8_t* atom = ob + (p >> 1) * (MPAD * 128);
          const uint32_t c0 = (p & 1) * 4;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            *reinterpret_cast<uint4*>(atom + sw128_chunk(r, c0 + j)) =
                make_uint4(o[4 * j], o[4 * j + 1], o[4 * j + 2], o[4 * j + 3]);
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ctl->op_full[buf]);
          mbar_arrive(&ctl->empty[s]);
        }
      }
      if (!ok) *abort_flag = 1;
    } else {
      // ------------------------------------------------- weight converters
      // They read only the static weights, so they start before the
      // activations exist (no dependency wait here).
      const uint32_t lane_base = ((warp & 3) * 32u) << 16;
      if (h == 0) {
        const int nn = n_tile * kBN + static_cast<int>(row);
        ctl->sw_s[row] = nn < g.N ? __ldg(s_w + nn) : 0.0f;
      }
      bool ok = true;

      auto drain = [&](int seg) -> bool {
        const int d = seg & 1;
        bool w = mbar_wait(&ctl->d_full[d], static_cast<uint32_t>(seg / 2) & 1u, g.wait_ns);
        if (!__all_sync(0xffffffffu, w && !*abort_flag)) return false;
        tc_fence_after();
        if constexpr (kHalf % 8 == 0) {
#pragma unroll
          for (int c = 0; c < kHalf; c += 8) {
            uint32_t t[8];
            tmem_ld_x8(tmem_d + lane_base + d * S::kDCols + h * kHalf + c, t);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 8; ++j) iacc[c + j] += __float2int_rn(__uint_as_float(t[j]));
          }
        } else {
#pragma unroll
          for (int c = 0; c < kHalf; c += 4) {
            uint32_t t[4];
            tmem_ld_x4(tmem_d + lane_base + d * S::kDCols + h * kHalf + c, t);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 4; ++j) iacc[c + j] += __float2int_rn(__uint_as_float(t[j]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->d_empty[d]);
        return true;
      };

      for (int i = 0; i < nk; ++i) {
        const int seg = i / kI8SegTiles, buf = i % kI8OpBufs, s = i % stages;
        if ((i % kI8SegTiles) == 0 && seg >= 2 && !drain(seg - 2)) {
          ok = false;
          break;
        }
        bool w = mbar_wait(&ctl->full[s], static_cast<uint32_t>(i / stages) & 1u, g.wait_ns);
        if (i >= kI8OpBufs)
          w = w && mbar_wait(&ctl->op_empty[buf], static_cast<uint32_t>(i / kI8OpBufs - 1) & 1u, g.wait_ns);
        if (!__all_sync(0xffffffffu, w && !*abort_flag)) {
          ok = false;
          break;
        }
        const uint8_t* st = smem + static_cast<size_t>(s) * kStage;
        // this thread's 64 weight bytes -> fp16 -> TMEM operand buffer
#pragma unroll
        for (int c = C::kChunks * h; c < C::kChunks * (h + 1); ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(st + sw128_chunk(row, c));
          uint32_t o[8];
          int8x4_to_f16x4(v.x, o[0], o[1]);
          int8x4_to_f16x4(v.y, o[2], o[3]);
          int8x4_to_f16x4(v.z, o[4], o[5]);
          int8x4_to_f16x4(v.w, o[6], o[7]);
          tmem_st_x8(tmem_a + lane_base + buf * S::kACols + c * 8, o);
        }
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&ctl->op_full[buf]);
          mbar_arrive(&ctl->empty[s]);
        }
      }
      if (ok) {
        for (int seg = nseg > 2 ? nseg - 2 : 0; seg < nseg; ++seg)
          if (!drain(seg)) {
            ok = false;
            break;
          }
      }
      if (!ok) *abort_flag = 1;
      mbar_wait(&ctl->done, 0, g.wait_ns);
    }
  }
  // ------------------------------------------- all roles done: TMEM free
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(ctl->tmem_base, S::kTmemCols);
  }
  const bool abort = ctl->abort_flag != 0;  // stable after the barrier: uniform
  pdl_wait();  // outputs are written only after the kernel this one depends on
  const int n = n_tile * kBN + static_cast<int>(row);
  const int ct = threadIdx.x - 64;
  // m: token of this block; r: row of the tile (scales staged in shared
  // memory); nn = n_tile*128 + r
  auto finish = [&](int m, int r, int nn, int32_t acc) {
    if (g.debug_acc) g.debug_acc[static_cast<int64_t>(m_base + m) * g.N + nn] = acc;
    const float y = (static_cast<float>(acc) * ctl->sa_s[m]) * ctl->sw_s[r];
    store_bf16(g.Y + static_cast<int64_t>(m_base + m) * g.ldy + nn, y);
  };

  const bool holds_acc = warp >= 2 && warp < C::kAWarp;
  if (PREW && holds_acc) {
    // no activation warps staged the token scales: the accumulator threads do
    if (ct < MPAD) ctl->sa_s[ct] = ct < Mb ? __ldg(g.s_a + m_base + ct) : 0.0f;
    named_bar_sync(1, C::kThreads);
  }
  if (clustered) {
    if (holds_acc) {
      cluster_wait();  // every peer's receive barrier is initialized
      // rows go out even after an abort, so that every owner's wait completes
      cluster_push_row(iacc, h * kHalf, static_cast<int>(row), split, g.splits, Mb, recv, &ctl->recv_bar);
      named_bar_sync(1, C::kThreads);  // this CTA's own rows, stored locally, are visible
      const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(&ctl->recv_bar, 0, g.wait_ns));
      if (got && !abort) {
        cluster_sum_rows<int32_t>(recv, split, g.splits, Mb, ct, C::kThreads, [&](int m, int r, int32_t sum) {
          const int nn = n_tile * kBN + r;
          if (nn < g.N) finish(m, r, nn, sum);
        });
      }
    } else if (!(FUSED && warp >= C::kAWarp)) {
      // the other warps pair their early arrive with a wait too (every peer
      // arrived right after its set-up, so this returns at once); the fused
      // quantizer warps waited before their row-maximum exchange
      cluster_wait();
    }
  } else if (holds_acc && !abort) {
    const bool n_ok = n < g.N;
    if (g.reduce == kReduceNone) {
      if (n_ok) {
#pragma unroll
        for (int j = 0; j < kHalf; ++j)
          if (h * kHalf + j < Mb) finish(h * kHalf + j, static_cast<int>(row), n, iacc[j]);
      }
    } else {
      int32_t* part = static_cast<int32_t*>(g.ws_part);
      if (n_ok) {
#pragma unroll
        for (int j = 0; j < kHalf; ++j) {
          const int m = h * kHalf + j;
          if (m < Mb) part[(static_cast<int64_t>(split) * g.M + m_base + m) * g.N + n] = iacc[j];
        }
      }
      __threadfence();
      named_bar_sync(1, C::kThreads);
      const int tile_id = blockIdx.x + blockIdx.z * gridDim.x;
      if (ct == 0) ctl->last_flag = (atomicAdd(g.ws_count + tile_id, 1) == g.splits - 1);
      named_bar_sync(1, C::kThreads);
      if (ctl->last_flag) {
        __threadfence();
        if (n_ok) {
          for (int j = 0; j < kHalf; ++j) {
            const int m = h * kHalf + j;
            if (m >= Mb) break;
            int32_t sum = 0;
            for (int s = 0; s < g.splits; ++s)
              sum += ld_cg_s32(part + (static_cast<int64_t>(s) * g.M + m_base + m) * g.N + n);
            finish(m, static_cast<int>(row), n, sum);
          }
        }
        if (ct == 0) g.ws_count[tile_id] = 0;
      }
    }
  }
  stamp_end(g.tstamp);
}

}  // namespace qg
