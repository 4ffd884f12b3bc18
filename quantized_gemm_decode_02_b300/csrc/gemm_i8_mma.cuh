// gemm_i8_mma.cuh -- W8A8_INT8 Swap-AB GEMM on the warp-level tensor-core
// instructions (mma.sync m16n8k16, f16 operands, f32 accumulate), with the
// int8 operands widened to f16 in registers.
//
// "W8A8_INT8: INT8 per-token activation and per-channel weight scaling"
// ("Building a High-Performance and Portable vLLM Linear Backend with
// Helion", section "Helion Linear Backend > Scope") needs the exact int32
// accumulator.  sm_103a has no int8 kind of tcgen05.mma, so every weight
// byte must be widened to f16 before a tensor core can use it.  The tcgen05
// kernel (gemm_i8.cuh) widens into a TMEM operand buffer and hands each
// k-tile to the MMA thread through mbarriers; here each warp widens its own
// weight rows straight into mma.sync fragment registers, so a k-tile needs
// no TMEM store, no fence and no handoff between warps.  Products of int8
// values are integers below 2^14 and every partial sum over at most 1024 K
// stays below 2^24, so the fp32 accumulators are exact for a 1024-K segment;
// segments are converted to int32 and summed in registers, as in the
// tcgen05 kernel.
//
// K order inside a fragment.  A sum over k does not depend on the order of
// its terms, so the kernel feeds both operands the same permutation of each
// 128-wide k-tile: for the 16-wide MMA step c (0..7), the lane with
// threadID_in_group t takes physical k = 32t + 4c + {0,1} as the fragment's
// logical k = 2t + {0,1} and physical 32t + 4c + {2,3} as logical
// 2t + 8 + {0,1}.  A lane thus reads 32 contiguous bytes of a row per
// k-tile (two 16-byte shared-memory loads), and one 32-bit word of four int8
// values becomes the two f16x2 fragment registers of one step.
//
// CTA = 2 + 8/TPW warps, one 128-row weight tile x one K range x one block
// of up to 32 tokens (NG groups of 8, the MMA N side):
//   warp 0      TMA: int8 W tile (128 x 128 B, 128-byte swizzle) and the
//               int8 activation tile (8*NG token rows, zero-filled past M)
//               into a `stages`-deep ring, weights and activations on
//               separate barriers (weights fetched before the dependency
//               wait);
//   MMA warps   8/TPW warps of 16*TPW weight rows each (TPW m16 tiles; TPW
//               = 2: four warps, TPW = 1: eight warps, twice the warps
//               to hide the widening's latency): per k-tile 4*TPW shared
//               loads of 16 bytes, 8 steps of widening and TPW*NG MMAs
//               per step;
//   last warp   widens the activation tile once per k-tile into f16
//               fragments in shared memory ([step][group][lane], 8 bytes),
//               read by every MMA warp.
// With S8 the products run on the int8 form of the instruction instead
// (mma.sync m16n8k32, s8 operands, s32 accumulate): no widening at all, and
// the exact int32 sum needs no segments.  The K permutation becomes: for the
// 32-wide step c (0..3) the lane takes physical k = 32t + 8c + {0..3} as the
// fragment's logical 4t + {0..3} and 32t + 8c + {4..7} as 16 + 4t + {0..3},
// so it still reads the same 32 contiguous bytes of each of its rows per
// k-tile, and each MMA warp takes its activation fragments straight from the
// stage's activation tile (the last warp only loads the activation scales).
// B300 runs this instruction far below its FP8 rate (about 143 TOPS measured
// on the part), which bounds the form to small token counts.
// With DPW > 0 (eight-warp layout, up to 16 tokens) the first 16*DPW weight
// rows go to DPW warps of dp4a threads instead (two per row, a K half each,
// exact int32 sums as in gemm_i8_dp4a.cuh): dp4a runs on the integer pipe,
// which the MMAs leave idle, so the two parts of the tile proceed side by
// side (with the widening form the widening competes for that pipe; with
// S8 nothing does).
// The epilogue, the Split-K reduction (cluster push or workspace) and the
// scales are those of the other Swap-AB kernels, one thread per weight row.
#pragma once
#include "common.cuh"
#include "gemm_f8.cuh"
#include "gemm_i8.cuh"

namespace qg {

// MMA warps (1 .. 8/TPW) of 16*TPW weight rows each, then the activation
// widening warp; the first four MMA warps' 128 threads run the per-row
// epilogue
__host__ __device__ constexpr int ms_mma_warps(int tpw) { return 8 / tpw; }
__host__ __device__ constexpr int ms_threads(int tpw) { return 32 * (ms_mma_warps(tpw) + 2); }
constexpr int kMsABufs = 3;                          // f16 activation fragment buffers in flight
constexpr int kMsMaxGroups = 4;                      // token groups of 8 per block (32 tokens)

struct alignas(8) CtrlMs {
  uint64_t full[16];    // weight tile of the stage landed
  uint64_t full_a[16];  // activation tile of the stage landed
  uint64_t empty[16];   // every lane of the MMA warps and of the activation warp is done with the stage
  uint64_t afull[kMsABufs];
  uint64_t aempty[kMsABufs];
  uint64_t recv_bar;    // split-K: peers' partial rows have landed
  uint64_t never;       // the forced-timeout test hook waits on it (nothing arrives)
  int last_flag;
  int abort_flag;
  float sa_s[8 * kMsMaxGroups];
  float sw_s[kBN];
};

template <int NG>
struct MsShape {
  static constexpr int kMpad = 8 * NG;                     // tokens per block (MMA N x groups)
  static constexpr uint32_t kWBytes = kBN * kBK;           // 16 KB int8 weights
  static constexpr uint32_t kABytes = kMpad * kBK;         // int8 activations
  // stage starts stay 1024-byte aligned (128-byte swizzle atoms)
  static constexpr uint32_t kStageBytes = (kWBytes + kABytes + 1023u) & ~1023u;
  static constexpr uint32_t kFragBytes = 8u * NG * 32u * 8u;  // [step][group][lane] x (b0, b1)
  static constexpr int kAccStride = kMpad + 4;              // int32 words per row of the epilogue tile
};

template <int NG>
__host__ __device__ constexpr size_t gemm_i8_mma_smem_bytes(int stages, int recv_bytes = 0) {
  return 1024 + static_cast<size_t>(stages) * MsShape<NG>::kStageBytes +
         static_cast<size_t>(kMsABufs) * MsShape<NG>::kFragBytes + recv_bytes + sizeof(CtrlMs);
}

// D += A . B for one m16n8k16 step: A 16x16 f16 (row), B 16x8 f16 (col), D f32.
__device__ __forceinline__ void mma_16816_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                              uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D += A . B for one m16n8k32 step: A 16x32 s8 (row), B 32x8 s8 (col), D s32.
__device__ __forceinline__ void mma_16832_s8(int32_t (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                             uint32_t b0, uint32_t b1) {
  asm("mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t word_of(const uint4& v, int j) {
  return j == 0 ? v.x : (j == 1 ? v.y : (j == 2 ? v.z : v.w));
}

template <int NG, int TPW, int DPW, bool S8>
__global__ void __launch_bounds__(ms_threads(TPW), 2)
    gemm_i8_mma_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA, GemmArgs g) {
  using S = MsShape<NG>;
  constexpr int MPAD = S::kMpad;
  static_assert(DPW == 0 || (TPW == 1 && NG <= 2 && DPW <= 4), "dp4a rows: eight-warp layout, up to 16 tokens");
  constexpr int kRD = 16 * DPW;                      // weight rows on dp4a (rows 0 .. kRD-1)
  constexpr int kMsWarps = ms_mma_warps(TPW) - DPW;  // MMA warps 1..kMsWarps (rows kRD ..)
  constexpr int kMsAWarp = 1 + kMsWarps + DPW;       // activation widening warp (dp4a warps before it)
  constexpr int kEpi = 128;                          // per-row epilogue threads (warps 1..4)
  stamp_start(g.tstamp);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stages = g.stages;
  uint8_t* frag = smem + static_cast<size_t>(stages) * S::kStageBytes;  // f16 activation fragments
  uint8_t* recv = frag + kMsABufs * S::kFragBytes;                       // split-K receive buffer
  CtrlMs* ctl = reinterpret_cast<CtrlMs*>(recv + g.recv_bytes);
  const bool clustered = g.reduce == kReduceCluster;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gid = lane >> 2, tig = lane & 3;  // the MMA fragment coordinates of this lane
  // the token blocks of one weight tile are adjacent block indices (weights
  // read from HBM once, then from L2)
  const int n_tile = static_cast<int>(blockIdx.x / g.m_tiles), split = blockIdx.y;
  const int m_blk = static_cast<int>(blockIdx.x % g.m_tiles);
  const GroupView grp = group_view(g);
  const int m_base = grp.tok0 + m_blk * MPAD;
  const int Mb = min(MPAD, grp.tok0 + grp.tokens - m_base);
  if (Mb <= 0) return;  // a token block past its group's tokens (the whole cluster alike)
  const int w_row0 = static_cast<int>(blockIdx.z) * g.N;
  const float* s_w = g.s_w + static_cast<int64_t>(blockIdx.z) * g.sw_group_stride;
  const int kb0 = static_cast<int>(static_cast<int64_t>(split) * g.kt_total / g.splits);
  const int kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * g.kt_total / g.splits);
  const int nk = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->full_a[i], 1);
      mbar_init(&ctl->empty[i], 32 * (kMsWarps + DPW + (S8 ? 0 : 1)));
    }
    for (int b = 0; b < kMsABufs; ++b) {
      mbar_init(&ctl->afull[b], 32);
      mbar_init(&ctl->aempty[b], 32 * kMsWarps);
    }
    mbar_init(&ctl->recv_bar, 1);
    mbar_init(&ctl->never, 1);
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
    if (threadIdx.x == 0)
      mbar_arrive_expect_tx(&ctl->recv_bar, static_cast<uint32_t>((g.splits - 1) * cluster_rows_of(split, g.splits) *
                                                                  cluster_mv(Mb) * 4));
    cluster_arrive_relaxed();
  }
  pdl_launch_dependents();
  volatile int* abort_flag = &ctl->abort_flag;

  // MMA warps: int32 sums of weight rows r0 = 32*cw + 16*t + gid and r0 + 8
  // for tokens 8*grp + 2*tig + {0,1} (the D fragment layout)
  // dp4a threads: int32 sums of their row's K half for every token
  int32_t dacc[DPW > 0 ? MPAD : 1];
#pragma unroll
  for (int m = 0; m < (DPW > 0 ? MPAD : 1); ++m) dacc[m] = 0;
  int32_t iacc[TPW][NG][4];
#pragma unroll
  for (int t = 0; t < TPW; ++t)
#pragma unroll
    for (int q = 0; q < NG; ++q)
#pragma unroll
      for (int j = 0; j < 4; ++j) iacc[t][q][j] = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      const int w_row = w_row0 + n_tile * kBN;
      const int pre = nk < stages ? nk : stages;
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = smem + static_cast<size_t>(i) * S::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full[i], S::kWBytes);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[i], pol_w);
      }
      for (int i = pre; i < nk && i < pre + g.l2_prefetch; ++i) tma_prefetch_l2_2d(&tmW, (kb0 + i) * kBK, w_row);
      pdl_wait();  // the activations come from the kernel this one depends on
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = smem + static_cast<size_t>(i) * S::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full_a[i], S::kABytes);
        tma_load_2d(st + S::kWBytes, &tmA, (kb0 + i) * kBK, m_base, &ctl->full_a[i], pol_a);
      }
      int issued = pre;
      for (int i = pre; i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
        if (!mbar_wait(&ctl->empty[s], ph ^ 1u, g.wait_ns) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(s) * S::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full[s], S::kWBytes);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[s], pol_w);
        if (g.l2_prefetch > 0 && i + g.l2_prefetch < nk) tma_prefetch_l2_2d(&tmW, (kb0 + i + g.l2_prefetch) * kBK, w_row);
        mbar_arrive_expect_tx(&ctl->full_a[s], S::kABytes);
        tma_load_2d(st + S::kWBytes, &tmA, (kb0 + i) * kBK, m_base, &ctl->full_a[s], pol_a);
        issued = i + 1;
      }
      // every issued copy lands before the CTA may exit or reuse the ring
      for (int j = issued > stages ? issued - stages : 0; j < issued; ++j) {
        mbar_wait(&ctl->full[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
        mbar_wait(&ctl->full_a[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
      }
    }
  } else if (warp == kMsAWarp) {
    // ------------------------------------------- activation widening warp
    pdl_wait();  // s_a is written by the kernel this one depends on
    if (lane < MPAD) ctl->sa_s[lane] = lane < Mb ? __ldg(g.s_a + m_base + lane) : 0.0f;
    bool ok = true;
    for (int i = 0; !S8 && i < nk; ++i) {
      const int s = i % stages, b = i % kMsABufs;
      bool w = mbar_wait(&ctl->full_a[s], static_cast<uint32_t>(i / stages) & 1u, g.wait_ns);
      if (i >= kMsABufs)
        w = w && mbar_wait(&ctl->aempty[b], static_cast<uint32_t>(i / kMsABufs - 1) & 1u, g.wait_ns);
      if (!__all_sync(0xffffffffu, w && !*abort_flag)) {
        ok = false;
        break;
      }
      const uint8_t* at = smem + static_cast<size_t>(s) * S::kStageBytes + S::kWBytes;
      uint8_t* fb = frag + b * S::kFragBytes;
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        const uint32_t r = static_cast<uint32_t>(8 * q + gid);  // token row of the tile
        const uint4 v0 = *reinterpret_cast<const uint4*>(at + sw128_chunk(r, 2 * tig));
        const uint4 v1 = *reinterpret_cast<const uint4*>(at + sw128_chunk(r, 2 * tig + 1));
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t lo, hi;
          int8x4_to_f16x4(word_of(c < 4 ? v0 : v1, c & 3), lo, hi);
          *reinterpret_cast<uint2*>(fb + ((c * NG + q) * 32 + lane) * 8) = make_uint2(lo, hi);
        }
      }
      mbar_arrive(&ctl->empty[s]);  // this lane's reads of the stage are done
      mbar_arrive(&ctl->afull[b]);  // this lane's fragments are written (release)
    }
    if (!ok) *abort_flag = 1;
  } else if (DPW > 0 && warp > kMsWarps) {
    // ---------------------------------------------------------- dp4a warps
    const int d = static_cast<int>(threadIdx.x) - 32 * (1 + kMsWarps);  // 0 .. 32*DPW-1
    const int row = d % (kRD > 0 ? kRD : 1), h = d / (kRD > 0 ? kRD : 1);  // weight row, K half
    bool ok = true;
    for (int i = 0; i < nk; ++i) {
      const int s = i % stages;
      const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
      const bool w = mbar_wait(&ctl->full[s], ph, g.wait_ns) && mbar_wait(&ctl->full_a[s], ph, g.wait_ns);
      if (!__all_sync(0xffffffffu, w && !*abort_flag)) {
        ok = false;
        break;
      }
      const uint8_t* wt = smem + static_cast<size_t>(s) * S::kStageBytes;
      const uint8_t* at = wt + S::kWBytes;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        const int c = 4 * h + cc;
        const uint4 wv = *reinterpret_cast<const uint4*>(wt + sw128_chunk(static_cast<uint32_t>(row), c));
#pragma unroll
        for (int m = 0; m < (DPW > 0 ? MPAD : 1); ++m) {
          const uint4 av = *reinterpret_cast<const uint4*>(at + sw128_chunk(static_cast<uint32_t>(m), c));
          int32_t a = dacc[m];
          a = __dp4a(static_cast<int>(wv.x), static_cast<int>(av.x), a);
          a = __dp4a(static_cast<int>(wv.y), static_cast<int>(av.y), a);
          a = __dp4a(static_cast<int>(wv.z), static_cast<int>(av.z), a);
          a = __dp4a(static_cast<int>(wv.w), static_cast<int>(av.w), a);
          dacc[m] = a;
        }
      }
      mbar_arrive(&ctl->empty[s]);  // this lane's reads of the stage are done
    }
    if (!ok) *abort_flag = 1;
  } else {
    // ---------------------------------------------------------- MMA warps
    const int cw = warp - 1;
    // test hook (qg_set_force_timeout): wait on a barrier nothing arrives on
    bool ok = !g.force_timeout || __all_sync(0xffffffffu, mbar_wait(&ctl->never, 0, g.wait_ns));
    if constexpr (S8) {
      for (int i = 0; ok && i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&ctl->full[s], ph, g.wait_ns) &&
                                         mbar_wait(&ctl->full_a[s], ph, g.wait_ns) && !*abort_flag)) {
          ok = false;
          break;
        }
        // this lane's 32 bytes of k of its weight rows and of its token rows
        const uint8_t* wt = smem + static_cast<size_t>(s) * S::kStageBytes;
        const uint8_t* at = wt + S::kWBytes;
        uint4 wv[TPW][2][2], av[NG][2];
#pragma unroll
        for (int t = 0; t < TPW; ++t)
#pragma unroll
          for (int rr = 0; rr < 2; ++rr) {
            const uint32_t row = static_cast<uint32_t>(kRD + 16 * TPW * cw + 16 * t + 8 * rr + gid);
#pragma unroll
            for (int hh = 0; hh < 2; ++hh)
              wv[t][rr][hh] = *reinterpret_cast<const uint4*>(wt + sw128_chunk(row, 2 * tig + hh));
          }
#pragma unroll
        for (int q = 0; q < NG; ++q)
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            av[q][hh] = *reinterpret_cast<const uint4*>(at + sw128_chunk(static_cast<uint32_t>(8 * q + gid), 2 * tig + hh));
        mbar_arrive(&ctl->empty[s]);  // both tiles are in registers
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int hh = c >> 1, j = 2 * (c & 1);
#pragma unroll
          for (int q = 0; q < NG; ++q) {
            const uint32_t b0 = word_of(av[q][hh], j), b1 = word_of(av[q][hh], j + 1);
#pragma unroll
            for (int t = 0; t < TPW; ++t)
              mma_16832_s8(iacc[t][q], word_of(wv[t][0][hh], j), word_of(wv[t][1][hh], j), word_of(wv[t][0][hh], j + 1),
                           word_of(wv[t][1][hh], j + 1), b0, b1);
          }
        }
      }
      if (!ok) *abort_flag = 1;
    } else {
    float facc[TPW][NG][4];
#pragma unroll
    for (int t = 0; t < TPW; ++t)
#pragma unroll
      for (int q = 0; q < NG; ++q)
#pragma unroll
        for (int j = 0; j < 4; ++j) facc[t][q][j] = 0.0f;
    for (int i = 0; ok && i < nk; ++i) {
      const int s = i % stages, b = i % kMsABufs;
      if (!__all_sync(0xffffffffu, mbar_wait(&ctl->full[s], static_cast<uint32_t>(i / stages) & 1u, g.wait_ns) &&
                                       !*abort_flag)) {
        ok = false;
        break;
      }
      // this lane's 32 bytes of k of the four rows it holds: [tile][row r0 / r0 + 8][16-byte half]
      const uint8_t* wt = smem + static_cast<size_t>(s) * S::kStageBytes;
      uint4 wv[TPW][2][2];
#pragma unroll
      for (int t = 0; t < TPW; ++t)
#pragma unroll
        for (int rr = 0; rr < 2; ++rr) {
          const uint32_t row = static_cast<uint32_t>(kRD + 16 * TPW * cw + 16 * t + 8 * rr + gid);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
            wv[t][rr][hh] = *reinterpret_cast<const uint4*>(wt + sw128_chunk(row, 2 * tig + hh));
        }
      if (!__all_sync(0xffffffffu,
                      mbar_wait(&ctl->afull[b], static_cast<uint32_t>(i / kMsABufs) & 1u, g.wait_ns) && !*abort_flag)) {
        ok = false;
        break;
      }
      const uint8_t* fb = frag + b * S::kFragBytes;
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        uint32_t a[TPW][4];
#pragma unroll
        for (int t = 0; t < TPW; ++t) {
          uint32_t lo0, hi0, lo1, hi1;
          int8x4_to_f16x4(word_of(wv[t][0][c >> 2], c & 3), lo0, hi0);
          int8x4_to_f16x4(word_of(wv[t][1][c >> 2], c & 3), lo1, hi1);
          a[t][0] = lo0;  // row gid,     k 2t, 2t+1
          a[t][1] = lo1;  // row gid + 8, k 2t, 2t+1
          a[t][2] = hi0;  // row gid,     k 2t+8, 2t+9
          a[t][3] = hi1;  // row gid + 8, k 2t+8, 2t+9
        }
#pragma unroll
        for (int q = 0; q < NG; ++q) {
          const uint2 bv = *reinterpret_cast<const uint2*>(fb + ((c * NG + q) * 32 + lane) * 8);
#pragma unroll
          for (int t = 0; t < TPW; ++t) mma_16816_f16(facc[t][q], a[t][0], a[t][1], a[t][2], a[t][3], bv.x, bv.y);
        }
      }
      mbar_arrive(&ctl->empty[s]);   // the weight bytes are consumed (in registers)
      mbar_arrive(&ctl->aempty[b]);  // the fragments are consumed
      // close an exact 1024-K segment (or the range) into int32
      if ((i % kI8SegTiles) == kI8SegTiles - 1 || i == nk - 1) {
#pragma unroll
        for (int t = 0; t < TPW; ++t)
#pragma unroll
          for (int q = 0; q < NG; ++q)
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              iacc[t][q][j] += __float2int_rn(facc[t][q][j]);
              facc[t][q][j] = 0.0f;
            }
      }
    }
    if (!ok) *abort_flag = 1;
    }
  }
  // ------------------------------------------------- per-row accumulators
  __syncthreads();  // the ring is idle: every issued copy was consumed by the MMA warps
  const bool abort = ctl->abort_flag != 0;  // stable after the barrier: uniform
  // [128 rows][kAccStride] over the idle ring, then (dp4a rows) the second
  // K half's sums [kRD rows][kAccStride]
  int32_t* acc_s = reinterpret_cast<int32_t*>(smem);
  int32_t* acc2_s = acc_s + kBN * S::kAccStride;
  if (warp >= 1 && warp <= kMsWarps) {
    const int cw = warp - 1;
#pragma unroll
    for (int t = 0; t < TPW; ++t)
#pragma unroll
      for (int q = 0; q < NG; ++q) {
        const int row = kRD + 16 * TPW * cw + 16 * t + gid, m = 8 * q + 2 * tig;
        *reinterpret_cast<int2*>(acc_s + row * S::kAccStride + m) = make_int2(iacc[t][q][0], iacc[t][q][1]);
        *reinterpret_cast<int2*>(acc_s + (row + 8) * S::kAccStride + m) = make_int2(iacc[t][q][2], iacc[t][q][3]);
      }
  } else if (DPW > 0 && warp > kMsWarps && warp < kMsAWarp) {
    const int d = static_cast<int>(threadIdx.x) - 32 * (1 + kMsWarps);
    const int row = d % (kRD > 0 ? kRD : 1), h = d / (kRD > 0 ? kRD : 1);
    int32_t* dst = (h == 0 ? acc_s : acc2_s) + row * S::kAccStride;
#pragma unroll
    for (int m = 0; m < (DPW > 0 ? MPAD : 1); ++m) dst[m] = dacc[m];
  }
  const bool holds_row = warp >= 1 && warp <= kEpi / 32;
  const int ct = threadIdx.x - 32;  // row of the tile (warps 1..4)
  if (holds_row) {
    const int nn = n_tile * kBN + ct;
    ctl->sw_s[ct] = nn < g.N ? __ldg(s_w + nn) : 0.0f;
  }
  __syncthreads();
  pdl_wait();  // outputs are written only after the kernel this one depends on
  int32_t acc[MPAD];
  if (holds_row) {
#pragma unroll
    for (int m = 0; m < MPAD; m += 2) {
      const int2 v = *reinterpret_cast<const int2*>(acc_s + ct * S::kAccStride + m);
      acc[m] = v.x;
      acc[m + 1] = v.y;
    }
    if (DPW > 0 && ct < kRD) {
#pragma unroll
      for (int m = 0; m < MPAD; ++m) acc[m] += acc2_s[ct * S::kAccStride + m];
    }
  }
  auto finish = [&](int m, int r, int nn, int32_t sum) {
    if (g.debug_acc) g.debug_acc[static_cast<int64_t>(m_base + m) * g.N + nn] = sum;
    const float y = (static_cast<float>(sum) * ctl->sa_s[m]) * ctl->sw_s[r];
    store_bf16(g.Y + static_cast<int64_t>(m_base + m) * g.ldy + nn, y);
  };
  const int n = n_tile * kBN + ct;
  if (clustered) {
    if (holds_row) {
      cluster_wait();  // every peer's receive barrier is initialized
      // rows go out even after an abort, so that every owner's wait completes
      cluster_push_row(acc, 0, ct, split, g.splits, Mb, recv, &ctl->recv_bar);
      named_bar_sync(1, kEpi);  // this CTA's own rows, stored locally, are visible
      const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(&ctl->recv_bar, 0, g.wait_ns));
      if (got && !abort) {
        cluster_sum_rows<int32_t>(recv, split, g.splits, Mb, ct, kEpi, [&](int m, int r, int32_t sum) {
          const int nn = n_tile * kBN + r;
          if (nn < g.N) finish(m, r, nn, sum);
        });
      }
    } else {
      // the other warps pair their early arrive with a wait too (every peer
      // arrived right after its set-up, so this returns at once)
      cluster_wait();
    }
  } else if (holds_row && !abort) {
    const bool n_ok = n < g.N;
    if (g.reduce == kReduceNone) {
      if (n_ok) {
#pragma unroll
        for (int m = 0; m < MPAD; ++m)
          if (m < Mb) finish(m, ct, n, acc[m]);
      }
    } else {
      int32_t* part = static_cast<int32_t*>(g.ws_part);
      if (n_ok) {
#pragma unroll
        for (int m = 0; m < MPAD; ++m)
          if (m < Mb) part[(static_cast<int64_t>(split) * g.M + m_base + m) * g.N + n] = acc[m];
      }
      __threadfence();
      named_bar_sync(1, kEpi);
      const int tile_id = blockIdx.x + blockIdx.z * gridDim.x;
      if (ct == 0) ctl->last_flag = (atomicAdd(g.ws_count + tile_id, 1) == g.splits - 1);
      named_bar_sync(1, kEpi);
      if (ctl->last_flag) {
        __threadfence();
        if (n_ok) {
          for (int m = 0; m < Mb; ++m) {
            int32_t sum = 0;
            for (int s = 0; s < g.splits; ++s)
              sum += ld_cg_s32(part + (static_cast<int64_t>(s) * g.M + m_base + m) * g.N + n);
            finish(m, ct, n, sum);
          }
        }
        if (ct == 0) g.ws_count[tile_id] = 0;
      }
    }
  }
  stamp_end(g.tstamp);
}

}  // namespace qg
