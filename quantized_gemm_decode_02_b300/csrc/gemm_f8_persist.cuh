// gemm_f8_persist.cuh -- persistent Standard-variant GEMM for FP8_Dynamic in
// the compute-bound regime (M of 64 and more tokens), with CTA pairs that
// share each weight tile.
//
// The Standard variant of "Building a High-Performance and Portable vLLM
// Linear Backend with Helion" (section "Kernel Implementation") puts the
// tokens on the MMA M side; the pages send token counts beyond their tuned
// range to other kernels ("Hybrid Dispatch"), here this library's own.
//
// Tiles: 128 tokens x RW weight rows per CTA (RW = 256, or 224 / 192 / 160
// so that a shape's tile count fills the resident clusters' last round
// better), D[128 x RW] fp32 in TMEM (tcgen05.mma.kind::f8f6f4, M = 128,
// N = RW, K = 32 per instruction).
// Pairs: the two CTAs of a thread-block cluster take the two 128-token
// halves of a 256-token pair tile and the same RW-row weight tile; CTA r
// loads weight rows [RW/2 r, RW/2 (r + 1)) of the tile with TMA multicast
// into both CTAs' shared memory, so each weight k-tile crosses from L2 to the
// SMs once per pair (at RW = 256 each CTA loads 16 KB of weights and 16 KB of
// activations per k-tile instead of 32 + 16).  A stage is refilled only when the MMAs of both
// CTAs are done with it (their commits arrive on both CTAs' empty barrier).
// Persistent: gridDim.x = 2 x clusters (at most one CTA per SM); cluster c
// takes pair tiles c, c + clusters, ..., token pair fastest, so the clusters
// running at the same time share weight tiles in L2.
// Double-buffered accumulator: two RW-column TMEM buffers; the MMA thread
// fills one tile's buffer while the epilogue warps drain the previous one.
//
// CTA = 6 warps: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer,
// warps 2..5 epilogue (thread = token row = TMEM lane).  Every wait is
// bounded; both CTAs of a pair end with a cluster barrier, so neither exits
// while its peer may still write into its shared memory.
//
// PAIR (QG_CONFIG_PAIR_MMA): the pair runs one tcgen05.mma.cta_group::2 per
// K step instead of one cta_group::1 MMA in each CTA: M = 256 tokens (128
// from each CTA's shared memory, each CTA's TMEM receiving its own 128
// rows), N = RW weight rows of which each CTA holds only its own half (the
// tensor cores of the pair exchange the halves), so at RW = 256 a stage is
// 16 KB of activations + 16 KB of weights per CTA (32 KB instead of 48:
// deeper ring) and no multicast is needed.  The even CTA (the leader) issues every MMA;
// both CTAs' TMA loads complete on the leader's full barrier (cta_group::2
// copies), its commits arrive on the barriers of both CTAs (multicast), the
// epilogue warps of both CTAs release an accumulator buffer by arriving on
// the leader's tempty barrier, and the TMEM is allocated and freed
// collectively by one warp of each CTA.
#pragma once
#include "common.cuh"
#include "gemm_f8.cuh"

namespace qg {

constexpr int kPsTok = 128;                       // tokens per CTA (MMA M)
constexpr int kPsRows = 256;                      // the largest weight-row tile (MMA N)
constexpr uint32_t kPsABytes = kPsTok * kBK;      // 16 KB

// A stage: the activation tile, then the weight rows of the tile (both
// multicast halves) or, PAIR, this CTA's half of them.
template <bool PAIR, int RW>
__host__ __device__ constexpr uint32_t ps_stage_bytes() {
  return kPsABytes + static_cast<uint32_t>(PAIR ? RW / 2 : RW) * kBK;
}

struct alignas(8) CtrlPs {
  uint64_t full[8];     // the stage's activation tile and both weight halves landed
  uint64_t empty[8];    // both CTAs' MMAs are done with the stage
  uint64_t tfull[2];    // accumulator buffer written (MMA commit)
  uint64_t tempty[2];   // accumulator buffer drained (epilogue)
  uint64_t never;       // the forced-timeout test hook waits on it
  uint64_t done;        // PAIR: every MMA of the pair has completed (leader's final commit)
  uint32_t tmem_base;
  int abort_flag;
  int epi_bad[4];          // per epilogue warp: its wait failed or the kernel aborted (this tile)
  float sw_s[2][kPsRows];  // per-channel scales of the buffer's weight tile
};

template <bool PAIR = false, int RW = kPsRows>
__host__ __device__ constexpr size_t gemm_f8_persist_smem_bytes(int stages) {
  return 1024 + static_cast<size_t>(stages) * ps_stage_bytes<PAIR, RW>() + sizeof(CtrlPs);
}

// 2-D TMA load multicast to the CTAs of ctaMask: the box lands at the same
// shared-memory offset in each of them and completes its bytes on the
// mbarrier at the same offset in each.
__device__ __forceinline__ void tma_load_2d_multicast(void* dst, const CUtensorMap* tm, int c0, int c1, uint64_t* bar,
                                                      uint16_t mask, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5, %6;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "h"(mask), "l"(policy)
      : "memory");
}
// Arrive on the mbarrier at the same offset in each CTA of ctaMask once every
// MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(mask)
               : "memory");
}

// ---- cta_group::2 forms (every tcgen05 instruction of a kernel takes the
// same cta_group) ----
// TMEM allocation for the CTA pair: one warp of each CTA executes it; the
// same columns are reserved in both CTAs' TMEM.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
// One MMA of the pair (issued by one thread of the leader): A rows from each
// CTA's shared memory at a_desc, B halves from each CTA's at b_desc, D rows
// of each CTA into its own TMEM at d_tmem.
__device__ __forceinline__ void mma_f8f6f4_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on the mbarrier at the same offset in each CTA of ctaMask once every
// pair MMA this thread issued before has completed.
__device__ __forceinline__ void tc_commit_pair_multicast(uint64_t* bar, uint16_t mask) {
  asm volatile("tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
                   smem_u32(bar)),
               "h"(mask)
               : "memory");
}
// 2-D TMA load into this CTA's shared memory whose bytes complete on the
// mbarrier at cluster address `cbar` (the leader's, for either CTA).
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* tm, int c0, int c1, uint32_t cbar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(tm)), "r"(c0), "r"(c1), "r"(cbar), "l"(policy)
      : "memory");
}
// Arrive (release, cluster scope) on the mbarrier at cluster address `cbar`.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cbar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cbar) : "memory");
}

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// One CTA of a pair.  g.m_tiles = pair tiles along the tokens (ceil(M/256)),
// g.kt_total = k-tiles; tiles = g.m_tiles * ceil(N/RW).  tmW's box is RW/2
// rows.
template <bool PAIR, int RW = kPsRows>
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f8_persist_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA, GemmArgs g) {
  static_assert(RW % 32 == 0 && RW >= 128 && RW <= kPsRows, "weight-row tiles of 128..256, halves of whole 16-row groups");
  constexpr uint32_t kStage = ps_stage_bytes<PAIR, RW>();
  constexpr int kHalfRows = RW / 2;                       // rows of one CTA's weight half
  constexpr uint32_t kTmemCols = pow2_cols(2 * RW);       // two accumulator buffers
  stamp_start(g.tstamp);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stages = g.stages;
  CtrlPs* ctl = reinterpret_cast<CtrlPs*>(smem + static_cast<size_t>(stages) * kStage);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();           // 0 or 1: token half of the pair tile
  const bool leader = rank == 0;
  const int cluster = static_cast<int>(blockIdx.x >> 1), clusters = static_cast<int>(gridDim.x >> 1);
  const int tp_count = g.m_tiles, wn_count = (g.N + RW - 1) / RW;
  const int tiles = tp_count * wn_count;
  const int nk = g.kt_total;

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], PAIR ? 1 : 2);  // PAIR: the leader's one commit; else one from each CTA
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->tfull[b], 1);
      mbar_init(&ctl->tempty[b], PAIR ? 8 : 128);  // PAIR: one arrive per epilogue warp of both CTAs
    }
    mbar_init(&ctl->never, 1);
    mbar_init(&ctl->done, 1);
    ctl->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmA);
  }
  // the peer's barriers are initialized before any copy or commit reaches
  // them (and, PAIR, before the collective TMEM allocation)
  cluster_sync();
  if (warp == 1) {
    if constexpr (PAIR) tmem_alloc_pair(&ctl->tmem_base, kTmemCols);
    else tmem_alloc(&ctl->tmem_base, kTmemCols);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_launch_dependents();
  volatile int* abort_flag = &ctl->abort_flag;
  // PAIR: cluster addresses of the leader's barriers
  const uint32_t full0 = dsmem_map(smem_u32(&ctl->full[0]), 0);
  const uint32_t tempty0 = dsmem_map(smem_u32(&ctl->tempty[0]), 0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      const uint16_t both = 0x3;
      // this CTA's weight half of tile t's k-tile kk into stage s (PAIR: its
      // own shared memory only; else multicast into both CTAs), and the
      // stage's activation tile
      auto load_w = [&](int s, int wn, int kk) {
        uint8_t* st = smem + static_cast<size_t>(s) * kStage;
        const int w_row = wn * RW + static_cast<int>(rank) * kHalfRows;
        if constexpr (PAIR)
          tma_load_2d_pair(st + kPsABytes, &tmW, kk * kBK, w_row, full0 + 8u * static_cast<uint32_t>(s), pol_w);
        else
          tma_load_2d_multicast(st + kPsABytes + rank * (kHalfRows * kBK), &tmW, kk * kBK, w_row, &ctl->full[s],
                                both, pol_w);
      };
      auto load_a = [&](int s, int a_row, int kk) {
        uint8_t* st = smem + static_cast<size_t>(s) * kStage;
        if constexpr (PAIR)
          tma_load_2d_pair(st, &tmA, kk * kBK, a_row, full0 + 8u * static_cast<uint32_t>(s), pol_a);
        else
          tma_load_2d(st, &tmA, kk * kBK, a_row, &ctl->full[s], pol_a);
      };
      // PAIR: the leader expects both CTAs' bytes of a stage on its barrier
      auto expect = [&](int s) {
        if (!PAIR) mbar_arrive_expect_tx(&ctl->full[s], kStage);
        else if (leader) mbar_arrive_expect_tx(&ctl->full[s], 2 * kStage);
      };
      // the weights of the first tile's first stages are requested before
      // the wait for the kernel this one depends on, its activations after
      const int first = cluster < tiles ? cluster : -1;
      const int pre = first >= 0 ? (nk < stages ? nk : stages) : 0;
      for (int kk = 0; kk < pre; ++kk) {
        expect(kk);
        load_w(kk, first / tp_count, kk);
      }
      // this CTA's weight half of the k-tile `ahead` k-tiles past (tile t,
      // k-tile kk) is requested into L2 (no shared memory): the ring then
      // only has to cover the L2 latency, not the HBM one
      const int ahead = g.l2_prefetch;
      auto prefetch_ahead = [&](int t, int kk) {
        int t2 = t, k2 = kk + ahead;
        while (k2 >= nk && t2 < tiles) {
          k2 -= nk;
          t2 += clusters;
        }
        if (t2 < tiles) tma_prefetch_l2_2d(&tmW, k2 * kBK, (t2 / tp_count) * RW + static_cast<int>(rank) * kHalfRows);
      };
      if (ahead > 0 && first >= 0)
        for (int kk = pre; kk < pre + ahead; ++kk) prefetch_ahead(first, kk - ahead);
      pdl_wait();
      int i = 0;  // k-tile counter over all of this CTA's tiles (the ring position)
      bool ok = true;
      for (int t = cluster; ok && t < tiles; t += clusters) {
        const int tp = t % tp_count, wn = t / tp_count;
        const int a_row = tp * 2 * kPsTok + static_cast<int>(rank) * kPsTok;
        for (int kk = 0; kk < nk; ++kk, ++i) {
          const int s = i % stages;
          if (ahead > 0 && i >= pre) prefetch_ahead(t, kk);
          if (i >= pre) {
            if (i >= stages && (!mbar_wait(&ctl->empty[s], (static_cast<uint32_t>(i / stages) & 1u) ^ 1u, g.wait_ns) ||
                                *abort_flag)) {
              ok = false;
              break;
            }
            expect(s);
            load_w(s, wn, kk);
          }
          load_a(s, a_row, kk);
        }
      }
      if (!ok) *abort_flag = 1;
      // every stage this CTA expects lands before the CTA may leave: its own
      // copies and the peer's half (the full barrier), or, for the PAIR
      // peer, whose copies complete on the leader's barrier, the MMAs that
      // consumed them (its empty barrier)
      for (int j = i > stages ? i - stages : 0; j < i; ++j) {
        if (PAIR && !leader)
          mbar_wait(&ctl->empty[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
        else
          mbar_wait(&ctl->full[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0 && (!PAIR || leader)) {
      // E4M3 x E4M3 -> F32: 128 x RW per CTA, or 256 x RW for the pair
      constexpr uint32_t idesc = make_idesc(PAIR ? 2 * kPsTok : kPsTok, RW, 0, 0);
      bool ok = !g.force_timeout || mbar_wait(&ctl->never, 0, g.wait_ns);
      int i = 0, lt = 0;
      for (int t = cluster; ok && t < tiles; t += clusters, ++lt) {
        const int b = lt & 1;
        if (lt >= 2) {
          const uint32_t par = (static_cast<uint32_t>(lt / 2) & 1u) ^ 1u;
          if (!(PAIR ? mbar_wait_cluster(&ctl->tempty[b], par, g.wait_ns) : mbar_wait(&ctl->tempty[b], par, g.wait_ns))) {
            ok = false;
            break;
          }
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b * RW);
        for (int kk = 0; kk < nk; ++kk, ++i) {
          const int s = i % stages;
          if (!mbar_wait(&ctl->full[s], static_cast<uint32_t>(i / stages) & 1u, g.wait_ns) || *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + static_cast<size_t>(s) * kStage);
          const uint32_t w_addr = a_addr + kPsABytes;
#pragma unroll
          for (int k4 = 0; k4 < kBK / 32; ++k4) {
            const uint32_t acc = (kk > 0 || k4 > 0) ? 1u : 0u;
            if constexpr (PAIR)
              mma_f8f6f4_pair(d, sw128_kmajor_desc(a_addr + k4 * 32), sw128_kmajor_desc(w_addr + k4 * 32), idesc, acc);
            else
              mma_f8f6f4(d, sw128_kmajor_desc(a_addr + k4 * 32), sw128_kmajor_desc(w_addr + k4 * 32), idesc, acc);
          }
          // the stage is free in both CTAs once both (PAIR: the pair's) MMAs committed
          if constexpr (PAIR) tc_commit_pair_multicast(&ctl->empty[s], 0x3);
          else tc_commit_multicast(&ctl->empty[s], 0x3);
        }
        if (!ok) break;
        if constexpr (PAIR) tc_commit_pair_multicast(&ctl->tfull[b], 0x3);
        else tc_commit(&ctl->tfull[b]);
      }
      if (!ok) {
        *abort_flag = 1;
        mbar_arrive(&ctl->tfull[0]);
        mbar_arrive(&ctl->tfull[1]);
      }
      // PAIR: both CTAs learn when every MMA (which writes both TMEMs and
      // reads both CTAs' shared memory) has completed
      if constexpr (PAIR) tc_commit_pair_multicast(&ctl->done, 0x3);
    }
    if (PAIR) {
      __syncwarp();
      mbar_wait(&ctl->done, 0, g.wait_ns);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();  // s_a is written, and Y may be written, only after the kernel this one depends on
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int et = threadIdx.x - 64;  // 0..127: token row of the CTA's tile
    int lt = 0;
    for (int t = cluster; t < tiles; t += clusters, ++lt) {
      const int tp = t % tp_count, wn = t / tp_count, b = lt & 1;
      const int m = tp * 2 * kPsTok + static_cast<int>(rank) * kPsTok + q * 32 + lane;
      const bool m_ok = m < g.M;
      // the tile's RW weight scales into the buffer's slot (the slot's
      // previous tile was drained before the barrier closing its iteration)
      for (int j = et; j < RW; j += 128) {
        const int n = wn * RW + j;
        ctl->sw_s[b][j] = n < g.N ? __ldg(g.s_w + n) : 0.0f;
      }
      const float sa = m_ok ? __ldg(g.s_a + m) : 0.0f;
      const bool w = mbar_wait(&ctl->tfull[b], static_cast<uint32_t>(lt / 2) & 1u, g.wait_ns);
      const bool bad = !__all_sync(0xffffffffu, w && !*abort_flag);
      if (lane == 0) ctl->epi_bad[q] = bad ? 1 : 0;
      named_bar_sync(1, 128);  // sw_s[b] and the four warps' verdicts are written
      if (ctl->epi_bad[0] | ctl->epi_bad[1] | ctl->epi_bad[2] | ctl->epi_bad[3]) {  // the same for every warp
        *abort_flag = 1;
        break;
      }
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < RW; c += 8) {
        uint32_t v[8];
        tmem_ld_x8(tmem + lane_base + static_cast<uint32_t>(b * RW + c), v);
        tmem_ld_wait();
        const int n0 = wn * RW + c;
        if (!m_ok || n0 >= g.N) continue;
        __nv_bfloat16* dst = g.Y + static_cast<int64_t>(m) * g.ldy + n0;
        if (n0 + 8 <= g.N && (reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
          uint32_t packed[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float y0 = (__uint_as_float(v[2 * j]) * sa) * ctl->sw_s[b][c + 2 * j];
            const float y1 = (__uint_as_float(v[2 * j + 1]) * sa) * ctl->sw_s[b][c + 2 * j + 1];
            __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
            packed[j] = *reinterpret_cast<uint32_t*>(&h);
          }
          *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
        } else {
          for (int j = 0; j < 8 && n0 + j < g.N; ++j)
            store_bf16(dst + j, (__uint_as_float(v[j]) * sa) * ctl->sw_s[b][c + j]);
        }
      }
      tc_fence_before();
      if constexpr (PAIR) {
        __syncwarp();  // the warp's TMEM reads of the buffer are done
        if (lane == 0) mbar_arrive_remote(tempty0 + 8u * static_cast<uint32_t>(b));
      } else {
        mbar_arrive(&ctl->tempty[b]);
      }
      named_bar_sync(1, 128);  // every thread is done with sw_s[b] and epi_bad before the next tile
    }
  }
  // ------------------------------------------- teardown: TMEM, then the pair
  tc_fence_before();
  __syncthreads();
  // PAIR: the leader's MMAs write both CTAs' TMEM, and the deallocation is
  // collective: both CTAs are past their last TMEM use (and the MMAs done)
  if (PAIR) cluster_sync();
  if (warp == 1) {
    tc_fence_after();
    if constexpr (PAIR) tmem_dealloc_pair(tmem, kTmemCols);
    else tmem_dealloc(tmem, kTmemCols);
  }
  // every copy this CTA issued into its peer, and the peer's into this CTA,
  // has been consumed (or the CTA gave up after a bounded wait) before
  // either CTA's shared memory is released
  cluster_sync();
  stamp_end(g.tstamp);
}

}  // namespace qg
