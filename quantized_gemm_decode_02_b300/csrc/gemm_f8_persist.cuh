// gemm_f8_persist.cuh -- persistent Standard-variant GEMM for FP8_Dynamic in
// the compute-bound regime (M of 64 and more tokens), with CTA pairs that
// share each weight tile.
//
// The Standard variant of "Building a High-Performance and Portable vLLM
// Linear Backend with Helion" (section "Kernel Implementation") puts the
// tokens on the MMA M side; the pages send token counts beyond their tuned
// range to other kernels ("Hybrid Dispatch"), here this library's own.
//
// Tiles: 128 tokens x 256 weight rows per CTA, D[128 x 256] fp32 in TMEM
// (tcgen05.mma.kind::f8f6f4, M = 128, N = 256, K = 32 per instruction).
// Pairs: the two CTAs of a thread-block cluster take the two 128-token
// halves of a 256-token pair tile and the same 256-row weight tile; CTA r
// loads weight rows [128 r, 128 r + 128) of the tile with TMA multicast into
// both CTAs' shared memory, so each weight k-tile crosses from L2 to the SMs
// once per pair (each CTA loads 16 KB of weights and 16 KB of activations per
// k-tile instead of 32 + 16).  A stage is refilled only when the MMAs of both
// CTAs are done with it (their commits arrive on both CTAs' empty barrier).
// Persistent: gridDim.x = 2 x clusters (at most one CTA per SM); cluster c
// takes pair tiles c, c + clusters, ..., token pair fastest, so the clusters
// running at the same time share weight tiles in L2.
// Double-buffered accumulator: two 256-column TMEM buffers; the MMA thread
// fills one tile's buffer while the epilogue warps drain the previous one.
//
// CTA = 6 warps: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer,
// warps 2..5 epilogue (thread = token row = TMEM lane).  Every wait is
// bounded; both CTAs of a pair end with a cluster barrier, so neither exits
// while its peer may still write into its shared memory.
#pragma once
#include "common.cuh"
#include "gemm_f8.cuh"

namespace qg {

constexpr int kPsTok = 128;                       // tokens per CTA (MMA M)
constexpr int kPsRows = 256;                      // weight rows per tile (MMA N)
constexpr uint32_t kPsABytes = kPsTok * kBK;      // 16 KB
constexpr uint32_t kPsWBytes = kPsRows * kBK;     // 32 KB (two multicast halves)
constexpr uint32_t kPsStageBytes = kPsABytes + kPsWBytes;
constexpr uint32_t kPsTmemCols = 2 * kPsRows;     // two accumulator buffers

struct alignas(8) CtrlPs {
  uint64_t full[8];     // the stage's activation tile and both weight halves landed
  uint64_t empty[8];    // both CTAs' MMAs are done with the stage
  uint64_t tfull[2];    // accumulator buffer written (MMA commit)
  uint64_t tempty[2];   // accumulator buffer drained (epilogue)
  uint64_t never;       // the forced-timeout test hook waits on it
  uint32_t tmem_base;
  int abort_flag;
  int epi_bad[4];          // per epilogue warp: its wait failed or the kernel aborted (this tile)
  float sw_s[2][kPsRows];  // per-channel scales of the buffer's weight tile
};

__host__ __device__ constexpr size_t gemm_f8_persist_smem_bytes(int stages) {
  return 1024 + static_cast<size_t>(stages) * kPsStageBytes + sizeof(CtrlPs);
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

__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// One CTA of a pair.  g.m_tiles = pair tiles along the tokens (ceil(M/256)),
// g.kt_total = k-tiles; tiles = g.m_tiles * ceil(N/256).
__global__ void __launch_bounds__(kThreads, 1)
    gemm_f8_persist_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA, GemmArgs g) {
  stamp_start(g.tstamp);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stages = g.stages;
  CtrlPs* ctl = reinterpret_cast<CtrlPs*>(smem + static_cast<size_t>(stages) * kPsStageBytes);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();           // 0 or 1: token half of the pair tile
  const int cluster = static_cast<int>(blockIdx.x >> 1), clusters = static_cast<int>(gridDim.x >> 1);
  const int tp_count = g.m_tiles, wn_count = (g.N + kPsRows - 1) / kPsRows;
  const int tiles = tp_count * wn_count;
  const int nk = g.kt_total;

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], 2);  // one commit from each CTA of the pair
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&ctl->tfull[b], 1);
      mbar_init(&ctl->tempty[b], 128);
    }
    mbar_init(&ctl->never, 1);
    ctl->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmA);
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, kPsTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_sync();  // the peer's barriers are initialized before any multicast reaches them
  const uint32_t tmem = ctl->tmem_base;
  pdl_launch_dependents();
  volatile int* abort_flag = &ctl->abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      const uint16_t both = 0x3;
      // the weights of the first tile's first stages are requested before
      // the wait for the kernel this one depends on, its activations after
      const int first = cluster < tiles ? cluster : -1;
      const int pre = first >= 0 ? (nk < stages ? nk : stages) : 0;
      if (pre > 0) {
        const int w_row = (first / tp_count) * kPsRows + static_cast<int>(rank) * kPsTok;
        for (int kk = 0; kk < pre; ++kk) {
          uint8_t* st = smem + static_cast<size_t>(kk) * kPsStageBytes;
          mbar_arrive_expect_tx(&ctl->full[kk], kPsStageBytes);
          tma_load_2d_multicast(st + kPsABytes + rank * (kPsWBytes / 2), &tmW, kk * kBK, w_row, &ctl->full[kk], both,
                                pol_w);
        }
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
        if (t2 < tiles) tma_prefetch_l2_2d(&tmW, k2 * kBK, (t2 / tp_count) * kPsRows + static_cast<int>(rank) * kPsTok);
      };
      if (ahead > 0 && first >= 0)
        for (int kk = pre; kk < pre + ahead; ++kk) prefetch_ahead(first, kk - ahead);
      pdl_wait();
      int i = 0;  // k-tile counter over all of this CTA's tiles (the ring position)
      bool ok = true;
      for (int t = cluster; ok && t < tiles; t += clusters) {
        const int tp = t % tp_count, wn = t / tp_count;
        const int a_row = tp * 2 * kPsTok + static_cast<int>(rank) * kPsTok;
        const int w_row = wn * kPsRows + static_cast<int>(rank) * kPsTok;
        for (int kk = 0; kk < nk; ++kk, ++i) {
          const int s = i % stages;
          uint8_t* st = smem + static_cast<size_t>(s) * kPsStageBytes;
          if (ahead > 0 && i >= pre) prefetch_ahead(t, kk);
          if (i >= pre) {
            if (i >= stages && (!mbar_wait(&ctl->empty[s], (static_cast<uint32_t>(i / stages) & 1u) ^ 1u, g.wait_ns) ||
                                *abort_flag)) {
              ok = false;
              break;
            }
            mbar_arrive_expect_tx(&ctl->full[s], kPsStageBytes);
            tma_load_2d_multicast(st + kPsABytes + rank * (kPsWBytes / 2), &tmW, kk * kBK, w_row, &ctl->full[s], both,
                                  pol_w);
          }
          tma_load_2d(st, &tmA, kk * kBK, a_row, &ctl->full[s], pol_a);
        }
      }
      if (!ok) *abort_flag = 1;
      // every stage this CTA expects lands (its own copies and the peer's
      // half) before the CTA may leave
      for (int j = i > stages ? i - stages : 0; j < i; ++j)
        mbar_wait(&ctl->full[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(kPsTok, kPsRows, 0, 0);  // E4M3 x E4M3 -> F32, 128 x 256
      bool ok = !g.force_timeout || mbar_wait(&ctl->never, 0, g.wait_ns);
      int i = 0, lt = 0;
      for (int t = cluster; ok && t < tiles; t += clusters, ++lt) {
        const int b = lt & 1;
        if (lt >= 2 && !mbar_wait(&ctl->tempty[b], (static_cast<uint32_t>(lt / 2) & 1u) ^ 1u, g.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + static_cast<uint32_t>(b * kPsRows);
        for (int kk = 0; kk < nk; ++kk, ++i) {
          const int s = i % stages;
          if (!mbar_wait(&ctl->full[s], static_cast<uint32_t>(i / stages) & 1u, g.wait_ns) || *abort_flag) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(smem + static_cast<size_t>(s) * kPsStageBytes);
          const uint32_t w_addr = a_addr + kPsABytes;
#pragma unroll
          for (int k4 = 0; k4 < kBK / 32; ++k4)
            mma_f8f6f4(d, sw128_kmajor_desc(a_addr + k4 * 32), sw128_kmajor_desc(w_addr + k4 * 32), idesc,
                       (kk > 0 || k4 > 0) ? 1u : 0u);
          tc_commit_multicast(&ctl->empty[s], 0x3);  // the stage is free in both CTAs once both committed
        }
        if (!ok) break;
        tc_commit(&ctl->tfull[b]);
      }
      if (!ok) {
        *abort_flag = 1;
        mbar_arrive(&ctl->tfull[0]);
        mbar_arrive(&ctl->tfull[1]);
      }
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
      // the tile's 256 weight scales into the buffer's slot (the slot's
      // previous tile was drained before the barrier closing its iteration)
      for (int j = et; j < kPsRows; j += 128) {
        const int n = wn * kPsRows + j;
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
      for (int c = 0; c < kPsRows; c += 8) {
        uint32_t v[8];
        tmem_ld_x8(tmem + lane_base + static_cast<uint32_t>(b * kPsRows + c), v);
        tmem_ld_wait();
        const int n0 = wn * kPsRows + c;
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
      mbar_arrive(&ctl->tempty[b]);
      named_bar_sync(1, 128);  // every thread is done with sw_s[b] and epi_bad before the next tile
    }
  }
  // ------------------------------------------- teardown: TMEM, then the pair
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kPsTmemCols);
  }
  // every copy this CTA issued into its peer, and the peer's into this CTA,
  // has been consumed (or the CTA gave up after a bounded wait) before
  // either CTA's shared memory is released
  cluster_sync();
  stamp_end(g.tstamp);
}

}  // namespace qg
