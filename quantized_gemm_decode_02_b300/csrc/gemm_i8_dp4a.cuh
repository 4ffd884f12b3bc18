// gemm_i8_dp4a.cuh -- W8A8_INT8 GEMM for the smallest token counts (M <= 8)
// on the CUDA cores: Swap-AB work split (one CTA per 128-row weight tile and
// K range), int8 dot products with dp4a into int32.
//
// "W8A8_INT8: INT8 per-token activation and per-channel weight scaling"
// ("Building a High-Performance and Portable vLLM Linear Backend with
// Helion", section "Helion Linear Backend > Scope") accumulates int8 x int8
// products in int32.  On sm_103a the tensor-core route has to widen every
// weight byte to fp16 first (no int8 MMA kind), and at M <= 8 that widening
// costs more issue slots than the whole product does on the CUDA cores:
// per 4 weight bytes and token one dp4a, against ~5 instructions of
// widening per 4 weight bytes before any MMA.  dp4a accumulates exactly in
// int32, so no segmenting is needed either.
//
// Per CTA (one 128-row weight tile x one K range):
//   warp 0      TMA: int8 W tile (128 x 128 B, 128-byte swizzle) and the
//               int8 activation tile (16 token rows, zero-filled past M)
//               into a `stages`-deep shared-memory ring;
//   warps 1..8  thread t: weight row t % 128, K half t / 128 of every
//               k-tile; per 16-byte chunk one weight load and, per token, one
//               broadcast activation load and four dp4a.  At the end the two
//               K halves of a row are added through shared memory and the
//               first half's threads run the epilogue (scales, bf16 store, or
//               the Split-K reduction shared with the tensor-core kernels).
#pragma once
#include "common.cuh"
#include "gemm_f8.cuh"

namespace qg {

constexpr int kDpWarps = 8;                    // compute warps (1..8)
constexpr int kDpThreads = 32 * (1 + kDpWarps);  // 288
constexpr int kDpMaxTokens = 8;
constexpr int kDpABox = 16;                    // activation rows per TMA box (rows >= M read as zero)

struct alignas(8) CtrlDp {
  uint64_t full[16];    // weight tile of the stage landed
  uint64_t full_a[16];  // activation tile of the stage landed
  uint64_t empty[16];
  uint64_t recv_bar;    // split-K: peers' partial rows have landed
  int last_flag;
  int abort_flag;
  float sa_s[kDpABox];
  float sw_s[kBN];
  int32_t half_s[kDpMaxTokens][kBN];  // second K half's sums, added by the first
};

struct DpShape {
  static constexpr uint32_t kWBytes = kBN * kBK;       // 16 KB int8 weights
  static constexpr uint32_t kABytes = kDpABox * kBK;   // 2 KB int8 activations
  static constexpr uint32_t kStageBytes = kWBytes + kABytes;
};

__host__ __device__ constexpr size_t gemm_dp4a_smem_bytes(int stages, int recv_bytes = 0) {
  return 1024 + static_cast<size_t>(stages) * DpShape::kStageBytes + recv_bytes + sizeof(CtrlDp);
}

// MT: tokens computed per CTA (1, 2, 4 or 8 >= M); rows M..MT-1 of the
// activation tile are zero, so their sums are zero and never stored.
template <int MT>
__global__ void __launch_bounds__(kDpThreads, 2)
    gemm_i8_dp4a_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA, GemmArgs g) {
  static_assert(MT == 1 || MT == 2 || MT == 4 || MT == 8, "MT");
  constexpr int MV = MT < 4 ? 4 : MT;  // accumulators padded to the 4-token groups of the cluster exchange
  stamp_start(g.tstamp);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stages = g.stages;
  uint8_t* recv = smem + static_cast<size_t>(stages) * DpShape::kStageBytes;  // split-K receive buffer
  CtrlDp* ctl = reinterpret_cast<CtrlDp*>(recv + g.recv_bytes);
  const bool clustered = g.reduce == kReduceCluster;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_tile = blockIdx.x, split = blockIdx.y;  // one token block (m_tiles == 1)
  const GroupView grp = group_view(g);
  const int m_base = grp.tok0;                 // tokens [m_base, m_base + Mb): at most 8
  const int Mb = min(MT, grp.tokens);
  if (Mb <= 0) return;  // an empty group (the whole cluster alike)
  const int w_row0 = static_cast<int>(blockIdx.z) * g.N;  // the group's weight rows
  const float* s_w = g.s_w + static_cast<int64_t>(blockIdx.z) * g.sw_group_stride;
  const int kb0 = static_cast<int>(static_cast<int64_t>(split) * g.kt_total / g.splits);
  const int kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * g.kt_total / g.splits);
  const int nk = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->full_a[i], 1);
      mbar_init(&ctl->empty[i], kDpWarps);
    }
    mbar_init(&ctl->recv_bar, 1);
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

  const int ct = threadIdx.x - 32;  // compute thread 0..255 (negative for the producer)
  const int row = ct & (kBN - 1), h = ct >> 7;
  int32_t acc[MV];
#pragma unroll
  for (int m = 0; m < MV; ++m) acc[m] = 0;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      const int w_row = w_row0 + n_tile * kBN;
      const int pre = nk < stages ? nk : stages;
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = smem + static_cast<size_t>(i) * DpShape::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full[i], DpShape::kWBytes);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[i], pol_w);
      }
      for (int i = pre; i < nk && i < pre + g.l2_prefetch; ++i) tma_prefetch_l2_2d(&tmW, (kb0 + i) * kBK, w_row);
      pdl_wait();  // the activations come from the kernel this one depends on
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = smem + static_cast<size_t>(i) * DpShape::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full_a[i], DpShape::kABytes);
        tma_load_2d(st + DpShape::kWBytes, &tmA, (kb0 + i) * kBK, m_base, &ctl->full_a[i], pol_a);
      }
      int issued = pre;
      for (int i = pre; i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
        if (!mbar_wait(&ctl->empty[s], ph ^ 1u, g.wait_ns) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(s) * DpShape::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full[s], DpShape::kWBytes);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[s], pol_w);
        if (g.l2_prefetch > 0 && i + g.l2_prefetch < nk) tma_prefetch_l2_2d(&tmW, (kb0 + i + g.l2_prefetch) * kBK, w_row);
        mbar_arrive_expect_tx(&ctl->full_a[s], DpShape::kABytes);
        tma_load_2d(st + DpShape::kWBytes, &tmA, (kb0 + i) * kBK, m_base, &ctl->full_a[s], pol_a);
        issued = i + 1;
      }
      // every issued copy lands before the CTA may exit
      for (int j = issued > stages ? issued - stages : 0; j < issued; ++j) {
        mbar_wait(&ctl->full[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
        mbar_wait(&ctl->full_a[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
      }
    }
  } else {
    // ------------------------------------------------------------- compute
    if (h == 0) {
      const int nn = n_tile * kBN + row;
      ctl->sw_s[row] = nn < g.N ? __ldg(s_w + nn) : 0.0f;
    }
    pdl_wait();  // s_a is written by the kernel this one depends on
    if (ct < kDpABox) ctl->sa_s[ct] = ct < Mb ? __ldg(g.s_a + m_base + ct) : 0.0f;
    for (int i = 0; i < nk; ++i) {
      const int s = i % stages;
      const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
      const bool w = mbar_wait(&ctl->full[s], ph, g.wait_ns) && mbar_wait(&ctl->full_a[s], ph, g.wait_ns);
      if (!__all_sync(0xffffffffu, w && !*abort_flag)) {
        *abort_flag = 1;
        break;
      }
      const uint8_t* wt = smem + static_cast<size_t>(s) * DpShape::kStageBytes;
      const uint8_t* at = wt + DpShape::kWBytes;
#pragma unroll(MT >= 8 ? 2 : 4)
      for (int c = 4 * h; c < 4 * h + 4; ++c) {
        const uint4 wv = *reinterpret_cast<const uint4*>(wt + sw128_chunk(row, c));
#pragma unroll
        for (int m = 0; m < MT; ++m) {
          // every lane of the warp reads the same 16 activation bytes
          const uint4 av = *reinterpret_cast<const uint4*>(at + sw128_chunk(m, c));
          int32_t a = acc[m];
          a = __dp4a(static_cast<int>(wv.x), static_cast<int>(av.x), a);
          a = __dp4a(static_cast<int>(wv.y), static_cast<int>(av.y), a);
          a = __dp4a(static_cast<int>(wv.z), static_cast<int>(av.z), a);
          a = __dp4a(static_cast<int>(wv.w), static_cast<int>(av.w), a);
          acc[m] = a;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->empty[s]);
    }
    // the second K half hands its sums to the first
    if (h == 1) {
#pragma unroll
      for (int m = 0; m < MT; ++m) ctl->half_s[m][row] = acc[m];
    }
    named_bar_sync(1, 32 * kDpWarps);
    if (h == 0) {
#pragma unroll
      for (int m = 0; m < MT; ++m) acc[m] += ctl->half_s[m][row];
    }
  }
  // ------------------------------------------------------------ epilogue
  __syncthreads();
  const bool abort = ctl->abort_flag != 0;  // stable after the barrier: uniform
  pdl_wait();  // outputs are written only after the kernel this one depends on
  const bool holds_acc = warp >= 1 && h == 0;  // warps 1..4: one full row each
  auto finish = [&](int m, int r, int nn, int32_t sum) {
    if (g.debug_acc) g.debug_acc[static_cast<int64_t>(m_base + m) * g.N + nn] = sum;
    const float y = (static_cast<float>(sum) * ctl->sa_s[m]) * ctl->sw_s[r];
    store_bf16(g.Y + static_cast<int64_t>(m_base + m) * g.ldy + nn, y);
  };
  const int n = n_tile * kBN + row;
  if (clustered) {
    if (holds_acc) {
      cluster_wait();  // every peer's receive barrier is initialized
      // rows go out even after an abort, so that every owner's wait completes
      cluster_push_row(acc, 0, row, split, g.splits, Mb, recv, &ctl->recv_bar);
      named_bar_sync(1, kBN);  // this CTA's own rows, stored locally, are visible
      const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(&ctl->recv_bar, 0, g.wait_ns));
      if (got && !abort) {
        cluster_sum_rows<int32_t>(recv, split, g.splits, Mb, ct, kBN, [&](int m, int r, int32_t sum) {
          const int nn = n_tile * kBN + r;
          if (nn < g.N) finish(m, r, nn, sum);
        });
      }
    } else {
      // the other warps pair their early arrive with a wait too (every peer
      // arrived right after its set-up, so this returns at once)
      cluster_wait();
    }
  } else if (holds_acc && !abort) {
    const bool n_ok = n < g.N;
    if (g.reduce == kReduceNone) {
      if (n_ok) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < Mb) finish(m, row, n, acc[m]);
      }
    } else {
      int32_t* part = static_cast<int32_t*>(g.ws_part);
      if (n_ok) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
          if (m < Mb) part[(static_cast<int64_t>(split) * g.M + m_base + m) * g.N + n] = acc[m];
      }
      __threadfence();
      named_bar_sync(1, kBN);
      const int tile_id = n_tile + blockIdx.z * gridDim.x;
      if (ct == 0) ctl->last_flag = (atomicAdd(g.ws_count + tile_id, 1) == g.splits - 1);
      named_bar_sync(1, kBN);
      if (ctl->last_flag) {
        __threadfence();
        if (n_ok) {
          for (int m = 0; m < Mb; ++m) {
            int32_t sum = 0;
            for (int s = 0; s < g.splits; ++s)
              sum += ld_cg_s32(part + (static_cast<int64_t>(s) * g.M + m_base + m) * g.N + n);
            finish(m, row, n, sum);
          }
        }
        if (ct == 0) g.ws_count[tile_id] = 0;
      }
    }
  }
  stamp_end(g.tstamp);
}

}  // namespace qg
