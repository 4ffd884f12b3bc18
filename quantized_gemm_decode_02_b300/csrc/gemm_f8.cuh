// gemm_f8.cuh -- tcgen05 (kind::f8f6f4) GEMM for the E4M3 formats
// FP8_Dynamic and Block_FP8:  Y[M,N] = bf16(dequant(A_q[M,K] . W_q[N,K]^T)).
//
// The three algorithm variants of "Building a High-Performance and Portable
// vLLM Linear Backend with Helion", section "Kernel Implementation":
//   Standard  D = A_q . W_q^T with tokens on the MMA M side (128 rows);
//   Swap-AB   D^T = W_q . A_q^T, so 128 weight rows take the MMA M side and
//             the few tokens (padded to MPAD) the MMA N side;
//   Split-K   K is cut into `splits` balanced ranges of whole 128-wide
//             k-tiles, one CTA per (tile, range), and the partial tiles are
//             summed in the fixed order 0..splits-1 (deterministic).  For
//             Swap-AB with at most 16 ranges the CTAs of one tile form a
//             thread-block cluster and add their partials through distributed
//             shared memory (no workspace); otherwise partials go to a caller
//             workspace and the last CTA to arrive on a tile sums them.
//
// CTA = 6 warps: warp 0 issues TMA loads into a `stages`-deep shared-memory
// ring (W tile 128x128 bytes + activation tile), warp 1 owns TMEM and issues
// the MMAs from one thread, warps 2..5 (128 threads, one per TMEM lane) run
// the epilogue.  Every mbarrier wait is bounded (see mbar_wait).  The Swap-AB
// kernel is sized so that two CTAs fit on one SM: while one drains its
// epilogue the other (or the next kernel's CTA, under programmatic dependent
// launch) keeps the weight stream going.
//
// Block_FP8 (1x128 activation groups, 128x128 weight blocks): each 128-wide
// k-tile is one scale group, so the MMA writes each k-tile's partial into its
// own TMEM buffer (NBUF-deep ring) and the epilogue warps promote it,
// acc += s_a[m,kb] * s_w[n/128,kb] * partial, while later MMAs run.
//
// Grid: x = weight tile * token blocks (the token blocks of one weight tile
// adjacent, so they share its loads in L2), y = K range, z = group of a
// grouped (mixture-of-experts) launch.  The Standard kernel also takes
// 256-row weight tiles (FP8_Dynamic, MMA N = 256).
#pragma once
#include "common.cuh"
#include "quant.cuh"

namespace qg {

enum : int { kReduceNone = 0, kReduceCluster = 1, kReduceGlobal = 2 };
constexpr int kMaxClusterSplits = 16;

struct GemmArgs {
  int M, N, K;
  int64_t ldy;          // Y row stride (elements)
  int kt_total;         // ceil(K / 128)
  int splits;           // >= 1
  int m_tiles;          // token blocks (Swap-AB) or 128-token tiles (Standard); blockIdx.x = n_tile * m_tiles + m
  // grouped launches (qg_gemm_w8a8_grouped): blockIdx.z is the group; its
  // tokens are rows [group_offsets[z], group_offsets[z+1]) of A_q / s_a / Y
  // (M counts all groups' tokens), its weights rows [z*N, z*N + N) of W_q,
  // its weight scales s_w + z*sw_group_stride.  Null: one group, M tokens.
  const int* group_offsets;
  int64_t sw_group_stride;
  int group_max;        // tokens of a group taken into account (the launch's max_tokens)
  int stages;           // shared-memory ring depth
  int l2_prefetch;      // L2 prefetch distance: weight k-tiles requested ahead of the ring's loads
  int reduce;           // kReduceNone / kReduceCluster / kReduceGlobal
  int recv_bytes;       // kReduceCluster: bytes of the shared-memory receive buffer (cluster_recv_bytes)
  const float* s_a;     // [M] or [M][kt_total]
  const float* s_w;     // [N] or [ceil(N/128)][kt_total]
  __nv_bfloat16* Y;     // [M][ldy]
  void* ws_part;        // kReduceGlobal: [splits][M][N] fp32 (or int32) partials
  int* ws_count;        // kReduceGlobal: one arrival counter per output tile, zero between launches
  int32_t* debug_acc;   // [M][N] int32 accumulators (W8A8_INT8 only) or null
  // fused activation quantization (qg_linear_w8a8): the kernel reads bf16
  // activations and quantizes them itself; A_q / s_a are optional copies
  const __nv_bfloat16* A;  // [M][lda] bf16
  int64_t lda;
  uint8_t* a_q_out;        // [M][K] codes, or null
  float* s_a_out;          // per-token scales, or null
  uint64_t wait_ns;     // bound of every pipeline wait
  int force_timeout;    // test hook: the MMA thread first waits on a barrier nothing arrives on
  unsigned long long* tstamp;  // launch timing slot pair (stamp_start / stamp_end), or null
};

constexpr int kBN = 128;         // weight rows per tile (and Block_FP8 block size)
constexpr int kBK = 128;         // bytes of K per k-tile (one 128-byte swizzle row)
constexpr int kThreads = 192;
// Block_FP8 with fused quantization adds four quantizer warps (6..9)
constexpr int kThreadsBlockFused = 320;
// Block_FP8 fused: ring of per-k-tile activation scales passed from the
// quantizer warps to the promotion warps (slots >= stages + 4 TMEM buffers)
constexpr int kSaRing = 16;
constexpr int kMaxStagesBlockFused = kSaRing - 4;
// pw: promotion / epilogue warps of the two-kernel form (4, or 8 for the
// Block_FP8 form with two warps per TMEM lane quarter)
__host__ __device__ constexpr int swap_threads(int fmt, bool fused, int pw = 4) {
  return (fmt == 2 && fused) ? kThreadsBlockFused : 64 + 32 * pw;
}
// Standard kernel: Block_FP8 promotes with eight epilogue warps
__host__ __device__ constexpr int std_threads(int fmt) { return fmt == 2 ? 320 : kThreads; }
constexpr uint64_t kDrainNs = 200000000ull;  // bound for draining in-flight copies on exit

__host__ __device__ constexpr uint32_t pow2_cols(uint32_t c) {
  return c <= 32 ? 32 : c <= 64 ? 64 : c <= 128 ? 128 : c <= 256 ? 256 : 512;
}

// Shared-memory control block that follows the ring.
struct alignas(16) Ctrl {
  uint64_t full[16];
  uint64_t empty[16];
  uint64_t acc_full;
  uint64_t tfull[8];
  uint64_t tempty[8];
  uint64_t never;
  uint64_t recv_bar;  // split-K: peers' partial rows have landed
  uint64_t amax_bar;  // fused quantization: peers' partial row maxima have landed
  uint64_t full_a[16];  // fused quantization: the stage's activation tile is written
  uint64_t sfull[kSaRing];  // Block_FP8 fused: the k-tile's activation scales are in amax_s (ring slot)
  uint32_t tmem_base;
  int last_flag;
  int abort_flag;
  float sa_s[64];   // per-token scales, staged for the epilogue
  float sw_s[128];  // per-channel scales of the tile's rows
  alignas(16) float amax_s[kMaxClusterSplits * 64];  // fused quantization: [source rank][token] partial row maxima
                                         // (Block_FP8 fused: [ring slot][token] activation scales;
                                         // Block_FP8 two-kernel form: [k-tile][token] scale products)
};

template <bool SWAP, int MPAD>
struct TileShape {
  static constexpr uint32_t kActRows = SWAP ? MPAD : 128;            // activation rows per tile
  static constexpr uint32_t kWBytes = kBN * kBK;                      // 16 KB
  static constexpr uint32_t kABytes = kActRows * kBK;
  static constexpr uint32_t kStageBytes = kWBytes + kABytes;          // multiple of 1024
  static constexpr uint32_t kMmaM = 128;
  static constexpr uint32_t kMmaN = SWAP ? MPAD : kBN;
};

template <bool SWAP, int MPAD>
__host__ __device__ constexpr size_t gemm_f8_smem_bytes(int stages, int recv_bytes = 0) {
  return 1024 + static_cast<size_t>(stages) * TileShape<SWAP, MPAD>::kStageBytes + recv_bytes + sizeof(Ctrl);
}
// Standard variant stage: BNW weight rows (128, or 256 for the wide tiles
// of FP8_Dynamic) and 128 token rows of one 128-byte k-tile.
template <int BNW>
struct StdShape {
  static constexpr uint32_t kWBytes = BNW * kBK;
  static constexpr uint32_t kABytes = 128 * kBK;
  static constexpr uint32_t kStageBytes = kWBytes + kABytes;  // multiple of 1024
};
template <int BNW>
__host__ __device__ constexpr size_t gemm_f8_std_smem_bytes(int stages) {
  return 1024 + static_cast<size_t>(stages) * StdShape<BNW>::kStageBytes + sizeof(Ctrl);
}

__device__ __forceinline__ void store_bf16(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

// This CTA's group (see GemmArgs::group_offsets): first token and token
// count.  The offsets are inputs, so a grouped launch waits for the kernel it
// depends on before reading them.
struct GroupView {
  int tok0, tokens;
};
__device__ __forceinline__ GroupView group_view(const GemmArgs& g) {
  if (g.group_offsets == nullptr) return GroupView{0, g.M};
  pdl_wait();
  // offsets outside [0, M] or decreasing are clamped (no row outside A_q /
  // Y), and a group's tokens beyond group_max are left out (the token blocks
  // and receive buffers are sized for group_max)
  const int t0 = min(max(g.group_offsets[blockIdx.z], 0), g.M);
  const int t1 = min(max(g.group_offsets[blockIdx.z + 1], t0), g.M);
  return GroupView{t0, min(t1 - t0, g.group_max)};
}

__device__ __forceinline__ uint8_t* align1024(uint8_t* p) {
  return reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// Split-K through distributed shared memory, push form.  The S CTAs of a
// tile form one cluster (cluster rank == split index).  Row r of the tile is
// owned by CTA r / R, R = ceil(128 / S).  Every CTA sends its partial of
// each row to the row's owner with st.async, which lands in the owner's
// receive buffer recv[s][j][..] (s = sending rank, j = row - owner*R; a row
// holds mv = M rounded up to 4 values, padded to an odd number of 16-byte
// chunks so that reads of consecutive rows hit different banks) and
// completes bytes on the owner's mbarrier; the owner waits for
// (S - 1) * rows * mv * 4 bytes, then adds the S partials of each of its
// elements in the fixed order 0..S-1.  One one-way transfer and one bounded
// wait; no CTA reads a peer, so none waits for its peers to finish.
__host__ __device__ constexpr int cluster_rows_per_rank(int S) { return (kBN + S - 1) / S; }
__host__ __device__ constexpr int cluster_mv(int M) { return (M + 3) & ~3; }
__host__ __device__ constexpr int cluster_row_stride(int M) { return 4 * ((cluster_mv(M) / 4) | 1); }
__host__ __device__ constexpr int cluster_recv_bytes(int S, int M) {
  return S * cluster_rows_per_rank(S) * cluster_row_stride(M) * 4;
}
__device__ __forceinline__ int cluster_rows_of(int rank, int S) {
  const int R = cluster_rows_per_rank(S);
  return max(0, min(kBN, rank * R + R) - rank * R);
}

// Send this thread's values v[0..N) of row `row` for tokens [m0, m0 + N)
// (m0 and N multiples of 4) to the row's owner; values for the thread's own
// rows are stored locally.
template <typename T, int N>
__device__ __forceinline__ void cluster_push_row(const T (&v)[N], int m0, int row, int rank, int S, int M,
                                                 uint8_t* recv, uint64_t* recv_bar) {
  const int R = cluster_rows_per_rank(S), mv = cluster_mv(M), rs = cluster_row_stride(M);
  const int o = row / R, j = row - o * R;
  const uint32_t base = smem_u32(recv), bar = smem_u32(recv_bar);
#pragma unroll
  for (int c = 0; c < N; c += 4) {
    const int m = m0 + c;
    if (m < mv) {
      const uint32_t off = static_cast<uint32_t>(((rank * R + j) * rs + m) * 4);
      const uint32_t w0 = reinterpret_cast<const uint32_t&>(v[c]);
      const uint32_t w1 = reinterpret_cast<const uint32_t&>(v[c + 1]);
      const uint32_t w2 = reinterpret_cast<const uint32_t&>(v[c + 2]);
      const uint32_t w3 = reinterpret_cast<const uint32_t&>(v[c + 3]);
      if (o == rank)
        *reinterpret_cast<uint4*>(recv + off) = make_uint4(w0, w1, w2, w3);
      else
        st_async_v4(dsmem_map(base + off, static_cast<uint32_t>(o)), w0, w1, w2, w3,
                    dsmem_map(bar, static_cast<uint32_t>(o)));
    }
  }
}

// Owner side, after the receive barrier completed: for each of this CTA's
// rows j and each group of 4 tokens, sum the S partials in order and call
// store(m, row, sum) for the tokens m < M.  Consecutive threads take
// consecutive rows, so each store instruction of a warp writes one
// contiguous run of a Y row.
template <typename T, typename Store>
__device__ __forceinline__ void cluster_sum_rows(const uint8_t* recv, int rank, int S, int M, int tid, int nthreads,
                                                 Store&& store) {
  const int R = cluster_rows_per_rank(S), rs = cluster_row_stride(M), rn = cluster_rows_of(rank, S);
  const int quads = cluster_mv(M) / 4;
  for (int e = tid; e < rn * quads; e += nthreads) {
    const int j = e % rn, m0 = 4 * (e / rn);
    const uint4 v0 = *reinterpret_cast<const uint4*>(recv + static_cast<size_t>((j * rs + m0) * 4));
    T sum[4] = {reinterpret_cast<const T&>(v0.x), reinterpret_cast<const T&>(v0.y), reinterpret_cast<const T&>(v0.z),
                reinterpret_cast<const T&>(v0.w)};
    for (int s = 1; s < S; ++s) {  // the receive buffer is this CTA's own shared memory
      const uint4 v = *reinterpret_cast<const uint4*>(recv + static_cast<size_t>(((s * R + j) * rs + m0) * 4));
      sum[0] += reinterpret_cast<const T&>(v.x);
      sum[1] += reinterpret_cast<const T&>(v.y);
      sum[2] += reinterpret_cast<const T&>(v.z);
      sum[3] += reinterpret_cast<const T&>(v.w);
    }
#pragma unroll
    for (int c = 0; c < 4; ++c)
      if (m0 + c < M) store(m0 + c, rank * R + j, sum[c]);
  }
}

// Fused activation quantization, part 1: the scale of every token of this
// CTA's block (the per-token formats, "Scope": one scale per token over the
// whole row).  `nthr` threads (index t, a multiple of 32) take the maximum
// |A| of each token over this CTA's K range [k0, k1); with Split-K in a
// cluster each CTA pushes its partial maxima to every peer (st.async into
// amax_s[src][token]) and waits for theirs, so every CTA holds the row
// maximum over all of K; then s = amax / qmax (IEEE, 1 for an all-zero row)
// goes to sa_s.  With Split-K through the workspace, [k0, k1) must be the
// whole row.  Ends with a barrier among the nthr threads.
__device__ __forceinline__ void fused_token_scales(const GemmArgs& g, int m_base, int Mb, int k0, int k1,
                                                   bool clustered, int rank, float qmax, float* amax_s, float* sa_s,
                                                   uint64_t* amax_bar, int t, int nthr, int bar_id,
                                                   bool write_scales) {
  const int warps = nthr / 32, w = t >> 5, lane = t & 31;
  for (int m = w; m < Mb; m += warps) {
    const __nv_bfloat16* row = g.A + static_cast<int64_t>(m_base + m) * g.lda;
    float mx = 0.0f;
    for (int k = k0 + lane * 8; k < k1; k += 256) {
      float v[8];
      load8(row + k, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) mx = fmaxf(mx, fabsf(v[i]));
    }
    mx = warp_max(mx);
    if (lane == 0) amax_s[rank * 64 + m] = mx;
  }
  named_bar_sync(bar_id, nthr);
  if (clustered) {
    cluster_wait();  // every peer's barriers are initialized
    if (t < Mb) {
      const uint32_t addr = smem_u32(&amax_s[rank * 64 + t]), bar = smem_u32(amax_bar);
      const uint32_t v = __float_as_uint(amax_s[rank * 64 + t]);
      for (int o = 0; o < g.splits; ++o)
        if (o != rank) st_async_b32(dsmem_map(addr, static_cast<uint32_t>(o)), v, dsmem_map(bar, static_cast<uint32_t>(o)));
    }
    mbar_wait_cluster(amax_bar, 0, g.wait_ns);
  }
  if (t < 64) {
    float mx = 0.0f;
    if (t < Mb) {
      if (clustered) {
        for (int o = 0; o < g.splits; ++o) mx = fmaxf(mx, amax_s[o * 64 + t]);
      } else {
        mx = amax_s[rank * 64 + t];
      }
    }
    sa_s[t] = t < Mb ? scale_from_amax(mx, qmax) : 0.0f;
    if (write_scales && t < Mb && g.s_a_out) g.s_a_out[m_base + t] = sa_s[t];
  }
  named_bar_sync(bar_id, nthr);
}

// Fused activation quantization, part 2: 32 consecutive activations of token
// row `row` starting at column k (zeros past K) as fp32.
// Raw bf16 activations A[row][k .. k+32) as four 16-byte words (zero past K;
// K % 16 == 0, so a word is either wholly inside the row or wholly past it).
__device__ __forceinline__ void load_act_raw(const GemmArgs& g, int row, int k, uint4 (&v)[4]) {
  const __nv_bfloat16* p = g.A + static_cast<int64_t>(row) * g.lda + k;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    v[c] = k + 8 * c < g.K ? *reinterpret_cast<const uint4*>(p + 8 * c) : make_uint4(0u, 0u, 0u, 0u);
}
__device__ __forceinline__ void unpack_act32(const uint4 (&v)[4], float (&x)[32]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint32_t w[4] = {v[c].x, v[c].y, v[c].z, v[c].w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
      x[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
}
__device__ __forceinline__ void load_act32(const GemmArgs& g, int row, int k, float (&x)[32]) {
  const __nv_bfloat16* p = g.A + static_cast<int64_t>(row) * g.lda + k;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    float v[8];
    if (k + 8 * c < g.K) {
      load8(p + 8 * c, v);
    } else {
#pragma unroll
      for (int i = 0; i < 8; ++i) v[i] = 0.0f;
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) x[8 * c + i] = v[i];
  }
}

// Block_FP8 fused quantization, run by warps 6..9 (qt = 0..127).  For each
// k-tile of the CTA's K range: the bf16 activations of the block's tokens,
// in pieces of 32 values (token row r, quarter p of the 128-wide group),
// are loaded one k-tile ahead; the four threads of a row agree on the
// group's maximum (two shuffles) and take s = amax / 448 ("Scope": one
// scale per 1x128 activation group); the codes (the correctly rounded
// quotient, round-to-nearest-even, saturated) go into the stage's
// activation tile once the MMAs of the stage's previous use are done, and
// the scales into the k-tile's ring slot for the promotion warps.  The CTAs
// of the first weight tile also write A_q / s_a when the caller gave them.
template <int MPAD>
__device__ __forceinline__ void block_fused_quantize(const GemmArgs& g, Ctrl* ctl, uint8_t* smem, uint32_t stage_bytes,
                                                     uint32_t w_bytes, int stages, int nk, int kb0, int m_base, int Mb,
                                                     int n_tile, volatile int* abort_flag) {
  pdl_wait();  // the activations are written by the kernel this one depends on
  const int qt = static_cast<int>(threadIdx.x) - 192, lane = threadIdx.x & 31;
  constexpr int kPP = (MPAD * 4 + 127) / 128;  // pieces per thread
  const bool write_out = g.a_q_out != nullptr && n_tile == 0;
  uint4 cur[kPP][4], nxt[kPP][4];
  auto fetch = [&](int i, uint4(&buf)[kPP][4]) {
#pragma unroll
    for (int q = 0; q < kPP; ++q) {
      const int piece = qt + 128 * q, r = piece >> 2, p = piece & 3;
      if (piece < MPAD * 4 && r < Mb)
        load_act_raw(g, m_base + r, (kb0 + i) * kBK + 32 * p, buf[q]);
      else
#pragma unroll
        for (int c = 0; c < 4; ++c) buf[q][c] = make_uint4(0u, 0u, 0u, 0u);
    }
  };
  fetch(0, cur);
  bool ok = true;
  for (int i = 0; i < nk; ++i) {
    const int s = i % stages, slot = i % kSaRing;
    if (i + 1 < nk) fetch(i + 1, nxt);
    if (i >= stages &&
        !__all_sync(0xffffffffu, mbar_wait(&ctl->empty[s], static_cast<uint32_t>(i / stages - 1) & 1u, g.wait_ns) &&
                                     !*abort_flag)) {
      ok = false;
      break;
    }
    const int kb = kb0 + i, kt0 = kb * kBK;
    uint8_t* at = smem + static_cast<size_t>(s) * stage_bytes + w_bytes;
#pragma unroll
    for (int q = 0; q < kPP; ++q) {
      const int piece = qt + 128 * q, r = piece >> 2, p = piece & 3;
      float x[32];
      unpack_act32(cur[q], x);
      float mx = 0.0f;
#pragma unroll
      for (int j = 0; j < 32; ++j) mx = fmaxf(mx, fabsf(x[j]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));  // the row's four quarters
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float sc = scale_from_amax(mx, 448.0f);
      if (piece < MPAD * 4) {
        float qv[32];
        Divider(sc).divide(x, qv);
        uint32_t w[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          w[j] = static_cast<uint32_t>(e4m3x2(qv[4 * j], qv[4 * j + 1])) |
                 (static_cast<uint32_t>(e4m3x2(qv[4 * j + 2], qv[4 * j + 3])) << 16);
        *reinterpret_cast<uint4*>(at + sw128_chunk(r, 2 * p)) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(at + sw128_chunk(r, 2 * p + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
        if (p == 0) ctl->amax_s[slot * 64 + r] = r < Mb ? sc : 0.0f;
        if (write_out && r < Mb) {
          uint8_t* dst = g.a_q_out + static_cast<int64_t>(m_base + r) * g.K + kt0 + 32 * p;
          *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
          *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
          if (p == 0 && g.s_a_out) g.s_a_out[static_cast<int64_t>(m_base + r) * g.kt_total + kb] = sc;
        }
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // the tile is read by the MMA (async proxy)
    __syncwarp();  // every lane's codes and scales are written
    if (lane == 0) {
      mbar_arrive(&ctl->full_a[s]);
      mbar_arrive(&ctl->sfull[slot]);
    }
#pragma unroll
    for (int q = 0; q < kPP; ++q)
#pragma unroll
      for (int c = 0; c < 4; ++c) cur[q][c] = nxt[q][c];
  }
  if (!ok) *abort_flag = 1;
}

// ------------------------------------------------------------ Swap-AB --
// One CTA per (128-row weight tile, K range, block of MPAD tokens).
// D^T[128 x MPAD] in TMEM.
// FUSED (qg_linear_w8a8's one-kernel form): the kernel reads bf16
// activations (g.A) and quantizes them itself; tmA is unused.
//   FP8_Dynamic: the epilogue warps, idle during the main loop, take the
//     per-token row maximum (agreed across a Split-K cluster) and write
//     each stage's activation tile.
//   Block_FP8: four more warps (6..9) quantize each k-tile's 1x128 groups
//     on their own -- a group's scale needs only its 128 values, so no CTA
//     waits for another -- write the stage's activation tile, and pass the
//     k-tile's scales to the promotion warps through a ring in shared
//     memory (amax_s, barriers sfull).
// PW (Block_FP8, two-kernel form): 4 promotion warps (2..5), or 8 (2..9):
// two per TMEM lane quarter, warp w taking the token half (w - 2) / 4 of
// every k-tile's partial, so each promotes half as many products per k-tile.
template <int FMT, int MPAD, bool FUSED, int PW = 4>
__global__ void __launch_bounds__(swap_threads(FMT, FUSED, PW),
                                  (FMT == kFmtBlock && FUSED && MPAD > 32) ? 1 : 2)  // (64-token blocks: registers)
    gemm_f8_swap_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA, GemmArgs g) {
  using TS = TileShape<true, MPAD>;
  constexpr bool BLOCK = (FMT == kFmtBlock);
  constexpr bool QWARPS = BLOCK && FUSED;                // quantizer warps 6..9
  constexpr int kT = swap_threads(FMT, FUSED, PW);
  constexpr int kEpi = 32 * PW;                          // promotion / epilogue threads
  constexpr int kTP = MPAD * 4 / PW;                     // tokens of each such thread
  static_assert(PW == 4 || (PW == 8 && BLOCK && !FUSED), "eight promotion warps: Block_FP8, two-kernel form");
  static_assert(kTP % 8 == 0, "token parts of whole 8-column TMEM loads");
  // Block_FP8: as many k-tile partial buffers as the 256 TMEM columns of one
  // of two CTAs per SM hold, up to 8 (the fused form keeps 4: its scale ring
  // holds stages + 4 k-tiles)
  constexpr int NBUF = BLOCK ? ((FUSED || MPAD > 32) ? 4 : 256 / MPAD > 8 ? 8 : 256 / MPAD) : 1;
  constexpr uint32_t kTmemCols = pow2_cols(NBUF * MPAD);
  static_assert(kTmemCols <= 256, "two CTAs per SM share the 512 TMEM columns");

  stamp_start(g.tstamp);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stages = g.stages;
  uint8_t* recv = smem + static_cast<size_t>(stages) * TS::kStageBytes;  // split-K receive buffer
  Ctrl* ctl = reinterpret_cast<Ctrl*>(recv + g.recv_bytes);
  const bool clustered = g.reduce == kReduceCluster;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the token blocks of one weight tile are adjacent block indices, so they
  // run together and all but the first find the tile's weights in L2
  const int n_tile = static_cast<int>(blockIdx.x / g.m_tiles);
  const int split = blockIdx.y;
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

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], 1);
    }
    mbar_init(&ctl->acc_full, 1);
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&ctl->tfull[b], 1);
      mbar_init(&ctl->tempty[b], kEpi / 32);  // one arrive per promotion warp
    }
    mbar_init(&ctl->never, 1);
    mbar_init(&ctl->recv_bar, 1);
    mbar_init(&ctl->amax_bar, 1);
    if (FUSED)
      for (int i = 0; i < stages; ++i) mbar_init(&ctl->full_a[i], 4);
    if (QWARPS)
      for (int j = 0; j < kSaRing; ++j) mbar_init(&ctl->sfull[j], 4);  // one arrive per quantizer warp
    ctl->last_flag = 0;
    ctl->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmW);
    if (!FUSED) prefetch_tmap(&tmA);
  }
  __syncthreads();
  if (clustered) {
    // the receive barriers expect the peers' rows (and, fused, their row
    // maxima); every thread then marks this CTA's barriers initialized for
    // the cluster (waited on before the first push)
    if (threadIdx.x == 0) {
      mbar_arrive_expect_tx(&ctl->recv_bar, static_cast<uint32_t>((g.splits - 1) * cluster_rows_of(split, g.splits) *
                                                                  cluster_mv(Mb) * 4));
      if (FUSED && !BLOCK) mbar_arrive_expect_tx(&ctl->amax_bar, static_cast<uint32_t>((g.splits - 1) * Mb * 4));
    }
    cluster_arrive_relaxed();
  }
  pdl_launch_dependents();
  volatile int* abort_flag = &ctl->abort_flag;
  float acc[kTP];  // epilogue threads: weight row n of the tile x tokens [t0, t0 + kTP)
#pragma unroll
  for (int m = 0; m < kTP; ++m) acc[m] = 0.0f;
  const int t0 = warp >= 2 ? ((warp - 2) >> 2) * kTP : 0;  // first token of this thread's part

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // Starts at once (it needs no TMEM): the weights are static, so their
    // first `pre` tiles are fetched before waiting on the kernel that
    // produced the activations.
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      const int w_row = w_row0 + n_tile * kBN;
      const int pre = nk < stages ? nk : stages;
      constexpr uint32_t kTx = FUSED ? TS::kWBytes : TS::kStageBytes;  // fused: threads write the activations
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = smem + static_cast<size_t>(i) * TS::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full[i], kTx);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[i], pol_w);
      }
      for (int i = pre; i < nk && i < pre + g.l2_prefetch; ++i) tma_prefetch_l2_2d(&tmW, (kb0 + i) * kBK, w_row);
      pdl_wait();
      if (!FUSED) {
        for (int i = 0; i < pre; ++i) {
          uint8_t* st = smem + static_cast<size_t>(i) * TS::kStageBytes;
          tma_load_2d(st + TS::kWBytes, &tmA, (kb0 + i) * kBK, m_base, &ctl->full[i], pol_a);
        }
      }
      int issued = pre;
      for (int i = pre; i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
        if (!mbar_wait(&ctl->empty[s], ph ^ 1u, g.wait_ns) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(s) * TS::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full[s], kTx);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[s], pol_w);
        if (g.l2_prefetch > 0 && i + g.l2_prefetch < nk) tma_prefetch_l2_2d(&tmW, (kb0 + i + g.l2_prefetch) * kBK, w_row);
        if (!FUSED) tma_load_2d(st + TS::kWBytes, &tmA, (kb0 + i) * kBK, m_base, &ctl->full[s], pol_a);
        issued = i + 1;
      }
      // Every issued copy lands before this CTA may exit or reuse the ring.
      for (int j = issued > stages ? issued - stages : 0; j < issued; ++j)
        mbar_wait(&ctl->full[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
    }
  } else {
    if (warp == 1) tmem_alloc(&ctl->tmem_base, kTmemCols);
    tc_fence_before();
    named_bar_sync(2, kT - 32);
    tc_fence_after();
    const uint32_t tmem = ctl->tmem_base;
    if (QWARPS && warp >= 6) {
      // --------------------------------- Block_FP8 activation quantizers
      block_fused_quantize<MPAD>(g, ctl, smem, TS::kStageBytes, TS::kWBytes, stages, nk, kb0, m_base, Mb, n_tile,
                                 abort_flag);
    } else if (warp == 1) {
      // -------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc = make_idesc(128, MPAD, 0, 0);  // E4M3 x E4M3 -> F32
        bool ok = true;
        if (g.force_timeout) ok = mbar_wait(&ctl->never, 0, g.wait_ns);
        for (int i = 0; ok && i < nk; ++i) {
          const int s = i % stages;
          const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
          const int buf = BLOCK ? i % NBUF : 0;
          if (BLOCK && i >= NBUF) {
            if (!mbar_wait(&ctl->tempty[buf], static_cast<uint32_t>(i / NBUF - 1) & 1u, g.wait_ns)) {
              ok = false;
              break;
            }
          }
          if (!mbar_wait(&ctl->full[s], ph, g.wait_ns) || (FUSED && !mbar_wait(&ctl->full_a[s], ph, g.wait_ns))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t w_addr = smem_u32(smem + static_cast<size_t>(s) * TS::kStageBytes);
          const uint32_t a_addr = w_addr + TS::kWBytes;
          const uint32_t d = tmem + static_cast<uint32_t>(buf * MPAD);
#pragma unroll
          for (int kk = 0; kk < kBK / 32; ++kk) {
            const uint32_t accumulate = BLOCK ? (kk > 0) : (i > 0 || kk > 0);
            mma_f8f6f4(d, sw128_kmajor_desc(w_addr + kk * 32), sw128_kmajor_desc(a_addr + kk * 32), idesc,
                       accumulate);
          }
          tc_commit(&ctl->empty[s]);
          if (BLOCK) tc_commit(&ctl->tfull[buf]);
        }
        if (!ok) {
          *abort_flag = 1;
          if (BLOCK)
            for (int b = 0; b < NBUF; ++b) mbar_arrive(&ctl->tfull[b]);
        }
        // Completes once every MMA issued above has finished (also on abort).
        tc_commit(&ctl->acc_full);
      }
    } else {
      // ---------------------------------------------- epilogue: TMEM -> acc
      pdl_wait();
      const int q = warp & 3;  // TMEM lane quarter this warp may access
      const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
      if constexpr (!BLOCK) {
        // scales for the epilogue, fetched while the main loop runs
        const int et0 = threadIdx.x - 64, r = q * 32 + lane, nn = n_tile * kBN + r;
        if (!FUSED && et0 < MPAD) ctl->sa_s[et0] = et0 < Mb ? __ldg(g.s_a + m_base + et0) : 0.0f;
        ctl->sw_s[r] = nn < g.N ? __ldg(s_w + nn) : 0.0f;
      }
      if constexpr (FUSED && !BLOCK) {
        // per-token scales, then every stage's activation tile as E4M3
        const int et0 = threadIdx.x - 64;
        const bool whole_row = !clustered && g.splits > 1;
        const int k0 = whole_row ? 0 : kb0 * kBK, k1 = whole_row ? g.K : min(g.K, kb1 * kBK);
        fused_token_scales(g, m_base, Mb, k0, k1, clustered, clustered ? split : 0, 448.0f, ctl->amax_s, ctl->sa_s,
                           &ctl->amax_bar, et0, 128, 3, n_tile == 0 && split == 0);
        const bool write_codes = g.a_q_out != nullptr && n_tile == 0;
        // Pieces of 32 activations (token row r, quarter p of the k-tile),
        // kPP per thread.  The next k-tile's pieces are loaded while this
        // one is quantized, and a stage's activation tile is written as soon
        // as the MMAs of the stage's previous use are done (empty[s]), ahead
        // of its weight tile.
        constexpr int kPP = (MPAD * 4 + 127) / 128;
        uint4 cur[kPP][4], nxt[kPP][4];
        auto fetch = [&](int i, uint4(&buf)[kPP][4]) {
#pragma unroll
          for (int q = 0; q < kPP; ++q) {
            const int piece = et0 + 128 * q, r = piece >> 2, p = piece & 3;
            if (piece < MPAD * 4 && r < Mb)
              load_act_raw(g, m_base + r, (kb0 + i) * kBK + 32 * p, buf[q]);
            else
#pragma unroll
              for (int c = 0; c < 4; ++c) buf[q][c] = make_uint4(0u, 0u, 0u, 0u);
          }
        };
        fetch(0, cur);
        for (int i = 0; i < nk; ++i) {
          const int s = i % stages;
          if (i + 1 < nk) fetch(i + 1, nxt);
          if (i >= stages &&
              !__all_sync(0xffffffffu, mbar_wait(&ctl->empty[s], static_cast<uint32_t>(i / stages - 1) & 1u, g.wait_ns) &&
                                           !*abort_flag)) {
            *abort_flag = 1;
            break;
          }
          const int kt0 = (kb0 + i) * kBK;
          uint8_t* at = smem + static_cast<size_t>(s) * TS::kStageBytes + TS::kWBytes;
#pragma unroll
          for (int q = 0; q < kPP; ++q) {
            const int piece = et0 + 128 * q, r = piece >> 2, p = piece & 3;
            if (piece >= MPAD * 4) continue;
            uint32_t w[8];
            if (r < Mb) {
              float x[32];
              unpack_act32(cur[q], x);
              float qv[32];
              Divider(ctl->sa_s[r]).divide(x, qv);
#pragma unroll
              for (int j = 0; j < 8; ++j)
                w[j] = static_cast<uint32_t>(e4m3x2(qv[4 * j], qv[4 * j + 1])) |
                       (static_cast<uint32_t>(e4m3x2(qv[4 * j + 2], qv[4 * j + 3])) << 16);
              if (write_codes) {
                uint8_t* dst = g.a_q_out + static_cast<int64_t>(m_base + r) * g.K + kt0 + 32 * p;
#pragma unroll
                for (int c = 0; c < 2; ++c)
                  if (kt0 + 32 * p + 16 * c < g.K)
                    *reinterpret_cast<uint4*>(dst + 16 * c) = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
              }
            } else {
#pragma unroll
              for (int j = 0; j < 8; ++j) w[j] = 0u;
            }
            *reinterpret_cast<uint4*>(at + sw128_chunk(r, 2 * p)) = make_uint4(w[0], w[1], w[2], w[3]);
            *reinterpret_cast<uint4*>(at + sw128_chunk(r, 2 * p + 1)) = make_uint4(w[4], w[5], w[6], w[7]);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->full_a[s]);
#pragma unroll
          for (int q = 0; q < kPP; ++q)
#pragma unroll
            for (int c = 0; c < 4; ++c) cur[q][c] = nxt[q][c];
        }
      }
      if constexpr (BLOCK) {
        const int nb = n_tile;  // 128-row tile == weight block row
        // Two-kernel form: the products s_a[m,kb] * s_w[nb,kb] (the k-tile's
        // coefficient for each token) are staged in amax_s (unused by this
        // form), so the promotion reads them as shared-memory broadcasts and
        // spends one paired FMA per two tokens:
        //   staged   the CTA's whole K range fits: loaded with every request
        //            in flight right after the dependency wait;
        //   chunked  otherwise: two halves of kChunkTiles k-tiles each, the
        //            next chunk loaded into registers one chunk ahead and
        //            stored at the chunk boundary (one barrier of the 128
        //            promotion threads per chunk).
        constexpr int kHalfCoefs = kMaxClusterSplits * 32;  // floats in one half of amax_s
        constexpr int kChunkTiles = kHalfCoefs / MPAD;
        constexpr int kCoefPer = kHalfCoefs / kEpi;         // per promotion thread and chunk
        const bool staged = !FUSED && nk * MPAD <= kMaxClusterSplits * 64;
        const bool chunked = !FUSED && !staged;
        const int et = threadIdx.x - 64;  // promotion thread 0 .. kEpi-1
        float cpre[kCoefPer];
        auto load_chunk = [&](int c) {
#pragma unroll
          for (int j = 0; j < kCoefPer; ++j) {
            const int e = et + kEpi * j;
            const int i = c * kChunkTiles + e / MPAD, t = e % MPAD;
            cpre[j] = (i < nk && t < Mb) ? __ldg(g.s_a + static_cast<int64_t>(m_base + t) * g.kt_total + kb0 + i) *
                                               __ldg(s_w + static_cast<int64_t>(nb) * g.kt_total + kb0 + i)
                                         : 0.0f;
          }
        };
        auto store_chunk = [&](int c) {
#pragma unroll
          for (int j = 0; j < kCoefPer; ++j) ctl->amax_s[(c & 1) * kHalfCoefs + et + kEpi * j] = cpre[j];
        };
        if (staged) {
          // loads issued in rounds of up to four before their products
          constexpr int kPer = kMaxClusterSplits * 64 / kEpi;
          constexpr int kRound = kPer > 4 ? 4 : kPer;
#pragma unroll
          for (int r0 = 0; r0 < kPer; r0 += kRound) {
            float ra[kRound], rw[kRound];
#pragma unroll
            for (int j = 0; j < kRound; ++j) {
              const int e = et + kEpi * (r0 + j);
              const int i = e / MPAD, t = e % MPAD;
              const bool ok_e = e < nk * MPAD && t < Mb;
              ra[j] = ok_e ? __ldg(g.s_a + static_cast<int64_t>(m_base + t) * g.kt_total + kb0 + i) : 0.0f;
              rw[j] = ok_e ? __ldg(s_w + static_cast<int64_t>(nb) * g.kt_total + kb0 + i) : 0.0f;
            }
#pragma unroll
            for (int j = 0; j < kRound; ++j)
              if (et + kEpi * (r0 + j) < nk * MPAD) ctl->amax_s[et + kEpi * (r0 + j)] = ra[j] * rw[j];
          }
          named_bar_sync(1, kEpi);
        } else if (chunked) {
          load_chunk(0);
          store_chunk(0);
          if (nk > kChunkTiles) load_chunk(1);
          named_bar_sync(1, kEpi);
        }
        // fused form: lane l holds s_a of tokens l, l + 32, ... for the
        // current k-tile
        constexpr int kSaw = (MPAD + 31) / 32;
        float sa_cur[kSaw];
        float sw_next = FUSED ? __ldg(s_w + static_cast<int64_t>(nb) * g.kt_total + kb0) : 0.0f;
        // After a failed wait a warp stays in the loop without working, so
        // that every promotion thread reaches every chunk barrier.
        bool dead = false;
        for (int i = 0; i < nk; ++i) {
          const int buf = i % NBUF;
          if (chunked && i > 0 && i % kChunkTiles == 0) {
            // chunk c's half was last read in chunk c - 2, which every
            // promotion thread left before the previous barrier
            const int c = i / kChunkTiles;
            store_chunk(c);
            if ((c + 1) * kChunkTiles < nk) load_chunk(c + 1);
            named_bar_sync(1, kEpi);
          }
          if (dead) continue;
          float sw_cur = 0.0f;
          if constexpr (FUSED) {
            // this k-tile's scales, from the quantizer warps through the ring
            const int slot = i % kSaRing;
            if (!__all_sync(0xffffffffu, mbar_wait(&ctl->sfull[slot], static_cast<uint32_t>(i / kSaRing) & 1u,
                                                   g.wait_ns) && !*abort_flag)) {
              *abort_flag = 1;
              dead = true;
              continue;
            }
#pragma unroll
            for (int j = 0; j < kSaw; ++j) {
              const int t = lane + 32 * j;
              sa_cur[j] = t < MPAD ? ctl->amax_s[slot * 64 + t] : 0.0f;
            }
            sw_cur = sw_next;
            if (i + 1 < nk) sw_next = __ldg(s_w + static_cast<int64_t>(nb) * g.kt_total + kb0 + i + 1);
          }
          const bool w = mbar_wait(&ctl->tfull[buf], static_cast<uint32_t>(i / NBUF) & 1u, g.wait_ns);
          if (!__all_sync(0xffffffffu, w && !*abort_flag)) {
            *abort_flag = 1;
            dead = true;
            continue;
          }
          tc_fence_after();
          uint32_t v[kTP];
          tmem_ld_cols(tmem + lane_base + static_cast<uint32_t>(buf * MPAD + t0), v);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();  // the warp's TMEM reads of the buffer are done
          if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
          if constexpr (!FUSED) {
            const float* coefs =
                (staged ? ctl->amax_s + i * MPAD
                        : ctl->amax_s + ((i / kChunkTiles) & 1) * kHalfCoefs + (i % kChunkTiles) * MPAD) + t0;
#pragma unroll
            for (int m = 0; m < kTP; m += 4) {
              const float4 c4 = *reinterpret_cast<const float4*>(coefs + m);
              const float2 r0 = __ffma2_rn(make_float2(c4.x, c4.y),
                                           make_float2(__uint_as_float(v[m]), __uint_as_float(v[m + 1])),
                                           make_float2(acc[m], acc[m + 1]));
              const float2 r1 = __ffma2_rn(make_float2(c4.z, c4.w),
                                           make_float2(__uint_as_float(v[m + 2]), __uint_as_float(v[m + 3])),
                                           make_float2(acc[m + 2], acc[m + 3]));
              acc[m] = r0.x;
              acc[m + 1] = r0.y;
              acc[m + 2] = r1.x;
              acc[m + 3] = r1.y;
            }
          } else {
#pragma unroll
            for (int m = 0; m < MPAD; ++m) {
              const float coef = __shfl_sync(0xffffffffu, sa_cur[m / 32], m & 31) * sw_cur;
              acc[m] = fmaf(coef, __uint_as_float(v[m]), acc[m]);
            }
          }
        }
        // the MMA thread's final commit: all MMAs done before teardown
        mbar_wait(&ctl->acc_full, 0, g.wait_ns);
      } else {
        if (!__all_sync(0xffffffffu, mbar_wait(&ctl->acc_full, 0, g.wait_ns))) *abort_flag = 1;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < MPAD; c += 8) {
          uint32_t t[8];
          tmem_ld_x8(tmem + lane_base + static_cast<uint32_t>(c), t);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[c + j] = __uint_as_float(t[j]);
        }
        tmem_ld_wait();
      }
    }
  }
  // ------------------------------------------- all roles done: TMEM free
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(ctl->tmem_base, kTmemCols);
  }
  const bool abort = ctl->abort_flag != 0;  // stable after the barrier: uniform
  const int row = (warp & 3) * 32 + lane;   // epilogue threads: weight row in the tile
  const int n = n_tile * kBN + row;
  const int et = threadIdx.x - 64;          // 0 .. kEpi-1 for the epilogue warps
  // m: token of this block; r: row of the tile (scales staged in shared
  // memory); nn = n_tile*128 + r
  auto out = [&](int m, int r, int nn, float sum) {
    const float y = BLOCK ? sum : (sum * ctl->sa_s[m]) * ctl->sw_s[r];
    store_bf16(g.Y + static_cast<int64_t>(m_base + m) * g.ldy + nn, y);
  };

  const bool epi = warp >= 2 && warp < 2 + PW;  // the epilogue warps hold the accumulators
  if (clustered) {
    if (epi) {
      if (!FUSED || BLOCK) cluster_wait();  // every peer's receive barrier is initialized (fused FP8: waited already)
      // rows go out even after an abort, so that every owner's wait completes
      cluster_push_row(acc, t0, row, split, g.splits, Mb, recv, &ctl->recv_bar);
      named_bar_sync(1, kEpi);  // this CTA's own rows, stored locally, are visible
      const bool got = __all_sync(0xffffffffu, mbar_wait_cluster(&ctl->recv_bar, 0, g.wait_ns));
      if (got && !abort) {
        cluster_sum_rows<float>(recv, split, g.splits, Mb, et, kEpi, [&](int m, int r, float sum) {
          const int nn = n_tile * kBN + r;
          if (nn < g.N) out(m, r, nn, sum);
        });
      }
    } else {
      // the producer, MMA (and quantizer) warps pair their early arrive with
      // a wait too (every peer arrived right after its set-up, so this
      // returns at once)
      cluster_wait();
    }
  } else if (epi && !abort) {
    const bool n_ok = n < g.N;
    if (g.reduce == kReduceNone) {
      if (n_ok) {
#pragma unroll
        for (int m = 0; m < kTP; ++m)
          if (t0 + m < Mb) out(t0 + m, row, n, acc[m]);
      }
    } else {
      float* part = static_cast<float*>(g.ws_part);
      if (n_ok) {
#pragma unroll
        for (int m = 0; m < kTP; ++m)
          if (t0 + m < Mb) part[(static_cast<int64_t>(split) * g.M + m_base + t0 + m) * g.N + n] = acc[m];
      }
      __threadfence();
      named_bar_sync(1, kEpi);
      const int tile_id = blockIdx.x + blockIdx.z * gridDim.x;
      if (et == 0) {
        const int old = atomicAdd(g.ws_count + tile_id, 1);
        ctl->last_flag = (old == g.splits - 1);
      }
      named_bar_sync(1, kEpi);
      if (ctl->last_flag) {
        __threadfence();
        if (n_ok) {
          for (int m = t0; m < min(Mb, t0 + kTP); ++m) {
            float sum = 0.0f;
            for (int s = 0; s < g.splits; ++s)
              sum += ld_cg_f32(part + (static_cast<int64_t>(s) * g.M + m_base + m) * g.N + n);
            out(m, row, n, sum);
          }
        }
        if (et == 0) g.ws_count[tile_id] = 0;  // ready for the next launch
      }
    }
  }
  stamp_end(g.tstamp);
}

// ----------------------------------------------------------- Standard --
// Tokens on the MMA M side: one CTA per (128-token tile, 128-row weight
// tile, K range); D[128 tokens x 128 weight rows] in TMEM.  Serves M > 32
// (and M <= 32 when the table picks it); Split-K uses the global workspace.
// BNW: weight rows per tile and MMA N (128; 256 for FP8_Dynamic's wide
// tiles, which halve the MMA instructions and the activation-tile loads per
// output).
// Block_FP8: each k-tile's partial lands in one of four TMEM buffers (all
// 512 columns: one CTA per SM) and eight promotion warps (two per TMEM lane
// quarter, each owning 64 of the tile's weight rows) add it, times the
// k-tile's coefficient s_a[m,kb] * s_w[nb,kb], into register accumulators.
template <int FMT, int BNW>
__global__ void __launch_bounds__(std_threads(FMT), 1)
    gemm_f8_std_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmA, GemmArgs g) {
  using TS = StdShape<BNW>;
  constexpr bool BLOCK = (FMT == kFmtBlock);
  static_assert(BNW == 128 || (BNW == 256 && !BLOCK), "wide tiles are FP8_Dynamic only");
  constexpr int NBUF = BLOCK ? 4 : 1;
  // D is 128 lanes x BNW cols per buffer
  constexpr uint32_t kBufCols = BNW;
  constexpr uint32_t kTmemCols = pow2_cols(NBUF * kBufCols);
  static_assert(kTmemCols <= 512, "TMEM budget");
  constexpr int kEpi = std_threads(FMT) - 64;        // epilogue threads (2 or 4 per TMEM lane)
  constexpr int kCols = BLOCK ? kBN / 2 : BNW;        // weight rows (TMEM columns) of each

  stamp_start(g.tstamp);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align1024(smem_raw);
  const int stages = g.stages;
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + static_cast<size_t>(stages) * TS::kStageBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // the token tiles of one weight tile are adjacent block indices (weights
  // read from HBM once, then from L2)
  const int n_tile = static_cast<int>(blockIdx.x / g.m_tiles);
  const int m_tile = static_cast<int>(blockIdx.x % g.m_tiles);
  const int split = blockIdx.y;
  const int kb0 = static_cast<int>(static_cast<int64_t>(split) * g.kt_total / g.splits);
  const int kb1 = static_cast<int>(static_cast<int64_t>(split + 1) * g.kt_total / g.splits);
  const int nk = kb1 - kb0;

  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&ctl->full[i], 1);
      mbar_init(&ctl->empty[i], 1);
    }
    mbar_init(&ctl->acc_full, 1);
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&ctl->tfull[b], 1);
      mbar_init(&ctl->tempty[b], kEpi / 32);  // one arrive per promotion warp
    }
    mbar_init(&ctl->never, 1);
    ctl->last_flag = 0;
    ctl->abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmA);
  }
  if (warp == 1) tmem_alloc(&ctl->tmem_base, kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  pdl_launch_dependents();
  volatile int* abort_flag = &ctl->abort_flag;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_a = policy_evict_last();
      const int w_row = n_tile * BNW;
      const int a_row = m_tile * 128;
      const int pre = nk < stages ? nk : stages;
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = smem + static_cast<size_t>(i) * TS::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full[i], TS::kStageBytes);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[i], pol_w);
      }
      for (int i = pre; i < nk && i < pre + g.l2_prefetch; ++i) tma_prefetch_l2_2d(&tmW, (kb0 + i) * kBK, w_row);
      pdl_wait();
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = smem + static_cast<size_t>(i) * TS::kStageBytes;
        tma_load_2d(st + TS::kWBytes, &tmA, (kb0 + i) * kBK, a_row, &ctl->full[i], pol_a);
      }
      int issued = pre;
      for (int i = pre; i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
        if (!mbar_wait(&ctl->empty[s], ph ^ 1u, g.wait_ns) || *abort_flag) {
          *abort_flag = 1;
          break;
        }
        uint8_t* st = smem + static_cast<size_t>(s) * TS::kStageBytes;
        mbar_arrive_expect_tx(&ctl->full[s], TS::kStageBytes);
        tma_load_2d(st, &tmW, (kb0 + i) * kBK, w_row, &ctl->full[s], pol_w);
        if (g.l2_prefetch > 0 && i + g.l2_prefetch < nk) tma_prefetch_l2_2d(&tmW, (kb0 + i + g.l2_prefetch) * kBK, w_row);
        tma_load_2d(st + TS::kWBytes, &tmA, (kb0 + i) * kBK, a_row, &ctl->full[s], pol_a);
        issued = i + 1;
      }
      for (int j = issued > stages ? issued - stages : 0; j < issued; ++j)
        mbar_wait(&ctl->full[j % stages], static_cast<uint32_t>(j / stages) & 1u, kDrainNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc = make_idesc(128, BNW, 0, 0);  // E4M3 x E4M3 -> F32
      bool ok = true;
      if (g.force_timeout) ok = mbar_wait(&ctl->never, 0, g.wait_ns);
      for (int i = 0; ok && i < nk; ++i) {
        const int s = i % stages;
        const uint32_t ph = static_cast<uint32_t>(i / stages) & 1u;
        const int buf = BLOCK ? i % NBUF : 0;
        if (BLOCK && i >= NBUF) {
          if (!mbar_wait(&ctl->tempty[buf], static_cast<uint32_t>(i / NBUF - 1) & 1u, g.wait_ns)) {
            ok = false;
            break;
          }
        }
        if (!mbar_wait(&ctl->full[s], ph, g.wait_ns)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t w_addr = smem_u32(smem + static_cast<size_t>(s) * TS::kStageBytes);
        const uint32_t a_addr = w_addr + TS::kWBytes;
        const uint32_t d = tmem + static_cast<uint32_t>(buf) * kBufCols;
#pragma unroll
        for (int kk = 0; kk < kBK / 32; ++kk) {
          const uint32_t accumulate = BLOCK ? (kk > 0) : (i > 0 || kk > 0);
          mma_f8f6f4(d, sw128_kmajor_desc(a_addr + kk * 32), sw128_kmajor_desc(w_addr + kk * 32), idesc, accumulate);
        }
        tc_commit(&ctl->empty[s]);
        if (BLOCK) tc_commit(&ctl->tfull[buf]);
      }
      if (!ok) {
        *abort_flag = 1;
        if (BLOCK)
          for (int b = 0; b < NBUF; ++b) mbar_arrive(&ctl->tfull[b]);
      }
      tc_commit(&ctl->acc_full);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // TMEM lane = token row m, columns = weight rows n; this thread's
    // columns are [c0, c0 + kCols).
    pdl_wait();
    const int q = warp & 3;
    const uint32_t lane_base = static_cast<uint32_t>(q * 32) << 16;
    const int et = threadIdx.x - 64;  // 0 .. kEpi-1
    const int c0 = ((warp - 2) >> 2) * kCols;
    const int m = m_tile * 128 + q * 32 + lane;
    const bool m_ok = m < g.M;
    float acc[BLOCK ? kCols : 1];  // Block: the promoted sums of this thread's columns
#pragma unroll
    for (int c = 0; c < (BLOCK ? kCols : 1); ++c) acc[c] = 0.0f;
    if constexpr (BLOCK) {
      const int nb = n_tile;
      // the k-tiles' scales, requested kAhead k-tiles ahead into a register
      // ring (an L2 round trip is several k-tiles of promotion) and
      // multiplied only when used, so no warp waits on a load it issued
      constexpr int kAhead = 4;
      float ring_a[kAhead], ring_w[kAhead];
      auto fetch = [&](int u, int i) {
        const bool ok_i = m_ok && i < nk;
        ring_a[u] = ok_i ? __ldg(g.s_a + static_cast<int64_t>(m) * g.kt_total + kb0 + i) : 0.0f;
        ring_w[u] = ok_i ? __ldg(g.s_w + static_cast<int64_t>(nb) * g.kt_total + kb0 + i) : 0.0f;
      };
#pragma unroll
      for (int u = 0; u < kAhead; ++u) fetch(u, u);
      bool ok = true;
      for (int i0 = 0; ok && i0 < nk; i0 += kAhead)
#pragma unroll
      for (int u = 0; u < kAhead; ++u) {
        const int i = i0 + u;
        if (i >= nk) break;
        const int buf = i % NBUF;
        const float sa_i = ring_a[u], sw_i = ring_w[u];
        fetch(u, i + kAhead);
        const bool w = mbar_wait(&ctl->tfull[buf], static_cast<uint32_t>(i / NBUF) & 1u, g.wait_ns);
        if (!__all_sync(0xffffffffu, w && !*abort_flag)) {
          *abort_flag = 1;
          ok = false;
          break;
        }
        tc_fence_after();
        const float coef = sa_i * sw_i;
        const float2 cc = make_float2(coef, coef);
        // the buffer's columns in two halves of 32 (registers)
#pragma unroll
        for (int h = 0; h < kCols; h += 32) {
          uint32_t v[32];
          tmem_ld_cols(tmem + lane_base + static_cast<uint32_t>(buf * kBufCols + c0 + h), v);
          tmem_ld_wait();
          if (h + 32 >= kCols) {
            tc_fence_before();
            __syncwarp();  // the warp's TMEM reads of the buffer are done
            if (lane == 0) mbar_arrive(&ctl->tempty[buf]);
          }
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const float2 r = __ffma2_rn(cc, make_float2(__uint_as_float(v[c]), __uint_as_float(v[c + 1])),
                                        make_float2(acc[h + c], acc[h + c + 1]));
            acc[h + c] = r.x;
            acc[h + c + 1] = r.y;
          }
        }
      }
      mbar_wait(&ctl->acc_full, 0, g.wait_ns);
    } else {
      if (!__all_sync(0xffffffffu, mbar_wait(&ctl->acc_full, 0, g.wait_ns))) *abort_flag = 1;
    }
    tc_fence_after();
    const bool abort = __any_sync(0xffffffffu, *abort_flag != 0);
    const float sa = (!BLOCK && m_ok) ? __ldg(g.s_a + m) : 1.0f;
    float* part = static_cast<float*>(g.ws_part);
    // this thread's 8 results of columns [c0 + c, c0 + c + 8) to Y (or to
    // its Split-K partial)
    auto emit = [&](int c, const uint32_t (&t)[8]) {
      const int n0 = n_tile * BNW + c0 + c;
      if (!m_ok) return;
      if (g.splits == 1) {
        if (n0 + 8 <= g.N) {
          uint32_t packed[4];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            float y0 = __uint_as_float(t[2 * j]), y1 = __uint_as_float(t[2 * j + 1]);
            if (!BLOCK) {
              y0 = (y0 * sa) * __ldg(g.s_w + n0 + 2 * j);
              y1 = (y1 * sa) * __ldg(g.s_w + n0 + 2 * j + 1);
            }
            __nv_bfloat162 h = __floats2bfloat162_rn(y0, y1);
            packed[j] = *reinterpret_cast<uint32_t*>(&h);
          }
          __nv_bfloat16* dst = g.Y + static_cast<int64_t>(m) * g.ldy + n0;
          if ((reinterpret_cast<uintptr_t>(dst) & 15) == 0) {
            *reinterpret_cast<uint4*>(dst) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
          } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) *reinterpret_cast<uint32_t*>(dst + 2 * j) = packed[j];
          }
        } else {
          for (int j = 0; j < 8 && n0 + j < g.N; ++j) {
            float y = __uint_as_float(t[j]);
            if (!BLOCK) y = (y * sa) * __ldg(g.s_w + n0 + j);
            store_bf16(g.Y + static_cast<int64_t>(m) * g.ldy + n0 + j, y);
          }
        }
      } else {
        for (int j = 0; j < 8 && n0 + j < g.N; ++j)
          part[(static_cast<int64_t>(split) * g.M + m) * g.N + n0 + j] = __uint_as_float(t[j]);
      }
    };
    if (!abort) {
      if constexpr (BLOCK) {
#pragma unroll
        for (int c = 0; c < kCols; c += 8) {
          uint32_t t[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) t[j] = __float_as_uint(acc[c + j]);
          emit(c, t);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < kCols; c += 8) {
          uint32_t t[8];
          tmem_ld_x8(tmem + lane_base + static_cast<uint32_t>(c), t);
          tmem_ld_wait();
          emit(c, t);
        }
      }
    }
    if (g.splits > 1 && !abort) {
      __threadfence();
      named_bar_sync(1, kEpi);
      const int tile_id = blockIdx.x;
      if (et == 0) {
        const int old = atomicAdd(g.ws_count + tile_id, 1);
        ctl->last_flag = (old == g.splits - 1);
      }
      named_bar_sync(1, kEpi);
      if (ctl->last_flag) {
        __threadfence();
        if (m_ok) {
          for (int c = c0; c < c0 + kCols; ++c) {
            const int n = n_tile * BNW + c;
            if (n >= g.N) break;
            float sum = 0.0f;
            for (int s = 0; s < g.splits; ++s) sum += ld_cg_f32(part + (static_cast<int64_t>(s) * g.M + m) * g.N + n);
            const float y = BLOCK ? sum : (sum * sa) * __ldg(g.s_w + n);
            store_bf16(g.Y + static_cast<int64_t>(m) * g.ldy + n, y);
          }
        }
        if (et == 0) g.ws_count[tile_id] = 0;
      }
    }
  }
  // ------------------------------------------------------------- teardown
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  stamp_end(g.tstamp);
}

}  // namespace qg
