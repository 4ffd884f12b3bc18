/*
 * qgemm.h -- C ABI of the B300 (sm_103a) quantized decode GEMM library.
 *
 * Computes the quantized linear layer
 *     Y[M,N] = bf16( dequant( A_q[M,K] . W_q[N,K]^T ) )
 * at decode token counts (M = 1..32, larger M also accepted) in the three
 * formats of "Building a High-Performance and Portable vLLM Linear Backend
 * with Helion" (discuss.pytorch.kr / PyTorch blog), section "Helion Linear
 * Backend > Scope":
 *   QG_FP8_DYNAMIC  E4M3 activations with one dynamic scale per token (row),
 *                   E4M3 weights with one scale per output channel;
 *   QG_W8A8_INT8    the same with symmetric int8 and an int32 accumulator;
 *   QG_BLOCK_FP8    E4M3 with one activation scale per 1x128 group and one
 *                   weight scale per 128x128 block;
 * with the Standard, Split-K and Swap-AB algorithm variants of its section
 * "Kernel Implementation", chosen per shape from a tuned table (sections
 * "Per-shape Config Tuning" and "Hybrid Dispatch"); plus a grouped form for
 * mixture-of-experts layers (its "Future work > Model coverage").
 *
 * Numerics (the page states no formulas; these are this library's readings):
 *   scale s = amax / 448 (E4M3) or amax / 127 (int8) in IEEE fp32, s = 1 for
 *   an all-zero row, group or block; q = round-to-nearest-even of the
 *   correctly rounded fp32 quotient x / s (one IEEE division, or Markstein's
 *   method, which gives the same quotient), saturated to +-448 / [-127, 127],
 *   the sign of a zero kept;
 *   FP8_Dynamic / INT8:  Y = bf16_rn((float(acc) * s_a[m]) * s_w[n]);
 *   Block_FP8:           Y = bf16_rn(sum_kb s_a[m,kb] * s_w[n/128,kb] * acc_kb).
 *
 * Conventions for every entry point:
 *   - returns a qg_status (0 = QG_OK); no exception crosses the ABI and
 *     nothing aborts; on error qg_last_error() describes the failure;
 *   - pointers named *_dev are device pointers owned by the caller; the
 *     library never allocates, frees or synchronizes on the call path and
 *     only enqueues kernels on `stream` (a cudaStream_t, NULL = legacy
 *     default stream), so the calls can be captured in a CUDA graph;
 *   - all matrices are row-major with K contiguous; K % 16 == 0 (TMA rows
 *     are 16-byte multiples); Block_FP8 also needs K % 128 == 0;
 *     A_q / W_q / A / W base pointers 16-byte aligned; scales 4-byte aligned;
 *   - kernel-side failures (a pipeline wait that exceeded its time bound) do
 *     not trap: they set a device status word read by qg_device_error().
 */
#ifndef QGEMM_H
#define QGEMM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define QG_API __attribute__((visibility("default")))
#else
#define QG_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { QG_FP8_DYNAMIC = 0, QG_W8A8_INT8 = 1, QG_BLOCK_FP8 = 2 } qg_format;

/* Algorithm variants ("Kernel Implementation"): Standard puts tokens on the
 * MMA M side; Swap-AB computes Y^T = W_q . A_q^T so the weight rows take the
 * MMA M side (small M); the *_SPLITK forms also cut K into split_k ranges.
 * QG_SWAPAB_DP4A(_SPLITK) keep the Swap-AB work split but run the int8 dot
 * products on the CUDA cores (dp4a, int32 accumulation) instead of the
 * tensor cores: W8A8_INT8 with M <= 8 only (QG_ERR_UNSUPPORTED_SHAPE
 * otherwise). */
typedef enum {
  QG_STANDARD = 0,
  QG_SPLITK = 1,
  QG_SWAPAB = 2,
  QG_SWAPAB_SPLITK = 3,
  QG_SWAPAB_DP4A = 4,
  QG_SWAPAB_DP4A_SPLITK = 5
} qg_variant;

#define QG_CONFIG_RING_MASK 31
#define QG_CONFIG_PREFETCH_SHIFT 5
#define QG_CONFIG_PREFETCH_MASK (127 << 5)
#define QG_CONFIG_MAX_PREFETCH 64
#define QG_CONFIG_WIDE (1 << 12)
#define QG_CONFIG_MMA_SYNC (1 << 13)
#define QG_CONFIG_MMA_NARROW (1 << 14)
#define QG_CONFIG_FUSED_QUANT (1 << 15)
#define QG_CONFIG_PERSIST (1 << 16)
#define QG_CONFIG_MMA_DP4A_SHIFT 17
#define QG_CONFIG_MMA_DP4A_MASK (7 << 17)
#define QG_CONFIG_MMA_S8 (1 << 20)
#define QG_CONFIG_PAIR_MMA (1 << 21)
#define QG_CONFIG_I8_PREWIDEN (1 << 22)
#define QG_CONFIG_I8_CONV16 (1 << 23)
#define QG_CONFIG_BLOCK_PROMO8 (1 << 24)
#define QG_CONFIG_PERSIST_ROWS_SHIFT 25
#define QG_CONFIG_PERSIST_ROWS_MASK (3 << 25)

typedef enum {
  QG_OK = 0,
  QG_ERR_INVALID_ARG = -1,        /* null pointer, bad enum, negative size ... */
  QG_ERR_UNSUPPORTED_SHAPE = -2,  /* K % 16 (or % 128), split_k range, M too large for the variant */
  QG_ERR_ALIGNMENT = -3,          /* a pointer or stride breaks the alignment rules above */
  QG_ERR_WORKSPACE_TOO_SMALL = -4,
  QG_ERR_NO_CONFIG = -5,          /* qg_select: shape absent from the table and defaults disallowed */
  QG_ERR_CUDA = -6,               /* a CUDA runtime / driver call failed */
  QG_ERR_DEVICE_TIMEOUT = -7,     /* reported by qg_device_error(): a kernel wait timed out */
  QG_ERR_TABLE_PARSE = -8
} qg_status;

/* Dynamic activation quantization ("Scope": per-token for FP8_Dynamic and
 * W8A8_INT8, 1x128 groups for Block_FP8).
 *   A_dev    bf16 [M][lda] (lda >= K, lda % 8 == 0), read-only;
 *   A_q_dev  [M][K] E4M3 codes (uint8) or int8, written;
 *   s_a_dev  fp32 [M] (per token) or [M][K/128] (Block_FP8), written.
 * M == 0 is a no-op. */
QG_API int qg_quant_act(int fmt, const void* A_dev, int64_t M, int64_t K, int64_t lda, void* A_q_dev, float* s_a_dev,
                 void* stream);

/* Static weight quantization (offline setup, not on the decode path).
 *   W_dev    fp32 [N][K], read-only;
 *   W_q_dev  [N][K] E4M3 codes or int8, written;
 *   s_w_dev  fp32 [N] (per output channel) or [ceil(N/128)][K/128]
 *            (Block_FP8, 128x128 blocks; the last block row may be ragged). */
QG_API int qg_quant_weight(int fmt, const float* W_dev, int64_t N, int64_t K, void* W_q_dev, float* s_w_dev,
                    void* stream);

/* The same weight quantization on the host, for offline packing of
 * checkpoints (codes and scales bit for bit those of qg_quant_weight).
 *   W_host    fp32 [N][K] row-major, read-only (host memory);
 *   W_q_host  [N][K] E4M3 codes or int8, written (host memory);
 *   s_w_host  fp32 [N] or [ceil(N/128)][K/128] (Block_FP8), written.
 * Synchronous; no device work.  Errors: QG_ERR_INVALID_ARG (format, sizes,
 * null pointers), QG_ERR_UNSUPPORTED_SHAPE (K % 16, Block_FP8 K % 128). */
QG_API int qg_pack_weight(int fmt, const float* W_host, int64_t N, int64_t K, void* W_q_host, float* s_w_host);

/* Workspace bytes qg_gemm_w8a8 needs for this shape and variant with every
 * config_id except QG_CONFIG_I8_PREWIDEN (0 when the splits reduce without a
 * workspace, in particular when split_k == 1).  Layout: per-tile arrival
 * counters (must be zero before the first use; the kernels leave them zero
 * again), then the split partials.  Returns 0 for an invalid configuration. */
QG_API size_t qg_workspace_bytes(int fmt, int64_t M, int64_t N, int64_t K, int variant, int split_k);

/* The same for a given config_id (exact for every config_id):
 * QG_CONFIG_I8_PREWIDEN adds, 256-byte aligned after the Split-K part, the
 * fp16 copy of the activations (M x K x 2 bytes), which qg_gemm_w8a8 writes
 * before its GEMM kernel reads it (no initial contents needed). */
QG_API size_t qg_workspace_bytes_config(int fmt, int64_t M, int64_t N, int64_t K, int variant, int split_k,
                                        int config_id);

/* Validate a configuration without launching anything: the checks of
 * qg_gemm_w8a8 that need no pointer (format, variant, sizes, config_id,
 * K % 16 / K % 128, split_k range, the W8A8_INT8 and dp4a restrictions).
 * Returns the status qg_gemm_w8a8 would return for them; QG_OK does not
 * check pointers, alignment or the workspace size.  qg_load_table applies
 * the same checks to every row at its token count. */
QG_API int qg_check_config(int fmt, int64_t M, int64_t N, int64_t K, int variant, int split_k, int config_id);

/* Zero a workspace's counters (cudaMemsetAsync on `stream`). */
QG_API int qg_workspace_init(void* workspace_dev, size_t ws_bytes, void* stream);

/* The quantized GEMM ("Kernel Implementation" plus the format's scaling).
 *   A_q_dev, s_a_dev   from qg_quant_act (same fmt, M, K);
 *   W_q_dev, s_w_dev   from qg_quant_weight (same fmt, N, K);
 *   Y_dev              bf16 [M][ldy] (ldy >= N), fully overwritten;
 *   variant, split_k   a qg_variant and the number of K ranges (1 ..
 *                      ceil(K/128); must be 1 for the non-SPLITK variants);
 *   config_id          ring | distance << QG_CONFIG_PREFETCH_SHIFT: the
 *                      shared-memory ring depth in k-tiles (0 = library
 *                      default: the deepest ring that lets two CTAs share
 *                      an SM; at most 16) and the L2 prefetch distance: each
 *                      CTA keeps that many 16 KB weight k-tiles requested
 *                      into L2 ahead of the ring's loads, the first of them
 *                      before it waits for the kernel it depends on (0 =
 *                      off; at most QG_CONFIG_MAX_PREFETCH); plus
 *                      QG_CONFIG_WIDE for FP8_Dynamic with QG_STANDARD /
 *                      QG_SPLITK: 256 weight rows per tile (MMA N = 256)
 *                      instead of 128 (QG_ERR_INVALID_ARG elsewhere); plus
 *                      QG_CONFIG_MMA_SYNC for W8A8_INT8 with QG_SWAPAB /
 *                      QG_SWAPAB_SPLITK: the int8 products run on the
 *                      warp-level tensor-core instructions (mma.sync, the
 *                      operands widened to f16 in registers, token blocks
 *                      of up to 32) instead of tcgen05 with the widened
 *                      weights in tensor memory; same exact int32 result
 *                      (QG_ERR_INVALID_ARG elsewhere, and in the one-kernel
 *                      form of qg_linear_w8a8, which then runs two kernels);
 *                      with QG_CONFIG_MMA_SYNC also QG_CONFIG_MMA_NARROW:
 *                      eight MMA warps of 16 weight rows instead of four
 *                      of 32 (more warps to hide the widening's latency),
 *                      and with that d << QG_CONFIG_MMA_DP4A_SHIFT (d = 1..4,
 *                      M <= 16): the first 16*d rows of each weight tile go
 *                      to d warps of dp4a threads instead, on the integer
 *                      pipe the widening leaves idle (same exact result;
 *                      QG_ERR_UNSUPPORTED_SHAPE for M > 16); and with
 *                      QG_CONFIG_MMA_SYNC (any of the forms above) also
 *                      QG_CONFIG_MMA_S8: the MMA warps run the int8 form
 *                      of the instruction (m16n8k32, s8 operands, s32
 *                      accumulate) on the unwidened bytes -- same exact
 *                      result, no widening, at B300's much lower int8 MMA
 *                      rate;
 *                      plus QG_CONFIG_FUSED_QUANT (Swap-AB variants on the
 *                      tcgen05 kernels): a hint for qg_linear_w8a8 to take
 *                      its one-kernel form even when A_q / s_a buffers are
 *                      given (qg_gemm_w8a8 accepts and ignores it);
 *                      plus QG_CONFIG_PERSIST for FP8_Dynamic with
 *                      QG_STANDARD (the compute-bound regime, M of 64 and
 *                      more): a persistent kernel (at most one CTA per SM)
 *                      whose thread-block cluster pairs take two 128-token
 *                      tiles of one 256-row weight tile, each loading half
 *                      of the weight tile by TMA multicast into both CTAs,
 *                      with two TMEM accumulators so that a tile's epilogue
 *                      overlaps the next tile's MMAs; only the ring depth,
 *                      the L2 prefetch distance (weight k-tiles of the
 *                      CTA's half requested ahead, across tiles) and the
 *                      fields below may be combined with it
 *                      (QG_ERR_INVALID_ARG else); with it
 *                      also QG_CONFIG_PAIR_MMA: the pair runs each MMA as one
 *                      tcgen05.mma.cta_group::2 (M = 256 tokens, each CTA
 *                      holding only its own half of the weight tile, no
 *                      multicast), issued by the pair's even CTA; and
 *                      r << QG_CONFIG_PERSIST_ROWS_SHIFT: weight tiles of
 *                      256 (r = 0), 224, 192 or 160 rows (r = 1..3; MMA N),
 *                      so that a shape's tile count fills the last round of
 *                      the resident pairs better;
 *                      plus QG_CONFIG_I8_PREWIDEN for W8A8_INT8 with
 *                      QG_SWAPAB / QG_SWAPAB_SPLITK on the tcgen05 kernel
 *                      (the compute-bound regime): the call first widens the
 *                      activations once into an exact fp16 copy in the
 *                      workspace (a second kernel), and the GEMM loads that
 *                      copy by TMA instead of widening it in every CTA, in
 *                      token blocks of 16 / 32 / 64 (M <= 64) or 128 -- each
 *                      weight tile widened once per 128 tokens; only the ring
 *                      depth and the L2 prefetch distance may be combined
 *                      with it, and it is not for grouped launches or the
 *                      one-kernel form of qg_linear_w8a8 (QG_ERR_INVALID_ARG);
 *                      its workspace (qg_workspace_bytes_config) then holds
 *                      that copy, which may cover where another call keeps
 *                      its Split-K arrival counters: give such calls a
 *                      workspace of their own;
 *                      plus QG_CONFIG_I8_CONV16 for W8A8_INT8 with QG_SWAPAB /
 *                      QG_SWAPAB_SPLITK on the tcgen05 kernel (with or
 *                      without QG_CONFIG_I8_PREWIDEN): sixteen weight
 *                      converter warps instead of eight and one CTA per SM
 *                      with the deepest ring that fits, so that more weight
 *                      bytes are in flight per SM while they are widened;
 *                      not for grouped launches or the one-kernel form of
 *                      qg_linear_w8a8 (QG_ERR_INVALID_ARG);
 *                      plus QG_CONFIG_BLOCK_PROMO8 for Block_FP8 with
 *                      QG_SWAPAB / QG_SWAPAB_SPLITK: eight warps instead of
 *                      four promote each k-tile's partial with its block
 *                      scales (two per TMEM lane quarter, each taking half
 *                      of the token block); same result; not for grouped
 *                      launches nor with QG_CONFIG_FUSED_QUANT
 *                      (QG_ERR_INVALID_ARG); qg_linear_w8a8 runs it as two
 *                      kernels (A_q / s_a buffers required);
 *   workspace_dev      qg_workspace_bytes_config() bytes (may be NULL when 0);
 *   debug_acc_dev      W8A8_INT8 only, optional: int32 [M][N] receives the
 *                      exact integer accumulators (NULL to skip).
 * Concurrent calls on different streams must use different workspaces. */
QG_API int qg_gemm_w8a8(int fmt, int64_t M, int64_t N, int64_t K, const void* A_q_dev, const float* s_a_dev,
                 const void* W_q_dev, const float* s_w_dev, void* Y_dev, int64_t ldy, int variant, int split_k,
                 int config_id, void* workspace_dev, size_t ws_bytes, int32_t* debug_acc_dev, void* stream);

/* Grouped quantized GEMM for mixture-of-experts layers (the "Model
 * coverage" item of the page's "Future work"): `groups` GEMMs with the
 * same N and K in one launch, group g computing
 *     Y[t][n] = dequant( sum_k A_q[t][k] * W_q[g][n][k] )
 * for the tokens t in [token_offsets[g], token_offsets[g+1]) (tokens sorted
 * by group, as a router's permutation leaves them).
 *   token_offsets_dev  int32 [groups + 1] on the device, nondecreasing
 *                      within [0, total_tokens] (values outside are
 *                      clamped); read by the kernel after its dependency
 *                      wait, so a routing kernel may write them;
 *   total_tokens       rows of A_q / s_a / Y (0 is a no-op);
 *   max_tokens         an upper bound of any group's token count: it sizes
 *                      the token blocks; a group's tokens beyond the first
 *                      max_tokens are not computed (their Y rows are left
 *                      as they were);
 *   A_q_dev, s_a_dev   [total_tokens][K] codes and their scales (per token,
 *                      or per token and 128-K group for Block_FP8);
 *   W_q_dev            [groups][N][K] codes;
 *   s_w_dev            fp32 [groups][N], or [groups][ceil(N/128)][K/128]
 *                      (Block_FP8);
 *   Y_dev              bf16 [total_tokens][ldy];
 *   variant            QG_SWAPAB, QG_SWAPAB_SPLITK or (W8A8_INT8,
 *                      max_tokens <= 8) QG_SWAPAB_DP4A(_SPLITK);
 *   split_k, config_id, workspace (qg_workspace_bytes_grouped bytes),
 *   debug_acc_dev ([total_tokens][N])   as qg_gemm_w8a8.
 * CTAs of token blocks past their group's tokens (and of empty groups) exit
 * at once, so only the groups with tokens stream their weights. */
QG_API int qg_gemm_w8a8_grouped(int fmt, int groups, const int32_t* token_offsets_dev, int64_t total_tokens,
                                int64_t max_tokens, int64_t N, int64_t K, const void* A_q_dev,
                                const float* s_a_dev, const void* W_q_dev, const float* s_w_dev, void* Y_dev,
                                int64_t ldy, int variant, int split_k, int config_id, void* workspace_dev,
                                size_t ws_bytes, int32_t* debug_acc_dev, void* stream);
/* Workspace bytes of qg_gemm_w8a8_grouped (0 when none is needed or the
 * arguments are invalid). */
QG_API size_t qg_workspace_bytes_grouped(int fmt, int groups, int64_t total_tokens, int64_t max_tokens, int64_t N,
                                         int64_t K, int variant, int split_k);

/* The whole quantized linear layer in one call: dynamic activation
 * quantization ("Scope": per token, or per 1x128 group for Block_FP8)
 * followed by the quantized GEMM ("Kernel Implementation"), i.e.
 * qg_quant_act then qg_gemm_w8a8 with the same results bit for bit.
 * Two forms:
 *  - two kernels (when A_q_dev and s_a_dev are given and config_id does not
 *    carry QG_CONFIG_FUSED_QUANT; the only form of the Standard, dp4a and
 *    mma.sync kernels): the quantization kernel writes A_q / s_a, the GEMM
 *    follows (with QG_LAUNCH_PDL it streams its weights while the
 *    quantization runs).  The faster form on B300 for the per-token formats.
 *  - one kernel (QG_SWAPAB / QG_SWAPAB_SPLITK on the tcgen05 kernels, when
 *    A_q_dev or s_a_dev is NULL, config_id carries QG_CONFIG_FUSED_QUANT,
 *    or QG_LAUNCH_FUSED_QUANT is set): each CTA quantizes the slice of the
 *    activations its K range needs.  FP8_Dynamic / W8A8_INT8: the CTAs of
 *    a Split-K cluster agree on every token's maximum over the whole row
 *    through distributed shared memory.  Block_FP8: a group's scale needs
 *    only its own 128 values, so four more warps of each CTA quantize every
 *    k-tile on their own, with no wait for another CTA: one kernel and one
 *    dependency wait per linear layer instead of two.  A_q / s_a are
 *    written only when given (by the CTAs of the first weight tile).
 *   A_dev      bf16 [M][lda] activations (lda >= K, lda % 8 == 0, 16-byte
 *              aligned), read-only;
 *   W_q_dev, s_w_dev, Y_dev, ldy, variant, split_k, config_id, workspace,
 *   ws_bytes, debug_acc_dev   as qg_gemm_w8a8;
 *   A_q_dev, s_a_dev  [M][K] codes and the scales (layouts of qg_quant_act).
 * Errors are those of qg_quant_act and qg_gemm_w8a8. */
QG_API int qg_linear_w8a8(int fmt, int64_t M, int64_t N, int64_t K, const void* A_dev, int64_t lda,
                          const void* W_q_dev, const float* s_w_dev, void* Y_dev, int64_t ldy, int variant,
                          int split_k, int config_id, void* workspace_dev, size_t ws_bytes, void* A_q_dev,
                          float* s_a_dev, int32_t* debug_acc_dev, void* stream);

/* Allocation-free form of qg_gemm_w8a8 (the pages have no counterpart; this
 * is a convenience of this library).  It is for callers that cannot call
 * cudaMalloc at all: code running inside a host framework or serving runtime
 * that owns the device allocator and forbids outside allocations, plugins
 * that receive only input and output buffers, or latency-critical paths that
 * must never enter the allocator.  Such callers cannot provide the Split-K
 * workspace that qg_gemm_w8a8 needs, so this entry point keeps the Split-K
 * partials and tile counters in one static device array of
 * QG_NOALLOC_SCRATCH_BYTES (4 MiB) inside the library; every GPU that loads
 * the library holds that array until the process exits.
 *   Arguments: as qg_gemm_w8a8 without workspace_dev / ws_bytes.
 *   Limit: a shape whose scratch (qg_workspace_bytes_config) exceeds
 *   QG_NOALLOC_SCRATCH_BYTES is rejected with QG_ERR_WORKSPACE_TOO_SMALL;
 *   use fewer splits, or qg_gemm_w8a8 with a caller workspace.
 *   Set-up: the first call in each CUDA context (normally once per device,
 *   in its primary context) looks up the array's device address with the
 *   caller's device current (cudaGetSymbolAddress) and keeps it for that
 *   context; make that first call before any stream capture, and again
 *   after a cudaDeviceReset (the new context has the array at another
 *   address).  It never calls cudaMalloc / cudaFree.
 *   Sharing: every call uses the same array, which keeps the last call's
 *   contents; each call clears the tile counters (cudaMemsetAsync on
 *   `stream`) before its kernel.  Calls whose kernels overlap on the GPU
 *   (other streams, concurrent graph launches) race on the array and give
 *   wrong results: serialize them. */
#define QG_NOALLOC_SCRATCH_BYTES (4u << 20)
QG_API int qg_gemm_w8a8_noalloc(int fmt, int64_t M, int64_t N, int64_t K, const void* A_q_dev, const float* s_a_dev,
                                const void* W_q_dev, const float* s_w_dev, void* Y_dev, int64_t ldy, int variant,
                                int split_k, int config_id, int32_t* debug_acc_dev, void* stream);

/* Per-shape config lookup ("Per-shape Config Tuning"): the row of the loaded
 * table for (fmt, N, K) and the smallest tuned token count >= M.  M larger
 * than every tuned count ("Hybrid Dispatch": beyond the tuned range) and,
 * when allowed, shapes missing from the table get the built-in default
 * config.  Returns QG_ERR_NO_CONFIG for a missing shape otherwise. */
QG_API int qg_select(int fmt, int64_t M, int64_t N, int64_t K, int* variant, int* split_k, int* config_id);

/* Load a tuned table (tab-separated "fmt N K M variant split_k config_id"
 * rows, '#' comments), replacing the current one.  NULL reads $QG_TABLE.
 * A row that does not parse, or whose configuration qg_check_config rejects
 * at the row's M, fails the load with QG_ERR_TABLE_PARSE (the current table
 * is kept).
 *
 * The table and the settings below (default configs, launch flags, wait
 * limit, forced timeout) are process-wide: any thread may change them, and a
 * change applies to the calls that start after it. */
QG_API int qg_load_table(const char* path);

/* Allow (1) or forbid (0, the initial state) qg_select's built-in default
 * config for shapes missing from the table. */
QG_API int qg_set_allow_default(int allow);

/* Launch flags: QG_LAUNCH_PDL enables programmatic dependent launch, so a
 * GEMM starts streaming its (static) weights while the previous kernel in
 * the stream finishes; W_q / s_w must then not be written by the kernels
 * directly preceding the GEMM in that stream. */
#define QG_LAUNCH_PDL 1
/* QG_LAUNCH_FUSED_QUANT makes qg_linear_w8a8 take its one-kernel form
 * (quantization fused into the GEMM) whenever the format and variant have
 * one, even when A_q / s_a buffers are given. */
#define QG_LAUNCH_FUSED_QUANT 2
QG_API int qg_set_launch_flags(int flags);

/* Bound, in nanoseconds, of every pipeline wait inside the kernels (default
 * 2e9).  0 restores the default. */
QG_API int qg_set_wait_limit_ns(uint64_t ns);

/* Test hook: when nonzero, the next GEMM launches make their MMA thread wait
 * on a barrier that nothing arrives on, so the bounded wait runs out and the
 * kernel reports QG_ERR_DEVICE_TIMEOUT instead of computing. */
QG_API int qg_set_force_timeout(int on);

/* Synchronize the current device, then read and clear its status word:
 * *code = 0 or the first qg_status a kernel reported.  After a reported
 * QG_ERR_DEVICE_TIMEOUT the Y of the launches since the last check is
 * unspecified, and a Split-K workspace they used may hold stale arrival
 * counters: run qg_workspace_init on it before its next use
 * (qg_gemm_w8a8_noalloc clears its own counters on every call). */
QG_API int qg_device_error(int* code);

/* Launch timing inside a stream or a captured graph, where timing events
 * would sit between kernels and break programmatic dependent launch.  While
 * a log is set, every kernel launch of qg_quant_act, qg_gemm_w8a8 and the
 * entry points built on them takes the next slot pair of the log, in launch
 * order: log_dev[2*i] receives the earliest CTA start and log_dev[2*i + 1]
 * the latest CTA end of launch i, in %globaltimer nanoseconds (atomicMin /
 * atomicMax: the caller fills the start slots with UINT64_MAX and the end
 * slots with 0 before the launches run, e.g. before every graph replay).
 * Launches beyond `slots` pairs, and every launch while no log is set, are
 * not timed and cost nothing extra.  A graph captured while the log is set
 * keeps writing its slots on every replay.
 *   log_dev  device array of 2 * slots uint64, owned by the caller, or NULL
 *            to turn the log off;  slots >= 0.
 * Setting a log (or NULL) restarts the slot count at 0.  The log is
 * process-wide, like the settings above.  Errors: QG_ERR_INVALID_ARG for
 * slots < 0 or an unaligned log. */
QG_API int qg_set_timing_log(uint64_t* log_dev, int slots);

/* Slot pairs handed out since the last qg_set_timing_log (may exceed the
 * log's capacity: the launches past it were not timed). */
QG_API int qg_timing_log_count(void);

/* Thread-local description of the last failure (never NULL). */
QG_API const char* qg_last_error(void);

/* Library version string. */
QG_API const char* qg_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QGEMM_H */
