// qgemm.cu -- C ABI of the quantized decode GEMM (see include/qgemm.h):
// argument validation, TMA tensor-map encoding, variant dispatch, the tuned
// config table and error reporting.  All arithmetic runs in the kernels of
// quant.cuh, gemm_f8.cuh, gemm_i8.cuh and gemm_i8_dp4a.cuh.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_fp8.h>

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/qgemm.h"
#include "common.cuh"
#include "gemm_f8.cuh"
#include "gemm_i8.cuh"
#include "gemm_i8_dp4a.cuh"
#include "gemm_i8_mma.cuh"
#include "gemm_f8_persist.cuh"
#include "quant.cuh"

namespace {

thread_local std::string g_err = "";

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(QG_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Process-wide settings: any thread may change them, and a change applies to
// the calls that start after it (a call running meanwhile may see either).
std::mutex g_mu;  // guards the table and g_allow_default
std::atomic<int> g_launch_flags{0};
std::atomic<uint64_t> g_wait_ns{2000000000ull};
std::atomic<int> g_force_timeout{0};
bool g_allow_default = false;
// launch timing log (qg_set_timing_log): slot pairs handed out in launch order
std::atomic<unsigned long long*> g_ts_log{nullptr};
std::atomic<int> g_ts_cap{0};
std::atomic<int> g_ts_next{0};

unsigned long long* next_ts_slot() {
  unsigned long long* log = g_ts_log.load(std::memory_order_relaxed);
  if (!log) return nullptr;
  const int i = g_ts_next.fetch_add(1, std::memory_order_relaxed);
  return i < g_ts_cap.load(std::memory_order_relaxed) ? log + 2 * static_cast<int64_t>(i) : nullptr;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

// ------------------------------------------------------------ tensor maps
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2-D uint8 tensor map over rows x K bytes (row pitch `pitch` bytes), box of
// 128 bytes x box_rows rows, 128-byte swizzle; rows past the end read zero.
int make_map(CUtensorMap* tm, const void* base, int64_t rows, int64_t K, int64_t pitch, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(QG_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(pitch)};
  cuuint32_t box[2] = {128u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(QG_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
  return QG_OK;
}

// 2-D fp16 tensor map over rows x K elements (dense rows), box of 64
// elements (128 bytes) x box_rows rows, 128-byte swizzle: one MMA operand
// swizzle atom of 64 K; rows past the end read zero.
int make_map_f16(CUtensorMap* tm, const void* base, int64_t rows, int64_t K, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(QG_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(K * 2)};
  cuuint32_t box[2] = {64u, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  CUresult r = fn(tm, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(QG_ERR_CUDA, "cuTensorMapEncodeTiled (fp16) failed (%d)", static_cast<int>(r));
  return QG_OK;
}

// -------------------------------------------------------------- launching
struct DevInfo {
  int sms = 0;
  size_t smem_optin = 0;     // largest dynamic shared memory one CTA may opt into
  size_t smem_per_sm = 0;    // shared memory of one SM
  size_t smem_reserved = 0;  // shared memory the system reserves per CTA
};
// Properties of the current device, queried once per device (thread-safe).
DevInfo dev_info() {
  static DevInfo cache[64];
  static std::once_flag once[64];
  int d = 0;
  cudaGetDevice(&d);
  if (d < 0 || d >= 64) d = 0;
  std::call_once(once[d], [d] {
    cudaDeviceProp p;
    DevInfo& c = cache[d];
    if (cudaGetDeviceProperties(&p, d) == cudaSuccess) {
      c.sms = p.multiProcessorCount;
      c.smem_optin = p.sharedMemPerBlockOptin;
      c.smem_per_sm = p.sharedMemPerMultiprocessor;
      c.smem_reserved = p.reservedSharedMemPerBlock;
    } else {  // no device to ask (host-only callers): B300's figures
      c.sms = 148;
      c.smem_optin = 232448;
      c.smem_per_sm = 233472;
      c.smem_reserved = 1024;
    }
  });
  return cache[d];
}

// Dynamic shared memory one CTA may use so that two CTAs share an SM.
size_t two_per_sm_smem() {
  const DevInfo d = dev_info();
  return (d.smem_per_sm - 2 * d.smem_reserved) / 2;
}

// Launch with the library's launch flags; cluster_y > 1 groups that many
// consecutive blockIdx.y into one thread-block cluster (cluster_x likewise
// along x).
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster_xy(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              unsigned cluster_x, unsigned cluster_y, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  int n = 0;
  if (g_launch_flags.load(std::memory_order_relaxed) & QG_LAUNCH_PDL) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1 || cluster_y > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = cluster_x;
    attr[n].val.clusterDim.y = cluster_y;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                           unsigned cluster_y, Args&&... args) {
  return launch_cluster_xy(kernel, grid, block, smem, stream, 1u, cluster_y, std::forward<Args>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                   Args&&... args) {
  return launch_cluster(kernel, grid, block, smem, stream, 1u, std::forward<Args>(args)...);
}

template <typename K>
cudaError_t set_smem(K kernel, size_t bytes) {
  return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(bytes));
}

// ------------------------------------------------------------ GEMM shapes
constexpr int kMaxStages = 16;

struct Plan {
  int groups = 1;      // grouped launches: grid z
  bool swap = false;
  bool dp4a = false;   // W8A8_INT8 Swap-AB on the CUDA cores (M <= 8)
  bool mma = false;    // W8A8_INT8 Swap-AB on mma.sync (QG_CONFIG_MMA_SYNC)
  bool persist = false;  // FP8_Dynamic Standard as the persistent pair kernel (QG_CONFIG_PERSIST)
  int persist_rows = 256;  // its weight rows per tile (QG_CONFIG_PERSIST_ROWS_MASK)
  bool prew = false;     // W8A8_INT8 Swap-AB on activations widened once per launch (QG_CONFIG_I8_PREWIDEN)
  int64_t prew_bytes = 0;  // their fp16 copy in the workspace (after the Split-K part)
  int mpad = 0;        // swap: MMA N (tokens padded), 16 / 32 / 64 (mma.sync: 8 / 16 / 24 / 32)
  int ctr_tiles = 0;   // Split-K arrival counters of one group: enough for every kernel's token blocks
  int n_tiles = 0, m_tiles = 0, kt = 0, splits = 1;
  int reduce = qg::kReduceNone;  // how split partials are summed
};

int64_t ws_counter_bytes(int64_t tiles) { return cdiv(tiles * 4, 256) * 256; }

int make_plan(int fmt, int64_t M, int64_t N, int64_t K, int variant, int split_k, int config_id, Plan* p) {
  p->dp4a = (variant == QG_SWAPAB_DP4A || variant == QG_SWAPAB_DP4A_SPLITK);
  p->swap = (variant == QG_SWAPAB || variant == QG_SWAPAB_SPLITK) || p->dp4a;
  p->mma = (config_id & QG_CONFIG_MMA_SYNC) != 0;
  p->persist = (config_id & QG_CONFIG_PERSIST) != 0;
  p->persist_rows = 256 - 32 * ((config_id & QG_CONFIG_PERSIST_ROWS_MASK) >> QG_CONFIG_PERSIST_ROWS_SHIFT);
  p->prew = (config_id & QG_CONFIG_I8_PREWIDEN) != 0;
  if (p->prew && (fmt != QG_W8A8_INT8 || !(variant == QG_SWAPAB || variant == QG_SWAPAB_SPLITK) || p->mma))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_I8_PREWIDEN is for W8A8_INT8 with QG_SWAPAB / QG_SWAPAB_SPLITK");
  if (p->persist && (fmt != QG_FP8_DYNAMIC || variant != QG_STANDARD))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_PERSIST is for FP8_Dynamic with QG_STANDARD");
  if (p->dp4a && (fmt != QG_W8A8_INT8 || M > qg::kDpMaxTokens))
    return fail(QG_ERR_UNSUPPORTED_SHAPE, "the dp4a variants take W8A8_INT8 with M <= %d", qg::kDpMaxTokens);
  if (p->mma && (fmt != QG_W8A8_INT8 || !p->swap || p->dp4a))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_MMA_SYNC is for W8A8_INT8 with QG_SWAPAB / QG_SWAPAB_SPLITK");
  if ((config_id & QG_CONFIG_MMA_DP4A_MASK) && M > 16)
    return fail(QG_ERR_UNSUPPORTED_SHAPE, "QG_CONFIG_MMA_DP4A takes at most 16 tokens");
  p->kt = static_cast<int>(cdiv(K, 128));
  p->n_tiles = static_cast<int>(cdiv(N, 128));
  // counters for blocks of 16 tokens cover every kernel's token blocking
  // (16 / 32 / 64, mma.sync 8..32, Standard 128), so qg_workspace_bytes needs
  // no config_id
  const int64_t ctr = cdiv(N, 128) * cdiv(M, 16);
  if (ctr > 0x7FFFFFFF) return fail(QG_ERR_UNSUPPORTED_SHAPE, "too many output tiles");
  p->ctr_tiles = static_cast<int>(ctr);
  if (p->mma) {
    // token groups of 8 on the MMA N side; more than 32 tokens run as blocks of 32
    p->mpad = M <= 8 ? 8 : (M <= 16 ? 16 : (M <= 24 ? 24 : 32));
    p->m_tiles = static_cast<int>(cdiv(M, p->mpad));
    if (p->m_tiles > 65535) return fail(QG_ERR_UNSUPPORTED_SHAPE, "M too large");
  } else if (p->prew) {
    // tokens padded to 16 / 32 / 64, blocks of 128 above 64 tokens
    p->mpad = M <= 16 ? 16 : (M <= 32 ? 32 : (M <= 64 ? 64 : 128));
    p->m_tiles = static_cast<int>(cdiv(M, p->mpad));
    if (p->m_tiles > 65535) return fail(QG_ERR_UNSUPPORTED_SHAPE, "M too large");
  } else if (p->swap) {
    // tokens padded to the MMA N side; more than 64 tokens run as blocks of 64
    p->mpad = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    p->m_tiles = static_cast<int>(cdiv(M, p->mpad));
    if (p->m_tiles > 65535) return fail(QG_ERR_UNSUPPORTED_SHAPE, "M too large");
  } else if (p->persist) {
    // pair tiles of 256 tokens x persist_rows weight rows
    p->m_tiles = static_cast<int>(cdiv(M, 256));
    p->n_tiles = static_cast<int>(cdiv(N, p->persist_rows));
    if (static_cast<int64_t>(p->m_tiles) * p->n_tiles > 0x7FFFFFFF) return fail(QG_ERR_UNSUPPORTED_SHAPE, "M too large");
  } else {
    p->m_tiles = static_cast<int>(cdiv(M, 128));
    if (p->m_tiles > 65535) return fail(QG_ERR_UNSUPPORTED_SHAPE, "M too large");
  }
  if (static_cast<int64_t>(p->n_tiles) * p->m_tiles > 0x7FFFFFFF)
    return fail(QG_ERR_UNSUPPORTED_SHAPE, "too many output tiles");
  const bool split_variant = (variant == QG_SPLITK || variant == QG_SWAPAB_SPLITK || variant == QG_SWAPAB_DP4A_SPLITK);
  if (split_k < 1 || split_k > p->kt)
    return fail(QG_ERR_UNSUPPORTED_SHAPE, "split_k=%d outside [1, ceil(K/128)=%d]", split_k, p->kt);
  if (!split_variant && split_k != 1)
    return fail(QG_ERR_INVALID_ARG, "split_k=%d needs a *_SPLITK variant", split_k);
  if (split_k > 65535) return fail(QG_ERR_UNSUPPORTED_SHAPE, "split_k too large");
  if (fmt == QG_W8A8_INT8 && !p->swap)
    return fail(QG_ERR_UNSUPPORTED_SHAPE, "W8A8_INT8 runs the Swap-AB variants");
  p->splits = split_k;
  // Swap-AB splits of one tile reduce inside a thread-block cluster (no
  // workspace) when there are at most 16 of them; otherwise through the
  // caller workspace.
  p->reduce = split_k == 1 ? qg::kReduceNone
              : (p->swap && split_k <= qg::kMaxClusterSplits) ? qg::kReduceCluster
                                                              : qg::kReduceGlobal;
  return QG_OK;
}

// rows: the token rows of A_q / Y (all groups' tokens for grouped launches).
// The counters are those of 128-row tiles (see gemm_entry).
// PREW adds the fp16 copy of the activations (rows x K), 256-byte aligned,
// after the Split-K part.
int64_t split_workspace_bytes(const Plan& p, int64_t rows, int64_t N) {
  if (p.reduce != qg::kReduceGlobal) return 0;
  return ws_counter_bytes(static_cast<int64_t>(p.groups) * p.ctr_tiles) + static_cast<int64_t>(p.splits) * rows * N * 4;
}
int64_t prew_offset(const Plan& p, int64_t rows, int64_t N) { return cdiv(split_workspace_bytes(p, rows, N), 256) * 256; }
int64_t workspace_bytes(const Plan& p, int64_t rows, int64_t N, int64_t K) {
  return p.prew ? prew_offset(p, rows, N) + cdiv(rows * K * 2, 256) * 256 : split_workspace_bytes(p, rows, N);
}

// config_id = ring | distance << 5 (see qgemm.h).  Ring depth: ring > 0
// asks for that many stages (capped by the opt-in limit); 0 takes the
// deepest ring that still lets two CTAs share an SM.
template <typename SmemFn>
int pick_stages(int config_id, SmemFn smem_bytes, int* stages) {
  config_id &= QG_CONFIG_RING_MASK;
  const size_t optin = dev_info().smem_optin, two = two_per_sm_smem();
  int max_stages = kMaxStages;
  while (max_stages > 2 && smem_bytes(max_stages) > optin) --max_stages;
  int def = max_stages;
  while (def > 2 && smem_bytes(def) > two) --def;
  int st = config_id > 0 ? config_id : def;
  if (st > max_stages) st = max_stages;
  if (st < 2) return fail(QG_ERR_INVALID_ARG, "config_id (stages) must be >= 2");
  *stages = st;
  return QG_OK;
}

template <typename Kernel>
int launch_gemm(Kernel kernel, const Plan& p, dim3 grid, unsigned threads, size_t smem, const CUtensorMap& tmW,
                const CUtensorMap& tmA, qg::GemmArgs& g, cudaStream_t stream) {
  cudaError_t e = set_smem(kernel, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  unsigned cluster_y = 1;
  if (p.reduce == qg::kReduceCluster) {
    cluster_y = static_cast<unsigned>(p.splits);
    if (cluster_y > 8) {
      e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute(non-portable cluster)");
    }
  }
  g.reduce = p.reduce;
  e = launch_cluster(kernel, grid, dim3(threads), smem, stream, cluster_y, tmW, tmA, g);
  if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
  return QG_OK;
}

template <int FMT, int MPAD, bool FUSED, int PW = 4>
int run_f8_swap(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
                cudaStream_t stream) {
  const int rb = g.recv_bytes;
  int rc = pick_stages(config_id, [rb](int st) { return qg::gemm_f8_smem_bytes<true, MPAD>(st, rb); }, &g.stages);
  if (rc != QG_OK) return rc;
  // Block_FP8 fused: the scale ring holds stages + 4 k-tiles
  if (FMT == qg::kFmtBlock && FUSED && g.stages > qg::kMaxStagesBlockFused) g.stages = qg::kMaxStagesBlockFused;
  return launch_gemm(qg::gemm_f8_swap_kernel<FMT, MPAD, FUSED, PW>, p,
                     dim3(p.n_tiles * p.m_tiles, p.splits, p.groups), qg::swap_threads(FMT, FUSED, PW),
                     qg::gemm_f8_smem_bytes<true, MPAD>(g.stages, rb), tmW, tmA, g, stream);
}

template <int FMT, int BNW>
int run_f8_std(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
               cudaStream_t stream) {
  // Block_FP8's four partial buffers take all the TMEM (one CTA per SM):
  // the deepest ring that fits by default
  if (FMT == qg::kFmtBlock && (config_id & QG_CONFIG_RING_MASK) == 0) config_id |= kMaxStages;
  int rc = pick_stages(config_id, [](int st) { return qg::gemm_f8_std_smem_bytes<BNW>(st); }, &g.stages);
  if (rc != QG_OK) return rc;
  return launch_gemm(qg::gemm_f8_std_kernel<FMT, BNW>, p, dim3(p.n_tiles * p.m_tiles, p.splits, p.groups),
                     qg::std_threads(FMT), qg::gemm_f8_std_smem_bytes<BNW>(g.stages), tmW, tmA, g, stream);
}

template <int MPAD>
int run_f8_swap_fmt(int fmt, bool fused, const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA,
                    qg::GemmArgs& g, int config_id, cudaStream_t stream) {
  if (fmt == QG_FP8_DYNAMIC) {
    if (fused) return run_f8_swap<qg::kFmtFP8, MPAD, true>(p, tmW, tmA, g, config_id, stream);
    return run_f8_swap<qg::kFmtFP8, MPAD, false>(p, tmW, tmA, g, config_id, stream);
  }
  if (fused) return run_f8_swap<qg::kFmtBlock, MPAD, true>(p, tmW, tmA, g, config_id, stream);
  // QG_CONFIG_BLOCK_PROMO8: eight promotion warps
  if (config_id & QG_CONFIG_BLOCK_PROMO8) return run_f8_swap<qg::kFmtBlock, MPAD, false, 8>(p, tmW, tmA, g, config_id, stream);
  return run_f8_swap<qg::kFmtBlock, MPAD, false>(p, tmW, tmA, g, config_id, stream);
}

template <int MPAD, bool FUSED, bool PREW = false, int CW = qg::kI8ConvWarps>
int run_i8(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
           cudaStream_t stream) {
  const int rb = g.recv_bytes;
  // the forms that run one CTA per SM take the deepest ring that fits by default
  if (qg::i8_one_per_sm(MPAD, PREW, CW) && (config_id & QG_CONFIG_RING_MASK) == 0) config_id |= kMaxStages;
  int rc = pick_stages(config_id, [rb](int st) { return qg::gemm_i8_smem_bytes<MPAD, PREW>(st, rb); }, &g.stages);
  if (rc != QG_OK) return rc;
  return launch_gemm(qg::gemm_i8_kernel<MPAD, FUSED, PREW, CW>, p, dim3(p.n_tiles * p.m_tiles, p.splits, p.groups),
                     qg::i8_threads(PREW, CW), qg::gemm_i8_smem_bytes<MPAD, PREW>(g.stages, rb), tmW, tmA, g, stream);
}

template <int NG, int TPW, int DPW, bool S8 = false>
int run_i8_mma_t(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
                 cudaStream_t stream) {
  const int rb = g.recv_bytes;
  int rc = pick_stages(config_id, [rb](int st) { return qg::gemm_i8_mma_smem_bytes<NG>(st, rb); }, &g.stages);
  if (rc != QG_OK) return rc;
  return launch_gemm(qg::gemm_i8_mma_kernel<NG, TPW, DPW, S8>, p, dim3(p.n_tiles * p.m_tiles, p.splits, p.groups),
                     qg::ms_threads(TPW), qg::gemm_i8_mma_smem_bytes<NG>(g.stages, rb), tmW, tmA, g, stream);
}
// QG_CONFIG_MMA_NARROW: eight MMA warps of 16 weight rows instead of four of
// 32; with it, QG_CONFIG_MMA_DP4A rows of 16 go to dp4a warps (up to 16
// tokens); QG_CONFIG_MMA_S8: the int8 form of the instruction (no widening)
template <int NG, bool S8>
int run_i8_mma_form(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
                    cudaStream_t stream) {
  if (!(config_id & QG_CONFIG_MMA_NARROW)) return run_i8_mma_t<NG, 2, 0, S8>(p, tmW, tmA, g, config_id, stream);
  if constexpr (NG <= 2) {
    switch ((config_id & QG_CONFIG_MMA_DP4A_MASK) >> QG_CONFIG_MMA_DP4A_SHIFT) {
      case 1: return run_i8_mma_t<NG, 1, 1, S8>(p, tmW, tmA, g, config_id, stream);
      case 2: return run_i8_mma_t<NG, 1, 2, S8>(p, tmW, tmA, g, config_id, stream);
      case 3: return run_i8_mma_t<NG, 1, 3, S8>(p, tmW, tmA, g, config_id, stream);
      case 4: return run_i8_mma_t<NG, 1, 4, S8>(p, tmW, tmA, g, config_id, stream);
      default: break;
    }
  }
  return run_i8_mma_t<NG, 1, 0, S8>(p, tmW, tmA, g, config_id, stream);
}
template <int NG>
int run_i8_mma(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
               cudaStream_t stream) {
  if (config_id & QG_CONFIG_MMA_S8) return run_i8_mma_form<NG, true>(p, tmW, tmA, g, config_id, stream);
  return run_i8_mma_form<NG, false>(p, tmW, tmA, g, config_id, stream);
}

// Persistent pair kernel: one CTA per SM at most (two per cluster); the
// ring takes the deepest depth that fits one CTA's shared memory unless
// config_id asks for fewer stages.  PAIR: the cta_group::2 form
// (QG_CONFIG_PAIR_MMA).
template <bool PAIR, int RW>
int run_f8_persist_t(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
                     cudaStream_t stream) {
  const DevInfo d = dev_info();
  int st = 8;
  while (st > 2 && qg::gemm_f8_persist_smem_bytes<PAIR, RW>(st) > d.smem_optin) --st;
  const int want = config_id & QG_CONFIG_RING_MASK;
  if (want >= 2 && want < st) st = want;
  g.stages = st;
  const size_t smem = qg::gemm_f8_persist_smem_bytes<PAIR, RW>(st);
  cudaError_t e = set_smem(qg::gemm_f8_persist_kernel<PAIR, RW>, smem);
  if (e != cudaSuccess) return cuda_fail(e, "cudaFuncSetAttribute");
  const int64_t tiles = static_cast<int64_t>(p.m_tiles) * p.n_tiles;
  // the tile schedule is static, so only clusters that can all be resident
  // at once are launched (a cluster placed later would finish its share late)
  int resident = 0;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2);
    cfg.blockDim = dim3(qg::kThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&resident, qg::gemm_f8_persist_kernel<PAIR, RW>, &cfg) != cudaSuccess) {
      cudaGetLastError();  // clear the query's error; fall back to one pair per two SMs
      resident = 0;
    }
  }
  const int sms = d.sms > 0 ? d.sms : 148;
  if (resident <= 0 || resident > sms / 2) resident = sms / 2;
  const int clusters = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(tiles, resident)));
  g.reduce = qg::kReduceNone;
  e = launch_cluster_xy(qg::gemm_f8_persist_kernel<PAIR, RW>, dim3(2 * clusters), dim3(qg::kThreads), smem, stream, 2u,
                        1u, tmW, tmA, g);
  if (e != cudaSuccess) return cuda_fail(e, "gemm launch");
  return QG_OK;
}
template <int RW>
int run_f8_persist_rw(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
                      cudaStream_t stream) {
  return (config_id & QG_CONFIG_PAIR_MMA) ? run_f8_persist_t<true, RW>(p, tmW, tmA, g, config_id, stream)
                                          : run_f8_persist_t<false, RW>(p, tmW, tmA, g, config_id, stream);
}
int run_f8_persist(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
                   cudaStream_t stream) {
  switch (p.persist_rows) {
    case 224: return run_f8_persist_rw<224>(p, tmW, tmA, g, config_id, stream);
    case 192: return run_f8_persist_rw<192>(p, tmW, tmA, g, config_id, stream);
    case 160: return run_f8_persist_rw<160>(p, tmW, tmA, g, config_id, stream);
    default: return run_f8_persist_rw<256>(p, tmW, tmA, g, config_id, stream);
  }
}

template <int MT>
int run_dp4a(const Plan& p, const CUtensorMap& tmW, const CUtensorMap& tmA, qg::GemmArgs& g, int config_id,
             cudaStream_t stream) {
  const int rb = g.recv_bytes;
  int rc = pick_stages(config_id, [rb](int st) { return qg::gemm_dp4a_smem_bytes(st, rb); }, &g.stages);
  if (rc != QG_OK) return rc;
  return launch_gemm(qg::gemm_i8_dp4a_kernel<MT>, p, dim3(p.n_tiles, p.splits, p.groups), qg::kDpThreads,
                     qg::gemm_dp4a_smem_bytes(g.stages, rb), tmW, tmA, g, stream);
}

// The config_id checks of qg_gemm_w8a8: known bits, ring depth, prefetch
// distance, and wide tiles only for the FP8_Dynamic Standard / Split-K forms.
int check_config_bits(int fmt, int variant, int config_id) {
  if (config_id < 0 ||
      (config_id & ~(QG_CONFIG_WIDE | QG_CONFIG_MMA_SYNC | QG_CONFIG_MMA_NARROW | QG_CONFIG_FUSED_QUANT |
                     QG_CONFIG_PERSIST | QG_CONFIG_MMA_DP4A_MASK | QG_CONFIG_MMA_S8 | QG_CONFIG_PAIR_MMA |
                     QG_CONFIG_I8_PREWIDEN | QG_CONFIG_I8_CONV16 | QG_CONFIG_BLOCK_PROMO8 |
                     QG_CONFIG_PERSIST_ROWS_MASK | QG_CONFIG_RING_MASK | QG_CONFIG_PREFETCH_MASK)) ||
      (config_id & QG_CONFIG_RING_MASK) > kMaxStages ||
      ((config_id & QG_CONFIG_PREFETCH_MASK) >> QG_CONFIG_PREFETCH_SHIFT) > QG_CONFIG_MAX_PREFETCH)
    return fail(QG_ERR_INVALID_ARG, "config_id %d: unknown bits, ring depth above %d or prefetch distance above %d",
                config_id, kMaxStages, QG_CONFIG_MAX_PREFETCH);
  if ((config_id & QG_CONFIG_WIDE) && (fmt != QG_FP8_DYNAMIC || !(variant == QG_STANDARD || variant == QG_SPLITK)))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_WIDE is for the FP8_Dynamic Standard / Split-K variants");
  if ((config_id & QG_CONFIG_MMA_SYNC) && (fmt != QG_W8A8_INT8 || !(variant == QG_SWAPAB || variant == QG_SWAPAB_SPLITK)))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_MMA_SYNC is for W8A8_INT8 with QG_SWAPAB / QG_SWAPAB_SPLITK");
  if ((config_id & QG_CONFIG_MMA_NARROW) && !(config_id & QG_CONFIG_MMA_SYNC))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_MMA_NARROW needs QG_CONFIG_MMA_SYNC");
  if ((config_id & QG_CONFIG_MMA_DP4A_MASK) &&
      (!(config_id & QG_CONFIG_MMA_NARROW) || ((config_id & QG_CONFIG_MMA_DP4A_MASK) >> QG_CONFIG_MMA_DP4A_SHIFT) > 4))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_MMA_DP4A needs QG_CONFIG_MMA_NARROW and at most 4 groups of 16 rows");
  if ((config_id & QG_CONFIG_MMA_S8) && !(config_id & QG_CONFIG_MMA_SYNC))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_MMA_S8 needs QG_CONFIG_MMA_SYNC");
  if ((config_id & QG_CONFIG_I8_PREWIDEN) &&
      (fmt != QG_W8A8_INT8 || !(variant == QG_SWAPAB || variant == QG_SWAPAB_SPLITK) ||
       (config_id & (QG_CONFIG_MMA_SYNC | QG_CONFIG_FUSED_QUANT | QG_CONFIG_WIDE | QG_CONFIG_PERSIST))))
    return fail(QG_ERR_INVALID_ARG,
                "QG_CONFIG_I8_PREWIDEN is for W8A8_INT8 with QG_SWAPAB / QG_SWAPAB_SPLITK on the tcgen05 kernel");
  if ((config_id & QG_CONFIG_I8_CONV16) &&
      (fmt != QG_W8A8_INT8 || !(variant == QG_SWAPAB || variant == QG_SWAPAB_SPLITK) ||
       (config_id & (QG_CONFIG_MMA_SYNC | QG_CONFIG_FUSED_QUANT | QG_CONFIG_WIDE | QG_CONFIG_PERSIST))))
    return fail(QG_ERR_INVALID_ARG,
                "QG_CONFIG_I8_CONV16 is for W8A8_INT8 with QG_SWAPAB / QG_SWAPAB_SPLITK on the tcgen05 kernel");
  if ((config_id & QG_CONFIG_BLOCK_PROMO8) &&
      (fmt != QG_BLOCK_FP8 || !(variant == QG_SWAPAB || variant == QG_SWAPAB_SPLITK) ||
       (config_id & (QG_CONFIG_FUSED_QUANT | QG_CONFIG_WIDE | QG_CONFIG_PERSIST | QG_CONFIG_MMA_SYNC))))
    return fail(QG_ERR_INVALID_ARG,
                "QG_CONFIG_BLOCK_PROMO8 is for Block_FP8 with QG_SWAPAB / QG_SWAPAB_SPLITK, two-kernel form");
  if ((config_id & QG_CONFIG_PAIR_MMA) && !(config_id & QG_CONFIG_PERSIST))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_PAIR_MMA is a form of the QG_CONFIG_PERSIST kernel");
  if ((config_id & QG_CONFIG_PERSIST_ROWS_MASK) && !(config_id & QG_CONFIG_PERSIST))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_PERSIST_ROWS_MASK is a field of the QG_CONFIG_PERSIST kernel");
  if ((config_id & QG_CONFIG_PERSIST) &&
      (fmt != QG_FP8_DYNAMIC || variant != QG_STANDARD ||
       (config_id & (QG_CONFIG_WIDE | QG_CONFIG_MMA_SYNC | QG_CONFIG_FUSED_QUANT | QG_CONFIG_MMA_DP4A_MASK |
                     QG_CONFIG_MMA_S8))))
    return fail(QG_ERR_INVALID_ARG,
                "QG_CONFIG_PERSIST is for FP8_Dynamic with QG_STANDARD (ring depth and prefetch distance only)");
  if ((config_id & QG_CONFIG_FUSED_QUANT) &&
      (!(variant == QG_SWAPAB || variant == QG_SWAPAB_SPLITK) || (config_id & QG_CONFIG_MMA_SYNC)))
    return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_FUSED_QUANT is for the Swap-AB variants on the tcgen05 kernels");
  if ((config_id & QG_CONFIG_RING_MASK) == 1) return fail(QG_ERR_INVALID_ARG, "config_id (stages) must be >= 2");
  return QG_OK;
}

// Every check of qg_gemm_w8a8 that needs no pointer: format, variant, sizes,
// config_id, K alignment, and the variant's plan (split_k range, token and
// tile limits, the INT8 and dp4a restrictions).
int check_shape_config(int fmt, int64_t M, int64_t N, int64_t K, int variant, int split_k, int config_id) {
  if (fmt < 0 || fmt > 2) return fail(QG_ERR_INVALID_ARG, "unknown format %d", fmt);
  if (variant < 0 || variant > QG_SWAPAB_DP4A_SPLITK) return fail(QG_ERR_INVALID_ARG, "unknown variant %d", variant);
  if (M < 1 || N <= 0 || K <= 0)
    return fail(QG_ERR_INVALID_ARG, "bad sizes M=%lld N=%lld K=%lld", (long long)M, (long long)N, (long long)K);
  int rc = check_config_bits(fmt, variant, config_id);
  if (rc != QG_OK) return rc;
  if (K % 16) return fail(QG_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a multiple of 16", (long long)K);
  if (fmt == QG_BLOCK_FP8 && K % 128) return fail(QG_ERR_UNSUPPORTED_SHAPE, "Block_FP8 needs K %% 128 == 0");
  if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF) return fail(QG_ERR_UNSUPPORTED_SHAPE, "sizes too large");
  Plan p;
  return make_plan(fmt, M, N, K, variant, split_k, config_id, &p);
}

// ------------------------------------------------------------------ table
struct Key {
  int fmt;
  int64_t n, k;
  int m;
  bool operator<(const Key& o) const { return std::tie(fmt, n, k, m) < std::tie(o.fmt, o.n, o.k, o.m); }
};
struct Row {
  int variant, split_k, config_id;
};
std::map<Key, Row> g_table;
bool g_table_env_checked = false;

// Built-in default config ("a default config for functional testing", section
// "Toward a Practical Adoption Model"): Swap-AB for M <= 32 (always for INT8,
// in blocks of 64 tokens above 64), Standard above; split K so that tiles x
// splits roughly fills the two CTA slots of every SM, with at least two
// 128-wide k-tiles per split and (for Swap-AB) no more splits than one
// cluster reduces.
void default_config(int fmt, int64_t M, int64_t N, int64_t K, int* variant, int* split_k, int* config_id) {
  const int sms = dev_info().sms > 0 ? dev_info().sms : 148;
  const bool swap = (fmt == QG_W8A8_INT8) || (M <= 32);
  const int64_t tiles = cdiv(N, 128) * (swap ? cdiv(M, M <= 16 ? 16 : (M <= 32 ? 32 : 64)) : cdiv(M, 128));
  const int64_t kt = cdiv(K, 128);
  int64_t s = (2 * static_cast<int64_t>(sms)) / std::max<int64_t>(tiles, 1);
  s = std::min<int64_t>(s, kt / 2);
  if (swap) s = std::min<int64_t>(s, qg::kMaxClusterSplits);
  if (s < 1) s = 1;
  *variant = swap ? (s > 1 ? QG_SWAPAB_SPLITK : QG_SWAPAB) : (s > 1 ? QG_SPLITK : QG_STANDARD);
  *split_k = static_cast<int>(s);
  *config_id = 0;
}

int load_table_file(const char* path) {
  FILE* f = fopen(path, "r");
  if (!f) return fail(QG_ERR_TABLE_PARSE, "cannot open table '%s'", path);
  std::map<Key, Row> t;
  char line[512];
  int lineno = 0;
  while (fgets(line, sizeof(line), f)) {
    ++lineno;
    char* hash = strchr(line, '#');
    if (hash) *hash = 0;
    char* s = line;
    while (*s == ' ' || *s == '\t' || *s == '\r' || *s == '\n') ++s;
    if (!*s) continue;
    int fmt, m, variant, split_k, config_id;
    long long n, k;
    if (sscanf(s, "%d %lld %lld %d %d %d %d", &fmt, &n, &k, &m, &variant, &split_k, &config_id) != 7 || fmt < 0 ||
        fmt > 2 || n <= 0 || k <= 0 || m <= 0 || variant < 0 || variant > QG_SWAPAB_DP4A_SPLITK || split_k < 1 || config_id < 0) {
      fclose(f);
      return fail(QG_ERR_TABLE_PARSE, "%s:%d: malformed row", path, lineno);
    }
    // a row must be a configuration the GEMM accepts at its token count (and
    // so at every smaller one qg_select sends to it)
    if (check_shape_config(fmt, m, n, k, variant, split_k, config_id) != QG_OK) {
      const std::string why = g_err;
      fclose(f);
      return fail(QG_ERR_TABLE_PARSE, "%s:%d: invalid configuration: %s", path, lineno, why.c_str());
    }
    t[Key{fmt, n, k, m}] = Row{variant, split_k, config_id};
  }
  fclose(f);
  g_table.swap(t);
  return QG_OK;
}

// Shared body of qg_gemm_w8a8 and qg_linear_w8a8.  With `fused` the kernel
// reads bf16 activations and quantizes them itself (A_q / s_a optional
// outputs); otherwise A_q / s_a are the quantized inputs.
struct FusedIn {
  const void* A;
  int64_t lda;
};
// Grouped launch (qg_gemm_w8a8_grouped): M is then the largest group's
// token count, which sizes the token blocks.
struct GroupIn {
  int groups;
  const int32_t* offsets;
  int64_t total_tokens;
};
int gemm_entry(int fmt, int64_t M, int64_t N, int64_t K, const void* A_q_dev, const float* s_a_dev,
               const void* W_q_dev, const float* s_w_dev, void* Y_dev, int64_t ldy, int variant, int split_k,
               int config_id, void* workspace_dev, size_t ws_bytes, int32_t* debug_acc_dev, void* stream,
               const FusedIn* fused, const GroupIn* grouped = nullptr) {
  if (fmt < 0 || fmt > 2) return fail(QG_ERR_INVALID_ARG, "unknown format %d", fmt);
  if (variant < 0 || variant > QG_SWAPAB_DP4A_SPLITK) return fail(QG_ERR_INVALID_ARG, "unknown variant %d", variant);
  if (M < 0 || N <= 0 || K <= 0 || ldy < N)
    return fail(QG_ERR_INVALID_ARG, "bad sizes M=%lld N=%lld K=%lld ldy=%lld", (long long)M, (long long)N, (long long)K, (long long)ldy);
  const bool wide = (config_id & QG_CONFIG_WIDE) != 0;
  const int crc = check_config_bits(fmt, variant, config_id);
  if (crc != QG_OK) return crc;
  if (M == 0) return QG_OK;
  if ((!fused && (!A_q_dev || !s_a_dev)) || !W_q_dev || !s_w_dev || !Y_dev)
    return fail(QG_ERR_INVALID_ARG, "null pointer");
  if (fused && (!fused->A || fused->lda < K || fused->lda % 8 || !aligned(fused->A, 16)))
    return fail(fused->A ? QG_ERR_ALIGNMENT : QG_ERR_INVALID_ARG,
                "A must be 16-byte aligned bf16 with lda >= K and lda %% 8 == 0");
  if (K % 16) return fail(QG_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a multiple of 16", (long long)K);
  if (fmt == QG_BLOCK_FP8 && K % 128) return fail(QG_ERR_UNSUPPORTED_SHAPE, "Block_FP8 needs K %% 128 == 0");
  if (M > 0x7FFFFFFF || N > 0x7FFFFFFF || K > 0x7FFFFFFF || cdiv(N, 128) > 0x7FFFFFFF)
    return fail(QG_ERR_UNSUPPORTED_SHAPE, "sizes too large");
  if (!aligned(A_q_dev, 16) || !aligned(W_q_dev, 16) || !aligned(s_a_dev, 4) || !aligned(s_w_dev, 4) ||
      !aligned(Y_dev, 2) || (debug_acc_dev && !aligned(debug_acc_dev, 4)))
    return fail(QG_ERR_ALIGNMENT, "A_q/W_q need 16-byte alignment, scales 4, Y 2");
  if (debug_acc_dev && fmt != QG_W8A8_INT8) return fail(QG_ERR_INVALID_ARG, "debug_acc is W8A8_INT8 only");
  // rows of A_q / s_a / Y: M, or all groups' tokens
  const int64_t rows = grouped ? grouped->total_tokens : M;
  if (grouped) {
    if (grouped->groups < 1 || grouped->groups > 65535)
      return fail(QG_ERR_UNSUPPORTED_SHAPE, "groups=%d outside [1, 65535]", grouped->groups);
    if (!grouped->offsets || !aligned(grouped->offsets, 4)) return fail(QG_ERR_INVALID_ARG, "token offsets: null or unaligned");
    if (fused || wide || !(variant == QG_SWAPAB || variant == QG_SWAPAB_SPLITK || variant == QG_SWAPAB_DP4A ||
                           variant == QG_SWAPAB_DP4A_SPLITK))
      return fail(QG_ERR_INVALID_ARG, "grouped launches run the Swap-AB variants");
    if (config_id & (QG_CONFIG_I8_PREWIDEN | QG_CONFIG_I8_CONV16 | QG_CONFIG_BLOCK_PROMO8))
      return fail(QG_ERR_INVALID_ARG,
                  "grouped launches take none of QG_CONFIG_I8_PREWIDEN, QG_CONFIG_I8_CONV16, QG_CONFIG_BLOCK_PROMO8");
    if (rows < 0 || rows > 0x7FFFFFFF || static_cast<int64_t>(grouped->groups) * N > 0x7FFFFFFF)
      return fail(QG_ERR_UNSUPPORTED_SHAPE, "sizes too large");
    if (rows == 0) return QG_OK;
  }
  Plan p;
  int rc = make_plan(fmt, M, N, K, variant, split_k, config_id, &p);
  if (rc != QG_OK) return rc;
  if (grouped) p.groups = grouped->groups;
  if (wide) p.n_tiles = static_cast<int>(cdiv(N, 256));
  const int64_t need = workspace_bytes(p, rows, N, K);
  if (need > 0) {
    if (!workspace_dev) return fail(QG_ERR_WORKSPACE_TOO_SMALL, "split_k=%d needs a %lld-byte workspace", split_k, (long long)need);
    if (static_cast<int64_t>(ws_bytes) < need)
      return fail(QG_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %lld needed", ws_bytes, (long long)need);
    if (!aligned(workspace_dev, 256)) return fail(QG_ERR_ALIGNMENT, "workspace must be 256-byte aligned");
  }
  CUtensorMap tmW, tmA;
  // the persistent kernel loads weight tiles in halves of persist_rows / 2 rows
  const uint32_t w_box = p.persist ? static_cast<uint32_t>(p.persist_rows / 2) : (wide ? 256u : 128u);
  rc = make_map(&tmW, W_q_dev, static_cast<int64_t>(p.groups) * N, K, K, w_box);
  if (rc != QG_OK) return rc;
  if (fused) {
    tmA = tmW;  // unused: the kernel reads the bf16 activations directly
  } else {
    rc = make_map(&tmA, A_q_dev, rows, K, K, p.swap ? static_cast<uint32_t>(p.mpad) : 128u);
    if (rc != QG_OK) return rc;
  }
  // PREW: the GEMM reads the fp16 copy of the activations in the workspace
  uint8_t* a16 = nullptr;
  if (p.prew) {
    if (grouped || fused)
      return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_I8_PREWIDEN takes the quantized activations of one group");
    a16 = static_cast<uint8_t*>(workspace_dev) + prew_offset(p, rows, N);
    rc = make_map_f16(&tmA, a16, rows, K, static_cast<uint32_t>(p.mpad));
    if (rc != QG_OK) return rc;
  }

  qg::GemmArgs g = {};
  g.M = static_cast<int>(rows);
  if (grouped) {
    g.group_offsets = grouped->offsets;
    g.sw_group_stride = fmt == QG_BLOCK_FP8 ? cdiv(N, 128) * p.kt : N;
    g.group_max = static_cast<int>(M);
  }
  g.N = static_cast<int>(N);
  g.K = static_cast<int>(K);
  g.ldy = ldy;
  g.kt_total = p.kt;
  g.splits = p.splits;
  g.m_tiles = p.m_tiles;
  g.s_a = s_a_dev;
  g.s_w = s_w_dev;
  g.Y = static_cast<__nv_bfloat16*>(Y_dev);
  if (p.reduce == qg::kReduceGlobal) {
    // the partials start after the counters of 128-row tiles even for wide
    // tiles, so that no configuration's partials overlap another's counters
    g.ws_count = static_cast<int*>(workspace_dev);
    g.ws_part = static_cast<uint8_t*>(workspace_dev) + ws_counter_bytes(static_cast<int64_t>(p.groups) * p.ctr_tiles);
  }
  g.reduce = p.reduce;
  g.recv_bytes = p.reduce == qg::kReduceCluster
                     ? qg::cluster_recv_bytes(p.splits, static_cast<int>(std::min<int64_t>(M, p.mpad)))
                     : 0;
  g.debug_acc = debug_acc_dev;
  if (fused) {
    g.A = static_cast<const __nv_bfloat16*>(fused->A);
    g.lda = fused->lda;
    g.a_q_out = static_cast<uint8_t*>(const_cast<void*>(A_q_dev));
    g.s_a_out = const_cast<float*>(s_a_dev);
  }
  g.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
  g.force_timeout = g_force_timeout.load(std::memory_order_relaxed);
  g.l2_prefetch = (config_id & QG_CONFIG_PREFETCH_MASK) >> QG_CONFIG_PREFETCH_SHIFT;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  g.tstamp = next_ts_slot();

  const bool fz = fused != nullptr;
  if (p.dp4a) {
    if (fz) return fail(QG_ERR_INVALID_ARG, "the dp4a variants take quantized activations");
    if (M <= 1) return run_dp4a<1>(p, tmW, tmA, g, config_id, s);
    if (M <= 2) return run_dp4a<2>(p, tmW, tmA, g, config_id, s);
    if (M <= 4) return run_dp4a<4>(p, tmW, tmA, g, config_id, s);
    return run_dp4a<8>(p, tmW, tmA, g, config_id, s);
  }
  if (p.persist) {
    if (fz) return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_PERSIST takes quantized activations");
    return run_f8_persist(p, tmW, tmA, g, config_id, s);
  }
  if (p.mma) {
    if (fz) return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_MMA_SYNC takes quantized activations");
    if (p.mpad == 8) return run_i8_mma<1>(p, tmW, tmA, g, config_id, s);
    if (p.mpad == 16) return run_i8_mma<2>(p, tmW, tmA, g, config_id, s);
    if (p.mpad == 24) return run_i8_mma<3>(p, tmW, tmA, g, config_id, s);
    return run_i8_mma<4>(p, tmW, tmA, g, config_id, s);
  }
  if (p.prew) {
    // the activations widened once (no timing slot: its time falls to the GEMM)
    const int64_t n16 = rows * K / 16;
    const int blocks = static_cast<int>(std::max<int64_t>(1, std::min<int64_t>(cdiv(n16, 256), 4 * dev_info().sms)));
    cudaError_t e = launch_cluster_xy(qg::widen_i8_kernel, dim3(blocks), dim3(256), 0, s, 1u, 1u,
                                      static_cast<const uint8_t*>(A_q_dev), reinterpret_cast<uint4*>(a16), n16);
    if (e != cudaSuccess) return cuda_fail(e, "widen launch");
    if (config_id & QG_CONFIG_I8_CONV16) {
      if (p.mpad == 16) return run_i8<16, false, true, 16>(p, tmW, tmA, g, config_id, s);
      if (p.mpad == 32) return run_i8<32, false, true, 16>(p, tmW, tmA, g, config_id, s);
      return p.mpad == 64 ? run_i8<64, false, true, 16>(p, tmW, tmA, g, config_id, s)
                          : run_i8<128, false, true, 16>(p, tmW, tmA, g, config_id, s);
    }
    if (p.mpad == 16) return run_i8<16, false, true>(p, tmW, tmA, g, config_id, s);
    if (p.mpad == 32) return run_i8<32, false, true>(p, tmW, tmA, g, config_id, s);
    return p.mpad == 64 ? run_i8<64, false, true>(p, tmW, tmA, g, config_id, s)
                        : run_i8<128, false, true>(p, tmW, tmA, g, config_id, s);
  }
  if (fmt == QG_W8A8_INT8 && (config_id & QG_CONFIG_I8_CONV16)) {
    if (fz) return fail(QG_ERR_INVALID_ARG, "QG_CONFIG_I8_CONV16 takes quantized activations");
    if (p.mpad == 16) return run_i8<16, false, false, 16>(p, tmW, tmA, g, config_id, s);
    if (p.mpad == 32) return run_i8<32, false, false, 16>(p, tmW, tmA, g, config_id, s);
    return run_i8<64, false, false, 16>(p, tmW, tmA, g, config_id, s);
  }
  if (fmt == QG_W8A8_INT8) {
    if (p.mpad == 16) return fz ? run_i8<16, true>(p, tmW, tmA, g, config_id, s) : run_i8<16, false>(p, tmW, tmA, g, config_id, s);
    if (p.mpad == 32) return fz ? run_i8<32, true>(p, tmW, tmA, g, config_id, s) : run_i8<32, false>(p, tmW, tmA, g, config_id, s);
    return fz ? run_i8<64, true>(p, tmW, tmA, g, config_id, s) : run_i8<64, false>(p, tmW, tmA, g, config_id, s);
  }
  if (p.swap) {
    if (p.mpad == 16) return run_f8_swap_fmt<16>(fmt, fz, p, tmW, tmA, g, config_id, s);
    if (p.mpad == 32) return run_f8_swap_fmt<32>(fmt, fz, p, tmW, tmA, g, config_id, s);
    return run_f8_swap_fmt<64>(fmt, fz, p, tmW, tmA, g, config_id, s);
  }
  if (fmt == QG_FP8_DYNAMIC)
    return wide ? run_f8_std<qg::kFmtFP8, 256>(p, tmW, tmA, g, config_id, s)
                : run_f8_std<qg::kFmtFP8, 128>(p, tmW, tmA, g, config_id, s);
  return run_f8_std<qg::kFmtBlock, 128>(p, tmW, tmA, g, config_id, s);
}

}  // namespace

// Static device scratch of qg_gemm_w8a8_noalloc (Split-K counters and
// partials for callers that cannot allocate).  In host code this name is only
// a host-side stand-in: kernels get the device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[QG_NOALLOC_SCRATCH_BYTES];

namespace {

std::mutex g_noalloc_mu;
// The scratch array's device address belongs to one CUDA context (a reset
// device or a caller's own context loads the library's module again, at
// another address), so the looked-up address is cached per context, keyed on
// the context's process-unique ID (cuCtxGetId), never on the device ordinal.
struct NoallocEntry {
  unsigned long long ctx_id;
  void* addr;
};
std::vector<NoallocEntry> g_noalloc_cache;

using CtxGetCurrentFn = CUresult (*)(CUcontext*);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long*);

template <typename Fn>
Fn driver_fn(const char* name, int version) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, version, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<Fn>(p);
  return nullptr;
}

// ID of the calling thread's current context (0 when none is current yet).
int current_ctx_id(unsigned long long* id) {
  static CtxGetCurrentFn get_current = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    get_current = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent", 4000);
    get_id = driver_fn<CtxGetIdFn>("cuCtxGetId", 12000);
  });
  if (!get_current || !get_id) return fail(QG_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId entry points unavailable");
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return fail(QG_ERR_CUDA, "cuCtxGetCurrent failed");
  *id = 0;
  if (ctx && get_id(ctx, id) != CUDA_SUCCESS) return fail(QG_ERR_CUDA, "cuCtxGetId failed");
  return QG_OK;
}

// Device address of g_noalloc_scratch in the current context, looked up
// (cudaGetSymbolAddress) the first time a context calls, with the caller's
// device current.
int noalloc_scratch(void** out) {
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  unsigned long long id = 0;
  int rc = current_ctx_id(&id);
  if (rc != QG_OK) return rc;
  if (id != 0)
    for (const NoallocEntry& e : g_noalloc_cache)
      if (e.ctx_id == id) {
        *out = e.addr;
        return QG_OK;
      }
  // first call in this context (or no context yet: the lookup makes the
  // device's primary context current)
  void* p = nullptr;
  cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(noalloc scratch)");
  rc = current_ctx_id(&id);
  if (rc != QG_OK) return rc;
  if (id == 0) return fail(QG_ERR_CUDA, "no current CUDA context after the symbol lookup");
  g_noalloc_cache.push_back(NoallocEntry{id, p});
  *out = p;
  return QG_OK;
}

}  // namespace

// ------------------------------------------------- host weight packing
// qg_pack_weight: the weight quantization of qg_quant_weight on the host
// (fp32 IEEE arithmetic, one division per scale and per code), for callers
// that quantize checkpoints offline and upload codes and scales.
namespace {

float pack_scale(float amax, float qmax) { return amax > 0.0f ? amax / qmax : 1.0f; }

uint8_t pack_code(bool int8, float x, float s) {
  const float q = x / s;
  if (int8) {
    const float r = std::min(127.0f, std::max(-127.0f, std::nearbyint(q)));  // ties to even
    return static_cast<uint8_t>(static_cast<int8_t>(r));
  }
  return static_cast<uint8_t>(__nv_cvt_float_to_fp8(q, __NV_SATFINITE, __NV_E4M3));
}

}  // namespace

// ====================================================================== ABI
extern "C" {

const char* qg_last_error(void) { return g_err.c_str(); }
const char* qg_version(void) { return "qgemm-b300 0.1 (sm_103a)"; }

int qg_set_launch_flags(int flags) {
  if (flags & ~(QG_LAUNCH_PDL | QG_LAUNCH_FUSED_QUANT))
    return fail(QG_ERR_INVALID_ARG, "unknown launch flag bits 0x%x", flags);
  g_launch_flags.store(flags, std::memory_order_relaxed);
  return QG_OK;
}
int qg_set_wait_limit_ns(uint64_t ns) {
  g_wait_ns.store(ns ? ns : 2000000000ull, std::memory_order_relaxed);
  return QG_OK;
}
int qg_set_timing_log(uint64_t* log_dev, int slots) {
  if (slots < 0) return fail(QG_ERR_INVALID_ARG, "slots=%d < 0", slots);
  if (log_dev && !aligned(log_dev, 8)) return fail(QG_ERR_INVALID_ARG, "timing log must be 8-byte aligned");
  g_ts_log.store(nullptr, std::memory_order_relaxed);
  g_ts_cap.store(log_dev ? slots : 0, std::memory_order_relaxed);
  g_ts_next.store(0, std::memory_order_relaxed);
  g_ts_log.store(reinterpret_cast<unsigned long long*>(log_dev), std::memory_order_relaxed);
  return QG_OK;
}
int qg_timing_log_count(void) { return g_ts_next.load(std::memory_order_relaxed); }
int qg_set_force_timeout(int on) {
  g_force_timeout.store(on ? 1 : 0, std::memory_order_relaxed);
  return QG_OK;
}
int qg_set_allow_default(int allow) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_allow_default = allow != 0;
  return QG_OK;
}

int qg_device_error(int* code) {
  if (!code) return fail(QG_ERR_INVALID_ARG, "code is NULL");
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  int v = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&v, qg::g_device_status, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "read device status");
  e = cudaMemcpyToSymbol(qg::g_device_status, &zero, sizeof(int));
  if (e != cudaSuccess) return cuda_fail(e, "clear device status");
  *code = v;
  return QG_OK;
}

int qg_quant_act(int fmt, const void* A_dev, int64_t M, int64_t K, int64_t lda, void* A_q_dev, float* s_a_dev,
                 void* stream) {
  if (fmt < 0 || fmt > 2) return fail(QG_ERR_INVALID_ARG, "unknown format %d", fmt);
  if (M < 0 || K <= 0 || lda < K) return fail(QG_ERR_INVALID_ARG, "bad sizes M=%lld K=%lld lda=%lld", (long long)M, (long long)K, (long long)lda);
  if (M == 0) return QG_OK;
  if (!A_dev || !A_q_dev || !s_a_dev) return fail(QG_ERR_INVALID_ARG, "null pointer");
  if (K % 16) return fail(QG_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a multiple of 16", (long long)K);
  if (fmt == QG_BLOCK_FP8 && K % 128) return fail(QG_ERR_UNSUPPORTED_SHAPE, "Block_FP8 needs K %% 128 == 0");
  if (lda % 8 || !aligned(A_dev, 16) || !aligned(A_q_dev, 16) || !aligned(s_a_dev, 4))
    return fail(QG_ERR_ALIGNMENT, "A/A_q must be 16-byte aligned with lda %% 8 == 0");
  if (M > 0x7FFFFFFF || K > 0x7FFFFFFF) return fail(QG_ERR_UNSUPPORTED_SHAPE, "sizes too large");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const __nv_bfloat16* A = static_cast<const __nv_bfloat16*>(A_dev);
  uint8_t* Q = static_cast<uint8_t*>(A_q_dev);
  unsigned long long* ts = next_ts_slot();
  cudaError_t e;
  if (fmt == QG_BLOCK_FP8) {
    constexpr int W = 8;
    const int64_t groups = M * (K / 128);
    e = launch(qg::quant_groups_kernel<W>, dim3(static_cast<unsigned>(cdiv(groups, W))), dim3(W * 32), 0, s, A, lda,
               static_cast<int>(M), static_cast<int>(K), Q, s_a_dev, ts);
  } else if (K <= 512 * 8 * 8) {
    // rows held in registers: 1, 2, 4 or 8 chunks of 8 values per thread
    const int ch = K <= 4096 ? 1 : (K <= 8192 ? 2 : (K <= 16384 ? 4 : 8));
    const bool fp8 = fmt == QG_FP8_DYNAMIC;
    const float qmax = fp8 ? 448.0f : 127.0f;
    const dim3 grid(static_cast<unsigned>(M)), block(512);
    const int k = static_cast<int>(K);
    if (ch == 1)
      e = fp8 ? launch(qg::quant_rows_reg_kernel<qg::kFmtFP8, 1>, grid, block, 0, s, A, lda, k, Q, s_a_dev, qmax, ts)
              : launch(qg::quant_rows_reg_kernel<qg::kFmtINT8, 1>, grid, block, 0, s, A, lda, k, Q, s_a_dev, qmax, ts);
    else if (ch == 2)
      e = fp8 ? launch(qg::quant_rows_reg_kernel<qg::kFmtFP8, 2>, grid, block, 0, s, A, lda, k, Q, s_a_dev, qmax, ts)
              : launch(qg::quant_rows_reg_kernel<qg::kFmtINT8, 2>, grid, block, 0, s, A, lda, k, Q, s_a_dev, qmax, ts);
    else if (ch == 4)
      e = fp8 ? launch(qg::quant_rows_reg_kernel<qg::kFmtFP8, 4>, grid, block, 0, s, A, lda, k, Q, s_a_dev, qmax, ts)
              : launch(qg::quant_rows_reg_kernel<qg::kFmtINT8, 4>, grid, block, 0, s, A, lda, k, Q, s_a_dev, qmax, ts);
    else
      e = fp8 ? launch(qg::quant_rows_reg_kernel<qg::kFmtFP8, 8>, grid, block, 0, s, A, lda, k, Q, s_a_dev, qmax, ts)
              : launch(qg::quant_rows_reg_kernel<qg::kFmtINT8, 8>, grid, block, 0, s, A, lda, k, Q, s_a_dev, qmax, ts);
  } else if (fmt == QG_FP8_DYNAMIC) {
    e = launch(qg::quant_rows_kernel<__nv_bfloat16, qg::kFmtFP8, 512>, dim3(static_cast<unsigned>(M)), dim3(512), 0, s,
               A, lda, static_cast<int>(K), Q, s_a_dev, 448.0f, ts);
  } else {
    e = launch(qg::quant_rows_kernel<__nv_bfloat16, qg::kFmtINT8, 512>, dim3(static_cast<unsigned>(M)), dim3(512), 0,
               s, A, lda, static_cast<int>(K), Q, s_a_dev, 127.0f, ts);
  }
  if (e != cudaSuccess) return cuda_fail(e, "quant_act launch");
  return QG_OK;
}

int qg_pack_weight(int fmt, const float* W_host, int64_t N, int64_t K, void* W_q_host, float* s_w_host) {
  if (fmt < 0 || fmt > 2) return fail(QG_ERR_INVALID_ARG, "unknown format %d", fmt);
  if (N <= 0 || K <= 0) return fail(QG_ERR_INVALID_ARG, "bad sizes N=%lld K=%lld", (long long)N, (long long)K);
  if (!W_host || !W_q_host || !s_w_host) return fail(QG_ERR_INVALID_ARG, "null pointer");
  if (K % 16) return fail(QG_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a multiple of 16", (long long)K);
  if (fmt == QG_BLOCK_FP8 && K % 128) return fail(QG_ERR_UNSUPPORTED_SHAPE, "Block_FP8 needs K %% 128 == 0");
  uint8_t* Q = static_cast<uint8_t*>(W_q_host);
  if (fmt == QG_BLOCK_FP8) {
    const int64_t kblocks = K / 128;
    for (int64_t n0 = 0; n0 < N; n0 += 128) {
      const int64_t n1 = std::min(N, n0 + 128);
      for (int64_t kb = 0; kb < kblocks; ++kb) {
        float amax = 0.0f;
        for (int64_t n = n0; n < n1; ++n)
          for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) amax = std::max(amax, std::fabs(W_host[n * K + k]));
        const float sc = pack_scale(amax, 448.0f);
        s_w_host[(n0 / 128) * kblocks + kb] = sc;
        for (int64_t n = n0; n < n1; ++n)
          for (int64_t k = kb * 128; k < kb * 128 + 128; ++k) Q[n * K + k] = pack_code(false, W_host[n * K + k], sc);
      }
    }
    return QG_OK;
  }
  const bool int8 = fmt == QG_W8A8_INT8;
  for (int64_t n = 0; n < N; ++n) {
    const float* w = W_host + n * K;
    float amax = 0.0f;
    for (int64_t k = 0; k < K; ++k) amax = std::max(amax, std::fabs(w[k]));
    const float sc = pack_scale(amax, int8 ? 127.0f : 448.0f);
    s_w_host[n] = sc;
    for (int64_t k = 0; k < K; ++k) Q[n * K + k] = pack_code(int8, w[k], sc);
  }
  return QG_OK;
}

int qg_quant_weight(int fmt, const float* W_dev, int64_t N, int64_t K, void* W_q_dev, float* s_w_dev, void* stream) {
  if (fmt < 0 || fmt > 2) return fail(QG_ERR_INVALID_ARG, "unknown format %d", fmt);
  if (N <= 0 || K <= 0) return fail(QG_ERR_INVALID_ARG, "bad sizes N=%lld K=%lld", (long long)N, (long long)K);
  if (!W_dev || !W_q_dev || !s_w_dev) return fail(QG_ERR_INVALID_ARG, "null pointer");
  if (K % 16) return fail(QG_ERR_UNSUPPORTED_SHAPE, "K=%lld must be a multiple of 16", (long long)K);
  if (fmt == QG_BLOCK_FP8 && K % 128) return fail(QG_ERR_UNSUPPORTED_SHAPE, "Block_FP8 needs K %% 128 == 0");
  if (!aligned(W_dev, 16) || !aligned(W_q_dev, 16) || !aligned(s_w_dev, 4))
    return fail(QG_ERR_ALIGNMENT, "W/W_q must be 16-byte aligned");
  if (N > 0x7FFFFFFF || K > 0x7FFFFFFF || cdiv(N, 128) > 65535) return fail(QG_ERR_UNSUPPORTED_SHAPE, "sizes too large");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint8_t* Q = static_cast<uint8_t*>(W_q_dev);
  cudaError_t e;
  if (fmt == QG_BLOCK_FP8) {
    e = launch(qg::quant_blocks_kernel, dim3(static_cast<unsigned>(K / 128), static_cast<unsigned>(cdiv(N, 128))),
               dim3(256), 0, s, W_dev, static_cast<int>(N), static_cast<int>(K), Q, s_w_dev);
  } else if (fmt == QG_FP8_DYNAMIC) {
    e = launch(qg::quant_rows_kernel<float, qg::kFmtFP8, 256>, dim3(static_cast<unsigned>(N)), dim3(256), 0, s, W_dev,
               K, static_cast<int>(K), Q, s_w_dev, 448.0f, nullptr);
  } else {
    e = launch(qg::quant_rows_kernel<float, qg::kFmtINT8, 256>, dim3(static_cast<unsigned>(N)), dim3(256), 0, s, W_dev,
               K, static_cast<int>(K), Q, s_w_dev, 127.0f, nullptr);
  }
  if (e != cudaSuccess) return cuda_fail(e, "quant_weight launch");
  return QG_OK;
}

size_t qg_workspace_bytes_config(int fmt, int64_t M, int64_t N, int64_t K, int variant, int split_k, int config_id) {
  Plan p;
  if (fmt < 0 || fmt > 2 || M <= 0 || N <= 0 || K <= 0 || variant < 0 || variant > QG_SWAPAB_DP4A_SPLITK) return 0;
  if (check_config_bits(fmt, variant, config_id) != QG_OK) return 0;
  if (make_plan(fmt, M, N, K, variant, split_k, config_id, &p) != QG_OK) return 0;
  return static_cast<size_t>(workspace_bytes(p, M, N, K));
}
size_t qg_workspace_bytes(int fmt, int64_t M, int64_t N, int64_t K, int variant, int split_k) {
  return qg_workspace_bytes_config(fmt, M, N, K, variant, split_k, 0);
}

int qg_check_config(int fmt, int64_t M, int64_t N, int64_t K, int variant, int split_k, int config_id) {
  return check_shape_config(fmt, M, N, K, variant, split_k, config_id);
}

int qg_workspace_init(void* workspace_dev, size_t ws_bytes, void* stream) {
  if (!workspace_dev || ws_bytes == 0) return QG_OK;
  cudaError_t e = cudaMemsetAsync(workspace_dev, 0, ws_bytes, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
  return QG_OK;
}

int qg_gemm_w8a8(int fmt, int64_t M, int64_t N, int64_t K, const void* A_q_dev, const float* s_a_dev,
                 const void* W_q_dev, const float* s_w_dev, void* Y_dev, int64_t ldy, int variant, int split_k,
                 int config_id, void* workspace_dev, size_t ws_bytes, int32_t* debug_acc_dev, void* stream) {
  return gemm_entry(fmt, M, N, K, A_q_dev, s_a_dev, W_q_dev, s_w_dev, Y_dev, ldy, variant, split_k, config_id,
                    workspace_dev, ws_bytes, debug_acc_dev, stream, nullptr);
}

int qg_gemm_w8a8_grouped(int fmt, int groups, const int32_t* token_offsets_dev, int64_t total_tokens,
                         int64_t max_tokens, int64_t N, int64_t K, const void* A_q_dev, const float* s_a_dev,
                         const void* W_q_dev, const float* s_w_dev, void* Y_dev, int64_t ldy, int variant,
                         int split_k, int config_id, void* workspace_dev, size_t ws_bytes, int32_t* debug_acc_dev,
                         void* stream) {
  if (max_tokens < 0 || total_tokens < 0) return fail(QG_ERR_INVALID_ARG, "negative token counts");
  const GroupIn gi{groups, token_offsets_dev, total_tokens};
  return gemm_entry(fmt, max_tokens, N, K, A_q_dev, s_a_dev, W_q_dev, s_w_dev, Y_dev, ldy, variant, split_k,
                    config_id, workspace_dev, ws_bytes, debug_acc_dev, stream, nullptr, &gi);
}

size_t qg_workspace_bytes_grouped(int fmt, int groups, int64_t total_tokens, int64_t max_tokens, int64_t N, int64_t K,
                                  int variant, int split_k) {
  Plan p;
  if (fmt < 0 || fmt > 2 || groups < 1 || total_tokens < 0 || max_tokens <= 0 || N <= 0 || K <= 0 || variant < 0 ||
      variant > QG_SWAPAB_DP4A_SPLITK)
    return 0;
  if (make_plan(fmt, max_tokens, N, K, variant, split_k, 0, &p) != QG_OK) return 0;
  p.groups = groups;
  return static_cast<size_t>(workspace_bytes(p, total_tokens, N, K));
}

int qg_linear_w8a8(int fmt, int64_t M, int64_t N, int64_t K, const void* A_dev, int64_t lda, const void* W_q_dev,
                   const float* s_w_dev, void* Y_dev, int64_t ldy, int variant, int split_k, int config_id,
                   void* workspace_dev, size_t ws_bytes, void* A_q_dev, float* s_a_dev, int32_t* debug_acc_dev,
                   void* stream) {
  if (fmt < 0 || fmt > 2) return fail(QG_ERR_INVALID_ARG, "unknown format %d", fmt);
  const bool fusable = (variant == QG_SWAPAB || variant == QG_SWAPAB_SPLITK) &&
                       !(config_id & (QG_CONFIG_MMA_SYNC | QG_CONFIG_I8_PREWIDEN | QG_CONFIG_I8_CONV16 |
                                      QG_CONFIG_BLOCK_PROMO8));
  const bool buffers = A_q_dev != nullptr && s_a_dev != nullptr;
  if (fusable && (!buffers || (config_id & QG_CONFIG_FUSED_QUANT) ||
                  (g_launch_flags.load(std::memory_order_relaxed) & QG_LAUNCH_FUSED_QUANT))) {
    // one kernel: each CTA quantizes the activations its K range needs
    if ((A_q_dev && !aligned(A_q_dev, 16)) || (s_a_dev && !aligned(s_a_dev, 4)))
      return fail(QG_ERR_ALIGNMENT, "A_q needs 16-byte alignment, s_a 4");
    const FusedIn f{A_dev, lda};
    return gemm_entry(fmt, M, N, K, A_q_dev, s_a_dev, W_q_dev, s_w_dev, Y_dev, ldy, variant, split_k, config_id,
                      workspace_dev, ws_bytes, debug_acc_dev, stream, &f);
  }
  // two kernels: quantize into the caller's A_q / s_a, then the GEMM
  if (!buffers)
    return fail(QG_ERR_INVALID_ARG,
                "qg_linear_w8a8: the Standard, dp4a and mma.sync forms need A_q and s_a buffers");
  int rc = qg_quant_act(fmt, A_dev, M, K, lda, A_q_dev, s_a_dev, stream);
  if (rc != QG_OK) return rc;
  return gemm_entry(fmt, M, N, K, A_q_dev, s_a_dev, W_q_dev, s_w_dev, Y_dev, ldy, variant, split_k, config_id,
                    workspace_dev, ws_bytes, debug_acc_dev, stream, nullptr);
}

int qg_gemm_w8a8_noalloc(int fmt, int64_t M, int64_t N, int64_t K, const void* A_q_dev, const float* s_a_dev,
                         const void* W_q_dev, const float* s_w_dev, void* Y_dev, int64_t ldy, int variant,
                         int split_k, int config_id, int32_t* debug_acc_dev, void* stream) {
  const size_t need = qg_workspace_bytes_config(fmt, M, N, K, variant, split_k, config_id);
  if (need > QG_NOALLOC_SCRATCH_BYTES)
    return fail(QG_ERR_WORKSPACE_TOO_SMALL,
                "qg_gemm_w8a8_noalloc: this shape needs %zu bytes of Split-K scratch, more than the %u-byte static "
                "array; use fewer splits or qg_gemm_w8a8 with a workspace",
                need, static_cast<unsigned>(QG_NOALLOC_SCRATCH_BYTES));
  void* ws = nullptr;
  if (need > 0) {
    int rc = noalloc_scratch(&ws);
    if (rc != QG_OK) return rc;
    Plan p;
    rc = make_plan(fmt, M, N, K, variant, split_k, config_id, &p);
    if (rc != QG_OK) return rc;
    const int64_t counters = ws_counter_bytes(p.ctr_tiles);
    cudaError_t e = cudaMemsetAsync(ws, 0, static_cast<size_t>(counters), static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "clear noalloc counters");
  }
  return qg_gemm_w8a8(fmt, M, N, K, A_q_dev, s_a_dev, W_q_dev, s_w_dev, Y_dev, ldy, variant, split_k, config_id, ws,
                      need, debug_acc_dev, stream);
}

int qg_load_table(const char* path) {
  std::lock_guard<std::mutex> lk(g_mu);
  g_table_env_checked = true;
  if (!path) {
    path = getenv("QG_TABLE");
    if (!path) return fail(QG_ERR_INVALID_ARG, "no path given and $QG_TABLE unset");
  }
  return load_table_file(path);
}

int qg_select(int fmt, int64_t M, int64_t N, int64_t K, int* variant, int* split_k, int* config_id) {
  if (fmt < 0 || fmt > 2) return fail(QG_ERR_INVALID_ARG, "unknown format %d", fmt);
  if (M <= 0 || N <= 0 || K <= 0) return fail(QG_ERR_INVALID_ARG, "bad sizes");
  if (!variant || !split_k || !config_id) return fail(QG_ERR_INVALID_ARG, "null output pointer");
  std::lock_guard<std::mutex> lk(g_mu);
  if (!g_table_env_checked) {
    g_table_env_checked = true;
    const char* env = getenv("QG_TABLE");
    if (env) {
      int rc = load_table_file(env);
      if (rc != QG_OK) return rc;
    }
  }
  // smallest tuned token count >= M for this (fmt, N, K)
  const Row* best = nullptr;
  int max_m = 0;
  for (auto it = g_table.lower_bound(Key{fmt, N, K, 0}); it != g_table.end(); ++it) {
    if (it->first.fmt != fmt || it->first.n != N || it->first.k != K) break;
    max_m = std::max(max_m, it->first.m);
    if (it->first.m >= M && !best) best = &it->second;
  }
  if (best) {
    *variant = best->variant;
    *split_k = best->split_k;
    *config_id = best->config_id;
    return QG_OK;
  }
  if (max_m > 0 || g_allow_default) {  // beyond the tuned range, or defaults allowed
    default_config(fmt, M, N, K, variant, split_k, config_id);
    return QG_OK;
  }
  return fail(QG_ERR_NO_CONFIG, "no tuned config for fmt=%d N=%lld K=%lld M=%lld", fmt, (long long)N, (long long)K,
              (long long)M);
}

}  // extern "C"
