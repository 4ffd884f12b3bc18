"""ctypes binding of libqgemm.so (include/qgemm.h), argument marshalling only.

Every function keeps the C name and order of arguments; torch tensors are
accepted where the C side takes device pointers, and ``stream`` defaults to
torch's current stream.  All computation happens in the library's sm_103a
kernels: importing this module fails loudly when the library is missing.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libqgemm.so")

QG_FP8_DYNAMIC, QG_W8A8_INT8, QG_BLOCK_FP8 = 0, 1, 2
QG_STANDARD, QG_SPLITK, QG_SWAPAB, QG_SWAPAB_SPLITK, QG_SWAPAB_DP4A, QG_SWAPAB_DP4A_SPLITK = 0, 1, 2, 3, 4, 5
QG_OK = 0
QG_ERR_INVALID_ARG, QG_ERR_UNSUPPORTED_SHAPE, QG_ERR_ALIGNMENT = -1, -2, -3
QG_ERR_WORKSPACE_TOO_SMALL, QG_ERR_NO_CONFIG, QG_ERR_CUDA = -4, -5, -6
QG_ERR_DEVICE_TIMEOUT, QG_ERR_TABLE_PARSE = -7, -8
QG_LAUNCH_PDL = 1
QG_LAUNCH_FUSED_QUANT = 2

FORMATS = {"FP8_Dynamic": QG_FP8_DYNAMIC, "W8A8_INT8": QG_W8A8_INT8, "Block_FP8": QG_BLOCK_FP8}
VARIANTS = {"Standard": QG_STANDARD, "Split-K": QG_SPLITK, "Swap-AB": QG_SWAPAB, "Swap-AB+Split-K": QG_SWAPAB_SPLITK,
            "Swap-AB dp4a": QG_SWAPAB_DP4A, "Swap-AB dp4a+Split-K": QG_SWAPAB_DP4A_SPLITK}

QG_NOALLOC_SCRATCH_BYTES = 4 << 20
QG_CONFIG_RING_MASK, QG_CONFIG_PREFETCH_SHIFT, QG_CONFIG_MAX_PREFETCH = 31, 5, 64
QG_CONFIG_WIDE = 1 << 12
QG_CONFIG_MMA_SYNC = 1 << 13
QG_CONFIG_MMA_NARROW = 1 << 14
QG_CONFIG_FUSED_QUANT = 1 << 15
QG_CONFIG_PERSIST = 1 << 16
QG_CONFIG_MMA_DP4A_SHIFT = 17
QG_CONFIG_MMA_S8 = 1 << 20
QG_CONFIG_PAIR_MMA = 1 << 21
QG_CONFIG_I8_PREWIDEN = 1 << 22
QG_CONFIG_I8_CONV16 = 1 << 23
QG_CONFIG_BLOCK_PROMO8 = 1 << 24
QG_CONFIG_PERSIST_ROWS_SHIFT = 25
QG_CONFIG_PERSIST_ROWS_MASK = 3 << 25
PERSIST_ROWS = (256, 224, 192, 160)


def config_id(ring: int = 0, prefetch: int = 0, wide: bool = False, mma_sync: bool = False,
              narrow: bool = False, fused: bool = False, persist: bool = False, dp4a_rows16: int = 0,
              s8: bool = False, pair_mma: bool = False, prewiden: bool = False, conv16: bool = False,
              promo8: bool = False, persist_rows: int = 256) -> int:
    """config_id of a ring depth (0 = default), an L2 prefetch distance,
    (FP8_Dynamic Standard / Split-K) 256-row weight tiles, (W8A8_INT8
    Swap-AB) the mma.sync kernel with eight narrow MMA warps if `narrow`,
    (Swap-AB on the tcgen05 kernels) qg_linear_w8a8's one-kernel form, and
    (FP8_Dynamic Standard) the persistent pair kernel; dp4a_rows16 groups
    of 16 weight rows on dp4a warps (implies the narrow mma.sync kernel);
    `s8`: the mma.sync kernel on the int8 form of the instruction (implies
    mma_sync); `pair_mma`: the persistent kernel with tcgen05.mma.cta_group::2
    (implies persist); `prewiden`: W8A8_INT8 Swap-AB on activations widened
    once per launch into the workspace (QG_CONFIG_I8_PREWIDEN); `conv16`:
    its tcgen05 kernel with sixteen converter warps, one CTA per SM
    (QG_CONFIG_I8_CONV16); `promo8`: Block_FP8 Swap-AB with eight promotion
    warps (QG_CONFIG_BLOCK_PROMO8); `persist_rows`: the persistent kernel's
    weight rows per tile, one of 256, 224, 192, 160 (not 256 implies
    persist)."""
    if persist_rows not in PERSIST_ROWS:
        raise ValueError(f"persist_rows must be one of {PERSIST_ROWS}")
    rows_code = PERSIST_ROWS.index(persist_rows)
    persist = persist or rows_code > 0
    narrow = narrow or dp4a_rows16 > 0
    return (ring | (prefetch << QG_CONFIG_PREFETCH_SHIFT) | (QG_CONFIG_WIDE if wide else 0)
            | (QG_CONFIG_MMA_SYNC if mma_sync or narrow or s8 else 0) | (QG_CONFIG_MMA_NARROW if narrow else 0)
            | (QG_CONFIG_MMA_S8 if s8 else 0)
            | (QG_CONFIG_FUSED_QUANT if fused else 0) | (QG_CONFIG_PERSIST if persist or pair_mma else 0)
            | (QG_CONFIG_PAIR_MMA if pair_mma else 0) | (QG_CONFIG_I8_PREWIDEN if prewiden else 0)
            | (QG_CONFIG_I8_CONV16 if conv16 else 0) | (QG_CONFIG_BLOCK_PROMO8 if promo8 else 0)
            | (rows_code << QG_CONFIG_PERSIST_ROWS_SHIFT)
            | (dp4a_rows16 << QG_CONFIG_MMA_DP4A_SHIFT))

EXPORTS = ("qg_quant_act", "qg_quant_weight", "qg_pack_weight", "qg_workspace_bytes", "qg_workspace_bytes_config",
           "qg_check_config", "qg_workspace_init", "qg_gemm_w8a8",
           "qg_linear_w8a8", "qg_gemm_w8a8_noalloc", "qg_gemm_w8a8_grouped", "qg_workspace_bytes_grouped",
           "qg_select", "qg_load_table", "qg_set_allow_default", "qg_set_launch_flags", "qg_set_wait_limit_ns",
           "qg_set_force_timeout", "qg_set_timing_log", "qg_timing_log_count", "qg_device_error", "qg_last_error",
           "qg_version")


class QGError(RuntimeError):
    def __init__(self, code: int, where: str, msg: str):
        super().__init__(f"{where} failed with status {code}: {msg}")
        self.code = code


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise ImportError(f"libqgemm.so not built at {path}; run quantized_gemm_decode_02_b300/build.py")
    lib = ctypes.CDLL(path)
    P, I64, I, SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.qg_quant_act.argtypes = [I, P, I64, I64, I64, P, P, P]
    lib.qg_quant_weight.argtypes = [I, P, I64, I64, P, P, P]
    lib.qg_pack_weight.argtypes = [I, P, I64, I64, P, P]
    lib.qg_workspace_bytes.argtypes = [I, I64, I64, I64, I, I]
    lib.qg_workspace_bytes.restype = SZ
    lib.qg_workspace_bytes_config.argtypes = [I, I64, I64, I64, I, I, I]
    lib.qg_workspace_bytes_config.restype = SZ
    lib.qg_check_config.argtypes = [I, I64, I64, I64, I, I, I]
    lib.qg_workspace_init.argtypes = [P, SZ, P]
    lib.qg_gemm_w8a8.argtypes = [I, I64, I64, I64, P, P, P, P, P, I64, I, I, I, P, SZ, P, P]
    lib.qg_gemm_w8a8_noalloc.argtypes = [I, I64, I64, I64, P, P, P, P, P, I64, I, I, I, P, P]
    lib.qg_gemm_w8a8_grouped.argtypes = [I, I, P, I64, I64, I64, I64, P, P, P, P, P, I64, I, I, I, P, SZ, P, P]
    lib.qg_workspace_bytes_grouped.argtypes = [I, I, I64, I64, I64, I64, I, I]
    lib.qg_workspace_bytes_grouped.restype = SZ
    lib.qg_linear_w8a8.argtypes = [I, I64, I64, I64, P, I64, P, P, P, I64, I, I, I, P, SZ, P, P, P, P]
    lib.qg_select.argtypes = [I, I64, I64, I64, ctypes.POINTER(I), ctypes.POINTER(I), ctypes.POINTER(I)]
    lib.qg_load_table.argtypes = [ctypes.c_char_p]
    lib.qg_set_allow_default.argtypes = [I]
    lib.qg_set_launch_flags.argtypes = [I]
    lib.qg_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    lib.qg_set_force_timeout.argtypes = [I]
    lib.qg_set_timing_log.argtypes = [P, I]
    lib.qg_timing_log_count.argtypes = []
    lib.qg_device_error.argtypes = [ctypes.POINTER(I)]
    lib.qg_last_error.restype = ctypes.c_char_p
    lib.qg_version.restype = ctypes.c_char_p
    return lib


_lib = load_library()


def _check(rc: int, where: str) -> int:
    if rc != QG_OK:
        raise QGError(rc, where, _lib.qg_last_error().decode())
    return rc


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _fmt(fmt) -> int:
    return FORMATS[fmt] if isinstance(fmt, str) else int(fmt)


def qg_quant_act(fmt, A, M, K, lda, A_q, s_a, stream=None) -> None:
    _check(_lib.qg_quant_act(_fmt(fmt), _ptr(A), M, K, lda, _ptr(A_q), _ptr(s_a), _stream(stream)), "qg_quant_act")


def qg_quant_weight(fmt, W, N, K, W_q, s_w, stream=None) -> None:
    _check(_lib.qg_quant_weight(_fmt(fmt), _ptr(W), N, K, _ptr(W_q), _ptr(s_w), _stream(stream)), "qg_quant_weight")


def qg_pack_weight(fmt, W, N, K, W_q, s_w) -> None:
    """Host weight quantization: W (fp32 [N, K]), W_q (1-byte [N, K]) and s_w
    (fp32 [N] or [ceil(N/128), K/128]) are contiguous CPU tensors."""
    f = _fmt(fmt)
    n_scales = -(-N // 128) * (K // 128) if f == QG_BLOCK_FP8 else N
    for t, dt, n, name in ((W, torch.float32, N * K, "W"), (W_q, None, N * K, "W_q"), (s_w, torch.float32, n_scales, "s_w")):
        if not isinstance(t, torch.Tensor):
            continue
        if t.is_cuda or not t.is_contiguous():
            raise ValueError("qg_pack_weight takes contiguous host tensors")
        if (dt is not None and t.dtype != dt) or (dt is None and t.element_size() != 1) or t.numel() < n:
            raise ValueError(f"qg_pack_weight: {name} must hold {n} {'fp32' if dt else '1-byte'} values")
    _check(_lib.qg_pack_weight(_fmt(fmt), _ptr(W), N, K, _ptr(W_q), _ptr(s_w)), "qg_pack_weight")


def qg_workspace_bytes(fmt, M, N, K, variant, split_k) -> int:
    return int(_lib.qg_workspace_bytes(_fmt(fmt), M, N, K, variant, split_k))


def qg_workspace_bytes_config(fmt, M, N, K, variant, split_k, config_id=0) -> int:
    return int(_lib.qg_workspace_bytes_config(_fmt(fmt), M, N, K, variant, split_k, config_id))


def qg_check_config(fmt, M, N, K, variant, split_k, config_id=0) -> int:
    """Status qg_gemm_w8a8 would return for this configuration's pointer-free
    checks (QG_OK = accepted); no exception, no launch."""
    return int(_lib.qg_check_config(_fmt(fmt), M, N, K, variant, split_k, config_id))


def qg_workspace_init(workspace, ws_bytes, stream=None) -> None:
    _check(_lib.qg_workspace_init(_ptr(workspace), ws_bytes, _stream(stream)), "qg_workspace_init")


def qg_gemm_w8a8(fmt, M, N, K, A_q, s_a, W_q, s_w, Y, ldy, variant, split_k, config_id=0, workspace=None,
                 ws_bytes=0, debug_acc=None, stream=None) -> None:
    _check(_lib.qg_gemm_w8a8(_fmt(fmt), M, N, K, _ptr(A_q), _ptr(s_a), _ptr(W_q), _ptr(s_w), _ptr(Y), ldy, variant,
                             split_k, config_id, _ptr(workspace), ws_bytes, _ptr(debug_acc), _stream(stream)),
           "qg_gemm_w8a8")


def qg_linear_w8a8(fmt, M, N, K, A, lda, W_q, s_w, Y, ldy, variant, split_k, config_id=0, workspace=None,
                   ws_bytes=0, A_q=None, s_a=None, debug_acc=None, stream=None) -> None:
    """Activation quantization and the GEMM in one call: two kernels when
    A_q and s_a are given, else (FP8_Dynamic / W8A8_INT8 with Swap-AB, or
    with QG_LAUNCH_FUSED_QUANT set) one kernel."""
    _check(_lib.qg_linear_w8a8(_fmt(fmt), M, N, K, _ptr(A), lda, _ptr(W_q), _ptr(s_w), _ptr(Y), ldy, variant,
                               split_k, config_id, _ptr(workspace), ws_bytes, _ptr(A_q), _ptr(s_a), _ptr(debug_acc),
                               _stream(stream)), "qg_linear_w8a8")


def qg_gemm_w8a8_grouped(fmt, groups, token_offsets, total_tokens, max_tokens, N, K, A_q, s_a, W_q, s_w, Y, ldy,
                         variant, split_k, config_id=0, workspace=None, ws_bytes=0, debug_acc=None,
                         stream=None) -> None:
    """Grouped (mixture-of-experts) GEMM: group g's tokens are rows
    token_offsets[g] .. token_offsets[g+1] of A_q / Y, its weights W_q[g]."""
    _check(_lib.qg_gemm_w8a8_grouped(_fmt(fmt), groups, _ptr(token_offsets), total_tokens, max_tokens, N, K,
                                     _ptr(A_q), _ptr(s_a), _ptr(W_q), _ptr(s_w), _ptr(Y), ldy, variant, split_k,
                                     config_id, _ptr(workspace), ws_bytes, _ptr(debug_acc), _stream(stream)),
           "qg_gemm_w8a8_grouped")


def qg_workspace_bytes_grouped(fmt, groups, total_tokens, max_tokens, N, K, variant, split_k) -> int:
    return int(_lib.qg_workspace_bytes_grouped(_fmt(fmt), groups, total_tokens, max_tokens, N, K, variant, split_k))


def qg_gemm_w8a8_noalloc(fmt, M, N, K, A_q, s_a, W_q, s_w, Y, ldy, variant, split_k, config_id=0, debug_acc=None,
                         stream=None) -> None:
    """qg_gemm_w8a8 without a caller workspace: Split-K scratch comes from the
    library's static 4 MiB device array (for callers that cannot allocate)."""
    _check(_lib.qg_gemm_w8a8_noalloc(_fmt(fmt), M, N, K, _ptr(A_q), _ptr(s_a), _ptr(W_q), _ptr(s_w), _ptr(Y), ldy,
                                     variant, split_k, config_id, _ptr(debug_acc), _stream(stream)),
           "qg_gemm_w8a8_noalloc")


def qg_select(fmt, M, N, K) -> tuple[int, int, int]:
    v, s, c = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
    _check(_lib.qg_select(_fmt(fmt), M, N, K, ctypes.byref(v), ctypes.byref(s), ctypes.byref(c)), "qg_select")
    return v.value, s.value, c.value


def qg_load_table(path) -> None:
    _check(_lib.qg_load_table(None if path is None else os.fsencode(path)), "qg_load_table")


def qg_set_allow_default(allow: bool) -> None:
    _check(_lib.qg_set_allow_default(1 if allow else 0), "qg_set_allow_default")


def qg_set_launch_flags(flags: int) -> None:
    _check(_lib.qg_set_launch_flags(flags), "qg_set_launch_flags")


def qg_set_wait_limit_ns(ns: int) -> None:
    _check(_lib.qg_set_wait_limit_ns(ns), "qg_set_wait_limit_ns")


def qg_set_force_timeout(on: bool) -> None:
    _check(_lib.qg_set_force_timeout(1 if on else 0), "qg_set_force_timeout")


def qg_set_timing_log(log, slots: int) -> None:
    """Give every following launch a slot pair of `log` (uint64 device
    tensor of 2 * slots: earliest CTA start, latest CTA end); None turns
    the log off."""
    _check(_lib.qg_set_timing_log(_ptr(log), slots), "qg_set_timing_log")


def qg_timing_log_count() -> int:
    return int(_lib.qg_timing_log_count())


def qg_device_error() -> int:
    code = ctypes.c_int()
    _check(_lib.qg_device_error(ctypes.byref(code)), "qg_device_error")
    return code.value


def qg_last_error() -> str:
    return _lib.qg_last_error().decode()


def qg_version() -> str:
    return _lib.qg_version().decode()
