"""Plain CPU oracle for the quantized decode GEMM -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this module.  The product
library never loads it and shares no code with it.

The arithmetic lives in ``qg_oracle.c`` (plain C, element by element, exact
int64 / fp64 accumulation); this module compiles it with gcc, marshals numpy
arrays through ctypes and splits large GEMMs over host threads (each thread
computes a disjoint set of output columns; ctypes releases the GIL for
the duration of each C call).  See the header of ``qg_oracle.c`` for the method's source,
"Building a High-Performance and Portable vLLM Linear Backend with Helion",
and for the readings taken where that page is silent.

Formats (the page's section "Helion Linear Backend > Scope"):
  ``"FP8_Dynamic"`` per-token E4M3 activations, per-channel E4M3 weights
  ``"W8A8_INT8"``   per-token int8 activations, per-channel int8 weights
  ``"Block_FP8"``   1x128 E4M3 activation groups, 128x128 E4M3 weight blocks
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "qg_oracle.c")
BUILD_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "libqg_oracle.so")

FORMATS = ("FP8_Dynamic", "W8A8_INT8", "Block_FP8")

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile qg_oracle.c into a shared library (strict IEEE: no fast-math,
    no FMA contraction).  Returns the library path."""
    os.makedirs(BUILD_DIR, exist_ok=True)
    if force or not os.path.exists(LIB_PATH) or os.path.getmtime(LIB_PATH) < os.path.getmtime(SRC):
        tmp = LIB_PATH + f".tmp{os.getpid()}"
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                        "-fno-fast-math", "-o", tmp, SRC, "-lm"], check=True)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        I = ctypes.c_int64
        lib.orc_e4m3_decode.restype = ctypes.c_double
        lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.orc_e4m3_encode.restype = ctypes.c_uint8
        lib.orc_e4m3_encode.argtypes = [ctypes.c_float]
        lib.orc_int8_encode.restype = ctypes.c_int8
        lib.orc_int8_encode.argtypes = [ctypes.c_float]
        lib.orc_bf16_from_double.restype = ctypes.c_uint16
        lib.orc_bf16_from_double.argtypes = [ctypes.c_double]
        for name in ("orc_quant_rows_fp8", "orc_quant_rows_int8", "orc_quant_groups_fp8", "orc_quant_blocks_fp8"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [P, I, I, P, P]
        for name in ("orc_gemm_int8", "orc_gemm_fp8", "orc_gemm_blockfp8"):
            getattr(lib, name).restype = None
            getattr(lib, name).argtypes = [P, P, P, P, I, I, P, I, P, P]
        lib.orc_abs_mag_fp8.restype = None
        lib.orc_abs_mag_fp8.argtypes = [P, P, P, P, I, I, P, I, ctypes.c_int, P]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _f32(x) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(x, dtype=np.float32))


# ------------------------------------------------------------------ scalars --

def e4m3_decode(codes) -> np.ndarray:
    """Decode E4M3FN codes (uint8 array) to float64, element by element."""
    lib = _load()
    c = np.asarray(codes, dtype=np.uint8)
    return np.array([lib.orc_e4m3_decode(int(v)) for v in c.ravel()], dtype=np.float64).reshape(c.shape)


def e4m3_encode(x) -> np.ndarray:
    """Encode fp32 values to E4M3FN codes (RNE, saturating to +-448)."""
    lib = _load()
    a = _f32(x)
    return np.array([lib.orc_e4m3_encode(float(v)) for v in a.ravel()], dtype=np.uint8).reshape(a.shape)


def int8_encode(x) -> np.ndarray:
    """Encode fp32 values to symmetric int8 (RNE, clamp to [-127, 127])."""
    lib = _load()
    a = _f32(x)
    return np.array([lib.orc_int8_encode(float(v)) for v in a.ravel()], dtype=np.int8).reshape(a.shape)


def bf16_from_double(y) -> np.ndarray:
    """Round fp64 values once to bf16 (RNE); returns uint16 bit patterns."""
    lib = _load()
    a = np.asarray(y, dtype=np.float64)
    return np.array([lib.orc_bf16_from_double(float(v)) for v in a.ravel()], dtype=np.uint16).reshape(a.shape)


def bf16_bits_to_f32(bits) -> np.ndarray:
    """Widen bf16 bit patterns (uint16) to float32 (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32)


# ------------------------------------------------------------- quantization --

def quant_act(fmt: str, A) -> tuple[np.ndarray, np.ndarray]:
    """Dynamic activation quantization of A [M, K] (fp32 values, e.g. widened
    bf16).  Returns (A_q [M, K] uint8 E4M3 codes or int8, s_a fp32) with s_a
    of shape [M] (FP8_Dynamic, W8A8_INT8) or [M, ceil(K/128)] (Block_FP8)."""
    lib = _load()
    A = _f32(A)
    M, K = A.shape
    if fmt == "FP8_Dynamic":
        q = np.empty((M, K), np.uint8); s = np.empty(M, np.float32)
        lib.orc_quant_rows_fp8(_ptr(A), M, K, _ptr(q), _ptr(s))
    elif fmt == "W8A8_INT8":
        q = np.empty((M, K), np.int8); s = np.empty(M, np.float32)
        lib.orc_quant_rows_int8(_ptr(A), M, K, _ptr(q), _ptr(s))
    elif fmt == "Block_FP8":
        q = np.empty((M, K), np.uint8); s = np.empty((M, (K + 127) // 128), np.float32)
        lib.orc_quant_groups_fp8(_ptr(A), M, K, _ptr(q), _ptr(s))
    else:
        raise ValueError(fmt)
    return q, s


def quant_weight(fmt: str, W) -> tuple[np.ndarray, np.ndarray]:
    """Static weight quantization of W [N, K] (fp32).  Returns (W_q [N, K],
    s_w) with s_w of shape [N] (per-channel) or [ceil(N/128), ceil(K/128)]
    (Block_FP8, 128x128 blocks)."""
    lib = _load()
    W = _f32(W)
    N, K = W.shape
    if fmt == "FP8_Dynamic":
        q = np.empty((N, K), np.uint8); s = np.empty(N, np.float32)
        lib.orc_quant_rows_fp8(_ptr(W), N, K, _ptr(q), _ptr(s))
    elif fmt == "W8A8_INT8":
        q = np.empty((N, K), np.int8); s = np.empty(N, np.float32)
        lib.orc_quant_rows_int8(_ptr(W), N, K, _ptr(q), _ptr(s))
    elif fmt == "Block_FP8":
        q = np.empty((N, K), np.uint8); s = np.empty(((N + 127) // 128, (K + 127) // 128), np.float32)
        lib.orc_quant_blocks_fp8(_ptr(W), N, K, _ptr(q), _ptr(s))
    else:
        raise ValueError(fmt)
    return q, s


# -------------------------------------------------------------------- GEMM --

def _split(ns: np.ndarray, parts: int):
    parts = max(1, min(parts, len(ns)))
    return [c for c in np.array_split(ns, parts) if len(c)]


def gemm(fmt: str, Aq, sa, Wq, sw, ns=None, threads: int | None = None):
    """Exact quantized GEMM for all M rows and the output columns ``ns``
    (default: every column).  Returns (acc, y) of shape [M, len(ns)]:
    acc is int64 (W8A8_INT8), the exact fp64 sum (FP8_Dynamic) or the scaled
    fp64 sum (Block_FP8); y holds the bf16 output bit patterns (uint16)."""
    lib = _load()
    Aq = np.ascontiguousarray(Aq); Wq = np.ascontiguousarray(Wq)
    sa = _f32(sa); sw = _f32(sw)
    M, K = Aq.shape
    N = Wq.shape[0]
    assert Wq.shape[1] == K
    ns = np.arange(N, dtype=np.int64) if ns is None else np.ascontiguousarray(np.asarray(ns, dtype=np.int64))
    assert ns.size == 0 or (ns.min() >= 0 and ns.max() < N)
    if fmt == "W8A8_INT8":
        fn, acc_t = lib.orc_gemm_int8, np.int64
        assert Aq.dtype == np.int8 and Wq.dtype == np.int8
    elif fmt == "FP8_Dynamic":
        fn, acc_t = lib.orc_gemm_fp8, np.float64
        assert Aq.dtype == np.uint8 and Wq.dtype == np.uint8
    elif fmt == "Block_FP8":
        fn, acc_t = lib.orc_gemm_blockfp8, np.float64
        assert Aq.dtype == np.uint8 and Wq.dtype == np.uint8
    else:
        raise ValueError(fmt)
    acc = np.empty((M, ns.size), acc_t)
    y = np.empty((M, ns.size), np.uint16)
    threads = threads or os.cpu_count() or 1
    chunks = _split(ns, threads if M * K * ns.size > (1 << 22) else 1)

    def run(chunk):
        a = np.empty((M, chunk.size), acc_t); b = np.empty((M, chunk.size), np.uint16)
        fn(_ptr(Aq), _ptr(sa), _ptr(Wq), _ptr(sw), M, K, _ptr(chunk), chunk.size, _ptr(a), _ptr(b))
        return a, b

    if len(chunks) <= 1:
        parts = [run(c) for c in chunks]
    else:
        with ThreadPoolExecutor(len(chunks)) as ex:
            parts = list(ex.map(run, chunks))
    col = 0
    for (a, b), c in zip(parts, chunks):
        acc[:, col:col + c.size] = a
        y[:, col:col + c.size] = b
        col += c.size
    return acc, y


def abs_magnitude(fmt: str, Aq, sa, Wq, sw, ns=None) -> np.ndarray:
    """For the FP8 formats: sum_k |a_q * w_q| with the format's scales applied
    (per-token x per-channel, or per 128-K group for Block_FP8), for every row
    and the listed columns.  It is the magnitude the FP8 accuracy bound
    multiplies."""
    lib = _load()
    Aq = np.ascontiguousarray(Aq); Wq = np.ascontiguousarray(Wq)
    sa = _f32(sa); sw = _f32(sw)
    M, K = Aq.shape
    N = Wq.shape[0]
    ns = np.arange(N, dtype=np.int64) if ns is None else np.ascontiguousarray(np.asarray(ns, dtype=np.int64))
    out = np.empty((M, ns.size), np.float64)
    blocked = 1 if fmt == "Block_FP8" else 0
    chunks = _split(ns, (os.cpu_count() or 1) if M * K * ns.size > (1 << 22) else 1)

    def run(chunk):
        o = np.empty((M, chunk.size), np.float64)
        lib.orc_abs_mag_fp8(_ptr(Aq), _ptr(sa), _ptr(Wq), _ptr(sw), M, K, _ptr(chunk), chunk.size, blocked, _ptr(o))
        return o

    with ThreadPoolExecutor(max(1, len(chunks))) as ex:
        parts = list(ex.map(run, chunks))
    col = 0
    for o, c in zip(parts, chunks):
        out[:, col:col + c.size] = o
        col += c.size
    return out
