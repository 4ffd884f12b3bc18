"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle on the same seeded inputs.

Tolerances (the accuracy contract of the path, restated):
  * quantizer outputs (A_q, s_a, W_q, s_w): bit-exact, both sides take the
    correctly rounded fp32 quotient and round-to-nearest-even encodes;
  * W8A8_INT8: the int32 accumulators bit-exact (debug output), Y within one
    bf16 ulp of the oracle (the GPU epilogue rounds three times in fp32, the
    oracle once from the exact value);
  * FP8_Dynamic / Block_FP8: |Y_gpu - y_exact| <= 8e-3 * magnitude, where the
    magnitude is s_a*s_w*sum_k|a_q*w_q| (per 128-K group for Block_FP8);
    and the tight bound that the arithmetic gives:
        |Y_gpu - y_exact| <= 2^-8 * |y_exact| + (K/16 + 8 + S) * 2^-23 * magnitude
    (one bf16 rounding of the fp32 result; E4M3 products are exact in fp32,
    and each fp32 addition that forms the sum -- one per MMA instruction of
    K = 32 into the accumulator, one per Block_FP8 promotion of a 128-K
    group with its fp32 scale product, one per Split-K partial, a few for
    the adder tree inside an instruction and the scale multiplications --
    is counted as one rounding of at most 2^-23 of the magnitude), plus the
    whole-output check that the relative RMS error stays within 2^-8, the
    size of a bf16 rounding: a scale that is 1% off fails both.
"""
from __future__ import annotations

import numpy as np
import torch

import seeded_inputs as si
from quantized_gemm_decode_02_b300 import qgemm as q

FP8_BOUND = 8e-3
MAX_SPLITS = 32  # Split-K partials added in any test configuration (the tight bound's S)

DEV = "cuda:0"


def quant_weight_gpu(fmt: str, W: torch.Tensor):
    N, K = W.shape
    Wq = torch.empty((N, K), dtype=torch.uint8, device=W.device)
    if fmt == "Block_FP8":
        sw = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=W.device)
    else:
        sw = torch.empty((N,), dtype=torch.float32, device=W.device)
    q.qg_quant_weight(fmt, W, N, K, Wq, sw)
    return Wq, sw


def quant_act_gpu(fmt: str, A: torch.Tensor):
    M, K = A.shape
    Aq = torch.empty((M, K), dtype=torch.uint8, device=A.device)
    if fmt == "Block_FP8":
        sa = torch.empty((M, K // 128), dtype=torch.float32, device=A.device)
    else:
        sa = torch.empty((M,), dtype=torch.float32, device=A.device)
    q.qg_quant_act(fmt, A, M, K, A.stride(0), Aq, sa)
    return Aq, sa


def gemm_gpu(fmt, Aq, sa, Wq, sw, N, variant, split_k, config_id=0, debug=False, Y=None, ws=None):
    M, K = Aq.shape
    if Y is None:
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=Aq.device)
    need = q.qg_workspace_bytes_config(fmt, M, N, K, variant, split_k, config_id)
    if need and ws is None:
        ws = torch.zeros(need, dtype=torch.uint8, device=Aq.device)
    dbg = torch.full((M, N), -7, dtype=torch.int32, device=Aq.device) if debug else None
    q.qg_gemm_w8a8(fmt, M, N, K, Aq, sa, Wq, sw, Y, Y.stride(0), variant, split_k, config_id,
                   ws, need, dbg)
    return Y, dbg


def oracle_dtype(fmt):
    return np.int8 if fmt == "W8A8_INT8" else np.uint8


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().view(torch.int16).numpy().view(np.uint16)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Distance in bf16 ulps between two bf16 bit arrays (same-sign values)."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, -(x & 0x7FFF), x)
    return np.abs(ordered(a) - ordered(b))


def check_quant(orc, fmt, A_cpu_bf16, W_cpu_f32, Aq, sa, Wq, sw, rows=None):
    """Bit-exact quantizer parity (optionally only for weight rows `rows`)."""
    A32 = si.bf16_to_f32_numpy(A_cpu_bf16)
    oAq, osa = orc.quant_act(fmt, A32)
    assert np.array_equal(Aq.cpu().numpy().view(oracle_dtype(fmt)), oAq), "A_q mismatch"
    assert np.array_equal(sa.cpu().numpy(), osa), "s_a mismatch"
    if rows is None:
        oWq, osw = orc.quant_weight(fmt, W_cpu_f32)
        assert np.array_equal(Wq.cpu().numpy().view(oracle_dtype(fmt)), oWq), "W_q mismatch"
        assert np.array_equal(sw.cpu().numpy(), osw), "s_w mismatch"
        return oAq, osa, oWq, osw
    return oAq, osa, None, None


def check_gemm(orc, fmt, oAq, osa, oWq, osw, Y, dbg=None, ns=None):
    """Compare GPU output Y (and INT8 debug accumulators) with the oracle for
    all rows and columns ns (default all)."""
    acc, y = orc.gemm(fmt, oAq, osa, oWq, osw, ns=ns)
    Yb = bf16_bits(Y)
    if ns is not None:
        Yb = Yb[:, ns]
    if fmt == "W8A8_INT8":
        if dbg is not None:
            d = dbg.cpu().numpy().astype(np.int64)
            if ns is not None:
                d = d[:, ns]
            assert np.array_equal(d, acc), f"int32 accumulators differ at {np.argwhere(d != acc)[:5].tolist()}"
        ud = bf16_ulp_diff(Yb, y)
        assert ud.max() <= 1, f"INT8 Y differs by {ud.max()} bf16 ulp"
        return
    mag = orc.abs_magnitude(fmt, oAq, osa, oWq, osw, ns=ns)
    if fmt == "Block_FP8":
        exact = acc
    else:
        exact = acc * osa.astype(np.float64)[:, None] * (osw.astype(np.float64)[None, :] if ns is None
                                                           else osw.astype(np.float64)[np.asarray(ns)][None, :])
    got = (Yb.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    err = np.abs(got - exact)
    bound = FP8_BOUND * mag
    bad = err > bound
    assert not np.isnan(got).any(), "NaN in output (unwritten element?)"
    assert not bad.any(), f"{bad.sum()} elements outside bound; worst ratio {np.max(err / np.maximum(bound, 1e-300)):.3g}"
    check_fp8_tight(exact, got, mag, oAq.shape[1])


def check_fp8_tight(exact, got, mag, K, splits=MAX_SPLITS):
    """The tight FP8 bound of the module docstring, element by element, and
    the relative RMS error of the whole output."""
    err = np.abs(got - exact)
    tight = 2.0 ** -8 * np.abs(exact) + (K / 16 + 8 + splits) * 2.0 ** -23 * mag
    bad = err > tight
    assert not bad.any(), (f"{bad.sum()} elements outside the tight bound; worst ratio "
                           f"{np.max(err / np.maximum(tight, 1e-300)):.3g}")
    ss = float((exact ** 2).sum())
    if ss > 0:
        rms = float(np.sqrt((err ** 2).sum() / ss))
        assert rms <= 2.0 ** -8, f"relative RMS error {rms:.3g} above 2^-8"


def run_case(orc, fmt, M, N, K, variant, split_k, seed=0, outliers=False, config_id=0, debug=True):
    A = si.activations(M, K, seed=seed, outliers=outliers)
    W = si.weights(N, K, seed=seed)
    Ad = A.to(DEV)
    Wd = torch.from_numpy(W).to(DEV)
    Wq, sw = quant_weight_gpu(fmt, Wd)
    Aq, sa = quant_act_gpu(fmt, Ad)
    Y, dbg = gemm_gpu(fmt, Aq, sa, Wq, sw, N, variant, split_k, config_id=config_id,
                      debug=(debug and fmt == "W8A8_INT8"))
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    oAq, osa, oWq, osw = check_quant(orc, fmt, A, W, Aq, sa, Wq, sw)
    check_gemm(orc, fmt, oAq, osa, oWq, osw, Y, dbg)
    return Y, dbg
