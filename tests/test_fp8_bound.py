"""The FP8 parity checker itself, on the CPU: an output that is the exact
GEMM rounded once to bf16 passes the tight bound and the RMS check of
tests/gpu_cases.py, and outputs with a planted error (a 1% scale error, a
dropped 128-K tile, a wrong per-token scale) fail them.  The errors are
planted into the oracle's exact values, never into GPU results."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import seeded_inputs as si


def _bf16(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


@pytest.fixture(scope="module")
def gc():
    import gpu_cases
    return gpu_cases


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "Block_FP8"])
@pytest.mark.parametrize("K", [256, 4096])
def test_tight_bound_accepts_one_rounding_and_rejects_planted_errors(orc, gc, fmt, K):
    M, N = 8, 256
    A = si.bf16_to_f32_numpy(si.activations(M, K, seed=K + 1, outliers=True))
    W = si.weights(N, K, seed=K + 2)
    Aq, sa = orc.quant_act(fmt, A)
    Wq, sw = orc.quant_weight(fmt, W)
    acc, _ = orc.gemm(fmt, Aq, sa, Wq, sw)
    mag = orc.abs_magnitude(fmt, Aq, sa, Wq, sw)
    exact = acc if fmt == "Block_FP8" else acc * sa.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
    gc.check_fp8_tight(exact, _bf16(exact), mag, K)                    # one bf16 rounding: passes
    with pytest.raises(AssertionError):
        gc.check_fp8_tight(exact, _bf16(exact * 1.01), mag, K)         # a scale 1% off
    # the last 128-K tile left out of every sum
    Wq_cut = Wq.copy()
    Wq_cut[:, K - 128:] = 0
    acc_cut, _ = orc.gemm(fmt, Aq, sa, Wq_cut, sw)
    cut = acc_cut if fmt == "Block_FP8" else acc_cut * sa.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :]
    with pytest.raises(AssertionError):
        gc.check_fp8_tight(exact, _bf16(cut), mag, K)
    # one token's output scaled by the next token's scale
    if fmt == "FP8_Dynamic":
        wrong = exact.copy()
        wrong[0] = exact[0] * float(sa[1]) / float(sa[0])
        with pytest.raises(AssertionError):
            gc.check_fp8_tight(exact, _bf16(wrong), mag, K)
