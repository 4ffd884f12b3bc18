"""qg_gemm_w8a8_noalloc: the allocation-free GEMM entry point.

Some callers cannot call cudaMalloc (a serving runtime or host framework that
owns the device allocator, a plugin that only receives its input and output
buffers, a latency-critical path that must not enter the allocator), so they
cannot hand qg_gemm_w8a8 a Split-K workspace.  qg_gemm_w8a8_noalloc keeps
that scratch in a static 4 MiB device array inside the library.  These tests
check, through the C ABI, that two calls in a row give the same output as the
workspace entry point (INT8: identical int32 accumulators and Y within one
bf16 ulp; FP8 formats: within 8e-3 * s_a*s_w*sum|a_q*w_q|), that a call
without Split-K needs no scratch, and that a shape whose scratch exceeds the
array is rejected with a clear error.

This file is collected last so that a run stopping at the first failure has
already run every other test; it passes alone in a fresh process as well.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gc():
    import gpu_cases
    return gpu_cases


@pytest.fixture(scope="module")
def q():
    from quantized_gemm_decode_02_b300 import qgemm
    return qgemm


def _inputs(gc, fmt, M, N, K, seed):
    import seeded_inputs as si
    A = si.activations(M, K, seed=seed, outliers=True).to(gc.DEV)
    W = torch.from_numpy(si.weights(N, K, seed=seed)).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu(fmt, W)
    Aq, sa = gc.quant_act_gpu(fmt, A)
    return Aq, sa, Wq, sw


def _close(orc, gc, fmt, Aq, sa, Wq, sw, Y, Y_ref, dbg, dbg_ref):
    if fmt == "W8A8_INT8":
        assert torch.equal(dbg, dbg_ref)
        assert gc.bf16_ulp_diff(gc.bf16_bits(Y), gc.bf16_bits(Y_ref)).max() <= 1
        return
    dt = gc.oracle_dtype(fmt)
    mag = orc.abs_magnitude(fmt, Aq.cpu().numpy().view(dt), sa.cpu().numpy(), Wq.cpu().numpy().view(dt),
                            sw.cpu().numpy())
    diff = (Y.float() - Y_ref.float()).abs().double().cpu().numpy()
    assert not np.isnan(diff).any()
    assert np.all(diff <= gc.FP8_BOUND * mag)


@pytest.mark.parametrize("fmt", ["W8A8_INT8", "FP8_Dynamic", "Block_FP8"])
def test_noalloc_matches_workspace_entry_point_on_two_calls(orc, gc, q, fmt):
    # 20 K ranges: more than a thread-block cluster reduces, so the partials
    # go through the scratch array (491,776 bytes of the 4 MiB)
    M, N, K, S = 16, 384, 4096, 20
    assert q.qg_workspace_bytes(fmt, M, N, K, q.QG_SWAPAB_SPLITK, S) > 0
    Aq, sa, Wq, sw = _inputs(gc, fmt, M, N, K, seed=31)
    is_int8 = fmt == "W8A8_INT8"
    Y_ref, dbg_ref = gc.gemm_gpu(fmt, Aq, sa, Wq, sw, N, q.QG_SWAPAB_SPLITK, S, debug=is_int8)
    torch.cuda.synchronize()
    for _ in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=gc.DEV)
        dbg = torch.full((M, N), -7, dtype=torch.int32, device=gc.DEV) if is_int8 else None
        q.qg_gemm_w8a8_noalloc(fmt, M, N, K, Aq, sa, Wq, sw, Y, N, q.QG_SWAPAB_SPLITK, S, 0, dbg)
        torch.cuda.synchronize()
        _close(orc, gc, fmt, Aq, sa, Wq, sw, Y, Y_ref, dbg, dbg_ref)
    assert q.qg_device_error() == 0


def test_noalloc_without_split_k(orc, gc, q):
    fmt, M, N, K = "W8A8_INT8", 5, 260, 1024
    # no Split-K, and Split-K reduced inside a thread-block cluster, need no scratch
    assert q.qg_workspace_bytes(fmt, M, N, K, q.QG_SWAPAB, 1) == 0
    assert q.qg_workspace_bytes(fmt, M, N, K, q.QG_SWAPAB_SPLITK, 4) == 0
    Aq, sa, Wq, sw = _inputs(gc, fmt, M, N, K, seed=32)
    Y_ref, dbg_ref = gc.gemm_gpu(fmt, Aq, sa, Wq, sw, N, q.QG_SWAPAB, 1, debug=True)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=gc.DEV)
    dbg = torch.empty((M, N), dtype=torch.int32, device=gc.DEV)
    q.qg_gemm_w8a8_noalloc(fmt, M, N, K, Aq, sa, Wq, sw, Y, N, q.QG_SWAPAB, 1, 0, dbg)
    torch.cuda.synchronize()
    _close(orc, gc, fmt, Aq, sa, Wq, sw, Y, Y_ref, dbg, dbg_ref)


def test_noalloc_prewidened_activations(orc, gc, q):
    # QG_CONFIG_I8_PREWIDEN keeps its fp16 activation copy in the static
    # array too: the same accumulators as the workspace entry point, twice
    fmt, M, N, K = "W8A8_INT8", 100, 384, 2304
    cfg = q.config_id(prewiden=True)
    need = q.qg_workspace_bytes_config(fmt, M, N, K, q.QG_SWAPAB_SPLITK, 3, cfg)
    assert 0 < need <= q.QG_NOALLOC_SCRATCH_BYTES
    Aq, sa, Wq, sw = _inputs(gc, fmt, M, N, K, seed=33)
    Y_ref, dbg_ref = gc.gemm_gpu(fmt, Aq, sa, Wq, sw, N, q.QG_SWAPAB_SPLITK, 3, config_id=cfg, debug=True)
    torch.cuda.synchronize()
    for _ in range(2):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=gc.DEV)
        dbg = torch.full((M, N), -7, dtype=torch.int32, device=gc.DEV)
        q.qg_gemm_w8a8_noalloc(fmt, M, N, K, Aq, sa, Wq, sw, Y, N, q.QG_SWAPAB_SPLITK, 3, cfg, dbg)
        torch.cuda.synchronize()
        _close(orc, gc, fmt, Aq, sa, Wq, sw, Y, Y_ref, dbg, dbg_ref)
    assert q.qg_device_error() == 0


def test_noalloc_rejects_scratch_beyond_the_array(gc, q):
    M, N, K, S = 32, 12288, 4096, 17          # 17 * 32 * 12288 * 4 bytes = 25.5 MiB of partials
    need = q.qg_workspace_bytes("FP8_Dynamic", M, N, K, q.QG_SWAPAB_SPLITK, S)
    assert need > q.QG_NOALLOC_SCRATCH_BYTES
    d = torch.zeros(16, dtype=torch.uint8, device=gc.DEV)
    f = torch.zeros(4, dtype=torch.float32, device=gc.DEV)
    with pytest.raises(q.QGError) as e:
        q.qg_gemm_w8a8_noalloc("FP8_Dynamic", M, N, K, d, f, d, f, d, N, q.QG_SWAPAB_SPLITK, S)
    assert e.value.code == q.QG_ERR_WORKSPACE_TOO_SMALL
    assert "static" in str(e.value)
