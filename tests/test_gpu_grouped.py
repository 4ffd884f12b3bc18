"""qg_gemm_w8a8_grouped (mixture-of-experts GEMM, "Future work > Model
coverage"): every group is one GEMM of the format over its own tokens and
weights, so each group's slice of the output is checked against the CPU
oracle's GEMM of that group alone (INT8 accumulators bit-exact and Y within
one bf16 ulp, FP8 within 8e-3 * s_a*s_w*sum|a_q*w_q|).  Groups include empty
ones and ragged token counts; N is ragged; Split-K reduces in a cluster or
through the workspace; more than 64 tokens in a group use several token
blocks."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu

SW, SWS, DP, DPS = 2, 3, 4, 5


@pytest.fixture(scope="module")
def gc():
    import gpu_cases
    return gpu_cases


@pytest.fixture(scope="module")
def q():
    from quantized_gemm_decode_02_b300 import qgemm
    return qgemm


def run_grouped(orc, gc, q, fmt, counts, N, K, variant, split, seed):
    dev = gc.DEV
    G = len(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    total, max_tokens = int(offs[-1]), max(1, int(max(counts)))
    A = si.activations(total, K, seed=seed, outliers=True)
    W = si.weights(G * N, K, seed=seed).reshape(G, N, K)
    Aq, sa = gc.quant_act_gpu(fmt, A.to(dev))
    Wq = torch.empty((G, N, K), dtype=torch.uint8, device=dev)
    sw_shape = (G, (N + 127) // 128, K // 128) if fmt == "Block_FP8" else (G, N)
    sw = torch.empty(sw_shape, dtype=torch.float32, device=dev)
    for g in range(G):  # one weight quantization per group (Block_FP8 blocks do not straddle groups)
        wq, s = gc.quant_weight_gpu(fmt, torch.from_numpy(np.ascontiguousarray(W[g])).to(dev))
        Wq[g].copy_(wq)
        sw[g].copy_(s.reshape(sw_shape[1:]))
    offs_d = torch.from_numpy(offs).to(dev)
    need = q.qg_workspace_bytes_grouped(fmt, G, total, max_tokens, N, K, variant, split)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    Y = torch.full((max(total, 1), N), float("nan"), dtype=torch.bfloat16, device=dev)
    is_int8 = fmt == "W8A8_INT8"
    dbg = torch.full((max(total, 1), N), -7, dtype=torch.int32, device=dev) if is_int8 else None
    q.qg_gemm_w8a8_grouped(fmt, G, offs_d, total, max_tokens, N, K, Aq, sa, Wq, sw, Y, N, variant, split, 0,
                           ws, need, dbg)
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    oAq, osa = orc.quant_act(fmt, si.bf16_to_f32_numpy(A))
    for g in range(G):
        t0, t1 = int(offs[g]), int(offs[g + 1])
        if t1 == t0:
            continue
        oWq, osw = orc.quant_weight(fmt, np.ascontiguousarray(W[g]))
        gc.check_gemm(orc, fmt, oAq[t0:t1], osa[t0:t1], oWq, osw, Y[t0:t1], None if dbg is None else dbg[t0:t1])
    return Y, dbg


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 3), (SWS, 18)])
def test_grouped(orc, gc, q, fmt, variant, split):
    run_grouped(orc, gc, q, fmt, [3, 0, 16, 1, 7], 300, 2304, variant, split, seed=700 + split)


@pytest.mark.parametrize("variant,split", [(DP, 1), (DPS, 4), (DPS, 18)])
def test_grouped_int8_dp4a(orc, gc, q, variant, split):
    run_grouped(orc, gc, q, "W8A8_INT8", [3, 0, 8, 1, 5, 2], 300, 2304, variant, split, seed=710 + split)


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8"])
def test_grouped_token_blocks(orc, gc, q, fmt):
    # 70 tokens in one group: blocks of 64 tokens, the second ragged
    run_grouped(orc, gc, q, fmt, [70, 5, 0], 264, 1024, SWS, 2, seed=720)


def test_grouped_equals_separate_gemms(orc, gc, q):
    # the grouped launch gives each group's output of the plain GEMM, bit for bit
    fmt, counts, N, K = "W8A8_INT8", [4, 9, 1], 256, 2048
    Y, dbg = run_grouped(orc, gc, q, fmt, counts, N, K, SWS, 2, seed=730)
    offs = np.concatenate([[0], np.cumsum(counts)])
    A = si.activations(int(offs[-1]), K, seed=730, outliers=True).to(gc.DEV)
    W = si.weights(len(counts) * N, K, seed=730).reshape(len(counts), N, K)
    Aq, sa = gc.quant_act_gpu(fmt, A)
    for g in range(len(counts)):
        t0, t1 = int(offs[g]), int(offs[g + 1])
        wq, s = gc.quant_weight_gpu(fmt, torch.from_numpy(np.ascontiguousarray(W[g])).to(gc.DEV))
        Yg, dg = gc.gemm_gpu(fmt, Aq[t0:t1].contiguous(), sa[t0:t1].contiguous(), wq, s, N, SWS, 2, debug=True)
        torch.cuda.synchronize()
        assert torch.equal(dg, dbg[t0:t1])
        assert torch.equal(Yg, Y[t0:t1])


@pytest.mark.parametrize("variant,split", [(SWS, 3), (SWS, 18), (DPS, 2)])
def test_grouped_tokens_beyond_max_are_left_out(orc, gc, q, variant, split):
    # a group with more tokens than max_tokens: its first max_tokens rows are
    # computed, the rest of Y stays untouched (no write outside the sized
    # token blocks and receive buffers)
    dev = gc.DEV
    fmt, N, K, counts, max_tokens = "W8A8_INT8", 256, 2304, [3, 11, 2], 4
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    total = int(offs[-1])
    A = si.activations(total, K, seed=740)
    W = si.weights(len(counts) * N, K, seed=740)
    Aq, sa = gc.quant_act_gpu(fmt, A.to(dev))
    Wq, sw = gc.quant_weight_gpu(fmt, torch.from_numpy(W).to(dev))
    need = q.qg_workspace_bytes_grouped(fmt, len(counts), total, max_tokens, N, K, variant, split)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    Y = torch.full((total, N), 7.0, dtype=torch.bfloat16, device=dev)
    q.qg_gemm_w8a8_grouped(fmt, len(counts), torch.from_numpy(offs).to(dev), total, max_tokens, N, K, Aq, sa, Wq,
                           sw, Y, N, variant, split, 0, ws, need)
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    oAq, osa = orc.quant_act(fmt, si.bf16_to_f32_numpy(A))
    oWq, osw = orc.quant_weight(fmt, W)
    for g in range(len(counts)):
        t0 = int(offs[g])
        t1 = min(int(offs[g + 1]), t0 + max_tokens)
        gc.check_gemm(orc, fmt, oAq[t0:t1], osa[t0:t1], oWq[g * N:(g + 1) * N], osw[g * N:(g + 1) * N], Y[t0:t1])
        assert torch.all(Y[t1:int(offs[g + 1])] == 7.0)


def test_grouped_validation(gc, q):
    d = torch.zeros(1 << 16, dtype=torch.uint8, device=gc.DEV)
    f = torch.ones(4096, dtype=torch.float32, device=gc.DEV)
    offs = torch.tensor([0, 2, 4], dtype=torch.int32, device=gc.DEV)
    with pytest.raises(q.QGError) as e:   # Standard variant
        q.qg_gemm_w8a8_grouped("FP8_Dynamic", 2, offs, 4, 2, 256, 256, d, f, d, f, d, 256, 0, 1)
    assert e.value.code == q.QG_ERR_INVALID_ARG
    with pytest.raises(q.QGError) as e:   # no offsets
        q.qg_gemm_w8a8_grouped("FP8_Dynamic", 2, None, 4, 2, 256, 256, d, f, d, f, d, 256, SW, 1)
    assert e.value.code == q.QG_ERR_INVALID_ARG
    with pytest.raises(q.QGError) as e:   # dp4a needs at most 8 tokens per group
        q.qg_gemm_w8a8_grouped("W8A8_INT8", 2, offs, 4, 9, 256, 256, d, f, d, f, d, 256, DP, 1)
    assert e.value.code == q.QG_ERR_UNSUPPORTED_SHAPE
    q.qg_gemm_w8a8_grouped("FP8_Dynamic", 2, offs, 0, 2, 256, 256, d, f, d, f, d, 256, SW, 1)  # no tokens: no-op
