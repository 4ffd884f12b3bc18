"""GPU parity at the benchmark's full sizes, in the launch configuration the
benchmark times (the committed tuned table through qg_select).

Weights are drawn on the device (N x K up to 51200 x 5120), quantized by the
library, and the oracle checks whole 128-row blocks of the output: the first,
one in the middle and the last.  For those rows it re-quantizes the same fp32
weights on the CPU (bit-exact codes and scales), recomputes the activations'
quantization (bit-exact) and the exact GEMM: INT8 accumulators bit-exact and
Y within one bf16 ulp; FP8 formats within 8e-3 * s_a*s_w*sum|a_q*w_q|.

Also covered: the M = 64..512 regime of every Qwen3-8B layer in the tuned
table's configuration, and the Standard variant with and without Split-K for
the E4M3 formats, with sampled rows."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TABLE = os.path.join(ROOT, "quantized_gemm_decode_02_b300", "tables", "b300.tsv")

# (format, model, token counts) of the benchmark's workloads
FULL = [
    ("W8A8_INT8", "Qwen3-1.7B", si.TUNED_M),
    ("FP8_Dynamic", "Qwen3-1.7B", (1,)),
    ("Block_FP8", "Qwen3-8B", (1, 7, 16, 17, 32)),
    ("FP8_Dynamic", "Qwen3-32B", (1, 8, 32)),
]
CASES = [(f, m, layer, M) for (f, m, ms) in FULL for layer in ("qkv", "o", "gate_up", "down") for M in ms
         if not (f == "FP8_Dynamic" and m == "Qwen3-1.7B" and layer != "o")]


@pytest.fixture(scope="module")
def gc():
    import gpu_cases
    return gpu_cases


@pytest.fixture(scope="module")
def q():
    from quantized_gemm_decode_02_b300 import qgemm
    qgemm.qg_load_table(TABLE)
    qgemm.qg_set_allow_default(True)
    yield qgemm
    qgemm.qg_set_allow_default(False)


def sampled_blocks(N: int) -> list[int]:
    nb = (N + 127) // 128
    return sorted({0, nb // 2, nb - 1})


def run_sampled(orc, gc, q, fmt, M, N, K, variant, split, cfg, seed, outliers=False):
    dev = gc.DEV
    A = si.activations(M, K, seed=seed, outliers=outliers)
    W = si.weights_device(N, K, seed=seed, device=dev)
    Wq, sw = gc.quant_weight_gpu(fmt, W)
    Aq, sa = gc.quant_act_gpu(fmt, A.to(dev))
    Y, dbg = gc.gemm_gpu(fmt, Aq, sa, Wq, sw, N, variant, split, config_id=cfg, debug=(fmt == "W8A8_INT8"))
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    blocks = sampled_blocks(N)
    rows = np.concatenate([np.arange(b * 128, min(N, b * 128 + 128)) for b in blocks])
    rows_t = torch.from_numpy(rows).to(dev)
    W_rows = W.index_select(0, rows_t).cpu().numpy()
    oWq, osw = orc.quant_weight(fmt, W_rows)
    dt = gc.oracle_dtype(fmt)
    assert np.array_equal(Wq.index_select(0, rows_t).cpu().numpy().view(dt), oWq), "W_q mismatch"
    if fmt == "Block_FP8":
        assert np.array_equal(sw.cpu().numpy()[blocks], osw), "s_w mismatch"
    else:
        assert np.array_equal(sw.cpu().numpy()[rows], osw), "s_w mismatch"
    oAq, osa = orc.quant_act(fmt, si.bf16_to_f32_numpy(A))
    assert np.array_equal(Aq.cpu().numpy().view(dt), oAq), "A_q mismatch"
    assert np.array_equal(sa.cpu().numpy(), osa), "s_a mismatch"
    Y_rows = Y.index_select(1, rows_t)
    dbg_rows = dbg.index_select(1, rows_t) if dbg is not None else None
    gc.check_gemm(orc, fmt, oAq, osa, oWq, osw, Y_rows, dbg_rows)


@pytest.mark.parametrize("fmt,model,layer,M", CASES)
def test_full_size_sampled_parity(orc, gc, q, fmt, model, layer, M):
    K, N = si.QWEN3_LINEARS[model][layer]
    variant, split, cfg = q.qg_select(fmt, M, N, K)
    run_sampled(orc, gc, q, fmt, M, N, K, variant, split, cfg, seed=1000 + M, outliers=(fmt == "Block_FP8"))


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
@pytest.mark.parametrize("M", [64, 100, 256, 512])
def test_large_token_counts(orc, gc, q, fmt, M):
    # Qwen3-8B o_proj shape: the config the table selects, and (E4M3 formats)
    # the Standard variant with and without Split-K
    K, N = si.QWEN3_LINEARS["Qwen3-8B"]["o"]
    variant, split, cfg = q.qg_select(fmt, M, N, K)
    run_sampled(orc, gc, q, fmt, M, N, K, variant, split, cfg, seed=2000 + M, outliers=True)
    if fmt != "W8A8_INT8":
        for v, sp in ((q.QG_STANDARD, 1), (q.QG_SPLITK, 3)):
            run_sampled(orc, gc, q, fmt, M, N, K, v, sp, 0, seed=2100 + M, outliers=True)


LARGE_M = [(f, layer, M) for f in ("FP8_Dynamic", "W8A8_INT8", "Block_FP8") for layer in ("qkv", "o", "gate_up", "down")
           for M in (64, 128, 256, 384, 512) if not (layer == "o" and M in (64, 256, 512))]


@pytest.mark.parametrize("fmt,layer,M", LARGE_M)
def test_large_m_table_configs(orc, gc, q, fmt, layer, M):
    # every Qwen3-8B layer at M = 64..512 in the configuration the tuned
    # table selects (persistent FP8 tiles of 192..256 weight rows, CTA pairs,
    # Block_FP8 promotion with eight warps, Swap-AB token blocks for INT8)
    K, N = si.QWEN3_LINEARS["Qwen3-8B"][layer]
    variant, split, cfg = q.qg_select(fmt, M, N, K)
    run_sampled(orc, gc, q, fmt, M, N, K, variant, split, cfg, seed=4000 + M, outliers=(fmt == "Block_FP8"))


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
@pytest.mark.parametrize("M,split", [(65, 1), (130, 3), (200, 20)])
def test_swap_ab_token_blocks(orc, gc, fmt, M, split):
    # more than 64 tokens through Swap-AB: blocks of 64 with a ragged last
    # block; split 3 reduces in a cluster, split 20 through the workspace
    SW, SWS = 2, 3
    gc.run_case(orc, fmt, M, 264, 2560, SW if split == 1 else SWS, split, seed=3000 + M)
