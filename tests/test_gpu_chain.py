"""GPU parity of the benchmark's chained step: all three formats on one
Qwen3-8B layer's four linears, captured into one CUDA graph with
programmatic dependent launch, as `bench.py --workload layer_qwen3_8b` runs
it (shared weights, activations with 1% outliers x20), on a slice of its
token counts: M in {1, 17, 32}.

Under programmatic dependent launch a GEMM starts streaming its weights
before the kernel ahead of it has finished, so an ordering fault across
formats (a GEMM reading activation codes or scales that its quantization
kernel has not written yet, or a quantization kernel overwriting codes a
GEMM still reads) shows only in such a chain.  Every GEMM's output is
checked against the oracle on whole sampled 128-column blocks (the first,
a middle and the last block of N): the oracle quantizes the same seeded
fp32 weights and bf16 activations itself; W8A8_INT8 within one bf16 ulp,
the FP8 formats within the FP8 bound.  Two replays in a row must give
identical outputs."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu

MS = (1, 17, 32)


@pytest.fixture(scope="module")
def gc():
    import gpu_cases
    return gpu_cases


@pytest.fixture(scope="module")
def chain():
    import bench
    items = [(f, "Qwen3-8B", layer, M) for f in bench.FORMATS for M in MS for layer in bench.LAYERS]
    wl = bench.Workload("layer_qwen3_8b", "cuda:0", seed=0, pdl=True, items=items)
    stream = torch.cuda.Stream(device="cuda:0")
    graph = wl.capture_step(stream)
    outs = []
    for _ in range(2):
        wl.Y_all.fill_(0xFF)          # NaN in every bf16 output
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        outs.append(wl.Y_all.clone())
    assert wl.q.qg_device_error() == 0
    yield wl, outs
    del graph


def test_chain_replays_are_identical(chain):
    wl, outs = chain
    assert torch.equal(outs[0], outs[1])


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
def test_chain_outputs_match_the_oracle(orc, gc, chain, fmt):
    wl, outs = chain
    for r in wl.recs:
        if r["fmt"] != fmt:
            continue
        M, N, K = r["M"], r["N"], r["K"]
        nb = (N + 127) // 128
        blocks = sorted({0, nb // 2, nb - 1})
        cols = np.concatenate([np.arange(b * 128, min(N, b * 128 + 128)) for b in blocks])
        cols_t = torch.from_numpy(cols).to(gc.DEV)
        W = si.weights_device(N, K, seed=r["wseed"], device=gc.DEV)
        W_rows = W.index_select(0, cols_t).cpu().numpy()
        del W
        # the sample is made of whole 128-row blocks (N is a multiple of 128
        # on these shapes), so for Block_FP8 the oracle's block j of the
        # sample is weight block blocks[j] of the GEMM
        oWq, osw = orc.quant_weight(fmt, W_rows)
        oAq, osa = orc.quant_act(fmt, si.bf16_to_f32_numpy(r["A"]))
        gc.check_gemm(orc, fmt, oAq, osa, oWq, osw, r["Y"].index_select(1, cols_t))
