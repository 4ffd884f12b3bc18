"""qg_linear_w8a8 in its two forms: activation quantization fused into the
GEMM kernel (QG_LAUNCH_FUSED_QUANT, or no A_q / s_a buffers), and the
quantization kernel followed by the GEMM (the default with buffers).

Against the CPU oracle on the same seeded inputs: the quantized activations
and scales the kernel writes out are bit-exact (the kernel divides with
Markstein's method, the oracle with one IEEE division: they must agree on
every code, including ties), INT8 accumulators are bit-exact and Y within one
bf16 ulp, FP8 within 8e-3 * s_a*s_w*sum|a_q*w_q|.  Against the two-kernel path
(qg_quant_act + qg_gemm_w8a8) with the same config: identical outputs.

Cases span one CTA per tile, Split-K in clusters (the per-token row maximum
is agreed across the cluster), Split-K through the workspace (each CTA reads
the whole row), blocks of 64 tokens, ragged N and K, and rows built so that
x / s falls exactly on E4M3 / int8 rounding ties."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import seeded_inputs as si

pytestmark = pytest.mark.gpu

SW, SWS, ST = 2, 3, 0


@pytest.fixture(scope="module")
def gc():
    import gpu_cases
    return gpu_cases


@pytest.fixture(scope="module")
def q():
    from quantized_gemm_decode_02_b300 import qgemm
    return qgemm


def tie_rows(fmt: str, M: int, K: int, rng) -> torch.Tensor:
    """Activations whose quotients x / s land on rounding ties: every row (for
    Block_FP8 every 1x128 group) has its maximum at a power of two times
    QMAX, so s is a power of two and x = s * midpoint is exact in bf16."""
    A = np.zeros((M, K), np.float32)
    if fmt == "W8A8_INT8":
        mids = (np.arange(-126, 127) + 0.5).astype(np.float32)   # k + 1/2
        qmax = 127.0
    else:
        codes = np.array([v for v in range(0x7F) if v not in (0x7F,)], np.uint8)
        from oracle import oracle as orc
        vals = np.unique(np.abs(orc.e4m3_decode(codes)))
        mids = ((vals[1:] + vals[:-1]) / 2).astype(np.float32)     # E4M3 rounding midpoints
        mids = np.concatenate([mids, -mids])
        qmax = 448.0
    span = 128 if fmt == "Block_FP8" else K                       # the scale's span: a 1x128 group or the row
    for m in range(M):
        for k0 in range(0, K, span):
            s = np.float32(2.0 ** int(rng.integers(-12, 4)))
            seg = rng.choice(mids, size=span) * s
            seg[int(rng.integers(0, span))] = qmax * s              # the maximum: s = amax / qmax exactly
            A[m, k0:k0 + span] = seg
    t = torch.from_numpy(A).to(torch.bfloat16)
    assert torch.equal(t.float(), torch.from_numpy(A)), "tie rows must be exact in bf16"
    return t


def run_linear(orc, gc, q, fmt, M, N, K, variant, split, seed, A=None, check_two_kernel=True, fused=True):
    dev = gc.DEV
    if A is None:
        A = si.activations(M, K, seed=seed, outliers=True)
    W = si.weights(N, K, seed=seed)
    Wq, sw = gc.quant_weight_gpu(fmt, torch.from_numpy(W).to(dev))
    Ad = A.to(dev)
    is_int8 = fmt == "W8A8_INT8"
    need = q.qg_workspace_bytes(fmt, M, N, K, variant, split)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=dev)
    Aq = torch.full((M, K), 0x5A, dtype=torch.uint8, device=dev)
    sa_shape = (M, K // 128) if fmt == "Block_FP8" else (M,)
    sa = torch.full(sa_shape, -1.0, dtype=torch.float32, device=dev)
    dbg = torch.full((M, N), -7, dtype=torch.int32, device=dev) if is_int8 else None
    q.qg_set_launch_flags(q.QG_LAUNCH_FUSED_QUANT if fused else 0)
    try:
        q.qg_linear_w8a8(fmt, M, N, K, Ad, K, Wq, sw, Y, N, variant, split, 0, ws, need, Aq, sa, dbg)
    finally:
        q.qg_set_launch_flags(0)
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    oAq, osa, oWq, osw = gc.check_quant(orc, fmt, A, W, Aq, sa, Wq, sw)
    gc.check_gemm(orc, fmt, oAq, osa, oWq, osw, Y, dbg)
    if check_two_kernel:
        Aq2, sa2 = gc.quant_act_gpu(fmt, Ad)
        Y2, dbg2 = gc.gemm_gpu(fmt, Aq2, sa2, Wq, sw, N, variant, split, debug=is_int8)
        torch.cuda.synchronize()
        assert torch.equal(Y, Y2), "fused and two-kernel outputs differ"
        if is_int8:
            assert torch.equal(dbg, dbg2)
    return Y


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8"])
@pytest.mark.parametrize("M,split", [(1, 1), (5, 3), (16, 8), (17, 2), (32, 16), (24, 17), (48, 5), (100, 3)])
def test_fused_linear(orc, gc, q, fmt, M, split):
    # K = 2320: 19 k-tiles, the last ragged (16 of 128 columns); ragged N
    run_linear(orc, gc, q, fmt, M, 328, 2320, SWS if split > 1 else SW, split, seed=400 + M + split)


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8"])
@pytest.mark.parametrize("split", [1, 4, 20])
def test_fused_quantization_ties(orc, gc, q, fmt, split):
    M, N, K = 32, 256, 2560
    rng = np.random.Generator(np.random.PCG64(77 + split))
    A = tie_rows(fmt, M, K, rng)
    run_linear(orc, gc, q, fmt, M, N, K, SWS if split > 1 else SW, split, seed=5, A=A)


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8"])
@pytest.mark.parametrize("split", [1, 3])
def test_fused_signed_zeros(orc, gc, q, fmt, split):
    # -0.0 quantizes to the E4M3 code 0x80 (its sign kept), +0.0 to 0x00
    M, N, K = 6, 256, 1024
    A = si.activations(M, K, seed=31, outliers=True)
    A[0, ::3] = -0.0
    A[1, 1::5] = 0.0
    A[2, :] = -0.0  # an all-zero row: s = 1, every code a signed zero
    run_linear(orc, gc, q, fmt, M, N, K, SWS if split > 1 else SW, split, seed=31, A=A)


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8"])
@pytest.mark.parametrize("K", [2560, 12288, 25600])
def test_quant_act_ties(orc, gc, fmt, K):
    # the activation quantization kernel on rows whose quotients land on
    # rounding ties, bit-exact against the oracle
    rng = np.random.Generator(np.random.PCG64(K))
    A = tie_rows(fmt, 8, K, rng)
    Aq, sa = gc.quant_act_gpu(fmt, A.to(gc.DEV))
    torch.cuda.synchronize()
    oAq, osa = orc.quant_act(fmt, si.bf16_to_f32_numpy(A))
    assert np.array_equal(Aq.cpu().numpy().view(gc.oracle_dtype(fmt)), oAq)
    assert np.array_equal(sa.cpu().numpy(), osa)


def test_fused_linear_without_optional_outputs(orc, gc, q):
    fmt, M, N, K = "W8A8_INT8", 8, 384, 2048
    A = si.activations(M, K, seed=9)
    W = si.weights(N, K, seed=9)
    Wq, sw = gc.quant_weight_gpu(fmt, torch.from_numpy(W).to(gc.DEV))
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=gc.DEV)
    q.qg_linear_w8a8(fmt, M, N, K, A.to(gc.DEV), K, Wq, sw, Y, N, SWS, 4)
    torch.cuda.synchronize()
    oAq, osa = orc.quant_act(fmt, si.bf16_to_f32_numpy(A))
    oWq, osw = orc.quant_weight(fmt, W)
    gc.check_gemm(orc, fmt, oAq, osa, oWq, osw, Y)


DP, DPS, STS = 4, 5, 1


@pytest.mark.parametrize("fmt,variant,split,M", [
    ("Block_FP8", SWS, 3, 12), ("Block_FP8", SW, 1, 12), ("FP8_Dynamic", ST, 1, 12), ("FP8_Dynamic", STS, 3, 40),
    ("FP8_Dynamic", SW, 1, 5), ("FP8_Dynamic", SWS, 4, 24), ("FP8_Dynamic", SWS, 18, 7),
    ("W8A8_INT8", SW, 1, 9), ("W8A8_INT8", SWS, 3, 32), ("W8A8_INT8", SWS, 18, 3),
    ("W8A8_INT8", DP, 1, 1), ("W8A8_INT8", DPS, 5, 4), ("W8A8_INT8", DPS, 18, 8)])
def test_two_kernel_linear(orc, gc, q, fmt, variant, split, M):
    # the quantization kernel writes the caller's buffers, the GEMM reads
    # them; every kernel family, every reduction (none, cluster, workspace);
    # K = 2304 (18 k-tiles)
    run_linear(orc, gc, q, fmt, M, 264, 2304, variant, split, seed=11 + M, fused=False)


@pytest.mark.parametrize("pdl", [False, True])
def test_two_kernel_linear_graph_replays(orc, gc, q, pdl):
    # a captured chain of linear layers (quantization + GEMM pairs, with and
    # without programmatic dependent launch) replayed many times: every
    # replay gives the results of a direct run
    dev = gc.DEV
    cases = [("W8A8_INT8", 1, DPS, 4), ("W8A8_INT8", 16, SWS, 3), ("FP8_Dynamic", 8, SWS, 5), ("Block_FP8", 4, SW, 1),
             ("FP8_Dynamic", 64, ST, 1), ("W8A8_INT8", 2, DP, 1)]
    N, K = 384, 2048
    layers = []
    for i, (fmt, M, v, s) in enumerate(cases):
        A = si.activations(M, K, seed=60 + i).to(dev)
        W = torch.from_numpy(si.weights(N, K, seed=60 + i)).to(dev)
        Wq, sw = gc.quant_weight_gpu(fmt, W)
        need = q.qg_workspace_bytes(fmt, M, N, K, v, s)
        ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
        Aq = torch.empty((M, K), dtype=torch.uint8, device=dev)
        sa = torch.empty((M, K // 128) if fmt == "Block_FP8" else (M,), dtype=torch.float32, device=dev)
        Y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        layers.append((fmt, M, v, s, A, Wq, sw, ws, need, Aq, sa, Y))
    stream = torch.cuda.Stream()

    def run_all():
        for (fmt, M, v, s, A, Wq, sw, ws, need, Aq, sa, Y) in layers:
            q.qg_linear_w8a8(fmt, M, N, K, A, K, Wq, sw, Y, N, v, s, 0, ws, need, Aq, sa, None, stream=stream)

    with torch.cuda.stream(stream):
        run_all()
    torch.cuda.synchronize()
    ref = [L[-1].clone() for L in layers]
    q.qg_set_launch_flags(q.QG_LAUNCH_PDL if pdl else 0)
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            run_all()
    finally:
        q.qg_set_launch_flags(0)
    for rep in range(40):
        for L in layers:
            L[-1].fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert q.qg_device_error() == 0
        for L, r in zip(layers, ref):
            assert torch.equal(L[-1], r), f"replay {rep}"


def test_linear_needs_buffers_when_not_fused(q, gc):
    d = torch.zeros(1024, dtype=torch.uint8, device=gc.DEV)
    f = torch.zeros(64, dtype=torch.float32, device=gc.DEV)
    for fmt, v, cfg in (("Block_FP8", ST, 0), ("W8A8_INT8", DP, 0), ("W8A8_INT8", SW, q.config_id(mma_sync=True))):
        with pytest.raises(q.QGError) as e:
            q.qg_linear_w8a8(fmt, 4, 128, 128, d, 128, d, f, d, 128, v, 1, cfg)
        assert e.value.code == q.QG_ERR_INVALID_ARG


@pytest.mark.parametrize("M,split", [(1, 1), (5, 3), (16, 8), (17, 2), (32, 16), (24, 17), (48, 5), (100, 3)])
def test_fused_linear_block_fp8(orc, gc, q, M, split):
    # Block_FP8 in one kernel: quantizer warps scale every 1x128 group
    # themselves; K = 2304 (18 k-tiles), ragged N; cluster and workspace
    # Split-K; 17 ranges through the workspace; blocks of 64 tokens above 64
    run_linear(orc, gc, q, "Block_FP8", M, 328, 2304, SWS if split > 1 else SW, split, seed=450 + M + split)


@pytest.mark.parametrize("split", [1, 4, 20])
def test_fused_block_fp8_ties_and_zeros(orc, gc, q, split):
    # groups whose quotients land on E4M3 rounding ties (per-group scales are
    # powers of two), signed zeros and an all-zero group
    M, N, K = 32, 256, 2560
    rng = np.random.Generator(np.random.PCG64(91 + split))
    A = tie_rows("Block_FP8", M, K, rng)
    A[0, :128] = -0.0
    A[1, 256:384] = 0.0
    A[2, ::7] = -0.0
    run_linear(orc, gc, q, "Block_FP8", M, N, K, SWS if split > 1 else SW, split, seed=6, A=A)


@pytest.mark.parametrize("ring", [2, 6, 12, 16])
def test_fused_block_fp8_ring_depths(orc, gc, q, ring):
    # the scale ring between the quantizer and promotion warps holds
    # stages + 4 k-tiles; a requested ring deeper than 12 is capped
    M, N, K = 20, 256, 4096
    A = si.activations(M, K, seed=70 + ring, outliers=True)
    W = si.weights(N, K, seed=70 + ring)
    Wq, sw = gc.quant_weight_gpu("Block_FP8", torch.from_numpy(W).to(gc.DEV))
    Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=gc.DEV)
    Aq = torch.empty((M, K), dtype=torch.uint8, device=gc.DEV)
    sa = torch.empty((M, K // 128), dtype=torch.float32, device=gc.DEV)
    q.qg_linear_w8a8("Block_FP8", M, N, K, A.to(gc.DEV), K, Wq, sw, Y, N, SW, 1, q.config_id(ring, fused=True),
                     None, 0, Aq, sa)
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    oAq, osa, oWq, osw = gc.check_quant(orc, "Block_FP8", A, W, Aq, sa, Wq, sw)
    gc.check_gemm(orc, "Block_FP8", oAq, osa, oWq, osw, Y)


def test_fused_quant_config_bit_selects_one_kernel(orc, gc, q):
    # with A_q / s_a buffers given, the table bit asks for the one-kernel
    # form: the GEMM writes the buffers itself (same codes as the
    # quantization kernel) and the outputs match the two-kernel form
    fmt, M, N, K = "Block_FP8", 9, 384, 2048
    A = si.activations(M, K, seed=71, outliers=True).to(gc.DEV)
    W = torch.from_numpy(si.weights(N, K, seed=71)).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu(fmt, W)
    outs = []
    for cfg in (0, q.config_id(fused=True)):
        Y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=gc.DEV)
        Aq = torch.full((M, K), 0x5A, dtype=torch.uint8, device=gc.DEV)
        sa = torch.full((M, K // 128), -1.0, dtype=torch.float32, device=gc.DEV)
        q.qg_linear_w8a8(fmt, M, N, K, A, K, Wq, sw, Y, N, SWS, 4, cfg, None, 0, Aq, sa)
        torch.cuda.synchronize()
        outs.append((Y, Aq, sa))
    assert torch.equal(outs[0][1], outs[1][1]) and torch.equal(outs[0][2], outs[1][2])
    assert torch.equal(outs[0][0], outs[1][0])
    assert q.qg_device_error() == 0
