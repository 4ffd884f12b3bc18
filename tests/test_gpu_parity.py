"""GPU parity: the sm_103a kernels, called through the C ABI, against the CPU
oracle on the same seeded inputs (quantizers bit-exact; INT8 accumulators
bit-exact and Y within 1 bf16 ulp; FP8 within 8e-3 * s_a*s_w*sum|a_q*w_q|).

Sizes here span several 128-row tiles, a ragged N tail, ragged K (FP8) and
several 1024-K exactness segments (INT8), with M over the decode range."""
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


SW, SWS, ST, STS = 2, 3, 0, 1  # Swap-AB, Swap-AB+Split-K, Standard, Split-K


@pytest.mark.parametrize("M", [1, 5, 16, 17, 32])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 3), (ST, 1), (STS, 2)])
def test_fp8_dynamic(orc, gc, M, variant, split):
    gc.run_case(orc, "FP8_Dynamic", M, 424, 656, variant, split, seed=M)


@pytest.mark.parametrize("M", [1, 40, 128, 129, 300])
@pytest.mark.parametrize("variant,split,ring", [(ST, 1, 0), (STS, 3, 0), (ST, 1, 4), (STS, 2, 3)])
def test_fp8_dynamic_wide_tiles(orc, q, gc, M, variant, split, ring):
    # 256-row weight tiles: N = 424 gives one full and one ragged wide tile;
    # M spans several 128-token tiles (ragged); Split-K through the workspace
    gc.run_case(orc, "FP8_Dynamic", M, 424, 656, variant, split, seed=50 + M, config_id=q.config_id(ring, 0, True))


def test_wide_tiles_rejected_outside_fp8_standard(q, gc):
    d = torch.zeros(1 << 16, dtype=torch.uint8, device=gc.DEV)
    f = torch.ones(4096, dtype=torch.float32, device=gc.DEV)
    for fmt, v in (("FP8_Dynamic", SW), ("Block_FP8", ST), ("W8A8_INT8", SW)):
        with pytest.raises(q.QGError) as e:
            q.qg_gemm_w8a8(fmt, 8, 256, 256, d, f, d, f, d, 256, v, 1, q.config_id(0, 0, True))
        assert e.value.code == q.QG_ERR_INVALID_ARG


@pytest.mark.parametrize("M", [1, 7, 16, 24, 32])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 2), (SWS, 5), (ST, 1), (STS, 3)])
def test_block_fp8(orc, gc, M, variant, split):
    gc.run_case(orc, "Block_FP8", M, 392, 768, variant, split, seed=100 + M)


@pytest.mark.parametrize("M", [5, 20, 48])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 2)])
def test_block_fp8_long_k_ranges(orc, gc, M, variant, split):
    # K ranges whose scale products (k-tiles x token block) exceed the
    # staged table of 1024: the promotion stages them in chunks of 32, 16 or
    # 8 k-tiles (blocks of 16, 32, 64 tokens), 73 k-tiles per range, so the
    # last chunk is ragged and both halves of the table are reused; split 2
    # reduces in a cluster
    K = 73 * 128 * split
    gc.run_case(orc, "Block_FP8", M, 264, K, variant, split, seed=4100 + M + split)


@pytest.mark.parametrize("M,N,K,split", [(33, 264, 4608, 1), (200, 392, 2560, 1), (130, 264, 3840, 3),
                                           (300, 136, 1280, 6)])
def test_block_fp8_standard_register_promotion(orc, gc, M, N, K, split):
    # the Standard kernel's Block_FP8 promotion: four partial buffers, eight
    # promotion warps with register accumulators; ragged token and weight
    # tiles, long K ranges, Split-K through the workspace
    gc.run_case(orc, "Block_FP8", M, N, K, ST if split == 1 else STS, split, seed=4500 + M)


@pytest.mark.parametrize("M,K,variant,split", [(1, 768, SW, 1), (7, 768, SWS, 2), (16, 768, SWS, 5),
                                               (24, 3840, SWS, 20), (32, 768, SW, 1), (5, 9344, SW, 1),
                                               (20, 9344, SW, 1), (48, 18688, SWS, 2), (65, 2560, SW, 1),
                                               (130, 2560, SWS, 3), (200, 2560, SWS, 20), (257, 4096, SW, 1)])
def test_block_fp8_eight_promotion_warps(orc, gc, q, M, K, variant, split):
    # QG_CONFIG_BLOCK_PROMO8: two promotion warps per TMEM lane quarter, each
    # with half of the token block (blocks of 16, 32, 64), through every
    # reduction (none, cluster, workspace), staged and chunked scale
    # products, ragged token blocks and weight tiles
    gc.run_case(orc, "Block_FP8", M, 264, K, variant, split, seed=4300 + M,
                config_id=q.config_id(promo8=True))


@pytest.mark.parametrize("variant,promo8", [(SW, False), (SW, True), (ST, False)])
def test_block_fp8_chunked_promotion_timeout(orc, gc, q, variant, promo8):
    # a forced wait time-out on the chunked promotion path (four or eight
    # promotion warps; and the Standard kernel's eight promotion warps): the
    # warps that gave up still pass every chunk barrier, the time-out is
    # reported, and the context stays usable
    import seeded_inputs as si
    M, N, K = 20, 256, 4608  # 36 k-tiles x a 32-token block > 1024 products
    cfg = q.config_id(promo8=promo8)
    A = si.activations(M, K, seed=3)
    W = si.weights(N, K, seed=3)
    Ad, Wd = A.to(gc.DEV), torch.from_numpy(W).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu("Block_FP8", Wd)
    Aq, sa = gc.quant_act_gpu("Block_FP8", Ad)
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    q.qg_set_wait_limit_ns(2_000_000)  # 2 ms
    q.qg_set_force_timeout(True)
    try:
        gc.gemm_gpu("Block_FP8", Aq, sa, Wq, sw, N, variant, 1, config_id=cfg)
        assert q.qg_device_error() == q.QG_ERR_DEVICE_TIMEOUT
    finally:
        q.qg_set_force_timeout(False)
        q.qg_set_wait_limit_ns(0)
    assert q.qg_device_error() == 0
    Y, _ = gc.gemm_gpu("Block_FP8", Aq, sa, Wq, sw, N, variant, 1, config_id=cfg)
    torch.cuda.synchronize()
    oAq, osa, oWq, osw = gc.check_quant(orc, "Block_FP8", A, W, Aq, sa, Wq, sw)
    gc.check_gemm(orc, "Block_FP8", oAq, osa, oWq, osw, Y)


@pytest.mark.parametrize("M", [1, 3, 16, 20, 32, 48])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 2), (SWS, 7)])
def test_w8a8_int8(orc, gc, M, variant, split):
    # K = 2304: 18 k-tiles -> three exact 1024-K segments at split 1
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=200 + M, outliers=True)


DP, DPS = 4, 5  # the CUDA-core (dp4a) forms of Swap-AB and Swap-AB+Split-K


@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("variant,split", [(DP, 1), (DPS, 2), (DPS, 7), (DPS, 16), (DPS, 18)])
def test_w8a8_int8_dp4a(orc, gc, M, variant, split):
    # K = 2304 (18 k-tiles); 16 ranges reduce in a cluster, 18 through the
    # workspace; ragged N; the int32 accumulators bit-exact
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=250 + M, outliers=True)


@pytest.mark.parametrize("fmt,M,variant,split", [("FP8_Dynamic", 3, SWS, 2), ("FP8_Dynamic", 40, STS, 2),
                                                  ("Block_FP8", 9, SW, 1), ("W8A8_INT8", 20, SWS, 3),
                                                  ("W8A8_INT8", 2, DPS, 3)])
@pytest.mark.parametrize("dist", [1, 4, 64])
def test_l2_prefetch_distance(orc, q, gc, fmt, M, variant, split, dist):
    # the prefetch distance only adds L2 requests ahead of the ring (64:
    # beyond every CTA's K range); results stay those of the oracle
    gc.run_case(orc, fmt, M, 300, 2304, variant, split, seed=400 + dist, config_id=q.config_id(0, dist))


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
@pytest.mark.parametrize("split", [2, 8, 9, 13, 14, 16, 17])
def test_split_k_cluster_and_workspace_reductions(orc, gc, fmt, split):
    # 2..16 ranges reduce across a thread-block cluster (9..16: non-portable
    # cluster sizes; 13 and 14 leave the last CTA few or no rows), 17 through
    # the workspace.  K = 2304 (18 k-tiles), ragged N, M across 32.
    M = 24 if fmt != "Block_FP8" else 19
    gc.run_case(orc, fmt, M, 328, 2304, SWS, split, seed=300 + split)


def test_int8_accumulators_identical_across_variants(gc):
    import seeded_inputs as si
    M, N, K = 32, 256, 4096
    A = si.activations(M, K, seed=5, outliers=True).to(gc.DEV)
    W = torch.from_numpy(si.weights(N, K, seed=5)).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu("W8A8_INT8", W)
    Aq, sa = gc.quant_act_gpu("W8A8_INT8", A)
    outs = [gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, v, s, debug=True) for v, s in
            [(SW, 1), (SWS, 2), (SWS, 3), (SWS, 8), (SWS, 32)]]
    torch.cuda.synchronize()
    for Y, d in outs[1:]:
        assert torch.equal(d, outs[0][1])
        assert torch.equal(Y, outs[0][0])


@pytest.mark.parametrize("M", [1, 4, 8])
def test_int8_dp4a_and_tensor_core_variants_identical(gc, M):
    # the CUDA-core (dp4a) and the tensor-core (exact fp32 segments) forms of
    # Swap-AB compute the same int32 accumulators and the same Y
    import seeded_inputs as si
    N, K = 384, 4096
    A = si.activations(M, K, seed=15 + M, outliers=True).to(gc.DEV)
    W = torch.from_numpy(si.weights(N, K, seed=15 + M)).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu("W8A8_INT8", W)
    Aq, sa = gc.quant_act_gpu("W8A8_INT8", A)
    outs = [gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, v, s, debug=True) for v, s in
            [(SW, 1), (SWS, 4), (DP, 1), (DPS, 3), (DPS, 16), (DPS, 32)]]
    torch.cuda.synchronize()
    for Y, d in outs[1:]:
        assert torch.equal(d, outs[0][1])
        assert torch.equal(Y, outs[0][0])


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "Block_FP8", "W8A8_INT8"])
def test_split_k_is_deterministic(gc, fmt):
    import seeded_inputs as si
    M, N, K = 16, 384, 2048
    A = si.activations(M, K, seed=9).to(gc.DEV)
    W = torch.from_numpy(si.weights(N, K, seed=9)).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu(fmt, W)
    Aq, sa = gc.quant_act_gpu(fmt, A)
    ys = [gc.gemm_gpu(fmt, Aq, sa, Wq, sw, N, SWS, 5)[0] for _ in range(4)]
    for y in ys[1:]:
        assert torch.equal(y, ys[0])


def test_zero_rows_and_columns(orc, gc):
    import seeded_inputs as si
    for fmt in ("FP8_Dynamic", "W8A8_INT8", "Block_FP8"):
        M, N, K = 6, 260, 512
        A = si.activations(M, K, seed=3)
        A[2] = 0
        W = si.weights(N, K, seed=3)
        W[7] = 0
        W[130:140] = 0
        Ad, Wd = A.to(gc.DEV), torch.from_numpy(W).to(gc.DEV)
        Wq, sw = gc.quant_weight_gpu(fmt, Wd)
        Aq, sa = gc.quant_act_gpu(fmt, Ad)
        Y, dbg = gc.gemm_gpu(fmt, Aq, sa, Wq, sw, N, SWS, 2, debug=fmt == "W8A8_INT8")
        torch.cuda.synchronize()
        Yc = Y.float().cpu()
        assert torch.all(Yc[2] == 0) and torch.all(Yc[:, 7] == 0)
        oAq, osa, oWq, osw = gc.check_quant(orc, fmt, A, W, Aq, sa, Wq, sw)
        gc.check_gemm(orc, fmt, oAq, osa, oWq, osw, Y, dbg)


def test_output_stride_and_untouched_padding(gc):
    import seeded_inputs as si
    M, N, K, ldy = 9, 200, 384, 264
    A = si.activations(M, K, seed=4).to(gc.DEV)
    W = torch.from_numpy(si.weights(N, K, seed=4)).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu("FP8_Dynamic", W)
    Aq, sa = gc.quant_act_gpu("FP8_Dynamic", A)
    big = torch.full((M, ldy), 123.0, dtype=torch.bfloat16, device=gc.DEV)
    gc.gemm_gpu("FP8_Dynamic", Aq, sa, Wq, sw, N, SWS, 3, Y=big)
    ref, _ = gc.gemm_gpu("FP8_Dynamic", Aq, sa, Wq, sw, N, SW, 1)
    torch.cuda.synchronize()
    assert torch.all(big[:, N:] == 123.0)
    assert torch.allclose(big[:, :N].float(), ref.float(), rtol=1e-2, atol=1e-3)


def test_m_zero_is_a_noop(q, gc):
    d = torch.zeros(16, dtype=torch.uint8, device=gc.DEV)
    f = torch.zeros(4, dtype=torch.float32, device=gc.DEV)
    q.qg_quant_act("FP8_Dynamic", d, 0, 16, 16, d, f)
    q.qg_gemm_w8a8("FP8_Dynamic", 0, 16, 16, d, f, d, f, d, 16, SW, 1)
    torch.cuda.synchronize()


def test_graph_capture_and_pdl_replay(orc, gc, q):
    import seeded_inputs as si
    fmt, M, N, K = "W8A8_INT8", 8, 512, 2048
    A = si.activations(M, K, seed=12)
    W = si.weights(N, K, seed=12)
    Ad = A.to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu(fmt, torch.from_numpy(W).to(gc.DEV))
    Aq = torch.empty((M, K), dtype=torch.uint8, device=gc.DEV)
    sa = torch.empty((M,), dtype=torch.float32, device=gc.DEV)
    Y = torch.empty((M, N), dtype=torch.bfloat16, device=gc.DEV)
    need = q.qg_workspace_bytes(fmt, M, N, K, SWS, 4)
    ws = torch.zeros(need, dtype=torch.uint8, device=gc.DEV)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    q.qg_set_launch_flags(q.QG_LAUNCH_PDL)
    try:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            for _ in range(3):
                q.qg_quant_act(fmt, Ad, M, K, K, Aq, sa)
                q.qg_gemm_w8a8(fmt, M, N, K, Aq, sa, Wq, sw, Y, N, SWS, 4, 0, ws, need)
        for _ in range(3):
            Y.fill_(float("nan"))
            g.replay()
            torch.cuda.synchronize()
            oAq, osa, oWq, osw = gc.check_quant(orc, fmt, A, W, Aq, sa, Wq, sw)
            gc.check_gemm(orc, fmt, oAq, osa, oWq, osw, Y)
    finally:
        q.qg_set_launch_flags(0)
    assert q.qg_device_error() == 0


@pytest.mark.parametrize("fmt,mma_sync", [("FP8_Dynamic", False), ("W8A8_INT8", False), ("W8A8_INT8", True),
                                          ("W8A8_INT8", "s8"), ("W8A8_INT8", "conv16"), ("Block_FP8", False)])
def test_bounded_wait_reports_timeout_and_context_survives(orc, gc, q, fmt, mma_sync):
    import seeded_inputs as si
    M, N, K = 4, 256, 1024
    A = si.activations(M, K, seed=1)
    W = si.weights(N, K, seed=1)
    Ad, Wd = A.to(gc.DEV), torch.from_numpy(W).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu(fmt, Wd)
    Aq, sa = gc.quant_act_gpu(fmt, Ad)
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    q.qg_set_wait_limit_ns(2_000_000)  # 2 ms
    q.qg_set_force_timeout(True)
    cfg = q.config_id(0, 0, mma_sync=mma_sync is True, s8=mma_sync == "s8", conv16=mma_sync == "conv16")
    try:
        gc.gemm_gpu(fmt, Aq, sa, Wq, sw, N, SW, 1, config_id=cfg)
        assert q.qg_device_error() == q.QG_ERR_DEVICE_TIMEOUT
    finally:
        q.qg_set_force_timeout(False)
        q.qg_set_wait_limit_ns(0)
    assert q.qg_device_error() == 0
    Y, dbg = gc.gemm_gpu(fmt, Aq, sa, Wq, sw, N, SW, 1, config_id=cfg, debug=fmt == "W8A8_INT8")
    torch.cuda.synchronize()
    oAq, osa, oWq, osw = gc.check_quant(orc, fmt, A, W, Aq, sa, Wq, sw)
    gc.check_gemm(orc, fmt, oAq, osa, oWq, osw, Y, dbg)


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
def test_scales_exact_across_binades(orc, gc, q, fmt):
    # every scale amax / qmax (448 or 127; Markstein's method with the
    # constant's reciprocal, __fdiv_rn below amax = 2^-100) equals the oracle's
    # IEEE quotient, and so do the codes: fp32 weight rows / 128x128 blocks
    # (full 24-bit mantissas) and bf16 activation rows / 1x128 groups whose
    # maxima span 2^-126 .. 2^125, across the 2^-100 threshold
    import seeded_inputs as si
    rng = np.random.default_rng(11)
    R, K = 512, 256
    exps = np.concatenate([rng.integers(-126, 126, R - 16), np.arange(-104, -96, 0.5)])
    amax = (1.0 + rng.random(R)) * np.exp2(exps)
    amax = amax.astype(np.float32)
    W = (rng.uniform(-1.0, 1.0, (R, K)) * amax[:, None]).astype(np.float32)
    W[np.arange(R), rng.integers(0, K, R)] = amax * np.where(rng.random(R) < 0.5, -1.0, 1.0).astype(np.float32)
    if fmt == "Block_FP8":
        # one binade per 128x128 block: scale whole blocks by their own factor
        blk = np.exp2(rng.integers(-120, 120, (R // 128, K // 128))).astype(np.float32)
        W = (W / amax[:, None] * np.repeat(np.repeat(blk, 128, 0), 128, 1)).astype(np.float32)
    Wd = torch.from_numpy(W).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu(fmt, Wd)
    # activations: bf16 rows (groups) with maxima over the bf16 exponent range
    A32 = (rng.uniform(-1.0, 1.0, (R, K)) * amax[:, None]).astype(np.float32)
    A32[np.arange(R), rng.integers(0, K, R)] = amax
    A = torch.from_numpy(A32).to(torch.bfloat16)
    Aq, sa = gc.quant_act_gpu(fmt, A.to(gc.DEV))
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    gc.check_quant(orc, fmt, A, W, Aq, sa, Wq, sw)


def test_quant_act_row_stride(orc, gc, q):
    import seeded_inputs as si
    M, K, lda = 5, 512, 640
    big = si.activations(M, lda, seed=77)
    A = big[:, :K].contiguous()
    Ad = big.to(gc.DEV)
    for fmt in ("FP8_Dynamic", "W8A8_INT8", "Block_FP8"):
        Aq = torch.empty((M, K), dtype=torch.uint8, device=gc.DEV)
        sa = torch.empty((M, K // 128) if fmt == "Block_FP8" else (M,), dtype=torch.float32, device=gc.DEV)
        q.qg_quant_act(fmt, Ad, M, K, lda, Aq, sa)
        torch.cuda.synchronize()
        oAq, osa = orc.quant_act(fmt, si.bf16_to_f32_numpy(A))
        assert np.array_equal(Aq.cpu().numpy().view(gc.oracle_dtype(fmt)), oAq)
        assert np.array_equal(sa.cpu().numpy(), osa)


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8"])
@pytest.mark.parametrize("K", [16, 656, 4096, 4112, 8192, 12288, 16400, 25600, 32768, 32784])
def test_quant_act_row_lengths(orc, gc, fmt, K):
    # every register-resident row kernel (1, 2, 4, 8 chunks of 8 values per
    # thread, ragged last chunk) and the looping kernel beyond 32768
    # elements; outliers put the row maximum anywhere in the row
    import seeded_inputs as si
    M = 3
    A = si.activations(M, K, seed=K, outliers=True)
    A[1, ::7] = -0.0  # negative zeros keep their sign in E4M3 (code 0x80)
    A[2, 5::11] = 0.0
    Aq, sa = gc.quant_act_gpu(fmt, A.to(gc.DEV))
    torch.cuda.synchronize()
    oAq, osa = orc.quant_act(fmt, si.bf16_to_f32_numpy(A))
    assert np.array_equal(Aq.cpu().numpy().view(gc.oracle_dtype(fmt)), oAq)
    assert np.array_equal(sa.cpu().numpy(), osa)


@pytest.mark.parametrize("M", [1, 5, 8, 9, 16, 17, 24, 25, 32, 33, 70])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 2), (SWS, 7), (SWS, 16), (SWS, 18)])
def test_w8a8_int8_mma_sync(orc, q, gc, M, variant, split):
    # the mma.sync form of Swap-AB: token groups of 8 (M = 1..32 in one
    # block of 8/16/24/32, M = 33 and 70 in blocks of 32 with a ragged last
    # block); K = 2304: 18 k-tiles, three exact 1024-K segments at split 1;
    # 16 ranges reduce in a cluster, 18 through the workspace; ragged N; the
    # int32 accumulators bit-exact
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=600 + M, outliers=True,
                config_id=q.config_id(0, 0, mma_sync=True))


@pytest.mark.parametrize("M", [1, 9, 24, 32, 70])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 3), (SWS, 16), (SWS, 18)])
def test_w8a8_int8_mma_sync_narrow_warps(orc, q, gc, M, variant, split):
    # eight MMA warps of 16 weight rows (QG_CONFIG_MMA_NARROW): same checks
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=700 + M, outliers=True,
                config_id=q.config_id(0, 0, narrow=True))


@pytest.mark.parametrize("M", [1, 5, 8, 9, 16, 17, 24, 25, 32, 33, 70])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 2), (SWS, 7), (SWS, 16), (SWS, 18)])
def test_w8a8_int8_mma_sync_s8(orc, q, gc, M, variant, split):
    # the int8 form of mma.sync (m16n8k32, s8 operands, s32 accumulate, no
    # widening): token groups of 8, blocks of up to 32 with a ragged last
    # block, cluster and workspace reductions, ragged N; the int32
    # accumulators bit-exact
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=1600 + M, outliers=True,
                config_id=q.config_id(0, 0, s8=True))


@pytest.mark.parametrize("M", [1, 9, 24, 32, 70])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 3), (SWS, 16), (SWS, 18)])
def test_w8a8_int8_mma_sync_s8_narrow_warps(orc, q, gc, M, variant, split):
    # the s8 form with eight MMA warps of 16 weight rows
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=1700 + M, outliers=True,
                config_id=q.config_id(0, 0, narrow=True, s8=True))


@pytest.mark.parametrize("M,K", [(4, 2320), (13, 4096 + 48), (32, 144)])
@pytest.mark.parametrize("ring", [2, 5])
def test_w8a8_int8_mma_sync_s8_ragged_k(orc, q, gc, M, K, ring):
    # K not a multiple of 128: the last k-tile's zero fill adds nothing;
    # shallow and deeper rings
    gc.run_case(orc, "W8A8_INT8", M, 256, K, SWS, 2, seed=1800 + M + ring, outliers=True,
                config_id=q.config_id(ring, 0, s8=True))


@pytest.mark.parametrize("M", [1, 17, 64, 65, 100, 128, 200, 300, 513])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 2), (SWS, 7), (SWS, 18)])
def test_w8a8_int8_prewidened_activations(orc, q, gc, M, variant, split):
    # QG_CONFIG_I8_PREWIDEN: activations widened once per launch into the
    # workspace and loaded by TMA; token blocks of 64 (M <= 64) or 128 with
    # a ragged last block; three exact 1024-K segments; cluster and
    # workspace reductions; ragged N; int32 bit-exact
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=1900 + M + split, outliers=True,
                config_id=q.config_id(0, 0, prewiden=True))


@pytest.mark.parametrize("M,K", [(130, 2320), (64, 144)])
@pytest.mark.parametrize("ring", [2, 3])
def test_w8a8_int8_prewidened_ragged_k_and_rings(orc, q, gc, M, K, ring):
    # K not a multiple of 64 (the last fp16 atom partly past K) and shallow rings
    gc.run_case(orc, "W8A8_INT8", M, 256, K, SWS, 2, seed=1950 + M + ring, outliers=True,
                config_id=q.config_id(ring, 0, prewiden=True))


@pytest.mark.parametrize("M", [9, 16, 17, 32, 33, 64, 70])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 2), (SWS, 7), (SWS, 18)])
def test_w8a8_int8_sixteen_converter_warps(orc, q, gc, M, variant, split):
    # QG_CONFIG_I8_CONV16: sixteen weight converter warps (k-tiles in four
    # parts, accumulators drained in four token parts: 4 tokens each at
    # M <= 16), one CTA per SM with the deepest ring; int32 bit-exact
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=2000 + M + split, outliers=True,
                config_id=q.config_id(0, 0, conv16=True))


@pytest.mark.parametrize("M", [64, 100, 300])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 3), (SWS, 18)])
def test_w8a8_int8_prewidened_sixteen_converter_warps(orc, q, gc, M, variant, split):
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=2100 + M + split, outliers=True,
                config_id=q.config_id(0, 0, prewiden=True, conv16=True))


def test_int8_prewidened_identical_to_other_kernels(gc, q):
    # the same int32 accumulators and Y as the tcgen05 kernel that widens the
    # activations itself, and through qg_linear_w8a8 (quantization, widening
    # and GEMM: three kernels)
    import seeded_inputs as si
    M, N, K = 300, 640, 4096
    A = si.activations(M, K, seed=61, outliers=True).to(gc.DEV)
    W = torch.from_numpy(si.weights(N, K, seed=61)).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu("W8A8_INT8", W)
    Aq, sa = gc.quant_act_gpu("W8A8_INT8", A)
    Y0, d0 = gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 3, debug=True)
    cfg = q.config_id(0, 0, prewiden=True)
    Y1, d1 = gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 3, config_id=cfg, debug=True)
    Y3, d3 = gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 3, config_id=q.config_id(conv16=True), debug=True)
    Y4, d4 = gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 3, config_id=q.config_id(prewiden=True, conv16=True),
                         debug=True)
    Y2 = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device=gc.DEV)
    need = q.qg_workspace_bytes_config("W8A8_INT8", M, N, K, SWS, 3, cfg)
    assert need >= M * K * 2 and need > q.qg_workspace_bytes("W8A8_INT8", M, N, K, SWS, 3)
    ws = torch.zeros(need, dtype=torch.uint8, device=gc.DEV)
    Aq2, sa2 = torch.empty_like(Aq), torch.empty_like(sa)
    q.qg_linear_w8a8("W8A8_INT8", M, N, K, A, K, Wq, sw, Y2, N, SWS, 3, cfg, ws, need, Aq2, sa2, None)
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    assert torch.equal(d0, d1) and torch.equal(Y0, Y1) and torch.equal(Y0, Y2)
    assert torch.equal(d0, d3) and torch.equal(Y0, Y3) and torch.equal(d0, d4) and torch.equal(Y0, Y4)


def test_prewidened_config_rejected_elsewhere(q, gc):
    d = torch.zeros(1 << 20, dtype=torch.uint8, device=gc.DEV)
    f = torch.ones(4096, dtype=torch.float32, device=gc.DEV)
    pw = q.QG_CONFIG_I8_PREWIDEN
    for fmt, v, s, cfg in (("FP8_Dynamic", SW, 1, pw), ("Block_FP8", SW, 1, pw), ("W8A8_INT8", DP, 1, pw),
                           ("W8A8_INT8", SW, 1, pw | q.QG_CONFIG_MMA_SYNC), ("W8A8_INT8", SW, 1, pw | q.QG_CONFIG_FUSED_QUANT),
                           ("FP8_Dynamic", SW, 1, q.QG_CONFIG_I8_CONV16),
                           ("W8A8_INT8", SW, 1, q.QG_CONFIG_I8_CONV16 | q.QG_CONFIG_MMA_SYNC)):
        with pytest.raises(q.QGError) as e:
            q.qg_gemm_w8a8(fmt, 64, 256, 256, d, f, d, f, d, 256, v, s, cfg, d, d.numel())
        assert e.value.code == q.QG_ERR_INVALID_ARG
    with pytest.raises(q.QGError) as e:  # the fp16 copy needs the workspace
        q.qg_gemm_w8a8("W8A8_INT8", 64, 256, 256, d, f, d, f, d, 256, SW, 1, pw)
    assert e.value.code == q.QG_ERR_WORKSPACE_TOO_SMALL


@pytest.mark.parametrize("M", [3, 12, 32])
@pytest.mark.parametrize("ring", [2, 3, 6])
def test_w8a8_int8_mma_sync_ring_depths(orc, q, gc, M, ring):
    # shallow and deep rings (the ring wraps many times over 32 k-tiles)
    gc.run_case(orc, "W8A8_INT8", M, 256, 4096, SWS, 1 if ring != 3 else 2, seed=650 + ring,
                config_id=q.config_id(ring, 0, mma_sync=True))


def test_int8_mma_sync_identical_to_tensor_memory_kernel(gc, q):
    # the mma.sync kernel and the tcgen05 kernel compute the same int32
    # accumulators and the same Y
    import seeded_inputs as si
    M, N, K = 29, 384, 4096
    A = si.activations(M, K, seed=31, outliers=True).to(gc.DEV)
    W = torch.from_numpy(si.weights(N, K, seed=31)).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu("W8A8_INT8", W)
    Aq, sa = gc.quant_act_gpu("W8A8_INT8", A)
    Y0, d0 = gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 4, debug=True)
    Y1, d1 = gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 4, config_id=q.config_id(0, 0, mma_sync=True),
                         debug=True)
    Y2, d2 = gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 4, config_id=q.config_id(0, 0, narrow=True),
                         debug=True)
    Y3, d3 = gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 4, config_id=q.config_id(0, 0, s8=True),
                         debug=True)
    Y4, d4 = gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 4, config_id=q.config_id(0, 0, narrow=True, s8=True),
                         debug=True)
    torch.cuda.synchronize()
    assert torch.equal(d0, d1) and torch.equal(Y0, Y1)
    assert torch.equal(d0, d2) and torch.equal(Y0, Y2)
    assert torch.equal(d0, d3) and torch.equal(Y0, Y3)
    assert torch.equal(d0, d4) and torch.equal(Y0, Y4)


def test_mma_sync_config_rejected_outside_int8_swap_ab(q, gc):
    d = torch.zeros(1 << 16, dtype=torch.uint8, device=gc.DEV)
    f = torch.ones(4096, dtype=torch.float32, device=gc.DEV)
    for fmt, v in (("FP8_Dynamic", SW), ("Block_FP8", SW), ("W8A8_INT8", 4), ("W8A8_INT8", ST)):
        with pytest.raises(q.QGError) as e:
            q.qg_gemm_w8a8(fmt, 8, 256, 256, d, f, d, f, d, 256, v, 1, q.config_id(0, 0, mma_sync=True))
        assert e.value.code == q.QG_ERR_INVALID_ARG
    with pytest.raises(q.QGError) as e:  # the narrow form is a form of the mma.sync kernel only
        q.qg_gemm_w8a8("W8A8_INT8", 8, 256, 256, d, f, d, f, d, 256, SW, 1, q.QG_CONFIG_MMA_NARROW)
    assert e.value.code == q.QG_ERR_INVALID_ARG


@pytest.mark.parametrize("pair_mma", [False, True])
@pytest.mark.parametrize("M", [64, 100, 256, 300, 513])
@pytest.mark.parametrize("N,K", [(424, 656), (1024, 2048)])
def test_fp8_persistent_pairs(orc, q, gc, M, N, K, pair_mma):
    # the persistent pair kernel (QG_CONFIG_PERSIST): 256-token pair tiles
    # (the second CTA of the last pair partly or wholly past M), 256-row
    # weight tiles (N = 424: one full, one ragged), ragged K (656: the last
    # k-tile 16 wide); with pair_mma each MMA is one cta_group::2 instruction
    # of the pair (M = 256) on the two CTAs' weight halves
    gc.run_case(orc, "FP8_Dynamic", M, N, K, ST, 1, seed=800 + M + N, outliers=True,
                config_id=q.config_id(persist=True, pair_mma=pair_mma))


@pytest.mark.parametrize("pair_mma", [False, True])
@pytest.mark.parametrize("rows", [224, 192, 160])
@pytest.mark.parametrize("M,N,K", [(100, 424, 656), (513, 1000, 1024), (300, 4096, 512)])
def test_fp8_persistent_narrow_weight_tiles(orc, q, gc, M, N, K, rows, pair_mma):
    # weight tiles of 224 / 192 / 160 rows (QG_CONFIG_PERSIST_ROWS_MASK):
    # TMA boxes of rows/2, MMA N = rows, the last tile ragged (424, 1000 and
    # 4096 are not multiples of any of them; for 4096 the last tile's second
    # half lies wholly past N), ragged K and token pairs
    gc.run_case(orc, "FP8_Dynamic", M, N, K, ST, 1, seed=860 + M + rows, outliers=True,
                config_id=q.config_id(persist=True, pair_mma=pair_mma, persist_rows=rows))


@pytest.mark.parametrize("pair_mma", [False, True])
@pytest.mark.parametrize("ring", [2, 3])
def test_fp8_persistent_many_tiles_per_pair(orc, q, gc, ring, pair_mma):
    # 3 x 80 = 240 pair tiles: every cluster takes several tiles, so both
    # TMEM accumulators and the weight-scale slots are reused; shallow rings
    # wrap many times.  Sampled columns against the oracle.
    import seeded_inputs as si
    M, N, K = 600, 20480, 512
    A = si.activations(M, K, seed=820 + ring, outliers=True)
    W = si.weights(N, K, seed=820 + ring)
    Wq, sw = gc.quant_weight_gpu("FP8_Dynamic", torch.from_numpy(W).to(gc.DEV))
    Aq, sa = gc.quant_act_gpu("FP8_Dynamic", A.to(gc.DEV))
    Y, _ = gc.gemm_gpu("FP8_Dynamic", Aq, sa, Wq, sw, N, ST, 1,
                       config_id=q.config_id(ring, persist=True, pair_mma=pair_mma))
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    ns = np.concatenate([np.arange(0, 300), np.arange(10000, 10300), np.arange(N - 300, N)])
    oAq, osa = orc.quant_act("FP8_Dynamic", si.bf16_to_f32_numpy(A))
    oWq, osw = orc.quant_weight("FP8_Dynamic", W)
    assert np.array_equal(Aq.cpu().numpy(), oAq)
    gc.check_gemm(orc, "FP8_Dynamic", oAq, osa, oWq, osw, Y, ns=ns)
    assert not torch.isnan(Y.float()).any()


@pytest.mark.parametrize("rows", [256, 160])
@pytest.mark.parametrize("pair_mma", [False, True])
def test_fp8_persistent_bounded_wait_and_recovery(orc, q, gc, pair_mma, rows):
    import seeded_inputs as si
    M, N, K = 300, 1024, 1024
    A = si.activations(M, K, seed=830)
    W = si.weights(N, K, seed=830)
    Wq, sw = gc.quant_weight_gpu("FP8_Dynamic", torch.from_numpy(W).to(gc.DEV))
    Aq, sa = gc.quant_act_gpu("FP8_Dynamic", A.to(gc.DEV))
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    cfg = q.config_id(persist=True, pair_mma=pair_mma, persist_rows=rows)
    q.qg_set_wait_limit_ns(2_000_000)
    q.qg_set_force_timeout(True)
    try:
        gc.gemm_gpu("FP8_Dynamic", Aq, sa, Wq, sw, N, ST, 1, config_id=cfg)
        assert q.qg_device_error() == q.QG_ERR_DEVICE_TIMEOUT
    finally:
        q.qg_set_force_timeout(False)
        q.qg_set_wait_limit_ns(0)
    Y, _ = gc.gemm_gpu("FP8_Dynamic", Aq, sa, Wq, sw, N, ST, 1, config_id=cfg)
    torch.cuda.synchronize()
    assert q.qg_device_error() == 0
    oAq, osa, oWq, osw = gc.check_quant(orc, "FP8_Dynamic", A, W, Aq, sa, Wq, sw)
    gc.check_gemm(orc, "FP8_Dynamic", oAq, osa, oWq, osw, Y)


def test_persist_config_rejected_elsewhere(q, gc):
    d = torch.zeros(1 << 16, dtype=torch.uint8, device=gc.DEV)
    f = torch.ones(4096, dtype=torch.float32, device=gc.DEV)
    for fmt, v, s, cfg in (("Block_FP8", ST, 1, q.config_id(persist=True)),
                           ("FP8_Dynamic", SW, 1, q.config_id(persist=True)),
                           ("FP8_Dynamic", STS, 2, q.config_id(persist=True)),
                           ("FP8_Dynamic", ST, 1, q.config_id(persist=True, wide=True)),
                           ("FP8_Dynamic", ST, 1, q.QG_CONFIG_PAIR_MMA)):
        with pytest.raises(q.QGError) as e:
            q.qg_gemm_w8a8(fmt, 64, 256, 256, d, f, d, f, d, 256, v, s, cfg)
        assert e.value.code == q.QG_ERR_INVALID_ARG


@pytest.mark.parametrize("s8", [False, True])
@pytest.mark.parametrize("dpw", [1, 2, 4])
@pytest.mark.parametrize("M", [1, 8, 13, 16])
@pytest.mark.parametrize("variant,split", [(SW, 1), (SWS, 3), (SWS, 18)])
def test_w8a8_int8_mma_sync_with_dp4a_rows(orc, q, gc, dpw, M, variant, split, s8):
    # the first 16*dpw rows of each weight tile on dp4a warps, the rest on
    # mma.sync (widened or s8): ragged N (the last tile's dp4a rows partly
    # past N), three exact segments, cluster and workspace reductions; int32
    # bit-exact
    gc.run_case(orc, "W8A8_INT8", M, 300, 2304, variant, split, seed=900 + 10 * dpw + M + 100 * s8, outliers=True,
                config_id=q.config_id(0, 0, dp4a_rows16=dpw, s8=s8))


def test_int8_dp4a_rows_identical_to_other_kernels(gc, q):
    import seeded_inputs as si
    M, N, K = 11, 384, 4096
    A = si.activations(M, K, seed=41, outliers=True).to(gc.DEV)
    W = torch.from_numpy(si.weights(N, K, seed=41)).to(gc.DEV)
    Wq, sw = gc.quant_weight_gpu("W8A8_INT8", W)
    Aq, sa = gc.quant_act_gpu("W8A8_INT8", A)
    outs = [gc.gemm_gpu("W8A8_INT8", Aq, sa, Wq, sw, N, SWS, 4, config_id=c, debug=True)
            for c in (0, q.config_id(mma_sync=True), q.config_id(dp4a_rows16=3),
                      q.config_id(dp4a_rows16=2, s8=True))]
    torch.cuda.synchronize()
    for Y, d in outs[1:]:
        assert torch.equal(d, outs[0][1]) and torch.equal(Y, outs[0][0])


def test_dp4a_rows_rejected_beyond_16_tokens_and_without_narrow(q, gc):
    d = torch.zeros(1 << 16, dtype=torch.uint8, device=gc.DEV)
    f = torch.ones(4096, dtype=torch.float32, device=gc.DEV)
    with pytest.raises(q.QGError) as e:
        q.qg_gemm_w8a8("W8A8_INT8", 17, 256, 256, d, f, d, f, d, 256, SW, 1, q.config_id(dp4a_rows16=2))
    assert e.value.code == q.QG_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(q.QGError) as e:
        q.qg_gemm_w8a8("W8A8_INT8", 8, 256, 256, d, f, d, f, d, 256, SW, 1,
                       q.QG_CONFIG_MMA_SYNC | (2 << q.QG_CONFIG_MMA_DP4A_SHIFT))
    assert e.value.code == q.QG_ERR_INVALID_ARG


@pytest.mark.parametrize("pair_mma", [False, True])
@pytest.mark.parametrize("dist", [4, 16, 64])
def test_fp8_persistent_l2_prefetch(orc, q, gc, dist, pair_mma):
    # L2 prefetch of the weight halves ahead of the ring, across tiles (64:
    # beyond every CTA's remaining k-tiles); results unchanged
    gc.run_case(orc, "FP8_Dynamic", 300, 1024, 2048, ST, 1, seed=840 + dist, outliers=True,
                config_id=q.config_id(0, dist, persist=True, pair_mma=pair_mma))
