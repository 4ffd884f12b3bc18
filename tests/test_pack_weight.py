"""qg_pack_weight: the host weight quantizer of the C ABI, against the CPU
oracle's weight quantization (per output channel for FP8_Dynamic and
W8A8_INT8, 128x128 blocks for Block_FP8, "Helion Linear Backend > Scope"):
codes and scales bit for bit.  Runs without a GPU; on a GPU the device
quantizer (qg_quant_weight) must give the same bytes."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import seeded_inputs as si


@pytest.fixture(scope="module")
def q():
    from quantized_gemm_decode_02_b300 import qgemm
    return qgemm


def pack(q, fmt, W):
    N, K = W.shape
    Wq = torch.empty((N, K), dtype=torch.uint8)
    sw = torch.empty(((N + 127) // 128, K // 128) if fmt == "Block_FP8" else (N,), dtype=torch.float32)
    q.qg_pack_weight(fmt, torch.from_numpy(np.ascontiguousarray(W)), N, K, Wq, sw)
    return Wq, sw


def oracle_view(fmt, Wq):
    return Wq.numpy().view(np.int8) if fmt == "W8A8_INT8" else Wq.numpy()


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
@pytest.mark.parametrize("N,K", [(300, 2304), (128, 128), (257, 640)])
def test_pack_weight_matches_oracle(orc, q, fmt, N, K):
    W = si.weights(N, K, seed=N + K)
    W[1, :] = 0.0                      # a zero row: s = 1, all codes 0
    W[2, ::5] = -0.0                   # signed zeros
    W[3, 7] = 40.0                     # an outlier sets the row / block maximum
    Wq, sw = pack(q, fmt, W)
    oWq, osw = orc.quant_weight(fmt, W)
    assert np.array_equal(oracle_view(fmt, Wq), oWq)
    assert np.array_equal(sw.numpy(), osw)


def test_pack_weight_rounding_ties(orc, q):
    # rows whose quotients land exactly on int8 and E4M3 rounding midpoints
    K = 256
    rows = []
    for s in (2.0 ** -6, 2.0 ** -3, 1.0):
        r = (np.arange(K, dtype=np.float32) % 200 - 100 + 0.5) * np.float32(s)
        r[0] = np.float32(127.0 * s)
        rows.append(r)
    W = np.stack(rows).astype(np.float32)
    for fmt in ("W8A8_INT8", "FP8_Dynamic"):
        Wq, sw = pack(q, fmt, W)
        oWq, osw = orc.quant_weight(fmt, W)
        assert np.array_equal(oracle_view(fmt, Wq), oWq)
        assert np.array_equal(sw.numpy(), osw)


def test_pack_weight_errors(q):
    W = torch.zeros((4, 96), dtype=torch.float32)
    Wq = torch.zeros((4, 96), dtype=torch.uint8)
    sw = torch.zeros(4, dtype=torch.float32)
    with pytest.raises(q.QGError) as e:
        q.qg_pack_weight("Block_FP8", W, 4, 96, Wq, sw)       # K % 128
    assert e.value.code == q.QG_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(q.QGError) as e:
        q.qg_pack_weight("FP8_Dynamic", W, 4, 90, Wq, sw)     # K % 16
    assert e.value.code == q.QG_ERR_UNSUPPORTED_SHAPE
    with pytest.raises(q.QGError) as e:
        q.qg_pack_weight(7, W, 4, 96, Wq, sw)
    assert e.value.code == q.QG_ERR_INVALID_ARG


def test_pack_weight_binding_rejects_short_or_mistyped_host_tensors(q):
    """The host quantizer writes N*K codes and the scales through raw
    pointers: the binding refuses tensors that cannot hold them."""
    N, K = 4, 128
    W = torch.zeros((N, K), dtype=torch.float32)
    Wq = torch.zeros((N, K), dtype=torch.uint8)
    sw = torch.zeros(N, dtype=torch.float32)
    bad = [
        (W[:, :64].contiguous(), Wq, sw),            # W too short
        (W.double(), Wq, sw),                        # W not fp32
        (W, Wq[:2].contiguous(), sw),                # W_q too short
        (W, Wq.to(torch.int16), sw),                 # W_q not 1-byte
        (W, Wq, sw[:3].contiguous()),                # s_w too short
        (W, Wq, torch.zeros((N, 2), dtype=torch.float32)[:, 0]),  # not contiguous
    ]
    for w, wq, s in bad:
        with pytest.raises(ValueError):
            q.qg_pack_weight("FP8_Dynamic", w, N, K, wq, s)
    with pytest.raises(ValueError):                  # Block_FP8: one scale per 128x128 block
        q.qg_pack_weight("Block_FP8", torch.zeros((200, K)), 200, K, torch.zeros((200, K), dtype=torch.uint8),
                         torch.zeros(1, dtype=torch.float32))
    q.qg_pack_weight("Block_FP8", torch.zeros((200, K)), 200, K, torch.zeros((200, K), dtype=torch.uint8),
                     torch.zeros(2, dtype=torch.float32))


@pytest.mark.gpu
@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
def test_pack_weight_equals_device_quantizer(q, fmt):
    import gpu_cases as gc
    W = si.weights(384, 1024, seed=5)
    Wq, sw = pack(q, fmt, W)
    dWq, dsw = gc.quant_weight_gpu(fmt, torch.from_numpy(W).to(gc.DEV))
    torch.cuda.synchronize()
    assert torch.equal(dWq.cpu().view(torch.uint8).reshape(Wq.shape), Wq)
    assert torch.equal(dsw.cpu().reshape(sw.shape), sw)
