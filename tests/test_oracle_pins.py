"""Pins for the CPU oracle against facts fixed outside it.

Nothing here re-types the oracle's formulas: each check compares it with a
library routine (torch's float8_e4m3fn / bfloat16 casts, numpy and torch
integer matmuls, numpy fp64 matmul of exactly representable products), with
exact rational arithmetic (``fractions.Fraction``), with a brute-force search,
with hand-derived golden values (tests/golden), or with invariants of the
definitions (identity weights, one-hot weights, K permutation, round-trip
bounds).  The formats are those of "Building a High-Performance and Portable
vLLM Linear Backend with Helion", section "Helion Linear Backend > Scope".
"""
from __future__ import annotations

import math
import os
import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import seeded_inputs as si

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ------------------------------------------------------------ independent helpers

def torch_e4m3_values() -> np.ndarray:
    """float64 value of every E4M3FN code, decoded by torch."""
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def torch_e4m3_encode(x: np.ndarray) -> np.ndarray:
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def frac_bf16_bits(y) -> int:
    """bf16 RNE of an exact value (float or Fraction) by rational arithmetic,
    independent of the oracle's bit manipulation: find the grid spacing,
    round the exact quotient half-to-even, re-pack via struct."""
    if isinstance(y, float) and y == 0.0:
        return 0x8000 if math.copysign(1.0, y) < 0 else 0
    a = Fraction(y)
    if a == 0:
        return 0
    sign = 0x8000 if a < 0 else 0
    a = abs(a)
    e = a.numerator.bit_length() - a.denominator.bit_length()   # 2^e <= a*2^? : fix below
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1                                            # now 2^e <= a < 2^(e+1)
    spacing = Fraction(2) ** (e - 7) if e >= -126 else Fraction(2) ** -133
    q = a / spacing
    fl = math.floor(q)
    r = q - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    v = fl * spacing
    if v >= Fraction(2) ** 128:
        return sign | 0x7F80
    bits = struct.unpack("<I", struct.pack("<f", float(v)))[0]
    assert bits & 0xFFFF == 0
    return sign | (bits >> 16)


def parse_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = line.split(":", 1)
            out[k.strip()] = v.split()
    return out


def frac_list(vals):
    return [Fraction(v) for v in vals]


# -------------------------------------------------------------------- E4M3 codec

def test_e4m3_decode_all_codes_match_torch(orc):
    ours = orc.e4m3_decode(np.arange(256, dtype=np.uint8))
    ref = torch_e4m3_values()
    nan = np.isnan(ref)
    assert set(np.nonzero(nan)[0].tolist()) == {0x7F, 0xFF}
    assert np.isnan(ours[nan]).all()
    assert np.array_equal(ours[~nan], ref[~nan])


def test_e4m3_decode_landmarks(orc):
    d = orc.e4m3_decode(np.array([0x00, 0x01, 0x07, 0x08, 0x38, 0x7E, 0x80, 0xFE], np.uint8))
    assert d.tolist() == [0.0, 2.0 ** -9, 7 * 2.0 ** -9, 2.0 ** -6, 1.0, 448.0, -0.0, -448.0]


def test_e4m3_roundtrip_every_finite_code(orc):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = orc.e4m3_decode(codes).astype(np.float32)
    assert np.array_equal(orc.e4m3_encode(vals), codes)


def test_e4m3_encode_matches_torch_in_range(orc):
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.uniform(-448, 448, 4000),
        rng.standard_normal(4000) * 3,
        rng.standard_normal(2000) * 0.01,           # subnormal region
        np.ldexp(rng.uniform(-1, 1, 2000), -8),
    ]).astype(np.float32)
    vals = torch_e4m3_values()
    fin = np.sort(np.unique(vals[np.isfinite(vals)]))
    mids = ((fin[1:] + fin[:-1]) / 2).astype(np.float32)  # exact in fp32
    x = np.concatenate([x, mids, -mids, np.nextafter(mids, np.float32(np.inf)), np.nextafter(mids, np.float32(-np.inf))])
    x = x[np.abs(x) <= 448]
    assert np.array_equal(orc.e4m3_encode(x), torch_e4m3_encode(x))


def test_e4m3_encode_bruteforce_nearest_ties_even(orc):
    vals = torch_e4m3_values()
    pos_codes = np.arange(0, 0x7F)  # 0x00..0x7E finite non-negative
    pos_vals = vals[pos_codes]
    fin = np.sort(pos_vals)
    mids = (fin[1:] + fin[:-1]) / 2
    rng = np.random.default_rng(1)
    xs = np.concatenate([mids, rng.uniform(0, 448, 3000), np.ldexp(rng.uniform(0, 1, 500), -7)]).astype(np.float32)
    got = orc.e4m3_encode(xs)
    for x, g in zip(xs.tolist(), got.tolist()):
        dist = np.abs(pos_vals - x)
        best = np.nonzero(dist == dist.min())[0]
        if len(best) == 1:
            want = int(pos_codes[best[0]])
        else:  # a tie between two neighbours: the even code (even mantissa) wins
            want = int([c for c in pos_codes[best] if c % 2 == 0][0])
        assert g == want, (x, g, want)
    # negative side mirrors with the sign bit
    assert np.array_equal(orc.e4m3_encode(-xs[xs > 0]), got[xs > 0] | 0x80)


def test_e4m3_encode_saturates_by_definition(orc):
    # torch gives NaN out of range; saturation is pinned by the satfinite reading.
    big = np.array([448.0, 449.0, 463.9, 464.0, 480.0, 1e6, 3.0e38, np.inf], np.float32)
    assert orc.e4m3_encode(big).tolist() == [0x7E] * len(big)
    assert orc.e4m3_encode(-big).tolist() == [0xFE] * len(big)


def test_e4m3_encode_underflow(orc):
    x = np.array([2.0 ** -10, 2.0 ** -10 * 1.0001, 2.0 ** -11, 1e-30, 0.0, 3 * 2.0 ** -10], np.float32)
    # 2^-10 is the midpoint of 0 and 2^-9 -> even code 0; just above -> 0x01; 3*2^-10 ties 1 vs 2 -> 2
    assert orc.e4m3_encode(x).tolist() == [0x00, 0x01, 0x00, 0x00, 0x00, 0x02]


# -------------------------------------------------------------------- INT8 codec

def test_int8_encode_matches_numpy_rint(orc):
    rng = np.random.default_rng(2)
    x = np.concatenate([rng.uniform(-140, 140, 5000), np.arange(-130, 130) + 0.5, np.arange(-130, 130).astype(float)]).astype(np.float32)
    want = np.clip(np.rint(x), -127, 127).astype(np.int8)  # numpy rint: half to even
    assert np.array_equal(orc.int8_encode(x), want)


def test_int8_ties_and_clamp(orc):
    x = np.array([2.5, 3.5, -2.5, -3.5, 0.5, -0.5, 126.5, 127.49, 200.0, -127.5, -128.0, -1e9], np.float32)
    assert orc.int8_encode(x).tolist() == [2, 4, -2, -4, 0, 0, 126, 127, 127, -127, -127, -127]


# -------------------------------------------------------------------- bf16 rounding

def test_bf16_from_double_matches_exact_rational(orc):
    rng = np.random.default_rng(3)
    ys = np.concatenate([
        rng.standard_normal(3000) * 10.0 ** rng.integers(-10, 10, 3000),
        np.ldexp(rng.uniform(0.5, 1, 300), rng.integers(-140, -120, 300)),  # bf16 subnormal range
        np.array([0.0, -0.0, 1.0, -1.0, 3.0e38, 3.4e38, -3.4e38, 1.00390625, 1.01171875]),
    ])
    # exact ties: 8 significant bits + a half-ulp bit
    t = (rng.integers(128, 256, 400) * 2 + 1).astype(np.float64) * np.ldexp(1.0, rng.integers(-30, 30, 400))
    ys = np.concatenate([ys, t, -t])
    got = orc.bf16_from_double(ys)
    for y, g in zip(ys.tolist(), got.tolist()):
        assert g == frac_bf16_bits(y), (y, hex(g), hex(frac_bf16_bits(y)))


def test_bf16_from_double_matches_torch_on_fp32_inputs(orc):
    rng = np.random.default_rng(4)
    x = (rng.standard_normal(20000) * 100).astype(np.float32)
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(orc.bf16_from_double(x.astype(np.float64)), want)


# -------------------------------------------------------------------- golden files

def _golden_case(orc, name, fmt):
    g = parse_golden(name)
    M, N, K = int(g["M"][0]), int(g["N"][0]), int(g["K"][0])
    if "A" in g:
        A = np.array([float(v) for v in g["A"]], np.float32).reshape(M, K)
        W = np.array([float(v) for v in g["W"]], np.float32).reshape(N, K)
    else:
        A = np.zeros((M, K), np.float32); W = np.zeros((N, K), np.float32)
        for kv in g["A_sparse"]:
            k, v = kv.split("="); A[0, int(k)] = float(v)
        for kv in g["W_sparse"]:
            k, v = kv.split("="); W[0, int(k)] = float(v)
    Aq, sa = orc.quant_act(fmt, A)
    Wq, sw = orc.quant_weight(fmt, W)
    for got, want in ((sa.ravel(), frac_list(g["s_a"])), (sw.ravel(), frac_list(g["s_w"]))):
        assert len(got) == len(want)
        for a, b in zip(got.tolist(), want):
            assert abs(Fraction(a) - b) <= abs(b) * Fraction(1, 2 ** 23)
    if "A_q" in g:
        assert Aq.view(np.uint8).ravel().tolist() == [int(v, 16) for v in g["A_q"]]
        assert Wq.view(np.uint8).ravel().tolist() == [int(v, 16) for v in g["W_q"]]
    else:
        for key, arr in (("A_q_sparse", Aq), ("W_q_sparse", Wq)):
            flat = arr.view(np.uint8).ravel()
            want = np.zeros_like(flat)
            for kv in g[key]:
                k, v = kv.split("="); want[int(k)] = int(v, 16)
            assert np.array_equal(flat, want)
    acc, y = orc.gemm(fmt, Aq, sa, Wq, sw)
    if "acc" in g:
        assert [int(round(float(v))) for v in acc.ravel()] == [int(v) for v in g["acc"]]
    assert y.ravel().tolist() == [int(v, 16) for v in g["Y"]]


def test_golden_fp8_dynamic_tiny(orc):
    _golden_case(orc, "fp8_dynamic_tiny.txt", "FP8_Dynamic")


def test_golden_fp8_dynamic_cancel(orc):
    _golden_case(orc, "fp8_dynamic_cancel.txt", "FP8_Dynamic")


def test_golden_w8a8_int8_ties(orc):
    _golden_case(orc, "w8a8_int8_ties.txt", "W8A8_INT8")


def test_golden_block_fp8_two_groups(orc):
    _golden_case(orc, "block_fp8_two_groups.txt", "Block_FP8")


# -------------------------------------------------------------------- quantizers

@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
def test_quant_amax_element_hits_qmax_and_roundtrip_bound(orc, fmt):
    A = si.bf16_to_f32_numpy(si.activations(5, 384, seed=11, outliers=True))
    A[2] = 0.0                                          # an all-zero token row
    q, s = orc.quant_act(fmt, A)
    tv = torch_e4m3_values()
    if fmt == "W8A8_INT8":
        deq = q.astype(np.float64) * s[:, None]
        assert np.all(np.abs(deq - A) <= s[:, None] * 0.5 * (1 + 1e-6))
        for m in (0, 1, 3, 4):
            i = np.argmax(np.abs(A[m])); assert abs(int(q[m, i])) == 127
        assert s[2] == 1.0 and not q[2].any()
        return
    if fmt == "FP8_Dynamic":
        sfull = np.repeat(s[:, None], A.shape[1], 1).astype(np.float64)
    else:
        sfull = np.repeat(s, 128, axis=1)[:, :A.shape[1]].astype(np.float64)
    deq = tv[q] * sfull
    x = A.astype(np.float64)
    normal = np.abs(x) >= sfull * 2.0 ** -6
    # E4M3 has 3 mantissa bits: relative error <= 2^-4 for normals, <= 2^-10 * s absolute below
    assert np.all(np.abs(deq - x)[normal] <= np.abs(x)[normal] * 2.0 ** -4 * (1 + 1e-6))
    assert np.all(np.abs(deq - x)[~normal] <= sfull[~normal] * 2.0 ** -10 * (1 + 1e-6))
    assert np.all(q[2] == 0) and np.all(s[2] == 1.0)
    if fmt == "FP8_Dynamic":
        for m in (0, 1, 3, 4):
            i = np.argmax(np.abs(A[m])); assert q[m, i] & 0x7F == 0x7E
    else:
        for m in (0, 1, 3, 4):
            for gi in range(3):
                seg = A[m, gi * 128:(gi + 1) * 128]
                i = np.argmax(np.abs(seg)); assert q[m, gi * 128 + i] & 0x7F == 0x7E


def test_block_weight_scales_cover_ragged_edges(orc):
    W = si.weights(200, 256, seed=5)                     # N ragged (200 = 128 + 72)
    q, s = orc.quant_weight("Block_FP8", W)
    assert s.shape == (2, 2)
    for bn in range(2):
        for bk in range(2):
            blk = W[bn * 128:min(200, bn * 128 + 128), bk * 128:bk * 128 + 128]
            assert abs(float(s[bn, bk]) - float(np.abs(blk).max()) / 448) <= float(s[bn, bk]) * 2 ** -22
    tv = torch_e4m3_values()
    deq = tv[q] * np.repeat(np.repeat(s, 128, 0), 128, 1)[:200, :256]
    assert np.all(np.abs(deq - W) <= np.abs(W) * 2.0 ** -4 + 1e-12 + np.repeat(np.repeat(s, 128, 0), 128, 1)[:200, :256] * 2 ** -10)


# -------------------------------------------------------------------- GEMM pins

_TV = None


def _frac_e4m3(code: int) -> Fraction:
    global _TV
    if _TV is None:
        _TV = [Fraction(float(v)) if np.isfinite(v) else None for v in torch_e4m3_values()]
    return _TV[code]


def _frac_gemm_y(fmt, Aq, sa, Wq, sw, ns):
    """Exact rational GEMM + one bf16 rounding of the exact value (brute force,
    tiny sizes), for all rows and the columns ``ns``."""
    M, K = Aq.shape
    acc = np.empty((M, len(ns)), object); ybits = np.empty((M, len(ns)), np.uint16)
    nbk = (K + 127) // 128
    for m in range(M):
        for j, n in enumerate(ns):
            if fmt == "W8A8_INT8":
                a = sum(Fraction(int(Aq[m, k])) * int(Wq[n, k]) for k in range(K))
                y = a * Fraction(float(sa[m])) * Fraction(float(sw[n]))
            elif fmt == "FP8_Dynamic":
                a = sum(_frac_e4m3(int(Aq[m, k])) * _frac_e4m3(int(Wq[n, k])) for k in range(K))
                y = a * Fraction(float(sa[m])) * Fraction(float(sw[n]))
            else:
                a = Fraction(0)
                mag = Fraction(0)
                for kb in range(nbk):
                    part = sum(_frac_e4m3(int(Aq[m, k])) * _frac_e4m3(int(Wq[n, k]))
                               for k in range(kb * 128, min(K, kb * 128 + 128)))
                    term = Fraction(float(sa[m, kb])) * Fraction(float(sw[n // 128, kb])) * part
                    a += term
                    mag += abs(term)
                y = a
                a = (a, mag)
            acc[m, j] = a
            ybits[m, j] = frac_bf16_bits(y)
    return acc, ybits


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8"])
@pytest.mark.parametrize("shape", [(1, 1, 1), (3, 5, 7), (8, 8, 8), (2, 7, 16)])
def test_gemm_bruteforce_fraction_tiny(orc, fmt, shape):
    M, N, K = shape
    A = si.bf16_to_f32_numpy(si.activations(M, K, seed=M * 100 + N * 10 + K))
    W = si.weights(N, K, seed=K)
    Aq, sa = orc.quant_act(fmt, A)
    Wq, sw = orc.quant_weight(fmt, W)
    acc, y = orc.gemm(fmt, Aq, sa, Wq, sw)
    facc, fy = _frac_gemm_y(fmt, Aq, sa, Wq, sw, list(range(N)))
    for m in range(M):
        for n in range(N):
            assert Fraction(int(acc[m, n]) if fmt == "W8A8_INT8" else float(acc[m, n])) == facc[m, n]
    # single rounding from the exact value may differ from rounding the fp64 product only at a
    # bf16 midpoint; with random data that never happens, so demand equality.
    assert np.array_equal(y, fy)


def test_gemm_block_bruteforce_fraction_ragged(orc):
    M, N, K = 2, 130, 256                               # two weight block rows (ragged), two K groups
    A = si.bf16_to_f32_numpy(si.activations(M, K, seed=21))
    W = si.weights(N, K, seed=22)
    Aq, sa = orc.quant_act("Block_FP8", A)
    Wq, sw = orc.quant_weight("Block_FP8", W)
    ns = [0, 1, 127, 128, 129]
    acc, y = orc.gemm("Block_FP8", Aq, sa, Wq, sw, ns=ns)
    facc, fy = _frac_gemm_y("Block_FP8", Aq, sa, Wq, sw, ns)
    for m in range(M):
        for j in range(len(ns)):
            exact, mag = facc[m, j]
            # fp64: one rounding per scaled partial and per addition -> <= 2 * nbk * 2^-53 * sum|terms|
            assert abs(Fraction(float(acc[m, j])) - exact) <= mag * Fraction(2 * 2, 2 ** 53)
            assert y[m, j] == fy[m, j]


def test_gemm_int8_matches_numpy_and_torch_int_mm(orc):
    M, N, K = 32, 96, 512
    A = si.bf16_to_f32_numpy(si.activations(M, K, seed=31, outliers=True))
    W = si.weights(N, K, seed=32)
    Aq, sa = orc.quant_act("W8A8_INT8", A)
    Wq, sw = orc.quant_weight("W8A8_INT8", W)
    acc, _ = orc.gemm("W8A8_INT8", Aq, sa, Wq, sw)
    ref = Aq.astype(np.int64) @ Wq.astype(np.int64).T
    assert np.array_equal(acc, ref)
    ti = torch._int_mm(torch.from_numpy(Aq), torch.from_numpy(np.ascontiguousarray(Wq.T)))
    assert np.array_equal(acc, ti.numpy().astype(np.int64))


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "Block_FP8"])
def test_gemm_fp8_acc_matches_numpy_fp64(orc, fmt):
    M, N, K = 16, 200, 384
    A = si.bf16_to_f32_numpy(si.activations(M, K, seed=41, outliers=True))
    W = si.weights(N, K, seed=42)
    Aq, sa = orc.quant_act(fmt, A)
    Wq, sw = orc.quant_weight(fmt, W)
    acc, y = orc.gemm(fmt, Aq, sa, Wq, sw)
    tv = torch_e4m3_values()
    a = tv[Aq]; w = tv[Wq]
    if fmt == "FP8_Dynamic":
        ref = a @ w.T                                    # every partial sum exact in fp64
        assert np.array_equal(acc, ref)
        yref = ref * (sa.astype(np.float64)[:, None] * sw.astype(np.float64)[None, :])
    else:
        nbk = K // 128
        yref = np.zeros((M, N))
        for kb in range(nbk):
            sl = slice(kb * 128, kb * 128 + 128)
            part = a[:, sl] @ w[:, sl].T
            yref += (sa[:, kb].astype(np.float64)[:, None] * np.repeat(sw[:, kb], 128)[:N][None, :].astype(np.float64)) * part
        assert np.allclose(acc, yref, rtol=1e-13, atol=0)
    want = torch.from_numpy(yref).to(torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    # torch rounds fp64 -> fp32 -> bf16 (two roundings); allow that to differ by one ulp
    diff = np.abs(y.astype(np.int32) - want.astype(np.int32))
    assert diff.max() <= 1 and (diff == 0).mean() > 0.99


def test_gemm_identity_weight_returns_dequantized_activation(orc):
    K = 256
    A = si.bf16_to_f32_numpy(si.activations(4, K, seed=51))
    W = np.eye(K, dtype=np.float32)
    tv = torch_e4m3_values()
    for fmt in ("FP8_Dynamic", "W8A8_INT8", "Block_FP8"):
        Aq, sa = orc.quant_act(fmt, A)
        Wq, sw = orc.quant_weight(fmt, W)
        if fmt == "W8A8_INT8":
            assert np.all(np.diag(Wq) == 127) and np.all(sw == np.float32(1) / np.float32(127))
            deq = Aq.astype(np.float64) * sa[:, None] * (127 * np.float64(sw[0]))
        elif fmt == "FP8_Dynamic":
            assert np.all(np.diag(Wq) == 0x7E)
            deq = tv[Aq] * sa[:, None] * (448 * np.float64(sw[0]))
        else:
            assert sw[0, 1] == 1.0 and sw[1, 0] == 1.0           # all-zero off-diagonal blocks
            deq = tv[Aq] * np.repeat(sa, 128, 1) * (448 * np.float64(sw[0, 0]))
        _, y = orc.gemm(fmt, Aq, sa, Wq, sw)
        want = np.array([frac_bf16_bits(float(v)) for v in deq.ravel()], np.uint16).reshape(deq.shape)
        assert np.array_equal(y, want), fmt


def test_gemm_one_hot_weight_picks_a_column(orc):
    K, N = 128, 5
    A = si.bf16_to_f32_numpy(si.activations(3, K, seed=61))
    W = np.zeros((N, K), np.float32)
    cols = [0, 17, 64, 100, 127]
    for n, c in enumerate(cols):
        W[n, c] = -0.75 if n % 2 else 2.0
    for fmt in ("FP8_Dynamic", "W8A8_INT8"):
        Aq, sa = orc.quant_act(fmt, A)
        Wq, sw = orc.quant_weight(fmt, W)
        acc, _ = orc.gemm(fmt, Aq, sa, Wq, sw)
        for n, c in enumerate(cols):
            qw = int(Wq[n, c]) if fmt == "W8A8_INT8" else torch_e4m3_values()[Wq[n, c]]
            qa = Aq[:, c].astype(np.float64) if fmt == "W8A8_INT8" else torch_e4m3_values()[Aq[:, c]]
            assert np.array_equal(acc[:, n].astype(np.float64), qa * qw)
            assert (Wq[n, c] == (-127 if n % 2 else 127)) if fmt == "W8A8_INT8" else (Wq[n, c] == (0xFE if n % 2 else 0x7E))


@pytest.mark.parametrize("fmt", ["FP8_Dynamic", "W8A8_INT8", "Block_FP8"])
def test_gemm_invariant_under_k_permutation(orc, fmt):
    # The order in which K is split or walked (Split-K, Swap-AB, tiles) must not
    # change the exact accumulator.  Permuting K inside 128-groups keeps the
    # Block_FP8 grouping; the other formats take any permutation.
    M, N, K = 4, 40, 512
    A = si.bf16_to_f32_numpy(si.activations(M, K, seed=71))
    W = si.weights(N, K, seed=72)
    Aq, sa = orc.quant_act(fmt, A)
    Wq, sw = orc.quant_weight(fmt, W)
    rng = np.random.default_rng(7)
    if fmt == "Block_FP8":
        perm = np.concatenate([g * 128 + rng.permutation(128) for g in range(K // 128)])
    else:
        perm = rng.permutation(K)
    acc0, y0 = orc.gemm(fmt, Aq, sa, Wq, sw)
    acc1, y1 = orc.gemm(fmt, np.ascontiguousarray(Aq[:, perm]), sa, np.ascontiguousarray(Wq[:, perm]), sw)
    if fmt == "Block_FP8":
        assert np.allclose(acc0, acc1, rtol=1e-12, atol=0)
    else:
        assert np.array_equal(acc0, acc1)
    assert np.array_equal(y0, y1)


def test_gemm_column_subset_equals_full(orc):
    M, N, K = 3, 300, 256
    A = si.bf16_to_f32_numpy(si.activations(M, K, seed=81))
    W = si.weights(N, K, seed=82)
    for fmt in ("FP8_Dynamic", "W8A8_INT8", "Block_FP8"):
        Aq, sa = orc.quant_act(fmt, A)
        Wq, sw = orc.quant_weight(fmt, W)
        acc, y = orc.gemm(fmt, Aq, sa, Wq, sw)
        ns = np.array([299, 0, 128, 5, 255])
        acc2, y2 = orc.gemm(fmt, Aq, sa, Wq, sw, ns=ns)
        assert np.array_equal(acc[:, ns], acc2) and np.array_equal(y[:, ns], y2)


def test_abs_magnitude_bounds_the_accumulator(orc):
    M, N, K = 4, 64, 256
    A = si.bf16_to_f32_numpy(si.activations(M, K, seed=91))
    W = si.weights(N, K, seed=92)
    for fmt in ("FP8_Dynamic", "Block_FP8"):
        Aq, sa = orc.quant_act(fmt, A)
        Wq, sw = orc.quant_weight(fmt, W)
        acc, _ = orc.gemm(fmt, Aq, sa, Wq, sw)
        mag = orc.abs_magnitude(fmt, Aq, sa, Wq, sw)
        y = acc if fmt == "Block_FP8" else acc * sa[:, None].astype(np.float64) * sw[None, :].astype(np.float64)
        assert np.all(np.abs(y) <= mag * (1 + 1e-12))
        tv = torch_e4m3_values()
        if fmt == "FP8_Dynamic":
            ref = (np.abs(tv[Aq]) @ np.abs(tv[Wq]).T) * sa[:, None].astype(np.float64) * sw[None, :].astype(np.float64)
            assert np.allclose(mag, ref, rtol=1e-13)


def _blocky_inputs(M, N, K, seed):
    """Activations and weights whose 1x128 groups and 128x128 blocks have
    clearly different magnitudes (factor 1 + group / block index), so that a
    scale taken from the wrong group or block changes the result by several
    percent."""
    A = si.bf16_to_f32_numpy(si.activations(M, K, seed=seed))
    A = A * np.repeat(1.0 + np.arange((K + 127) // 128), 128)[None, :K].astype(np.float32)
    A = si.bf16_to_f32_numpy(torch.from_numpy(A.astype(np.float32)).to(torch.bfloat16))
    W = si.weights(N, K, seed=seed + 1)
    fac = (1.0 + 2.0 * np.arange((N + 127) // 128))[:, None] * (1.0 + 0.5 * np.arange((K + 127) // 128))[None, :]
    W = (W * np.repeat(np.repeat(fac, 128, 0), 128, 1)[:N, :K]).astype(np.float32)
    return A, W


def test_block_abs_magnitude_equals_exact_rationals(orc):
    # Fraction brute force of the magnitude the Block_FP8 bound multiplies,
    # sum_kb s_a[m,kb] * s_w[n/128,kb] * sum_{k in kb} |a_q * w_q|, term by
    # term from independent decode tables (ragged N: the third block row
    # has 44 rows)
    M, N, K = 2, 300, 384
    A, W = _blocky_inputs(M, N, K, seed=93)
    Aq, sa = orc.quant_act("Block_FP8", A)
    Wq, sw = orc.quant_weight("Block_FP8", W)
    ns = np.array([0, 127, 128, 200, 255, 256, 299])
    mag = orc.abs_magnitude("Block_FP8", Aq, sa, Wq, sw, ns=ns)
    for m in range(M):
        for j, n in enumerate(ns):
            exact = Fraction(0)
            for kb in range(K // 128):
                part = sum(abs(_frac_e4m3(int(Aq[m, k])) * _frac_e4m3(int(Wq[n, k])))
                           for k in range(kb * 128, kb * 128 + 128))
                exact += Fraction(float(sa[m, kb])) * Fraction(float(sw[n // 128, kb])) * part
            assert abs(Fraction(float(mag[m, j])) - exact) <= exact * Fraction(1, 2 ** 45)


def test_block_abs_magnitude_per_block_numpy(orc):
    # the same magnitude from numpy, one 128-K group at a time with that
    # group's activation scale and the weight scale of the row's block
    M, N, K = 3, 300, 512
    A, W = _blocky_inputs(M, N, K, seed=95)
    Aq, sa = orc.quant_act("Block_FP8", A)
    Wq, sw = orc.quant_weight("Block_FP8", W)
    assert len(np.unique(sw)) == sw.size               # every block has its own scale
    tv = np.abs(torch_e4m3_values())
    ref = np.zeros((M, N))
    for kb in range(K // 128):
        ks = slice(kb * 128, kb * 128 + 128)
        part = tv[Aq[:, ks]] @ tv[Wq[:, ks]].T                           # [M, N]
        coef = sa[:, kb].astype(np.float64)[:, None] * sw[np.arange(N) // 128, kb].astype(np.float64)[None, :]
        ref += coef * part
    mag = orc.abs_magnitude("Block_FP8", Aq, sa, Wq, sw)
    assert np.allclose(mag, ref, rtol=1e-13, atol=0)
    # a plausible slip, a per-channel magnitude (one scale per row and column),
    # is far from it
    wrong = (tv[Aq] @ tv[Wq].T) * sa[:, :1].astype(np.float64) * sw[np.arange(N) // 128, :1].T.astype(np.float64)
    assert np.max(np.abs(wrong - ref) / ref) > 0.05
