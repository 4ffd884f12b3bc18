"""Host-side checks of the C ABI (no GPU): the library loads and exports every
symbol include/qgemm.h declares, argument validation returns the documented
status codes before any device work, workspace sizing, and the per-shape
config table ("Per-shape Config Tuning" / "Hybrid Dispatch" of "Building a
High-Performance and Portable vLLM Linear Backend with Helion")."""
from __future__ import annotations

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "qgemm.h")


@pytest.fixture(scope="module")
def q():
    from quantized_gemm_decode_02_b300 import qgemm
    return qgemm


def header_symbols():
    txt = open(HEADER).read()
    return sorted(set(re.findall(r"QG_API\s+[\w\s\*]*?\b(qg_\w+)\s*\(", txt)))


def test_header_declares_the_entry_points():
    syms = header_symbols()
    for s in ("qg_quant_act", "qg_quant_weight", "qg_gemm_w8a8", "qg_select", "qg_workspace_bytes",
              "qg_load_table", "qg_last_error"):
        assert s in syms


def test_library_exports_every_declared_symbol(q):
    out = subprocess.run(["nm", "-D", "--defined-only", q.LIB_PATH], capture_output=True, text=True, check=True).stdout
    exported = set(re.findall(r"\bT (qg_\w+)", out))
    missing = [s for s in header_symbols() if s not in exported]
    assert not missing, missing
    assert set(q.EXPORTS) == set(header_symbols())
    lib = ctypes.CDLL(q.LIB_PATH)
    for s in header_symbols():
        assert getattr(lib, s) is not None


def test_header_compiles_as_c():
    src = '#include "qgemm.h"\nint main(void){ return QG_OK + QG_SWAPAB_SPLITK * 0; }\n'
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), "-x", "c", "-",
                        "-fsyntax-only"], input=src, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def _raw(q):
    return q._lib


BAD16 = 0x10008  # 8-byte aligned only; never dereferenced (validation fails first)
OK16 = 0x10000


def test_quant_act_validation(q):
    lib = _raw(q)
    assert lib.qg_quant_act(7, OK16, 1, 128, 128, OK16, OK16, None) == q.QG_ERR_INVALID_ARG
    assert lib.qg_quant_act(0, None, 1, 128, 128, OK16, OK16, None) == q.QG_ERR_INVALID_ARG
    assert lib.qg_quant_act(0, OK16, 1, 120, 120, OK16, OK16, None) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert lib.qg_quant_act(2, OK16, 1, 144, 144, OK16, OK16, None) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert lib.qg_quant_act(0, BAD16, 1, 128, 128, OK16, OK16, None) == q.QG_ERR_ALIGNMENT
    assert lib.qg_quant_act(0, OK16, 1, 128, 132, OK16, OK16, None) == q.QG_ERR_ALIGNMENT
    assert lib.qg_quant_act(0, OK16, 1, 128, 64, OK16, OK16, None) == q.QG_ERR_INVALID_ARG
    assert lib.qg_quant_act(0, None, 0, 128, 128, None, None, None) == q.QG_OK  # M == 0: no-op
    assert "K" in q.qg_last_error() or q.qg_last_error() != ""


def test_quant_weight_validation(q):
    lib = _raw(q)
    assert lib.qg_quant_weight(1, OK16, 0, 128, OK16, OK16, None) == q.QG_ERR_INVALID_ARG
    assert lib.qg_quant_weight(1, OK16, 4, 40, OK16, OK16, None) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert lib.qg_quant_weight(1, BAD16, 4, 128, OK16, OK16, None) == q.QG_ERR_ALIGNMENT


def _gemm(q, fmt=0, M=4, N=256, K=256, A=OK16, sa=OK16, W=OK16, sw=OK16, Y=OK16, ldy=None, variant=2, split=1,
          cfg=0, ws=None, wsb=0, dbg=None):
    return _raw(q).qg_gemm_w8a8(fmt, M, N, K, A, sa, W, sw, Y, N if ldy is None else ldy, variant, split, cfg, ws,
                                wsb, dbg, None)


def test_gemm_validation(q):
    assert _gemm(q, fmt=5) == q.QG_ERR_INVALID_ARG
    assert _gemm(q, variant=9) == q.QG_ERR_INVALID_ARG
    assert _gemm(q, ldy=100) == q.QG_ERR_INVALID_ARG
    assert _gemm(q, A=None) == q.QG_ERR_INVALID_ARG
    assert _gemm(q, K=200) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert _gemm(q, fmt=2, K=272) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert _gemm(q, A=BAD16) == q.QG_ERR_ALIGNMENT
    assert _gemm(q, W=BAD16) == q.QG_ERR_ALIGNMENT
    assert _gemm(q, split=2) == q.QG_ERR_INVALID_ARG                    # split needs a *_SPLITK variant
    assert _gemm(q, variant=3, split=3) == q.QG_ERR_UNSUPPORTED_SHAPE     # > ceil(K/128) = 2
    assert _gemm(q, variant=3, split=0) == q.QG_ERR_UNSUPPORTED_SHAPE
    # Split-K through the workspace: Standard split-K, or Swap-AB with more
    # than 16 ranges (up to 16 reduce inside a thread-block cluster)
    assert _gemm(q, variant=1, split=2) == q.QG_ERR_WORKSPACE_TOO_SMALL   # no workspace
    assert _gemm(q, variant=1, split=2, ws=OK16, wsb=16) == q.QG_ERR_WORKSPACE_TOO_SMALL
    assert _gemm(q, K=4096, variant=3, split=20) == q.QG_ERR_WORKSPACE_TOO_SMALL
    assert _gemm(q, fmt=1, M=8, variant=0) == q.QG_ERR_UNSUPPORTED_SHAPE  # INT8 runs Swap-AB
    # the CUDA-core (dp4a) variants: W8A8_INT8 with M <= 8 only
    assert _gemm(q, fmt=1, M=9, variant=q.QG_SWAPAB_DP4A) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert _gemm(q, fmt=0, M=1, variant=q.QG_SWAPAB_DP4A) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert _gemm(q, fmt=1, M=1, variant=q.QG_SWAPAB_DP4A, split=2) == q.QG_ERR_INVALID_ARG
    assert _gemm(q, fmt=1, M=1, variant=6) == q.QG_ERR_INVALID_ARG
    assert _gemm(q, fmt=0, dbg=OK16) == q.QG_ERR_INVALID_ARG              # debug acc is INT8 only
    assert _gemm(q, cfg=17) == q.QG_ERR_INVALID_ARG                       # ring depth above 16
    assert _gemm(q, cfg=q.config_id(0, 65)) == q.QG_ERR_INVALID_ARG       # prefetch distance above 64
    assert _gemm(q, cfg=1 << 13) == q.QG_ERR_INVALID_ARG                  # unknown bit
    assert _gemm(q, cfg=q.config_id(0, 0, True)) == q.QG_ERR_INVALID_ARG  # wide tiles: FP8 Standard only
    assert _gemm(q, cfg=-1) == q.QG_ERR_INVALID_ARG
    assert _gemm(q, M=0) == q.QG_OK


def test_workspace_bytes(q):
    assert q.qg_workspace_bytes(0, 4, 256, 1024, q.QG_SWAPAB, 1) == 0
    # Swap-AB with <= 16 ranges reduces in distributed shared memory: no workspace
    assert q.qg_workspace_bytes(0, 4, 256, 1024, q.QG_SWAPAB_SPLITK, 3) == 0
    assert q.qg_workspace_bytes(1, 32, 4096, 2048, q.QG_SWAPAB_SPLITK, 16) == 0
    # counters (tiles x 4 bytes, rounded up to 256) + splits * M * N * 4
    assert q.qg_workspace_bytes(1, 32, 4096, 4096, q.QG_SWAPAB_SPLITK, 17) == 256 + 17 * 32 * 4096 * 4
    assert q.qg_workspace_bytes(0, 300, 256, 1024, q.QG_SPLITK, 2) == 256 + 2 * 300 * 256 * 4
    assert q.qg_workspace_bytes(0, 4, 256, 1024, q.QG_SWAPAB_SPLITK, 99) == 0  # invalid -> 0
    assert q.qg_workspace_bytes(1, 8, 4096, 4096, q.QG_SWAPAB_DP4A_SPLITK, 16) == 0
    assert q.qg_workspace_bytes(1, 8, 4096, 4096, q.QG_SWAPAB_DP4A_SPLITK, 17) == 256 + 17 * 8 * 4096 * 4
    assert q.qg_workspace_bytes(1, 9, 4096, 4096, q.QG_SWAPAB_DP4A_SPLITK, 2) == 0  # M > 8 -> invalid


def _grouped(q, fmt=0, groups=4, offs=OK16, total=8, max_tokens=4, N=256, K=256, variant=2, split=1, cfg=0):
    return _raw(q).qg_gemm_w8a8_grouped(fmt, groups, offs, total, max_tokens, N, K, OK16, OK16, OK16, OK16, OK16, N,
                                        variant, split, cfg, None, 0, None, None)


def test_workspace_bytes_config(q):
    pw = q.QG_CONFIG_I8_PREWIDEN
    # the fp16 activation copy after the (256-byte aligned) Split-K part
    assert q.qg_workspace_bytes_config(1, 300, 640, 4096, q.QG_SWAPAB_SPLITK, 3, pw) == 300 * 4096 * 2
    split_part = ((5 * 19 * 4 + 255) // 256) * 256 + 18 * 300 * 640 * 4
    assert q.qg_workspace_bytes(1, 300, 640, 4096, q.QG_SWAPAB_SPLITK, 18) == split_part
    assert q.qg_workspace_bytes_config(1, 300, 640, 4096, q.QG_SWAPAB_SPLITK, 18, pw) == \
        (split_part + 255) // 256 * 256 + 300 * 4096 * 2
    assert q.qg_workspace_bytes_config(1, 7, 640, 4112, q.QG_SWAPAB, 1, pw) == (7 * 4112 * 2 + 255) // 256 * 256
    # other configs: as qg_workspace_bytes; invalid ones: 0
    assert q.qg_workspace_bytes_config(0, 16, 640, 4096, q.QG_SWAPAB_SPLITK, 18, 0) == \
        q.qg_workspace_bytes(0, 16, 640, 4096, q.QG_SWAPAB_SPLITK, 18)
    assert q.qg_workspace_bytes_config(0, 16, 640, 4096, q.QG_SWAPAB, 1, pw) == 0


def test_grouped_validation(q):
    # every check below returns before any device work
    assert _grouped(q, groups=0) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert _grouped(q, groups=70000) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert _grouped(q, offs=None) == q.QG_ERR_INVALID_ARG
    assert _grouped(q, offs=OK16 + 2) == q.QG_ERR_INVALID_ARG            # unaligned offsets
    assert _grouped(q, variant=0) == q.QG_ERR_INVALID_ARG                # Standard
    assert _grouped(q, variant=4, fmt=0) == q.QG_ERR_UNSUPPORTED_SHAPE   # dp4a is INT8 only
    assert _grouped(q, variant=4, fmt=1, max_tokens=9) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert _grouped(q, K=200) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert _grouped(q, total=-1) == q.QG_ERR_INVALID_ARG
    assert _grouped(q, split=17, K=4096, variant=3) == q.QG_ERR_WORKSPACE_TOO_SMALL
    assert _grouped(q, fmt=1, cfg=q.QG_CONFIG_I8_PREWIDEN) == q.QG_ERR_INVALID_ARG   # not for grouped launches
    assert _grouped(q, fmt=1, cfg=q.QG_CONFIG_I8_CONV16) == q.QG_ERR_INVALID_ARG
    assert _grouped(q, fmt=2, cfg=q.QG_CONFIG_BLOCK_PROMO8) == q.QG_ERR_INVALID_ARG
    assert _grouped(q, total=0) == q.QG_OK                               # no tokens: nothing to do
    assert _grouped(q, max_tokens=0) == q.QG_OK


def test_grouped_workspace_bytes(q):
    # cluster reductions need none; the workspace holds counters for every
    # group's tiles and [splits][total_tokens][N] partials
    assert q.qg_workspace_bytes_grouped(0, 8, 40, 16, 4096, 4096, q.QG_SWAPAB_SPLITK, 4) == 0
    tiles = 8 * 32 * 1
    assert q.qg_workspace_bytes_grouped(0, 8, 40, 16, 4096, 4096, q.QG_SWAPAB_SPLITK, 17) == \
        ((tiles * 4 + 255) // 256) * 256 + 17 * 40 * 4096 * 4
    assert q.qg_workspace_bytes_grouped(1, 8, 40, 9, 4096, 4096, q.QG_SWAPAB_DP4A_SPLITK, 17) == 0  # invalid
    assert q.qg_workspace_bytes_grouped(0, 0, 40, 16, 4096, 4096, q.QG_SWAPAB, 1) == 0


def test_launch_flag_and_limits(q):
    assert _raw(q).qg_set_launch_flags(6) == q.QG_ERR_INVALID_ARG
    q.qg_set_launch_flags(0)
    q.qg_set_wait_limit_ns(0)


def test_table_select(q, tmp_path):
    t = tmp_path / "t.tsv"
    t.write_text("# fmt N K M variant split config\n"
                 "1\t2048\t2048\t1\t3\t8\t0\n"
                 "1\t2048\t2048\t8\t3\t4\t6\n"
                 "1\t2048\t2048\t32\t2\t1\t0\n")
    q.qg_load_table(str(t))
    q.qg_set_allow_default(False)
    assert q.qg_select("W8A8_INT8", 1, 2048, 2048) == (3, 8, 0)
    assert q.qg_select("W8A8_INT8", 2, 2048, 2048) == (3, 4, 6)    # next tuned M >= 2 is 8
    assert q.qg_select("W8A8_INT8", 24, 2048, 2048) == (2, 1, 0)
    v, s, c = q.qg_select("W8A8_INT8", 100, 2048, 2048)             # beyond the tuned range -> default
    assert v in (q.QG_SWAPAB, q.QG_SWAPAB_SPLITK, q.QG_STANDARD, q.QG_SPLITK) and s >= 1
    with pytest.raises(q.QGError) as e:
        q.qg_select("W8A8_INT8", 1, 4096, 2048)                     # missing shape
    assert e.value.code == q.QG_ERR_NO_CONFIG
    q.qg_set_allow_default(True)
    v, s, c = q.qg_select("W8A8_INT8", 1, 4096, 2048)
    assert v == q.QG_SWAPAB_SPLITK and 1 <= s <= 16
    q.qg_set_allow_default(False)
    bad = tmp_path / "bad.tsv"
    bad.write_text("1 2048 2048 1 3\n")
    with pytest.raises(q.QGError) as e:
        q.qg_load_table(str(bad))
    assert e.value.code == q.QG_ERR_TABLE_PARSE
    with pytest.raises(q.QGError):
        q.qg_load_table(str(tmp_path / "missing.tsv"))
    empty = tmp_path / "empty.tsv"
    empty.write_text("# nothing\n")
    q.qg_load_table(str(empty))


def test_default_config_fills_the_gpu(q):
    q.qg_set_allow_default(True)
    try:
        for (M, N, K) in [(1, 2048, 2048), (32, 12288, 2048), (1, 5120, 25600), (32, 51200, 5120)]:
            v, s, c = q.qg_select("FP8_Dynamic", M, N, K)
            tiles = (N + 127) // 128
            assert v in (q.QG_SWAPAB, q.QG_SWAPAB_SPLITK)
            assert s == 1 or tiles * s <= 2 * 148      # two CTA slots per SM
            assert s <= 16                              # one cluster reduces the splits
            assert s <= max(1, ((K + 127) // 128) // 2)
        v, s, c = q.qg_select("FP8_Dynamic", 256, 4096, 4096)
        assert v in (q.QG_STANDARD, q.QG_SPLITK)
    finally:
        q.qg_set_allow_default(False)


def test_check_config_returns_the_gemm_status(q):
    """qg_check_config gives, without pointers, the status qg_gemm_w8a8
    returns for the same configuration's pointer-free checks."""
    cases = [dict(fmt=5), dict(variant=9), dict(K=200), dict(fmt=2, K=272), dict(split=2), dict(variant=3, split=3),
             dict(variant=3, split=0), dict(fmt=1, M=8, variant=0), dict(fmt=1, M=9, variant=q.QG_SWAPAB_DP4A),
             dict(fmt=0, M=1, variant=q.QG_SWAPAB_DP4A), dict(cfg=17), dict(cfg=q.config_id(0, 65)),
             dict(cfg=1 << 13), dict(cfg=q.config_id(0, 0, True)), dict(cfg=-1), dict(cfg=1),
             dict(fmt=1, M=8, cfg=q.QG_CONFIG_MMA_S8),                               # s8 without mma.sync
             dict(fmt=0, M=8, cfg=q.config_id(s8=True)),
             dict(fmt=0, M=300, variant=0, cfg=q.QG_CONFIG_PAIR_MMA),                # pair MMA without persist
             dict(fmt=2, M=300, variant=0, cfg=q.config_id(pair_mma=True)),
             dict(fmt=0, M=300, cfg=q.QG_CONFIG_I8_PREWIDEN),                          # prewiden: INT8 only
             dict(fmt=1, M=300, cfg=q.QG_CONFIG_I8_PREWIDEN | q.QG_CONFIG_MMA_SYNC),
             dict(fmt=1, M=300, variant=q.QG_SWAPAB_DP4A, cfg=q.QG_CONFIG_I8_PREWIDEN),
             dict(fmt=2, M=32, cfg=q.QG_CONFIG_I8_CONV16),                              # conv16: INT8 only
             dict(fmt=1, M=32, cfg=q.QG_CONFIG_I8_CONV16 | q.QG_CONFIG_FUSED_QUANT),
             dict(fmt=0, M=32, cfg=q.QG_CONFIG_BLOCK_PROMO8),                           # promo8: Block_FP8 only
             dict(fmt=1, M=32, cfg=q.QG_CONFIG_BLOCK_PROMO8),
             dict(fmt=2, M=300, variant=0, cfg=q.QG_CONFIG_BLOCK_PROMO8),               # Swap-AB only
             dict(fmt=2, M=32, cfg=q.QG_CONFIG_BLOCK_PROMO8 | q.QG_CONFIG_FUSED_QUANT),
             dict(fmt=0, M=300, variant=0, cfg=1 << q.QG_CONFIG_PERSIST_ROWS_SHIFT)]  # rows without persist
    for c in cases:
        fmt, M, K = c.get("fmt", 0), c.get("M", 4), c.get("K", 256)
        v, s, cfg = c.get("variant", 2), c.get("split", 1), c.get("cfg", 0)
        want = _gemm(q, fmt=fmt, M=M, K=K, variant=v, split=s, cfg=cfg)
        assert want != q.QG_OK
        assert q.qg_check_config(fmt, M, 256, K, v, s, cfg) == want, c
    # accepted configurations (never launched here)
    assert q.qg_check_config(1, 8, 4096, 2048, q.QG_SWAPAB_DP4A_SPLITK, 16, 0) == q.QG_OK
    assert q.qg_check_config(1, 24, 4096, 4096, q.QG_SWAPAB_SPLITK, 4, q.config_id(s8=True)) == q.QG_OK
    assert q.qg_check_config(1, 8, 4096, 4096, q.QG_SWAPAB, 1, q.config_id(narrow=True, s8=True)) == q.QG_OK
    assert q.qg_check_config(1, 16, 4096, 4096, q.QG_SWAPAB, 1, q.config_id(dp4a_rows16=4, s8=True)) == q.QG_OK
    assert q.qg_check_config(1, 17, 4096, 4096, q.QG_SWAPAB, 1,
                             q.config_id(dp4a_rows16=1, s8=True)) == q.QG_ERR_UNSUPPORTED_SHAPE
    assert q.qg_check_config(0, 300, 4096, 4096, q.QG_SPLITK, 3, q.config_id(4, 0, True)) == q.QG_OK
    assert q.qg_check_config(0, 512, 24576, 4096, q.QG_STANDARD, 1, q.config_id(3, 8, pair_mma=True)) == q.QG_OK
    assert q.qg_check_config(1, 16, 4096, 4096, q.QG_SWAPAB_SPLITK, 4, q.config_id(conv16=True)) == q.QG_OK
    assert q.qg_check_config(1, 300, 4096, 4096, q.QG_SWAPAB, 1, q.config_id(prewiden=True, conv16=True)) == q.QG_OK
    assert q.qg_check_config(2, 512, 4096, 4096, q.QG_SWAPAB_SPLITK, 2, q.config_id(6, promo8=True)) == q.QG_OK
    for rows in (224, 192, 160):
        assert q.qg_check_config(0, 512, 24576, 4096, q.QG_STANDARD, 1,
                                 q.config_id(pair_mma=True, persist_rows=rows)) == q.QG_OK
    with pytest.raises(ValueError):
        q.config_id(persist_rows=200)
    assert q.qg_check_config(2, 32, 4096, 12288, q.QG_SWAPAB_SPLITK, 96, q.config_id(12, 64)) == q.QG_OK
    assert q.qg_check_config(0, 0, 256, 256, 2, 1, 0) == q.QG_ERR_INVALID_ARG   # a configuration has M >= 1


def test_table_rows_are_checked_at_load(q, tmp_path):
    good = tmp_path / "good.tsv"
    good.write_text("1\t2048\t2048\t8\t5\t2\t0\n")
    q.qg_load_table(str(good))
    for row, why in [("1\t2048\t2048\t16\t5\t2\t0\n", "dp4a above 8 tokens"),
                     ("1\t2048\t2048\t8\t0\t1\t0\n", "INT8 Standard"),
                     ("0\t2048\t2048\t8\t3\t17\t0\n", "split_k above ceil(K/128)"),
                     ("0\t2048\t2048\t8\t2\t1\t4096\n", "wide tiles on Swap-AB"),
                     ("2\t2048\t2000\t8\t2\t1\t0\n", "Block_FP8 K % 128")]:
        bad = tmp_path / "bad.tsv"
        bad.write_text("# ok row first\n1\t4096\t2048\t1\t4\t1\t0\n" + row)
        with pytest.raises(q.QGError) as e:
            q.qg_load_table(str(bad))
        assert e.value.code == q.QG_ERR_TABLE_PARSE, why
        assert "bad.tsv:3" in q.qg_last_error(), why
    # a rejected file leaves the loaded table in place
    q.qg_set_allow_default(False)
    assert q.qg_select("W8A8_INT8", 5, 2048, 2048) == (q.QG_SWAPAB_DP4A_SPLITK, 2, 0)
    with pytest.raises(q.QGError):
        q.qg_select("W8A8_INT8", 1, 4096, 2048)


def test_shipped_table_covers_every_bench_workload(q):
    """Every (format, shape, token count) bench.py and its workloads launch
    has a tuned row, and the row is a configuration the GEMM accepts."""
    import bench
    import seeded_inputs as si
    q.qg_load_table(bench.TABLE)
    q.qg_set_allow_default(False)
    seen = set()
    for name, wl in bench.WORKLOADS.items():
        for fmt, model, layer, M in wl["items"]:
            K, N = si.QWEN3_LINEARS[model][layer]
            if (fmt, M, N, K) in seen:
                continue
            seen.add((fmt, M, N, K))
            v, s, c = q.qg_select(fmt, M, N, K)
            assert q.qg_check_config(fmt, M, N, K, v, s, c) == q.QG_OK, (name, fmt, model, layer, M)
    assert len(seen) > 300


def test_tuner_candidates_are_accepted(q):
    """The offline sweep only times configurations the GEMM accepts."""
    from quantized_gemm_decode_02_b300 import tune
    n = 0
    for fmt in tune.FMT_ID:
        for shapes in tune.SHAPES.values():
            for K, N in shapes.values():
                for M in tune.TUNED_M + (64, 128, 256, 384, 512):
                    for v, s, c in tune.candidates(fmt, M, N, K, 148):
                        assert q.qg_check_config(fmt, M, N, K, v, s, c) == q.QG_OK, (fmt, M, N, K, v, s, c)
                        n += 1
    assert n > 1000
