"""Offline per-shape config sweep: writes the table that qg_select reads.

"Per-shape Config Tuning" of "Building a High-Performance and Portable vLLM
Linear Backend with Helion" tunes every (model GEMM shape x num_tokens)
separately, with the candidates benchmarked under CUDA graphs the way they
will run ("Enable CUDA Graph for Autotuner Benchmarking").  This sweep keeps
that method and replaces the page's LLM-seeded tree search with an exhaustive
walk over a small grid: for every format, shape and tuned token count it
times each candidate (variant, split_k, ring depth) as a CUDA graph of R
GEMM launches (qg_gemm_w8a8; with --linear, whole linear layers through
qg_linear_w8a8 instead) over rotated weight copies (more than three L2
capacities, so the weights stream from HBM), with programmatic dependent
launch on, and keeps the fastest.  With --prefetch-pass a second pass tries
the winner with an L2 prefetch distance of 1, 2 and 4 weight k-tiles
(config_id's upper bits) and keeps one only when it is more than 1% faster.
The shipped table is swept without it: distances that won in these
same-shape chains lost in the mixed-shape chains of bench.py.

Rows already present in the output table are skipped, so an interrupted
sweep resumes where it stopped.

With --layer-context TABLE_IN the rows are re-tuned where they run (for
Block_FP8 also the one-kernel form of the linear, QG_CONFIG_FUSED_QUANT): for
each token count the candidates of one linear are timed inside the chain
of the whole decoder layer (activation quantization and GEMM of qkv, o,
gate_up and down in order, one CUDA graph with programmatic dependent
launch), the other linears keeping their current rows, one linear after
the other.  A linear's best configuration depends on its neighbours there
(which SMs the previous GEMM still holds when its thread-block clusters
are placed, how much of its weights it streams before its dependency
wait), which a chain of one shape does not show.

Usage:  python -m quantized_gemm_decode_02_b300.tune --out TABLE
            [--formats FP8_Dynamic,W8A8_INT8,Block_FP8]
            [--models Qwen3-1.7B,Qwen3-8B,Qwen3-32B] [--ms 1,2,4,8,16,24,32]
The decode table covers the tuned token counts; a second pass with
--ms 64,128,256,384,512 adds rows for the compute-bound regime.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import sys
import time

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from quantized_gemm_decode_02_b300 import qgemm as q  # noqa: E402

# Linear-layer shapes (K = in_features, N = out_features) of the Qwen3 models
# whose GEMMs the pages tune.
SHAPES = {
    "Qwen3-1.7B": {"qkv": (2048, 4096), "o": (2048, 2048), "gate_up": (2048, 12288), "down": (6144, 2048)},
    "Qwen3-8B": {"qkv": (4096, 6144), "o": (4096, 4096), "gate_up": (4096, 24576), "down": (12288, 4096)},
    "Qwen3-32B": {"qkv": (5120, 10240), "o": (8192, 5120), "gate_up": (5120, 51200), "down": (25600, 5120)},
}
TUNED_M = (1, 2, 4, 8, 16, 24, 32)
FMT_ID = {"FP8_Dynamic": 0, "W8A8_INT8": 1, "Block_FP8": 2}
POOL_BYTES = 512 << 20
PREFETCH_DISTANCES = (1, 2, 4)  # weight k-tiles each CTA keeps requested into L2 ahead of its ring
# kernel forms that qg_linear_w8a8 runs only as quantization kernel + GEMM
NOT_FUSABLE = (q.QG_CONFIG_MMA_SYNC | q.QG_CONFIG_I8_PREWIDEN | q.QG_CONFIG_I8_CONV16 | q.QG_CONFIG_BLOCK_PROMO8)


def candidates(fmt: str, M: int, N: int, K: int, sms: int):
    """(variant, split_k, config_id) candidates for one shape: Swap-AB with
    and without Split-K (reduced in a cluster, up to 16 ranges) for every M
    (in blocks of 64 tokens above 64); for W8A8_INT8 at M <= 8 also their
    CUDA-core (dp4a) forms, and for W8A8_INT8 at every M the mma.sync forms
    (QG_CONFIG_MMA_SYNC, widened or QG_CONFIG_MMA_S8), and from 64 tokens on
    its pre-widened form (QG_CONFIG_I8_PREWIDEN); for Block_FP8 Swap-AB with
    eight promotion warps (QG_CONFIG_BLOCK_PROMO8); above 32 tokens also the Standard variant of the
    E4M3 formats (FP8_Dynamic also with 256-row weight tiles).  Ring depth:
    0 = two CTAs per SM, 12 = one deep ring per SM (6 for Standard, whose
    stages are twice as large)."""
    n_tiles = (N + 127) // 128
    kt = (K + 127) // 128
    mpad = 16 if M <= 16 else (32 if M <= 32 else 64)
    tiles = n_tiles * -(-M // mpad)
    out = []
    swap_forms = [(q.QG_SWAPAB, q.QG_SWAPAB_SPLITK)]
    if fmt == "W8A8_INT8" and M <= 8:
        swap_forms.append((q.QG_SWAPAB_DP4A, q.QG_SWAPAB_DP4A_SPLITK))
    cfgs = [0, 12]
    if fmt == "W8A8_INT8" and M > 8:
        # sixteen converter warps, one CTA per SM, the deepest ring
        cfgs.append(q.config_id(0, 0, conv16=True))
    if fmt == "Block_FP8":
        # eight promotion warps (QG_CONFIG_BLOCK_PROMO8)
        cfgs += [q.config_id(0, promo8=True), q.config_id(12, promo8=True)]
    for cfg in cfgs:
        for single, split in swap_forms:
            if cfg & q.QG_CONFIG_I8_CONV16 and single != q.QG_SWAPAB:
                continue
            out.append((single, 1, cfg))
            for s in range(2, min(16, kt) + 1):
                if tiles * s > 12 * sms or kt // s < 1:
                    continue
                out.append((split, s, cfg))
    if fmt == "W8A8_INT8":
        # the mma.sync form of Swap-AB (token groups of 8, blocks of 32)
        mma_tiles = n_tiles * -(-M // (8 * min(4, -(-M // 8))))
        # on f16-widened operands, and on the int8 form of the instruction
        # (no widening, B300's low int8 MMA rate: worth it at small M)
        forms = [q.config_id(ring, 0, mma_sync=True, narrow=narrow, s8=s8)
                 for s8 in (False, True) for ring, narrow in ((0, False), (12, False), (0, True), (12, True))]
        if M <= 16:
            # dp4a warps on the first 16*d rows of each tile, s8 mma.sync on
            # the rest: two pipes side by side (with the widening form the
            # dp4a rows were never faster on B300 and are not swept)
            forms += [q.config_id(0, 0, dp4a_rows16=d, s8=True) for d in (1, 2, 3, 4)]
        for cfg in forms:
            out.append((q.QG_SWAPAB, 1, cfg))
            for s in range(2, min(16, kt) + 1):
                if mma_tiles * s > 12 * sms or kt // s < 1:
                    continue
                out.append((q.QG_SWAPAB_SPLITK, s, cfg))
    if fmt == "W8A8_INT8" and M >= 64:
        # activations widened once per launch (QG_CONFIG_I8_PREWIDEN), token
        # blocks of 64 / 128: the compute-bound regime
        pw_tiles = n_tiles * -(-M // (64 if M <= 64 else 128))
        for ring, c16 in ((0, False), (3, False), (0, True)):
            cfg = q.config_id(ring, 0, prewiden=True, conv16=c16)
            out.append((q.QG_SWAPAB, 1, cfg))
            for s in range(2, min(16, kt) + 1):
                if pw_tiles * s > 4 * sms or kt // s < 1:
                    continue
                out.append((q.QG_SWAPAB_SPLITK, s, cfg))
    if M > 32 and fmt != "W8A8_INT8":
        std_tiles = n_tiles * -(-M // 128)
        for cfg in (0, 6):
            out.append((q.QG_STANDARD, 1, cfg))
            for s in (2, 3, 4, 6, 8):
                if s <= kt and std_tiles * s <= 4 * sms:
                    out.append((q.QG_SPLITK, s, cfg))
        if fmt == "FP8_Dynamic":
            # the persistent pair kernel (one CTA per SM, two TMEM
            # accumulators; the weight tile shared by TMA multicast, or each
            # CTA holding its half under cta_group::2 MMAs): deepest ring or
            # shallower ones (L2 prefetch distances were never faster)
            for pair in (False, True):
                for ring in (0, 3, 4):
                    out.append((q.QG_STANDARD, 1, q.config_id(ring, 0, persist=True, pair_mma=pair)))
            # narrower weight tiles, so that the tile count fills the last
            # round of the resident pairs better (cta_group::2 form)
            for rows in q.PERSIST_ROWS[1:]:
                out.append((q.QG_STANDARD, 1, q.config_id(0, 0, pair_mma=True, persist_rows=rows)))
            # 256-row weight tiles: ring of 2 (two CTAs per SM) or 4 (one)
            wide_tiles = -(-N // 256) * -(-M // 128)
            for cfg in (q.config_id(0, 0, True), q.config_id(4, 0, True)):
                out.append((q.QG_STANDARD, 1, cfg))
                for s in (2, 3, 4):
                    if s <= kt and wide_tiles * s <= 4 * sms:
                        out.append((q.QG_SPLITK, s, cfg))
    return out


class Bench:
    """Device buffers shared by every candidate: a pool of random weight
    bytes that launches take disjoint windows of, activations, scales, Y."""

    def __init__(self, device):
        self.device = device
        g = torch.Generator(device=device)
        g.manual_seed(1234)
        # random bytes: valid int8 codes; as E4M3 they include NaN codes,
        # which do not change the kernels' speed
        self.pool = torch.randint(0, 256, (POOL_BYTES,), dtype=torch.uint8, device=device, generator=g)
        self.A = torch.randn(512 * 25600, device=device, generator=g).to(torch.bfloat16)
        self.Aq = torch.randint(0, 256, (512 * 25600,), dtype=torch.uint8, device=device, generator=g)
        self.sa = torch.ones(512 * 256, dtype=torch.float32, device=device)
        self.sw = torch.ones(65536 * 4, dtype=torch.float32, device=device)
        self.Y = torch.empty(512 * 51200, dtype=torch.bfloat16, device=device)
        self.ws = torch.zeros(64 << 20, dtype=torch.uint8, device=device)
        # QG_CONFIG_I8_PREWIDEN candidates write their fp16 activation copy into
        # the workspace: a separate one keeps it off the Split-K counters
        self.ws_prew = torch.zeros(64 << 20, dtype=torch.uint8, device=device)
        self.stream = torch.cuda.Stream(device=device)

    def time_config(self, fmt, M, N, K, variant, split, cfg, min_bytes=3 * 126e6, reps=5, linear=False):
        """Microseconds per GEMM: median over `reps` replays of a graph of R
        launches, each on its own window of the weight pool."""
        wbytes = N * K
        R = int(min(64, max(2, -(-min_bytes // wbytes))))
        step = (wbytes + 255) // 256 * 256
        if step * R > POOL_BYTES:
            R = max(2, POOL_BYTES // step)
        need = q.qg_workspace_bytes_config(fmt, M, N, K, variant, split, cfg)
        ws = self.ws_prew if cfg & q.QG_CONFIG_I8_PREWIDEN else self.ws
        q.qg_set_launch_flags(q.QG_LAUNCH_PDL)
        try:
            graph = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph, stream=self.stream):
                for r in range(R):
                    W = self.pool[r * step:r * step + wbytes]
                    if not linear:
                        q.qg_gemm_w8a8(fmt, M, N, K, self.Aq, self.sa, W, self.sw, self.Y, N, variant, split, cfg,
                                       ws if need else None, need, None, stream=self.stream)
                        continue
                    # the linear call's two-kernel form (quantization into
                    # Aq / sa, then the GEMM), as bench.py runs it
                    q.qg_linear_w8a8(fmt, M, N, K, self.A, K, W, self.sw, self.Y, N, variant, split, cfg,
                                     ws if need else None, need, self.Aq, self.sa, None, stream=self.stream)
        finally:
            q.qg_set_launch_flags(0)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        times = []
        for _ in range(reps):
            with torch.cuda.stream(self.stream):
                e0.record(self.stream)
                graph.replay()
                e1.record(self.stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1e3 / R)
        del graph
        return statistics.median(times)


def time_layer_chain(bench, fmt, M, layers, cfgs, passes=3, reps=5):
    """Microseconds per pass of one decoder layer's linears, in order, each
    a qg_linear_w8a8 call (quantization kernel + GEMM) with its config from
    `cfgs`, captured as one CUDA graph with programmatic dependent launch:
    `passes` x `windows` passes, each window with its own weights (two
    windows when they fit the pool: a layer's weights are then re-read only
    after the other window's; one window when the layer alone exceeds
    L2 several times)."""
    sizes = [N * K for (K, N) in layers]
    windows = 2 if 2 * sum((sz + 255) // 256 * 256 for sz in sizes) <= POOL_BYTES else 1
    offs, o = [], 0
    for w in range(windows):
        row = []
        for sz in sizes:
            row.append(o)
            o += (sz + 255) // 256 * 256
        offs.append(row)
    if o > POOL_BYTES:
        raise ValueError("layer weights exceed the pool")
    q.qg_set_launch_flags(q.QG_LAUNCH_PDL)
    try:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=bench.stream):
            for _ in range(passes):
                for w in range(windows):
                    for (K, N), off, (v, sp, c) in zip(layers, offs[w], cfgs):
                        need = q.qg_workspace_bytes_config(fmt, M, N, K, v, sp, c)
                        W = bench.pool[off:off + N * K]
                        ws = bench.ws_prew if c & q.QG_CONFIG_I8_PREWIDEN else bench.ws
                        q.qg_linear_w8a8(fmt, M, N, K, bench.A, K, W, bench.sw, bench.Y, N, v, sp, c,
                                         ws if need else None, need, bench.Aq, bench.sa, None,
                                         stream=bench.stream)
    finally:
        q.qg_set_launch_flags(0)
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    times = []
    for _ in range(reps):
        with torch.cuda.stream(bench.stream):
            e0.record(bench.stream)
            graph.replay()
            e1.record(bench.stream)
        e1.synchronize()
        times.append(e0.elapsed_time(e1) * 1e3 / (passes * windows))
    del graph
    return statistics.median(times)


def layer_context_pass(bench, table_in, out_path, fmts, models, ms, sms, log=None):
    """Coordinate descent over one layer's linears in their decoder order:
    for every token count, each linear's candidates are timed inside the
    whole layer chain (the other linears keep their current rows), and the
    best chain time keeps its row.  Writes a complete table."""
    rows = read_table(table_in)
    for fmt in fmts:
        fid = FMT_ID[fmt]
        for model in models:
            layers = list(SHAPES[model].items())
            shapes = [ks for _, ks in layers]
            for M in ms:
                cfgs = []
                for (K, N) in shapes:
                    key = (fid, N, K, M)
                    cfgs.append(rows[key] if key in rows else q.qg_select(fmt, M, N, K))
                base = time_layer_chain(bench, fmt, M, shapes, cfgs)
                best_total = base
                for li, (layer, (K, N)) in enumerate(layers):
                    cands = candidates(fmt, M, N, K, sms)
                    if M <= 8:
                        # the one-kernel form of the linear (quantization inside the
                        # GEMM): every CTA reads whole activation rows, cheap at a few
                        # tokens, and the linear has one kernel boundary instead of two
                        cands += [(v, sp, c | q.QG_CONFIG_FUSED_QUANT) for (v, sp, c) in cands
                                  if v in (q.QG_SWAPAB, q.QG_SWAPAB_SPLITK) and not c & NOT_FUSABLE]
                    for cand in cands:
                        if cand == cfgs[li]:
                            continue
                        trial = list(cfgs)
                        trial[li] = cand
                        us = time_layer_chain(bench, fmt, M, shapes, trial)
                        if log:
                            log.write(json.dumps({"pass": "layer", "fmt": fmt, "model": model, "layer": layer, "M": M,
                                                  "variant": cand[0], "split_k": cand[1], "config_id": cand[2],
                                                  "chain_us": us}) + "\n")
                        if us < 0.995 * best_total:
                            best_total, cfgs = us, trial
                for (K, N), cfg in zip(shapes, cfgs):
                    rows[(fid, N, K, M)] = tuple(cfg)
                print(f"{fmt:12s} {model:10s} M={M:2d}: layer chain {base:7.2f} -> {best_total:7.2f} us  "
                      f"{[tuple(c) for c in cfgs]}", flush=True)
    with open(out_path, "w") as fh:
        fh.write("# fmt\tN\tK\tM\tvariant\tsplit_k\tconfig_id   (written by quantized_gemm_decode_02_b300/tune.py)\n")
        for (f, n, k, m) in sorted(rows):
            v, sp, c = rows[(f, n, k, m)]
            fh.write(f"{f}\t{n}\t{k}\t{m}\t{v}\t{sp}\t{c}\n")


def read_table(path):
    rows = {}
    if os.path.exists(path):
        for line in open(path):
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            f, n, k, m, v, s, c = (int(x) for x in line.split())
            rows[(f, n, k, m)] = (v, s, c)
    return rows


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", required=True)
    ap.add_argument("--formats", default="FP8_Dynamic,W8A8_INT8,Block_FP8")
    ap.add_argument("--models", default="Qwen3-1.7B,Qwen3-8B,Qwen3-32B")
    ap.add_argument("--ms", default=",".join(str(m) for m in TUNED_M))
    ap.add_argument("--log", default=None, help="JSON lines with every candidate's time")
    ap.add_argument("--linear", action="store_true",
                    help="time qg_linear_w8a8 (quantization kernel + GEMM) instead of the GEMM alone")
    ap.add_argument("--prefetch-pass", action="store_true",
                    help="also try the winner with an L2 prefetch distance (config_id upper bits)")
    ap.add_argument("--layer-context", metavar="TABLE_IN",
                    help="re-tune the rows of TABLE_IN inside whole-layer chains (quantization + GEMM of qkv, o, "
                         "gate_up, down in order) and write the complete table to --out")
    args = ap.parse_args(argv)
    device = "cuda:0"
    torch.cuda.set_device(0)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    bench = Bench(device)
    if args.layer_context:
        q.qg_load_table(args.layer_context)
        q.qg_set_allow_default(True)
        log = open(args.log, "a") if args.log else None
        layer_context_pass(bench, args.layer_context, args.out, args.formats.split(","), args.models.split(","),
                           [int(m) for m in args.ms.split(",")], sms, log)
        if log:
            log.close()
        return 0
    done = read_table(args.out)
    os.makedirs(os.path.dirname(os.path.abspath(args.out)), exist_ok=True)
    new_file = not os.path.exists(args.out)
    out = open(args.out, "a")
    if new_file:
        out.write("# fmt\tN\tK\tM\tvariant\tsplit_k\tconfig_id   (written by quantized_gemm_decode_02_b300/tune.py)\n")
    log = open(args.log, "a") if args.log else None
    t0 = time.time()
    for fmt in args.formats.split(","):
        fid = FMT_ID[fmt]
        for model in args.models.split(","):
            for layer, (K, N) in SHAPES[model].items():
                for M in (int(m) for m in args.ms.split(",")):
                    if (fid, N, K, M) in done:
                        continue
                    best = None
                    def timed(v, s, c):
                        us = bench.time_config(fmt, M, N, K, v, s, c, linear=args.linear)
                        if log:
                            log.write(json.dumps({"fmt": fmt, "model": model, "layer": layer, "M": M, "N": N, "K": K,
                                                  "variant": v, "split_k": s, "config_id": c, "us": us}) + "\n")
                        return us

                    for (v, s, c) in candidates(fmt, M, N, K, sms):
                        us = timed(v, s, c)
                        if best is None or us < best[0]:
                            best = (us, v, s, c)
                    # optional second pass: the winner with an L2 prefetch
                    # distance, kept only when it is more than 1% faster
                    us0, v, s, c0 = best
                    for dist in (PREFETCH_DISTANCES if args.prefetch_pass else ()):
                        c = q.config_id(c0, dist)
                        us = timed(v, s, c)
                        if us < 0.99 * us0 and us < best[0]:
                            best = (us, v, s, c)
                    us, v, s, c = best
                    gbs = (N * K + M * K + 2 * M * N) / (us * 1e-6) / 1e9
                    out.write(f"{fid}\t{N}\t{K}\t{M}\t{v}\t{s}\t{c}\t# {model} {layer} {us:.2f} us {gbs:.0f} GB/s\n")
                    out.flush()
                    print(f"{fmt:12s} {model:10s} {layer:8s} M={M:2d}: variant {v} split {s:2d} cfg {c:2d} "
                          f"{us:7.2f} us {gbs:6.0f} GB/s  [{time.time() - t0:.0f} s]", flush=True)
    out.close()
    if log:
        log.close()
    return 0


if __name__ == "__main__":
    sys.exit(main())
