"""Benchmark of the grouped (mixture-of-experts) quantized GEMM on B300.

Workload: the expert layers of a Qwen3-30B-A3B-shaped MoE block (128 experts,
8 routed per token; hidden 2048, expert intermediate 768): for each decode
token count M in {1,2,4,8,16,24,32}, the M*8 routed (token, expert) rows,
sorted by expert, go through
    activation quantization (qg_quant_act) -> grouped gate_up GEMM (N = 1536, K = 2048)
    activation quantization                -> grouped down GEMM    (N = 2048, K = 768)
with qg_gemm_w8a8_grouped, every expert's weights distinct, the whole step
captured in one CUDA graph with programmatic dependent launch.  Routing is
drawn from a seeded generator (each token picks 8 distinct experts
uniformly); activations and weights are seeded synthetic data (the page's
MoE item names no model or dataset).

Metric: HBM GB/s = algorithmic bytes per step / step time, where a grouped
GEMM must move the weights of the experts that received tokens (the others
are never read), the routed activations, scales and outputs once.

Usage:  python -m quantized_gemm_decode_02_b300.bench_moe [--fmt FP8_Dynamic] [--steps K] [--warmup W]
Prints one JSON line.
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from quantized_gemm_decode_02_b300 import qgemm as q  # noqa: E402

EXPERTS, TOPK, HIDDEN, INTER = 128, 8, 2048, 768
LAYERS = (("gate_up", 2 * INTER, HIDDEN), ("down", HIDDEN, INTER))  # (name, N, K)
TUNED_M = (1, 2, 4, 8, 16, 24, 32)


def routing(M: int, rng) -> np.ndarray:
    """Token offsets [EXPERTS + 1] of the M*TOPK routed rows sorted by expert."""
    picks = np.stack([rng.choice(EXPERTS, size=TOPK, replace=False) for _ in range(M)]).reshape(-1)
    counts = np.bincount(picks, minlength=EXPERTS)
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("--fmt", default="FP8_Dynamic", choices=sorted(q.FORMATS))
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every step's kernels directly instead of replaying the captured graph (profilers)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if not torch.cuda.is_available():
        raise SystemExit("bench_moe needs a CUDA device")
    import bench  # the repository's benchmark: clock sampling and the measured peaks
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    fmt = args.fmt
    rng = np.random.Generator(np.random.PCG64(0))
    gen = torch.Generator(device=dev)
    gen.manual_seed(0)
    q.qg_set_allow_default(True)
    if os.path.exists(bench.TABLE):
        q.qg_load_table(bench.TABLE)

    # expert weights: random N(0, 0.02) per expert, quantized on the device
    weights = {}
    for name, N, K in LAYERS:
        Wq = torch.empty((EXPERTS, N, K), dtype=torch.uint8, device=dev)
        sw_shape = (EXPERTS, (N + 127) // 128, K // 128) if fmt == "Block_FP8" else (EXPERTS, N)
        sw = torch.empty(sw_shape, dtype=torch.float32, device=dev)
        for e in range(EXPERTS):
            W = torch.randn((N, K), device=dev, generator=gen) * 0.02
            q.qg_quant_weight(fmt, W, N, K, Wq[e], sw[e])
        weights[name] = (Wq, sw)
    torch.cuda.synchronize()

    items, bytes_step, weight_bytes = [], 0, 0
    for M in TUNED_M:
        offs = routing(M, rng)
        rows = int(offs[-1])
        active = int(np.count_nonzero(np.diff(offs)))
        max_tokens = int(np.diff(offs).max())
        offs_d = torch.from_numpy(offs).to(dev)
        for name, N, K in LAYERS:
            A = torch.randn((rows, K), device=dev, generator=gen).to(torch.bfloat16)
            Aq = torch.empty((rows, K), dtype=torch.uint8, device=dev)
            sa = torch.empty((rows, K // 128) if fmt == "Block_FP8" else (rows,), dtype=torch.float32, device=dev)
            Y = torch.empty((rows, N), dtype=torch.bfloat16, device=dev)
            # every expert with tokens brings its own weight tiles, so the
            # grid is already ~active x N/128 tiles: no Split-K; INT8 groups
            # of at most 4 tokens on the CUDA cores
            v, s, c = (q.QG_SWAPAB_DP4A if fmt == "W8A8_INT8" and max_tokens <= 4 else q.QG_SWAPAB), 1, 0
            need = q.qg_workspace_bytes_grouped(fmt, EXPERTS, rows, max_tokens, N, K, v, s)
            ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
            scale_bytes = (4 * ((N + 127) // 128) * (K // 128) if fmt == "Block_FP8" else 4 * N) * active
            act_scales = 4 * rows * (K // 128 if fmt == "Block_FP8" else 1)
            gemm_bytes = active * N * K + rows * K + 2 * rows * N + scale_bytes + act_scales
            quant_bytes = 2 * rows * K + rows * K + act_scales
            bytes_step += gemm_bytes + quant_bytes
            weight_bytes += active * N * K
            items.append(dict(M=M, layer=name, N=N, K=K, rows=rows, active=active, max_tokens=max_tokens,
                              offs=offs_d, A=A, Aq=Aq, sa=sa, Y=Y, v=v, s=s, c=c, ws=ws, need=need))

    stream = torch.cuda.Stream(device=dev)

    def enqueue():
        for it in items:
            Wq, sw = weights[it["layer"]]
            q.qg_quant_act(fmt, it["A"], it["rows"], it["K"], it["K"], it["Aq"], it["sa"], stream=stream)
            q.qg_gemm_w8a8_grouped(fmt, EXPERTS, it["offs"], it["rows"], it["max_tokens"], it["N"], it["K"],
                                   it["Aq"], it["sa"], Wq, sw, it["Y"], it["N"], it["v"], it["s"], it["c"],
                                   it["ws"], it["need"], None, stream=stream)

    if args.no_graph:
        class _Direct:
            """Stand-in for the step graph: enqueue the step's kernels."""
            def replay(self):
                with torch.cuda.stream(stream):
                    q.qg_set_launch_flags(q.QG_LAUNCH_PDL)
                    enqueue()
                    q.qg_set_launch_flags(0)
        graph = _Direct()
    else:
        q.qg_set_launch_flags(q.QG_LAUNCH_PDL)
        graph = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(graph, stream=stream):
                enqueue()
        finally:
            q.qg_set_launch_flags(0)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    clocks = bench.ClockSampler(0)
    clocks.start()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            graph.replay()
        e1.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    assert q.qg_device_error() == 0
    ms = e0.elapsed_time(e1) / args.steps
    hbm_peak, _, peak_kind = bench.load_peaks()
    value = bytes_step / (ms * 1e-3) / 1e9
    line = {
        "metric": "HBM GB/s (% of B300 peak) of grouped (MoE) quantized GEMMs at decode token counts",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 6), "higher_is_better": True, "dtype": {"FP8_Dynamic": "e4m3", "Block_FP8": "e4m3",
                                                                          "W8A8_INT8": "int8"}[fmt],
        "data": "synthetic", "pct_of_peak": round(100 * value / hbm_peak, 1), "peak_gbs": hbm_peak,
        "peak_kind": peak_kind, "clocks": clk,
        "config": {"workload": f"moe_qwen3_30b_a3b_{fmt}", "experts": EXPERTS, "top_k": TOPK, "hidden": HIDDEN,
                   "expert_intermediate": INTER, "M": list(TUNED_M), "grouped_gemms_per_step": len(items),
                   "kernels_per_step": 2 * len(items), "bytes_per_step": bytes_step,
                   "weight_bytes_streamed_per_step": weight_bytes,
                   "graph": ("direct launches" if args.no_graph else "one CUDA graph per step")
                            + ", programmatic dependent launch"},
        "per_gemm": [{"M": it["M"], "layer": it["layer"], "routed_rows": it["rows"], "experts_with_tokens": it["active"],
                      "max_tokens": it["max_tokens"], "variant": it["v"], "split_k": it["s"]} for it in items],
    }
    print(json.dumps(line))
    return 0


if __name__ == "__main__":
    sys.exit(main())
