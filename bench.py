"""Benchmark of the quantized decode GEMM hot path on B300.

Workload (default, `layer_qwen3_8b`): all three formats (FP8_Dynamic,
W8A8_INT8, Block_FP8) on one Qwen3-8B layer's four linears (qkv K=4096
N=6144, o K=4096 N=4096, gate_up K=4096 N=24576, down K=12288 N=4096) at
every decode token count M = 1..32, activations A ~ N(0,1) with 1% outliers
x20.  One step is one pass of the whole hot path over that batch: for each
(format, M, layer) one qg_linear_w8a8 call, i.e. a dynamic activation
quantization kernel (per token, or per 1x128 group for Block_FP8) and the
quantized GEMM kernel with the variant the tuned table selects (qg_select);
384 + 384 kernels captured once into one CUDA graph with programmatic
dependent launch and replayed.  Weights: one copy per (format, layer) and
token-count parity, so two uses of a copy are separated by the other
linears' 193 MB of weights (> 126 MB L2): no GEMM finds its weights in L2.

Other workloads (--workload): W8A8_INT8 over the Qwen3-1.7B linears at
M in {1,2,4,8,16,24,32}; Block_FP8 over the Qwen3-8B linears at M=1..32;
FP8_Dynamic over the Qwen3-32B linears; FP8_Dynamic at M=1 on the Qwen3-1.7B
o_proj shape; FP8_Dynamic / W8A8_INT8 over the Qwen3-8B linears;
`large_m_qwen3_8b`, the layer at M = 64..512 (compute-bound: TFLOP/s
against the tensor peak of each format's MMA kind).

Metric: HBM GB/s = algorithmic bytes per step / step time (the kernels must
move the weights, activations, scales and outputs once), plus us per GEMM;
TFLOP/s = 2*M*N*K per step / step time for the compute-bound workload.

Also reported: the roofline of the GEMM kernels from an in-chain timeline
(the same graph, programmatic dependent launch kept, every kernel stamping
its first CTA start and last CTA end with %globaltimer through the library's
timing log: a kernel's time is from its predecessor's end to its own end, so
the kernels' times add up to the step), an end-to-end figure through the C
ABI with the activations copied from pinned host memory and the outputs
copied back inside the timed region (two buffer sets, so one step's copies
overlap its neighbours' kernels), SM clocks sampled during the timed region,
and the CPU oracle timed on the host cores on a bounded sample
(cpu_baseline).  `--impl reference` times that oracle alone as the
reference arm.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import seeded_inputs as si  # noqa: E402

TABLE = os.path.join(ROOT, "quantized_gemm_decode_02_b300", "tables", "b300.tsv")
PEAKS = os.path.join(ROOT, "MEASURED_PEAKS.json")

LAYERS = ("qkv", "o", "gate_up", "down")
FORMATS = ("FP8_Dynamic", "W8A8_INT8", "Block_FP8")


def _items(fmts, model, layers, ms):
    """(format, model, layer, M) in launch order: format, then token count,
    then the layer's linears in forward order."""
    return [(f, model, layer, M) for f in fmts for M in ms for layer in layers]


# name: items, whether items share weights (one copy per (format, layer) and
# token-count parity), roofline bound; activations with 1% outliers x20 for
# every format (`outliers`), else for Block_FP8 only
WORKLOADS = {
    "int8_qwen3_1.7b": dict(items=_items(["W8A8_INT8"], "Qwen3-1.7B", LAYERS, si.TUNED_M), shared=False, bound="hbm"),
    "fp8_qwen3_1.7b_o_m1": dict(items=_items(["FP8_Dynamic"], "Qwen3-1.7B", ("o",), (1,)), shared=False, bound="hbm"),
    # the same linear 64 times in one graph (distinct weights, 268 MB): its cost
    # inside a chain, without one graph launch per linear
    "fp8_qwen3_1.7b_o_m1_chain64": dict(items=_items(["FP8_Dynamic"], "Qwen3-1.7B", ("o",), (1,)) * 64, shared=False,
                                        bound="hbm"),
    "blockfp8_qwen3_8b": dict(items=_items(["Block_FP8"], "Qwen3-8B", LAYERS, range(1, 33)), shared=False,
                              bound="hbm"),
    "fp8_qwen3_32b": dict(items=_items(["FP8_Dynamic"], "Qwen3-32B", LAYERS, si.TUNED_M), shared=False, bound="hbm"),
    "fp8_qwen3_8b": dict(items=_items(["FP8_Dynamic"], "Qwen3-8B", LAYERS, si.TUNED_M), shared=False, bound="hbm"),
    "int8_qwen3_8b": dict(items=_items(["W8A8_INT8"], "Qwen3-8B", LAYERS, si.TUNED_M), shared=False, bound="hbm"),
    # all three formats on one Qwen3-8B layer's four linears, chained in one
    # graph, at every token count 1..32
    "layer_qwen3_8b": dict(items=_items(FORMATS, "Qwen3-8B", LAYERS, range(1, 33)), shared=True, bound="hbm",
                           outliers=True),
    # the compute-bound regime beyond the decode range
    "large_m_qwen3_8b": dict(items=_items(FORMATS, "Qwen3-8B", LAYERS, (64, 128, 256, 384, 512)), shared=True,
                             bound="tensor", outliers=True),
}
DEFAULT_WORKLOAD = "layer_qwen3_8b"
METRIC_HBM = "HBM GB/s (% of B300 peak) and us/GEMM at M=1..32 on Qwen3 linear shapes"
METRIC_TENSOR = "TFLOP/s (% of B300 tensor peak) at M=64..512 on Qwen3 linear shapes"


def gemm_bytes(fmt: str, M: int, N: int, K: int) -> int:
    """Algorithmic bytes of one quantized GEMM: weights, quantized
    activations, bf16 output and the scales, each moved once."""
    if fmt == "Block_FP8":
        return N * K + M * K + 2 * M * N + 4 * ((N + 127) // 128) * (K // 128) + 4 * M * (K // 128)
    return N * K + M * K + 2 * M * N + 4 * N + 4 * M


def quant_bytes(fmt: str, M: int, K: int) -> int:
    """Algorithmic bytes of one activation quantization: bf16 in, codes and scales out."""
    scales = M * (K // 128) if fmt == "Block_FP8" else M
    return 2 * M * K + M * K + 4 * scales


def workload_dtype(items) -> str:
    fmts = sorted({f for f, _, _, _ in items})
    names = {"FP8_Dynamic": "e4m3", "Block_FP8": "e4m3", "W8A8_INT8": "int8"}
    return "+".join(sorted({names[f] for f in fmts}))


# ------------------------------------------------------------------ workload

class Workload:
    """Device buffers and the captured graphs for one workload."""

    def __init__(self, name: str, device: str, seed: int = 0, pdl: bool = True, fused: bool = False,
                 table: str = TABLE, items=None):
        """`items`: (format, model, layer, M) list replacing the workload's
        own (a slice of it, for tests), with the workload's other settings."""
        from quantized_gemm_decode_02_b300 import qgemm as q
        self.q = q
        self.name = name
        self.fused = fused
        spec = WORKLOADS[name]
        spec_items = spec["items"] if items is None else list(items)
        self.bound = spec["bound"]
        self.device = device
        self.pdl = pdl
        self.items = []  # (fmt, M, layer, N, K)
        for fmt, model, layer, M in spec_items:
            K, N = si.QWEN3_LINEARS[model][layer]
            self.items.append((fmt, M, layer, N, K))
        self.formats = sorted({it[0] for it in self.items})
        self.models = sorted({m for _, m, _, _ in spec_items})
        self.layers = list(dict.fromkeys(layer for _, _, layer, _ in spec_items))
        self.ms = list(dict.fromkeys(M for _, _, _, M in spec_items))
        if os.path.exists(table):
            q.qg_load_table(table)
        q.qg_set_allow_default(True)
        # one contiguous activation buffer (bf16) and one output buffer (bf16),
        # sliced per item at 256-byte boundaries, so e2e copies are single copies
        def align(n):
            return (n + 255) // 256 * 256
        a_off, y_off, a_tot, y_tot = [], [], 0, 0
        for (_, M, _, N, K) in self.items:
            a_off.append(a_tot); a_tot += align(M * K * 2)
            y_off.append(y_tot); y_tot += align(M * N * 2)
        self.A_all = torch.empty(a_tot, dtype=torch.uint8, device=device)
        self.Y_all = torch.empty(y_tot, dtype=torch.uint8, device=device)
        self.a_off, self.y_off = a_off, y_off
        self.recs = []
        ws_need = 0
        ws_prew = 0  # QG_CONFIG_I8_PREWIDEN items: a workspace of their own (their fp16 copy must not land on
                     # the Split-K arrival counters of other items)
        weights = {}
        wseeds = {}  # weight copy -> seed of its fp32 weights (si.weights_device)
        for i, (fmt, M, layer, N, K) in enumerate(self.items):
            variant, split, cfg = q.qg_select(fmt, M, N, K)
            need = q.qg_workspace_bytes_config(fmt, M, N, K, variant, split, cfg)
            if cfg & q.QG_CONFIG_I8_PREWIDEN:
                ws_prew = max(ws_prew, need)
            else:
                ws_need = max(ws_need, need)
            A = self.A_all[a_off[i]:a_off[i] + M * K * 2].view(torch.bfloat16).view(M, K)
            A.copy_(si.activations_device(M, K, seed=seed * 1000 + i, device=device,
                                          outliers=spec.get("outliers", False) or fmt == "Block_FP8"))
            # distinct weights per item, or (shared workloads) one copy per
            # (format, layer) and token-count parity: consecutive uses of a
            # copy are separated by the other linears' weights (> L2)
            wkey = (fmt, layer, self.ms.index(M) % 2) if spec["shared"] else i
            if wkey not in weights:
                wseeds[wkey] = seed * 1000 + len(weights)
                W = si.weights_device(N, K, seed=wseeds[wkey], device=device)
                Wq = torch.empty((N, K), dtype=torch.uint8, device=device)
                if fmt == "Block_FP8":
                    sw = torch.empty(((N + 127) // 128, K // 128), dtype=torch.float32, device=device)
                else:
                    sw = torch.empty((N,), dtype=torch.float32, device=device)
                q.qg_quant_weight(fmt, W, N, K, Wq, sw)
                del W
                weights[wkey] = (Wq, sw)
            Wq, sw = weights[wkey]
            sa = torch.empty((M, K // 128) if fmt == "Block_FP8" else (M,), dtype=torch.float32, device=device)
            Aq = torch.empty((M, K), dtype=torch.uint8, device=device)
            Y = self.Y_all[y_off[i]:y_off[i] + M * N * 2].view(torch.bfloat16).view(M, N)
            self.recs.append(dict(fmt=fmt, M=M, layer=layer, N=N, K=K, A=A, Aq=Aq, sa=sa, Wq=Wq, sw=sw, Y=Y,
                                  variant=variant, split=split, cfg=cfg, ws_need=need, wseed=wseeds[wkey]))
        self.ws = torch.zeros(max(ws_need, 256), dtype=torch.uint8, device=device)
        self.ws_bytes = ws_need
        self.ws_prew = torch.zeros(max(ws_prew, 256), dtype=torch.uint8, device=device)
        self.ws_prew_bytes = ws_prew
        torch.cuda.synchronize()
        self.bytes_gemm = sum(gemm_bytes(r["fmt"], r["M"], r["N"], r["K"]) for r in self.recs)
        self.bytes_quant = sum(quant_bytes(r["fmt"], r["M"], r["K"]) for r in self.recs)
        self.bytes_step = self.bytes_gemm + self.bytes_quant
        self.flops_step = sum(2 * r["M"] * r["N"] * r["K"] for r in self.recs)
        self.weight_bytes = sum({id(r["Wq"]): r["N"] * r["K"] for r in self.recs}.values())
        self.weight_bytes_streamed = sum(r["N"] * r["K"] for r in self.recs)

    def fused_item(self, i: int) -> bool:
        """Whether item i runs as one kernel (activation quantization inside
        the GEMM): the Swap-AB variants on the tcgen05 kernels when the
        table row asks for it (QG_CONFIG_FUSED_QUANT) or with --fused."""
        r = self.recs[i]
        fusable = r["variant"] in (self.q.QG_SWAPAB, self.q.QG_SWAPAB_SPLITK) and not r["cfg"] & self.q.QG_CONFIG_MMA_SYNC
        return fusable and (self.fused or bool(r["cfg"] & self.q.QG_CONFIG_FUSED_QUANT))

    def kernels(self, i: int) -> int:
        if self.fused_item(i):
            return 1
        # QG_CONFIG_I8_PREWIDEN: quantization, activation widening, GEMM
        return 3 if self.recs[i]["cfg"] & self.q.QG_CONFIG_I8_PREWIDEN else 2

    def rebind(self, A_all, Y_all):
        """The items with their activations and outputs in other buffers of
        the same layout (a second buffer set for pipelined e2e steps)."""
        out = []
        for i, r in enumerate(self.recs):
            M, N, K = r["M"], r["N"], r["K"]
            A = A_all[self.a_off[i]:self.a_off[i] + M * K * 2].view(torch.bfloat16).view(M, K)
            Y = Y_all[self.y_off[i]:self.y_off[i] + M * N * 2].view(torch.bfloat16).view(M, N)
            out.append(dict(r, A=A, Y=Y))
        return out

    def enqueue(self, stream, i: int, recs=None):
        """One linear layer through qg_linear_w8a8: activation quantization +
        GEMM (two kernels; one fused kernel with --fused where the format and
        variant have one)."""
        r = (recs or self.recs)[i]
        q = self.q
        fz = self.fused and self.fused_item(i)
        prew = bool(r["cfg"] & q.QG_CONFIG_I8_PREWIDEN)
        q.qg_linear_w8a8(r["fmt"], r["M"], r["N"], r["K"], r["A"], r["K"], r["Wq"], r["sw"], r["Y"], r["N"],
                         r["variant"], r["split"], r["cfg"], self.ws_prew if prew else self.ws,
                         self.ws_prew_bytes if prew else self.ws_bytes,
                         None if fz else r["Aq"], None if fz else r["sa"], None, stream=stream)

    def capture_step(self, stream, recs=None, timing_log=None) -> torch.cuda.CUDAGraph:
        """The whole step (quant + GEMM for every item) as one graph; with a
        timing log every kernel of the step stamps its slot pair (launch
        order: each item's quantization kernel, then its GEMM)."""
        q = self.q
        q.qg_set_launch_flags(q.QG_LAUNCH_PDL if self.pdl else 0)
        if timing_log is not None:
            q.qg_set_timing_log(timing_log, timing_log.numel() // 2)
        g = torch.cuda.CUDAGraph()
        try:
            with torch.cuda.graph(g, stream=stream):
                for i in range(len(self.recs)):
                    self.enqueue(stream, i, recs)
            if timing_log is not None and q.qg_timing_log_count() != timing_log.numel() // 2:
                raise RuntimeError(f"timing log: {q.qg_timing_log_count()} launches, expected "
                                   f"{timing_log.numel() // 2}")
        finally:
            q.qg_set_launch_flags(0)
            if timing_log is not None:
                q.qg_set_timing_log(None, 0)
        return g

    def kernel_roles(self):
        """(item index, 'quant' | 'gemm' | 'fused') of every kernel of a step, in launch order."""
        out = []
        for i in range(len(self.recs)):
            if self.fused_item(i):
                out.append((i, "fused"))
            else:
                out += [(i, "quant"), (i, "gemm")]
        return out


def timeline(wl, stream, reps: int, direct: bool = False):
    """Per-kernel times inside the step graph, programmatic dependent launch
    kept.  Every kernel stamps its earliest CTA start and latest CTA end
    (%globaltimer) into its slot pair; a kernel's time is from the latest
    end of the kernels before it to its own end (the first kernel: from its
    own start), so the times of a step's kernels add up to the step's span.
    Returns (mean time per kernel in us, mean step span in us)."""
    roles = wl.kernel_roles()
    n = len(roles)
    log = torch.zeros(2 * n, dtype=torch.int64, device=wl.device)
    q = wl.q

    class _Direct:
        """The step's kernels launched directly, each with its slot pair."""
        def replay(self):
            q.qg_set_launch_flags(q.QG_LAUNCH_PDL if wl.pdl else 0)
            q.qg_set_timing_log(log, n)
            try:
                for i in range(len(wl.recs)):
                    wl.enqueue(stream, i)
            finally:
                q.qg_set_launch_flags(0)
                q.qg_set_timing_log(None, 0)

    g = _Direct() if direct else wl.capture_step(stream, timing_log=log)
    start_fill = torch.full((n,), -1, dtype=torch.int64, device=wl.device)  # UINT64_MAX for atomicMin
    acc = np.zeros(n)
    span = 0.0
    for r in range(reps + 3):
        with torch.cuda.stream(stream):
            log.view(n, 2)[:, 0].copy_(start_fill)
            log.view(n, 2)[:, 1].zero_()
            g.replay()
        torch.cuda.synchronize()
        if r < 3:
            continue
        t = log.view(n, 2).cpu().numpy().view(np.uint64).astype(np.float64)
        starts, ends = t[:, 0], t[:, 1]
        prev = np.maximum.accumulate(np.concatenate([[starts[0]], ends[:-1]]))
        acc += np.maximum(ends - prev, 0.0)
        span += ends.max() - starts[0]
    return acc / reps / 1e3, span / reps / 1e3


# ------------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"qg_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        self.t0 = time.time()

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2])); smax.append(float(parts[3]))
                power.append(float(parts[4]))
            except ValueError:
                continue
            for nm, v in zip(names, parts[6:10]):
                if v.lower() in ("active", "1"):
                    reasons.add(nm)
        os.unlink(self.path)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm), "power_w_max": max(power) if power else None}


# --------------------------------------------------------------- cpu oracle

def _oracle_items(name):
    """(format, M, N, K) of every item of the workload."""
    out = []
    for fmt, model, layer, M in WORKLOADS[name]["items"]:
        K, N = si.QWEN3_LINEARS[model][layer]
        out.append((fmt, M, N, K))
    return out


def _oracle_pass(orc, name, cols, cache, cores, items=None):
    """quant_act + GEMM in the oracle for the workload's items (or the listed
    item indices), all token rows, the first `cols` output columns.  The
    quantized weights and the activations are prepared once and cached
    (set-up, not timed).  Returns (seconds, bytes, flops)."""
    t_total, processed, flops = 0.0, 0, 0
    all_items = _oracle_items(name)
    for idx in (range(len(all_items)) if items is None else items):
        fmt, M, N, K = all_items[idx]
        nc = min(cols, N)
        wkey = (fmt, N, K, nc)
        if wkey not in cache:
            cache[wkey] = orc.quant_weight(fmt, si.weights(nc, K, seed=idx))
        Wq, sw = cache[wkey]
        akey = ("A", idx)
        if akey not in cache:
            cache[akey] = si.bf16_to_f32_numpy(si.activations(M, K, seed=idx))
        A = cache[akey]
        t0 = time.perf_counter()
        Aq, sa = orc.quant_act(fmt, A)
        orc.gemm(fmt, Aq, sa, Wq, sw, threads=cores)
        t_total += time.perf_counter() - t0
        processed += gemm_bytes(fmt, M, nc, K) + quant_bytes(fmt, M, K)
        flops += 2 * M * nc * K
    return t_total, processed, flops


def _rate(bound, b, f, t):
    return (b / t / 1e9, "GB/s") if bound == "hbm" else (f / t / 1e12, "TFLOP/s")


def cpu_oracle_leg(name: str, budget_s: float = 12.0) -> dict:
    """Time the CPU oracle on a bounded sample of the workload: every item,
    all token rows, the first `cols` output columns of each layer (doubling
    `cols` up to the full width while a pass stays short), then repeated
    passes until `budget_s` seconds of oracle work are timed.  The rate
    counts the algorithmic bytes (or flops) of the sampled part with the
    same accounting as the GPU path."""
    from oracle import oracle as orc
    orc.build()
    cores = os.cpu_count() or 1
    n_max = max(n for _, _, n, _ in _oracle_items(name))
    cols, cache = 16, {}
    while True:
        t, b, f = _oracle_pass(orc, name, cols, cache, cores)
        if t >= budget_s / 4 or cols >= n_max:
            break
        cols = min(cols * 2, n_max)
    passes = 1
    while t < budget_s and passes < 64:
        t1, b1, f1 = _oracle_pass(orc, name, cols, cache, cores)
        t, b, f, passes = t + t1, b + b1, f + f1, passes + 1
    v, unit = _rate(WORKLOADS[name]["bound"], b, f, t)
    return {"value": v, "unit": unit, "cores": cores, "kind": "oracle",
            "sample": f"{name}: all {len(_oracle_items(name))} (format, M, layer) items, all token rows, the first "
                      f"{cols} output columns per layer, {passes} passes; quant_act + GEMM in the C oracle on "
                      f"{cores} threads ({t:.1f} s timed)"}


# --------------------------------------------------------------------- main

def load_peaks():
    """(HBM GB/s, bf16 dense TFLOP/s burst, kind): the measured copy and GEMM
    peaks of this machine, else the fallback figures."""
    try:
        with open(PEAKS) as fh:
            p = json.load(fh)
        return p.get("hbm_gbs", 6400.0), p.get("bf16_tflops", 1800.0), "measured"
    except (OSError, ValueError):
        return 6400.0, 1800.0, "fallback"


TRAFFIC = os.path.join(ROOT, "profiles", "gemm_traffic.json")


def kernel_sources_sha() -> str:
    """SHA-256 over the library's kernel sources (csrc/*.cuh, sorted by name;
    the host-side ABI file is not part of it)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_gemm_decode_02_b300", "csrc")
    for name in sorted(n for n in os.listdir(csrc) if n.endswith(".cuh")):
        with open(os.path.join(csrc, name), "rb") as fh:
            h.update(name.encode() + b"\0" + fh.read())
    return h.hexdigest()


def measured_traffic(workload: str, fused: bool):
    """DRAM bytes (read + write) per GEMM launch from the committed ncu
    capture of this workload, or None when there is none or the kernel
    sources changed since it was taken."""
    try:
        with open(TRAFFIC) as fh:
            rec = json.load(fh).get(workload)
    except (OSError, ValueError):
        return None, "no committed capture"
    if not rec or fused:
        return None, "no committed capture for this workload and path"
    if rec.get("kernel_sources_sha256") != kernel_sources_sha():
        return None, "kernel sources changed since the capture"
    return rec["dram_bytes_per_launch"], rec["capture"]


def tensor_peak(fmt: str, bf16_tflops: float) -> float:
    """Dense tensor peak of the MMA kind a format runs on: E4M3 runs
    kind::f8f6f4 (nominally twice the bf16 rate), W8A8_INT8 runs kind::f16 on
    widened operands (the bf16 rate)."""
    return bf16_tflops * (2.0 if fmt in ("FP8_Dynamic", "Block_FP8") else 1.0)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, v: float, device) -> float:
    if world <= 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _config(name, wl_items):
    """The workload's description: formats, linear shapes (K, N) and token counts."""
    fmts = sorted({f for f, _, _, _ in wl_items})
    shapes = {}
    for _, model, layer, _ in wl_items:
        shapes.setdefault(f"{model} {layer}", list(si.QWEN3_LINEARS[model][layer]))
    return {"workload": name, "formats": fmts, "shapes_k_n": shapes,
            "layers": list(dict.fromkeys(layer for _, _, layer, _ in wl_items)),
            "M": list(dict.fromkeys(M for _, _, _, M in wl_items))}


REFERENCE_BUDGET_S = 120.0  # wall time of a whole --impl reference run, warm-up included


def reference_plan(n_items: int, t_item: float, t_pass16: float, runs: int, budget_s: float = REFERENCE_BUDGET_S):
    """Per-step sample of the reference arm so that `runs` steps (warm-up
    included) take about `budget_s` seconds: (columns, items per step).  The
    whole workload per step at the widest column count whose pass fits the
    per-step share; when even 16 columns over every item do not fit, a
    rotating subset of the items, at least one per step."""
    per_step = budget_s / max(1, runs)
    if t_pass16 <= per_step:
        cols = 16
        while cols < 8192 and t_pass16 * (cols * 2) / 16 <= per_step:
            cols *= 2
        return cols, n_items
    return 16, max(1, min(n_items, int(per_step / max(t_item, 1e-9))))


def run_reference(args, world, rank):
    """The reference arm: the CPU oracle as it stands, each step a bounded
    sample of the workload sized so the whole run stays within ~2 minutes."""
    if rank != 0:
        return 0
    from oracle import oracle as orc
    orc.build()
    name = args.workload
    spec = WORKLOADS[name]
    cores = os.cpu_count() or 1
    cache = {}
    n_items = len(_oracle_items(name))
    _oracle_pass(orc, name, 16, cache, cores)                      # inputs prepared, not timed
    w0 = time.perf_counter()
    _oracle_pass(orc, name, 16, cache, cores)                      # calibration (wall time)
    t_pass16 = time.perf_counter() - w0
    cols, per_step = reference_plan(n_items, t_pass16 / n_items, t_pass16, args.steps + args.warmup,
                                    budget_s=args.reference_budget_s)
    nxt = 0

    def step():
        nonlocal nxt
        idx = [(nxt + i) % n_items for i in range(per_step)]
        nxt = (nxt + per_step) % n_items
        return _oracle_pass(orc, name, cols, cache, cores, items=idx)

    for _ in range(args.warmup):
        step()
    t_sum, b_sum, f_sum = 0.0, 0, 0
    for _ in range(args.steps):
        t, b, f = step()
        t_sum += t
        b_sum += b
        f_sum += f
    value, unit = _rate(spec["bound"], b_sum, f_sum, t_sum)
    which = (f"all {n_items} (format, M, layer) items" if per_step == n_items else
             f"{per_step} of the {n_items} (format, M, layer) items in turn")
    sample = (f"{name}: {which}, all token rows, the first {cols} output columns per layer, per step; "
              f"quant_act + GEMM in the C oracle on {cores} threads")
    line = {"metric": METRIC_HBM if spec["bound"] == "hbm" else METRIC_TENSOR,
            "value": value, "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": t_sum / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": workload_dtype(spec["items"]), "data": "synthetic",
            "config": _config(name, spec["items"]),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=100)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--reference-budget-s", type=float, default=REFERENCE_BUDGET_S,
                    help="wall time of a whole --impl reference run, warm-up included")
    ap.add_argument("--workload", choices=sorted(WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--table", default=TABLE, help="tuned config table to load (default: the shipped B300 table)")
    ap.add_argument("--fused", action="store_true",
                    help="quantize activations inside the GEMM kernel (qg_linear_w8a8's one-kernel form) instead "
                         "of in their own kernel; measured slower on B300, so not the default")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=200)
    ap.add_argument("--launches-only", action="store_true",
                    help="run the warm-up and timed steps only and print a short line (for a kernel profiler's "
                         "launch list); no timeline, e2e or CPU legs")
    ap.add_argument("--no-graph", action="store_true",
                    help="launch every step's kernels directly instead of replaying the captured graph "
                         "(for profilers that cannot follow graph nodes; not used for reported numbers)")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the compute path is the sm_103a library)")
    device = f"cuda:{local}"
    torch.cuda.set_device(local)
    wl = Workload(args.workload, device, seed=rank, pdl=not args.no_pdl, fused=args.fused, table=args.table)
    stream = torch.cuda.Stream(device=device)
    graph = wl.capture_step(stream)
    torch.cuda.synchronize()

    if args.no_graph:
        class _Direct:
            """Stand-in for the step graph: enqueue the step's kernels."""
            def replay(self_inner):
                with torch.cuda.stream(stream):
                    wl.q.qg_set_launch_flags(wl.q.QG_LAUNCH_PDL if wl.pdl else 0)
                    for i in range(len(wl.recs)):
                        wl.enqueue(stream, i)
                    wl.q.qg_set_launch_flags(0)
        graph = _Direct()

    # ---- timed region: K graph replays (one step each)
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    barrier(world)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.25)  # let the sampler's first reading land
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        t_start.record(stream)
        for _ in range(args.steps):
            graph.replay()
        t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms_step = t_start.elapsed_time(t_end) / args.steps
    ms_step = max_over_ranks(world, ms_step, device)
    hbm = wl.bound == "hbm"

    def rate(b, f, ms):
        return b / (ms * 1e-3) / 1e9 if hbm else f / (ms * 1e-3) / 1e12

    value = world * rate(wl.bytes_step, wl.flops_step, ms_step)
    assert wl.q.qg_device_error() == 0
    n_gemm = len(wl.recs)
    n_kernels = sum(wl.kernels(i) for i in range(n_gemm))
    if args.launches_only:
        # for a kernel profiler's launch list: the timed steps only
        if rank == 0:
            print(json.dumps({"workload": args.workload, "steps": args.steps, "warmup": args.warmup,
                              "ms_per_step": round(ms_step, 6), "kernels_per_step": n_kernels,
                              "launches_only": True}), flush=True)
        return 0

    # ---- in-chain timeline: each kernel's time inside the step (stamps)
    reps = max(10, min(100, args.steps))
    per_kernel_us, span_us = timeline(wl, stream, reps, direct=args.no_graph)
    assert wl.q.qg_device_error() == 0
    roles = wl.kernel_roles()
    gemm_us = np.zeros(n_gemm)   # the GEMM kernel's time (fused: quantize + GEMM)
    quant_us = np.zeros(n_gemm)  # the activation quantization kernel's time
    for (i, role), t in zip(roles, per_kernel_us):
        if role == "quant":
            quant_us[i] += t
        else:
            gemm_us[i] += t
    hbm_peak, bf16_peak, peak_kind = load_peaks()
    timing_note = ("in-chain timeline of the step graph (programmatic dependent launch kept): every kernel stamps "
                   "its first CTA start and last CTA end with %globaltimer; a kernel's time runs from the latest "
                   "end of the kernels before it to its own end, so the kernels' times add up to the step span")
    chain = {"step_span_us": round(span_us, 3), "ms_per_step_us": round(ms_step * 1e3, 3),
             "gemm_us_per_step": round(float(gemm_us.sum()), 3),
             "quant_us_per_step": round(float(quant_us.sum()), 3)}
    # roofline of the GEMM kernels: algorithmic bytes (HBM-bound decode) or
    # flops (compute-bound large M) over their in-chain time
    if hbm:
        units = [gemm_bytes(r["fmt"], r["M"], r["N"], r["K"]) +
                 (quant_bytes(r["fmt"], r["M"], r["K"]) if wl.fused_item(i) else 0) for i, r in enumerate(wl.recs)]
        avg_units = sum(units) / n_gemm
        avg_us = float(gemm_us.sum()) / n_gemm
        achieved = sum(units) / (float(gemm_us.sum()) * 1e-6) / 1e9
        peak = hbm_peak
        by_fmt = {}
        for fmt in wl.formats:
            idx = [i for i, r in enumerate(wl.recs) if r["fmt"] == fmt]
            b = sum(units[i] for i in idx)
            ach = b / (float(gemm_us[idx].sum()) * 1e-6) / 1e9
            by_fmt[fmt] = {"achieved": round(ach, 1), "frac": round(ach / peak, 4),
                           "gemm_us": round(float(gemm_us[idx].sum()), 3)}
        traffic, traffic_note = measured_traffic(args.workload, wl.fused)
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                "frac": round(achieved / peak, 4), "traffic": traffic, "traffic_note": traffic_note,
                "kernel": ("fused quantize+gemm" if wl.fused else "gemm") + " (" + "+".join(wl.formats) + ")",
                "peak_kind": peak_kind, "avg_launch_us": round(avg_us, 3),
                "avg_bytes_per_launch": round(avg_units), "by_format": by_fmt, "timing": timing_note,
                "chain": chain,
                "step_frac": round(value / world / peak, 4)}
    else:
        # the E4M3 GEMMs (the dominant kernels) against the kind::f8f6f4 peak;
        # every format's own figure follows
        by_fmt = {}
        for fmt in wl.formats:
            idx = [i for i, r in enumerate(wl.recs) if r["fmt"] == fmt]
            fl = sum(2 * wl.recs[i]["M"] * wl.recs[i]["N"] * wl.recs[i]["K"] for i in idx)
            t = float(gemm_us[idx].sum())
            ach = fl / (t * 1e-6) / 1e12
            pk = tensor_peak(fmt, bf16_peak)
            by_fmt[fmt] = {"achieved": round(ach, 1), "peak": round(pk, 1), "frac": round(ach / pk, 4),
                           "gemm_us": round(t, 3)}
        main_fmt = "FP8_Dynamic" if "FP8_Dynamic" in by_fmt else wl.formats[0]
        avg_us = float(gemm_us.sum()) / n_gemm
        roof = {"bound": "tensor", "achieved": by_fmt[main_fmt]["achieved"], "peak": by_fmt[main_fmt]["peak"],
                "unit": "TFLOP/s", "frac": by_fmt[main_fmt]["frac"], "traffic": None,
                "kernel": f"gemm ({main_fmt})", "peak_kind": peak_kind + " bf16 x nominal kind ratio",
                "by_format": by_fmt, "avg_launch_us": round(avg_us, 3),
                "avg_flops_per_launch": round(wl.flops_step / n_gemm), "timing": timing_note, "chain": chain}

    # ---- end to end through the C ABI: pinned host activations in, outputs out.
    # Two buffer sets and two graphs: while step i's kernels run, a copy
    # stream uploads step i+1's activations and downloads step i-1's outputs
    # (every step still copies its own inputs in and its outputs out inside
    # the timed region).
    host_A = torch.empty(wl.A_all.numel(), dtype=torch.uint8, pin_memory=True)
    host_A.copy_(wl.A_all.cpu())
    host_Y = [torch.empty(wl.Y_all.numel(), dtype=torch.uint8, pin_memory=True) for _ in range(2)]
    e2e_steps = max(10, args.e2e_steps)
    A2, Y2 = torch.empty_like(wl.A_all), torch.empty_like(wl.Y_all)
    if args.no_graph:
        class _Direct2:
            def __init__(self, recs):
                self.recs = recs

            def replay(self):
                with torch.cuda.stream(stream):
                    wl.q.qg_set_launch_flags(wl.q.QG_LAUNCH_PDL if wl.pdl else 0)
                    for i in range(len(self.recs)):
                        wl.enqueue(stream, i, self.recs)
                    wl.q.qg_set_launch_flags(0)
        graph2 = _Direct2(wl.rebind(A2, Y2))
    else:
        graph2 = wl.capture_step(stream, wl.rebind(A2, Y2))
    sets = [(wl.A_all, wl.Y_all, graph), (A2, Y2, graph2)]
    copy_stream = torch.cuda.Stream(device=device)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = torch.cuda.Event()

    def pipelined(n):
        with torch.cuda.stream(copy_stream):
            sets[0][0].copy_(host_A, non_blocking=True)
            ev_in[0].record(copy_stream)
        for i in range(n):
            A_i, Y_i, g_i = sets[i % 2]
            stream.wait_event(ev_in[i % 2])
            g_i.replay()
            ev_done[i % 2].record(stream)
            with torch.cuda.stream(copy_stream):
                if i + 1 < n:  # after step i-1's download in this stream: its buffers are free
                    sets[(i + 1) % 2][0].copy_(host_A, non_blocking=True)
                    ev_in[(i + 1) % 2].record(copy_stream)
                copy_stream.wait_event(ev_done[i % 2])
                host_Y[i % 2].copy_(Y_i, non_blocking=True)
        ev_out.record(copy_stream)
        stream.wait_event(ev_out)

    with torch.cuda.stream(stream):
        pipelined(5)
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        copy_stream.wait_event(e0)
        pipelined(e2e_steps)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, e0.elapsed_time(e1) / e2e_steps, device)
    e2e_val = world * rate(wl.bytes_step, wl.flops_step, e2e_ms)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_oracle_leg(args.workload)

    per_gemm = [{"fmt": r["fmt"], "M": r["M"], "layer": r["layer"], "N": r["N"], "K": r["K"],
                 "variant": r["variant"], "split_k": r["split"], "us": round(float(gemm_us[i]), 3),
                 "quant_us": round(float(quant_us[i]), 3),
                 "GBps": round(gemm_bytes(r["fmt"], r["M"], r["N"], r["K"]) / (max(gemm_us[i], 1e-3) * 1e-6) / 1e9, 1),
                 "TFLOPs": round(2 * r["M"] * r["N"] * r["K"] / (max(gemm_us[i], 1e-3) * 1e-6) / 1e12, 2)}
                for i, r in enumerate(wl.recs)]
    if rank == 0:
        unit = "GB/s" if hbm else "TFLOP/s"
        cfg = _config(args.workload, WORKLOADS[args.workload]["items"])
        cfg.update({
            "gemms_per_step": n_gemm, "kernels_per_step": n_kernels,
            "activation_quantization": ("fused into the GEMM kernel wherever one kernel does both (--fused)"
                                        if wl.fused else
                                        f"qg_linear_w8a8: {sum(wl.fused_item(i) for i in range(n_gemm))} of {n_gemm} "
                                        "linears in one kernel (table rows with QG_CONFIG_FUSED_QUANT), the others "
                                        "a quantization kernel and the GEMM"),
            "bytes_per_step": wl.bytes_step, "flops_per_step": wl.flops_step,
            "weight_bytes_streamed_per_step": wl.weight_bytes_streamed,
            "l2": (f"inputs larger than L2: {wl.weight_bytes_streamed / 1e6:.0f} MB of weights streamed per step "
                   + ("(distinct weights per GEMM)" if not WORKLOADS[args.workload]["shared"] else
                      f"({wl.weight_bytes / 1e6:.0f} MB distinct; a reuse is separated by > 126 MB of other "
                      "weights)")),
            "graph": "one CUDA graph per step" + ("" if args.no_pdl else ", programmatic dependent launch"),
            "parallelism": f"replicas x{world}",
            "us_per_gemm": round(ms_step * 1e3 / n_gemm, 3)})
        if hbm:
            cfg["pct_of_peak"] = round(100 * value / world / hbm_peak, 1)
        line = {
            "metric": METRIC_HBM if hbm else METRIC_TENSOR,
            "value": round(value, 2), "unit": unit, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 6), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": workload_dtype(WORKLOADS[args.workload]["items"]), "data": "synthetic",
            "config": cfg,
            "roofline": roof,
            "e2e": {"value": round(e2e_val, 2), "unit": unit, "h2d_bytes_per_step": int(wl.A_all.numel()),
                    "d2h_bytes_per_step": int(wl.Y_all.numel()), "ms_per_step": round(e2e_ms, 6),
                    "pipelining": "two buffer sets: step i+1's upload and step i-1's download overlap step i's "
                                  "kernels (copy stream)"},
            "gpu_launches": n_kernels * args.steps,
            "clocks": clk,
            "cpu_baseline": cpu,
            "per_gemm": per_gemm,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
