"""Launch one GEMM configuration a few times, plainly (no graph, no
programmatic dependent launch), for a kernel profiler such as ncu.

Each launch reads its own window of a pool of random weight bytes (several
hundred MB, beyond L2), so the profiled launch streams its weights from HBM.

Usage:  python -m quantized_gemm_decode_02_b300.profile_gemm FORMAT M N K VARIANT SPLIT_K CONFIG_ID REPS
e.g.    python -m quantized_gemm_decode_02_b300.profile_gemm W8A8_INT8 32 12288 2048 3 2 0 4
"""
from __future__ import annotations

import argparse
import os
import sys

import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from quantized_gemm_decode_02_b300 import qgemm as q  # noqa: E402


def main(argv=None) -> int:
    ap = argparse.ArgumentParser()
    ap.add_argument("fmt", choices=sorted(q.FORMATS))
    for name in ("M", "N", "K", "variant", "split_k", "config_id", "reps"):
        ap.add_argument(name, type=int)
    a = ap.parse_args(argv)
    dev = "cuda:0"
    g = torch.Generator(device=dev)
    g.manual_seed(1)
    wb = a.N * a.K
    copies = max(2, min(16, -(-400_000_000 // wb)))
    pool = torch.randint(0, 256, (copies * wb,), dtype=torch.uint8, device=dev, generator=g)
    Aq = torch.randint(0, 256, (a.M * a.K,), dtype=torch.uint8, device=dev, generator=g)
    sa = torch.ones(a.M * ((a.K + 127) // 128) + 1, dtype=torch.float32, device=dev)
    sw = torch.ones(max(a.N, ((a.N + 127) // 128) * ((a.K + 127) // 128)), dtype=torch.float32, device=dev)
    Y = torch.empty(a.M * a.N, dtype=torch.bfloat16, device=dev)
    need = q.qg_workspace_bytes_config(a.fmt, a.M, a.N, a.K, a.variant, a.split_k, a.config_id)
    ws = torch.zeros(max(need, 256), dtype=torch.uint8, device=dev)
    for r in range(a.reps):
        W = pool[(r % copies) * wb:(r % copies + 1) * wb]
        q.qg_gemm_w8a8(a.fmt, a.M, a.N, a.K, Aq, sa, W, sw, Y, a.N, a.variant, a.split_k, a.config_id, ws, need, None)
    torch.cuda.synchronize()
    if q.qg_device_error() != 0:
        raise SystemExit("device status reported an error")
    print("ok", a.fmt, a.M, a.N, a.K, a.variant, a.split_k, a.config_id, a.reps)
    return 0


if __name__ == "__main__":
    sys.exit(main())
