"""bench.py with more than one GPU runs independent replicas (the path has no
exchange step): every rank runs the same workload, the ranks meet at a
barrier around the timed region, the step time is the maximum over ranks,
and only rank 0 prints (the reference arm too).  The host side of that is
checked here with two gloo ranks on the CPU."""
from __future__ import annotations

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    os.environ.update({"MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port), "RANK": str(rank),
                       "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank)})
    sys.path.insert(0, ROOT)
    import io
    import contextlib
    import torch.distributed as dist
    import bench
    w, r, _ = bench.dist_setup()
    bench.barrier(w)
    step_ms = [3.0, 7.5][r]
    slowest = bench.max_over_ranks(w, step_ms, "cpu")
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        rc = bench.run_reference(None, w, r) if r != 0 else 0  # non-zero ranks: no work, no output
    bench.barrier(w)
    dist.destroy_process_group()
    out.put((r, w, slowest, rc, buf.getvalue()))


@pytest.mark.timeout(120)
def test_two_gloo_replicas():
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=100) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for r, w, slowest, rc, printed in got:
        assert w == 2
        assert slowest == 7.5          # the step time is the slowest rank's
        assert rc == 0
    assert got[1][4] == ""             # rank 1 of the reference arm prints nothing
