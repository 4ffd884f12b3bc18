"""Host logic of bench.py that runs without a GPU: the reference arm (the
CPU oracle timed on a bounded sample) keeps its whole run within its time
budget for any step count, and prints the contract's JSON line."""
from __future__ import annotations

import io
import json
from contextlib import redirect_stdout

import pytest


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


@pytest.mark.parametrize("runs", [4, 23, 103, 1000, 20100, 10 ** 6])
@pytest.mark.parametrize("t_pass16", [0.001, 0.03, 9.0])
def test_reference_plan_fits_the_budget(bench, runs, t_pass16):
    n_items = 28
    cols, per_step = bench.reference_plan(n_items, t_pass16 / n_items, t_pass16, runs, budget_s=120.0)
    assert 16 <= cols <= 8192 and 1 <= per_step <= n_items
    # the plan's own estimate of a step: a pass is at least the 16-column pass
    est_step = t_pass16 * max(1.0, cols / 16) * per_step / n_items
    if per_step > 1 or cols > 16:
        assert runs * est_step <= 120.0 * 1.0001
    if per_step < n_items:
        assert cols == 16                      # subsets only once 16 columns of every item do not fit
    if runs * t_pass16 <= 120.0:
        assert per_step == n_items             # the whole workload whenever it fits


def test_reference_arm_prints_the_contract_line(bench):
    out = io.StringIO()
    with redirect_stdout(out):
        rc = bench.main(["--impl", "reference", "--steps", "2", "--warmup", "3", "--reference-budget-s", "10"])
    assert rc == 0
    line = json.loads(out.getvalue().strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3
    assert line["value"] > 0 and line["unit"] == "GB/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["value"] == line["value"]
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["e2e"]["value"] == line["value"]
    assert line["config"]["workload"] == bench.DEFAULT_WORKLOAD
    assert not {"model", "models", "global_batch", "seq_len"} & set(line["config"])  # a workload, not a model
    assert line["config"]["shapes_k_n"]["Qwen3-8B down"] == [12288, 4096]
    assert line["config"]["formats"] == ["Block_FP8", "FP8_Dynamic", "W8A8_INT8"]


def test_cpu_baseline_leg_reports_a_bounded_sample(bench):
    r = bench.cpu_oracle_leg(bench.DEFAULT_WORKLOAD, budget_s=0.5)
    assert r["kind"] == "oracle" and r["unit"] == "GB/s" and r["value"] > 0 and r["cores"] >= 1
    assert "all 384 (format, M, layer) items" in r["sample"]
