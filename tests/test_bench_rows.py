"""bench.py's extra rows, on the host: the plain default single-GPU run also
times the other workloads and E4M3 pools after the headline one and reports
them in the same (single) JSON line; the profiling commands and multi-rank
runs do not; a row that fails leaves its error in the line and the headline
numbers intact.  The measurement itself is stubbed: only the control flow runs
here."""
from __future__ import annotations

import json

import pytest

import bench


def fake_result(args):
    return {"metric": bench.METRIC, "value": 1.0, "unit": bench.UNIT, "ms_per_step": 2.0,
            "config": {"workload": bench.DESCR[args.workload]}, "gpu_launches": 3,
            "clocks": {"sm_mhz": 2070.0},
            "roofline": {"kernel": bench.KERNEL_OF[args.workload][0], "avg_launch_ms": 0.5,
                         "achieved": 100.0, "frac": 0.5, "algorithmic_bytes_per_launch": 50,
                         "traffic": None}}


@pytest.mark.parametrize("argv,ws,want", [
    ([], 1, True),
    (["--gpus", "1", "--steps", "20", "--warmup", "5"], 1, True),
    ([], 2, False),                                     # replicas under torchrun
    (["--workload", "wide"], 1, False),
    (["--kv", "fp8"], 1, False),
    (["--no-e2e"], 1, False),                           # the profiling commands
    (["--no-cpu-baseline"], 1, False),
    (["--queries", "64"], 1, False),
    (["--fused"], 1, False),
    (["--row", "offline"], 1, False),
    (["--impl", "reference"], 1, False),
    (["--no-extra-rows"], 1, False),
])
def test_which_runs_add_rows(argv, ws, want):
    assert bench.wants_extra_rows(bench.parse_args(argv), ws) is want


def test_rows_use_the_headline_measurement_with_fewer_steps():
    seen = []

    def run(a):
        seen.append(a)
        return fake_result(a)

    rows = bench.run_extra_rows(bench.parse_args(["--steps", "20", "--warmup", "5"]), run=run)
    assert [(r["workload"], r["kv"]) for r in rows] == bench.EXTRA_ROWS
    for a in seen:
        assert a.steps == 10 and a.warmup == 5
        assert a.no_e2e and a.no_cpu_baseline and not a.fused
        assert a.queries == a.pool_items == a.layers == 0
    assert all(r["frac"] == 0.5 and r["kernel"] == bench.KERNEL_OF[r["workload"]][0] for r in rows)


def test_a_failing_row_is_reported_and_the_rest_still_run():
    def run(a):
        if a.workload == "paged" and a.kv == "fp8":
            raise RuntimeError("device status 2")
        return fake_result(a)

    rows = bench.run_extra_rows(bench.parse_args([]), run=run)
    bad = [r for r in rows if "error" in r]
    assert len(bad) == 1 and bad[0]["workload"] == "paged" and "device status 2" in bad[0]["error"]
    assert len(rows) == len(bench.EXTRA_ROWS)


def test_the_default_run_prints_one_line_with_the_rows(monkeypatch, capsys):
    monkeypatch.setattr(bench, "run_ours", fake_result)
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main([])
    lines = [ln for ln in capsys.readouterr().out.splitlines() if ln.strip()]
    assert len(lines) == 1
    res = json.loads(lines[0])
    assert res["value"] == 1.0
    assert [(r["workload"], r["kv"]) for r in res["rows"]] == bench.EXTRA_ROWS


def test_profiling_runs_print_no_rows(monkeypatch, capsys):
    monkeypatch.setattr(bench, "run_ours", fake_result)
    monkeypatch.setenv("WORLD_SIZE", "1")
    bench.main(["--steps", "2", "--warmup", "3", "--no-cpu-baseline", "--no-e2e"])
    res = json.loads(capsys.readouterr().out.strip())
    assert "rows" not in res
