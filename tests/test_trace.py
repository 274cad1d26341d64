"""Time accounting of the role trace, pinned to the explainer's worked example
(tests/golden/worked_example.json): a fixed 32-unit crew on a 256-unit GPU
against one-way switching, reproduced as synthetic traces."""
import json
import os

import numpy as np

from comm_persistent_gemm_gb300.trace import as_records, chrome_trace, summarize

G = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "worked_example.json")))
MS = 1_000_000  # ns per ms


def _fixed_split_trace():
    rows = []
    n, crew = G["units_total"], G["crew"]
    gemm = G["gemm_full_ms"] / G["retained_throughput"]
    # builders: one tile each spanning the reduced-throughput GEMM, then idle
    for c in range(crew, n):
        rows.append((0, 0, int(round(gemm * MS)), 2, c, c))
    # the crew reduces during the GEMM and carries the tail alone
    for c in range(crew):
        rows.append((0, 0, int(round((gemm + G["tail_fixed_ms"]) * MS)), 3, c, c))
    return as_records(rows)


def _switch_trace():
    rows = []
    n, crew = G["units_total"], G["crew"]
    gemm = G["gemm_full_ms"] / G["retained_throughput"]
    tail = G["tail_switch_ms"]
    for c in range(crew, n):
        rows.append((0, 0, int(round(gemm * MS)), 2, c, c))
        # builders join the reduction when the tiles run out (one-way switch)
        rows.append((int(round(gemm * MS)), int(round(gemm * MS)), int(round((gemm + tail) * MS)), 3, n + c, c))
    for c in range(crew):
        rows.append((0, 0, int(round((gemm + tail) * MS)), 3, c, c))
    return as_records(rows)


def test_worked_example_reduced_gemm_time():
    assert round(G["gemm_full_ms"] / G["retained_throughput"], 2) == G["gemm_reduced_ms"]


def test_worked_example_fixed_vs_switch():
    f = summarize(_fixed_split_trace())
    s = summarize(_switch_trace())
    assert abs(f["makespan"] / MS - G["total_fixed_ms"]) < 0.01
    assert abs(s["makespan"] / MS - G["total_switch_ms"]) < 0.01
    assert round(f["makespan"] / s["makespan"], 2) == G["speedup"]
    # in the fixed split every builder idles through the tail
    n, crew = G["units_total"], G["crew"]
    assert abs(f["idle"] / MS - (n - crew) * G["tail_fixed_ms"]) < 0.5
    assert s["idle"] < f["idle"]
    assert s["kinds"]["REDUCE"]["ctas"] == n


def test_accounting_definitions_and_chrome_export(tmp_path):
    recs = as_records([(0, 5, 15, 2, 0, 0), (15, 15, 20, 2, 1, 0), (0, 0, 10, 1, 0, 1)])
    s = summarize(recs)
    assert s["makespan"] == 20
    assert s["kinds"]["TILE"] == {"entries": 2, "busy": 15, "wait": 5, "ctas": 1}
    assert s["kinds"]["TRANSFER"]["busy"] == 10
    assert s["idle"] == 2 * 20 - (20 + 10)
    ev = chrome_trace(recs, str(tmp_path / "t.json"))
    assert len(ev) == 4 and json.load(open(tmp_path / "t.json"))["traceEvents"]
