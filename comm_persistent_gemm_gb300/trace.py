"""Role-trace analysis: time accounting per role and a Chrome-trace export.

A trace record (one per claimed entry, see kosmos_trace_rec in kosmos.h) has
t_claim (ticket taken), t_ready (its readiness wait ended), t_done (its work
finished), kind, ticket and cta.  The accounting follows the explainer's
worked example (paragraph "A worked example"): for each role the busy time
(work), the time spent waiting for data, and the idle time of CTAs between
entries and after their last entry up to the end of the launch.
"""
from __future__ import annotations

import json
from typing import Dict, Iterable, List, Optional

import numpy as np

KIND_NAMES = {1: "TRANSFER", 2: "TILE", 3: "REDUCE", 4: "ROUTE", 5: "DISPATCH", 6: "TILE_GU", 7: "TILE_D",
              8: "PUSH", 9: "FOLD", 10: "TILE_HALF", 11: "QUANT", 16: "ZPAD", 17: "GRADIN", 18: "RBWD",
              19: "RDX", 20: "DH", 21: "DGU", 22: "DWD", 23: "DWGU", 24: "DWR"}
TRACE_DTYPE = np.dtype([("t_claim", "<i8"), ("t_ready", "<i8"), ("t_done", "<i8"), ("kind", "<i4"),
                        ("ticket", "<i4"), ("cta", "<i4"), ("pad", "<i4")])


def as_records(rows: Iterable) -> np.ndarray:
    """Records from an iterable of (t_claim, t_ready, t_done, kind, ticket, cta)."""
    rows = list(rows)
    out = np.zeros(len(rows), dtype=TRACE_DTYPE)
    for i, r in enumerate(rows):
        out[i] = (r[0], r[1], r[2], r[3], r[4], r[5], 0)
    return out


def summarize(recs: np.ndarray, n_ctas: Optional[int] = None) -> Dict[str, object]:
    """Time accounting of one launch.

    makespan   : last t_done - first t_claim
    per kind   : entries, busy (t_done - t_ready), wait (t_ready - t_claim)
    idle       : sum over CTAs of (makespan - time covered by that CTA's entries)
    utilisation: sum of busy / (CTAs x makespan)
    Times are in the records' unit (ns for the GPU's globaltimer).
    """
    recs = recs[recs["kind"] != 0]
    if len(recs) == 0:
        return {"makespan": 0, "kinds": {}, "idle": 0, "utilisation": 0.0, "ctas": 0}
    t0 = int(recs["t_claim"].min())
    t1 = int(recs["t_done"].max())
    span = t1 - t0
    ctas = np.unique(recs["cta"])
    n = n_ctas if n_ctas is not None else len(ctas)
    kinds = {}
    for k in np.unique(recs["kind"]):
        r = recs[recs["kind"] == k]
        kinds[KIND_NAMES.get(int(k), str(int(k)))] = {
            "entries": int(len(r)),
            "busy": int((r["t_done"] - r["t_ready"]).sum()),
            "wait": int((r["t_ready"] - r["t_claim"]).sum()),
            "ctas": int(len(np.unique(r["cta"]))),
        }
    covered = 0
    for c in ctas:
        r = recs[recs["cta"] == c]
        covered += int((r["t_done"] - r["t_claim"]).sum())
    busy = sum(v["busy"] for v in kinds.values())
    idle = n * span - covered
    return {"makespan": span, "kinds": kinds, "idle": int(idle), "utilisation": busy / (n * span) if span else 0.0,
            "ctas": int(n)}


def chrome_trace(recs: np.ndarray, path: Optional[str] = None) -> List[dict]:
    """Chrome / Perfetto trace events: one row per CTA, a wait slice and a
    work slice per entry (microseconds)."""
    recs = recs[recs["kind"] != 0]
    t0 = int(recs["t_claim"].min()) if len(recs) else 0
    ev = []
    for r in recs:
        name = KIND_NAMES.get(int(r["kind"]), str(int(r["kind"])))
        if r["t_ready"] > r["t_claim"]:
            ev.append({"name": f"wait {name}", "ph": "X", "pid": 0, "tid": int(r["cta"]),
                       "ts": (int(r["t_claim"]) - t0) / 1e3, "dur": (int(r["t_ready"]) - int(r["t_claim"])) / 1e3})
        ev.append({"name": name, "ph": "X", "pid": 0, "tid": int(r["cta"]), "ts": (int(r["t_ready"]) - t0) / 1e3,
                   "dur": max(0, int(r["t_done"]) - int(r["t_ready"])) / 1e3, "args": {"ticket": int(r["ticket"])}})
    if path:
        with open(path, "w") as fh:
            json.dump({"traceEvents": ev}, fh)
    return ev
