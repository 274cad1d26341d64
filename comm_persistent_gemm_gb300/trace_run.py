"""Runs one traced launch of each fused operator on the full-size synthetic
workloads and writes Chrome traces plus the role time accounting.

    python -m comm_persistent_gemm_gb300.trace_run --out DIR [--only ag,rs,moe,mxfp8,moe_mxfp8,moe_bwd]

Output: DIR/<name>.trace.json (chrome://tracing / Perfetto) and one JSON line
per traced launch on stdout with the summary of trace.summarize().
"""
from __future__ import annotations

import argparse
import json
import os
import sys

import numpy as np


def _trace_ag(K, out, name, o):
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    w = WORKLOADS["ag_bf16_p8"]
    inp = workload_inputs(w)
    xs = [x.cuda() for x in inp["x"]]
    W = inp["w"].cuda()
    xg = torch.empty(w.P * w.m, w.k, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(w.P * w.m, w.n, dtype=torch.bfloat16, device="cuda")
    ws = K.workspace(K.OP_AG_GEMM, w.P, w.m, w.n, w.k, o=o)
    for _ in range(3):
        K.ag_gemm(xs, W, xg, y, ws, o)
    K.check(ws, name)
    ws.zero_()
    K.ag_gemm(xs, W, xg, y, ws, o)
    K.check(ws, name)
    return K.trace_records(K.OP_AG_GEMM, w.P, w.m, w.n, w.k, ws, o)


def _trace_mxfp8(K, out, name, o):
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    w = WORKLOADS["ag_mxfp8_p8"]
    inp = workload_inputs(w)

    def quant(x, along):
        r, c = x.shape
        q = torch.empty(r, c, dtype=torch.uint8, device="cuda")
        sc = torch.empty(K.mxfp8_scale_bytes(r, c, along), dtype=torch.uint8, device="cuda")
        K.mxfp8_quantize(x.cuda(), q, sc, along)
        return q, sc

    qs, ss = zip(*[quant(x, True) for x in inp["x"]])
    qw, sw = quant(inp["w"], False)
    xg = torch.empty(w.P * w.m, w.k, dtype=torch.uint8, device="cuda")
    y = torch.empty(w.P * w.m, w.n, dtype=torch.bfloat16, device="cuda")
    ws = K.workspace(K.OP_AG_GEMM, w.P, w.m, w.n, w.k, dtype=K.MXFP8_E4M3, o=o)
    run = lambda: K.ag_gemm(list(qs), qw, xg, y, ws, o, dtype=K.MXFP8_E4M3, x_scales=list(ss), w_scales=sw)
    for _ in range(3):
        run()
    K.check(ws, name)
    ws.zero_()
    run()
    K.check(ws, name)
    return K.trace_records(K.OP_AG_GEMM, w.P, w.m, w.n, w.k, ws, o, dtype=K.MXFP8_E4M3)


def _trace_rs(K, out, name, o):
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    w = WORKLOADS["rs_bf16_p8"]
    inp = workload_inputs(w)
    xs = [x.cuda() for x in inp["x"]]
    ws_ = [x.cuda() for x in inp["w"]]
    ys = [torch.empty(w.m // w.P, w.n, dtype=torch.bfloat16, device="cuda") for _ in range(w.P)]
    ws = K.workspace(K.OP_GEMM_RS, w.P, w.m, w.n, w.k, o=o)
    for _ in range(2):
        K.gemm_rs(xs, ws_, ys, ws, o)
    K.check(ws, name)
    ws.zero_()
    K.gemm_rs(xs, ws_, ys, ws, o)
    K.check(ws, name)
    return K.trace_records(K.OP_GEMM_RS, w.P, w.m, w.n, w.k, ws, o)


def _quant_experts(K, w, P):
    import torch
    E, Kd, N = w.shape
    nb = K.mxfp8_scale_bytes(Kd, N, False)
    codes, scales = [], []
    for q in range(P):
        c = torch.empty(E // P, Kd, N, dtype=torch.uint8, device="cuda")
        s = torch.empty((E // P) * nb, dtype=torch.uint8, device="cuda")
        for j in range(E // P):
            K.mxfp8_quantize(w[q * (E // P) + j].cuda(), c[j], s[j * nb:(j + 1) * nb], False)
        codes.append(c)
        scales.append(s)
    return codes, scales


def _trace_moe(K, out, name, o, mx=False):
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    from .trace import TRACE_DTYPE
    w = WORKLOADS["moe_fwd_p8"]
    inp = workload_inputs(w)
    P, T, H, E, Kt, I = w.P, w.T, w.H, w.E, w.topk, w.I
    xs = [t.cuda() for t in torch.chunk(inp["x"], P, 0)]
    wr = inp["w_router"].cuda()
    kw = {}
    if mx:
        (wg, sg), (wu, su), (wd, sd) = (_quant_experts(K, inp[n], P) for n in ("w_gate", "w_up", "w_down"))
        kw = {"dtype": K.MXFP8_E4M3, "w_gate_scales": sg, "w_up_scales": su, "w_down_scales": sd}
    else:
        sp = lambda t: [t[q * (E // P):(q + 1) * (E // P)].contiguous().cuda() for q in range(P)]
        wg, wu, wd = sp(inp["w_gate"]), sp(inp["w_up"]), sp(inp["w_down"])
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    idx = torch.empty(T, Kt, dtype=torch.int32, device="cuda")
    gate = torch.empty(T, Kt, dtype=torch.float32, device="cuda")
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    pos = torch.empty(T, Kt, dtype=torch.int32, device="cuda")
    dt = K.MXFP8_E4M3 if mx else K.BF16
    ws = K.moe_workspace(P, T, H, E, Kt, I, o, dtype=dt)
    for _ in range(2):
        K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, cnt, pos, ws, Kt, o, **kw)
    K.check(ws, name)
    ws.zero_()
    K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, cnt, pos, ws, Kt, o, **kw)
    K.check(ws, name)
    raw = K.moe_debug_view(K.MOE_VIEW_TRACE, P, T, H, E, Kt, I, ws, dtype=dt).cpu().numpy()
    recs = raw.view(TRACE_DTYPE)
    return recs[recs["kind"] != 0]


def _trace_moe_bwd(K, out, name, o):
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    from .trace import TRACE_DTYPE
    w = WORKLOADS["moe_fwd_p8"]
    inp = workload_inputs(w)
    P, T, H, E, Kt, I = w.P, w.T, w.H, w.E, w.topk, w.I
    xs = [t.cuda() for t in torch.chunk(inp["x"], P, 0)]
    wr = inp["w_router"].cuda()
    sp = lambda t: [t[q * (E // P):(q + 1) * (E // P)].contiguous().cuda() for q in range(P)]
    wg, wu, wd = sp(inp["w_gate"]), sp(inp["w_up"]), sp(inp["w_down"])
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    idx = torch.empty(T, Kt, dtype=torch.int32, device="cuda")
    gate = torch.empty(T, Kt, dtype=torch.float32, device="cuda")
    cnt = torch.empty(E, dtype=torch.int32, device="cuda")
    pos = torch.empty(T, Kt, dtype=torch.int32, device="cuda")
    fws = K.moe_workspace(P, T, H, E, Kt, I)
    K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, cnt, pos, fws, Kt)
    K.check(fws, "moe_fwd")
    g = torch.Generator().manual_seed(11)
    dys = [t.cuda() for t in torch.chunk(torch.randn(T, H, generator=g).to(torch.bfloat16), P, 0)]
    dxs = [torch.empty(T // P, H, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    dwr = torch.empty(H, E, dtype=torch.float32, device="cuda")
    dwg, dwu, dwd = [torch.empty_like(t) for t in wg], [torch.empty_like(t) for t in wu], [torch.empty_like(t) for t in wd]
    bws = K.moe_bwd_workspace(P, T, H, E, Kt, I, o)
    run = lambda: K.moe_bwd(xs, wr, wg, wu, wd, idx, gate, fws, dys, dxs, dwr, dwg, dwu, dwd, bws, o)
    for _ in range(2):
        run()
    K.check(bws, name)
    bws.zero_()
    run()
    K.check(bws, name)
    raw = K.moe_bwd_debug_view(K.MOE_BWD_VIEW_TRACE, P, T, H, E, Kt, I, bws).cpu().numpy()
    recs = raw.view(TRACE_DTYPE)
    return recs[recs["kind"] != 0]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--out", required=True)
    ap.add_argument("--only", default="ag,rs,moe")
    ap.add_argument("--tail-split", type=int, default=None, help="all-gather: kosmos_opts.tail_split")
    a = ap.parse_args(argv)
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import comm_persistent_gemm_gb300 as K
    from .trace import chrome_trace, summarize
    K.build()
    os.makedirs(a.out, exist_ok=True)
    sms = K.num_sms()
    runs = []
    only = set(a.only.split(","))
    if "ag" in only:
        ts = a.tail_split
        runs += [("ag_self", _trace_ag, K.opts(trace=1, tail_split=ts)),
                 ("ag_fixed19", _trace_ag, K.opts(trace=1, sched=K.SCHED_FIXED, fixed_comm_ctas=-(-sms // 8),
                                                  tail_split=ts))]
    if "mxfp8" in only:
        runs += [("ag_mxfp8_self", _trace_mxfp8, K.opts(trace=1))]
    if "rs" in only:
        runs += [("rs_band", _trace_rs, K.opts(trace=1)), ("rs_row", _trace_rs, K.opts(trace=1, order=K.ORDER_ROW))]
    if "moe" in only:
        runs += [("moe_fwd", _trace_moe, K.opts(trace=1))]
    if "moe_bwd" in only:
        runs += [("moe_bwd", _trace_moe_bwd, K.opts(trace=1))]
    if "moe_mxfp8" in only:
        runs += [("moe_fwd_mxfp8", lambda *a: _trace_moe(*a, mx=True), K.opts(trace=1))]
    for name, fn, o in runs:
        recs = fn(K, a.out, name, o)
        s = summarize(recs, n_ctas=sms)
        chrome_trace(recs, os.path.join(a.out, f"{name}.trace.json"))
        s["name"] = name
        # per-CTA finish spread: when each CTA's last entry ended, relative to the launch start
        t0 = int(recs["t_claim"].min())
        last = np.array([int(recs["t_done"][recs["cta"] == c].max()) - t0 for c in np.unique(recs["cta"])])
        s["cta_finish_ns"] = {"min": int(last.min()), "median": int(np.median(last)), "max": int(last.max())}
        print(json.dumps(s))
    return 0


if __name__ == "__main__":
    sys.exit(main())
