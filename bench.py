#!/usr/bin/env python3
"""Benchmark of the fused all-gather + GEMM persistent kernel (KOSMOS method)
on the 8-rank workload X_r [1024, 8192] x 8, W [8192, 3584] (bf16, fp32
accumulate), with the fixed-split and unfused baselines, the GEMM+RS and MoE
kernels when built, the CPU oracle timed on the host cores, and the
roofline of the dominant kernel.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

Prints ONE JSON line (rank 0).  N > 1 (under torchrun) runs N independent
replicas, one per GPU: the emulated ranks live in one GPU's HBM, so nothing
shards across GPUs ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "ag_bf16_p8"
METRIC = "Fused AG/RS-GEMM TFLOP/s & % BF16 tensor peak on 1 GB300; MoE layer tokens/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}

# DRAM bytes (read + write) of one ag_gemm_pair_kernel launch on the 8-rank AG
# workload, from an ncu capture; valid only while the kernel sources hash to
# src_sha (otherwise the bench reports traffic = null).
TRAFFIC_CAPTURE = {"bytes": 830933248, "src_sha": "5fac42c3390fb242"}
KERNEL_SOURCES = ["comm_persistent_gemm_gb300/csrc/ag_gemm.cu", "comm_persistent_gemm_gb300/csrc/engine.cuh",
                  "comm_persistent_gemm_gb300/csrc/engine2.cuh", "comm_persistent_gemm_gb300/csrc/ptx.cuh",
                  "comm_persistent_gemm_gb300/csrc/common.cuh"]


def kernel_src_sha() -> str:
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as fh:
            d = json.load(fh)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """SM clock and throttle-reason samples taken during the timed region.

    A thread of this process reads NVML every 2 ms (read-only queries: the SM
    clock, the maximum SM clock and the active clock-event reasons), so a
    timed region of a few milliseconds still holds samples.  Where the NVML
    library cannot be loaded, nvidia-smi polling every 200 ms is used instead."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    # clock-event reason bits of NVML's public header
    REASON_BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8, "sw_thermal_slowdown": 0x20,
                   "hw_thermal_slowdown": 0x40}
    NVML_CLOCK_SM = 1
    PERIOD_S = 0.002

    def __init__(self, device):
        import torch
        self.index = device.index if device.index is not None else 0
        try:
            self.uuid = "GPU-" + str(torch.cuda.get_device_properties(self.index).uuid)
        except (AttributeError, RuntimeError):
            self.uuid = None
        self.proc = None
        self.nvml = None
        self.samples = []
        self.path = os.path.join("/tmp", f"kosmos_clocks_{os.getpid()}.csv")

    # ---- NVML in-process sampler
    def _nvml_open(self):
        import ctypes
        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return False
        h = ctypes.c_void_p()
        ok = self.uuid is not None and nv.nvmlDeviceGetHandleByUUID(self.uuid.encode(), ctypes.byref(h)) == 0
        if not ok and nv.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(self.index), ctypes.byref(h)) != 0:
            nv.nvmlShutdown()
            return False
        mx = ctypes.c_uint()
        self.sm_max = (float(mx.value) if nv.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0
                       else None)
        try:
            self.reasons_fn = nv.nvmlDeviceGetCurrentClocksEventReasons
        except AttributeError:
            self.reasons_fn = nv.nvmlDeviceGetCurrentClocksThrottleReasons
        self.nvml, self.handle = nv, h
        return True

    def _poll(self):
        import ctypes
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while True:
            if (self.nvml.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, ctypes.byref(clk)) == 0
                    and self.reasons_fn(self.handle, ctypes.byref(rs)) == 0):
                self.samples.append((float(clk.value), int(rs.value)))
            if self.stop.wait(self.PERIOD_S):
                return

    def __enter__(self):
        import threading
        try:
            opened = self._nvml_open()
        except (OSError, AttributeError):
            opened = False
        if opened:
            self.stop = threading.Event()
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            t0 = time.time()
            while not self.samples and time.time() - t0 < 1.0:
                time.sleep(0.001)
            return self
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", self.uuid or str(self.index),
                                          f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.fh, stderr=subprocess.DEVNULL)
            # the timed region starts once nvidia-smi has written its first
            # sample (its start-up would otherwise overlap the first steps)
            t0 = time.time()
            while time.time() - t0 < 5.0 and self.proc.poll() is None:
                if os.path.getsize(self.path) > 0:
                    break
                time.sleep(0.01)
            time.sleep(0.05)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.nvml is not None:
            self.stop.set()
            self.thread.join(timeout=5)
            self.nvml.nvmlShutdown()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.fh.close()

    @staticmethod
    def _summarise(sm, smax, reasons, source):
        busy = [s for s in sm if smax and s > 0.5 * smax] or sm
        return {"sm_mhz": statistics.median(busy) if busy else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm), "source": source}

    def summary(self):
        if self.nvml is not None:
            reasons = {nm for nm, bit in self.REASON_BITS.items() for _, r in self.samples if r & bit}
            return self._summarise([s for s, _ in self.samples], self.sm_max, reasons,
                                   f"NVML every {self.PERIOD_S * 1e3:.0f} ms")
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax = float(parts[2])
            except ValueError:
                continue
            for nm, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        os.unlink(self.path)
        return self._summarise(sm, smax, reasons, "nvidia-smi every 200 ms")


def dist_max(value: float, device=None) -> float:
    """Maximum of a per-rank value over all ranks (the value itself when not
    running distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(work_per_rank: float, step_ms_max: float, world: int) -> float:
    """Units per second processed by all ranks, timed by the slowest rank."""
    return world * work_per_rank / (step_ms_max * 1e-3)


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


# --------------------------------------------------------------------------- CPU oracle timing
def time_oracle_ag(inp, target_s: float = 12.0):
    """The oracle, as it stands, on a bounded sample of output rows of the
    AG workload; returns TFLOP/s on the host cores."""
    import numpy as np
    import oracle
    from kosmos_inputs import bf16_bits
    oracle.build()
    xs = [bf16_bits(x) for x in inp["x"]]
    w = bf16_bits(inp["w"])
    P = len(xs)
    m, k = xs[0].shape
    n = w.shape[1]
    rows = np.arange(0, P * m, max(1, (P * m) // 32), dtype=np.int64)[:32]
    t0 = time.perf_counter()
    oracle.ag_gemm(xs, w, rows=rows)
    dt = time.perf_counter() - t0
    want = int(min(P * m, max(32, len(rows) * target_s / max(dt, 1e-3))))
    rows = np.linspace(0, P * m - 1, want).astype(np.int64)
    t0 = time.perf_counter()
    oracle.ag_gemm(xs, w, rows=rows)
    dt = time.perf_counter() - t0
    flops = 2.0 * len(rows) * k * n
    return {"value": flops / dt / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{len(rows)} of {P * m} output rows of Y = concat(X_r) W (fp64, {dt:.1f} s)"}


# --------------------------------------------------------------------------- GPU timing
def time_kernel_steps(fn, steps, warmup, flush, stream):
    """Per-step CUDA-event times (ms) on `stream`, L2 flushed before each step
    (outside the events)."""
    import torch
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    times = []
    for _ in range(steps):
        flush()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        fn()
        b.record(stream)
        b.synchronize()
        times.append(a.elapsed_time(b))
    return times


def paired_medians(fn_a, fn_b, flush, stream, rounds=5, steps=10):
    """Median per-round mean step time (ms) of two configurations timed in
    alternation (a, b, a, b, ...).  A sweep's best point is the maximum of
    noisy samples, biased upward against a configuration timed once; the
    paired comparison of the sweep's choice removes that bias."""
    ta, tb = [], []
    for _ in range(rounds):
        ta.append(statistics.mean(time_kernel_steps(fn_a, steps, 2, flush, stream)))
        tb.append(statistics.mean(time_kernel_steps(fn_b, steps, 2, flush, stream)))
    return statistics.median(ta), statistics.median(tb)


def _split_experts(w, P):
    E = w.shape[0]
    return [w[q * (E // P):(q + 1) * (E // P)].contiguous() for q in range(P)]


def bench_rs(K, dev, steps, warmup, flush, stream, peak):
    """GEMM + reduce-scatter, 8 ranks x [8192, 3584] . [3584, 8192]: band order
    (the method), the row-order ablation, the fixed-split crew sweep and the
    unfused GEMM-then-reduce baseline."""
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    w = WORKLOADS["rs_bf16_p8"]
    inp = workload_inputs(w)
    P, m, k, n = w.P, w.m, w.k, w.n
    xs = [x.to(dev) for x in inp["x"]]
    ws_ = [x.to(dev) for x in inp["w"]]
    del inp
    ys = [torch.empty(m // P, n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    flops = w.flops()

    def timed(o):
        wsb = K.workspace(K.OP_GEMM_RS, P, m, n, k, o=o, device=dev)
        f = lambda: K.gemm_rs(xs, ws_, ys, wsb, o, stream=stream)
        f()
        K.check(wsb, "gemm_rs")
        t = time_kernel_steps(f, steps, warmup, flush, stream)
        K.check(wsb, "gemm_rs")
        del wsb
        return statistics.mean(t)

    band = timed(K.opts(order=K.ORDER_BAND))
    row = timed(K.opts(order=K.ORDER_ROW))
    fixed = {}
    for crew in (1, 2, 3):  # reducer pairs per rank
        fixed[str(crew)] = flops / (timed(K.opts(sched=K.SCHED_FIXED, fixed_comm_ctas=crew)) * 1e-3) / 1e12
    unf = timed(K.opts(sched=K.SCHED_UNFUSED))
    single = timed(K.opts(cta_pair=0))
    tfl = lambda ms: flops / (ms * 1e-3) / 1e12
    link = {"self": tfl(timed(K.opts(link_gbs=LINK_GBS))),
            "fixed_sweep": {str(c): tfl(timed(K.opts(sched=K.SCHED_FIXED, fixed_comm_ctas=c, link_gbs=LINK_GBS)))
                            for c in (1, 2, 3)},
            "unfused": tfl(timed(K.opts(sched=K.SCHED_UNFUSED, link_gbs=LINK_GBS)))}
    link["fixed_best"] = max(link["fixed_sweep"].values())
    tf = flops / (band * 1e-3) / 1e12
    best = max(fixed, key=fixed.get)
    return {"workload": "rs_bf16_p8", "ms": band, "tflops": tf, "frac_of_peak": tf / peak, "link": link,
            "row_order_ms": row, "row_over_band": row / band,
            "fixed_split_best": {"tflops": fixed[best], "crew_per_rank": int(best), "sweep": fixed},
            "unfused": {"tflops": flops / (unf * 1e-3) / 1e12, "launches_per_step": 2},
            "self_single_sm_tiles_tflops": flops / (single * 1e-3) / 1e12,
            "vs_fixed_split_best": tf / fixed[best], "vs_unfused": tf / (flops / (unf * 1e-3) / 1e12)}


# Launch options of the --quick configurations (grid size, plain launch for
# profilers); the full run always uses the defaults.
QUICK_OPTS = {}


def bench_rs_quick(K, dev, steps, warmup, flush, stream):
    """The band-ordered GEMM + reduce-scatter alone (8 ranks, [8192, 3584] x [3584, 8192])."""
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    w = WORKLOADS["rs_bf16_p8"]
    inp = workload_inputs(w)
    P, m, k, n = w.P, w.m, w.k, w.n
    xs = [x.to(dev) for x in inp["x"]]
    ws_ = [x.to(dev) for x in inp["w"]]
    del inp
    ys = [torch.empty(m // P, n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    o = K.opts(**QUICK_OPTS)
    wsb = K.workspace(K.OP_GEMM_RS, P, m, n, k, o=o, device=dev)
    f = lambda: K.gemm_rs(xs, ws_, ys, wsb, o, stream=stream)
    t = statistics.mean(time_kernel_steps(f, steps, warmup, flush, stream))
    K.check(wsb, "gemm_rs")
    return {"workload": "rs_bf16_p8", "ms": t, "tflops": w.flops() / (t * 1e-3) / 1e12}


# Algorithmic HBM bytes of one MoE forward step (2048 tokens, hidden 4096,
# 128 experts top-8, inter 1536, bf16): every expert weight read once
# (128 x 3 x 4096 x 1536 x 2 = 4.83 GB), router weights, token reads and
# writes of the dispatch (read x rows, write received rows), the grouped GEMMs'
# reads of received rows, h writes and reads, y writes, push reads and writes,
# fold reads of the slots and the output write.
def moe_algorithmic_bytes(T, H, E, K, I):
    rows = T * K
    weights = E * 3 * H * I * 2 + H * E * 2
    dispatch = 2 * rows * H * 2
    gemm_in = rows * H * 2 + rows * I * 2
    h_out = rows * I * 2
    y_out = rows * H * 2
    push = 2 * rows * H * 2
    fold = rows * H * 2 + T * H * 2
    router_in = T * H * 2
    return weights + dispatch + gemm_in + h_out + y_out + push + fold + router_in


# MXFP8 layer: weights, tokens and h in E4M3 with one E8M0 byte per 32
# (router, expert outputs, slots and the fold stay bf16); adds the in-launch
# quantisation of the tokens (read bf16, write E4M3 + scales).
def moe_algorithmic_bytes_mxfp8(T, H, E, K, I):
    rows = T * K
    f8 = lambda n: n + n // 32  # E4M3 bytes plus their scales
    weights = f8(E * 3 * H * I) + H * E * 2
    quant = T * H * 2 + f8(T * H)
    dispatch = 2 * f8(rows * H)
    gemm_in = f8(rows * H) + f8(rows * I)
    h_out = f8(rows * I)
    y_out = rows * H * 2
    push = 2 * rows * H * 2
    fold = rows * H * 2 + T * H * 2
    router_in = T * H * 2
    return weights + quant + dispatch + gemm_in + h_out + y_out + push + fold + router_in


def _quant_experts_gpu(K, w, P, dev, stream):
    """E4M3 codes per rank and the experts' tiled scales one after the other."""
    import torch
    E, Kd, N = w.shape
    codes, scales = [], []
    nb = K.mxfp8_scale_bytes(Kd, N, False)
    for q in range(P):
        c = torch.empty(E // P, Kd, N, dtype=torch.uint8, device=dev)
        s = torch.empty((E // P) * nb, dtype=torch.uint8, device=dev)
        for j in range(E // P):
            K.mxfp8_quantize(w[q * (E // P) + j].to(dev), c[j], s[j * nb:(j + 1) * nb], False, stream=stream)
        codes.append(c)
        scales.append(s)
    return codes, scales


# Algorithmic HBM bytes of one MoE backward step (bf16): every expert weight
# read once and every weight gradient written once (2 x 4.83 GB at the
# benchmark shapes), plus the token-side and expert-side activations each
# read or written once: dout and the saved per-slot outputs, dy, g / u and
# dg / du, h and x for the weight gradients, dx of the expert rows, the slot
# push and fold, the router part.
def moe_bwd_algorithmic_bytes(T, H, E, K, I):
    rows = T * K
    w = E * 3 * H * I * 2
    token = T * H * 2 + rows * H * 2 + rows * H * 2 + rows * 4          # dout, y slots, dy, dgate
    dh = rows * H * 2 + 2 * rows * I * 2 + 2 * rows * I * 2             # dy, g/u, dg/du
    dgu = 2 * rows * I * 2 + rows * H * 2                               # dg/du, dx rows
    wgrad_in = rows * I * 2 + rows * H * 2 + rows * H * 2 + 2 * rows * I * 2  # h, dy, x, dg/du
    push_fold = 2 * rows * H * 2 + rows * H * 2 + T * H * 4 + T * H * 2
    router = T * E * 4 + T * E * 2 + H * E * 2 + T * H * 4 + T * H * 2 + H * E * 4
    return 2 * w + token + dh + dgu + wgrad_in + push_fold + router


def bench_moe_bwd(K, dev, steps, warmup, flush, stream, hbm_peak, tensor_peak, experts=0, unfused=False):
    """MoE layer backward (2048 tokens, hidden 4096, 128 experts top-8, 8 EP
    ranks, inter 1536) in one launch; the forward runs once untimed to fill
    the saved context."""
    import dataclasses
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    w = WORKLOADS["moe_fwd_p8"]
    if experts:  # a smaller expert count for profiler captures
        w = dataclasses.replace(w, E=experts, name=f"moe_fwd_p8_e{experts}")
    inp = workload_inputs(w)
    P, T, H, E, Kt, I = w.P, w.T, w.H, w.E, w.topk, w.I
    xs = [t.to(dev) for t in torch.chunk(inp["x"], P, 0)]
    wr = inp["w_router"].to(dev)
    wg = [t.to(dev) for t in _split_experts(inp["w_gate"], P)]
    wu = [t.to(dev) for t in _split_experts(inp["w_up"], P)]
    wd = [t.to(dev) for t in _split_experts(inp["w_down"], P)]
    del inp
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    idx = torch.empty(T, Kt, dtype=torch.int32, device=dev)
    gate = torch.empty(T, Kt, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    pos = torch.empty(T, Kt, dtype=torch.int32, device=dev)
    fws = K.moe_workspace(P, T, H, E, Kt, I, device=dev)
    K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, counts, pos, fws, Kt, stream=stream)
    K.check(fws, "moe_fwd")
    g = torch.Generator(device="cpu").manual_seed(11)
    dys = [t.to(dev) for t in torch.chunk(torch.randn(T, H, generator=g).to(torch.bfloat16), P, 0)]
    dxs = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    dwr = torch.empty(H, E, dtype=torch.float32, device=dev)
    dwg = [torch.empty_like(t) for t in wg]
    dwu = [torch.empty_like(t) for t in wu]
    dwd = [torch.empty_like(t) for t in wd]
    bws = K.moe_bwd_workspace(P, T, H, E, Kt, I, device=dev)
    f = lambda: K.moe_bwd(xs, wr, wg, wu, wd, idx, gate, fws, dys, dxs, dwr, dwg, dwu, dwd, bws, stream=stream)
    f()
    K.check(bws, "moe_bwd")
    t = statistics.mean(time_kernel_steps(f, steps, warmup, flush, stream))
    K.check(bws, "moe_bwd")
    byt = moe_bwd_algorithmic_bytes(T, H, E, Kt, I)
    flops = 12.0 * T * Kt * H * I + 4.0 * T * E * H
    gbs = byt / (t * 1e-3) / 1e9
    r = {"workload": w.name.replace("moe_fwd", "moe_bwd"), "ms": t, "tokens_per_s": T / (t * 1e-3),
         "tflops": flops / (t * 1e-3) / 1e12, "frac_of_tensor_peak": flops / (t * 1e-3) / 1e12 / tensor_peak,
         "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                      "bytes_per_launch": byt},
         "launches_per_step": 1}
    if unfused:  # head | DH | DWD | DGU | DWGU | DWR | push + fold, one launch each
        ou = K.opts(sched=K.SCHED_UNFUSED)
        fu = lambda: K.moe_bwd(xs, wr, wg, wu, wd, idx, gate, fws, dys, dxs, dwr, dwg, dwu, dwd, bws, ou,
                               stream=stream)
        fu()
        K.check(bws, "moe_bwd unfused")
        tu = statistics.mean(time_kernel_steps(fu, steps, warmup, flush, stream))
        K.check(bws, "moe_bwd unfused")
        r["unfused"] = {"ms": tu, "tokens_per_s": T / (tu * 1e-3), "launches_per_step": 7}
        r["vs_unfused"] = tu / t
    return r


def bench_moe(K, dev, steps, warmup, flush, stream, hbm_peak, tensor_peak, experts=0, mx=False, unfused=False):
    import dataclasses
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    w = WORKLOADS["moe_fwd_p8"]
    if experts:  # a smaller expert count for profiler captures (same kernel, fewer weights)
        w = dataclasses.replace(w, E=experts, name=f"moe_fwd_p8_e{experts}")
    if mx:
        w = dataclasses.replace(w, name=w.name.replace("moe_fwd", "moe_fwd_mxfp8"), dtype="mxfp8")
    inp = workload_inputs(w)
    P, T, H, E, Kt, I = w.P, w.T, w.H, w.E, w.topk, w.I
    xs = [t.to(dev) for t in torch.chunk(inp["x"], P, 0)]
    wr = inp["w_router"].to(dev)
    kw = {}
    if mx:
        (wg, sg), (wu, su), (wd, sd) = (_quant_experts_gpu(K, inp[n], P, dev, stream)
                                        for n in ("w_gate", "w_up", "w_down"))
        kw = {"dtype": K.MXFP8_E4M3, "w_gate_scales": sg, "w_up_scales": su, "w_down_scales": sd}
    else:
        wg = [t.to(dev) for t in _split_experts(inp["w_gate"], P)]
        wu = [t.to(dev) for t in _split_experts(inp["w_up"], P)]
        wd = [t.to(dev) for t in _split_experts(inp["w_down"], P)]
    del inp
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    idx = torch.empty(T, Kt, dtype=torch.int32, device=dev)
    gate = torch.empty(T, Kt, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    pos = torch.empty(T, Kt, dtype=torch.int32, device=dev)
    wsb = K.moe_workspace(P, T, H, E, Kt, I, device=dev, dtype=K.MXFP8_E4M3 if mx else K.BF16)
    o = K.opts(**QUICK_OPTS)
    f = lambda: K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, counts, pos, wsb, Kt, o, stream=stream, **kw)
    f()
    K.check(wsb, "moe_fwd")
    t = statistics.mean(time_kernel_steps(f, steps, warmup, flush, stream))
    K.check(wsb, "moe_fwd")
    byt = (moe_algorithmic_bytes_mxfp8 if mx else moe_algorithmic_bytes)(T, H, E, Kt, I)
    gbs = byt / (t * 1e-3) / 1e9
    r = {"workload": w.name, "ms": t, "tokens_per_s": T / (t * 1e-3),
         "tflops": w.flops() / (t * 1e-3) / 1e12, "frac_of_tensor_peak": w.flops() / (t * 1e-3) / 1e12 / tensor_peak,
         "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm_peak, "unit": "GB/s", "frac": gbs / hbm_peak,
                      "bytes_per_launch": byt},
         "launches_per_step": 1}
    if unfused:  # the same kernel once per phase: route | dispatch | gate/up tiles | down tiles | push + fold
        ou = K.opts(sched=K.SCHED_UNFUSED)
        fu = lambda: K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, counts, pos, wsb, Kt, ou, stream=stream, **kw)
        fu()
        K.check(wsb, "moe_fwd unfused")
        tu = statistics.mean(time_kernel_steps(fu, steps, warmup, flush, stream))
        K.check(wsb, "moe_fwd unfused")
        r["unfused"] = {"ms": tu, "tokens_per_s": T / (tu * 1e-3), "launches_per_step": 5}
        r["vs_unfused"] = tu / t
    return r


def bench_mxfp8(K, dev, steps, warmup, flush, stream, bf16_peak, baselines=True):
    """All-gather + GEMM on MXFP8 operands (E4M3 + E8M0 per 32 K), the shapes
    of the 8-rank bf16 workload; quantisation on the GPU before timing (the
    kernel's inputs are the quantised bytes).  Peak: the measured bf16 dense
    peak x 2 (the nominal fp8 : bf16 dense ratio, 4.5 : 2.25 PFLOP/s)."""
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    w = WORKLOADS["ag_mxfp8_p8"]
    inp = workload_inputs(w)
    P, m, k, n = w.P, w.m, w.k, w.n

    def quant(x, along):
        r, c = x.shape
        q = torch.empty(r, c, dtype=torch.uint8, device=dev)
        sc = torch.empty(K.mxfp8_scale_bytes(r, c, along), dtype=torch.uint8, device=dev)
        K.mxfp8_quantize(x.to(dev), q, sc, along, stream=stream)
        return q, sc

    qs, ss = zip(*[quant(x, True) for x in inp["x"]])
    qw, sw = quant(inp["w"], False)
    del inp
    xg = torch.empty(P * m, k, dtype=torch.uint8, device=dev)
    y = torch.empty(P * m, n, dtype=torch.bfloat16, device=dev)
    flops = w.flops()
    peak = 2.0 * bf16_peak

    def timed(o):
        wsb = K.workspace(K.OP_AG_GEMM, P, m, n, k, dtype=K.MXFP8_E4M3, o=o, device=dev)
        f = lambda: K.ag_gemm(list(qs), qw, xg, y, wsb, o, dtype=K.MXFP8_E4M3, x_scales=list(ss), w_scales=sw,
                              stream=stream)
        f()
        K.check(wsb, "ag_gemm mxfp8")
        t = statistics.mean(time_kernel_steps(f, steps, warmup, flush, stream))
        K.check(wsb, "ag_gemm mxfp8")
        return flops / (t * 1e-3) / 1e12, t

    tf, ms = timed(K.opts(**(QUICK_OPTS if not baselines else {})))
    if not baselines:
        return {"workload": "ag_mxfp8_p8", "ms": ms, "tflops": tf, "peak": peak, "frac_of_peak": tf / peak}
    fx, _ = timed(K.opts(sched=K.SCHED_FIXED))
    un, _ = timed(K.opts(sched=K.SCHED_UNFUSED))
    sms = K.num_sms()
    link = {"self": timed(K.opts(link_gbs=LINK_GBS))[0],
            "fixed_sweep": {str(c): timed(K.opts(sched=K.SCHED_FIXED, fixed_comm_ctas=c, link_gbs=LINK_GBS))[0]
                            for c in sorted({max(1, sms // 8), max(1, sms // 4), max(1, 3 * sms // 8)})},
            "unfused": timed(K.opts(sched=K.SCHED_UNFUSED, link_gbs=LINK_GBS))[0]}
    link["fixed_best"] = max(link["fixed_sweep"].values())
    return {"workload": "ag_mxfp8_p8", "ms": ms, "tflops": tf, "peak": peak,
            "peak_source": "measured bf16 dense x 2 (nominal fp8/bf16 ratio)", "frac_of_peak": tf / peak,
            "fixed_split_tflops": fx, "unfused_tflops": un, "vs_fixed_split": tf / fx, "vs_unfused": tf / un,
            "link": link}


def bench_rs_mxfp8(K, dev, steps, warmup, flush, stream, bf16_peak, baselines=True):
    """GEMM + reduce-scatter on MXFP8 operands, the shapes of the 8-rank bf16
    workload (X_r [8192, 3584], W_r [3584, 8192]); band order, with the
    row-order ablation and the unfused baseline.  Peak as for the MXFP8
    all-gather: the measured bf16 dense peak x 2."""
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    w = WORKLOADS["rs_mxfp8_p8"]
    inp = workload_inputs(w)
    P, m, k, n = w.P, w.m, w.k, w.n

    def quant(x, along):
        r, c = x.shape
        q = torch.empty(r, c, dtype=torch.uint8, device=dev)
        sc = torch.empty(K.mxfp8_scale_bytes(r, c, along), dtype=torch.uint8, device=dev)
        K.mxfp8_quantize(x.to(dev), q, sc, along, stream=stream)
        return q, sc

    qx, sx = zip(*[quant(x, True) for x in inp["x"]])
    qw, sw = zip(*[quant(x, False) for x in inp["w"]])
    del inp
    ys = [torch.empty(m // P, n, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    flops = w.flops()
    peak = 2.0 * bf16_peak

    def timed(o):
        wsb = K.workspace(K.OP_GEMM_RS, P, m, n, k, dtype=K.MXFP8_E4M3, o=o, device=dev)
        f = lambda: K.gemm_rs(list(qx), list(qw), ys, wsb, o, stream=stream, dtype=K.MXFP8_E4M3,
                              x_scales=list(sx), w_scales=list(sw))
        f()
        K.check(wsb, "gemm_rs mxfp8")
        t = statistics.mean(time_kernel_steps(f, steps, warmup, flush, stream))
        K.check(wsb, "gemm_rs mxfp8")
        return flops / (t * 1e-3) / 1e12, t

    tf, ms = timed(K.opts(**(QUICK_OPTS if not baselines else {})))
    r = {"workload": "rs_mxfp8_p8", "ms": ms, "tflops": tf, "peak": peak, "frac_of_peak": tf / peak}
    if not baselines:
        return r
    row, row_ms = timed(K.opts(order=K.ORDER_ROW))
    fx, _ = timed(K.opts(sched=K.SCHED_FIXED))
    un, _ = timed(K.opts(sched=K.SCHED_UNFUSED))
    link = {"self": timed(K.opts(link_gbs=LINK_GBS))[0],
            "fixed_sweep": {str(c): timed(K.opts(sched=K.SCHED_FIXED, fixed_comm_ctas=c, link_gbs=LINK_GBS))[0]
                            for c in (1, 2, 3)},
            "unfused": timed(K.opts(sched=K.SCHED_UNFUSED, link_gbs=LINK_GBS))[0]}
    link["fixed_best"] = max(link["fixed_sweep"].values())
    r["link"] = link
    r.update({"peak_source": "measured bf16 dense x 2 (nominal fp8/bf16 ratio)", "row_order_ms": row_ms,
              "row_over_band": row_ms / ms, "fixed_split_tflops": fx, "unfused_tflops": un,
              "vs_fixed_split": tf / fx, "vs_unfused": tf / un})
    return r


# One GPU's per-direction NVLink 5 bandwidth: the emulated link of the
# attention-shape measurements (kosmos_opts.link_gbs).
LINK_GBS = 900


def bench_attn(K, dev, steps, warmup, flush, stream, peak):
    """Attention block of the layer: QKV all-gather + GEMM (8 ranks, X_r
    1024x8192, W 8192x1280) and output-projection GEMM + reduce-scatter
    (X_r 8192x1024, W_r 1024x8192), each with the copies free (one HBM) and
    through an emulated 900 GB/s link; self-scheduling, fixed crew and
    unfused."""
    import torch
    from kosmos_inputs import WORKLOADS, workload_inputs
    out = {"link_gbs": LINK_GBS}
    w = WORKLOADS["ag_qkv_p8"]
    inp = workload_inputs(w)
    P, m, k, n = w.P, w.m, w.k, w.n
    xs = [x.to(dev) for x in inp["x"]]
    W = inp["w"].to(dev)
    del inp
    xg = torch.empty(P * m, k, dtype=torch.bfloat16, device=dev)
    y = torch.empty(P * m, n, dtype=torch.bfloat16, device=dev)

    def mk_ag(**kw):
        o = K.opts(**kw)
        wsb = K.workspace(K.OP_AG_GEMM, P, m, n, k, o=o, device=dev)
        return (lambda: K.ag_gemm(xs, W, xg, y, wsb, o, stream=stream)), wsb

    def t_ag(**kw):
        f, wsb = mk_ag(**kw)
        f()
        K.check(wsb, "ag_gemm")
        t = statistics.mean(time_kernel_steps(f, steps, warmup, flush, stream))
        K.check(wsb, "ag_gemm")
        return w.flops() / (t * 1e-3) / 1e12

    res = {}
    for cap in (0, LINK_GBS):
        tag = "link" if cap else "free"
        fixed = {str(c): t_ag(sched=K.SCHED_FIXED, fixed_comm_ctas=c, link_gbs=cap) for c in (20, 40, 60)}
        res[tag] = {"self": t_ag(link_gbs=cap), "fixed_best": max(fixed.values()), "fixed_sweep": fixed,
                    "unfused": t_ag(sched=K.SCHED_UNFUSED, link_gbs=cap)}
        crew = int(max(fixed, key=fixed.get))
        (fa, wa), (fb, wb) = mk_ag(link_gbs=cap), mk_ag(sched=K.SCHED_FIXED, fixed_comm_ctas=crew, link_gbs=cap)
        ma, mb = paired_medians(fa, fb, flush, stream)
        K.check(wa, "ag_gemm paired")
        K.check(wb, "ag_gemm fixed paired")
        res[tag]["paired_self_fixed"] = {"crew": crew, "self": w.flops() / (ma * 1e-3) / 1e12,
                                         "fixed": w.flops() / (mb * 1e-3) / 1e12, "ratio": mb / ma}
    out["ag_qkv_p8"] = {"tflops": res, "frac_of_peak_free": res["free"]["self"] / peak,
                        "link_bound_us": (P - 1) * m * k * 2 / LINK_GBS / 1e3,
                        "gemm_at_peak_us": w.flops() / (peak * 1e12) * 1e6}
    del xs, W, xg, y
    torch.cuda.empty_cache()
    w = WORKLOADS["rs_oproj_p8"]
    inp = workload_inputs(w)
    P, m, k, n = w.P, w.m, w.k, w.n
    xs = [x.to(dev) for x in inp["x"]]
    ws_ = [x.to(dev) for x in inp["w"]]
    del inp
    ys = [torch.empty(m // P, n, dtype=torch.bfloat16, device=dev) for _ in range(P)]

    def t_rs(**kw):
        o = K.opts(**kw)
        wsb = K.workspace(K.OP_GEMM_RS, P, m, n, k, o=o, device=dev)
        f = lambda: K.gemm_rs(xs, ws_, ys, wsb, o, stream=stream)
        f()
        K.check(wsb, "gemm_rs")
        t = statistics.mean(time_kernel_steps(f, steps, warmup, flush, stream))
        K.check(wsb, "gemm_rs")
        return w.flops() / (t * 1e-3) / 1e12

    res = {}
    for cap in (0, LINK_GBS):
        tag = "link" if cap else "free"
        fixed = {str(c): t_rs(sched=K.SCHED_FIXED, fixed_comm_ctas=c, link_gbs=cap) for c in (1, 2, 4)}
        res[tag] = {"band": t_rs(link_gbs=cap), "row": t_rs(order=K.ORDER_ROW, link_gbs=cap),
                    "fixed_best": max(fixed.values()), "fixed_sweep_per_rank": fixed,
                    "unfused": t_rs(sched=K.SCHED_UNFUSED, link_gbs=cap)}
    out["rs_oproj_p8"] = {"tflops": res, "frac_of_peak_free": res["free"]["band"] / peak,
                          "link_bound_us": (P - 1) * m * n * 2 / LINK_GBS / 1e3,
                          "gemm_at_peak_us": w.flops() / (peak * 1e12) * 1e6}
    return out


def workload_config(w):
    """The `config` of both arms' lines: the workload and how the timed region
    treats L2 (identical dicts, so that the two arms compare)."""
    return {"workload": w.name, "P": w.P, "m_per_shard": w.m, "k": w.k, "n": w.n,
            "l2": "flushed (256 MiB write) before every GPU step"}


def run_reference(args):
    """The reference arm: the oracle (plain fp64 C, OpenMP) timed on the host
    cores.  Every step computes a bounded sample of the workload's output rows
    (the same sample in every step); ms_per_step is the measured time of that
    sample, and value is its TFLOP/s."""
    import numpy as np
    import oracle
    from kosmos_inputs import WORKLOADS, bf16_bits, workload_inputs
    ws, rank, local = dist_env()
    if ws > 1 and rank != 0:
        return 0
    w = WORKLOADS[WORKLOAD]
    inp = workload_inputs(w)
    oracle.build()
    xs = [bf16_bits(x) for x in inp["x"]]
    wb = bf16_bits(inp["w"])
    P, m, k, n = w.P, w.m, w.k, w.n
    # size the sample so that warm-up and timed steps take about 90 s in all
    probe = np.arange(0, P * m, (P * m) // 32, dtype=np.int64)[:32]
    t0 = time.perf_counter()
    oracle.ag_gemm(xs, wb, rows=probe)
    per_row = (time.perf_counter() - t0) / len(probe)
    budget_s = 90.0 / max(1, args.steps + args.warmup)
    nrows = int(min(P * m, max(16, budget_s / max(per_row, 1e-6))))
    rows = np.linspace(0, P * m - 1, nrows).astype(np.int64)
    for _ in range(args.warmup):
        oracle.ag_gemm(xs, wb, rows=rows)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.ag_gemm(xs, wb, rows=rows)
        times.append(time.perf_counter() - t0)
    step_s = statistics.mean(times)
    v = 2.0 * nrows * k * n / step_s / 1e12
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "TFLOP/s", "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": step_s * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic (seeded N(0,var) bf16)", "config": workload_config(w),
            "cpu_baseline": {"value": v, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                             "sample": f"{nrows} of {P * m} output rows of Y = concat(X_r) W per step (fp64); "
                                       f"ms_per_step is the time of that sample"},
            "e2e": {"value": v, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def sig(x, n=4):
    """x rounded to n significant digits (keeps the JSON line short)."""
    return float(f"{x:.{n}g}") if isinstance(x, float) else x


def compact_baselines(base):
    return {"fixed_split_best": {"tflops": sig(base["fixed_split_best"]["tflops"]),
                                 "crew": base["fixed_split_best"]["crew"]},
            "fixed_sweep": {c: sig(v) for c, v in base["fixed_split_best"]["sweep"].items()},
            "unfused": sig(base["unfused"]["tflops"]),
            "one_sm_tiles": sig(base["self_single_sm_tiles"]["tflops"]),
            "n_comm0_sweep": {c: sig(v) for c, v in base["self_n_comm0_sweep"].items()},
            "link_self_fixedbest_unfused": [sig(base["link"]["self"]), sig(base["link"]["fixed_best"]),
                                            sig(base["link"]["unfused"])],
            "paired_self_over_fixed": {"free": sig(base["paired_self_fixed"]["ratio"], 3),
                                       "link": sig(base["link"]["paired_self_fixed"]["ratio"], 3)}}


def compact_also(also):
    """Every other workload's key figures, short enough that the whole result
    line survives a log tail (TFLOP/s unless named otherwise; frac = fraction
    of the measured peak of the kernel's bound)."""
    out = {}
    r = also.get("gemm_rs")
    if r:
        out["rs_bf16_p8"] = {"tflops": sig(r["tflops"]), "frac": sig(r["frac_of_peak"], 3), "ms": sig(r["ms"]),
                             "row_over_band": sig(r["row_over_band"], 3),
                             "fixed_best": sig(r["fixed_split_best"]["tflops"]),
                             "unfused": sig(r["unfused"]["tflops"]),
                             "one_sm_tiles": sig(r["self_single_sm_tiles_tflops"]),
                             "link_self_fixedbest_unfused": [sig(r["link"]["self"]), sig(r["link"]["fixed_best"]),
                                                             sig(r["link"]["unfused"])]}
    r = also.get("ag_mxfp8")
    if r:
        out["ag_mxfp8_p8"] = {"tflops": sig(r["tflops"]), "frac": sig(r["frac_of_peak"], 3), "ms": sig(r["ms"]),
                              "fixed_best": sig(r["fixed_split_tflops"]), "unfused": sig(r["unfused_tflops"])}
        if "link" in r:
            out["ag_mxfp8_p8"]["link_self_fixedbest_unfused"] = [sig(r["link"]["self"]), sig(r["link"]["fixed_best"]),
                                                                 sig(r["link"]["unfused"])]
    r = also.get("rs_mxfp8")
    if r:
        out["rs_mxfp8_p8"] = {"tflops": sig(r["tflops"]), "frac": sig(r["frac_of_peak"], 3), "ms": sig(r["ms"]),
                              "row_over_band": sig(r.get("row_over_band"), 3),
                              "fixed_best": sig(r.get("fixed_split_tflops")), "unfused": sig(r.get("unfused_tflops"))}
        if "link" in r:
            out["rs_mxfp8_p8"]["link_self_fixedbest_unfused"] = [sig(r["link"]["self"]), sig(r["link"]["fixed_best"]),
                                                                 sig(r["link"]["unfused"])]
    for key, name in (("moe_fwd", "moe_fwd_p8"), ("moe_fwd_mxfp8", "moe_fwd_mxfp8_p8"), ("moe_bwd", "moe_bwd_p8")):
        r = also.get(key)
        if r:
            d = {"ms": sig(r["ms"]), "tok_s": sig(r["tokens_per_s"]), "tflops": sig(r["tflops"]),
                 "hbm_frac": sig(r["roofline"]["frac"], 3), "gbs": sig(r["roofline"]["achieved"])}
            if "unfused" in r:
                d["unfused_ms"] = sig(r["unfused"]["ms"])
                d["unfused_launches"] = r["unfused"]["launches_per_step"]
            out[name] = d
    r = also.get("attention")
    if r:
        a = {}
        for wl, k in (("ag_qkv_p8", "self"), ("rs_oproj_p8", "band")):
            for tag in ("free", "link"):
                t = r[wl]["tflops"][tag]
                a[f"{wl}_{tag}"] = [sig(t[k]), sig(t["fixed_best"]), sig(t["unfused"])]
        out["attention_self_fixedbest_unfused"] = a
        out["qkv_paired_self_over_fixed"] = {tag: sig(r["ag_qkv_p8"]["tflops"][tag]["paired_self_fixed"]["ratio"], 3)
                                             for tag in ("free", "link")}
    return out


def run_quick_other(args):
    """Quick mode for the other workloads: one configuration, timed region only."""
    import torch
    import comm_persistent_gemm_gb300 as K
    K.build()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    flush = lambda: flush_buf.fill_(1)
    peaks, _ = load_peaks()
    if args.workload == "rs":
        r = bench_rs_quick(K, dev, args.steps, args.warmup, flush, stream)
    elif args.workload == "moe":
        r = bench_moe(K, dev, args.steps, args.warmup, flush, stream, peaks["hbm_gbs"], peaks["bf16_tflops"],
                      experts=args.experts)
    elif args.workload == "moe_bwd":
        r = bench_moe_bwd(K, dev, args.steps, args.warmup, flush, stream, peaks["hbm_gbs"], peaks["bf16_tflops"],
                          experts=args.experts)
    elif args.workload == "attn":
        r = bench_attn(K, dev, args.steps, args.warmup, flush, stream, peaks["bf16_tflops"])
    elif args.workload == "moe_mxfp8":
        r = bench_moe(K, dev, args.steps, args.warmup, flush, stream, peaks["hbm_gbs"], 2 * peaks["bf16_tflops"],
                      experts=args.experts, mx=True)
    elif args.workload == "rs_mxfp8":
        r = bench_rs_mxfp8(K, dev, args.steps, args.warmup, flush, stream, peaks["bf16_tflops"], baselines=False)
    else:
        r = bench_mxfp8(K, dev, args.steps, args.warmup, flush, stream, peaks["bf16_tflops"], baselines=False)
    print(json.dumps({"quick": True, "workload": args.workload, **r}))
    return 0


def run_kosmos(args):
    import torch
    if args.quick and args.workload != "ag":
        return run_quick_other(args)
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    import comm_persistent_gemm_gb300 as K
    from kosmos_inputs import WORKLOADS, workload_inputs
    K.build()
    w = WORKLOADS[WORKLOAD]
    inp = workload_inputs(w)
    P, m, k, n = w.P, w.m, w.k, w.n
    xs = [x.to(dev) for x in inp["x"]]
    W = inp["w"].to(dev)
    xg = torch.empty(P * m, k, dtype=torch.bfloat16, device=dev)
    y = torch.empty(P * m, n, dtype=torch.bfloat16, device=dev)
    flush_buf = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def flush():
        flush_buf.fill_(1)

    def make(o):
        wsb = K.workspace(K.OP_AG_GEMM, P, m, n, k, o=o, device=dev)
        return (lambda: K.ag_gemm(xs, W, xg, y, wsb, o, stream=stream)), wsb

    flops = w.flops()
    sms = K.num_sms()
    peaks, src = load_peaks()
    peak = peaks["bf16_tflops"]
    o_self = K.opts(**QUICK_OPTS) if args.quick else K.opts()
    f_self, ws_self = make(o_self)
    # warm up + correctness gate of the timed configuration
    f_self()
    K.check(ws_self, "ag_gemm")

    # ---- timed region (the method), barrier + sync on both sides, max over ranks
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    with ClockSampler(dev) as clk:
        times = time_kernel_steps(f_self, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    K.check(ws_self, "ag_gemm")
    step_ms = dist_max(statistics.mean(times), dev)
    value = whole_job_rate(flops, step_ms, world) / 1e12
    clocks = clk.summary()
    if args.quick:
        if rank == 0:
            print(json.dumps({"quick": True, "metric": METRIC, "value": value, "unit": "TFLOP/s",
                              "ms_per_step": step_ms, "steps": args.steps, "warmup": args.warmup,
                              "config": {"workload": WORKLOAD}, "gpu_launches": args.steps}))
        return 0

    # ---- baselines on the same inputs (not the headline)
    base = {}
    fixed = {}
    for crew in sorted({max(1, sms // 16), max(1, sms // 8), max(1, sms // P), max(1, sms // 4)}):
        f, wsb = make(K.opts(sched=K.SCHED_FIXED, fixed_comm_ctas=crew))
        tt = time_kernel_steps(f, max(3, args.steps // 2), 2, flush, stream)
        K.check(wsb, "ag_gemm fixed")
        fixed[str(crew)] = flops / (statistics.mean(tt) * 1e-3) / 1e12
    best_crew = max(fixed, key=fixed.get)
    base["fixed_split_best"] = {"tflops": fixed[best_crew], "crew": int(best_crew), "sweep": fixed}
    f_fix, ws_fix = make(K.opts(sched=K.SCHED_FIXED, fixed_comm_ctas=int(best_crew)))
    ma, mb = paired_medians(f_self, f_fix, flush, stream)
    K.check(ws_self, "ag_gemm paired")
    K.check(ws_fix, "ag_gemm fixed paired")
    base["paired_self_fixed"] = {"crew": int(best_crew), "self": flops / (ma * 1e-3) / 1e12,
                                 "fixed": flops / (mb * 1e-3) / 1e12, "ratio": mb / ma}
    f, wsb = make(K.opts(sched=K.SCHED_UNFUSED))
    tt = time_kernel_steps(f, max(3, args.steps // 2), 2, flush, stream)
    K.check(wsb, "ag_gemm unfused")
    base["unfused"] = {"tflops": flops / (statistics.mean(tt) * 1e-3) / 1e12,
                       "launches_per_step": 2}
    f, wsb = make(K.opts(cta_pair=0))
    tt = time_kernel_steps(f, max(3, args.steps // 2), 2, flush, stream)
    K.check(wsb, "ag_gemm single-SM tiles")
    base["self_single_sm_tiles"] = {"tflops": flops / (statistics.mean(tt) * 1e-3) / 1e12,
                                    "note": "same schedule, 128x256 tiles on one SM each (tcgen05 cta_group::1)"}
    sweep = {}
    for nc in sorted({max(1, sms // 16), max(1, sms // 8), max(1, sms // 4)}):
        f, wsb = make(K.opts(n_comm0=nc))
        tt = time_kernel_steps(f, max(3, args.steps // 2), 2, flush, stream)
        K.check(wsb, "ag_gemm n_comm0")
        sweep[str(nc)] = flops / (statistics.mean(tt) * 1e-3) / 1e12
    base["self_n_comm0_sweep"] = sweep
    # the same comparison with every remote piece crossing an emulated link
    # (one GPU's per-direction NVLink 5 bandwidth): role dynamics of a slow link
    link = {}
    f, wsb = make(K.opts(link_gbs=LINK_GBS))
    tt = time_kernel_steps(f, max(3, args.steps // 2), 2, flush, stream)
    K.check(wsb, "ag_gemm link")
    link["self"] = flops / (statistics.mean(tt) * 1e-3) / 1e12
    lfixed = {}
    for crew in sorted({max(1, sms // 8), max(1, sms // 4), max(1, 3 * sms // 8)}):
        f, wsb = make(K.opts(sched=K.SCHED_FIXED, fixed_comm_ctas=crew, link_gbs=LINK_GBS))
        tt = time_kernel_steps(f, max(3, args.steps // 2), 2, flush, stream)
        K.check(wsb, "ag_gemm link fixed")
        lfixed[str(crew)] = flops / (statistics.mean(tt) * 1e-3) / 1e12
    link["fixed_sweep"] = lfixed
    link["fixed_best"] = max(lfixed.values())
    lcrew = int(max(lfixed, key=lfixed.get))
    f_ls, ws_ls = make(K.opts(link_gbs=LINK_GBS))
    f_lf, ws_lf = make(K.opts(sched=K.SCHED_FIXED, fixed_comm_ctas=lcrew, link_gbs=LINK_GBS))
    ma, mb = paired_medians(f_ls, f_lf, flush, stream)
    K.check(ws_ls, "ag_gemm link paired")
    K.check(ws_lf, "ag_gemm link fixed paired")
    link["paired_self_fixed"] = {"crew": lcrew, "self": flops / (ma * 1e-3) / 1e12,
                                 "fixed": flops / (mb * 1e-3) / 1e12, "ratio": mb / ma}
    f, wsb = make(K.opts(sched=K.SCHED_UNFUSED, link_gbs=LINK_GBS))
    tt = time_kernel_steps(f, max(3, args.steps // 2), 2, flush, stream)
    K.check(wsb, "ag_gemm link unfused")
    link["unfused"] = flops / (statistics.mean(tt) * 1e-3) / 1e12
    base["link"] = link

    # ---- e2e through the C ABI with host buffers (pinned), copies inside the timed region
    hx = [x.pin_memory() for x in inp["x"]]
    hy = torch.empty(P * m, n, dtype=torch.bfloat16).pin_memory()
    h2d = sum(x.numel() * 2 for x in hx)
    d2h = hy.numel() * 2

    # kosmos_ag_gemm_host: the shard copies (h2d stream) and output copies (d2h
    # stream) overlap the kernel through per-shard arrival words and output
    # tile counts; the timed stream waits for both copy streams every step
    h2d_s, d2h_s = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    o_host = K.opts()
    ws_host = K.workspace(K.OP_AG_GEMM, P, m, n, k, o=o_host, device=dev)

    def e2e_step():
        K.ag_gemm_host(hx, xs, W, xg, y, hy, ws_host, o_host, stream=stream, h2d_stream=h2d_s, d2h_stream=d2h_s)

    et = time_kernel_steps(e2e_step, args.steps, args.warmup, flush, stream)
    K.check(ws_host, "ag_gemm e2e")
    if not torch.equal(hy, y.cpu()):
        raise RuntimeError("e2e: host output differs from the device output")
    e2e_ms = dist_max(statistics.mean(et), dev)
    e2e = {"value": whole_job_rate(flops, e2e_ms, world) / 1e12, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h}


    achieved = flops / (step_ms * 1e-3) / 1e12
    traffic = TRAFFIC_CAPTURE["bytes"] if TRAFFIC_CAPTURE["src_sha"] == kernel_src_sha() else None
    roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
            "traffic": traffic, "peak_source": f"{src} bf16 dense (burst)", "kernel": "ag_gemm_pair_kernel",
            "flop_per_launch": flops}

    also = {}
    if not args.ag_only:
        also["gemm_rs"] = bench_rs(K, dev, max(3, args.steps // 2), 3, flush, stream, peak)
        torch.cuda.empty_cache()
        also["moe_fwd"] = bench_moe(K, dev, max(3, args.steps // 2), 3, flush, stream, peaks["hbm_gbs"], peak,
                                    unfused=True)
        torch.cuda.empty_cache()
        also["ag_mxfp8"] = bench_mxfp8(K, dev, max(3, args.steps // 2), 3, flush, stream, peak)
        torch.cuda.empty_cache()
        also["rs_mxfp8"] = bench_rs_mxfp8(K, dev, max(3, args.steps // 2), 3, flush, stream, peak)
        torch.cuda.empty_cache()
        also["moe_fwd_mxfp8"] = bench_moe(K, dev, max(3, args.steps // 2), 3, flush, stream, peaks["hbm_gbs"],
                                          2 * peak, mx=True, unfused=True)
        torch.cuda.empty_cache()
        also["attention"] = bench_attn(K, dev, max(3, args.steps // 2), 3, flush, stream, peak)
        torch.cuda.empty_cache()
        also["moe_bwd"] = bench_moe_bwd(K, dev, max(3, args.steps // 2), 3, flush, stream, peaks["hbm_gbs"], peak,
                                        unfused=True)
        torch.cuda.empty_cache()

    line = None
    if rank == 0:
        cpu = time_oracle_ag(inp) if world == 1 else None
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": step_ms, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,var) bf16)",
                "config": workload_config(w),
                "launch": {"sched": "self", "n_comm0": "ceil(S/P)", "sms": sms},
                "frac_of_peak": achieved / peak,
                "roofline": roof, "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks,
                "gpu_launches": args.steps, "baselines": compact_baselines(base),
                "vs_fixed_split_best": value / world / base["fixed_split_best"]["tflops"],
                "vs_unfused": value / world / base["unfused"]["tflops"], "also": compact_also(also)}
        if args.detail:
            with open(args.detail, "w") as fh:
                json.dump({**line, "baselines": base, "also": also}, fh, indent=1)
        print(json.dumps(line, separators=(",", ":")))
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="kosmos", choices=["kosmos", "reference"])
    ap.add_argument("--ag-only", action="store_true", help="skip the GEMM+RS and MoE measurements")
    ap.add_argument("--workload", default="ag", choices=["ag", "rs", "moe", "mxfp8", "rs_mxfp8", "moe_mxfp8", "attn", "moe_bwd"],
                    help="with --quick: which fused operator to time")
    ap.add_argument("--experts", type=int, default=0, help="with --quick --workload moe: expert count (0 = 128)")
    ap.add_argument("--num-ctas", type=int, default=0,
                    help="with --quick: persistent grid size (0 = one CTA per SM)")
    ap.add_argument("--plain-launch", action="store_true",
                    help="with --quick: launch without the cooperative attribute (for profilers)")
    ap.add_argument("--detail", default="", help="also write the full results (every sweep point) to this JSON file")
    ap.add_argument("--quick", action="store_true",
                    help="only the timed region of the fused kernel (no baselines, e2e or CPU oracle): "
                         "a short launch list for profilers")
    args = ap.parse_args()
    if args.quick:
        QUICK_OPTS.update({"num_ctas": args.num_ctas if args.num_ctas > 0 else None,
                           "plain_launch": 1 if args.plain_launch else None})
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_kosmos(args)


if __name__ == "__main__":
    sys.exit(main())
