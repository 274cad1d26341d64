"""Seeded synthetic inputs for the fused AG/RS-GEMM and MoE kernels.

This module is shared by the CUDA path's tests and benchmark and by the CPU
oracle's tests.  It holds the workload table (shapes, seeds, value
distributions) and draws random tensors; it contains none of the method's
arithmetic (no GEMM, no quantisation, no routing).

Generation recipe (the pages give only "~N(0, var)" and a seed):
  * one ``torch.Generator('cpu')`` seeded with the workload's seed;
  * AG and RS tensors are drawn in the order the workload lists them
    (AG: X_0..X_{P-1}, then W;  RS: X_0..X_{P-1}, then W_0..W_{P-1});
  * MoE tensors (X, W_router, then gate, up, down of each expert) each have
    their own generator seeded from the workload seed and the tensor's index,
    so the 384 expert matrices can be drawn in parallel;
  * each draw is ``randn(shape, float32) * sigma`` rounded once to bfloat16
    (round-to-nearest-even, torch's conversion).

Everything is returned as CPU torch tensors (bf16); ``bf16_bits`` gives the raw
uint16 view that the oracle consumes.
"""
from __future__ import annotations

import math
import os
from dataclasses import dataclass, field
from typing import Dict, List

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    """One synthetic workload.  Shapes follow the KOSMOS abstract's three fused
    ops (all-gather+GEMM, GEMM+reduce-scatter, one-launch expert layer)."""

    name: str
    op: str                 # "ag" | "rs" | "moe"
    seed: int
    P: int                  # emulated ranks
    m: int = 0              # AG: rows per shard; RS: rows of each X_r
    k: int = 0              # AG: K; RS: K per rank
    n: int = 0              # output columns
    dtype: str = "bf16"     # "bf16" | "mxfp8"
    var_x: float = 1.0
    var_w: float = 1.0
    # MoE only
    T: int = 0
    H: int = 0
    E: int = 0
    topk: int = 0
    I: int = 0
    note: str = ""

    def flops(self) -> float:
        if self.op == "ag":
            return 2.0 * self.P * self.m * self.k * self.n
        if self.op == "rs":
            return 2.0 * self.P * self.m * self.k * self.n
        if self.op == "moe":
            return 2.0 * self.T * self.H * self.E + 2.0 * self.T * self.topk * 3 * self.H * self.I
        raise ValueError(self.op)


# The five workloads.  Names say what they are; sizes are the full sizes.
WORKLOADS: Dict[str, Workload] = {
    "ag_tiny_p2": Workload("ag_tiny_p2", "ag", seed=0, P=2, m=64, k=128, n=128,
                           var_x=1.0, var_w=1.0 / 128,
                           note="AG-GEMM tiny, P=2, X_r 64x128, W 128x128"),
    "ag_bf16_p8": Workload("ag_bf16_p8", "ag", seed=1, P=8, m=1024, k=8192, n=3584,
                           var_x=1.0, var_w=1.0 / 8192,
                           note="AG-GEMM BF16, P=8, X_r 1024x8192, W 8192x3584 (70B-like MLP up-proj, TP=8)"),
    "rs_bf16_p8": Workload("rs_bf16_p8", "rs", seed=2, P=8, m=8192, k=3584, n=8192,
                           var_x=1.0, var_w=1.0 / 28672,
                           note="GEMM+RS BF16, P=8, X_r 8192x3584, W_r 3584x8192, chunks 1024x8192"),
    "ag_mxfp8_p8": Workload("ag_mxfp8_p8", "ag", seed=3, P=8, m=1024, k=8192, n=3584, dtype="mxfp8",
                            var_x=1.0, var_w=1.0 / 8192,
                            note="AG-GEMM MXFP8 (E4M3 + E8M0 per 32 K), shapes of ag_bf16_p8"),
    "rs_mxfp8_p8": Workload("rs_mxfp8_p8", "rs", seed=5, P=8, m=8192, k=3584, n=8192, dtype="mxfp8",
                            var_x=1.0, var_w=1.0 / 28672,
                            note="GEMM+RS MXFP8 (E4M3 + E8M0 per 32 K), shapes of rs_bf16_p8"),
    # attention block of the same layer (hidden 8192, 64 query heads and 8
    # key/value heads of 128): QKV projection as an all-gather + GEMM
    # (8192 + 2 * 1024 columns over 8 ranks = 1280 each) and the output
    # projection as a GEMM + reduce-scatter (8192 / 8 = 1024 K per rank)
    "ag_qkv_p8": Workload("ag_qkv_p8", "ag", seed=6, P=8, m=1024, k=8192, n=1280,
                          var_x=1.0, var_w=1.0 / 8192,
                          note="QKV AG-GEMM BF16, P=8, X_r 1024x8192, W_qkv 8192x1280 (rank 0's column shard)"),
    "rs_oproj_p8": Workload("rs_oproj_p8", "rs", seed=7, P=8, m=8192, k=1024, n=8192,
                            var_x=1.0, var_w=1.0 / 8192,
                            note="out-proj GEMM+RS BF16, P=8, X_r 8192x1024, W_r 1024x8192, chunks 1024x8192"),
    "moe_fwd_p8": Workload("moe_fwd_p8", "moe", seed=4, P=8, T=2048, H=4096, E=128, topk=8, I=1536,
                           var_x=1.0, var_w=1.0,
                           note="MoE forward, 2048 tokens, hidden 4096, 128 experts top-8, 8 EP ranks x 16, I=1536"),
}


def _draw(g: torch.Generator, shape, var: float) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if var != 1.0:
        x.mul_(math.sqrt(var))
    return x.to(torch.bfloat16)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU bf16 tensor, as a contiguous uint16 array."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def ag_inputs(P: int, m: int, k: int, n: int, seed: int, var_x: float = 1.0,
              var_w: float = 1.0) -> Dict[str, object]:
    """X_0..X_{P-1} ([m, k] each) then W ([k, n])."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    xs = [_draw(g, (m, k), var_x) for _ in range(P)]
    w = _draw(g, (k, n), var_w)
    return {"x": xs, "w": w}


def rs_inputs(P: int, m: int, k: int, n: int, seed: int, var_x: float = 1.0,
              var_w: float = 1.0) -> Dict[str, object]:
    """X_0..X_{P-1} ([m, k] each) then W_0..W_{P-1} ([k, n] each)."""
    g = torch.Generator(device="cpu").manual_seed(seed)
    xs = [_draw(g, (m, k), var_x) for _ in range(P)]
    ws = [_draw(g, (k, n), var_w) for _ in range(P)]
    return {"x": xs, "w": ws}


def _stream_seed(seed: int, stream: int) -> int:
    return (seed * 1_000_003 + stream) & 0x7FFFFFFFFFFFFFFF


def _draw_stream(seed: int, stream: int, shape, var: float) -> torch.Tensor:
    g = torch.Generator(device="cpu").manual_seed(_stream_seed(seed, stream))
    return _draw(g, shape, var)


def moe_inputs(T: int, H: int, E: int, I: int, seed: int, threads: int = 0) -> Dict[str, object]:
    """X [T, H] ~N(0,1), W_router [H, E] ~N(0, 1/H), then per expert
    gate [H, I] ~N(0, 1/H), up [H, I] ~N(0, 1/H), down [I, H] ~N(0, 1/I).

    Each tensor has its own generator, seeded (seed * 1000003 + stream) with
    stream 0 for X, 1 for W_router and 2 + 3e, 3 + 3e, 4 + 3e for expert e's
    gate, up and down; the draws run in parallel threads and the values do not
    depend on the thread count."""
    from concurrent.futures import ThreadPoolExecutor
    x = _draw_stream(seed, 0, (T, H), 1.0)
    wr = _draw_stream(seed, 1, (H, E), 1.0 / H)
    wg = torch.empty(E, H, I, dtype=torch.bfloat16)
    wu = torch.empty(E, H, I, dtype=torch.bfloat16)
    wd = torch.empty(E, I, H, dtype=torch.bfloat16)

    def one(e):
        wg[e] = _draw_stream(seed, 2 + 3 * e, (H, I), 1.0 / H)
        wu[e] = _draw_stream(seed, 3 + 3 * e, (H, I), 1.0 / H)
        wd[e] = _draw_stream(seed, 4 + 3 * e, (I, H), 1.0 / I)

    n = threads or min(32, os.cpu_count() or 1)
    prev = torch.get_num_threads()
    torch.set_num_threads(1)
    try:
        with ThreadPoolExecutor(max_workers=n) as ex:
            list(ex.map(one, range(E)))
    finally:
        torch.set_num_threads(prev)
    return {"x": x, "w_router": wr, "w_gate": wg, "w_up": wu, "w_down": wd}


def workload_inputs(w: Workload) -> Dict[str, object]:
    if w.op == "ag":
        return ag_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    if w.op == "rs":
        return rs_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    if w.op == "moe":
        return moe_inputs(w.T, w.H, w.E, w.I, w.seed)
    raise ValueError(w.op)


def per_block_indices(n_total: int, block: int, per_block: int, seed: int) -> np.ndarray:
    """Sorted distinct indices: per_block of every run of `block` indices (a
    shorter last run included), plus the first and last index, drawn from
    their own generator."""
    rng = np.random.default_rng(seed + 104729)
    pick = {0, n_total - 1}
    for b0 in range(0, n_total, block):
        n = min(block, n_total - b0)
        pick.update((b0 + rng.choice(n, size=min(per_block, n), replace=False)).tolist())
    return np.array(sorted(pick), dtype=np.int64)


def sample_indices(n_total: int, n_sample: int, seed: int) -> np.ndarray:
    """Sorted distinct indices in [0, n_total), always including the first and
    last index (edges and the ragged tail), drawn from their own generator."""
    n_sample = min(n_sample, n_total)
    rng = np.random.default_rng(seed + 7919)
    pick = set([0, n_total - 1])
    while len(pick) < n_sample:
        pick.add(int(rng.integers(0, n_total)))
    return np.array(sorted(pick), dtype=np.int64)
