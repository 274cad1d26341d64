"""CPU oracle for the KOSMOS fused operators -- TEST INFRASTRUCTURE ONLY.

Plain C (``oracle.c``), fp64 accumulation, OpenMP over output rows.  Only the
tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg use it;
the product path (``comm_persistent_gemm_gb300``) never imports it, and it
never imports the product.

``build()`` compiles ``liboracle.so`` next to this file with gcc.  The wrappers
below only marshal numpy arrays; all arithmetic is in the C file.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
from typing import List, Optional, Sequence

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle.  -ffp-contract=off keeps a*b+c unfused so x86 and
    Arm hosts produce the same doubles."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fvisibility=hidden", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def lib():
    global _lib
    if _lib is None:
        build()
        L = C.CDLL(_LIB_PATH)
        P = C.c_void_p
        i64 = C.c_int64
        L.orc_bf16_to_f64.restype = C.c_double
        L.orc_bf16_to_f64.argtypes = [C.c_uint16]
        L.orc_e4m3_to_f64.restype = C.c_double
        L.orc_e4m3_to_f64.argtypes = [C.c_uint8]
        L.orc_f64_to_e4m3.restype = C.c_uint8
        L.orc_f64_to_e4m3.argtypes = [C.c_double]
        L.orc_mx_scale_exp.restype = C.c_int
        L.orc_mx_scale_exp.argtypes = [C.c_double]
        L.orc_mxfp8_quantize.restype = C.c_int
        L.orc_mxfp8_quantize.argtypes = [i64, i64, P, C.c_int, P, P]
        L.orc_ag_gemm.restype = C.c_int
        L.orc_ag_gemm.argtypes = [C.c_int, i64, i64, i64, P, P, P, i64, P]
        L.orc_ag_gemm_mxfp8.restype = C.c_int
        L.orc_ag_gemm_mxfp8.argtypes = [C.c_int, i64, i64, i64, P, P, P, P, P, i64, P]
        L.orc_gemm_rs.restype = C.c_int
        L.orc_gemm_rs.argtypes = [C.c_int, i64, i64, i64, P, P, P, i64, P]
        L.orc_gemm_rs_mxfp8.restype = C.c_int
        L.orc_gemm_rs_mxfp8.argtypes = [C.c_int, i64, i64, i64, P, P, P, P, P, i64, P]
        L.orc_topk_f32.restype = C.c_int
        L.orc_topk_f32.argtypes = [i64, C.c_int, C.c_int, P, P]
        L.orc_moe_dispatch_tables.restype = C.c_int
        L.orc_moe_dispatch_tables.argtypes = [i64, C.c_int, C.c_int, P, P, P, P]
        L.orc_moe_route.restype = C.c_int
        L.orc_moe_route.argtypes = [i64, i64, C.c_int, C.c_int, P, P, P, P, P, P, P, P]
        L.orc_moe_experts_mxfp8.restype = C.c_int
        L.orc_moe_experts_mxfp8.argtypes = [i64, i64, C.c_int, C.c_int, i64, C.c_int, P, P, P, P,
                                            P, P, P, P, P, P, P, i64, P]
        L.orc_moe_bwd_tokens.restype = C.c_int
        L.orc_moe_bwd_tokens.argtypes = [i64, i64, C.c_int, C.c_int, i64, C.c_int, P, P, P, P, P, P, P, P, P,
                                         P, i64, P, P, P]
        L.orc_moe_bwd_experts.restype = C.c_int
        L.orc_moe_bwd_experts.argtypes = [i64, i64, C.c_int, C.c_int, i64, C.c_int, P, P, P, P, P, P, P, P,
                                          C.c_int, P, P, P]
        L.orc_moe_bwd_router_weight.restype = C.c_int
        L.orc_moe_bwd_router_weight.argtypes = [i64, i64, C.c_int, C.c_int, i64, C.c_int, P, P, P, P, P, P,
                                                P, P, P, P]
        L.orc_moe_experts.restype = C.c_int
        L.orc_moe_experts.argtypes = [i64, i64, C.c_int, C.c_int, i64, C.c_int, P, P, P,
                                      P, P, P, C.c_int, P, i64, P]
        L.orc_rail_ag.restype = i64
        L.orc_rail_ag.argtypes = [C.c_int, i64, i64, C.c_int, C.c_int, C.c_int, C.c_int, i64, P, P, P, P]
        L.orc_rail_rs.restype = i64
        L.orc_rail_rs.argtypes = [C.c_int, i64, i64, C.c_int, C.c_int, C.c_int, C.c_int,
                                  P, P, P, P]
        L.orc_num_threads.restype = C.c_int
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _ptr_array(arrs: Sequence[np.ndarray]):
    arr = (C.c_void_p * len(arrs))(*[_ptr(a) for a in arrs])
    return arr


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    assert a.dtype == np.uint16, a.dtype
    return a


def num_threads() -> int:
    return int(lib().orc_num_threads())


# -- number formats ---------------------------------------------------------

def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    f = np.vectorize(lambda b: lib().orc_bf16_to_f64(int(b)), otypes=[np.float64])
    return f(bits)


def e4m3_to_f64(q: int) -> float:
    return float(lib().orc_e4m3_to_f64(int(q)))


def f64_to_e4m3(v: float) -> int:
    return int(lib().orc_f64_to_e4m3(float(v)))


def mx_scale_exp(blockmax: float) -> int:
    return int(lib().orc_mx_scale_exp(float(blockmax)))


def mxfp8_quantize(x_bits: np.ndarray, along_cols: bool):
    """bf16 bits [rows, cols] -> (q uint8 [rows, cols], scales uint8)."""
    x_bits = _u16(x_bits)
    rows, cols = x_bits.shape
    q = np.empty((rows, cols), dtype=np.uint8)
    if along_cols:
        s = np.empty((rows, cols // 32), dtype=np.uint8)
    else:
        s = np.empty((cols, rows // 32), dtype=np.uint8)
    rc = lib().orc_mxfp8_quantize(rows, cols, _ptr(x_bits), 1 if along_cols else 0, _ptr(q), _ptr(s))
    if rc:
        raise ValueError("orc_mxfp8_quantize failed")
    return q, s


# -- all-gather + GEMM ------------------------------------------------------

def ag_gemm(x_bits: List[np.ndarray], w_bits: np.ndarray,
            rows: Optional[np.ndarray] = None) -> np.ndarray:
    P = len(x_bits)
    m, k = x_bits[0].shape
    n = w_bits.shape[1]
    xs = [_u16(x) for x in x_bits]
    w = _u16(w_bits)
    nrows = P * m if rows is None else len(rows)
    y = np.empty((nrows, n), dtype=np.float64)
    rp = None
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rp = _ptr(rows)
    rc = lib().orc_ag_gemm(P, m, k, n, _ptr_array(xs), _ptr(w), rp, nrows, _ptr(y))
    if rc:
        raise ValueError("orc_ag_gemm failed")
    return y


def ag_gemm_mxfp8(qx: List[np.ndarray], sx: List[np.ndarray], qw: np.ndarray, sw: np.ndarray,
                  rows: Optional[np.ndarray] = None) -> np.ndarray:
    P = len(qx)
    m, k = qx[0].shape
    n = qw.shape[1]
    nrows = P * m if rows is None else len(rows)
    y = np.empty((nrows, n), dtype=np.float64)
    qx = [np.ascontiguousarray(a) for a in qx]
    sx = [np.ascontiguousarray(a) for a in sx]
    qw = np.ascontiguousarray(qw)
    sw = np.ascontiguousarray(sw)
    rp = None
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rp = _ptr(rows)
    rc = lib().orc_ag_gemm_mxfp8(P, m, k, n, _ptr_array(qx), _ptr_array(sx), _ptr(qw), _ptr(sw),
                                 rp, nrows, _ptr(y))
    if rc:
        raise ValueError("orc_ag_gemm_mxfp8 failed")
    return y


# -- GEMM + reduce-scatter --------------------------------------------------

def gemm_rs(x_bits: List[np.ndarray], w_bits: List[np.ndarray],
            rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Rows of Y = sum_r X_r W_r (global row indices).  Chunk c of the scatter
    is rows [c*m/P, (c+1)*m/P)."""
    P = len(x_bits)
    m, k = x_bits[0].shape
    n = w_bits[0].shape[1]
    xs = [_u16(x) for x in x_bits]
    ws = [_u16(w) for w in w_bits]
    nrows = m if rows is None else len(rows)
    y = np.empty((nrows, n), dtype=np.float64)
    rp = None
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rp = _ptr(rows)
    rc = lib().orc_gemm_rs(P, m, k, n, _ptr_array(xs), _ptr_array(ws), rp, nrows, _ptr(y))
    if rc:
        raise ValueError("orc_gemm_rs failed")
    return y


def gemm_rs_mxfp8(qx: List[np.ndarray], sx: List[np.ndarray], qw: List[np.ndarray], sw: List[np.ndarray],
                  rows: Optional[np.ndarray] = None) -> np.ndarray:
    """Rows of Y = sum_r dequant(X_r) dequant(W_r); scales row-major [rows, k/32]
    for X_r and [n, k/32] for W_r (as mxfp8_quantize returns them)."""
    P = len(qx)
    m, k = qx[0].shape
    n = qw[0].shape[1]
    nrows = m if rows is None else len(rows)
    y = np.empty((nrows, n), dtype=np.float64)
    arrs = [[np.ascontiguousarray(a) for a in lst] for lst in (qx, sx, qw, sw)]
    rp = None
    if rows is not None:
        rows = np.ascontiguousarray(rows, dtype=np.int64)
        rp = _ptr(rows)
    rc = lib().orc_gemm_rs_mxfp8(P, m, k, n, *[_ptr_array(a) for a in arrs], rp, nrows, _ptr(y))
    if rc:
        raise ValueError("orc_gemm_rs_mxfp8 failed")
    return y


# -- MoE ------------------------------------------------------------------

def topk_f32(scores: np.ndarray, K: int) -> np.ndarray:
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    T, E = scores.shape
    idx = np.empty((T, K), dtype=np.int32)
    if lib().orc_topk_f32(T, E, K, _ptr(scores), _ptr(idx)):
        raise ValueError("orc_topk_f32 failed")
    return idx


def moe_dispatch_tables(idx: np.ndarray, E: int):
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    T, K = idx.shape
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E, dtype=np.int32)
    pos = np.empty((T, K), dtype=np.int32)
    if lib().orc_moe_dispatch_tables(T, E, K, _ptr(idx), _ptr(counts), _ptr(offsets), _ptr(pos)):
        raise ValueError("orc_moe_dispatch_tables failed")
    return counts, offsets, pos


def moe_route(x_bits: np.ndarray, wr_bits: np.ndarray, K: int):
    x = _u16(x_bits)
    wr = _u16(wr_bits)
    T, H = x.shape
    E = wr.shape[1]
    logits = np.empty((T, E), dtype=np.float64)
    idx = np.empty((T, K), dtype=np.int32)
    gate = np.empty((T, K), dtype=np.float64)
    counts = np.empty(E, dtype=np.int32)
    offsets = np.empty(E, dtype=np.int32)
    pos = np.empty((T, K), dtype=np.int32)
    rc = lib().orc_moe_route(T, H, E, K, _ptr(x), _ptr(wr), _ptr(logits), _ptr(idx), _ptr(gate),
                             _ptr(counts), _ptr(offsets), _ptr(pos))
    if rc:
        raise ValueError("orc_moe_route failed")
    return {"logits": logits, "idx": idx, "gate": gate, "counts": counts,
            "offsets": offsets, "pos": pos}


def moe_experts(x_bits: np.ndarray, idx: np.ndarray, gate: np.ndarray,
                wg_bits: List[np.ndarray], wu_bits: List[np.ndarray], wd_bits: List[np.ndarray],
                E: int, identity: bool = False,
                tokens: Optional[np.ndarray] = None) -> np.ndarray:
    """wg/wu/wd: one array per EP rank: [E/P, H, I], [E/P, H, I], [E/P, I, H]."""
    x = _u16(x_bits)
    T, H = x.shape
    K = idx.shape[1]
    P = len(wg_bits)
    I = wg_bits[0].shape[2]
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    wg = [_u16(a) for a in wg_bits]
    wu = [_u16(a) for a in wu_bits]
    wd = [_u16(a) for a in wd_bits]
    ntok = T if tokens is None else len(tokens)
    out = np.empty((ntok, H), dtype=np.float64)
    tp = None
    if tokens is not None:
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        tp = _ptr(tokens)
    rc = lib().orc_moe_experts(T, H, E, K, I, P, _ptr(x), _ptr(idx), _ptr(gate),
                               _ptr_array(wg), _ptr_array(wu), _ptr_array(wd),
                               1 if identity else 0, tp, ntok, _ptr(out))
    if rc:
        raise ValueError("orc_moe_experts failed")
    return out


def moe_experts_mxfp8(xq: np.ndarray, xs: np.ndarray, idx: np.ndarray, gate: np.ndarray,
                      wg: List[tuple], wu: List[tuple], wd: List[tuple],
                      tokens: Optional[np.ndarray] = None) -> np.ndarray:
    """MXFP8 experts.  xq [T, H] E4M3 codes, xs [T, H/32] scale bytes (as
    mxfp8_quantize(x, along_cols=True) returns them); wg/wu/wd: one
    (codes, scales) pair per EP rank, codes [E/P, H, I] (down: [E/P, I, H]),
    scales [E/P, I, H/32] (down: [E/P, H, I/32]) -- each expert quantised
    along its K dimension."""
    xq = np.ascontiguousarray(xq, dtype=np.uint8)
    xs = np.ascontiguousarray(xs, dtype=np.uint8)
    T, H = xq.shape
    K = idx.shape[1]
    P = len(wg)
    Eq, _, I = wg[0][0].shape
    idx = np.ascontiguousarray(idx, dtype=np.int32)
    gate = np.ascontiguousarray(gate, dtype=np.float64)
    arrs = [[np.ascontiguousarray(w[j], dtype=np.uint8) for w in lst] for lst in (wg, wu, wd) for j in (0, 1)]
    ntok = T if tokens is None else len(tokens)
    out = np.empty((ntok, H), dtype=np.float64)
    tp = None
    if tokens is not None:
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        tp = _ptr(tokens)
    rc = lib().orc_moe_experts_mxfp8(T, H, Eq * P, K, I, P, _ptr(xq), _ptr(xs), _ptr(idx), _ptr(gate),
                                     *[_ptr_array(a) for a in arrs], tp, ntok, _ptr(out))
    if rc:
        raise ValueError("orc_moe_experts_mxfp8 failed")
    return out


def moe_bwd_tokens(x_bits, wr_bits, route, dout_bits, wg_bits, wu_bits, wd_bits, tokens=None):
    """dx (expert and router paths), dgate and dl of the selected tokens
    (all when tokens is None).  route: orc.moe_route's output."""
    x = _u16(x_bits)
    T, H = x.shape
    wr = _u16(wr_bits)
    E = wr.shape[1]
    idx = np.ascontiguousarray(route["idx"], dtype=np.int32)
    K = idx.shape[1]
    gate = np.ascontiguousarray(route["gate"], dtype=np.float64)
    logits = np.ascontiguousarray(route["logits"], dtype=np.float64)
    dout = _u16(dout_bits)
    wg = [_u16(a) for a in wg_bits]
    wu = [_u16(a) for a in wu_bits]
    wd = [_u16(a) for a in wd_bits]
    P = len(wg)
    I = wg[0].shape[2]
    ntok = T if tokens is None else len(tokens)
    tp = None
    if tokens is not None:
        tokens = np.ascontiguousarray(tokens, dtype=np.int64)
        tp = _ptr(tokens)
    dx = np.empty((ntok, H))
    dgate = np.empty((ntok, K))
    dl = np.empty((ntok, E))
    rc = lib().orc_moe_bwd_tokens(T, H, E, K, I, P, _ptr(x), _ptr(wr), _ptr(logits), _ptr(idx), _ptr(gate),
                                  _ptr(dout), _ptr_array(wg), _ptr_array(wu), _ptr_array(wd), tp, ntok,
                                  _ptr(dx), _ptr(dgate), _ptr(dl))
    if rc:
        raise ValueError("orc_moe_bwd_tokens failed")
    return {"dx": dx, "dgate": dgate, "dl": dl}


def moe_bwd_experts(x_bits, route, dout_bits, wg_bits, wu_bits, wd_bits, experts):
    """(dWg, dWu, dWd) of the selected experts: [n, H, I], [n, H, I], [n, I, H]."""
    x = _u16(x_bits)
    T, H = x.shape
    idx = np.ascontiguousarray(route["idx"], dtype=np.int32)
    K = idx.shape[1]
    gate = np.ascontiguousarray(route["gate"], dtype=np.float64)
    dout = _u16(dout_bits)
    wg = [_u16(a) for a in wg_bits]
    wu = [_u16(a) for a in wu_bits]
    wd = [_u16(a) for a in wd_bits]
    P = len(wg)
    Eq, _, I = wg[0].shape
    ex = np.ascontiguousarray(experts, dtype=np.int32)
    n = len(ex)
    dwg = np.empty((n, H, I))
    dwu = np.empty((n, H, I))
    dwd = np.empty((n, I, H))
    rc = lib().orc_moe_bwd_experts(T, H, Eq * P, K, I, P, _ptr(x), _ptr(idx), _ptr(gate), _ptr(dout),
                                   _ptr_array(wg), _ptr_array(wu), _ptr_array(wd), _ptr(ex), n,
                                   _ptr(dwg), _ptr(dwu), _ptr(dwd))
    if rc:
        raise ValueError("orc_moe_bwd_experts failed")
    return dwg, dwu, dwd


def moe_bwd_router_weight(x_bits, wr_bits, route, dout_bits, wg_bits, wu_bits, wd_bits):
    """dWr [H, E] over every token."""
    x = _u16(x_bits)
    T, H = x.shape
    wr = _u16(wr_bits)
    E = wr.shape[1]
    idx = np.ascontiguousarray(route["idx"], dtype=np.int32)
    K = idx.shape[1]
    gate = np.ascontiguousarray(route["gate"], dtype=np.float64)
    logits = np.ascontiguousarray(route["logits"], dtype=np.float64)
    dout = _u16(dout_bits)
    wg = [_u16(a) for a in wg_bits]
    wu = [_u16(a) for a in wu_bits]
    wd = [_u16(a) for a in wd_bits]
    P = len(wg)
    I = wg[0].shape[2]
    dwr = np.empty((H, E))
    rc = lib().orc_moe_bwd_router_weight(T, H, E, K, I, P, _ptr(x), _ptr(wr), _ptr(logits), _ptr(idx),
                                         _ptr(gate), _ptr(dout), _ptr_array(wg), _ptr_array(wu), _ptr_array(wd),
                                         _ptr(dwr))
    if rc:
        raise ValueError("orc_moe_bwd_router_weight failed")
    return dwr


# -- rails ------------------------------------------------------------------

def rail_ag(P: int, m: int, n: int, R: int = 128, BN: int = 256, TR: Optional[int] = None, PR: int = 32,
            XS: int = 0):
    """Transfer rail (pieces of R rows in parts of PR rows) and tile rail
    (tiles of TR rows, BN columns; the last XS tiles as column halves)."""
    TR = R if TR is None else TR
    nt = C.c_int64()
    nb = C.c_int64()
    if lib().orc_rail_ag(P, m, n, R, BN, TR, PR, XS, None, C.byref(nt), None, C.byref(nb)) < 0:
        raise ValueError("inconsistent rail arguments")
    tr = np.zeros((nt.value, 4), dtype=np.int32)
    tl = np.zeros((nb.value, 4), dtype=np.int32)
    lib().orc_rail_ag(P, m, n, R, BN, TR, PR, XS, _ptr(tr), C.byref(nt), _ptr(tl), C.byref(nb))
    return tr, tl


def rail_rs(P: int, m: int, n: int, rank: int, order: int, R: int = 128, BN: int = 256):
    nb = C.c_int64()
    nr = C.c_int64()
    if lib().orc_rail_rs(P, m, n, R, BN, order, rank, None, C.byref(nb), None, C.byref(nr)) < 0:
        raise ValueError("m must be divisible by P")
    tl = np.zeros((nb.value, 4), dtype=np.int32)
    rd = np.zeros((nr.value, 4), dtype=np.int32)
    lib().orc_rail_rs(P, m, n, R, BN, order, rank, _ptr(tl), C.byref(nb), _ptr(rd), C.byref(nr))
    return tl, rd
