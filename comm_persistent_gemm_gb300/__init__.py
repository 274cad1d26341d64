"""Python binding of libkosmos.so (C ABI in include/kosmos.h).

Argument marshalling only: every step of the fused operators runs in the
CUDA kernels of the library.  Tensors are torch CUDA tensors (PyTorch supplies
device memory and streams).  There is no fallback: if the library is missing
or a call fails, a KosmosError is raised.
"""
from __future__ import annotations

import ctypes as C
import os
from typing import List, Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libkosmos.so")

KOSMOS_MAX_P = 8
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_WORKSPACE, ERR_CUDA, ERR_TIMEOUT, ERR_DEVICE = range(7)
STATUS_NAMES = {0: "OK", 1: "INVALID_ARG", 2: "UNSUPPORTED", 3: "WORKSPACE", 4: "CUDA", 5: "TIMEOUT",
                6: "DEVICE"}
BF16, MXFP8_E4M3 = 0, 1
OP_AG_GEMM, OP_GEMM_RS, OP_MOE_FWD = 0, 1, 2
SCHED_SELF, SCHED_FIXED, SCHED_UNFUSED = 0, 1, 2
ORDER_BAND, ORDER_ROW = 0, 1
INJECT_DROP_TRANSFER = 0x1
INJECT_DROP_PARTIAL = 0x2
INJECT_IDENTITY_EXPERTS = 0x4
INJECT_DROP_DISPATCH = 0x8
INJECT_DROP_ARRIVAL = 0x10
MOE_VIEW_LOGITS, MOE_VIEW_RECV, MOE_VIEW_H, MOE_VIEW_Y, MOE_VIEW_SLOT, MOE_VIEW_OFFSETS, MOE_VIEW_TRACE = range(7)
MOE_VIEW_RECV_SCALES, MOE_VIEW_XQ, MOE_VIEW_XS = 7, 8, 9  # MXFP8 only
KIND_NAMES = {1: "TRANSFER", 2: "TILE", 3: "REDUCE", 4: "ROUTE", 5: "DISPATCH", 6: "TILE_GU", 7: "TILE_D",
              8: "PUSH", 9: "FOLD", 10: "TILE_HALF", 11: "QUANT", 16: "ZPAD", 17: "GRADIN", 18: "RBWD",
              19: "RDX", 20: "DH", 21: "DGU", 22: "DWD", 23: "DWGU", 24: "DWR"}

EXPORTS = ["kosmos_default_opts", "kosmos_num_sms", "kosmos_workspace_bytes", "kosmos_workspace_init",
           "kosmos_ag_gemm", "kosmos_gemm_rs", "kosmos_moe_fwd", "kosmos_mxfp8_quantize", "kosmos_status_sync",
           "kosmos_trace_info", "kosmos_rail_decode", "kosmos_rail_decode_device", "kosmos_ag_gemm_noalloc",
           "kosmos_moe_workspace_bytes", "kosmos_moe_debug_view", "kosmos_ag_tile_plan", "kosmos_moe_bwd",
           "kosmos_moe_bwd_workspace_bytes", "kosmos_moe_bwd_debug_view", "kosmos_ag_gemm_host",
           "kosmos_noalloc_status_sync"]


class KosmosError(RuntimeError):
    def __init__(self, status: int, what: str, entry: int = -1):
        self.status = status
        self.entry = entry
        super().__init__(f"{what}: KOSMOS_{STATUS_NAMES.get(status, status)}"
                         + (f" (entry {entry})" if entry >= 0 else ""))


class Opts(C.Structure):
    _fields_ = [("sched", C.c_int32), ("n_comm0", C.c_int32), ("fixed_comm_ctas", C.c_int32),
                ("order", C.c_int32), ("num_ctas", C.c_int32), ("trace", C.c_int32),
                ("cta_pair", C.c_int32), ("plain_launch", C.c_int32),
                ("wait_limit_ns", C.c_uint64), ("inject", C.c_uint64), ("tail_split", C.c_int64),
                ("link_gbs", C.c_int64)]


class TraceRec(C.Structure):
    _fields_ = [("t_claim", C.c_int64), ("t_ready", C.c_int64), ("t_done", C.c_int64),
                ("kind", C.c_int32), ("ticket", C.c_int32), ("cta", C.c_int32), ("pad", C.c_int32)]


_lib = None


def build(force: bool = False, verbose: bool = False) -> str:
    from . import buildlib as _b
    return _b.build(force=force, verbose=verbose)


def lib():
    """The loaded library.  Raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with comm_persistent_gemm_gb300.build()")
    L = C.CDLL(LIB_PATH)
    vp, i64, i32 = C.c_void_p, C.c_int64, C.c_int
    L.kosmos_default_opts.argtypes = [C.POINTER(Opts)]
    L.kosmos_default_opts.restype = None
    L.kosmos_num_sms.restype = i32
    L.kosmos_workspace_bytes.argtypes = [i32, i32, i64, i64, i64, i32, C.POINTER(Opts)]
    L.kosmos_workspace_bytes.restype = C.c_size_t
    L.kosmos_workspace_init.argtypes = [vp, C.c_size_t, vp]
    L.kosmos_workspace_init.restype = i32
    L.kosmos_ag_gemm.argtypes = [vp, vp, i32, i64, i64, i64, vp, vp, i32, vp, vp, vp, C.c_size_t,
                                 C.POINTER(Opts), vp]
    L.kosmos_ag_gemm.restype = i32
    L.kosmos_gemm_rs.argtypes = [vp, vp, vp, vp, i32, i64, i64, i64, i32, vp, vp, C.c_size_t, C.POINTER(Opts), vp]
    L.kosmos_gemm_rs.restype = i32
    L.kosmos_moe_fwd.argtypes = [vp, vp, i32, i64, i64, i32, i32, i64, vp, vp, vp, vp, vp, vp, i32, vp, vp, vp, vp,
                                 vp, vp, C.c_size_t, C.POINTER(Opts), vp]
    L.kosmos_moe_fwd.restype = i32
    L.kosmos_mxfp8_quantize.argtypes = [vp, i64, i64, i32, vp, vp, vp]
    L.kosmos_mxfp8_quantize.restype = i32
    L.kosmos_status_sync.argtypes = [vp, vp, C.POINTER(i64)]
    L.kosmos_status_sync.restype = i32
    L.kosmos_trace_info.argtypes = [i32, i32, i64, i64, i64, i32, C.POINTER(Opts), vp, C.POINTER(vp),
                                    C.POINTER(C.c_int32), C.POINTER(C.c_int32)]
    L.kosmos_trace_info.restype = i32
    L.kosmos_rail_decode.argtypes = [i32, i32, i64, i64, i32, i32, i32, i32, i64, vp, i64]
    L.kosmos_rail_decode.restype = i64
    L.kosmos_rail_decode_device.argtypes = [i32, i32, i64, i64, i32, i32, i32, i32, i64, vp, i64, vp]
    L.kosmos_rail_decode_device.restype = i64
    L.kosmos_ag_gemm_noalloc.argtypes = [vp, vp, i32, i64, i64, i64, vp, vp, i32, vp, vp, C.POINTER(Opts), vp]
    L.kosmos_ag_gemm_noalloc.restype = i32
    L.kosmos_noalloc_status_sync.argtypes = [vp, C.POINTER(i64)]
    L.kosmos_noalloc_status_sync.restype = i32
    L.kosmos_moe_workspace_bytes.argtypes = [i32, i64, i64, i32, i32, i64, i32, C.POINTER(Opts)]
    L.kosmos_moe_workspace_bytes.restype = C.c_size_t
    L.kosmos_moe_debug_view.argtypes = [i32, i32, i64, i64, i32, i32, i64, i32, vp, C.POINTER(vp), C.POINTER(i64)]
    L.kosmos_moe_debug_view.restype = i32
    L.kosmos_ag_tile_plan.argtypes = [i32, i64, i64, i64, i32, C.POINTER(Opts), C.POINTER(i64), C.POINTER(C.c_int32)]
    L.kosmos_moe_bwd.argtypes = [vp, vp, i32, i64, i64, i32, i32, i64, vp, vp, vp, vp, vp, vp, C.c_size_t, vp, vp, vp,
                                 vp, vp, vp, vp, C.c_size_t, C.POINTER(Opts), vp]
    L.kosmos_moe_bwd.restype = i32
    L.kosmos_ag_gemm_host.argtypes = [vp, vp, i32, i64, i64, i64, vp, vp, vp, vp, vp, C.c_size_t, C.POINTER(Opts), vp,
                                      vp, vp]
    L.kosmos_ag_gemm_host.restype = i32
    L.kosmos_moe_bwd_workspace_bytes.argtypes = [i32, i64, i64, i32, i32, i64, C.POINTER(Opts)]
    L.kosmos_moe_bwd_workspace_bytes.restype = C.c_size_t
    L.kosmos_moe_bwd_debug_view.argtypes = [i32, i32, i64, i64, i32, i32, i64, vp, C.POINTER(vp), C.POINTER(i64)]
    L.kosmos_moe_bwd_debug_view.restype = i32
    L.kosmos_ag_tile_plan.restype = i32
    _lib = L
    return L


def opts(**kw) -> Opts:
    o = Opts()
    lib().kosmos_default_opts(C.byref(o))
    for k, v in kw.items():
        if v is None:
            continue
        if not hasattr(o, k):
            raise TypeError(f"unknown option {k}")
        setattr(o, k, int(v))
    return o


def _stream(stream) -> Optional[int]:
    import torch
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ptrs(ts: Sequence) -> C.Array:
    return (C.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _check_cuda(*ts):
    for t in ts:
        if t is None:
            continue
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError("kosmos tensors must be contiguous CUDA tensors")


def _raise(rc: int, what: str):
    if rc != OK:
        raise KosmosError(rc, what)


def num_sms() -> int:
    return int(lib().kosmos_num_sms())


def workspace_bytes(op: int, P: int, m: int, n: int, k: int, dtype: int = BF16, o: Optional[Opts] = None) -> int:
    return int(lib().kosmos_workspace_bytes(op, P, m, n, k, dtype, C.byref(o) if o is not None else None))


def workspace(op: int, P: int, m: int, n: int, k: int, dtype: int = BF16, o: Optional[Opts] = None,
              device=None):
    """A zeroed workspace tensor (uint8) sized for this call."""
    import torch
    nbytes = workspace_bytes(op, P, m, n, k, dtype, o)
    if nbytes == 0:
        raise KosmosError(ERR_INVALID_ARG, "workspace_bytes")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def workspace_init(ws, stream=None):
    _raise(lib().kosmos_workspace_init(ws.data_ptr(), ws.numel() * ws.element_size(), _stream(stream)),
           "kosmos_workspace_init")


def ag_gemm(x_shards: List, w, x_gathered, y, ws, o: Optional[Opts] = None, dtype: int = BF16,
            x_scales: Optional[List] = None, w_scales=None, stream=None):
    """Y = concat_r(x_shards[r]) @ w; x_gathered receives the concatenation."""
    _check_cuda(*x_shards, w, x_gathered, y, ws, *(x_scales or []), w_scales)
    P = len(x_shards)
    m, k = x_shards[0].shape
    n = w.shape[1]
    xs = _ptrs(x_shards)
    xsc = _ptrs(x_scales) if x_scales is not None else None
    rc = lib().kosmos_ag_gemm(xs, xsc, P, m, k, n, w.data_ptr(),
                              w_scales.data_ptr() if w_scales is not None else None, dtype,
                              x_gathered.data_ptr(), y.data_ptr(), ws.data_ptr(), ws.numel(),
                              C.byref(o) if o is not None else None, _stream(stream))
    _raise(rc, "kosmos_ag_gemm")


def ag_gemm_host(x_host: List, x_dev: List, w, x_gathered, y_dev, y_host, ws, o: Optional[Opts] = None,
                 stream=None, h2d_stream=None, d2h_stream=None):
    """ag_gemm from pinned host shards to a pinned host output; the copies run
    on h2d_stream / d2h_stream and overlap the kernel on `stream`."""
    _check_cuda(*x_dev, w, x_gathered, y_dev, ws)
    for t in list(x_host) + [y_host]:
        if t.is_cuda or not t.is_pinned() or not t.is_contiguous():
            raise ValueError("host tensors must be contiguous pinned CPU tensors")
    if h2d_stream is None or d2h_stream is None:
        raise ValueError("ag_gemm_host needs two copy streams")
    P = len(x_host)
    m, k = x_host[0].shape
    n = w.shape[1]
    rc = lib().kosmos_ag_gemm_host(_ptrs(x_host), _ptrs(x_dev), P, m, k, n, w.data_ptr(), x_gathered.data_ptr(),
                                   y_dev.data_ptr(), y_host.data_ptr(), ws.data_ptr(), ws.numel(),
                                   C.byref(o) if o is not None else None, _stream(stream), _stream(h2d_stream),
                                   _stream(d2h_stream))
    _raise(rc, "kosmos_ag_gemm_host")


def ag_gemm_noalloc(x_shards: List, w, x_gathered, y, o: Optional[Opts] = None, dtype: int = BF16,
                    x_scales: Optional[List] = None, w_scales=None, stream=None):
    """ag_gemm with the library's own static scratch instead of a workspace
    (for callers that cannot allocate device memory)."""
    _check_cuda(*x_shards, w, x_gathered, y, *(x_scales or []), w_scales)
    P = len(x_shards)
    m, k = x_shards[0].shape
    n = w.shape[1]
    xsc = _ptrs(x_scales) if x_scales is not None else None
    rc = lib().kosmos_ag_gemm_noalloc(_ptrs(x_shards), xsc, P, m, k, n, w.data_ptr(),
                                      w_scales.data_ptr() if w_scales is not None else None, dtype,
                                      x_gathered.data_ptr(), y.data_ptr(), C.byref(o) if o is not None else None,
                                      _stream(stream))
    _raise(rc, "kosmos_ag_gemm_noalloc")


def gemm_rs(x_shards: List, w_shards: List, y_chunks: List, ws, o: Optional[Opts] = None, stream=None,
            dtype: int = BF16, x_scales: Optional[List] = None, w_scales: Optional[List] = None):
    """y_chunks[c] = rows [c*m/P, (c+1)*m/P) of sum_r x_shards[r] @ w_shards[r]
    (MXFP8: E4M3 bytes with MMA-tiled E8M0 scales)."""
    _check_cuda(*x_shards, *w_shards, *y_chunks, ws, *(x_scales or []), *(w_scales or []))
    P = len(x_shards)
    m, k = x_shards[0].shape
    n = w_shards[0].shape[1]
    rc = lib().kosmos_gemm_rs(_ptrs(x_shards), _ptrs(x_scales) if x_scales else None, _ptrs(w_shards),
                              _ptrs(w_scales) if w_scales else None, P, m, k, n, dtype, _ptrs(y_chunks),
                              ws.data_ptr(), ws.numel(), C.byref(o) if o is not None else None, _stream(stream))
    _raise(rc, "kosmos_gemm_rs")


def moe_fwd(x_shards: List, w_router, w_gate: List, w_up: List, w_down: List, y_shards: List, topk_idx,
            topk_gate, expert_counts, dispatch_pos, ws, topk: int, o: Optional[Opts] = None, stream=None,
            dtype: int = BF16, w_gate_scales: Optional[List] = None, w_up_scales: Optional[List] = None,
            w_down_scales: Optional[List] = None):
    """One MoE layer forward.  MXFP8: w_gate / w_up / w_down hold E4M3 bytes
    ([E/P, hidden, inter], [E/P, inter, hidden] per rank) and *_scales their
    MMA-tiled E8M0 scales, expert after expert (each expert quantised along
    its K dimension as mxfp8_quantize(w[e], along_cols=False) does)."""
    _check_cuda(*x_shards, w_router, *w_gate, *w_up, *w_down, *y_shards, topk_idx, topk_gate, expert_counts,
                dispatch_pos, ws, *(w_gate_scales or []), *(w_up_scales or []), *(w_down_scales or []))
    P = len(x_shards)
    tokens = x_shards[0].shape[0] * P
    hidden = x_shards[0].shape[1]
    E = w_router.shape[1]
    inter = w_gate[0].shape[2]
    mx = dtype == MXFP8_E4M3
    if mx and (w_gate_scales is None or w_up_scales is None or w_down_scales is None):
        raise KosmosError(ERR_INVALID_ARG, "moe_fwd: MXFP8 needs the weight scales")
    rc = lib().kosmos_moe_fwd(_ptrs(x_shards), w_router.data_ptr(), P, tokens, hidden, E, topk, inter,
                              _ptrs(w_gate), _ptrs(w_gate_scales) if mx else None, _ptrs(w_up),
                              _ptrs(w_up_scales) if mx else None, _ptrs(w_down),
                              _ptrs(w_down_scales) if mx else None, dtype, _ptrs(y_shards), topk_idx.data_ptr(),
                              topk_gate.data_ptr(), expert_counts.data_ptr(), dispatch_pos.data_ptr(),
                              ws.data_ptr(), ws.numel(), C.byref(o) if o is not None else None, _stream(stream))
    _raise(rc, "kosmos_moe_fwd")


def moe_workspace(P: int, tokens: int, hidden: int, n_experts: int, topk: int, inter: int,
                  o: Optional[Opts] = None, device=None, dtype: int = BF16):
    """A zeroed workspace tensor (uint8) for kosmos_moe_fwd."""
    import torch
    nbytes = int(lib().kosmos_moe_workspace_bytes(P, tokens, hidden, n_experts, topk, inter, dtype,
                                                  C.byref(o) if o is not None else None))
    if nbytes == 0:
        raise KosmosError(ERR_INVALID_ARG, "kosmos_moe_workspace_bytes")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


def moe_debug_view(what: int, P: int, tokens: int, hidden: int, n_experts: int, topk: int, inter: int, ws,
                   dtype: int = BF16):
    """A uint8 view (torch tensor slice of ws) of one internal MoE buffer."""
    ptr = C.c_void_p()
    nb = C.c_int64()
    rc = lib().kosmos_moe_debug_view(what, P, tokens, hidden, n_experts, topk, inter, dtype, ws.data_ptr(),
                                     C.byref(ptr), C.byref(nb))
    _raise(rc, "kosmos_moe_debug_view")
    off = ptr.value - ws.data_ptr()
    return ws[off:off + nb.value]


def moe_bwd(x_shards: List, w_router, w_gate: List, w_up: List, w_down: List, topk_idx, topk_gate, fwd_ws,
            dy_shards: List, dx_shards: List, dw_router, dw_gate: List, dw_up: List, dw_down: List, ws,
            o: Optional[Opts] = None, stream=None):
    """Backward of a bf16 moe_fwd call whose workspace fwd_ws is passed
    unchanged: dx, dW_router (fp32), dW_gate / dW_up / dW_down (bf16)."""
    _check_cuda(*x_shards, w_router, *w_gate, *w_up, *w_down, topk_idx, topk_gate, fwd_ws, *dy_shards, *dx_shards,
                dw_router, *dw_gate, *dw_up, *dw_down, ws)
    P = len(x_shards)
    tokens = x_shards[0].shape[0] * P
    hidden = x_shards[0].shape[1]
    E = w_router.shape[1]
    topk = topk_idx.shape[1]
    inter = w_gate[0].shape[2]
    rc = lib().kosmos_moe_bwd(_ptrs(x_shards), w_router.data_ptr(), P, tokens, hidden, E, topk, inter, _ptrs(w_gate),
                              _ptrs(w_up), _ptrs(w_down), topk_idx.data_ptr(), topk_gate.data_ptr(), fwd_ws.data_ptr(),
                              fwd_ws.numel(), _ptrs(dy_shards), _ptrs(dx_shards), dw_router.data_ptr(),
                              _ptrs(dw_gate), _ptrs(dw_up), _ptrs(dw_down), ws.data_ptr(), ws.numel(),
                              C.byref(o) if o is not None else None, _stream(stream))
    _raise(rc, "kosmos_moe_bwd")


def moe_bwd_workspace(P: int, tokens: int, hidden: int, n_experts: int, topk: int, inter: int,
                      o: Optional[Opts] = None, device=None):
    import torch
    nbytes = int(lib().kosmos_moe_bwd_workspace_bytes(P, tokens, hidden, n_experts, topk, inter,
                                                      C.byref(o) if o is not None else None))
    if nbytes == 0:
        raise KosmosError(ERR_INVALID_ARG, "kosmos_moe_bwd_workspace_bytes")
    return torch.zeros(nbytes, dtype=torch.uint8, device=device or "cuda")


MOE_BWD_VIEW_DY, MOE_BWD_VIEW_DG, MOE_BWD_VIEW_DU, MOE_BWD_VIEW_DXB, MOE_BWD_VIEW_DSLOT = range(5)
MOE_BWD_VIEW_DGATE, MOE_BWD_VIEW_DL, MOE_BWD_VIEW_DXR, MOE_BWD_VIEW_TRACE = 5, 6, 7, 8


def moe_bwd_debug_view(what: int, P: int, tokens: int, hidden: int, n_experts: int, topk: int, inter: int, ws):
    """A uint8 view (torch tensor slice of ws) of one internal backward buffer."""
    ptr = C.c_void_p()
    nb = C.c_int64()
    _raise(lib().kosmos_moe_bwd_debug_view(what, P, tokens, hidden, n_experts, topk, inter, ws.data_ptr(),
                                           C.byref(ptr), C.byref(nb)), "kosmos_moe_bwd_debug_view")
    off = ptr.value - ws.data_ptr()
    return ws[off:off + nb.value]


def mxfp8_scale_bytes(rows: int, cols: int, along_cols: bool) -> int:
    """Bytes of the MMA-tiled E8M0 scale tensor for an operand [rows, cols]."""
    srows = rows if along_cols else cols
    kk = cols if along_cols else rows
    return -(-srows // 128) * 128 * (kk // 32)


def mxfp8_quantize(x, q, scales, along_cols: bool, stream=None):
    _check_cuda(x, q, scales)
    rows, cols = x.shape
    rc = lib().kosmos_mxfp8_quantize(x.data_ptr(), rows, cols, 1 if along_cols else 0, q.data_ptr(),
                                     scales.data_ptr(), _stream(stream))
    _raise(rc, "kosmos_mxfp8_quantize")


def status_sync(ws, stream=None):
    """(status, failing_entry) of the last call that used ws (synchronises)."""
    e = C.c_int64(-1)
    rc = lib().kosmos_status_sync(ws.data_ptr(), _stream(stream), C.byref(e))
    return int(rc), int(e.value)


def noalloc_status_sync(stream=None):
    """(status, failing_entry) of the last ag_gemm_noalloc call on the current
    device (synchronises); valid until the next such call."""
    e = C.c_int64(-1)
    rc = lib().kosmos_noalloc_status_sync(_stream(stream), C.byref(e))
    return int(rc), int(e.value)


def check(ws, what: str = "kosmos", stream=None):
    st, ent = status_sync(ws, stream)
    if st != OK:
        raise KosmosError(st, what, ent)


def trace_records(op: int, P: int, m: int, n: int, k: int, ws, o: Opts, dtype: int = BF16):
    """Copies the role trace out of the workspace: list of dicts, one per
    recorded entry (CTA ring order)."""
    import numpy as np
    import torch
    ptr = C.c_void_p()
    cap = C.c_int32()
    nct = C.c_int32()
    rc = lib().kosmos_trace_info(op, P, m, n, k, dtype, C.byref(o), ws.data_ptr(), C.byref(ptr), C.byref(cap),
                                 C.byref(nct))
    _raise(rc, "kosmos_trace_info")
    off = ptr.value - ws.data_ptr()
    nbytes = nct.value * cap.value * C.sizeof(TraceRec)
    raw = ws[off:off + nbytes].cpu().numpy()
    dt = np.dtype([("t_claim", "<i8"), ("t_ready", "<i8"), ("t_done", "<i8"), ("kind", "<i4"),
                   ("ticket", "<i4"), ("cta", "<i4"), ("pad", "<i4")])
    recs = raw.view(dt).reshape(nct.value, cap.value)
    return recs[recs["kind"] != 0]


def ag_tile_plan(P: int, m_per_shard: int, k: int, n: int, o: Optional[Opts] = None, dtype: int = BF16):
    """(tail_split, tile_m) that ag_gemm uses for these sizes and options on
    the current device: the arguments of its tile rail's decode."""
    sp = C.c_int64()
    tm = C.c_int32()
    if lib().kosmos_ag_tile_plan(P, m_per_shard, k, n, dtype, C.byref(o) if o is not None else None, C.byref(sp),
                                 C.byref(tm)) != 0:
        raise KosmosError(ERR_INVALID_ARG, "kosmos_ag_tile_plan")
    return sp.value, tm.value


def rail_decode(op: int, P: int, m: int, n: int, rail: int, order: int = ORDER_BAND, rank: int = 0,
                tile_m: int = 256, split: int = 0):
    """Host-compiled decode of one rail: int32 array [len, 4]."""
    import numpy as np
    ln = lib().kosmos_rail_decode(op, P, m, n, order, rank, rail, tile_m, split, None, 0)
    if ln < 0:
        raise KosmosError(ERR_INVALID_ARG, "kosmos_rail_decode")
    out = np.zeros((ln, 4), dtype=np.int32)
    lib().kosmos_rail_decode(op, P, m, n, order, rank, rail, tile_m, split, out.ctypes.data, ln)
    return out


def rail_decode_device(op: int, P: int, m: int, n: int, rail: int, order: int = ORDER_BAND, rank: int = 0,
                       tile_m: int = 256, split: int = 0, stream=None):
    import torch
    ln = lib().kosmos_rail_decode(op, P, m, n, order, rank, rail, tile_m, split, None, 0)
    if ln < 0:
        raise KosmosError(ERR_INVALID_ARG, "kosmos_rail_decode")
    out = torch.zeros((max(ln, 1), 4), dtype=torch.int32, device="cuda")
    r = lib().kosmos_rail_decode_device(op, P, m, n, order, rank, rail, tile_m, split, out.data_ptr(), ln,
                                        _stream(stream))
    if r < 0:
        raise KosmosError(ERR_CUDA, "kosmos_rail_decode_device")
    torch.cuda.synchronize()
    return out[:ln].cpu().numpy()
