"""kosmos_ag_gemm_noalloc: the all-gather + GEMM entry point for callers that
cannot allocate device memory (no workspace argument; the library's own
static scratch holds the tickets, flags and status).

Called through the C ABI (ctypes) twice in a row, on two different problems.
Both entry points run the same kernel with the same plan, so each result must
equal kosmos_ag_gemm's (with a caller workspace, same inputs) bit for bit;
the small problem is also checked against the oracle's fp64 all-gather +
GEMM within max|y - ref| <= 1e-2 * max|ref|.  A transfer whose flag is
never released (host-set injection, a bounded wait of 2 ms) must come back
as TIMEOUT through kosmos_noalloc_status_sync, and the next call must be
correct again.  Collected last so that a failure here comes after every
other test.
"""
import ctypes as C

import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
import numpy as np

from kosmos_inputs import ag_inputs, bf16_bits

pytestmark = pytest.mark.gpu
TOL = 1e-2


def _ptrs(ts):
    return (C.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def test_noalloc_matches_workspace_entry_point_twice(orc):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K = kosmos()
    lib = K.lib()
    stream = torch.cuda.current_stream().cuda_stream
    for (P, m, k, n, seed) in [(8, 1024, 8192, 3584, 1), (3, 200, 192, 264, 17)]:
        inp = ag_inputs(P, m, k, n, seed=seed, var_w=1.0 / k)
        xs = [x.cuda() for x in inp["x"]]
        w = inp["w"].cuda()
        # reference: the entry point with a caller-owned workspace
        xg_ref = torch.zeros(P * m, k, dtype=torch.bfloat16, device="cuda")
        y_ref = torch.zeros(P * m, n, dtype=torch.bfloat16, device="cuda")
        ws = K.workspace(K.OP_AG_GEMM, P, m, n, k)
        K.ag_gemm(xs, w, xg_ref, y_ref, ws)
        K.check(ws, "kosmos_ag_gemm")
        # the no-allocation entry point, through the C ABI
        xg = torch.zeros(P * m, k, dtype=torch.bfloat16, device="cuda")
        y = torch.full((P * m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = lib.kosmos_ag_gemm_noalloc(_ptrs(xs), None, P, m, k, n, w.data_ptr(), None, K.BF16,
                                        xg.data_ptr(), y.data_ptr(), None, stream)
        assert rc == K.OK, rc
        torch.cuda.synchronize()
        assert not torch.isnan(y).any()
        assert torch.equal(y, y_ref), rel_err(bf16_tensor_to_f64(y), bf16_tensor_to_f64(y_ref))
        assert torch.equal(xg, xg_ref)
        if P * m <= 1024:
            ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]))
            assert rel_err(bf16_tensor_to_f64(y), ref) <= TOL, rel_err(bf16_tensor_to_f64(y), ref)


def test_noalloc_rejects_oversized_and_trace():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K = kosmos()
    lib = K.lib()
    dummy = torch.zeros(16, dtype=torch.uint8, device="cuda")
    xs = _ptrs([dummy] * 8)
    # 8 shards of 2^20 rows need 8 * 8192 piece flags = 256 KiB > 64 KiB of static scratch
    rc = lib.kosmos_ag_gemm_noalloc(xs, None, 8, 1 << 20, 64, 64, dummy.data_ptr(), None, K.BF16,
                                    dummy.data_ptr(), dummy.data_ptr(), None, None)
    assert rc == K.ERR_WORKSPACE
    o = K.opts(trace=1)
    rc = lib.kosmos_ag_gemm_noalloc(xs, None, 2, 64, 64, 64, dummy.data_ptr(), None, K.BF16,
                                    dummy.data_ptr(), dummy.data_ptr(), C.byref(o), None)
    assert rc == K.ERR_UNSUPPORTED


def test_noalloc_reports_device_status(orc):
    """The static scratch's status word through kosmos_noalloc_status_sync: OK
    after a clean call; TIMEOUT with the waiting tile's ticket after a call
    whose first transfer never releases its flag; OK and bit-equal results
    on the next clean call (each call clears the part of the array it uses)."""
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    K = kosmos()
    P, m, k, n = 2, 128, 128, 256
    inp = ag_inputs(P, m, k, n, seed=9, var_w=1.0 / k)
    xs = [x.cuda() for x in inp["x"]]
    w = inp["w"].cuda()
    xg = torch.empty(P * m, k, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(P * m, n, dtype=torch.bfloat16, device="cuda")
    K.ag_gemm_noalloc(xs, w, xg, y)
    assert K.noalloc_status_sync() == (K.OK, -1)
    y_ok = y.clone()
    o = K.opts(inject=K.INJECT_DROP_TRANSFER | (0 << 32), wait_limit_ns=2_000_000)
    K.ag_gemm_noalloc(xs, w, xg, y, o)
    st, entry = K.noalloc_status_sync()
    assert st == K.ERR_TIMEOUT, (st, entry)
    # transfer 0 is part 0 of shard 1's piece 0; the first tile of shard 1 waits for it
    split, tm = K.ag_tile_plan(P, m, k, n, o)
    _, tl = orc.rail_ag(P, m, n, TR=tm, XS=split)
    assert entry == int(np.flatnonzero(tl[:, 1] == 1)[0]), entry
    y.fill_(float("nan"))
    K.ag_gemm_noalloc(xs, w, xg, y)
    assert K.noalloc_status_sync() == (K.OK, -1)
    assert torch.equal(y, y_ok)
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]))
    assert rel_err(bf16_tensor_to_f64(y), ref) <= TOL
