"""Attention-block shapes (QKV all-gather + GEMM, output-projection GEMM +
reduce-scatter) and the emulated link-bandwidth cap.

Parity against the oracle as for the MLP shapes (max|y - ref| <= 1e-2 *
max|ref|, sampled rows at full size); every schedule and the capped link give
bit-identical results (the cap only delays releases); a capped launch lasts at
least the link time of its remote bytes (one server of link_gbs GB/s)."""
import numpy as np
import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
from kosmos_inputs import WORKLOADS, ag_inputs, bf16_bits, per_block_indices, rs_inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2
LINK_GBS = 900  # one GPU's per-direction NVLink 5 bandwidth


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kosmos()


def _timed(fn):
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    fn()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) * 1e3  # us


def run_ag(K, inp, o):
    xs = [x.cuda() for x in inp["x"]]
    w = inp["w"].cuda()
    P = len(xs)
    m, k = xs[0].shape
    n = w.shape[1]
    xg = torch.zeros(P * m, k, dtype=torch.bfloat16, device="cuda")
    y = torch.full((P * m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = K.workspace(K.OP_AG_GEMM, P, m, n, k, o=o)
    K.ag_gemm(xs, w, xg, y, ws, o)  # warm-up
    K.check(ws, "ag_gemm")
    us = _timed(lambda: K.ag_gemm(xs, w, xg, y, ws, o))
    K.check(ws, "ag_gemm")
    assert torch.equal(xg.cpu(), torch.cat(inp["x"], 0))
    return y, us


def run_rs(K, inp, o):
    xs = [x.cuda() for x in inp["x"]]
    ws_ = [w.cuda() for w in inp["w"]]
    P = len(xs)
    m, k = xs[0].shape
    n = ws_[0].shape[1]
    ys = [torch.full((m // P, n), float("nan"), dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    wsb = K.workspace(K.OP_GEMM_RS, P, m, n, k, o=o)
    K.gemm_rs(xs, ws_, ys, wsb, o)
    K.check(wsb, "gemm_rs")
    us = _timed(lambda: K.gemm_rs(xs, ws_, ys, wsb, o))
    K.check(wsb, "gemm_rs")
    return torch.cat(ys, 0), us


SCHEDS = {"self": 0, "fixed": 1, "unfused": 2}


@pytest.mark.parametrize("sched", list(SCHEDS))
@pytest.mark.parametrize("pair", [1, 0])
def test_ag_link_cap_small(K, orc, sched, pair):
    P, m, k, n = 4, 256, 512, 384
    inp = ag_inputs(P, m, k, n, seed=31, var_w=1.0 / k)
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]))
    y0, _ = run_ag(K, inp, K.opts(sched=SCHEDS[sched], cta_pair=pair))
    gbs = 10
    y1, us = run_ag(K, inp, K.opts(sched=SCHEDS[sched], cta_pair=pair, link_gbs=gbs))
    assert rel_err(bf16_tensor_to_f64(y1), ref) <= TOL
    assert torch.equal(y0, y1)
    link_us = (P - 1) * m * k * 2 / gbs / 1e3
    assert us >= 0.97 * link_us, (us, link_us)


@pytest.mark.parametrize("sched", list(SCHEDS))
@pytest.mark.parametrize("pair", [1, 0])
def test_rs_link_cap_small(K, orc, sched, pair):
    P, m, k, n = 4, 1024, 128, 512
    inp = rs_inputs(P, m, k, n, seed=32, var_w=1.0 / (P * k))
    ref = orc.gemm_rs([bf16_bits(x) for x in inp["x"]], [bf16_bits(w) for w in inp["w"]])
    y0, _ = run_rs(K, inp, K.opts(sched=SCHEDS[sched], cta_pair=pair))
    gbs = 20
    y1, us = run_rs(K, inp, K.opts(sched=SCHEDS[sched], cta_pair=pair, link_gbs=gbs))
    assert rel_err(bf16_tensor_to_f64(y1), ref) <= TOL
    assert torch.equal(y0, y1)
    link_us = (P - 1) * m * n * 2 / gbs / 1e3  # every rank's partial, except the chunk owner's
    assert us >= 0.97 * link_us, (us, link_us)


def test_ag_qkv_full_size(K, orc):
    """QKV projection, 8 ranks, X_r 1024x8192 . W 8192x1280: sampled rows,
    all schedules and the 900 GB/s link give the same bits."""
    w = WORKLOADS["ag_qkv_p8"]
    inp = ag_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    y, _ = run_ag(K, inp, K.opts())
    for o in (K.opts(sched=1), K.opts(sched=2), K.opts(link_gbs=LINK_GBS), K.opts(sched=1, link_gbs=LINK_GBS)):
        y2, _ = run_ag(K, inp, o)
        assert torch.equal(y, y2)
    _, us = run_ag(K, inp, K.opts(link_gbs=LINK_GBS))
    assert us >= 0.97 * (w.P - 1) * w.m * w.k * 2 / LINK_GBS / 1e3
    rows = np.unique(np.concatenate([per_block_indices(w.P * w.m, 128, 1, seed=7), np.arange(w.P) * w.m,
                                     np.arange(w.P) * w.m + w.m - 1]))
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]), rows=rows)
    got = bf16_tensor_to_f64(y[torch.from_numpy(rows).cuda()])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)


def test_rs_oproj_full_size(K, orc):
    """Output projection, 8 ranks, X_r 8192x1024 . W_r 1024x8192: sampled
    rows; band, row, unfused and the capped link give the same bits."""
    w = WORKLOADS["rs_oproj_p8"]
    inp = rs_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    y, _ = run_rs(K, inp, K.opts())
    for o in (K.opts(order=1), K.opts(sched=2), K.opts(link_gbs=LINK_GBS), K.opts(sched=2, link_gbs=LINK_GBS)):
        y2, _ = run_rs(K, inp, o)
        assert torch.equal(y, y2)
    mc = w.m // w.P
    rows = np.unique(np.concatenate([per_block_indices(w.m, 128, 1, seed=8), np.arange(w.P) * mc,
                                     np.arange(w.P) * mc + mc - 1]))
    ref = orc.gemm_rs([bf16_bits(x) for x in inp["x"]], [bf16_bits(x) for x in inp["w"]], rows=rows)
    got = bf16_tensor_to_f64(y[torch.from_numpy(rows).cuda()])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)


def test_moe_rejects_link_cap(K):
    from kosmos_inputs import moe_inputs
    P, T, H, E, topk, I = 2, 256, 256, 64, 2, 128
    inp = moe_inputs(T, H, E, I, seed=3)
    dev = "cuda"
    xs = [t.to(dev) for t in torch.chunk(inp["x"], P, 0)]
    sp = lambda t: [t[q * (E // P):(q + 1) * (E // P)].contiguous().to(dev) for q in range(P)]
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    z = torch.empty(T, topk, dtype=torch.int32, device=dev)
    o = K.opts(link_gbs=100)
    ws = K.moe_workspace(P, T, H, E, topk, I, o)
    with pytest.raises(K.KosmosError):
        K.moe_fwd(xs, inp["w_router"].to(dev), sp(inp["w_gate"]), sp(inp["w_up"]), sp(inp["w_down"]), ys, z,
                  z.float(), z[:, 0].clone(), z, ws, topk, o)


@pytest.mark.parametrize("pair", [1, 0])
def test_ag_mxfp8_link_cap(K, orc, pair):
    """MXFP8 all-gather + GEMM through the emulated link: same bytes as
    without it, and at least the link time of the remote pieces and their
    scale blocks."""
    P, m, k, n = 4, 256, 512, 512
    inp = ag_inputs(P, m, k, n, seed=33, var_w=1.0 / k)

    def quant(x, along):
        r, c = x.shape
        q = torch.empty(r, c, dtype=torch.uint8, device="cuda")
        sc = torch.empty(K.mxfp8_scale_bytes(r, c, along), dtype=torch.uint8, device="cuda")
        K.mxfp8_quantize(x.cuda(), q, sc, along)
        return q, sc

    qs, ss = zip(*[quant(x, True) for x in inp["x"]])
    qw, sw = quant(inp["w"], False)
    xg = torch.zeros(P * m, k, dtype=torch.uint8, device="cuda")

    def run(o):
        y = torch.full((P * m, n), float("nan"), dtype=torch.bfloat16, device="cuda")
        ws = K.workspace(K.OP_AG_GEMM, P, m, n, k, dtype=K.MXFP8_E4M3, o=o)
        f = lambda: K.ag_gemm(list(qs), qw, xg, y, ws, o, dtype=K.MXFP8_E4M3, x_scales=list(ss), w_scales=sw)
        f()
        K.check(ws, "ag mxfp8")
        us = _timed(f)
        K.check(ws, "ag mxfp8")
        return y, us

    y0, _ = run(K.opts(cta_pair=pair))
    gbs = 10
    y1, us = run(K.opts(cta_pair=pair, link_gbs=gbs))
    assert torch.equal(y0, y1)
    assert not torch.isnan(y1).any()
    link_us = (P - 1) * m * k / gbs / 1e3
    assert us >= 0.97 * link_us, (us, link_us)
