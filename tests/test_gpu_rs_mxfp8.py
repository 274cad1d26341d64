"""GPU parity of the MXFP8 GEMM + reduce-scatter (SM-pair block-scaled tiles,
bf16 partials, fp32 rank-ordered reduction) against the oracle's fp64 sum of
its own dequantised operands.  Tolerance max|y - ref| <= 2e-2 * max|ref|;
schedules and orders must agree bit for bit (same tile arithmetic, same
reduction order)."""
import numpy as np
import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
from kosmos_inputs import WORKLOADS, bf16_bits, per_block_indices, rs_inputs

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kosmos()


def gpu_quantize(K, x, along_cols):
    rows, cols = x.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    sc = torch.empty(K.mxfp8_scale_bytes(rows, cols, along_cols), dtype=torch.uint8, device="cuda")
    K.mxfp8_quantize(x.cuda(), q, sc, along_cols)
    return q, sc


def run(K, inp, o, reps=1):
    P = len(inp["x"])
    m, k = inp["x"][0].shape
    n = inp["w"][0].shape[1]
    qx, sx = zip(*[gpu_quantize(K, x, True) for x in inp["x"]])
    qw, sw = zip(*[gpu_quantize(K, w, False) for w in inp["w"]])
    ys = [torch.empty(m // P, n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    ws = K.workspace(K.OP_GEMM_RS, P, m, n, k, dtype=K.MXFP8_E4M3, o=o)
    outs = []
    for _ in range(reps):
        for y in ys:
            y.fill_(float("nan"))
        K.gemm_rs(list(qx), list(qw), ys, ws, o, dtype=K.MXFP8_E4M3, x_scales=list(sx), w_scales=list(sw))
        K.check(ws, "gemm_rs mxfp8")
        outs.append(torch.cat(ys, 0).clone())
    return outs


def oracle(orc, inp, rows=None):
    qx, sx = zip(*[orc.mxfp8_quantize(bf16_bits(x), True) for x in inp["x"]])
    qw, sw = zip(*[orc.mxfp8_quantize(bf16_bits(w), False) for w in inp["w"]])
    return orc.gemm_rs_mxfp8(list(qx), list(sx), list(qw), list(sw), rows=rows)


SCHEDS = {"self": 0, "fixed": 1, "unfused": 2}


@pytest.mark.parametrize("P,m,k,n", [(2, 256, 128, 256), (3, 768, 256, 272), (4, 512, 384, 512), (1, 128, 128, 128)])
def test_rs_mxfp8_small_all_schedules(K, orc, P, m, k, n):
    inp = rs_inputs(P, m, k, n, seed=6000 + P * m + n, var_w=1.0 / (P * k))
    ref = oracle(orc, inp)
    base = None
    for sched in SCHEDS.values():
        for order in (0, 1):
            outs = run(K, inp, K.opts(sched=sched, order=order), reps=2 if base is None else 1)
            got = bf16_tensor_to_f64(outs[0])
            assert not np.isnan(got).any()
            assert rel_err(got, ref) <= TOL, (sched, order, rel_err(got, ref))
            if base is None:
                assert torch.equal(outs[0], outs[1]), "reruns differ"
                base = outs[0]
            assert torch.equal(outs[0], base), f"sched {sched} order {order} differs"


def test_rs_mxfp8_full_size_sampled(K, orc):
    """The 8-rank 8192x3584 . 3584x8192 shapes in MXFP8: one row of every
    128-row tile row plus every chunk's first and last row against the
    oracle."""
    w = WORKLOADS["rs_mxfp8_p8"]
    inp = rs_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    outs = run(K, inp, K.opts(), reps=2)
    assert torch.equal(outs[0], outs[1])
    mc = w.m // w.P
    rows = np.unique(np.concatenate([per_block_indices(w.m, 128, 1, seed=4), np.arange(w.P) * mc,
                                     np.arange(w.P) * mc + mc - 1]))
    ref = oracle(orc, inp, rows=rows)
    got = bf16_tensor_to_f64(outs[0][torch.from_numpy(rows).cuda()])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)


def test_rs_mxfp8_rejects_one_sm_tiles_and_bad_sizes(K):
    inp = rs_inputs(2, 256, 128, 256, seed=3, var_w=1.0 / 256)
    with pytest.raises(K.KosmosError):
        run(K, inp, K.opts(cta_pair=0))
    bad = rs_inputs(2, 192, 128, 256, seed=3, var_w=1.0 / 256)  # 96 rows per chunk: not a multiple of 128
    with pytest.raises(K.KosmosError):
        run(K, bad, K.opts())
