"""GPU parity of the MXFP8 path: the quantiser (bit-exact against the
oracle's E4M3/E8M0 codec) and the block-scaled all-gather + GEMM (against the
oracle's fp64 product of its own dequantised operands, tolerance
max|y - ref| <= 2e-2 * max|ref|)."""
import numpy as np
import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
from kosmos_inputs import WORKLOADS, ag_inputs, bf16_bits, per_block_indices

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kosmos()


def untile_scales(tiled, srows, kk):
    """MMA-tiled scale bytes -> row-major [srows, kk/32] (layout restated)."""
    kb = kk // 32
    r = np.arange(srows)[:, None]
    b = np.arange(kb)[None, :]
    off = ((r // 128) * (kb // 4) + b // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)
    return np.asarray(tiled)[off]


def gpu_quantize(K, x, along_cols):
    rows, cols = x.shape
    q = torch.empty(rows, cols, dtype=torch.uint8, device="cuda")
    sc = torch.full((K.mxfp8_scale_bytes(rows, cols, along_cols),), 0xEE, dtype=torch.uint8, device="cuda")
    K.mxfp8_quantize(x.cuda(), q, sc, along_cols)
    torch.cuda.synchronize()
    return q, sc


def _special(x, along_cols):
    x = x.clone()
    v = x if along_cols else x.t()
    v[0, 0:32] = 0.0                                   # all-zero block
    v[1, 32:64] = 0.375                                # equal values
    v[2, 0:32] = torch.tensor(448.0 * 2.0 ** -3)       # blockmax exactly 448 * 2^-3
    v[3, 64:96] = torch.linspace(-1e-6, 1e-6, 32)      # tiny values (subnormal E4M3 after scaling)
    v[4, 96:128] = torch.linspace(-3e4, 3e4, 32)       # large values
    return x


@pytest.mark.parametrize("along_cols", [True, False])
@pytest.mark.parametrize("rows,cols", [(200, 256), (128, 384), (33, 128)])
def test_quantize_bit_exact_vs_oracle(K, orc, along_cols, rows, cols):
    if not along_cols and rows % 128:
        rows = 256
    g = torch.Generator().manual_seed(rows * cols + along_cols)
    x = (torch.randn(rows, cols, generator=g) * 3).to(torch.bfloat16)
    if rows >= 5 and cols >= 128:
        x = _special(x, along_cols)
    q, sc = gpu_quantize(K, x, along_cols)
    qo, so = orc.mxfp8_quantize(bf16_bits(x), along_cols)
    assert np.array_equal(q.cpu().numpy(), qo)
    srows = rows if along_cols else cols
    kk = cols if along_cols else rows
    sct = sc.cpu().numpy()
    assert np.array_equal(untile_scales(sct, srows, kk), so)
    pad = untile_scales(sct, -(-srows // 128) * 128, kk)[srows:]
    assert np.all(pad == 127)


def run_f8(K, inp, o, reps=1):
    P = len(inp["x"])
    m, k = inp["x"][0].shape
    n = inp["w"].shape[1]
    qs, ss = zip(*[gpu_quantize(K, x, True) for x in inp["x"]])
    qw, sw = gpu_quantize(K, inp["w"], False)
    xg = torch.zeros(P * m, k, dtype=torch.uint8, device="cuda")
    y = torch.empty(P * m, n, dtype=torch.bfloat16, device="cuda")
    ws = K.workspace(K.OP_AG_GEMM, P, m, n, k, dtype=K.MXFP8_E4M3, o=o)
    outs = []
    for _ in range(reps):
        y.fill_(float("nan"))
        K.ag_gemm(list(qs), qw, xg, y, ws, o, dtype=K.MXFP8_E4M3, x_scales=list(ss), w_scales=sw)
        K.check(ws, "ag_gemm mxfp8")
        outs.append(y.clone())
    return qs, xg, outs


def oracle_f8(orc, inp, rows=None):
    qx, sx = zip(*[orc.mxfp8_quantize(bf16_bits(x), True) for x in inp["x"]])
    qw, sw = orc.mxfp8_quantize(bf16_bits(inp["w"]), False)
    return orc.ag_gemm_mxfp8(list(qx), list(sx), qw, sw, rows=rows)


SCHEDS = {"self": 0, "fixed": 1, "unfused": 2}
PAIR = {"pair": 1, "single": 0}


@pytest.mark.parametrize("mode", list(PAIR))
@pytest.mark.parametrize("sched", list(SCHEDS))
@pytest.mark.parametrize("P,m,k,n", [(2, 64, 128, 128), (3, 200, 256, 272), (1, 128, 384, 256), (4, 130, 128, 512),
                                     (2, 300, 256, 400)])
def test_ag_mxfp8_small(K, orc, sched, P, m, k, n, mode):
    inp = ag_inputs(P, m, k, n, seed=500 + P * m + n, var_w=1.0 / k)
    qs, xg, outs = run_f8(K, inp, K.opts(sched=SCHEDS[sched], cta_pair=PAIR[mode]), reps=2)
    ref = oracle_f8(orc, inp)
    got = bf16_tensor_to_f64(outs[0])
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(xg, torch.cat(qs, 0))


@pytest.mark.parametrize("mode", list(PAIR))
def test_ag_mxfp8_full_size_sampled(K, orc, mode):
    w = WORKLOADS["ag_mxfp8_p8"]
    inp = ag_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    qs, xg, outs = run_f8(K, inp, K.opts(cta_pair=PAIR[mode]), reps=2)
    rows = np.unique(np.concatenate([per_block_indices(w.P * w.m, 128, 1, seed=3), np.arange(w.P) * w.m,
                                     np.arange(w.P) * w.m + w.m - 1]))
    ref = oracle_f8(orc, inp, rows=rows)
    got = bf16_tensor_to_f64(outs[0][torch.from_numpy(rows).cuda()])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(xg, torch.cat(qs, 0))


def test_ag_mxfp8_pair_and_single_agree(K):
    """Both tile engines on the full 8-rank MXFP8 workload: the same sums in
    another order, equal within tolerance."""
    w = WORKLOADS["ag_mxfp8_p8"]
    inp = ag_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    _, _, a = run_f8(K, inp, K.opts(cta_pair=1))
    _, _, b = run_f8(K, inp, K.opts(cta_pair=0))
    assert rel_err(bf16_tensor_to_f64(a[0]), bf16_tensor_to_f64(b[0])) <= TOL


@pytest.mark.parametrize("n_comm0", [1, 40])
def test_ag_mxfp8_pair_mover_counts_and_few_ctas(K, orc, n_comm0):
    inp = ag_inputs(4, 256, 256, 512, seed=88, var_w=1.0 / 256)
    ref = oracle_f8(orc, inp)
    for o in (K.opts(cta_pair=1, n_comm0=n_comm0), K.opts(cta_pair=1, num_ctas=6, n_comm0=2),
              K.opts(cta_pair=1, num_ctas=4, sched=1, fixed_comm_ctas=2)):
        _, _, outs = run_f8(K, inp, o)
        assert rel_err(bf16_tensor_to_f64(outs[0]), ref) <= TOL
