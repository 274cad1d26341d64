"""GPU parity of the GEMM + reduce-scatter kernel against the fp64 CPU oracle.

Tolerance: max|y - ref| <= 1e-2 * max|ref| over each checked set of rows
(bf16 partials, fp32 rank-ordered sum, bf16 output).  Reruns, and the band
and row orders, must agree bit for bit (fixed rank order 0..P-1 in the sum,
fixed K order per tile)."""
import numpy as np
import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
from kosmos_inputs import WORKLOADS, bf16_bits, per_block_indices, rs_inputs

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kosmos()


def _run(K, inp, o, reps=1):
    xs = [x.cuda() for x in inp["x"]]
    ws_ = [w.cuda() for w in inp["w"]]
    P = len(xs)
    m, k = xs[0].shape
    n = ws_[0].shape[1]
    ys = [torch.empty(m // P, n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    wsb = K.workspace(K.OP_GEMM_RS, P, m, n, k, o=o)
    outs = []
    for _ in range(reps):
        for y in ys:
            y.fill_(float("nan"))
        K.gemm_rs(xs, ws_, ys, wsb, o)
        K.check(wsb, "gemm_rs")
        outs.append(torch.cat(ys, 0).clone())
    return outs, wsb


SCHEDS = {"self": 0, "fixed": 1, "unfused": 2}
PAIR = {"pair": 1, "single": 0}


@pytest.mark.parametrize("mode", list(PAIR))
@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("sched", list(SCHEDS))
@pytest.mark.parametrize("P,m,k,n", [(3, 600, 128, 264), (1, 130, 64, 256), (8, 1024, 256, 512),
                                     (2, 16, 64, 8), (4, 2048, 128, 512)])
def test_rs_small_full_compare(K, orc, P, m, k, n, sched, order, mode):
    inp = rs_inputs(P, m, k, n, seed=2000 + P * m + n, var_w=1.0 / (P * k))
    cp = PAIR[mode] if mode == "single" else -1  # auto: pairs where the grid allows
    outs, _ = _run(K, inp, K.opts(sched=SCHEDS[sched], order=order, cta_pair=cp), reps=2)
    ref = orc.gemm_rs([bf16_bits(x) for x in inp["x"]], [bf16_bits(w) for w in inp["w"]])
    got = bf16_tensor_to_f64(outs[0])
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)
    assert torch.equal(outs[0], outs[1])


def test_rs_reducer_counts_and_few_ctas(K, orc):
    inp = rs_inputs(4, 512, 128, 512, seed=4, var_w=1.0 / 512)
    ref = orc.gemm_rs([bf16_bits(x) for x in inp["x"]], [bf16_bits(w) for w in inp["w"]])
    groups = {
        # one tile engine per group: results must not depend on the schedule
        "pair": [K.opts(n_comm0=1, cta_pair=1), K.opts(n_comm0=5, cta_pair=1), K.opts(num_ctas=8, cta_pair=1),
                 K.opts(num_ctas=16, cta_pair=1), K.opts(num_ctas=32, sched=1, fixed_comm_ctas=1, cta_pair=1)],
        "single": [K.opts(cta_pair=0), K.opts(num_ctas=8, cta_pair=0), K.opts(num_ctas=4, cta_pair=0),
                   K.opts(num_ctas=12, sched=1, fixed_comm_ctas=1, cta_pair=0)],
    }
    for name, opts in groups.items():
        base = None
        for o in opts:
            outs, _ = _run(K, inp, o)
            assert rel_err(bf16_tensor_to_f64(outs[0]), ref) <= TOL
            if base is None:
                base = outs[0]
            assert torch.equal(outs[0], base), f"{name}: result depends on the schedule"


def test_rs_full_size_sampled_band_and_row(K, orc):
    """The 8-rank 8192x3584 . 3584x8192 workload: one row of every 128-row
    tile row plus every chunk's first and last row against the oracle; band order, row order
    and the unfused baseline agree bit for bit."""
    w = WORKLOADS["rs_bf16_p8"]
    inp = rs_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    band, _ = _run(K, inp, K.opts(order=0), reps=2)
    row, _ = _run(K, inp, K.opts(order=1))
    unf, _ = _run(K, inp, K.opts(sched=2))
    single, _ = _run(K, inp, K.opts(cta_pair=0))
    assert torch.equal(band[0], band[1])
    assert torch.equal(band[0], row[0])
    assert torch.equal(band[0], unf[0])
    assert rel_err(bf16_tensor_to_f64(single[0]), bf16_tensor_to_f64(band[0])) <= TOL
    mc = w.m // w.P
    rows = np.unique(np.concatenate([per_block_indices(w.m, 128, 1, seed=2), np.arange(w.P) * mc,
                                     np.arange(w.P) * mc + mc - 1]))
    ref = orc.gemm_rs([bf16_bits(x) for x in inp["x"]], [bf16_bits(x) for x in inp["w"]], rows=rows)
    got = bf16_tensor_to_f64(band[0][torch.from_numpy(rows).cuda()])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)


def test_rs_rail_decode_device_matches_oracle(K, orc):
    for order in (0, 1):
        for tm in (128, 256):
            for r in range(8):
                tl, rd = orc.rail_rs(8, 8192, 8192, rank=r, order=order, R=tm)
                assert np.array_equal(K.rail_decode_device(K.OP_GEMM_RS, 8, 8192, 8192, rail=0, order=order, rank=r,
                                                           tile_m=tm), tl)
                assert np.array_equal(K.rail_decode_device(K.OP_GEMM_RS, 8, 8192, 8192, rail=1, order=order, rank=r,
                                                           tile_m=tm), rd)


@pytest.mark.parametrize("mode", list(PAIR))
def test_rs_trace_every_entry_once(K, orc, mode):
    P, m, k, n = 4, 2048, 128, 512
    inp = rs_inputs(P, m, k, n, seed=6, var_w=1.0 / 512)
    o = K.opts(trace=1, cta_pair=PAIR[mode])
    outs, wsb = _run(K, inp, o)
    recs = K.trace_records(K.OP_GEMM_RS, P, m, n, k, wsb, o)
    tl, rd = orc.rail_rs(P, m, n, rank=0, order=0, R=256 if PAIR[mode] else 128)
    red_pairs = (P + 1) // 2  # one reducer CTA per rank from the start, two ranks per pair
    # one tile rail for all ranks: every ticket exactly once
    assert np.array_equal(np.sort(recs["ticket"][recs["kind"] == 2]), np.arange(len(tl)))
    r = recs[recs["kind"] == 3]
    if PAIR[mode]:
        rank_of = np.where(r["cta"] < 2 * red_pairs, r["cta"] % P, (r["cta"] // 2) % P)
    else:
        rank_of = r["cta"] % P
    for q in range(P):
        assert np.array_equal(np.sort(r["ticket"][rank_of == q]), np.arange(len(rd))), q
    red = recs[recs["kind"] == 3]
    assert np.all(red["t_done"] >= red["t_ready"])


def test_rs_dropped_partial_times_out_then_recovers(K, orc):
    P, m, k, n = 2, 256, 64, 256
    inp = rs_inputs(P, m, k, n, seed=8, var_w=1.0 / 128)
    xs = [x.cuda() for x in inp["x"]]
    wts = [w.cuda() for w in inp["w"]]
    ys = [torch.empty(m // P, n, dtype=torch.bfloat16, device="cuda") for _ in range(P)]
    o = K.opts(inject=K.INJECT_DROP_PARTIAL | (1 << 32), wait_limit_ns=2_000_000)
    wsb = K.workspace(K.OP_GEMM_RS, P, m, n, k, o=o)
    K.gemm_rs(xs, wts, ys, wsb, o)
    st, entry = K.status_sync(wsb)
    assert st == K.ERR_TIMEOUT
    assert (entry >> 40) == 1  # a reduce entry
    K.workspace_init(wsb)
    K.gemm_rs(xs, wts, ys, wsb, K.opts())
    K.check(wsb)
    ref = orc.gemm_rs([bf16_bits(x) for x in inp["x"]], [bf16_bits(w) for w in inp["w"]])
    assert rel_err(bf16_tensor_to_f64(torch.cat(ys, 0)), ref) <= TOL
