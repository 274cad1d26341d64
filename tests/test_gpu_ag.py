"""GPU parity of the all-gather + GEMM kernel against the fp64 CPU oracle.

Tolerance: max|y - ref| <= 1e-2 * max|ref| (bf16 output, fp32 accumulation).
The gathered buffer must equal the concatenated shards byte for byte, and
repeated runs must be bit-identical (fixed K order per tile, no split-K)."""
import numpy as np
import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
from kosmos_inputs import WORKLOADS, ag_inputs, bf16_bits, per_block_indices, sample_indices

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kosmos()


def _run(K, inp, o, reps=1):
    xs = [x.cuda() for x in inp["x"]]
    w = inp["w"].cuda()
    P = len(xs)
    m, k = xs[0].shape
    n = w.shape[1]
    xg = torch.empty(P * m, k, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(P * m, n, dtype=torch.bfloat16, device="cuda")
    ws = K.workspace(K.OP_AG_GEMM, P, m, n, k, o=o)
    outs = []
    for _ in range(reps):
        y.fill_(float("nan"))
        xg.zero_()
        K.ag_gemm(xs, w, xg, y, ws, o)
        K.check(ws, "ag_gemm")
        outs.append(y.clone())
    return xs, xg, outs, ws


def _check_full(orc, K, inp, o):
    xs, xg, outs, _ = _run(K, inp, o, reps=2)
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]))
    got = bf16_tensor_to_f64(outs[0])
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)
    assert torch.equal(outs[0], outs[1]), "reruns differ"
    assert torch.equal(xg.cpu(), torch.cat(inp["x"], 0)), "gathered buffer differs from the shards"


SCHEDS = {"self": 0, "fixed": 1, "unfused": 2}
PAIR = {"pair": 1, "single": 0}


@pytest.mark.parametrize("mode", list(PAIR))
@pytest.mark.parametrize("sched", list(SCHEDS))
def test_ag_tiny_workload(K, orc, sched, mode):
    w = WORKLOADS["ag_tiny_p2"]
    inp = ag_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    _check_full(orc, K, inp, K.opts(sched=SCHEDS[sched], cta_pair=PAIR[mode]))


@pytest.mark.parametrize("mode", list(PAIR))
@pytest.mark.parametrize("sched", list(SCHEDS))
@pytest.mark.parametrize("P,m,k,n", [(3, 200, 192, 264), (1, 130, 128, 256), (4, 128, 320, 512),
                                     (2, 37, 64, 8), (2, 300, 128, 520), (2, 1, 64, 8)])
def test_ag_ragged_multi_tile(K, orc, sched, P, m, k, n, mode):
    inp = ag_inputs(P, m, k, n, seed=1000 + P * m + n, var_w=1.0 / k)
    _check_full(orc, K, inp, K.opts(sched=SCHEDS[sched], cta_pair=PAIR[mode]))


@pytest.mark.parametrize("mode", list(PAIR))
@pytest.mark.parametrize("n_comm0", [1, 8, 40])
def test_ag_mover_counts(K, orc, n_comm0, mode):
    inp = ag_inputs(8, 256, 256, 512, seed=77, var_w=1.0 / 256)
    _check_full(orc, K, inp, K.opts(n_comm0=n_comm0, cta_pair=PAIR[mode]))


@pytest.mark.parametrize("mode", list(PAIR))
@pytest.mark.parametrize("split", [-1, 3, 10**6])
@pytest.mark.parametrize("P,m,k,n", [(3, 200, 192, 264), (2, 300, 128, 520), (4, 128, 320, 512)])
def test_ag_tail_split(K, orc, P, m, k, n, split, mode):
    """The last tiles run as two K halves (one wave, the last 3, all of
    them): results within tolerance of the oracle and of the unsplit rail,
    bit-identical on reruns (the two fp32 halves are added once, in either
    order: the sum is the same)."""
    inp = ag_inputs(P, m, k, n, seed=4000 + P * m + n, var_w=1.0 / k)
    o = K.opts(cta_pair=PAIR[mode], tail_split=split)
    assert K.ag_tile_plan(P, m, k, n, o)[0] > 0
    _check_full(orc, K, inp, o)
    _, _, a, _ = _run(K, inp, o)
    _, _, b, _ = _run(K, inp, K.opts(cta_pair=PAIR[mode], tail_split=0))
    assert rel_err(bf16_tensor_to_f64(a[0]), bf16_tensor_to_f64(b[0])) <= TOL


@pytest.mark.parametrize("mode", list(PAIR))
def test_ag_tail_split_full_size(K, orc, mode):
    """One wave of K-split tiles on the 8-rank workload: sampled rows against
    the oracle (the split tiles are the last ones: the last shard's rows)."""
    w = WORKLOADS["ag_bf16_p8"]
    inp = ag_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    o = K.opts(cta_pair=PAIR[mode], tail_split=-1)
    xs, xg, outs, _ = _run(K, inp, o, reps=2)
    rows = np.unique(np.concatenate([sample_indices(w.P * w.m, 16, seed=5),
                                     (w.P - 1) * w.m + np.arange(0, w.m, 97), [w.P * w.m - 1]]))
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]), rows=rows)
    got = bf16_tensor_to_f64(outs[0][torch.from_numpy(rows).cuda()])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)
    assert torch.equal(outs[0], outs[1])


def test_ag_tile_plan_split(K):
    """No split by default; tail_split = -1 is one wave: every tile engine that builds."""
    sms = K.num_sms()
    assert K.ag_tile_plan(8, 1024, 8192, 3584, K.opts(tail_split=0)) == (0, 256)
    assert K.ag_tile_plan(8, 1024, 64, 3584, K.opts(tail_split=-1))[0] == 0  # one K block: nothing to split
    sp, tm = K.ag_tile_plan(8, 1024, 8192, 3584, K.opts(tail_split=-1))
    assert tm == 256 and 1 <= sp <= sms // 2  # one per co-resident SM pair
    if sms == 152:
        assert sp == 76
    assert K.ag_tile_plan(8, 1024, 8192, 3584, K.opts(tail_split=10**6))[0] == 256  # the slot limit
    assert K.ag_tile_plan(2, 256, 8192, 512, K.opts(tail_split=10**6))[0] == 2 * 1 * 2  # clamped to the tiles
    assert K.ag_tile_plan(8, 1024, 8192, 3584, K.opts(tail_split=5))[0] == 5
    sp1, tm1 = K.ag_tile_plan(8, 1024, 8192, 3584, K.opts(cta_pair=0, tail_split=-1))
    assert tm1 == 128 and sp1 == min(sms, 8 * 8 * 14, 256)
    sp2, _ = K.ag_tile_plan(8, 1024, 8192, 3584, K.opts(cta_pair=0, sched=K.SCHED_FIXED, fixed_comm_ctas=10,
                                                         tail_split=-1))
    assert sp2 == sms - 10
    assert K.ag_tile_plan(8, 1024, 8192, 3584, K.opts(tail_split=-1), dtype=K.MXFP8_E4M3)[0] == 0


def test_ag_few_ctas(K, orc):
    """A grid much smaller than the tile count: CTAs loop over many entries."""
    inp = ag_inputs(4, 384, 256, 768, seed=5, var_w=1.0 / 256)
    _check_full(orc, K, inp, K.opts(num_ctas=6, n_comm0=2, cta_pair=0))
    _check_full(orc, K, inp, K.opts(num_ctas=3, sched=1, fixed_comm_ctas=1, cta_pair=0))
    _check_full(orc, K, inp, K.opts(num_ctas=6, n_comm0=2, cta_pair=1))
    _check_full(orc, K, inp, K.opts(num_ctas=4, sched=1, fixed_comm_ctas=2, cta_pair=1))


def test_ag_pair_and_single_agree(K, orc):
    """Both tile engines on the full 8-rank workload: equal within tolerance."""
    w = WORKLOADS["ag_bf16_p8"]
    inp = ag_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    _, _, a, _ = _run(K, inp, K.opts(cta_pair=1))
    _, _, b, _ = _run(K, inp, K.opts(cta_pair=0))
    assert rel_err(bf16_tensor_to_f64(a[0]), bf16_tensor_to_f64(b[0])) <= TOL


@pytest.mark.parametrize("sched", list(SCHEDS))
def test_ag_full_size_sampled(K, orc, sched):
    """The 8-rank 1024x8192 . 8192x3584 workload in the benchmark's launch
    configuration, checked on one row of every 128-row tile row plus every
    shard's first and last row, and for bit-identical reruns."""
    w = WORKLOADS["ag_bf16_p8"]
    inp = ag_inputs(w.P, w.m, w.k, w.n, w.seed, w.var_x, w.var_w)
    xs, xg, outs, _ = _run(K, inp, K.opts(sched=SCHEDS[sched]), reps=2)
    rows = np.unique(np.concatenate([per_block_indices(w.P * w.m, 128, 1, seed=1),
                                     np.arange(w.P) * w.m, np.arange(w.P) * w.m + w.m - 1]))
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]), rows=rows)
    got = bf16_tensor_to_f64(outs[0][torch.from_numpy(rows).cuda()])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)
    assert torch.equal(outs[0], outs[1])
    assert torch.equal(xg, torch.cat(xs, 0))


def test_ag_rail_decode_device_matches_oracle(K, orc):
    for (P, m, n) in [(8, 1024, 3584), (3, 200, 264)]:
        for tm in (128, 256):
            for split in (0, 76, 10**6):
                tr, tl = orc.rail_ag(P, m, n, TR=tm, XS=split)
                assert np.array_equal(K.rail_decode_device(K.OP_AG_GEMM, P, m, n, rail=0, tile_m=tm, split=split), tr)
                assert np.array_equal(K.rail_decode_device(K.OP_AG_GEMM, P, m, n, rail=1, tile_m=tm, split=split), tl)


@pytest.mark.parametrize("mode", list(PAIR))
def test_ag_trace_every_entry_once(K, orc, mode):
    inp = ag_inputs(4, 512, 128, 512, seed=3, var_w=1.0 / 128)
    o = K.opts(trace=1, cta_pair=PAIR[mode])
    xs, xg, outs, ws = _run(K, inp, o)
    recs = K.trace_records(K.OP_AG_GEMM, 4, 512, 512, 128, ws, o)
    split, tm = K.ag_tile_plan(4, 512, 128, 512, o)
    assert tm == (256 if PAIR[mode] else 128)
    tr, tl = orc.rail_ag(4, 512, 512, TR=tm, XS=split)
    tiles = np.sort(recs["ticket"][recs["kind"] == 2])
    transfers = np.sort(recs["ticket"][recs["kind"] == 1])
    assert np.array_equal(tiles, np.arange(len(tl)))
    assert np.array_equal(transfers, np.arange(len(tr)))
    t = recs[recs["kind"] == 2]
    assert np.all(t["t_done"] >= t["t_ready"]) and np.all(t["t_ready"] >= t["t_claim"])


@pytest.mark.parametrize("mode", list(PAIR))
def test_ag_blocked_builders_take_transfers(K, orc, mode):
    """One initial mover (pair) for 8 ranks: builders whose piece has not
    arrived take transfer parts themselves (self-scheduling only).  Every
    transfer and tile entry runs exactly once, the result matches the oracle,
    and the trace shows transfers run by CTAs that started as builders."""
    P, m, k, n = 8, 512, 512, 1024
    inp = ag_inputs(P, m, k, n, seed=91, var_w=1.0 / k)
    o = K.opts(trace=1, n_comm0=1, cta_pair=PAIR[mode])
    _check_full(orc, K, inp, K.opts(n_comm0=1, cta_pair=PAIR[mode]))
    xs, xg, outs, ws = _run(K, inp, o)
    recs = K.trace_records(K.OP_AG_GEMM, P, m, n, k, ws, o)
    split, tm = K.ag_tile_plan(P, m, k, n, o)
    tr, tl = orc.rail_ag(P, m, n, TR=tm, XS=split)
    assert np.array_equal(np.sort(recs["ticket"][recs["kind"] == 2]), np.arange(len(tl)))
    assert np.array_equal(np.sort(recs["ticket"][recs["kind"] == 1]), np.arange(len(tr)))
    first_builder = 2 if PAIR[mode] else 1  # CTAs below this one start as movers
    helpers = recs[(recs["kind"] == 1) & (recs["cta"] >= first_builder)]
    assert len(helpers) > 0, "no builder took a transfer part"
    assert torch.equal(xg.cpu(), torch.cat(inp["x"], 0))
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]))
    assert rel_err(bf16_tensor_to_f64(outs[0]), ref) <= TOL


def test_ag_fixed_crew_builders_never_move(K):
    """The fixed-split baseline keeps its partition: no transfer is run by a
    CTA outside the crew."""
    P, m, k, n = 8, 512, 512, 1024
    inp = ag_inputs(P, m, k, n, seed=92, var_w=1.0 / k)
    o = K.opts(trace=1, sched=K.SCHED_FIXED, fixed_comm_ctas=2)
    xs, xg, outs, ws = _run(K, inp, o)
    recs = K.trace_records(K.OP_AG_GEMM, P, m, n, k, ws, o)
    assert np.all(recs["cta"][recs["kind"] == 1] < 2)
    assert np.all(recs["cta"][recs["kind"] == 2] >= 2)


def test_ag_dropped_transfer_times_out_then_recovers(K, orc):
    """A transfer whose flag is never released: the waiting tile's bounded wait
    runs out, the call reports TIMEOUT with that tile's ticket, and after a
    workspace re-init the next call is correct."""
    P, m, k, n = 2, 128, 128, 256
    inp = ag_inputs(P, m, k, n, seed=9, var_w=1.0 / k)
    xs = [x.cuda() for x in inp["x"]]
    w = inp["w"].cuda()
    xg = torch.empty(P * m, k, dtype=torch.bfloat16, device="cuda")
    y = torch.empty(P * m, n, dtype=torch.bfloat16, device="cuda")
    o = K.opts(inject=K.INJECT_DROP_TRANSFER | (0 << 32), wait_limit_ns=2_000_000)
    ws = K.workspace(K.OP_AG_GEMM, P, m, n, k, o=o)
    K.ag_gemm(xs, w, xg, y, ws, o)
    st, entry = K.status_sync(ws)
    assert st == K.ERR_TIMEOUT
    # transfer 0 is part 0 of shard 1's piece 0; the first tile of shard 1 waits for it
    split, tm = K.ag_tile_plan(P, m, k, n, o)
    _, tl = orc.rail_ag(P, m, n, TR=tm, XS=split)
    assert entry == int(np.flatnonzero(tl[:, 1] == 1)[0])
    K.workspace_init(ws)
    K.ag_gemm(xs, w, xg, y, ws, K.opts())
    K.check(ws)
    ref = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]))
    assert rel_err(bf16_tensor_to_f64(y), ref) <= TOL
