"""GPU parity of the one-launch MoE expert layer (router -> dispatch -> expert
GEMMs -> push -> fold) against the fp64 CPU oracle.

Integer decisions:
  * the kernel's top-k must equal a stable descending sort of its own fp32
    logits (ties to the lower expert index), bit for bit;
  * against the oracle's fp64 routing, indices must match exactly wherever the
    oracle's decision margin exceeds the fp32 logit error (1e-3); elsewhere the
    kernel's picks must be valid (within the margin of the oracle's k-th);
  * counts and dispatch positions must equal their definition applied to the
    kernel's indices (expert-major, then token order), bit for bit.
  * every token's gates must equal the renormalised softmax of the oracle's
    fp64 logits over the experts the kernel picked.
Floating outputs: max|y - ref| <= 1e-2 * max|ref| over EVERY token, where ref
is the oracle's fp64 layer run on the kernel's own routing (its top-k indices
and gates), so that tokens whose routing sits inside the fp32 logit error are
compared too; identity experts must reproduce an fp32 restatement of the
k-ordered fold bit for bit; reruns must be bit-identical."""
import numpy as np
import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
from kosmos_inputs import WORKLOADS, bf16_bits, moe_inputs, per_block_indices

pytestmark = pytest.mark.gpu
TOL = 1e-2
MARGIN = 1e-3


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kosmos()


def _split(w, P):
    E = w.shape[0]
    return [w[q * (E // P):(q + 1) * (E // P)].contiguous() for q in range(P)]


def run_moe(K, inp, P, topk, o=None, reps=1):
    T, H = inp["x"].shape
    E = inp["w_router"].shape[1]
    I = inp["w_gate"].shape[2]
    dev = "cuda"
    xs = [t.to(dev) for t in torch.chunk(inp["x"], P, 0)]
    wr = inp["w_router"].to(dev)
    wg = [t.to(dev) for t in _split(inp["w_gate"], P)]
    wu = [t.to(dev) for t in _split(inp["w_up"], P)]
    wd = [t.to(dev) for t in _split(inp["w_down"], P)]
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    idx = torch.empty(T, topk, dtype=torch.int32, device=dev)
    gate = torch.empty(T, topk, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    pos = torch.empty(T, topk, dtype=torch.int32, device=dev)
    ws = K.moe_workspace(P, T, H, E, topk, I, o)
    outs = []
    for _ in range(reps):
        for y in ys:
            y.fill_(float("nan"))
        K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, counts, pos, ws, topk, o)
        K.check(ws, "moe_fwd")
        outs.append(torch.cat(ys, 0).clone())
    logits = K.moe_debug_view(K.MOE_VIEW_LOGITS, P, T, H, E, topk, I, ws).view(torch.float32).view(T, E)
    return {"y": outs, "idx": idx.cpu().numpy(), "gate": gate.cpu().numpy(), "counts": counts.cpu().numpy(),
            "pos": pos.cpu().numpy(), "logits": logits.cpu().numpy(), "ws": ws}


def dispatch_tables_np(idx, E):
    """Definition restated: counts, exclusive offsets, position of (t, k) in the
    expert-major then token-ordered receive buffer."""
    T, Kk = idx.shape
    counts = np.bincount(idx.ravel(), minlength=E).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)[:-1]]).astype(np.int32)
    order = np.lexsort((np.repeat(np.arange(T), Kk), idx.ravel()))  # by expert, then token
    pos = np.empty(T * Kk, dtype=np.int64)
    pos[order] = np.arange(T * Kk)
    return counts, offsets, pos.reshape(T, Kk).astype(np.int32)


def check_routing(out, route, topk):
    gl = out["logits"].astype(np.float64)
    # 1) the kernel's own top-k decision on its own fp32 logits
    ref = np.argsort(-out["logits"], axis=1, kind="stable")[:, :topk]
    assert np.array_equal(out["idx"], ref)
    # 2) against the oracle's fp64 routing
    L = route["logits"]
    assert np.max(np.abs(gl - L)) <= 1e-3 * max(1.0, np.max(np.abs(L)))
    srt = -np.sort(-L, axis=1)
    gaps = np.min(srt[:, :topk] - srt[:, 1:topk + 1], axis=1)
    clear = gaps > MARGIN
    assert np.array_equal(out["idx"][clear], route["idx"][clear])
    for t in np.where(~clear)[0]:
        kth = srt[t, topk - 1]
        assert np.all(L[t, out["idx"][t]] >= kth - MARGIN)
    np.testing.assert_allclose(out["gate"][clear], route["gate"][clear], rtol=1e-4, atol=1e-6)
    # every token's gates, near-ties included: the renormalised softmax of the
    # oracle's logits over the experts the kernel selected
    sel = np.take_along_axis(L, out["idx"].astype(np.int64), axis=1)
    ex = np.exp(sel - sel.max(axis=1, keepdims=True))
    np.testing.assert_allclose(out["gate"], ex / ex.sum(axis=1, keepdims=True), rtol=1e-4, atol=1e-6)
    # 3) counts and positions: definition applied to the kernel's indices
    E = L.shape[1]
    c, _, pos = dispatch_tables_np(out["idx"], E)
    assert np.array_equal(out["counts"], c)
    assert np.array_equal(out["pos"], pos)
    if clear.all():
        assert np.array_equal(out["counts"], route["counts"])
        assert np.array_equal(out["pos"], route["pos"])
    return clear


def kernel_route(out):
    """The kernel's own routing as the oracle's routing input: its top-k
    indices and gates, and its fp32 logits widened to fp64 (the router
    backward's operating point)."""
    return {"idx": np.ascontiguousarray(out["idx"]), "gate": out["gate"].astype(np.float64),
            "logits": out["logits"].astype(np.float64)}


def oracle_experts(orc, inp, route, P, tokens=None, identity=False):
    E = inp["w_router"].shape[1]
    return orc.moe_experts(bf16_bits(inp["x"]), route["idx"], route["gate"],
                           [bf16_bits(w) for w in _split(inp["w_gate"], P)],
                           [bf16_bits(w) for w in _split(inp["w_up"], P)],
                           [bf16_bits(w) for w in _split(inp["w_down"], P)], E=E, identity=identity, tokens=tokens)


@pytest.mark.parametrize("P,T,H,E,topk,I", [(4, 512, 512, 64, 4, 256), (2, 400, 256, 64, 8, 128),
                                            (1, 128, 256, 64, 2, 128), (8, 1024, 256, 128, 8, 256)])
def test_moe_small_full_compare(K, orc, P, T, H, E, topk, I):
    inp = moe_inputs(T, H, E, I, seed=300 + T + E + topk)
    out = run_moe(K, inp, P, topk, reps=2)
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), topk)
    check_routing(out, route, topk)
    ref = oracle_experts(orc, inp, kernel_route(out), P)
    got = bf16_tensor_to_f64(out["y"][0])
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)
    assert torch.equal(out["y"][0], out["y"][1])


def test_moe_identity_experts_fold_exact(K, orc):
    """Identity experts isolate router, dispatch, push and fold: the output
    must equal the fp32 k-ordered fold of the token rows bit for bit."""
    P, T, H, E, topk, I = 4, 512, 512, 64, 8, 128
    inp = moe_inputs(T, H, E, I, seed=77)
    out = run_moe(K, inp, P, topk, o=K.opts(inject=K.INJECT_IDENTITY_EXPERTS))
    x = inp["x"].float().numpy()
    g = out["gate"].astype(np.float32)
    acc = np.zeros((T, H), dtype=np.float32)
    for k in range(topk):
        acc = (acc + (g[:, k:k + 1] * x).astype(np.float32)).astype(np.float32)
    ref_bits = torch.from_numpy(acc).to(torch.bfloat16)
    assert torch.equal(out["y"][0].cpu(), ref_bits)
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), topk)
    check_routing(out, route, topk)
    ref = oracle_experts(orc, inp, kernel_route(out), P, identity=True)
    assert rel_err(bf16_tensor_to_f64(out["y"][0]), ref) <= TOL


def test_moe_router_ties_go_to_lower_index(K, orc):
    P, T, H, E, topk, I = 2, 256, 256, 64, 4, 128
    inp = moe_inputs(T, H, E, I, seed=5)
    wr = inp["w_router"].clone()
    for e in range(0, E, 2):
        wr[:, e + 1] = wr[:, e]          # every expert pair has identical logits
    inp["w_router"] = wr
    out = run_moe(K, inp, P, topk)
    gl = out["logits"]
    assert np.array_equal(gl[:, 0::2], gl[:, 1::2]), "duplicated router columns gave different logits"
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), topk)
    check_routing(out, route, topk)
    ref = oracle_experts(orc, inp, kernel_route(out), P)
    assert rel_err(bf16_tensor_to_f64(out["y"][0]), ref) <= TOL
    # within each token's emission list, an odd expert always follows its even twin
    for t in range(T):
        lst = list(out["idx"][t])
        for j, e in enumerate(lst):
            if e % 2 == 1 and (e - 1) in lst:
                assert lst.index(e - 1) < j


def test_moe_empty_expert_and_ragged_blocks(K, orc):
    """An expert no token selects (zero router column while the others are
    scaled up) and token blocks of 200 rows (a ragged second block)."""
    P, T, H, E, topk, I = 2, 400, 256, 64, 4, 128
    inp = moe_inputs(T, H, E, I, seed=11)
    wr = inp["w_router"].float() * 50.0
    wr[:, 7] = 0.0
    inp["w_router"] = wr.to(torch.bfloat16)
    out = run_moe(K, inp, P, topk)
    assert out["counts"][7] == 0
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), topk)
    check_routing(out, route, topk)
    ref = oracle_experts(orc, inp, kernel_route(out), P)
    got = bf16_tensor_to_f64(out["y"][0])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)


def test_moe_trace_every_entry_once(K, orc):
    P, T, H, E, topk, I = 4, 512, 512, 64, 4, 256
    inp = moe_inputs(T, H, E, I, seed=21)
    o = K.opts(trace=1)
    out = run_moe(K, inp, P, topk, o=o)
    raw = K.moe_debug_view(K.MOE_VIEW_TRACE, P, T, H, E, topk, I, out["ws"]).cpu().numpy()
    dt = np.dtype([("t_claim", "<i8"), ("t_ready", "<i8"), ("t_done", "<i8"), ("kind", "<i4"),
                   ("ticket", "<i4"), ("cta", "<i4"), ("pad", "<i4")])
    recs = raw.view(dt)
    recs = recs[recs["kind"] != 0]
    counts = out["counts"]
    units = [int(sum((counts[q * (E // P) + j] + 127) // 128 for j in range(E // P))) for q in range(P)]
    RB = (T // P + 127) // 128
    ND = H // 256
    NGU = I // 128
    kinds = recs["kind"]
    for q in range(P):
        mine = recs[(recs["cta"] % P) == q]
        main = np.sort(mine["ticket"][np.isin(mine["kind"], [4, 5, 6, 7])])
        assert np.array_equal(main, np.arange(RB + RB * topk + units[q] * (NGU + ND))), q
    assert (kinds == 8).sum() == sum(units) * ND      # one push per down tile
    assert (kinds == 9).sum() == P * RB * ND          # one fold per (token block, column tile)


def test_moe_full_size_sampled(K, orc):
    """2048 tokens, hidden 4096, 128 experts top-8 over 8 emulated EP ranks,
    inter 1536: routing over every token, outputs on two tokens of every
    128-token block (both ends included) against the oracle on the kernel's
    routing, bit-identical rerun."""
    w = WORKLOADS["moe_fwd_p8"]
    inp = moe_inputs(w.T, w.H, w.E, w.I, w.seed)
    out = run_moe(K, inp, w.P, w.topk, reps=2)
    assert torch.equal(out["y"][0], out["y"][1])
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), w.topk)
    check_routing(out, route, w.topk)
    tokens = per_block_indices(w.T, 128, 2, seed=4)
    ref = oracle_experts(orc, inp, kernel_route(out), w.P, tokens=tokens)
    got = bf16_tensor_to_f64(out["y"][0][torch.from_numpy(tokens).cuda()])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)


@pytest.mark.parametrize("P,T,H,E,topk,I", [(4, 512, 512, 64, 4, 256), (2, 400, 256, 64, 8, 128),
                                            (8, 2048, 4096, 128, 8, 1536)])
def test_moe_unfused_phases_match_one_launch(K, P, T, H, E, topk, I):
    """The unfused baseline runs the same kernel once per phase (route and
    plan | dispatch | gate/up tiles | down tiles | push and fold): every
    output and routing table equals the one-launch layer's bit for bit, and
    reruns are bit-identical."""
    inp = moe_inputs(T, H, E, I, seed=500 + T + E)
    one = run_moe(K, inp, P, topk)
    unf = run_moe(K, inp, P, topk, o=K.opts(sched=K.SCHED_UNFUSED), reps=2)
    assert torch.equal(unf["y"][0], unf["y"][1])
    assert torch.equal(one["y"][0], unf["y"][0])
    for key in ("idx", "gate", "counts", "pos"):
        assert np.array_equal(one[key], unf[key]), key


def test_moe_dropped_dispatch_times_out_then_recovers(K, orc):
    """A dispatch whose rows are never counted as arrived: the gate/up tiles
    waiting for them run out of their bounded wait, the call reports TIMEOUT
    (every CTA leaves; nothing hangs), and after a workspace re-init the next
    call matches the oracle."""
    P, T, H, E, topk, I = 2, 256, 256, 64, 2, 128
    inp = moe_inputs(T, H, E, I, seed=17)
    first_dispatch = (T // P + 127) // 128  # main-rail tickets: ROUTE entries first, then DISPATCH
    o = K.opts(inject=K.INJECT_DROP_DISPATCH | (first_dispatch << 32), wait_limit_ns=2_000_000)
    dev = "cuda"
    xs = [t.to(dev) for t in torch.chunk(inp["x"], P, 0)]
    wr = inp["w_router"].to(dev)
    wg = [t.to(dev) for t in _split(inp["w_gate"], P)]
    wu = [t.to(dev) for t in _split(inp["w_up"], P)]
    wd = [t.to(dev) for t in _split(inp["w_down"], P)]
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    idx = torch.empty(T, topk, dtype=torch.int32, device=dev)
    gate = torch.empty(T, topk, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    pos = torch.empty(T, topk, dtype=torch.int32, device=dev)
    ws = K.moe_workspace(P, T, H, E, topk, I, o)
    K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, counts, pos, ws, topk, o)
    st, entry = K.status_sync(ws)
    assert st == K.ERR_TIMEOUT, (st, entry)
    K.workspace_init(ws)
    K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, counts, pos, ws, topk, K.opts())
    K.check(ws, "moe_fwd after re-init")
    logits = K.moe_debug_view(K.MOE_VIEW_LOGITS, P, T, H, E, topk, I, ws).view(torch.float32).view(T, E)
    out = {"idx": idx.cpu().numpy(), "gate": gate.cpu().numpy(), "logits": logits.cpu().numpy()}
    ref = oracle_experts(orc, inp, kernel_route(out), P)
    assert rel_err(bf16_tensor_to_f64(torch.cat(ys, 0)), ref) <= TOL
