"""GPU parity of the one-launch MoE backward against the oracle's fp64
gradients of the forward layer (top-K routing held fixed).

The oracle runs on the kernel's own routing: the forward's top-K indices and
gates, and its fp32 logits (the router backward's operating point), so every
token and every expert is compared, near-tie tokens included.  Small cases:
dx of every token, dW_gate / dW_up / dW_down of every expert, dW_router;
full size: dx of two tokens per 128-token block, the weight gradients of one
expert per EP rank.  Each within max|got - ref| <= 1e-2 *
max|ref|; reruns bit-identical.  Every assertion message carries the
backward's status word and failing entry."""
import numpy as np
import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
from kosmos_inputs import WORKLOADS, bf16_bits, moe_inputs, per_block_indices
from test_gpu_moe import _split, check_routing, kernel_route

pytestmark = pytest.mark.gpu
TOL = 1e-2


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kosmos()


def dout_for(T, H, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(T, H, generator=g).to(torch.bfloat16)


def run_fwd_bwd(K, inp, dout, P, topk, reps=1, o=None):
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
    fws = K.moe_workspace(P, T, H, E, topk, I)
    K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, counts, pos, fws, topk)
    K.check(fws, "moe_fwd")
    dys = [t.to(dev) for t in torch.chunk(dout, P, 0)]
    dxs = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    dwr = torch.empty(H, E, dtype=torch.float32, device=dev)
    dwg = [torch.empty_like(w) for w in wg]
    dwu = [torch.empty_like(w) for w in wu]
    dwd = [torch.empty_like(w) for w in wd]
    bws = K.moe_bwd_workspace(P, T, H, E, topk, I, o)
    outs = []
    for _ in range(reps):
        for t in dxs + dwg + dwu + dwd + [dwr]:
            t.fill_(float("nan"))
        K.moe_bwd(xs, wr, wg, wu, wd, idx, gate, fws, dys, dxs, dwr, dwg, dwu, dwd, bws, o)
        K.check(bws, "moe_bwd")
        outs.append({"dx": torch.cat(dxs, 0).clone(), "dwr": dwr.clone(), "dwg": torch.cat(dwg, 0).clone(),
                     "dwu": torch.cat(dwu, 0).clone(), "dwd": torch.cat(dwd, 0).clone()})
    logits = K.moe_debug_view(K.MOE_VIEW_LOGITS, P, T, H, E, topk, I, fws).view(torch.float32).view(T, E)
    fwd = {"idx": idx.cpu().numpy(), "gate": gate.cpu().numpy(), "counts": counts.cpu().numpy(),
           "pos": pos.cpu().numpy(), "logits": logits.cpu().numpy()}
    return outs, fwd, bws


def oracle_args(inp, P):
    return ([bf16_bits(w) for w in _split(inp["w_gate"], P)], [bf16_bits(w) for w in _split(inp["w_up"], P)],
            [bf16_bits(w) for w in _split(inp["w_down"], P)])


def diag(K, bws):
    """The backward workspace's status word and failing entry, for assertion
    messages."""
    st, ent = K.status_sync(bws)
    return f"status={K.STATUS_NAMES.get(st, st)} failing_entry={ent}"


def first_diff(a, b):
    d = (a != b) & ~(torch.isnan(a) & torch.isnan(b))
    nz = torch.nonzero(d)
    return "equal" if nz.numel() == 0 else f"{int(d.sum())} differ, first at {tuple(nz[0].tolist())}"


def check_reruns(K, bws, outs):
    for key in ("dx", "dwr", "dwg", "dwu", "dwd"):
        assert torch.equal(outs[0][key], outs[1][key]), \
            f"{key}: reruns differ ({first_diff(outs[0][key], outs[1][key])}); {diag(K, bws)}"


def check_experts(K, bws, orc, got, x, kr, d, wg, wu, wd, experts):
    rg, ru, rd = orc.moe_bwd_experts(x, kr, d, wg, wu, wd, experts)
    sel = torch.tensor(experts)
    for key, r in (("dwg", rg), ("dwu", ru), ("dwd", rd)):
        gk = bf16_tensor_to_f64(got[key][sel])
        err = rel_err(gk, r)
        assert err <= TOL, f"{key}: rel_err {err:.3e} over experts {experts}; {diag(K, bws)}"


@pytest.mark.parametrize("P,T,H,E,topk,I", [(2, 256, 256, 64, 4, 256), (4, 512, 512, 64, 8, 512),
                                            (1, 128, 256, 64, 2, 256), (8, 1024, 256, 128, 8, 256),
                                            (2, 384, 512, 64, 3, 256)])
def test_moe_bwd_small_full_compare(K, orc, P, T, H, E, topk, I):
    inp = moe_inputs(T, H, E, I, seed=900 + T + E + topk)
    dout = dout_for(T, H, seed=T + H)
    outs, fwd, bws = run_fwd_bwd(K, inp, dout, P, topk, reps=2)
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), topk)
    check_routing(fwd, route, topk)
    kr = kernel_route(fwd)
    wg, wu, wd = oracle_args(inp, P)
    x, wr, d = bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), bf16_bits(dout)
    ref = orc.moe_bwd_tokens(x, wr, kr, d, wg, wu, wd)
    got = outs[0]
    for key in ("dx", "dwr", "dwg", "dwu", "dwd"):
        assert not torch.isnan(got[key]).any(), f"{key}: NaN left in the output; {diag(K, bws)}"
    check_reruns(K, bws, outs)
    gx = bf16_tensor_to_f64(got["dx"])
    err = rel_err(gx, ref["dx"])
    assert err <= TOL, f"dx: rel_err {err:.3e}; {diag(K, bws)}"
    check_experts(K, bws, orc, got, x, kr, d, wg, wu, wd, list(range(E)))
    rwr = orc.moe_bwd_router_weight(x, wr, kr, d, wg, wu, wd)
    err = rel_err(got["dwr"].cpu().double().numpy(), rwr)
    assert err <= TOL, f"dwr: rel_err {err:.3e}; {diag(K, bws)}"


def test_moe_bwd_empty_expert_and_ragged_blocks(K, orc):
    """An expert no token selects gets zero weight gradients; token blocks of
    192 rows (a ragged second block)."""
    P, T, H, E, topk, I = 2, 384, 256, 64, 4, 256
    inp = moe_inputs(T, H, E, I, seed=13)
    wr = inp["w_router"].float() * 50.0
    wr[:, 7] = 0.0
    inp["w_router"] = wr.to(torch.bfloat16)
    dout = dout_for(T, H, seed=3)
    outs, fwd, bws = run_fwd_bwd(K, inp, dout, P, topk)
    assert fwd["counts"][7] == 0
    got = outs[0]
    for key in ("dwg", "dwu", "dwd"):
        assert torch.count_nonzero(got[key][7]) == 0, f"{key}; {diag(K, bws)}"
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), topk)
    check_routing(fwd, route, topk)
    kr = kernel_route(fwd)
    wg, wu, wd = oracle_args(inp, P)
    x, d = bf16_bits(inp["x"]), bf16_bits(dout)
    ref = orc.moe_bwd_tokens(x, bf16_bits(inp["w_router"]), kr, d, wg, wu, wd)
    gx = bf16_tensor_to_f64(got["dx"])
    err = rel_err(gx, ref["dx"])
    assert err <= TOL, f"dx: rel_err {err:.3e}; {diag(K, bws)}"
    check_experts(K, bws, orc, got, x, kr, d, wg, wu, wd, list(range(E)))


def test_moe_bwd_trace_every_entry_once(K, orc):
    P, T, H, E, topk, I = 4, 512, 512, 64, 4, 256
    inp = moe_inputs(T, H, E, I, seed=23)
    o = K.opts(trace=1)
    outs, fwd, bws = run_fwd_bwd(K, inp, dout_for(T, H, 4), P, topk, o=o)
    raw = K.moe_bwd_debug_view(K.MOE_BWD_VIEW_TRACE, P, T, H, E, topk, I, bws).cpu().numpy()
    dt = np.dtype([("t_claim", "<i8"), ("t_ready", "<i8"), ("t_done", "<i8"), ("kind", "<i4"),
                   ("ticket", "<i4"), ("cta", "<i4"), ("pad", "<i4")])
    recs = raw.view(dt)
    recs = recs[recs["kind"] != 0]
    counts = fwd["counts"]
    Eq = E // P
    units = [int(sum((counts[q * Eq + j] + 127) // 128 for j in range(Eq))) for q in range(P)]
    RB = (T // P + 127) // 128
    NIC, NHC, NWI, NWH = I // 256, H // 256, I // 128, H // 128
    head = 1 + RB * topk + RB + RB * NHC
    # a DWD / DWGU ticket covers a group of 4 (else 2, else 1) tiles
    W1, W2 = NWI * NHC, NWH * NWI
    grp = lambda w: 4 if w % 4 == 0 else (2 if w % 2 == 0 else 1)
    for q in range(P):
        mine = recs[(recs["cta"] % P) == q]
        main = np.sort(mine["ticket"][np.isin(mine["kind"], list(range(16, 25)))])
        ndwr = len(range(q, NWH, P))
        n_tickets = head + (NIC + NHC) * units[q] + (W1 // grp(W1) + W2 // grp(W2)) * Eq + ndwr
        n_entries = head + (NIC + NHC) * units[q] + (W1 + W2) * Eq + ndwr
        assert np.array_equal(np.unique(main), np.arange(n_tickets)), q
        assert len(main) == n_entries, q
        wg = mine[np.isin(mine["kind"], [22, 23])]
        _, per_ticket = np.unique(wg["ticket"], return_counts=True)
        assert set(per_ticket.tolist()) <= {grp(W1), grp(W2)}, q
    kinds = recs["kind"]
    assert (kinds == 8).sum() == sum(units) * NHC        # one push per DGU tile
    assert (kinds == 9).sum() == P * RB * NHC            # one fold per (token block, column tile)


def test_moe_bwd_full_size_sampled(K, orc):
    """2048 tokens, hidden 4096, 128 experts top-8 over 8 EP ranks, inter
    1536: dx of two tokens per 128-token block and the weight gradients of
    one expert per EP rank (the first and last expert included), against the
    oracle on the kernel's routing; bit-identical rerun.  dW_router is
    compared in the small cases only: at this size the oracle would run the
    backward of every token (minutes of CPU time)."""
    w = WORKLOADS["moe_fwd_p8"]
    inp = moe_inputs(w.T, w.H, w.E, w.I, w.seed)
    dout = dout_for(w.T, w.H, seed=77)
    outs, fwd, bws = run_fwd_bwd(K, inp, dout, w.P, w.topk, reps=2)
    check_reruns(K, bws, outs)
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), w.topk)
    check_routing(fwd, route, w.topk)
    kr = kernel_route(fwd)
    wg, wu, wd = oracle_args(inp, w.P)
    x, wr, d = bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), bf16_bits(dout)
    tokens = per_block_indices(w.T, 128, 2, seed=6)
    ref = orc.moe_bwd_tokens(x, wr, kr, d, wg, wu, wd, tokens=tokens)
    got = bf16_tensor_to_f64(outs[0]["dx"][torch.from_numpy(tokens).cuda()])
    err = rel_err(got, ref["dx"])
    assert err <= TOL, f"dx: rel_err {err:.3e}; {diag(K, bws)}"
    Eq = w.E // w.P
    experts = [0] + [q * Eq + (5 * q + 3) % Eq for q in range(1, w.P - 1)] + [w.E - 1]
    check_experts(K, bws, orc, outs[0], x, kr, d, wg, wu, wd, experts)


def test_moe_bwd_refuses_a_context_that_is_not_a_complete_bf16_forward(K):
    """A forward workspace that no bf16 forward has completed on (a fresh one,
    or one an MXFP8 forward used): the backward reports INVALID_ARG."""
    P, T, H, E, topk, I = 2, 256, 256, 64, 2, 256
    inp = moe_inputs(T, H, E, I, seed=5)
    dev = "cuda"
    xs = [t.to(dev) for t in torch.chunk(inp["x"], P, 0)]
    wr = inp["w_router"].to(dev)
    wg = [t.to(dev) for t in _split(inp["w_gate"], P)]
    wu = [t.to(dev) for t in _split(inp["w_up"], P)]
    wd = [t.to(dev) for t in _split(inp["w_down"], P)]
    idx = torch.zeros(T, topk, dtype=torch.int32, device=dev)
    gate = torch.zeros(T, topk, dtype=torch.float32, device=dev)
    dys = [torch.zeros(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    dxs = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    dwr = torch.empty(H, E, dtype=torch.float32, device=dev)
    dwg, dwu, dwd = [torch.empty_like(w) for w in wg], [torch.empty_like(w) for w in wu], [torch.empty_like(w) for w in wd]
    fresh = K.moe_workspace(P, T, H, E, topk, I)
    bws = K.moe_bwd_workspace(P, T, H, E, topk, I)
    K.moe_bwd(xs, wr, wg, wu, wd, idx, gate, fresh, dys, dxs, dwr, dwg, dwu, dwd, bws)
    st, _ = K.status_sync(bws)
    assert st == K.ERR_INVALID_ARG
    # an MXFP8 forward's workspace (sized for bf16 so that the size check passes)
    K.workspace_init(bws)
    from test_gpu_moe_mxfp8 import gpu_quant_experts
    (qg, sg), (qu, su), (qd, sd) = (gpu_quant_experts(K, inp[n], P) for n in ("w_gate", "w_up", "w_down"))
    fws = K.moe_workspace(P, T, H, E, topk, I, dtype=K.MXFP8_E4M3)
    if fws.numel() < fresh.numel():
        fws = torch.cat([fws, torch.zeros(fresh.numel() - fws.numel(), dtype=torch.uint8, device=dev)])
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    cnt = torch.empty(E, dtype=torch.int32, device=dev)
    pos = torch.empty(T, topk, dtype=torch.int32, device=dev)
    K.moe_fwd(xs, wr, qg, qu, qd, ys, idx, gate, cnt, pos, fws, topk, dtype=K.MXFP8_E4M3, w_gate_scales=sg,
              w_up_scales=su, w_down_scales=sd)
    K.check(fws, "moe_fwd mxfp8")
    K.moe_bwd(xs, wr, wg, wu, wd, idx, gate, fws, dys, dxs, dwr, dwg, dwu, dwd, bws)
    st, _ = K.status_sync(bws)
    assert st == K.ERR_INVALID_ARG


@pytest.mark.parametrize("P,T,H,E,topk,I", [(4, 512, 512, 64, 8, 512), (2, 384, 512, 64, 3, 256)])
def test_moe_bwd_unfused_phases_match_one_launch(K, P, T, H, E, topk, I):
    """The unfused backward runs the same kernel once per phase (head |
    DH | DWD | DGU | DWGU | DWR | push and fold): every gradient equals the
    one-launch backward's bit for bit."""
    inp = moe_inputs(T, H, E, I, seed=960 + T + topk)
    dout = dout_for(T, H, seed=9)
    one, _, bws1 = run_fwd_bwd(K, inp, dout, P, topk)
    unf, _, bws2 = run_fwd_bwd(K, inp, dout, P, topk, reps=2, o=K.opts(sched=K.SCHED_UNFUSED))
    check_reruns(K, bws2, unf)
    for key in ("dx", "dwr", "dwg", "dwu", "dwd"):
        assert torch.equal(one[0][key], unf[0][key]), f"{key}: {first_diff(one[0][key], unf[0][key])}; {diag(K, bws2)}"


def test_moe_rejects_fixed_schedule_and_unfused_trace(K):
    P, T, H, E, topk, I = 2, 256, 256, 64, 2, 256
    inp = moe_inputs(T, H, E, I, seed=6)
    with pytest.raises(K.KosmosError):
        run_fwd_bwd(K, inp, dout_for(T, H, 1), P, topk, o=K.opts(sched=K.SCHED_FIXED))
    with pytest.raises(K.KosmosError):
        run_fwd_bwd(K, inp, dout_for(T, H, 1), P, topk, o=K.opts(sched=K.SCHED_UNFUSED, trace=1))
