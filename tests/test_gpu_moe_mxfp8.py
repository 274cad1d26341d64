"""GPU parity of the MXFP8 MoE layer (router in bf16; tokens, h and the expert
weights in E4M3 + E8M0 per 32 K) against the oracle's fp64 layer on its own
quantised operands.

Integer and byte work, bit for bit: routing as for the bf16 layer; the
kernel's quantised tokens and scales against the oracle's quantiser; every
dispatched row (codes and tiled scales) against its token, at the padded
position its unpadded dispatch_pos maps to.  Floating output:
max|y - ref| <= 2e-2 * max|ref| over every token, ref = the oracle's layer
run on the kernel's own routing (indices and gates); reruns bit-identical."""
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import pytest
import torch

from _helpers import bf16_tensor_to_f64, kosmos, rel_err
from kosmos_inputs import WORKLOADS, bf16_bits, moe_inputs, per_block_indices
from test_gpu_moe import check_routing, kernel_route

pytestmark = pytest.mark.gpu
TOL = 2e-2


@pytest.fixture(scope="module")
def K():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return kosmos()


def gpu_quant_experts(K, w, P):
    """Per EP rank: E4M3 codes [E/P, Kd, N] and the experts' tiled scales one
    after the other (each expert quantised along its K rows)."""
    E, Kd, N = w.shape
    codes, scales = [], []
    for q in range(P):
        ws = w[q * (E // P):(q + 1) * (E // P)].cuda()
        c = torch.empty(ws.shape, dtype=torch.uint8, device="cuda")
        nb = K.mxfp8_scale_bytes(Kd, N, False)
        s = torch.empty(ws.shape[0] * nb, dtype=torch.uint8, device="cuda")
        for e in range(ws.shape[0]):
            K.mxfp8_quantize(ws[e], c[e], s[e * nb:(e + 1) * nb], False)
        codes.append(c)
        scales.append(s)
    return codes, scales


def run_moe_mx(K, inp, P, topk, o=None, reps=1):
    T, H = inp["x"].shape
    E = inp["w_router"].shape[1]
    I = inp["w_gate"].shape[2]
    dev = "cuda"
    xs = [t.to(dev) for t in torch.chunk(inp["x"], P, 0)]
    wr = inp["w_router"].to(dev)
    (wg, sg), (wu, su), (wd, sd) = (gpu_quant_experts(K, inp[n], P) for n in ("w_gate", "w_up", "w_down"))
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    idx = torch.empty(T, topk, dtype=torch.int32, device=dev)
    gate = torch.empty(T, topk, dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    pos = torch.empty(T, topk, dtype=torch.int32, device=dev)
    ws = K.moe_workspace(P, T, H, E, topk, I, o, dtype=K.MXFP8_E4M3)
    outs = []
    for _ in range(reps):
        for y in ys:
            y.fill_(float("nan"))
        K.moe_fwd(xs, wr, wg, wu, wd, ys, idx, gate, counts, pos, ws, topk, o, dtype=K.MXFP8_E4M3,
                  w_gate_scales=sg, w_up_scales=su, w_down_scales=sd)
        K.check(ws, "moe_fwd mxfp8")
        outs.append(torch.cat(ys, 0).clone())

    def view(what):
        return K.moe_debug_view(what, P, T, H, E, topk, I, ws, dtype=K.MXFP8_E4M3).cpu().numpy()

    logits = view(K.MOE_VIEW_LOGITS).view(np.float32).reshape(T, E)
    return {"y": outs, "idx": idx.cpu().numpy(), "gate": gate.cpu().numpy(), "counts": counts.cpu().numpy(),
            "pos": pos.cpu().numpy(), "logits": logits, "ws": ws, "view": view}


def oracle_quant_experts(orc, w, P, only=None):
    """(codes, row-major scales) per rank from the oracle's quantiser; experts
    outside `only` are left zero (the oracle reads only the selected ones)."""
    E, Kd, N = w.shape
    Eq = E // P
    out = []
    jobs = []
    for q in range(P):
        c = np.zeros((Eq, Kd, N), dtype=np.uint8)
        s = np.zeros((Eq, N, Kd // 32), dtype=np.uint8)
        out.append((c, s))
        jobs += [(q, j) for j in range(Eq) if only is None or q * Eq + j in only]

    def one(job):
        q, j = job
        out[q][0][j], out[q][1][j] = orc.mxfp8_quantize(bf16_bits(w[q * Eq + j]), along_cols=False)

    # the oracle's C quantiser releases the GIL: experts in parallel threads
    with ThreadPoolExecutor(max_workers=min(16, os.cpu_count() or 1)) as ex:
        list(ex.map(one, jobs))
    return out


def oracle_mx(orc, inp, route, P, tokens=None):
    xq, xs = orc.mxfp8_quantize(bf16_bits(inp["x"]), along_cols=True)
    only = None if tokens is None else set(route["idx"][tokens].ravel().tolist())
    packs = [oracle_quant_experts(orc, inp[n], P, only) for n in ("w_gate", "w_up", "w_down")]
    return orc.moe_experts_mxfp8(xq, xs, route["idx"], route["gate"], *packs, tokens=tokens)


def untile(tiled, rows, kblocks):
    r = np.arange(rows)[:, None]
    b = np.arange(kblocks)[None, :]
    off = ((r // 128) * (kblocks // 4) + b // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + (b % 4)
    return tiled[off]


def check_quant_and_dispatch(orc, inp, out, topk):
    T, H = inp["x"].shape
    E = out["counts"].shape[0]
    xq, xs = orc.mxfp8_quantize(bf16_bits(inp["x"]), along_cols=True)
    assert np.array_equal(out["view"](8).reshape(T, H), xq)
    assert np.array_equal(out["view"](9).reshape(T, H // 32), xs)
    counts = out["counts"].astype(np.int64)
    offl = np.concatenate([[0], np.cumsum(counts)])
    offp = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    assert np.array_equal(out["view"](5).view(np.int32)[:E + 1], offp)
    phys = out["pos"] - offl[out["idx"]] + offp[out["idx"]]
    recv = out["view"](1).reshape(-1, H)
    rows = recv.shape[0]
    sf = untile(out["view"](7), rows, H // 32)
    tok = np.repeat(np.arange(T), topk)
    assert np.array_equal(recv[phys.ravel()], xq[tok])
    assert np.array_equal(sf[phys.ravel()], xs[tok])


@pytest.mark.parametrize("P,T,H,E,topk,I", [(4, 512, 512, 64, 4, 256), (2, 400, 256, 64, 8, 128),
                                            (1, 128, 256, 64, 2, 128), (8, 1024, 256, 128, 8, 256)])
def test_moe_mxfp8_small_full_compare(K, orc, P, T, H, E, topk, I):
    inp = moe_inputs(T, H, E, I, seed=700 + T + E + topk)
    out = run_moe_mx(K, inp, P, topk, reps=2)
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), topk)
    check_routing(out, route, topk)
    check_quant_and_dispatch(orc, inp, out, topk)
    ref = oracle_mx(orc, inp, kernel_route(out), P)
    got = bf16_tensor_to_f64(out["y"][0])
    assert not np.isnan(got).any()
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)
    assert torch.equal(out["y"][0], out["y"][1])


def test_moe_mxfp8_empty_expert_and_ragged_blocks(K, orc):
    P, T, H, E, topk, I = 2, 400, 256, 64, 4, 128
    inp = moe_inputs(T, H, E, I, seed=12)
    wr = inp["w_router"].float() * 50.0
    wr[:, 7] = 0.0
    inp["w_router"] = wr.to(torch.bfloat16)
    out = run_moe_mx(K, inp, P, topk)
    assert out["counts"][7] == 0
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), topk)
    check_routing(out, route, topk)
    check_quant_and_dispatch(orc, inp, out, topk)
    ref = oracle_mx(orc, inp, kernel_route(out), P)
    got = bf16_tensor_to_f64(out["y"][0])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)


def test_moe_mxfp8_rejects_identity_injection_and_missing_scales(K):
    P, T, H, E, topk, I = 2, 256, 256, 64, 2, 128
    inp = moe_inputs(T, H, E, I, seed=3)
    with pytest.raises(K.KosmosError):
        run_moe_mx(K, inp, P, topk, o=K.opts(inject=K.INJECT_IDENTITY_EXPERTS))
    dev = "cuda"
    xs = [t.to(dev) for t in torch.chunk(inp["x"], P, 0)]
    w = [torch.zeros(E // P, H, I, dtype=torch.uint8, device=dev) for _ in range(P)]
    ys = [torch.empty(T // P, H, dtype=torch.bfloat16, device=dev) for _ in range(P)]
    z = torch.empty(T, topk, dtype=torch.int32, device=dev)
    ws = K.moe_workspace(P, T, H, E, topk, I, dtype=K.MXFP8_E4M3)
    with pytest.raises(K.KosmosError):
        K.moe_fwd(xs, inp["w_router"].to(dev), w, w, w, ys, z, z.float(), z[:, 0].clone(), z, ws, topk,
                  dtype=K.MXFP8_E4M3)


def test_moe_mxfp8_full_size_sampled(K, orc):
    """2048 tokens, hidden 4096, 128 experts top-8 over 8 EP ranks, inter
    1536, MXFP8: routing and quantised dispatch over every token, outputs on
    two tokens of every 128-token block against the oracle on the kernel's
    routing, bit-identical rerun."""
    w = WORKLOADS["moe_fwd_p8"]
    inp = moe_inputs(w.T, w.H, w.E, w.I, w.seed)
    out = run_moe_mx(K, inp, w.P, w.topk, reps=2)
    assert torch.equal(out["y"][0], out["y"][1])
    route = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), w.topk)
    check_routing(out, route, w.topk)
    check_quant_and_dispatch(orc, inp, out, w.topk)
    tokens = per_block_indices(w.T, 128, 2, seed=5)
    ref = oracle_mx(orc, inp, kernel_route(out), w.P, tokens=tokens)
    got = bf16_tensor_to_f64(out["y"][0][torch.from_numpy(tokens).cuda()])
    assert rel_err(got, ref) <= TOL, rel_err(got, ref)


def test_moe_mxfp8_unfused_phases_match_one_launch(K):
    """MXFP8 layer, unfused baseline (the QUANT entries run in the first
    launch with the router): outputs bit-identical to the one-launch layer."""
    P, T, H, E, topk, I = 4, 512, 512, 64, 4, 256
    inp = moe_inputs(T, H, E, I, seed=41)
    one = run_moe_mx(K, inp, P, topk)
    unf = run_moe_mx(K, inp, P, topk, o=K.opts(sched=K.SCHED_UNFUSED), reps=2)
    assert torch.equal(unf["y"][0], unf["y"][1])
    assert torch.equal(one["y"][0], unf["y"][0])
    assert np.array_equal(one["idx"], unf["idx"]) and np.array_equal(one["pos"], unf["pos"])
