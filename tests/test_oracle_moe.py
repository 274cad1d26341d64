"""Pins for the oracle's MoE layer: top-k (brute force over subsets, ties),
dispatch tables (definitions, bijection), router (numpy softmax), identity
experts (out = token * sum of gates) and the E = P = 1, top-1 reduction to a
dense SwiGLU MLP."""
import itertools

import numpy as np
import pytest
import torch

from kosmos_inputs import bf16_bits, moe_inputs


def _order_key(vals, e):
    # larger value first, equal values: lower index first
    return (-vals[e], e)


def _brute_topk(vals, K):
    E = len(vals)
    winners = []
    for S in itertools.combinations(range(E), K):
        rest = [e for e in range(E) if e not in S]
        if all(_order_key(vals, a) < _order_key(vals, b) for a in S for b in rest):
            winners.append(S)
    assert len(winners) == 1
    return sorted(winners[0], key=lambda e: _order_key(vals, e))


def test_topk_bruteforce_with_ties(orc):
    rng = np.random.default_rng(0)
    for trial in range(200):
        E = int(rng.integers(2, 11))
        K = int(rng.integers(1, E + 1))
        vals = rng.integers(-3, 4, size=E).astype(np.float32)  # many ties
        got = orc.topk_f32(vals[None, :], K)[0]
        assert list(got) == _brute_topk(vals, K), (vals, K)


def test_topk_hand_ties(orc):
    s = np.array([[1.0, 2.0, 2.0, 0.5, 2.0]], dtype=np.float32)
    assert list(orc.topk_f32(s, 2)[0]) == [1, 2]
    assert list(orc.topk_f32(s, 4)[0]) == [1, 2, 4, 0]
    s = np.zeros((1, 6), dtype=np.float32)
    assert list(orc.topk_f32(s, 3)[0]) == [0, 1, 2]


def test_dispatch_tables_definition(orc):
    rng = np.random.default_rng(1)
    T, E, K = 50, 12, 3
    idx = np.stack([rng.permutation(E)[:K] for _ in range(T)]).astype(np.int32)
    counts, offsets, pos = orc.moe_dispatch_tables(idx, E)
    assert counts.sum() == T * K
    assert np.array_equal(counts, np.bincount(idx.ravel(), minlength=E))
    assert offsets[0] == 0 and np.array_equal(offsets[1:], np.cumsum(counts)[:-1])
    # bijection onto 0..T*K-1
    assert np.array_equal(np.sort(pos.ravel()), np.arange(T * K))
    # receive order: expert ascending, then token ascending
    order = sorted(((int(idx[t, k]), t, k) for t in range(T) for k in range(K)))
    for p, (e, t, k) in enumerate(order):
        assert pos[t, k] == p


def test_dispatch_tables_empty_expert(orc):
    idx = np.array([[0, 2], [2, 0], [0, 2]], dtype=np.int32)
    counts, offsets, pos = orc.moe_dispatch_tables(idx, 4)
    assert list(counts) == [3, 0, 3, 0]
    assert list(offsets) == [0, 3, 3, 6]
    assert pos.tolist() == [[0, 3], [4, 1], [2, 5]]


def _small_moe(T=24, H=32, E=8, I=16, seed=42):
    return moe_inputs(T=T, H=H, E=E, I=I, seed=seed)


def test_route_vs_numpy(orc):
    inp = _small_moe()
    K = 3
    r = orc.moe_route(bf16_bits(inp["x"]), bf16_bits(inp["w_router"]), K)
    X = inp["x"].double().numpy()
    Wr = inp["w_router"].double().numpy()
    L = X @ Wr
    np.testing.assert_allclose(r["logits"], L, rtol=1e-12, atol=1e-12)
    p = np.exp(L - L.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    for t in range(L.shape[0]):
        order = sorted(range(L.shape[1]), key=lambda e: (-L[t, e], e))[:K]
        assert list(r["idx"][t]) == order
        g = p[t, order] / p[t, order].sum()
        np.testing.assert_allclose(r["gate"][t], g, rtol=1e-12)
    np.testing.assert_allclose(r["gate"].sum(axis=1), 1.0, rtol=1e-13)
    assert r["counts"].sum() == L.shape[0] * K


def _split_ranks(w, P):
    E = w.shape[0]
    return [bf16_bits(w[q * (E // P):(q + 1) * (E // P)]) for q in range(P)]


def test_identity_experts_return_token_times_gate_sum(orc):
    inp = _small_moe()
    K, P, E = 3, 2, 8
    x = bf16_bits(inp["x"])
    r = orc.moe_route(x, bf16_bits(inp["w_router"]), K)
    out = orc.moe_experts(x, r["idx"], r["gate"], _split_ranks(inp["w_gate"], P),
                          _split_ranks(inp["w_up"], P), _split_ranks(inp["w_down"], P),
                          E=E, identity=True)
    X = inp["x"].double().numpy()
    np.testing.assert_allclose(out, X * r["gate"].sum(axis=1, keepdims=True), rtol=1e-14, atol=1e-14)
    np.testing.assert_allclose(out, X, rtol=1e-13, atol=1e-13)


def test_single_expert_top1_is_dense_swiglu(orc):
    T, H, I = 10, 24, 20
    inp = moe_inputs(T=T, H=H, E=1, I=I, seed=3)
    x = bf16_bits(inp["x"])
    r = orc.moe_route(x, bf16_bits(inp["w_router"]), 1)
    assert np.all(r["idx"] == 0) and np.allclose(r["gate"], 1.0)
    out = orc.moe_experts(x, r["idx"], r["gate"], [bf16_bits(inp["w_gate"])],
                          [bf16_bits(inp["w_up"])], [bf16_bits(inp["w_down"])], E=1)
    X = torch.from_numpy(inp["x"].double().numpy())
    g = X @ inp["w_gate"][0].double()
    u = X @ inp["w_up"][0].double()
    ref = (torch.nn.functional.silu(g) * u) @ inp["w_down"][0].double()
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-11, atol=1e-12)


def test_experts_vs_numpy_per_token(orc):
    inp = _small_moe(T=12, H=16, E=4, I=8, seed=8)
    K, P, E = 2, 2, 4
    x = bf16_bits(inp["x"])
    r = orc.moe_route(x, bf16_bits(inp["w_router"]), K)
    tokens = np.array([0, 5, 11], dtype=np.int64)
    out = orc.moe_experts(x, r["idx"], r["gate"], _split_ranks(inp["w_gate"], P),
                          _split_ranks(inp["w_up"], P), _split_ranks(inp["w_down"], P),
                          E=E, tokens=tokens)
    X = inp["x"].double()
    for s, t in enumerate(tokens):
        acc = torch.zeros(X.shape[1], dtype=torch.float64)
        for kk in range(K):
            e = int(r["idx"][t, kk])
            h = torch.nn.functional.silu(X[t] @ inp["w_gate"][e].double()) * (X[t] @ inp["w_up"][e].double())
            acc += r["gate"][t, kk] * (h @ inp["w_down"][e].double())
        np.testing.assert_allclose(out[s], acc.numpy(), rtol=1e-11, atol=1e-12)


# -- MXFP8 experts ---------------------------------------------------------

def _quant_experts(orc, w, P):
    """Per EP rank: (codes [E/P, K, N], scales [E/P, N, K/32]), each expert
    quantised along its K (row) dimension."""
    E = w.shape[0]
    out = []
    for q in range(P):
        qs = [orc.mxfp8_quantize(bf16_bits(w[e]), along_cols=False) for e in range(q * (E // P), (q + 1) * (E // P))]
        out.append((np.stack([a for a, _ in qs]), np.stack([b for _, b in qs])))
    return out


def _deq_rows(codes, scales):
    """codes [R, C] with one scale per row and 32 columns (scales [R, C/32])."""
    v = torch.from_numpy(np.ascontiguousarray(codes)).view(torch.float8_e4m3fn).double().numpy()
    return v * np.exp2(np.repeat(scales.astype(np.float64) - 127.0, 32, axis=1))


def _mx_round_blocks(h):
    """MXFP8 rounding of a vector in blocks of 32, restated with numpy and
    torch's E4M3 cast: 2^e with e the smallest integer such that
    blockmax <= 448 * 2^e, elements rounded to E4M3 at that scale."""
    out = np.empty_like(h)
    for b in range(0, len(h), 32):
        blk = h[b:b + 32]
        mx = np.abs(blk).max()
        if mx == 0.0:
            out[b:b + 32] = 0.0
            continue
        e = int(np.ceil(np.log2(mx / 448.0)))
        while mx > 448.0 * 2.0 ** e:
            e += 1
        while mx <= 448.0 * 2.0 ** (e - 1):
            e -= 1
        v = torch.from_numpy(blk / 2.0 ** e).to(torch.float8_e4m3fn).double().numpy()
        out[b:b + 32] = v * 2.0 ** e
    return out


def test_mxfp8_experts_vs_numpy(orc):
    """Every step restated: E4M3 decode by torch's float8 type, scales as
    powers of two, h rounded to MXFP8 per 32 intermediate columns."""
    T, H, E, I, K, P = 10, 64, 4, 96, 2, 2
    inp = moe_inputs(T=T, H=H, E=E, I=I, seed=21)
    x = bf16_bits(inp["x"])
    r = orc.moe_route(x, bf16_bits(inp["w_router"]), K)
    xq, xs = orc.mxfp8_quantize(x, along_cols=True)
    wg, wu, wd = (_quant_experts(orc, inp[n], P) for n in ("w_gate", "w_up", "w_down"))
    tokens = np.array([0, 3, 9], dtype=np.int64)
    out = orc.moe_experts_mxfp8(xq, xs, r["idx"], r["gate"], wg, wu, wd, tokens=tokens)
    X = _deq_rows(xq, xs)
    Eq = E // P

    def wdeq(pack, e):
        codes, scales = pack[e // Eq][0][e % Eq], pack[e // Eq][1][e % Eq]
        return _deq_rows(codes.T, scales).T  # scales run along the K rows of [K, N]

    for s, t in enumerate(tokens):
        acc = np.zeros(H)
        for kk in range(K):
            e = int(r["idx"][t, kk])
            g = X[t] @ wdeq(wg, e)
            u = X[t] @ wdeq(wu, e)
            h = _mx_round_blocks(g / (1.0 + np.exp(-g)) * u)
            acc += r["gate"][t, kk] * (h @ wdeq(wd, e))
        np.testing.assert_allclose(out[s], acc, rtol=1e-10, atol=1e-12)


def test_mxfp8_experts_close_to_bf16_layer_on_dequantised_inputs(orc):
    """The dequantised E4M3 x 2^e operands are exact bf16 values, so the bf16
    layer on them differs from the MXFP8 layer only by the rounding of h
    (at most 1/16 of each element)."""
    T, H, E, I, K, P = 16, 64, 8, 64, 3, 2
    inp = moe_inputs(T=T, H=H, E=E, I=I, seed=22)
    x = bf16_bits(inp["x"])
    r = orc.moe_route(x, bf16_bits(inp["w_router"]), K)
    xq, xs = orc.mxfp8_quantize(x, along_cols=True)
    packs = [_quant_experts(orc, inp[n], P) for n in ("w_gate", "w_up", "w_down")]
    mx = orc.moe_experts_mxfp8(xq, xs, r["idx"], r["gate"], *packs)

    def to_bf16_bits(a):
        t = torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16)
        assert np.array_equal(t.double().numpy(), a), "dequantised value not exact in bf16"
        return t.view(torch.int16).numpy().view(np.uint16)

    xb = to_bf16_bits(_deq_rows(xq, xs))
    wb = [[to_bf16_bits(np.stack([_deq_rows(c.T, s).T for c, s in zip(codes, scales)])) for codes, scales in pack]
          for pack in packs]
    ref = orc.moe_experts(xb, r["idx"], r["gate"], wb[0], wb[1], wb[2], E=E)
    err = np.abs(mx - ref).max() / np.abs(ref).max()
    assert 1e-4 < err < 0.06, err  # h rounding is visible, and bounded


# -- backward --------------------------------------------------------------

def _torch_layer(x, wr, wg, wu, wd, idx, K):
    """The forward layer restated in torch fp64 with the top-K indices held
    fixed (the routing decision is not differentiated)."""
    logits = x @ wr
    p = torch.softmax(logits, dim=1)
    sel = torch.gather(p, 1, idx)
    gate = sel / sel.sum(dim=1, keepdim=True)
    out = torch.zeros_like(x)
    for k in range(K):
        e = idx[:, k]
        g = torch.einsum("th,thi->ti", x, wg[e])
        u = torch.einsum("th,thi->ti", x, wu[e])
        y = torch.einsum("ti,tih->th", torch.nn.functional.silu(g) * u, wd[e])
        out = out + gate[:, k:k + 1] * y
    return out


def _bwd_case(T=12, H=32, E=8, I=16, K=3, P=2, seed=51):
    inp = moe_inputs(T=T, H=H, E=E, I=I, seed=seed)
    g = torch.Generator().manual_seed(seed + 1)
    dout = (torch.randn(T, H, generator=g)).to(torch.bfloat16)
    return inp, dout, K, P


def test_moe_bwd_vs_torch_autograd(orc):
    inp, dout, K, P = _bwd_case()
    E = inp["w_router"].shape[1]
    x = bf16_bits(inp["x"])
    r = orc.moe_route(x, bf16_bits(inp["w_router"]), K)
    wg, wu, wd = (_split_ranks(inp[n], P) for n in ("w_gate", "w_up", "w_down"))
    tok = orc.moe_bwd_tokens(x, bf16_bits(inp["w_router"]), r, bf16_bits(dout), wg, wu, wd)
    dwg, dwu, dwd = orc.moe_bwd_experts(x, r, bf16_bits(dout), wg, wu, wd, np.arange(E))
    dwr = orc.moe_bwd_router_weight(x, bf16_bits(inp["w_router"]), r, bf16_bits(dout), wg, wu, wd)
    leaves = {n: inp[n].double().clone().requires_grad_(True) for n in ("x", "w_router", "w_gate", "w_up", "w_down")}
    idx = torch.from_numpy(r["idx"].astype(np.int64))
    out = _torch_layer(leaves["x"], leaves["w_router"], leaves["w_gate"], leaves["w_up"], leaves["w_down"], idx, K)
    (out * dout.double()).sum().backward()
    np.testing.assert_allclose(tok["dx"], leaves["x"].grad.numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dwr, leaves["w_router"].grad.numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dwg, leaves["w_gate"].grad.numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dwu, leaves["w_up"].grad.numpy(), rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(dwd, leaves["w_down"].grad.numpy(), rtol=1e-9, atol=1e-12)


def test_moe_bwd_finite_differences(orc):
    """Central differences of <dout, out(x + eps v)> with the routing fixed
    match <dx, v>; likewise for one expert's W_down and the router."""
    inp, dout, K, P = _bwd_case(T=10, H=24, E=8, I=16, K=2, seed=52)
    x = bf16_bits(inp["x"])
    r = orc.moe_route(x, bf16_bits(inp["w_router"]), K)
    wg, wu, wd = (_split_ranks(inp[n], P) for n in ("w_gate", "w_up", "w_down"))
    tok = orc.moe_bwd_tokens(x, bf16_bits(inp["w_router"]), r, bf16_bits(dout), wg, wu, wd)
    dwr = orc.moe_bwd_router_weight(x, bf16_bits(inp["w_router"]), r, bf16_bits(dout), wg, wu, wd)
    e0 = int(r["idx"][0, 0])
    _, _, dwd = orc.moe_bwd_experts(x, r, bf16_bits(dout), wg, wu, wd, [e0])
    idx = torch.from_numpy(r["idx"].astype(np.int64))
    base = {n: inp[n].double() for n in ("x", "w_router", "w_gate", "w_up", "w_down")}
    D = dout.double()
    L = lambda t: float((_torch_layer(t["x"], t["w_router"], t["w_gate"], t["w_up"], t["w_down"], idx, K) * D).sum())
    g = torch.Generator().manual_seed(9)
    eps = 1e-6
    for name, grad in (("x", tok["dx"]), ("w_router", dwr)):
        v = torch.randn(base[name].shape, generator=g, dtype=torch.float64)
        plus = dict(base); plus[name] = base[name] + eps * v
        minus = dict(base); minus[name] = base[name] - eps * v
        fd = (L(plus) - L(minus)) / (2 * eps)
        assert abs(fd - float((torch.from_numpy(grad) * v).sum())) <= 1e-6 * max(1.0, abs(fd)), name
    v = torch.randn(base["w_down"].shape[1:], generator=g, dtype=torch.float64)
    plus = dict(base); plus["w_down"] = base["w_down"].clone(); plus["w_down"][e0] += eps * v
    minus = dict(base); minus["w_down"] = base["w_down"].clone(); minus["w_down"][e0] -= eps * v
    fd = (L(plus) - L(minus)) / (2 * eps)
    assert abs(fd - float((torch.from_numpy(dwd[0]) * v).sum())) <= 1e-6 * max(1.0, abs(fd))
