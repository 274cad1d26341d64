"""Pins for the oracle's all-gather+GEMM, GEMM+reduce-scatter and MXFP8 GEMM.

Independent checks: brute-force Python loops on tiny shapes, numpy float64
matmul of the concatenated operands (the closed forms the method reduces to),
unit-vector inputs whose products are exact, and P = 1 reductions."""
import numpy as np
import pytest
import torch

from kosmos_inputs import ag_inputs, bf16_bits, rs_inputs


def _f64(t):
    return t.double().numpy()


def test_ag_bruteforce_tiny(orc):
    inp = ag_inputs(P=2, m=3, k=5, n=4, seed=123, var_w=0.5)
    xs = [bf16_bits(x) for x in inp["x"]]
    y = orc.ag_gemm(xs, bf16_bits(inp["w"]))
    xf = [_f64(x) for x in inp["x"]]
    wf = _f64(inp["w"])
    for g in range(6):
        r, i = divmod(g, 3)
        for j in range(4):
            s = 0.0
            for kk in range(5):
                s += xf[r][i][kk] * wf[kk][j]
            assert abs(y[g, j] - s) <= 1e-12 * max(1.0, abs(s))


@pytest.mark.parametrize("P,m,k,n", [(1, 17, 33, 40), (3, 70, 96, 48), (8, 16, 64, 24)])
def test_ag_equals_gemm_of_concatenation(orc, P, m, k, n):
    inp = ag_inputs(P=P, m=m, k=k, n=n, seed=P * 100 + m, var_w=1.0 / k)
    y = orc.ag_gemm([bf16_bits(x) for x in inp["x"]], bf16_bits(inp["w"]))
    ref = np.concatenate([_f64(x) for x in inp["x"]], axis=0) @ _f64(inp["w"])
    assert y.shape == (P * m, n)
    np.testing.assert_allclose(y, ref, rtol=1e-12, atol=1e-12)


def test_ag_row_subset_matches_full(orc):
    inp = ag_inputs(P=3, m=20, k=32, n=16, seed=9)
    xs = [bf16_bits(x) for x in inp["x"]]
    full = orc.ag_gemm(xs, bf16_bits(inp["w"]))
    rows = np.array([0, 19, 20, 41, 59], dtype=np.int64)
    sub = orc.ag_gemm(xs, bf16_bits(inp["w"]), rows=rows)
    assert np.array_equal(sub, full[rows])


def test_ag_unit_rows_select_w_rows(orc):
    """X rows that are unit vectors e_{c} pick row c of W exactly; shard order
    is checked by giving each shard a different column pattern."""
    P, m, k, n = 3, 4, 8, 5
    w = torch.arange(k * n, dtype=torch.float32).reshape(k, n).to(torch.bfloat16)
    xs = []
    for r in range(P):
        x = torch.zeros(m, k)
        for i in range(m):
            x[i, (r * m + i) % k] = 1.0
        xs.append(x.to(torch.bfloat16))
    y = orc.ag_gemm([bf16_bits(x) for x in xs], bf16_bits(w))
    wf = w.double().numpy()
    for g in range(P * m):
        assert np.array_equal(y[g], wf[g % k])


def test_rs_equals_k_concatenated_gemm(orc):
    P, m, k, n = 4, 24, 40, 32
    inp = rs_inputs(P=P, m=m, k=k, n=n, seed=77, var_w=1.0 / (P * k))
    y = orc.gemm_rs([bf16_bits(x) for x in inp["x"]], [bf16_bits(w) for w in inp["w"]])
    X = np.concatenate([_f64(x) for x in inp["x"]], axis=1)
    W = np.concatenate([_f64(w) for w in inp["w"]], axis=0)
    np.testing.assert_allclose(y, X @ W, rtol=1e-12, atol=1e-12)


def test_rs_single_rank_and_linearity(orc):
    P, m, k, n = 3, 9, 16, 8
    inp = rs_inputs(P=P, m=m, k=k, n=n, seed=5)
    xs = [bf16_bits(x) for x in inp["x"]]
    ws = [bf16_bits(w) for w in inp["w"]]
    # P = 1 is a plain GEMM
    y1 = orc.gemm_rs(xs[:1], ws[:1])
    np.testing.assert_allclose(y1, _f64(inp["x"][0]) @ _f64(inp["w"][0]), rtol=1e-13, atol=1e-13)
    # zeroing every rank but q leaves X_q W_q: a dropped or doubled rank fails
    zero = np.zeros_like(xs[0])
    for q in range(P):
        xz = [xs[r] if r == q else zero for r in range(P)]
        yq = orc.gemm_rs(xz, ws)
        np.testing.assert_allclose(yq, _f64(inp["x"][q]) @ _f64(inp["w"][q]), rtol=1e-13, atol=1e-13)


def test_rs_bruteforce_tiny(orc):
    P, m, k, n = 2, 2, 3, 2
    inp = rs_inputs(P=P, m=m, k=k, n=n, seed=1)
    y = orc.gemm_rs([bf16_bits(x) for x in inp["x"]], [bf16_bits(w) for w in inp["w"]])
    for i in range(m):
        for j in range(n):
            s = 0.0
            for r in range(P):
                for kk in range(k):
                    s += float(inp["x"][r][i, kk]) * float(inp["w"][r][kk, j])
            assert abs(y[i, j] - s) <= 1e-12


def test_mxfp8_gemm_vs_dequantised_numpy(orc):
    P, m, k, n = 2, 12, 64, 16
    inp = ag_inputs(P=P, m=m, k=k, n=n, seed=31, var_w=1.0 / k)
    qx, sx = zip(*[orc.mxfp8_quantize(bf16_bits(x), along_cols=True) for x in inp["x"]])
    qw, sw = orc.mxfp8_quantize(bf16_bits(inp["w"]), along_cols=False)
    y = orc.ag_gemm_mxfp8(list(qx), list(sx), qw, sw)

    def deq(q, s, along_cols):
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
        e = s.astype(np.int64) - 127
        sc = np.repeat(e, 32, axis=1) if along_cols else np.repeat(e, 32, axis=1).T
        return np.ldexp(v, sc)

    X = np.concatenate([deq(q, s, True) for q, s in zip(qx, sx)], axis=0)
    W = deq(qw, sw, False)
    np.testing.assert_allclose(y, X @ W, rtol=1e-12, atol=1e-12)
    # and quantisation error vs the bf16 product is small (sanity of layouts:
    # a transposed scale layout would blow this up)
    ref = np.concatenate([_f64(x) for x in inp["x"]]) @ _f64(inp["w"])
    assert np.max(np.abs(y - ref)) <= 0.1 * np.max(np.abs(ref))


def test_mxfp8_rs_vs_dequantised_numpy_and_bf16_path(orc):
    """MXFP8 RS = sum_r of the dequantised products (numpy, torch's E4M3
    decode); equals the bf16 RS oracle on the dequantised values (exactly
    representable in bf16); a rank-order or scale-layout mistake fails."""
    P, m, k, n = 3, 12, 64, 16
    inp = rs_inputs(P, m, k, n, seed=32, var_w=1.0 / (P * k))
    qx, sx = zip(*[orc.mxfp8_quantize(bf16_bits(x), along_cols=True) for x in inp["x"]])
    qw, sw = zip(*[orc.mxfp8_quantize(bf16_bits(w), along_cols=False) for w in inp["w"]])
    y = orc.gemm_rs_mxfp8(list(qx), list(sx), list(qw), list(sw))

    def deq(q, s, along_cols):
        v = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
        e = s.astype(np.int64) - 127
        sc = np.repeat(e, 32, axis=1) if along_cols else np.repeat(e, 32, axis=1).T
        return np.ldexp(v, sc)

    Xd = [deq(q, s, True) for q, s in zip(qx, sx)]
    Wd = [deq(q, s, False) for q, s in zip(qw, sw)]
    np.testing.assert_allclose(y, sum(a @ b for a, b in zip(Xd, Wd)), rtol=1e-12, atol=1e-12)
    # the dequantised operands are bf16 values: the bf16 oracle gives the same sums
    to_bits = lambda a: torch.from_numpy(a).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert all(np.array_equal(torch.from_numpy(a).to(torch.bfloat16).double().numpy(), a) for a in Xd + Wd)
    y2 = orc.gemm_rs([to_bits(a) for a in Xd], [to_bits(b) for b in Wd])
    np.testing.assert_allclose(y, y2, rtol=1e-13, atol=1e-13)
    rows = np.array([0, 5, 11])
    np.testing.assert_array_equal(orc.gemm_rs_mxfp8(list(qx), list(sx), list(qw), list(sw), rows=rows), y[rows])
