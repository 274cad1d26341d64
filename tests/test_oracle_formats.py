"""Pins for the oracle's number formats: bf16 decode, E4M3 codec, MX block scale
and the MXFP8 quantiser.  Every expected value comes from the format
definitions (golden fixture) or from an independent library conversion
(torch's bfloat16 / float8_e4m3fn casts)."""
import json
import os

import numpy as np
import pytest
import torch

GOLD = os.path.join(os.path.dirname(__file__), "golden", "e4m3_mx_cases.json")


def test_bf16_decode_all_patterns(orc):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy().astype(np.float64)
    got = orc.bf16_to_f64(bits)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])
    # sign of zero kept
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_e4m3_golden(orc):
    g = json.load(open(GOLD))
    for c in g["decode"]:
        assert orc.e4m3_to_f64(c["code"]) == c["value"], c
    for c in g["encode"]:
        assert orc.f64_to_e4m3(c["value"]) == c["code"], c
    for c in g["scale_exp"]:
        assert orc.mx_scale_exp(c["blockmax"]) == c["e"], c


def test_e4m3_decode_all_codes_vs_torch(orc):
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    got = np.array([orc.e4m3_to_f64(int(c)) for c in codes])
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], ref[~nan])


def test_e4m3_roundtrip_all_finite_codes(orc):
    for c in range(256):
        v = orc.e4m3_to_f64(c)
        if np.isnan(v):
            continue
        if v == 0.0:
            # +-0 keep their sign bit
            assert orc.f64_to_e4m3(v) == c
            continue
        assert orc.f64_to_e4m3(v) == c, (c, v)


def test_e4m3_encode_vs_torch_rne(orc):
    """Random values across the whole finite range (normal and subnormal),
    plus every exact midpoint between neighbouring codes."""
    rng = np.random.default_rng(5)
    mags = np.exp2(rng.uniform(-12, np.log2(448.0), size=4000))
    vals = np.concatenate([mags, -mags])
    finite = sorted({orc.e4m3_to_f64(c) for c in range(128) if not np.isnan(orc.e4m3_to_f64(c))})
    mids = [(a + b) / 2 for a, b in zip(finite[:-1], finite[1:])]
    vals = np.concatenate([vals, np.array(mids), -np.array(mids)])
    ref = torch.from_numpy(vals).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = np.array([orc.f64_to_e4m3(float(v)) for v in vals], dtype=np.uint8)
    assert np.array_equal(got, ref)


def test_mx_scale_brackets_blockmax(orc):
    rng = np.random.default_rng(11)
    for bm in np.exp2(rng.uniform(-40, 40, size=2000)):
        e = orc.mx_scale_exp(bm)
        assert bm <= 448.0 * 2.0 ** e
        assert bm > 448.0 * 2.0 ** (e - 1)
    for k in range(-20, 21):
        assert orc.mx_scale_exp(448.0 * 2.0 ** k) == k


def _dequant_torch(q, s, along_cols):
    """Independent decode: torch's float8_e4m3fn cast and an exact power of two."""
    vals = torch.from_numpy(q).view(torch.float8_e4m3fn).double().numpy()
    e = s.astype(np.int64) - 127
    if along_cols:
        scale = np.repeat(e, 32, axis=1)
    else:
        scale = np.repeat(e, 32, axis=1).T
    return np.ldexp(vals, scale)


@pytest.mark.parametrize("along_cols", [True, False])
def test_mxfp8_quantize_properties(orc, along_cols):
    rng = np.random.default_rng(3)
    x = torch.from_numpy(rng.standard_normal((64, 96)).astype(np.float32)).to(torch.bfloat16)
    if along_cols:
        x[5, 32:64] = 0.0                 # an all-zero block
        x[6, 0:32] = 0.75                 # a block of equal values
        x[7, 64:96] = torch.tensor(448.0 * 2.0 ** -3)  # blockmax exactly 448 * 2^-3
    else:
        x[32:64, 5] = 0.0
        x[0:32, 6] = 0.75
        x[32:64, 7] = torch.tensor(448.0 * 2.0 ** -3)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    q, s = orc.mxfp8_quantize(bits, along_cols)
    xd = x.double().numpy()
    deq = _dequant_torch(q, s, along_cols)
    # element error of RNE with 3 mantissa bits: half an ulp of the scaled value
    # (relative 2^-4 in the normal range; absolute 2^-10 * 2^e in the subnormal range)
    e = (s.astype(np.int64) - 127)
    ee = np.repeat(e, 32, axis=1) if along_cols else np.repeat(e, 32, axis=1).T
    bound = np.maximum(np.abs(xd) * 2.0 ** -4, 2.0 ** (-10 + ee))
    assert np.all(np.abs(deq - xd) <= bound)
    if along_cols:
        assert s[5, 1] == 127 and np.all(q[5, 32:64] == 0)
        assert np.all(q[6, 0:32] == q[6, 0])
        assert s[7, 2] == 127 - 3 and np.all(q[7, 64:96] == 0x7E)
    else:
        assert s[5, 1] == 127 and np.all(q[32:64, 5] == 0)
        assert np.all(q[0:32, 6] == q[0, 6])
        assert s[7, 1] == 127 - 3 and np.all(q[32:64, 7] == 0x7E)
    # every block's max magnitude lands in (224, 448] after scaling
    blk = np.abs(xd).reshape(64, 3, 32).max(axis=2) if along_cols else \
        np.abs(xd).T.reshape(96, 2, 32).max(axis=2)
    nz = blk > 0
    scaled = blk[nz] / 2.0 ** e[nz]
    assert np.all(scaled <= 448.0) and np.all(scaled > 224.0)
