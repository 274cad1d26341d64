"""C-ABI checks that need no GPU: the library builds and loads, exports every
symbol include/kosmos.h declares, validates arguments on the host, and its
rail decode (the same functions the kernels run, compiled for the host)
matches the oracle's independently built rails bit for bit."""
import ctypes as C

import numpy as np
import pytest

from _helpers import header_exports, kosmos


@pytest.fixture(scope="module")
def K():
    return kosmos()


def test_exports_every_declared_symbol(K):
    names = header_exports()
    assert len(names) >= 12
    lib = C.CDLL(K.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(K.EXPORTS) == names


def _header_prototypes():
    """name -> list of parameter declarations, from include/kosmos.h."""
    import os
    import re
    from _helpers import ROOT
    src = open(os.path.join(ROOT, "include", "kosmos.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    out = {}
    for m in re.finditer(r"KOSMOS_API\s+[\w\s\*]+?\b(kosmos_\w+)\s*\(([^)]*)\)\s*;", src):
        params = [p.strip() for p in m.group(2).split(",") if p.strip()]
        out[m.group(1)] = [] if params == ["void"] else params
    return out


def test_binding_argument_lists_match_the_header(K):
    """Every ctypes prototype has the header's parameter count, and 64-bit
    integer / size / pointer parameters line up with the header's types."""
    protos = _header_prototypes()
    assert sorted(protos) == sorted(K.EXPORTS)
    L = K.lib()
    for name, params in protos.items():
        argt = getattr(L, name).argtypes
        if argt is None:
            assert params == [], name
            continue
        assert len(argt) == len(params), (name, len(argt), len(params))
        for a, decl in zip(argt, params):
            if "*" in decl:
                assert a is C.c_void_p or issubclass(a, C._Pointer) or a is C.c_char_p, (name, decl, a)
            elif "int64_t" in decl:
                assert a is C.c_int64, (name, decl, a)
            elif "size_t" in decl:
                assert a is C.c_size_t, (name, decl, a)
            elif decl.split()[0] in ("int", "int32_t"):
                assert a in (C.c_int, C.c_int32), (name, decl, a)


def test_binding_constants_match_the_header(K):
    """Every numeric #define and enum value of include/kosmos.h that the
    binding exposes (under its name without the KOSMOS_ prefix) is equal, and
    every fault-injection bit is exposed."""
    import os
    import re
    from _helpers import ROOT
    src = open(os.path.join(ROOT, "include", "kosmos.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    vals = {}
    for m in re.finditer(r"#define\s+KOSMOS_(\w+)\s+(0x[0-9a-fA-F]+|\d+)(?:ull|u|ll)?\b", src):
        vals[m.group(1)] = int(m.group(2), 0)
    for body in re.findall(r"enum\s*(?:\w+\s*)?\{([^}]*)\}", src):
        for m in re.finditer(r"KOSMOS_(\w+)\s*=\s*(-?(?:0x[0-9a-fA-F]+|\d+))", body):
            vals[m.group(1)] = int(m.group(2), 0)
    inject = [n for n in vals if n.startswith("INJECT_")]
    assert len(inject) >= 5
    for n in inject:
        assert hasattr(K, n), n
    checked = 0
    for n, v in vals.items():
        if hasattr(K, n) and isinstance(getattr(K, n), int):
            assert getattr(K, n) == v, n
            checked += 1
    assert checked >= 15


def test_default_opts(K):
    o = K.opts()
    assert o.sched == K.SCHED_SELF and o.n_comm0 == -1 and o.order == K.ORDER_BAND
    assert o.num_ctas == -1 and o.trace == 0 and o.inject == 0 and o.cta_pair == -1


def test_workspace_sizes(K):
    ag = K.workspace_bytes(K.OP_AG_GEMM, 8, 1024, 3584, 8192)
    assert ag >= 256 + 8 * 8 * 4
    rs = K.workspace_bytes(K.OP_GEMM_RS, 8, 8192, 8192, 3584)
    assert rs >= 8 * 8192 * 8192 * 2  # bf16 partials of every rank
    assert K.workspace_bytes(K.OP_GEMM_RS, 3, 100, 256, 64) == 0  # m % P != 0
    assert K.workspace_bytes(K.OP_AG_GEMM, 9, 64, 64, 64) == 0     # P > 8
    t = K.workspace_bytes(K.OP_AG_GEMM, 8, 1024, 3584, 8192, o=K.opts(trace=1))
    assert t > ag


def test_host_validation_rejects_bad_args(K):
    lib = K.lib()
    P = 2
    buf = (C.c_uint8 * 4096)()
    base = (C.addressof(buf) + 15) // 16 * 16
    xs = (C.c_void_p * P)(base, base)
    # P out of range
    assert lib.kosmos_ag_gemm(xs, None, 0, 64, 128, 128, base, None, 0, base, base, base, 4096, None, None) == 1
    assert lib.kosmos_ag_gemm(xs, None, 9, 64, 128, 128, base, None, 0, base, base, base, 4096, None, None) == 1
    # k not a multiple of 64, n not a multiple of 8
    assert lib.kosmos_ag_gemm(xs, None, P, 64, 100, 128, base, None, 0, base, base, base, 4096, None, None) == 1
    assert lib.kosmos_ag_gemm(xs, None, P, 64, 128, 100, base, None, 0, base, base, base, 4096, None, None) == 1
    # misaligned pointer
    bad = (C.c_void_p * P)(base + 2, base)
    assert lib.kosmos_ag_gemm(bad, None, P, 64, 128, 128, base, None, 0, base, base, base, 4096, None, None) == 1
    # null output
    assert lib.kosmos_ag_gemm(xs, None, P, 64, 128, 128, base, None, 0, base, None, base, 4096, None, None) == 1
    # workspace too small
    assert lib.kosmos_ag_gemm(xs, None, P, 64, 128, 128, base, None, 0, base, base, base, 16, None, None) == 3
    # RS: m not divisible by P
    ys = (C.c_void_p * P)(base, base)
    assert lib.kosmos_gemm_rs(xs, None, xs, None, P, 63, 64, 64, 0, ys, base, 1 << 20, None, None) == 1
    # RS MXFP8 without scales
    assert lib.kosmos_gemm_rs(xs, None, xs, None, P, 256, 128, 64, 1, ys, base, 1 << 20, None, None) == 1
    # quantiser: blocked extent not a multiple of 32
    assert lib.kosmos_mxfp8_quantize(base, 4, 96, 1, base, base, None) == 1
    # emulated link: out of range, or more link time than half the wait bound
    for gbs in (-1, 2000000):
        o = K.opts(link_gbs=gbs)
        assert lib.kosmos_ag_gemm(xs, None, P, 64, 128, 128, base, None, 0, base, base, base, 1 << 20,
                                  C.byref(o), None) == 1
        assert lib.kosmos_gemm_rs(xs, None, xs, None, P, 256, 64, 64, 0, ys, base, 1 << 20, C.byref(o), None) == 1
    o = K.opts(link_gbs=1, wait_limit_ns=1000)  # 16 KB over 1 GB/s = 16 us > 0.5 us
    assert lib.kosmos_ag_gemm(xs, None, P, 64, 128, 128, base, None, 0, base, base, base, 1 << 20,
                              C.byref(o), None) == 1


@pytest.mark.parametrize("split", [0, 3, 76, 10**6])
@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("P,m,n", [(2, 64, 128), (8, 1024, 3584), (3, 200, 264), (1, 5, 8)])
def test_ag_rail_decode_matches_oracle(K, orc, P, m, n, tile_m, split):
    tr, tl = orc.rail_ag(P, m, n, R=128, BN=256, TR=tile_m, PR=32, XS=split)
    assert np.array_equal(K.rail_decode(K.OP_AG_GEMM, P, m, n, rail=0, tile_m=tile_m, split=split), tr)
    assert np.array_equal(K.rail_decode(K.OP_AG_GEMM, P, m, n, rail=1, tile_m=tile_m, split=split), tl)


@pytest.mark.parametrize("tile_m", [128, 256])
@pytest.mark.parametrize("order", [0, 1])
@pytest.mark.parametrize("P,m,n", [(8, 8192, 8192), (3, 600, 520), (1, 128, 256)])
def test_rs_rail_decode_matches_oracle(K, orc, P, m, n, order, tile_m):
    for r in range(P):
        tl, rd = orc.rail_rs(P, m, n, rank=r, order=order, R=tile_m, BN=256)
        assert np.array_equal(K.rail_decode(K.OP_GEMM_RS, P, m, n, rail=0, order=order, rank=r, tile_m=tile_m), tl)
        assert np.array_equal(K.rail_decode(K.OP_GEMM_RS, P, m, n, rail=1, order=order, rank=r, tile_m=tile_m), rd)
