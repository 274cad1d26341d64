"""Pins for the oracle's rails: every entry appears exactly once, and the
order follows consumer demand (the explainer's queue-order paragraph):
  * AG: remote transfers are ordered by the first tile that consumes them, the
    local shard's tiles come first, and no tile's input is transferred after a
    later tile's input;
  * RS band order: band b of every rank and chunk before band b+1, one rank
    at a time inside a band; row order finishes chunk c before chunk c+1."""
import numpy as np
import pytest


@pytest.mark.parametrize("PR", [32, 128])
@pytest.mark.parametrize("P,m,n", [(2, 64, 128), (8, 1024, 3584), (3, 320, 200)])
def test_ag_rail_exactly_once_and_demand_order(orc, P, m, n, PR):
    R, BN = 128, 256
    tr_all, tl = orc.rail_ag(P, m, n, R=R, BN=BN, PR=PR)
    pieces = -(-m // R)
    parts = R // PR
    tn = -(-n // BN)
    assert len(tr_all) == P * pieces * parts
    assert len({tuple(e) for e in tr_all}) == len(tr_all)
    assert set(tr_all[:, 3].tolist()) == set(range(parts))
    # the parts of one piece are adjacent and in row order; dropping the part
    # field leaves the piece rail
    assert np.array_equal(tr_all[:, 3], np.tile(np.arange(parts), P * pieces))
    tr = tr_all[::parts]
    assert np.array_equal(np.repeat(tr[:, 1:3], parts, axis=0), tr_all[:, 1:3])
    assert len(tl) == P * pieces * tn
    assert len({tuple(e) for e in tl}) == len(tl)
    assert np.all(tr[:, 0] == 1) and np.all(tl[:, 0] == 2)
    # local shard tiles first
    assert np.all(tl[: pieces * tn, 1] == 0)
    # first consumer ticket of each remote transfer is non-decreasing along the rail
    first = {}
    for t, (_, s, i, c) in enumerate(tl):
        first.setdefault((int(s), int(i)), t)
    remote = [(int(s), int(j)) for (_, s, j, _) in tr if s != 0]
    cons = [first[x] for x in remote]
    assert cons == sorted(cons)
    # the local shard's own copies come last (nothing waits on them)
    assert all(int(s) == 0 for (_, s, _, _) in tr[len(remote):])


@pytest.mark.parametrize("P,m,n", [(8, 8192, 8192), (3, 768, 520)])
@pytest.mark.parametrize("order", [0, 1])
def test_rs_rails(orc, order, P, m, n):
    R, BN = 128, 256
    bands = -(-(m // P) // R)
    tn = -(-n // BN)
    tl = None
    for r in range(P):
        t_r, rd = orc.rail_rs(P, m, n, rank=r, order=order, R=R, BN=BN)
        if tl is None:
            tl = t_r
        assert np.array_equal(t_r, tl)  # one tile rail for every rank
        assert len(rd) == bands * tn and len({tuple(e) for e in rd}) == len(rd)
        assert np.all(rd[:, 1] == r)
        # the reduce rail follows the order in which its chunk's tiles complete:
        # the last of the P partials of (chunk r, b, j) moves forward along it
        pos = {(int(a), int(b), int(j)): t for t, (_, a, b, j) in enumerate(tl)}
        last = [max(pos[(q * P + r, int(b), int(j))] for q in range(P)) for (_, _, b, j) in rd]
        assert last == sorted(last)
    q, c = tl[:, 1] // P, tl[:, 1] % P
    assert len(tl) == P * P * bands * tn and len({tuple(e) for e in tl}) == len(tl)
    assert set(q.tolist()) == set(range(P)) and set(c.tolist()) == set(range(P))
    if order == 0:
        # band-major; inside a band one rank at a time; chunk innermost
        key = tl[:, 2] * P + q
        assert list(key) == sorted(key)
        assert np.array_equal(c, np.tile(np.arange(P), len(tl) // P))
        # every chunk's band 0 is complete after the first P*P*tn tickets
        assert np.all(tl[: P * P * tn, 2] == 0)
    else:
        key = (c * bands + tl[:, 2]) * P + q
        assert list(key) == sorted(key)


def test_rs_rail_rejects_indivisible(orc):
    with pytest.raises(ValueError):
        orc.rail_rs(3, 100, 256, rank=0, order=0)


def test_ag_rail_rejects_uneven_parts(orc):
    with pytest.raises(ValueError):
        orc.rail_ag(2, 64, 128, R=128, PR=48)


@pytest.mark.parametrize("P,m,n,TR,XS", [(8, 1024, 3584, 256, 76), (3, 320, 200, 128, 5), (2, 64, 128, 128, 99),
                                         (4, 512, 520, 256, 0)])
def test_ag_rail_tail_halves_cover_every_output_once(orc, P, m, n, TR, XS):
    """The split rail keeps the unsplit prefix, replaces only the last XS
    tiles by their two K halves (adjacent, first half first), and covers
    every (output element, K half) exactly once."""
    BN = 256
    _, full = orc.rail_ag(P, m, n, TR=TR, BN=BN)
    _, tl = orc.rail_ag(P, m, n, TR=TR, BN=BN, XS=XS)
    xs = min(XS, len(full))
    keep = len(full) - xs
    assert np.array_equal(tl[:keep], full[:keep])
    assert len(tl) == keep + 2 * xs
    halves = tl[keep:]
    assert np.all(halves[:, 0] == 10)
    assert np.array_equal(halves[0::2, 1:3], full[keep:, 1:3])
    assert np.array_equal(halves[1::2, 1:3], full[keep:, 1:3])
    assert np.array_equal(halves[0::2, 3], 2 * full[keep:, 3])
    assert np.array_equal(halves[1::2, 3], 2 * full[keep:, 3] + 1)
    cover = np.zeros((P, -(-m // TR) * TR, -(-n // BN) * BN, 2), dtype=np.int32)
    for kind, s, i, c in tl:
        if kind == 2:
            cover[s, i * TR:(i + 1) * TR, c * BN:(c + 1) * BN, :] += 1
        else:
            cover[s, i * TR:(i + 1) * TR, (c // 2) * BN:(c // 2 + 1) * BN, c % 2] += 1
    assert np.all(cover == 1)
