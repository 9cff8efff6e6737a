"""Oracle pins for per-channel ring orders and for the direct all-gather mode."""
import itertools

import numpy as np
import pytest

import oracle
from collective_communication_gb300 import inputs as gen
from golden_io import rows

PROTOS = [oracle.LL, oracle.LL128, oracle.SIMPLE]


def page_rings(n):
    return [[int(v) for v in ring.split("-")] for nr, _ch, ring in rows("channel_rings.txt") if int(nr) == n]


def test_page_ring_table_shape():
    r4 = page_rings(4)
    assert len(r4) == 12 and r4[6:] == r4[:6]
    assert sorted(map(tuple, r4[:6])) == sorted((0,) + p for p in itertools.permutations((1, 2, 3)))
    assert all(r == [0, 1] for r in page_rings(2))
    r3 = page_rings(3)
    assert r3.count([0, 1, 2]) == 6 and r3.count([0, 2, 1]) == 6
    for n in (2, 3, 4):
        for ring in page_rings(n):
            oracle.ring_setup(ring)  # every listed order is a valid ring


@pytest.mark.parametrize("proto", PROTOS)
@pytest.mark.parametrize("n", [2, 3, 4])
def test_per_channel_rings_sim_equals_closed(proto, n):
    rings = page_rings(n)
    x = gen.draw("normal", n, 200003, 20 + n, gen.F32)
    outs, *_ = oracle.ring_allreduce_sim(list(x), rings, 0xFFF, proto, 0 if proto != oracle.SIMPLE else 65536)
    closed = oracle.ring_allreduce_closed(list(x), rings, 0xFFF, proto, 0 if proto != oracle.SIMPLE else 65536)
    for o, c in zip(outs, closed):
        assert o.tobytes() == c.tobytes()


def test_per_channel_result_is_each_channels_own_ring():
    """Channel k's elements equal the single-ring result computed with ring k."""
    n, mask = 4, 0xFFF
    rings = page_rings(n)
    x = gen.draw("normal", n, 100000, 7, gen.F32)
    got = oracle.ring_allreduce_closed(list(x), rings, mask, oracle.SIMPLE, 65536)[0]
    geo = oracle.geometry(oracle.SIMPLE, oracle.F32, n, mask, 100000, 65536, 4)
    differs = 0
    for k, (off, cnt) in enumerate(geo["channels"]):
        single = oracle.ring_allreduce_closed(list(x), rings[k], mask, oracle.SIMPLE, 65536)[0]
        assert got[off:off + cnt].tobytes() == single[off:off + cnt].tobytes()
        other = oracle.ring_allreduce_closed(list(x), rings[(k + 1) % 12], mask, oracle.SIMPLE, 65536)[0]
        differs += int(got[off:off + cnt].tobytes() != other[off:off + cnt].tobytes())
    assert differs > 0  # the ring order really changes rounding somewhere


def test_rejects_wrong_ring_count():
    x = gen.draw("normal", 4, 100, 1, gen.F32)
    with pytest.raises(oracle.OracleError):
        oracle.ring_allreduce_closed(list(x), page_rings(4)[:5], 0xFFF, oracle.SIMPLE, 65536)


@pytest.mark.parametrize("seed", range(10))
def test_direct_allgather_sim_equals_closed(seed):
    rng = np.random.default_rng(300 + seed)
    n = int(rng.integers(2, 9))
    dtype = gen.F32 if seed % 2 == 0 else gen.BF16
    mask = int(rng.integers(1, 1 << 6))
    count = int(rng.integers(1, 60000))
    bs = 4096 * int(rng.integers(1, 6))
    cs = int(rng.choice([1, 2, 4]))
    ring = rng.permutation(n).tolist()
    x = gen.draw("normal", n, count, seed, dtype)
    outs, sends, recvs, loops = oracle.ring_allreduce_sim(list(x), ring, mask, oracle.SIMPLE, bs, cs, direct=True)
    closed = oracle.ring_allreduce_closed(list(x), ring, mask, oracle.SIMPLE, bs, cs)
    for o, c in zip(outs, closed):
        assert o.tobytes() == c.tobytes()
    g = oracle.geometry(oracle.SIMPLE, 0 if dtype == gen.F32 else 1, n, mask, count, bs, cs)
    expect = int(loops.sum()) * 2 * (n - 1) * g["slices_per_chunk"]
    assert (sends == expect).all() and (recvs == expect).all()
    # in place
    xin = [a.copy() for a in x]
    oracle.ring_allreduce_sim(xin, ring, mask, oracle.SIMPLE, bs, cs, outputs=xin, direct=True)
    for o, c in zip(xin, closed):
        assert o.tobytes() == c.tobytes()


def test_direct_needs_simple():
    x = gen.draw("normal", 4, 100, 1, gen.F32)
    with pytest.raises(oracle.OracleError):
        oracle.ring_allreduce_sim(list(x), [0, 1, 2, 3], 1, oracle.LL, direct=True)


def test_direct_integer_exact_with_page_rings():
    x = gen.draw("int8", 4, 50000, 3, gen.F32)
    exact = x.astype(np.int64).sum(axis=0).astype(np.float32)
    outs, *_ = oracle.ring_allreduce_sim(list(x), page_rings(4), 0xFFF, oracle.SIMPLE, 65536, direct=True)
    for o in outs:
        assert np.array_equal(o, exact)
