"""Pins of the oracle's ReduceScatter and AllGather (the two halves of the
ring AllReduce run as collectives of their own).

The pages state AllReduce = ReduceScatter + AllGather and print rank 0's
seven rows with the phase of each ("NCCL 专家课程 12", sections
"Ring AllReduce 不只是“绕一圈”", "rank0 的完整操作序列", "源码步骤三"); the
collectives' shapes (ReduceScatter: nranks blocks in, the rank's own block
out; AllGather: one block in, all blocks out) are the plain reading. Pins:
the page's rows, exact sums of integer-valued inputs, the composition
AllGather(ReduceScatter(x)) == AllReduce(x), the start of the fold taken from
the page's first-send table, and the step simulation against the closed form.
"""
import numpy as np
import pytest

import oracle
from golden_io import rows

PRIM = {v: k for k, v in oracle.PRIM_NAMES.items()}


def _bits(a):
    return a.view(np.uint32) if a.dtype == np.float32 else a


def _same(xs, ys):
    return all(np.array_equal(_bits(x), _bits(y)) for x, y in zip(xs, ys))


def _int_inputs(rng, n, size, dtype, lo=-8, hi=9):
    vals = [rng.integers(lo, hi, size).astype(np.float32) for _ in range(n)]
    if dtype == "bf16":
        return [oracle.bf16_round(v) for v in vals], vals
    return vals, vals


def _normal_inputs(rng, n, size, dtype):
    vals = [rng.standard_normal(size).astype(np.float32) for _ in range(n)]
    return [oracle.bf16_round(v) for v in vals] if dtype == "bf16" else vals


def test_rows_are_the_pages_rows_split_at_the_owner():
    # rank 0, ring 0-1-2-3: the page's seven rows are ReduceScatter (rows 0-2),
    # the fused owner row (3), AllGather (rows 4-6)
    page = rows("rank0_schedule.txt")
    assert [r[1] for r in page] == ["RS", "RS", "RS", "fused", "AG", "AG", "AG"]
    chunks = [int(r[3]) for r in page]
    prims = [PRIM[r[2]] for r in page]
    rs = oracle.schedule_kind(oracle.REDUCE_SCATTER, 4, 0)
    ag = oracle.schedule_kind(oracle.ALL_GATHER, 4, 0)
    assert [c for _, c in rs] == chunks[:4]
    assert [c for _, c in ag] == chunks[3:]
    # the halves keep the page's primitives, except the owner row: its
    # recv+reduce ends ReduceScatter and its send starts AllGather
    assert [p for p, _ in rs] == prims[:3] + [oracle.RECV_REDUCE_COPY]
    assert [p for p, _ in ag] == [oracle.COPY_SEND] + prims[4:]


@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_rows_of_every_ring_index(n):
    for i in range(n):
        full = []
        prim = np.zeros(2 * n, np.int32)
        chunk = np.zeros(2 * n, np.int32)
        assert oracle.lib().orc_schedule(n, i, oracle._ptr(prim), oracle._ptr(chunk)) == 0
        full = list(zip(prim[:2 * n - 1].tolist(), chunk[:2 * n - 1].tolist()))
        rs = oracle.schedule_kind(oracle.REDUCE_SCATTER, n, i)
        ag = oracle.schedule_kind(oracle.ALL_GATHER, n, i)
        assert len(rs) == len(ag) == n
        assert [c for _, c in rs] == [c for _, c in full[:n]]
        assert [c for _, c in ag] == [c for _, c in full[n - 1:]]
        # ReduceScatter ends with the rank's own chunk; AllGather starts with it
        assert rs[-1][1] == i and ag[0][1] == i
        # every chunk once per half
        assert sorted(c for _, c in rs) == list(range(n)) == sorted(c for _, c in ag)


def test_first_send_sets_the_start_of_the_fold():
    """The page's first-send table (ring 0-1-2-3): rank q sends chunk f(q)
    first, so the partial of block b starts at the rank whose first send is b.
    Put 2**24 there and 1 everywhere else: starting at the big value, every
    later +1 rounds back to 2**24 (ties to even); any other start would leave
    at least 2**24 + 2."""
    first = {int(r[0]): int(r[1]) for r in rows("first_send.txt")}
    n, m = 4, 64
    xs = [np.ones(n * m, np.float32) for _ in range(n)]
    for q, b in first.items():
        xs[q][b * m:(b + 1) * m] = 2.0 ** 24
    for proto in (oracle.SIMPLE, oracle.LL, oracle.LL128):
        out, _, _, _ = oracle.ring_halves_sim(oracle.REDUCE_SCATTER, xs, [0, 1, 2, 3], 0x1, proto,
                                              buff_size=65536)
        for r in range(n):
            assert np.all(out[r] == np.float32(2.0 ** 24)), (proto, r)


CASES = [
    # (n, block elements, mask, proto, buff_size, chunk_steps)
    (4, 1000, 0x3, oracle.SIMPLE, 65536, 4),
    (4, 4096 * 3 + 5, 0x5, oracle.SIMPLE, 65536, 2),
    (8, 777, 0xFF, oracle.SIMPLE, 32768, 1),
    (3, 5000, 0x1, oracle.LL, 32768, 4),
    (5, 3001, 0x6, oracle.LL128, 65536, 4),
    (2, 1, 0x3, oracle.SIMPLE, 65536, 4),
    (8, 3, 0xF0, oracle.LL, 32768, 4),
    (6, 0, 0x3, oracle.SIMPLE, 65536, 4),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", CASES)
def test_reduce_scatter_integer_inputs_give_exact_block_sums(case, dtype):
    n, m, mask, proto, bs, cs = case
    rng = np.random.default_rng(11 + n + m)
    # bf16: integers up to 256 in magnitude are exact, their sums need not
    # be, so the result shows that the binary32 sum is rounded once
    xs, vals = _int_inputs(rng, n, n * m, dtype, *((-200, 201) if dtype == "bf16" else (-8, 9)))
    ring = list(rng.permutation(n))
    out, sends, recvs, loops = oracle.ring_halves_sim(oracle.REDUCE_SCATTER, xs, ring, mask, proto,
                                                      buff_size=bs, chunk_steps=cs)
    for r in range(n):
        exact = np.sum([v[r * m:(r + 1) * m].astype(np.float64) for v in vals], axis=0)
        want = exact.astype(np.float32)
        if dtype == "bf16":
            want = oracle.bf16_round(want)
        assert np.array_equal(_bits(out[r]), _bits(want)), r
    # every rank sends and receives n-1 slices per slice position of a loop
    geo = oracle.geometry(proto, oracle.F32 if dtype == "f32" else oracle.BF16, n, mask, m, bs, cs)
    assert np.all(sends == sends[0]) and np.all(recvs == sends)
    assert sends[0] == loops.sum() * geo["slices_per_chunk"] * (n - 1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", CASES)
def test_all_gather_is_the_concatenation(case, dtype):
    n, m, mask, proto, bs, cs = case
    rng = np.random.default_rng(5 + n + m)
    xs = _normal_inputs(rng, n, m, dtype)
    ring = list(rng.permutation(n))
    want = np.concatenate(xs) if m else np.zeros(0, xs[0].dtype)
    modes = [False, True] if proto == oracle.SIMPLE else [False]
    for direct in modes:
        out, sends, recvs, _ = oracle.ring_halves_sim(oracle.ALL_GATHER, xs, ring, mask, proto,
                                                      buff_size=bs, chunk_steps=cs, direct=direct)
        for r in range(n):
            assert np.array_equal(_bits(out[r]), _bits(want)), (direct, r)
        assert np.all(sends == recvs)
    closed = oracle.ring_halves_closed(oracle.ALL_GATHER, xs, ring, mask, proto, bs, cs)
    assert all(np.array_equal(_bits(c), _bits(want)) for c in closed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("proto,bs", [(oracle.SIMPLE, 65536), (oracle.LL, 32768), (oracle.LL128, 65536)])
@pytest.mark.parametrize("n", [2, 4, 7])
def test_allgather_of_reducescatter_is_allreduce(n, proto, bs, dtype):
    """AllReduce = ReduceScatter + AllGather, bit for bit, where the two cut
    the buffer alike: ring 0..n-1 (chunk c and block c have the same owner),
    one channel, and one loop whose chunk is exactly a block."""
    geo = oracle.geometry(proto, oracle.F32, n, 0x1, 0, bs, 4)
    align = 4 if dtype == "f32" else 8
    m = (min(geo["chunk_elems"], 3000) // align) * align
    rng = np.random.default_rng(n * 100 + proto)
    xs = _normal_inputs(rng, n, n * m, dtype)
    ring = list(range(n))
    ar = oracle.ring_allreduce_closed(xs, ring, 0x1, proto, bs, 4)
    rs, _, _, _ = oracle.ring_halves_sim(oracle.REDUCE_SCATTER, xs, ring, 0x1, proto, buff_size=bs)
    ag, _, _, _ = oracle.ring_halves_sim(oracle.ALL_GATHER, rs, ring, 0x1, proto, buff_size=bs)
    assert _same(ag, ar)


@pytest.mark.parametrize("n", [3, 8])
def test_composition_with_integer_inputs_for_any_ring_and_channels(n):
    rng = np.random.default_rng(n)
    m = 2053
    xs, _ = _int_inputs(rng, n, n * m, "f32")
    rings = [list(rng.permutation(n)) for _ in range(3)]
    ar = oracle.ring_allreduce_closed(xs, rings, 0x0B, oracle.SIMPLE, 65536, 2)
    rs, _, _, _ = oracle.ring_halves_sim(oracle.REDUCE_SCATTER, xs, rings, 0x0B, oracle.SIMPLE,
                                         buff_size=65536, chunk_steps=2)
    ag, _, _, _ = oracle.ring_halves_sim(oracle.ALL_GATHER, rs, rings[::-1], 0x0B, oracle.SIMPLE,
                                         buff_size=65536, chunk_steps=2)
    assert _same(ag, ar)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("case", CASES)
def test_reduce_scatter_sim_matches_closed_form(case, dtype):
    n, m, mask, proto, bs, cs = case
    rng = np.random.default_rng(3 * n + m)
    xs = _normal_inputs(rng, n, n * m, dtype)
    nch = len(oracle.mask_channels(mask))
    rings = [list(rng.permutation(n)) for _ in range(nch)]
    sim, _, _, _ = oracle.ring_halves_sim(oracle.REDUCE_SCATTER, xs, rings, mask, proto,
                                          buff_size=bs, chunk_steps=cs)
    closed = oracle.ring_halves_closed(oracle.REDUCE_SCATTER, xs, rings, mask, proto, bs, cs)
    assert _same(sim, closed)


def test_fold_start_is_visible_in_the_result():
    """The first-send pin can tell fold starts apart: with the big value at
    the owner (the last rank of the fold) instead of the first sender, the
    three +1 come first and the result is 2**24 + 4, not 2**24."""
    n, m = 4, 16
    xs = [np.ones(n * m, np.float32) for _ in range(n)]
    for b in range(n):
        xs[b][b * m:(b + 1) * m] = 2.0 ** 24  # at the owner, not the first sender
    out = oracle.ring_halves_closed(oracle.REDUCE_SCATTER, xs, [0, 1, 2, 3], 0x1, oracle.SIMPLE)
    for r in range(n):
        assert np.all(out[r] == np.float32(2.0 ** 24 + 4))


def test_bad_arguments():
    xs = [np.zeros(8, np.float32) for _ in range(2)]
    with pytest.raises(oracle.OracleError):
        oracle.ring_halves_sim(oracle.REDUCE_SCATTER, xs, [0, 1], 0x1, oracle.SIMPLE, direct=True)
    with pytest.raises(oracle.OracleError):
        oracle.ring_halves_sim(oracle.ALL_GATHER, xs, [0, 1], 0x1, oracle.LL, direct=True)
    with pytest.raises(ValueError):
        oracle.ring_halves_sim(oracle.REDUCE_SCATTER, [np.zeros(9, np.float32)] * 2, [0, 1], 0x1,
                               oracle.SIMPLE)
