"""Oracle pins on the result of the collective: exact integer sums, hand-derived
association-order values, step simulation == closed form, error bounds."""
import itertools

import numpy as np
import pytest
import torch

import oracle
from collective_communication_gb300 import inputs as gen
from golden_io import rows

PROTOS = [oracle.LL, oracle.LL128, oracle.SIMPLE]
SMALL_BUF = {oracle.SIMPLE: 65536, oracle.LL: 16384, oracle.LL128: 16384}


def dt_code(dtype):
    return oracle.F32 if dtype == gen.F32 else oracle.BF16


def as_f64(a):
    if a.dtype == np.uint16:
        return (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    return a.astype(np.float64)


@pytest.mark.parametrize("proto", PROTOS)
def test_integer_inputs_sum_exactly(proto):
    """4 KiB per rank of integers in [-8, 8], N=4: every ordering of the sum is
    exact, so ring result == the integer sum, for every protocol."""
    case = gen.small_case()
    x = case.inputs()
    exact = x.astype(np.int64).sum(axis=0).astype(np.float32)
    bs = case.buff_size if proto == oracle.SIMPLE else 0
    outs, sends, recvs, loops = oracle.ring_allreduce_sim(list(x), case.ring, case.mask, proto, bs,
                                                          case.chunk_steps)
    for o in outs:
        assert np.array_equal(o, exact)
    closed = oracle.ring_allreduce_closed(list(x), case.ring, case.mask, proto, bs, case.chunk_steps)
    for o in closed:
        assert np.array_equal(o, exact)


def test_ring_order_association_golden():
    g = rows("ring_order_association.txt")
    per_rank = {0: -16777216.0, 1: 1.0, 2: 16777216.0, 3: 1.0}
    x = [np.full(16, per_rank[r], np.float32) for r in range(4)]
    for proto in PROTOS:
        outs, *_ = oracle.ring_allreduce_sim(x, [0, 2, 3, 1], 1, proto)
        closed = oracle.ring_allreduce_closed(x, [0, 2, 3, 1], 1, proto)
        for o in outs + closed:
            for a, b, v in g:
                assert (o[int(a):int(b) + 1] == np.float32(float(v))).all()


def test_oneshot_association_golden():
    (v,), = rows("oneshot_association.txt")
    bits = lambda f: oracle.bf16_round(np.array([f], np.float32))
    x = [bits(256.0), bits(1.0), bits(-256.0), bits(1.0)]
    outs = oracle.oneshot(x)
    for o in outs:
        assert o[0] == bits(float(v))[0]


def test_oneshot_single_rank_is_identity():
    x = gen.draw("normal", 1, 777, 4, gen.BF16)
    (o,) = oracle.oneshot([x[0]])
    assert np.array_equal(o, x[0])


def test_oneshot_integer_bf16_exact():
    x = gen.draw("int8", 8, 5000, 9, gen.BF16)
    outs = oracle.oneshot(list(x))
    exact = as_f64(x).sum(axis=0)
    for o in outs:
        assert np.array_equal(as_f64(o), exact)


def _tiny_cases():
    rng = np.random.default_rng(1234)
    cases = []
    for k in range(40):
        n = int(rng.integers(2, 9))
        proto = PROTOS[k % 3]
        dtype = gen.F32 if (k // 3) % 2 == 0 else gen.BF16
        mask = int(rng.integers(1, 1 << 6))
        count = int(rng.integers(0, 30000)) if k % 5 else int(rng.integers(0, 40))
        bs = {oracle.SIMPLE: 4096 * int(rng.integers(1, 5)), oracle.LL: 4096,
              oracle.LL128: 4096 * int(rng.integers(2, 5))}[proto]
        cs = int(rng.choice([1, 2, 4]))
        ring = rng.permutation(n).tolist()
        cases.append((n, proto, dtype, mask, count, bs, cs, ring, int(rng.integers(0, 1 << 30))))
    return cases


@pytest.mark.parametrize("case", _tiny_cases())
def test_sim_equals_closed_form(case):
    n, proto, dtype, mask, count, bs, cs, ring, seed = case
    x = gen.draw("normal", n, count, seed, dtype)
    outs, sends, recvs, loops = oracle.ring_allreduce_sim(list(x), ring, mask, proto, bs, cs)
    closed = oracle.ring_allreduce_closed(list(x), ring, mask, proto, bs, cs)
    for o, c in zip(outs, closed):
        assert o.tobytes() == c.tobytes()
    # every rank's output is identical
    for o in outs[1:]:
        assert o.tobytes() == outs[0].tobytes()
    # 2(N-1) sends and receives per rank per loop and slice
    g = oracle.geometry(proto, dt_code(dtype), n, mask, count, bs, cs)
    expect = int(loops.sum()) * 2 * (n - 1) * g["slices_per_chunk"]
    assert (sends == expect).all() and (recvs == expect).all()
    # in place gives the same bytes
    xin = [a.copy() for a in x]
    oracle.ring_allreduce_sim(xin, ring, mask, proto, bs, cs, outputs=xin)
    for o, c in zip(xin, closed):
        assert o.tobytes() == c.tobytes()


@pytest.mark.parametrize("dtype", [gen.F32, gen.BF16])
def test_error_bound_against_exact_sum(dtype):
    """f32: |ring - exact| <= N 2^-24 sum|x| (recursive summation bound).
    bf16: the result is the binary32 ring sum rounded once, so it lies within
    half a bf16 ulp of a value that meets the same bound."""
    n = 8
    ring = gen.ring_permutation(n, 3)
    x = gen.draw("normal", n, 50000, 3, dtype)
    (out,) = oracle.ring_allreduce_closed(list(x), ring, 0xFFF, oracle.SIMPLE, 65536, 4)[:1]
    xf = as_f64(x)
    exact = xf.sum(axis=0)
    bound = n * 2.0 ** -24 * np.abs(xf).sum(axis=0)
    got = as_f64(out)
    if dtype == gen.F32:
        assert (np.abs(got - exact) <= bound).all()
    else:
        half_ulp = np.ldexp(1.0, np.frexp(np.abs(got))[1] - 9)
        assert (np.abs(got - exact) <= bound + half_ulp).all()


def test_closed_form_at_samples():
    rng = np.random.default_rng(5)
    for proto in PROTOS:
        for dtype in (gen.F32, gen.BF16):
            n, count, mask = 8, 100003, 0b101101011011
            ring = gen.ring_permutation(n, 5)
            x = gen.draw("normal", n, count, 6, dtype)
            full = oracle.ring_allreduce_closed(list(x), ring, mask, proto, SMALL_BUF[proto], 4)[0]
            idx = np.sort(rng.choice(count, 500, replace=False))
            vals, chunks = oracle.ring_closed_at([xr[idx] for xr in x], ring, mask, proto, idx, count,
                                                 SMALL_BUF[proto], 4)
            assert vals.tobytes() == full[idx].tobytes()
            assert ((chunks >= 0) & (chunks < n)).all()


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(7)
    x = np.concatenate([
        rng.standard_normal(200000).astype(np.float32),
        (rng.standard_normal(20000) * 1e-40).astype(np.float32),  # subnormals
        np.array([1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -(1.0 + 2.0 ** -8), 3.3895314e38, 3.4e38,
                  np.inf, -np.inf, 0.0, -0.0, 2.0 ** -126], np.float32),
        rng.integers(0, 2 ** 32, 100000, dtype=np.uint64).astype(np.uint32).view(np.float32),
    ])
    ours = oracle.bf16_round(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    fin = np.isfinite(x) | np.isinf(x)
    assert np.array_equal(ours[fin], ref[fin])
    nan = np.isnan(x)
    ob = (ours[nan].astype(np.uint32) << 16).view(np.float32)
    assert np.isnan(ob).all()


@pytest.mark.parametrize("n", [2, 4, 8])
def test_chunk_steps_8_deadlocks(n):
    """With chunkSteps = NCCL_STEPS = 8 one chunk fills a connector's whole
    credit window: sending slice (s, k) then needs the next rank to have
    received its own slice (s, k) first, around the whole ring -- a cycle. The
    simulation must report the deadlock (the library refuses chunkSteps 8)."""
    x = gen.draw("normal", n, 4096, 1, gen.F32)
    with pytest.raises(oracle.OracleError) as e:
        oracle.ring_allreduce_sim(list(x), list(range(n)), 1, oracle.SIMPLE, 65536, 8)
    assert e.value.code == oracle.EDEADLOCK
    # chunkSteps 4 on the same input completes
    oracle.ring_allreduce_sim(list(x), list(range(n)), 1, oracle.SIMPLE, 65536, 4)
