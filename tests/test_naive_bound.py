"""The naive-sum accuracy check (tests/naive_bound.py) on the oracle's ring
results, on the CPU: the oracle's ring-order fold meets it on every element
(f32 and bf16, N = 2..8, rings, channels and protocols as in the workloads),
integer inputs give the naive sum exactly, the cancellation and order rules
are needed and hold, and plausible mistakes fail it."""
import numpy as np
import pytest

import oracle
from collective_communication_gb300 import inputs as gen
from naive_bound import U, bf16_key, exact_sum, f32_bound, naive_sum_f32, violations

OPROTO = {"LL": oracle.LL, "LL128": oracle.LL128, "Simple": oracle.SIMPLE}


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("proto", ["LL", "LL128", "Simple"])
@pytest.mark.parametrize("n", [2, 3, 5, 8])
def test_oracle_ring_meets_the_naive_bound(n, proto, dtype):
    count = 200003
    x = gen.draw("normal", n, count, 700 + n, dtype)
    ring = gen.ring_permutation(n, 710 + n)
    mask = gen.SPARSE_MASK
    bs = 65536 if proto == "Simple" else 0
    out = oracle.ring_allreduce_closed(list(x), ring, mask, OPROTO[proto], bs, 4)
    bad = violations(x, out[0], dtype).bad
    assert not bad.any(), np.nonzero(bad)[0][:8]


def test_integer_inputs_give_the_naive_sum_exactly():
    case = gen.small_case()
    x = case.inputs()
    out = oracle.ring_allreduce_closed(list(x), case.ring, case.mask, oracle.SIMPLE, case.buff_size, 4)
    assert np.array_equal(out[0], naive_sum_f32(x))
    chk = violations(x, out[0], "f32")
    assert not chk.bad.any() and chk.order == 0


def test_bf16_cancellation_rule_is_needed_and_holds():
    """Normal bf16 data with 8 ranks has elements whose sum nearly cancels:
    there the f32 interval spans several bf16 ulps of the result, the rule
    for them applies, and the oracle's result still meets it."""
    n, count = 8, 1 << 20
    x = gen.draw("normal", n, count, 720, "bf16")
    out = oracle.ring_allreduce_closed(list(x), gen.ring_permutation(n, 3), 0xFFF, oracle.SIMPLE, 1 << 20, 4)
    chk = violations(x, out[0], "bf16")
    assert not chk.bad.any()
    assert chk.wide > 0


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_planted_mistakes_fail(dtype):
    n, count = 8, 100000
    x = gen.draw("normal", n, count, 730, dtype)
    ring = gen.ring_permutation(n, 3)
    good = oracle.ring_allreduce_closed(list(x), ring, 0xFFF, oracle.SIMPLE, 1 << 20, 4)[0]
    # a dropped term: the sum of ranks 1..N-1 only
    dropped = oracle.oneshot(list(x[1:]))[0]
    bad = violations(x, dropped, dtype).bad
    assert bad.mean() > 0.9
    # a result two or more bf16 ulps / many f32 ulps away on a few elements
    if dtype == "f32":
        wrong = good.copy()
        wrong[::997] = np.nextafter(wrong[::997] * np.float32(1.0 + 2.0 ** -12), np.float32(np.inf))
    else:
        wrong = good.copy()
        k = bf16_key(wrong[::997])
        wrong[::997] = np.where(k >= 0, wrong[::997] + 2, wrong[::997] - 2).astype(np.uint16)
    bad = violations(x, wrong, dtype).bad
    assert bad[::997].mean() > 0.9
    assert not np.delete(bad, np.arange(0, count, 997)).any()


def test_order_rule_is_needed_and_holds():
    """Three ranks, ring 2-0-1: on a few elements per million the ring's
    binary32 sum and the naive one fall on opposite sides of the exact sum,
    each within gamma_2 * sum|x| of it (the bound of any binary32 order of
    three terms), so they differ by more than 3 * 2^-24 * sum|x|; the order
    rule accepts exactly those, and a result moved twice that bound from the
    exact sum on those elements fails."""
    n = 3
    x = gen.draw("normal", n, 1 << 20, 760, "f32")
    ring = oracle.ring_allreduce_closed(list(x), [2, 0, 1], 0b1, oracle.SIMPLE, 1 << 20, 4)[0]
    chk = violations(x, ring, "f32")
    assert not chk.bad.any() and chk.order > 0
    naive = naive_sum_f32(x).astype(np.float64)
    exact, _ = exact_sum(x)
    b = f32_bound(x)
    r = ring.astype(np.float64)
    took = np.abs(r - naive) > b
    assert took.sum() == chk.order
    sabs = np.abs(x.astype(np.float64)).sum(axis=0)
    gamma = (n - 1) * U / (1 - (n - 1) * U)
    assert np.all(np.abs(r - exact) <= gamma * sabs) and np.all(np.abs(naive - exact) <= gamma * sabs)
    assert np.all(np.sign(r - exact)[took] == -np.sign(naive - exact)[took])
    wrong = ring.copy()
    wrong[took] = (exact[took] + 2 * b[took]).astype(np.float32)
    bad = violations(x, wrong, "f32").bad
    assert bad[took].all() and not bad[~took].any()
