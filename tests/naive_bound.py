"""The accuracy criterion against a naive sum: the ring's result compared with
the plain left-to-right binary32 sum over user ranks 0..N-1.

Criterion, per element. The ring fixes its own association order, so its
result differs from the naive order's by rounding only; with cancellation a
plain relative error is unbounded, so the error is measured relative to the
sum of magnitudes, with B = N * 2^-24 * sum_r |x_r|:
  f32:  |ring - naive| <= B  (the naive rule);
        where that fails, |ring - exact| <= B  (the order rule).
  bf16: ring within 1 bf16 ulp of bf16_RNE(naive), except where the f32
        interval [naive - B, naive + B] itself rounds to bf16 values 2 or
        more ulps apart (heavy cancellation): there the ring result lies
        between bf16_RNE of the interval's two ends (the cancellation rule);
        where both fail, the ring result lies between bf16_RNE of the ends of
        [exact - B, exact + B] (the order rule).
Why the order rule: a binary32 sum of N terms in any association order lies
within gamma_{N-1} * sum|x| of the exact sum (N - 1 roundings, each at most
2^-24 of a partial sum no larger than sum|x|; gamma_k = k u / (1 - k u),
u = 2^-24), and gamma_{N-1} < N u. Two orders can therefore differ by up to
2 gamma_{N-1} sum|x|, which exceeds B for N >= 3 when their rounding errors
fall on opposite sides of the exact sum (the oracle's own ring order does so
on a few elements per million at N = 3). There the ring result must be as
close to the exact sum as the naive order is guaranteed to be. The bf16 rules
follow from the f32 ones: the ring's binary32 sum lies in the interval, and
rounding to bf16 is monotone.

Plain numpy: a binary32 add of two float32 arrays is one IEEE round-to-
nearest-even per element. The exact sum is taken in binary64 (its own error,
at most (N - 1) 2^-53 sum|x|, is added to B for the order rule). bf16 values
are converted to binary32 exactly; the rounding back to bf16 is torch's CPU
conversion (round to nearest even).
"""
from typing import NamedTuple

import numpy as np

U = 2.0 ** -24


class Check(NamedTuple):
    bad: np.ndarray   # elements that break the criterion
    wide: int         # bf16 elements that took the cancellation rule
    order: int        # elements that took the order rule


def bf16_bits_to_f32(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16_bits(x):
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def bf16_key(bits):
    """bf16 bit patterns -> integers ordered like the values (+0 and -0 equal),
    so that a difference of keys counts the ulps between two values."""
    b = np.asarray(bits, np.uint16).astype(np.int32)
    mag = b & 0x7FFF
    return np.where(b >> 15 == 1, -mag, mag)


def naive_sum_f32(xs):
    """Left-to-right binary32 sum over the rows of xs ([N, m] float32)."""
    acc = np.array(xs[0], np.float32, copy=True)
    for r in range(1, len(xs)):
        acc += xs[r]
    return acc


def f32_bound(xs):
    """N * 2^-24 * sum_r |x_r| per element, in binary64."""
    return len(xs) * U * np.abs(np.asarray(xs, np.float32).astype(np.float64)).sum(axis=0)


def exact_sum(xs):
    """The sum of the binary32 rows in binary64, and a bound on its own error."""
    x64 = np.asarray(xs, np.float32).astype(np.float64)
    return x64.sum(axis=0), (len(xs) - 1) * 2.0 ** -53 * np.abs(x64).sum(axis=0)


def _interval_keys(centre64, half64):
    """bf16 keys of RNE of the binary32 ends of [centre - half, centre + half],
    each end rounded outward to binary32."""
    lo64 = centre64 - half64
    hi64 = centre64 + half64
    lo = lo64.astype(np.float32)
    lo = np.where(lo.astype(np.float64) > lo64, np.nextafter(lo, np.float32(-np.inf)), lo)
    hi = hi64.astype(np.float32)
    hi = np.where(hi.astype(np.float64) < hi64, np.nextafter(hi, np.float32(np.inf)), hi)
    return bf16_key(f32_to_bf16_bits(lo)), bf16_key(f32_to_bf16_bits(hi))


def violations(xs, got, dtype):
    """Check of one rank's results against the criterion.

    xs: [N, m] inputs (float32, or uint16 bf16 bits); got: [m] results of one
    rank in the same representation."""
    if dtype == "f32":
        xf = np.asarray(xs, np.float32)
        naive = naive_sum_f32(xf)
        g64 = np.asarray(got, np.float32).astype(np.float64)
        b = f32_bound(xf)
        ok_naive = np.abs(g64 - naive.astype(np.float64)) <= b
        exact, err = exact_sum(xf)
        ok_order = np.abs(g64 - exact) <= b + err
        return Check(~(ok_naive | ok_order), 0, int((~ok_naive & ok_order).sum()))
    xf = bf16_bits_to_f32(xs)
    naive = naive_sum_f32(xf)
    b = f32_bound(xf)
    klo, khi = _interval_keys(naive.astype(np.float64), b)
    kn = bf16_key(f32_to_bf16_bits(naive))
    kr = bf16_key(got)
    wide = khi - klo >= 2
    ok_naive = np.where(wide, (kr >= klo) & (kr <= khi), np.abs(kr - kn) <= 1)
    exact, err = exact_sum(xf)
    elo, ehi = _interval_keys(exact, b + err)
    ok_order = (kr >= elo) & (kr <= ehi)
    return Check(~(ok_naive | ok_order), int(wide.sum()), int((~ok_naive & ok_order).sum()))
