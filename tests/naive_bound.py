"""The accuracy criterion against a naive sum: the ring's result compared with
the plain left-to-right binary32 sum over user ranks 0..N-1.

Criterion, per element. The ring fixes its own association order, so its
result differs from the naive order's by rounding only; with cancellation a
plain relative error is unbounded, so the error is measured relative to the
sum of magnitudes (each order takes N-1 binary32 roundings, each at most
2^-24 of a partial sum no larger than the sum of magnitudes; the criterion
allows N such units between the two orders):
  f32:  |ring - naive| <= N * 2^-24 * sum_r |x_r|
  bf16: ring within 1 bf16 ulp of bf16_RNE(naive), except where the f32
        interval [naive - B, naive + B] (B the f32 bound above) itself rounds
        to bf16 values 2 or more ulps apart (heavy cancellation); there the
        ring result lies between bf16_RNE of the interval's two ends.
The bf16 rule follows from the f32 one: the ring's binary32 sum lies in the
interval, and rounding to bf16 is monotone.

Plain numpy: a binary32 add of two float32 arrays is one IEEE round-to-
nearest-even per element. bf16 values are converted to binary32 exactly; the
rounding back to bf16 is torch's CPU conversion (round to nearest even).
"""
import numpy as np

U = 2.0 ** -24


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


def violations(xs, got, dtype):
    """Boolean mask of the elements whose result breaks the criterion, and the
    number of bf16 elements that took the cancellation rule.

    xs: [N, m] inputs (float32, or uint16 bf16 bits); got: [m] results of one
    rank in the same representation."""
    if dtype == "f32":
        xf = np.asarray(xs, np.float32)
        naive = naive_sum_f32(xf)
        d = np.abs(np.asarray(got, np.float32).astype(np.float64) - naive.astype(np.float64))
        return d > f32_bound(xf), 0
    xf = bf16_bits_to_f32(xs)
    naive = naive_sum_f32(xf)
    b = f32_bound(xf)
    lo64 = naive.astype(np.float64) - b
    hi64 = naive.astype(np.float64) + b
    lo = lo64.astype(np.float32)
    lo = np.where(lo.astype(np.float64) > lo64, np.nextafter(lo, np.float32(-np.inf)), lo)
    hi = hi64.astype(np.float32)
    hi = np.where(hi.astype(np.float64) < hi64, np.nextafter(hi, np.float32(np.inf)), hi)
    klo = bf16_key(f32_to_bf16_bits(lo))
    khi = bf16_key(f32_to_bf16_bits(hi))
    kn = bf16_key(f32_to_bf16_bits(naive))
    kr = bf16_key(got)
    wide = khi - klo >= 2
    ok = np.where(wide, (kr >= klo) & (kr <= khi), np.abs(kr - kn) <= 1)
    return ~ok, int(wide.sum())
