"""Pins of the oracle's LL session simulation and the flag-wrap test mode.

[C23] "LL：Data 与 Flag 同 Line": production LL flags are step + 1, a
monotonic generation, so a reused slot's old lines never match; a test
macro makes the flag wrap at 0x100, and then a cleanup (the sender writes the
current generation into the rest of its slot) is what keeps lines the slice
did not cover from carrying an old flag of the same value. The session
simulation keeps FIFOs and step counters across calls and lets receivers
take each line on its own, so the hazard is observable: the pins show it
with the cleanup taken out (a mistake planted in the oracle) and show its
absence with production flags and with the cleanup.
"""
import numpy as np
import pytest

import oracle


def _draw(n, count, seed, dtype="f32"):
    rng = np.random.default_rng(seed)
    vals = [rng.standard_normal(count).astype(np.float32) for _ in range(n)]
    return [oracle.bf16_round(v) for v in vals] if dtype == "bf16" else vals


def _exact(outs, calls, ring, mask, bs):
    for k, c in enumerate(calls):
        want = oracle.ring_allreduce_closed(c, ring, mask, oracle.LL, bs)
        for a, b in zip(outs[k], want):
            if a.tobytes() != b.tobytes():
                return False
    return True


def aba_session(n=5, bs=4096):
    """A large call (every line of every slot written), then tiny calls that
    write only the first line of their slots and advance each connection by
    exactly 248 steps, then a large call: its first use of every slot comes
    256 steps after that slot's last full write, so with 256-step flags the
    old lines carry exactly the expected flag.
    LL buffer 4096 B: 512-byte steps of 32 lines, 64-element f32 chunks; a
    loop of n chunks is 2n - 2 = 8 steps per connection for n = 5."""
    assert n == 5 and bs == 4096
    big = n * 64 * 4  # 4 loops: 32 steps
    calls = [_draw(n, big, 1)] + [_draw(n, 8, 2 + k) for k in range(31)] + [_draw(n, big, 100)]
    return calls, list(range(n)), 0x1, bs


def test_production_flags_never_match_old_lines():
    calls, ring, mask, bs = aba_session()
    outs, stale, age = oracle.ll_session_sim(calls, ring, mask, bs, flag_max=0)
    assert stale == 0
    assert age == 256  # the old lines are polled, 256 steps old, and rejected
    assert _exact(outs, calls, ring, mask, bs)


def test_wrap_without_cleanup_takes_stale_lines():
    """The planted mistake: flags wrap at 0x100 and nobody cleans. The old
    lines of the large call's slots carry the flag of the step 256 later, are
    taken before the sender writes them, and the results are wrong."""
    calls, ring, mask, bs = aba_session()
    outs, stale, age = oracle.ll_session_sim(calls, ring, mask, bs, flag_max=256, cleanup=False)
    assert stale > 0
    assert age == 256
    assert not _exact(outs, calls, ring, mask, bs)


def test_wrap_with_cleanup_is_exact():
    calls, ring, mask, bs = aba_session()
    outs, stale, age = oracle.ll_session_sim(calls, ring, mask, bs, flag_max=256, cleanup=True)
    assert stale == 0
    assert 0 < age <= 128  # no polled line is older than half a flag period
    assert _exact(outs, calls, ring, mask, bs)


def test_zeroed_lines_are_not_taken_for_flag_zero():
    """With 64-step flags, step 63 expects flag 0, the value of never-written
    lines. N=3: a loop is 4 steps per connection. One full loop (slots 0-3),
    14 one-line calls (steps 4-59), then three full loops (steps 60-71): step
    63 uses slot 7, whose lines past the first were never written. Without
    the cleanup they are taken as data; with it, slot 7 was cleaned at step
    31 and its lines carry flag 32."""
    n, bs = 3, 4096
    calls = [_draw(n, 3 * 64, 7)] + [_draw(n, 5, 8 + k) for k in range(14)] + [_draw(n, 3 * 64 * 3, 60)]
    outs, stale, age = oracle.ll_session_sim(calls, list(range(n)), 0x1, bs, flag_max=64, cleanup=True)
    assert stale == 0 and age <= 32
    assert _exact(outs, calls, list(range(n)), 0x1, bs)
    outs, stale, _ = oracle.ll_session_sim(calls, list(range(n)), 0x1, bs, flag_max=64, cleanup=False)
    assert stale > 0


@pytest.mark.parametrize("flag_max", [64, 256])
@pytest.mark.parametrize("seed", range(6))
def test_random_sessions_across_many_wraps(seed, flag_max):
    rng = np.random.default_rng(500 + seed)
    n = int(rng.integers(2, 7))
    mask = int(rng.integers(1, 8))
    nch = bin(mask).count("1")
    rings = [rng.permutation(n).tolist() for _ in range(nch)] if seed % 2 else rng.permutation(n).tolist()
    bs = 4096 * int(rng.integers(1, 3))
    dtype = "bf16" if seed % 3 == 0 else "f32"
    calls = []
    for k in range(int(rng.integers(20, 40))):
        count = int(rng.choice([0, 1, 5, 40, 300, 2000, 9000]))
        calls.append(_draw(n, count, 1000 * seed + k, dtype))
    outs, stale, age = oracle.ll_session_sim(calls, rings, mask, bs, flag_max=flag_max, cleanup=True)
    assert stale == 0
    assert age <= flag_max // 2
    assert _exact(outs, calls, rings, mask, bs)


def test_session_with_production_flags_matches_single_calls():
    """Step counters that carry over change no result: every call of a
    session equals the same call on a fresh workspace."""
    rng = np.random.default_rng(3)
    calls = [_draw(4, int(c), 40 + k) for k, c in enumerate(rng.integers(1, 5000, 12))]
    outs, stale, _ = oracle.ll_session_sim(calls, [0, 2, 3, 1], 0x3, 8192)
    assert stale == 0
    for k, c in enumerate(calls):
        single, _, _, _ = oracle.ring_allreduce_sim(c, [0, 2, 3, 1], 0x3, oracle.LL, 8192)
        assert all(a.tobytes() == b.tobytes() for a, b in zip(outs[k], single))


def test_bad_flag_periods():
    calls = [_draw(2, 10, 0)]
    for bad in (32, 100, 255):
        with pytest.raises(oracle.OracleError):
            oracle.ll_session_sim(calls, [0, 1], 0x1, 4096, flag_max=bad)
