"""GPU parity in the LL flag-wrap test mode (rar_debug_set_ll_flag_wrap):
sessions of calls on one workspace whose step counters cross the flag period
many times, including the sequences that make the oracle take stale lines
when the cleanup is left out. With the cleanup every call must equal the
oracle's result bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_communication_gb300 import binding as B
from gpu_util import device_rows_numpy, guarded_outputs, check_guards, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    B.load_library()
    B.set_spin_timeout_ns(5_000_000_000)
    yield
    B.debug_set_ll_flag_wrap(0)


def _draw(n, count, seed, dtype="f32"):
    rng = np.random.default_rng(seed)
    vals = [rng.standard_normal(count).astype(np.float32) for _ in range(n)]
    return [oracle.bf16_round(v) for v in vals] if dtype == "bf16" else vals


def run_session(calls, rings, mask, bs, flag_max):
    """Every call on one fresh workspace under the given flag mode; each
    result compared with the oracle's session (which also reports that no
    stale line was taken)."""
    n = len(calls[0])
    dtype = "f32" if calls[0][0].dtype == np.float32 else "bf16"
    want, stale, age = oracle.ll_session_sim(calls, rings, mask, bs, flag_max=flag_max, cleanup=True)
    assert stale == 0
    B.debug_set_ll_flag_wrap(flag_max)
    try:
        ws = B.Workspace(n, mask, "LL", bs)
        for k, c in enumerate(calls):
            count = c[0].size
            if count == 0:
                continue
            _, send = to_device(np.stack(c), dtype)
            big_out, recv = guarded_outputs(n, count, dtype)
            B.allreduce_ex(send, recv, rings, mask, "LL", ws, bs, 4)
            assert B.get_status(ws) == B.Status.OK, k
            check_guards(big_out, count, dtype)
            got = device_rows_numpy(recv, dtype)
            for r in range(n):
                assert got[r].tobytes() == want[k][r].tobytes(), f"call {k} rank {r}"
    finally:
        B.debug_set_ll_flag_wrap(0)


def test_wrap_at_0x100_after_248_steps_of_one_line_calls():
    """The sequence that makes the oracle take stale lines without the cleanup
    (N=5, LL buffer 4096 B): a large call, 31 one-line calls (248 steps per
    connection), a large call whose first use of each slot is 256 steps after
    its last full write."""
    n = 5
    big = n * 64 * 4
    calls = [_draw(n, big, 1)] + [_draw(n, 8, 2 + k) for k in range(31)] + [_draw(n, big, 100)]
    run_session(calls, list(range(n)), 0x1, 4096, 256)


def test_wrap_at_64_reaches_flag_zero():
    n = 3
    calls = [_draw(n, 3 * 64, 7)] + [_draw(n, 5, 8 + k) for k in range(14)] + [_draw(n, 3 * 64 * 3, 60)]
    run_session(calls, list(range(n)), 0x1, 4096, 64)


@pytest.mark.parametrize("flag_max", [64, 256])
@pytest.mark.parametrize("seed", range(4))
def test_random_sessions(seed, flag_max):
    rng = np.random.default_rng(900 + seed)
    n = int(rng.integers(2, 9))
    mask = int(rng.integers(1, 1 << 6))
    nch = bin(mask).count("1")
    rings = [rng.permutation(n).tolist() for _ in range(nch)] if seed % 2 else rng.permutation(n).tolist()
    bs = 4096 * int(rng.integers(1, 4))
    dtype = "bf16" if seed % 2 == 0 else "f32"
    calls = [_draw(n, int(rng.choice([1, 5, 40, 300, 2000, 20000])), 50 * seed + k, dtype)
             for k in range(int(rng.integers(25, 45)))]
    run_session(calls, rings, mask, bs, flag_max)


def test_production_mode_after_wrap_mode_needs_a_fresh_workspace_only():
    """Back in production mode, a fresh workspace gives exact results."""
    n = 4
    calls = [_draw(n, c, 70 + c) for c in (1000, 3, 50000)]
    want, stale, _ = oracle.ll_session_sim(calls, [0, 2, 3, 1], 0x3, 0)
    assert stale == 0
    ws = B.Workspace(n, 0x3, "LL", 0)
    for k, c in enumerate(calls):
        _, send = to_device(np.stack(c), "f32")
        _, recv = guarded_outputs(n, c[0].size, "f32")
        B.allreduce(send, recv, [0, 2, 3, 1], 0x3, "LL", ws, 0, 4)
        assert B.get_status(ws) == B.Status.OK
        got = device_rows_numpy(recv, "f32")
        for r in range(n):
            assert got[r].tobytes() == want[k][r].tobytes()
