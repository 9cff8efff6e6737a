"""GPU parity of the staged one-shot AllReduce (rar_oneshot_staged) against
the CPU oracle's one-shot sum, bit-exact: single calls, many calls on one
workspace (the staging slots wrap), CUDA graph replay with no reset, in
place, and the guard: with acknowledgements dropped, exactly the first four
calls (one per staging slot) complete and the fifth runs out of time."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_communication_gb300 import binding as B
from collective_communication_gb300 import inputs as gen
from gpu_util import check_guards, device_rows_numpy, guarded_outputs, to_device

pytestmark = pytest.mark.gpu
SLOTS = 4  # staging slots per rank


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    B.load_library()
    B.set_spin_timeout_ns(5_000_000_000)
    yield


def _exact(got, want):
    for r in range(len(want)):
        a, b = got[r], want[r]
        bad = np.nonzero(a.view(np.uint8) != b.view(np.uint8))[0]
        assert bad.size == 0, f"rank {r}: {bad.size} mismatching bytes"


def run_staged(n, count, dtype, seed, ws=None, in_place=False, kind="normal"):
    x = gen.draw(kind, n, count, seed, dtype)
    big_in, send = to_device(x, dtype)
    if in_place:
        recv = send
    else:
        big_out, recv = guarded_outputs(n, count, dtype)
    ws = ws or B.OneShotWorkspace(n, count, dtype)
    B.oneshot_staged(send, recv, ws)
    assert B.get_status(ws) == B.Status.OK
    if not in_place:
        check_guards(big_out, count, dtype)
    _exact(device_rows_numpy(recv, dtype), oracle.oneshot(list(x)))
    return ws


@pytest.mark.parametrize("case", gen.oneshot_cases(), ids=lambda c: c.name)
def test_staged_bf16_n8(case):
    run_staged(case.nranks, case.count, case.dtype, case.seed, kind=case.kind)


@pytest.mark.parametrize("count", [1, 7, 8, 9, 1000, 2048, 4095, 123457])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n", [1, 2, 3, 8, 16])
def test_staged_ragged(n, count, dtype):
    run_staged(n, count, dtype, 20 + n)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 32])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_staged_every_rank_count(n, dtype):
    """Every rank count of the fixed-count kernels (1..8) and of the kernel
    for more than 8 ranks (slots read in batches of 8), each rank's blocks
    taking many reduce chunks, with a ragged end."""
    ws = run_staged(n, 1300007, dtype, 80 + n)
    run_staged(n, 1300007, dtype, 90 + n, ws=ws)  # the next slot of the same workspace


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_staged_in_place(dtype):
    for n, count in ((2, 5), (8, 7168 * 8), (5, 100003)):
        run_staged(n, count, dtype, 7, in_place=True)


def test_many_calls_on_one_workspace():
    """Calls of varying sizes (at most the workspace's) reuse the 4 slots
    round-robin; every result is exact."""
    n, max_count = 8, 7168 * 64
    ws = B.OneShotWorkspace(n, max_count, "bf16")
    for k in range(3 * SLOTS + 1):
        run_staged(n, [max_count, 7168, 1, 99999][k % 4], "bf16", 100 + k, ws=ws)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_graph_replay_needs_no_reset(dtype):
    """One call captured in a CUDA graph and replayed 3 * SLOTS + 2 times with
    new inputs each time: the sequence numbers and done counters live in the
    workspace and only grow, so every replay is exact."""
    n, count = 8, 7168 * 8
    ws = B.OneShotWorkspace(n, count, dtype)
    x0 = gen.draw("normal", n, count, 0, dtype)
    big_in, send = to_device(x0, dtype)
    big_out, recv = guarded_outputs(n, count, dtype)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        B.oneshot_staged(send, recv, ws, stream=s)  # warm-up call, outside the graph
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        B.oneshot_staged(send, recv, ws, stream=s)
    torch.cuda.synchronize()
    for k in range(3 * SLOTS + 2):
        x = gen.draw("normal", n, count, 1000 + k, dtype)
        _, src = to_device(x, dtype)
        for r in range(n):
            send[r].copy_(src[r])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert B.get_status(ws) == B.Status.OK
        check_guards(big_out, count, dtype)
        _exact(device_rows_numpy(recv, dtype), oracle.oneshot(list(x)))


def test_guard_fires_after_one_call_per_slot():
    """Fault 2: no rank acknowledges its reads. A staging slot is reused every
    SLOTS calls, so calls 1..SLOTS complete (exactly) and call SLOTS+1 waits for
    an acknowledgement that never comes, until the time limit. The workspace
    then stays aborted until it is initialised again."""
    n, count = 4, 5000
    ws = B.OneShotWorkspace(n, count, "f32")
    B.set_spin_timeout_ns(200_000_000)
    try:
        B.debug_set_fault(2)
        for k in range(SLOTS):
            run_staged(n, count, "f32", 200 + k, ws=ws)
        x = gen.draw("normal", n, count, 300, "f32")
        _, send = to_device(x, "f32")
        _, recv = guarded_outputs(n, count, "f32")
        B.oneshot_staged(send, recv, ws)
        assert B.get_status(ws) == B.Status.ERR_TIMEOUT
        B.debug_set_fault(0)
        B.oneshot_staged(send, recv, ws)
        assert B.get_status(ws) == B.Status.ERR_ABORT
    finally:
        B.debug_set_fault(0)
        B.set_spin_timeout_ns(5_000_000_000)
    ws.init()
    run_staged(n, count, "f32", 301, ws=ws)


def test_workspace_of_another_configuration_is_refused():
    ws = B.OneShotWorkspace(4, 4096, "f32")
    x = gen.draw("normal", 2, 1024, 1, "f32")
    _, send = to_device(x, "f32")
    _, recv = guarded_outputs(2, 1024, "f32")
    B.oneshot_staged(send, recv, ws)  # 2 ranks on a 4-rank workspace
    assert B.get_status(ws) == B.Status.ERR_WORKSPACE
    ws.init()
    run_staged(4, 4096, "f32", 2, ws=ws)
