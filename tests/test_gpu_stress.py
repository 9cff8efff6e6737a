"""Many calls on long-lived workspaces: 240 ring AllReduce calls spread over
five workspaces (every protocol, 8 ranks on 12 channels and 4 ranks on a
sparse mask), each call with its own size (1 element to 1 Mi, so the line
protocols switch between their polling and bulk forms on one workspace),
type, ring order and in-place choice. Step counters and flags carry over
from call to call; every result must equal the oracle's bit for bit."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_communication_gb300 import binding as B
from collective_communication_gb300 import inputs as gen
from gpu_util import check_guards, device_rows_numpy, guarded_outputs, to_device

pytestmark = pytest.mark.gpu
OPROTO = {"LL": oracle.LL, "LL128": oracle.LL128, "Simple": oracle.SIMPLE}
SPACES = [(8, 0xFFF, "Simple", 1 << 20), (8, 0xFFF, "LL128", 0), (8, 0xFFF, "LL", 0),
          (4, 0b101000000101, "Simple", 65536), (4, 0b101000000101, "LL128", 0)]


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    B.load_library()
    B.set_spin_timeout_ns(5_000_000_000)
    yield


def test_many_calls_on_long_lived_workspaces():
    rng = np.random.default_rng(2024)
    spaces = [B.Workspace(n, mask, proto, bs) for n, mask, proto, bs in SPACES]
    for k in range(240):
        w = int(rng.integers(0, len(SPACES)))
        n, mask, proto, bs = SPACES[w]
        count = int(rng.integers(1, 1 << int(rng.integers(1, 21))))
        dtype = "bf16" if rng.integers(0, 2) else "f32"
        ring = rng.permutation(n).tolist()
        in_place = bool(rng.integers(0, 4) == 0)
        x = gen.draw("normal", n, count, 7000 + k, dtype)
        _, send = to_device(x, dtype)
        if in_place:
            recv = send
        else:
            big_out, recv = guarded_outputs(n, count, dtype)
        B.allreduce(send, recv, ring, mask, proto, spaces[w], bs, 4)
        st = B.get_status(spaces[w])
        assert st == B.Status.OK, (k, proto, count, st)
        if not in_place:
            check_guards(big_out, count, dtype)
        want = oracle.ring_allreduce_closed(list(x), ring, mask, OPROTO[proto], bs, 4)
        got = device_rows_numpy(recv, dtype)
        for r in range(n):
            assert got[r].tobytes() == want[r].tobytes(), (k, proto, dtype, count, r)
