"""The ring collectives under CUDA-graph replay: one call captured once and
replayed with new inputs each time. The step counters live in the workspace
and only grow, so no replay needs a reset, and every replay must equal the
oracle bit for bit (every protocol, both forms of the line protocols, the
two halves)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_communication_gb300 import binding as B
from collective_communication_gb300 import inputs as gen
from gpu_util import check_guards, device_rows_numpy, guarded_outputs, to_device

pytestmark = pytest.mark.gpu
OPROTO = {"LL": oracle.LL, "LL128": oracle.LL128, "Simple": oracle.SIMPLE}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    B.load_library()
    B.set_spin_timeout_ns(5_000_000_000)
    yield


def _replay(n, count, dtype, call, reference, nreplay=9):
    """Capture call(send, recv, stream) in a graph; replay it with new inputs."""
    x0 = gen.draw("normal", n, count[0], 0, dtype)
    _, send = to_device(x0, dtype)
    big_out, recv = guarded_outputs(n, count[1], dtype)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        call(send, recv, s)  # warm-up, outside the graph
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        call(send, recv, s)
    torch.cuda.synchronize()
    for k in range(nreplay):
        x = gen.draw("normal", n, count[0], 100 + k, dtype)
        _, src = to_device(x, dtype)
        for r in range(n):
            send[r].copy_(src[r])
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        check_guards(big_out, count[1], dtype)
        want = reference(list(x))
        got = device_rows_numpy(recv, dtype)
        for r in range(n):
            assert got[r].tobytes() == want[r].tobytes(), (k, r)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("proto,count", [("Simple", 300001), ("LL", 500), ("LL", 100003), ("LL128", 700),
                                         ("LL128", 200003)])
def test_allreduce_graph_replay(proto, count, dtype):
    n, mask, ring = 5, 0b1011, [3, 1, 4, 0, 2]
    bs = 65536 if proto == "Simple" else 0
    ws = B.Workspace(n, mask, proto, bs)

    def call(send, recv, s):
        B.allreduce(send, recv, ring, mask, proto, ws, bs, 4, stream=s)

    _replay(n, (count, count), dtype, call,
            lambda xs: oracle.ring_allreduce_closed(xs, ring, mask, OPROTO[proto], bs, 4))
    assert B.get_status(ws) == B.Status.OK


@pytest.mark.parametrize("proto", ["Simple", "LL128"])
@pytest.mark.parametrize("kind", ["rs", "ag"])
def test_halves_graph_replay(kind, proto):
    n, mask, ring, block, dtype = 4, 0b11, [0, 2, 3, 1], 40000, "f32"
    ws = B.Workspace(n, mask, proto, 0)
    if kind == "rs":
        def call(send, recv, s):
            B.reduce_scatter(send, recv, ring, mask, proto, ws, 0, 4, stream=s)
        counts = (n * block, block)
        ref = lambda xs: oracle.ring_halves_closed(oracle.REDUCE_SCATTER, xs, ring, mask, OPROTO[proto], 0, 4)
    else:
        def call(send, recv, s):
            B.all_gather(send, recv, ring, mask, proto, ws, 0, 4, stream=s)
        counts = (block, n * block)
        ref = lambda xs: oracle.ring_halves_closed(oracle.ALL_GATHER, xs, ring, mask, OPROTO[proto], 0, 4)
    _replay(n, counts, dtype, call, ref)
    assert B.get_status(ws) == B.Status.OK
