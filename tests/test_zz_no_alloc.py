"""rar_allreduce_static: the ring AllReduce entry point for callers that may not
allocate device memory (its workspace is a fixed library array in device
memory). Checked against rar_allreduce with a caller-allocated workspace and
against the oracle, on two calls in a row, through the C ABI. The cases run in
order on the one shared array: a Simple call (which clears only the header and
step counters) follows an LL call that left its lines in the array. This file
is collected last so that a run stopping at its first failure has already run
every other test."""
import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_communication_gb300 import binding as B
from collective_communication_gb300 import inputs as gen

pytestmark = pytest.mark.gpu

STATIC_BYTES = 16 << 20  # RAR_STATIC_WORKSPACE_BYTES
OPROTO = {"LL": oracle.LL, "LL128": oracle.LL128, "Simple": oracle.SIMPLE}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    B.load_library()
    yield


def _ptrs(ts):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


def _static_call(send, recv, case, stream):
    L = B.load_library()
    ring = (ctypes.c_int * case.nranks)(*case.ring)
    return L.rar_allreduce_static(_ptrs(send), _ptrs(recv), case.nranks, case.count,
                                  0 if case.dtype == "f32" else 1, 0, ring, case.mask,
                                  int(B.PROTO_BY_NAME[case.proto]), case.buff_size, case.chunk_steps, stream)


def _rows(x, dtype):
    n, count = x.shape
    stride = -(-count // 64) * 64
    if dtype == "f32":
        big = torch.zeros((n, stride), dtype=torch.float32, device="cuda")
        big[:, :count] = torch.from_numpy(x).cuda()
    else:
        big = torch.zeros((n, stride), dtype=torch.int16, device="cuda")
        big[:, :count] = torch.from_numpy(x.view(np.int16)).cuda()
        big = big.view(torch.bfloat16)
    return big, [big[r, :count] for r in range(n)]


CASES = [
    gen.RingCase("static_simple_n8_ch12", 8, gen.ring_permutation(8, 3), 0xFFF, gen.SIMPLE, 300007, gen.F32,
                 "normal", 31, 64 * 1024, 4),
    gen.RingCase("static_ll128_n4_sparse", 4, gen.RING_0231, 0b1011, gen.LL128, 123457, gen.BF16, "normal", 32,
                 256 * 1024, 4),
    gen.RingCase("static_ll_n5", 5, [4, 0, 3, 1, 2], 0b11, gen.LL, 77777, gen.F32, "normal", 33, 0, 4),
    gen.RingCase("static_simple_n4_after_ll", 4, gen.RING_0231, 0b101, gen.SIMPLE, 200003, gen.BF16, "normal", 34,
                 16 * 1024, 2),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: c.name)
def test_static_matches_allocating_entry_point(case):
    assert B.workspace_bytes(case.nranks, case.mask, case.proto, case.buff_size) <= STATIC_BYTES
    stream = torch.cuda.current_stream().cuda_stream
    ws = B.Workspace(case.nranks, case.mask, case.proto, case.buff_size)
    for call in range(2):  # two calls in a row, different data each time
        x = gen.draw(case.kind, case.nranks, case.count, case.seed + call, case.dtype)
        _, send = _rows(x, case.dtype)
        big_ref, ref = _rows(np.zeros_like(x), case.dtype)
        big_out, out = _rows(np.zeros_like(x), case.dtype)
        B.allreduce(send, ref, case.ring, case.mask, case.proto, ws, case.buff_size, case.chunk_steps)
        st = _static_call(send, out, case, stream)
        assert st == B.Status.OK, B.Status(st)
        torch.cuda.synchronize()
        assert B.get_status(ws) == B.Status.OK
        a = big_ref.view(torch.int32 if case.dtype == "f32" else torch.int16)
        b = big_out.view(torch.int32 if case.dtype == "f32" else torch.int16)
        assert bool(torch.equal(a, b)), f"call {call}: static workspace result differs"
        want = oracle.ring_allreduce_closed(list(x), case.ring, case.mask, OPROTO[case.proto], case.buff_size,
                                            case.chunk_steps)
        got = b[:, :case.count].cpu().numpy()
        for r in range(case.nranks):
            w = want[r].view(np.int32 if case.dtype == "f32" else np.int16)
            assert np.array_equal(got[r], w), f"call {call}, rank {r}: differs from the oracle"


def test_static_refuses_oversized_workspace():
    case = gen.RingCase("too_big", 8, list(range(8)), 0xFFF, gen.SIMPLE, 1024, gen.F32, "normal", 1, 1 << 20, 4)
    assert B.workspace_bytes(8, 0xFFF, gen.SIMPLE, 1 << 20) > STATIC_BYTES
    x = gen.draw("normal", 8, 1024, 1)
    _, send = _rows(x, "f32")
    _, out = _rows(np.zeros_like(x), "f32")
    st = _static_call(send, out, case, torch.cuda.current_stream().cuda_stream)
    assert st == B.Status.ERR_WORKSPACE
