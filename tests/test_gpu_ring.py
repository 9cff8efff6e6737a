"""GPU parity of the ring AllReduce (all protocols, f32 and bf16) against the
CPU oracle: bit-exact, element by element, on every rank, with guard bands
around every receive buffer, at every size up to 1 GiB per rank; and every
result element against the naive left-to-right sum's bound
(tests/naive_bound.py). Calls go through the C ABI (librar.so)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_communication_gb300 import binding as B
from collective_communication_gb300 import inputs as gen
from gpu_util import check_guards, device_rows_numpy, guarded_outputs, to_device
from naive_bound import violations

pytestmark = pytest.mark.gpu

OPROTO = {"LL": oracle.LL, "LL128": oracle.LL128, "Simple": oracle.SIMPLE}
ODT = {"f32": oracle.F32, "bf16": oracle.BF16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    B.load_library()
    B.set_spin_timeout_ns(5_000_000_000)
    yield


def run_ring(case, x=None, in_place=False, workspace=None, calls=1):
    x = case.inputs() if x is None else x
    big_in, send = to_device(x, case.dtype)
    if in_place:
        big_out, recv = big_in, send
    else:
        big_out, recv = guarded_outputs(case.nranks, case.count, case.dtype)
    ws = workspace or B.Workspace(case.nranks, case.mask, case.proto, case.buff_size)
    for _ in range(calls):
        if in_place and calls > 1:
            raise ValueError
        B.allreduce(send, recv, case.ring, case.mask, case.proto, ws, case.buff_size, case.chunk_steps)
    st = B.get_status(ws)
    assert st == B.Status.OK, st
    if not in_place:
        check_guards(big_out, case.count, case.dtype)
    return x, device_rows_numpy(recv, case.dtype), ws


def oracle_full(case, x):
    return oracle.ring_allreduce_closed(list(x), case.ring, case.mask, OPROTO[case.proto], case.buff_size,
                                        case.chunk_steps)


def assert_bit_exact(got, want_rows):
    for r in range(got.shape[0]):
        w = want_rows[r]
        g = got[r]
        bad = np.nonzero(g.view(np.uint32 if g.dtype == np.float32 else np.uint16) !=
                         w.view(np.uint32 if w.dtype == np.float32 else np.uint16))[0]
        assert bad.size == 0, f"rank {r}: {bad.size} mismatches, first at {bad[:8]}"


def assert_naive_bound(x, got, dtype, offset=0):
    """Every rank's result within the naive left-to-right sum's bound."""
    for r in range(got.shape[0]):
        idx = np.nonzero(violations(x, got[r], dtype).bad)[0]
        assert idx.size == 0, f"rank {r}: {idx.size} elements outside the naive-sum bound, first at {idx[:8] + offset}"


# ---------------------------------------------------------------------------
# the 4 KiB integer case: every protocol, exact sum
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("proto", ["Simple", "LL", "LL128"])
def test_small_integer_case_exact(proto):
    case = gen.small_case()
    case.proto = proto
    if proto != "Simple":
        case.buff_size = 0
    x, got, _ = run_ring(case)
    exact = x.astype(np.int64).sum(axis=0).astype(np.float32)
    for r in range(case.nranks):
        assert np.array_equal(got[r], exact)
    assert_bit_exact(got, oracle_full(case, x))
    assert_naive_bound(x, got, case.dtype)


# ---------------------------------------------------------------------------
# 512 KiB per rank, N=4: protocols x channels
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", gen.sweep_512k_cases(), ids=lambda c: c.name)
def test_sweep_512k(case):
    x, got, _ = run_ring(case)
    assert_bit_exact(got, oracle_full(case, x))
    assert_naive_bound(x, got, case.dtype)


# ---------------------------------------------------------------------------
# tiny and ragged cases, several tiles, random rings and masks, both dtypes
# ---------------------------------------------------------------------------
def _random_cases():
    rng = np.random.default_rng(77)
    out = []
    for k in range(36):
        n = int(rng.integers(2, 9))
        proto = ["LL", "LL128", "Simple"][k % 3]
        dtype = "f32" if (k // 3) % 2 == 0 else "bf16"
        mask = int(rng.integers(1, 1 << 8))
        count = [1, 3, 7, 13, 100, 1000][k % 6] if k < 12 else int(rng.integers(1, 300000))
        bs = {"Simple": 4096 * int(rng.integers(1, 9)), "LL": 4096 * int(rng.integers(1, 5)),
              "LL128": 4096 * int(rng.integers(1, 10))}[proto]
        cs = int(rng.choice([1, 2, 4]))
        ring = rng.permutation(n).tolist()
        out.append(gen.RingCase(f"rand{k}_{proto}_{dtype}_n{n}_c{count}", n, ring, mask, proto, count, dtype,
                                "normal", 1000 + k, bs, cs))
    return out


@pytest.mark.parametrize("case", _random_cases(), ids=lambda c: c.name)
def test_random_cases(case):
    x, got, _ = run_ring(case)
    assert_bit_exact(got, oracle_full(case, x))
    assert_naive_bound(x, got, case.dtype)


@pytest.mark.parametrize("proto", ["LL", "LL128", "Simple"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_in_place(proto, dtype):
    case = gen.RingCase("inplace", 5, [3, 1, 4, 0, 2], 0b1011, proto, 77777, dtype, "normal", 42,
                        8192 if proto == "Simple" else 0, 4)
    x = case.inputs()
    want = oracle_full(case, x)
    _, got, _ = run_ring(case, x=x, in_place=True)
    assert_bit_exact(got, want)


@pytest.mark.parametrize("proto", ["LL", "LL128", "Simple"])
def test_many_calls_reuse_workspace(proto):
    """Step counters carry over between calls: 7 calls with changing data,
    dtype and ring on one workspace, each bit-exact."""
    bs = 16384 if proto == "Simple" else 0
    ws = B.Workspace(4, 0b110, proto, bs)
    for k in range(7):
        dtype = "f32" if k % 2 == 0 else "bf16"
        ring = gen.ring_permutation(4, 500 + k)
        case = gen.RingCase("reuse", 4, ring, 0b110, proto, 5000 + 997 * k, dtype, "normal", 900 + k, bs,
                            [4, 2, 1][k % 3])
        x, got, _ = run_ring(case, workspace=ws)
        assert_bit_exact(got, oracle_full(case, x))


def test_block_to_channel_trace():
    """The kernel writes, per block, the channel id it mapped itself to; block
    b serves rank b // C and the (b % C)-th set bit of the mask."""
    mask = gen.SPARSE_MASK
    case = gen.RingCase("trace", 3, [0, 2, 1], mask, "Simple", 4096, "f32", "normal", 5, 65536, 4)
    _, _, ws = run_ring(case)
    ids = oracle.mask_channels(mask)
    C = len(ids)
    trace = ws.tensor[2048:2048 + 3 * C].cpu().numpy()
    for b in range(3 * C):
        assert trace[b] == ids[b % C]


# ---------------------------------------------------------------------------
# full size: N=8, 64 MiB per rank, and the sparse sweep up to 1 GiB per rank:
# every element of the result against the oracle's closed form (computed
# range by range, so host memory stays bounded) and the naive-sum bound
# ---------------------------------------------------------------------------
def _device_inputs(case):
    """Seeded inputs drawn on the device (too large to draw on the host
    quickly); rows padded to 64 elements so every rank's buffer is 16-byte
    aligned. Returns the [N, count] view."""
    g = torch.Generator(device="cuda")
    g.manual_seed(case.seed)
    stride = -(-case.count // 64) * 64
    x = torch.randn((case.nranks, stride), generator=g, device="cuda", dtype=torch.float32)
    if case.dtype == "bf16":
        x = x.to(torch.bfloat16)
    return x[:, :case.count]


def _host(t, dtype):
    if dtype == "f32":
        return t.cpu().numpy()
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def check_full(case, x, out_row, span=1 << 23):
    """out_row (rank 0's device result) against the oracle's closed form at
    every element, and against the naive-sum bound, span elements at a time."""
    wide = 0
    for a in range(0, case.count, span):
        b = min(case.count, a + span)
        xs = _host(x[:, a:b], case.dtype)
        got = _host(out_row[a:b], case.dtype)
        want, _ = oracle.ring_closed_at(list(xs), case.ring, case.mask, OPROTO[case.proto],
                                        np.arange(a, b, dtype=np.int64), case.count, case.buff_size,
                                        case.chunk_steps)
        bits = np.uint32 if case.dtype == "f32" else np.uint16
        bad = np.nonzero(got.view(bits) != want.view(bits))[0]
        assert bad.size == 0, f"{bad.size} mismatches in [{a}, {b}), first at {bad[:8] + a}"
        chk = violations(xs, got, case.dtype)
        wide += chk.wide
        idx = np.nonzero(chk.bad)[0]
        assert idx.size == 0, f"{idx.size} elements outside the naive-sum bound, first at {idx[:8] + a}"
    return wide


def _run_large(case):
    x = _device_inputs(case)
    send = [x[r] for r in range(case.nranks)]
    recv_big = torch.empty((case.nranks, x.stride(0)), dtype=x.dtype, device="cuda")[:, :case.count]
    recv = [recv_big[r] for r in range(case.nranks)]
    ws = B.Workspace(case.nranks, case.mask, case.proto, case.buff_size)
    B.allreduce(send, recv, case.ring, case.mask, case.proto, ws, case.buff_size, case.chunk_steps)
    assert B.get_status(ws) == B.Status.OK
    # every rank holds the same bytes as rank 0, which is checked element by element
    raw = recv_big.view(torch.int32 if case.dtype == "f32" else torch.int16)
    for r in range(1, case.nranks):
        assert bool(torch.equal(raw[r], raw[0])), f"rank {r} differs from rank 0"
    check_full(case, x, recv_big[0])


@pytest.mark.parametrize("case", gen.large_cases(), ids=lambda c: c.name)
def test_large_64MiB(case):
    _run_large(case)


def _chunk_elems_of(proto, dtype):
    return oracle.geometry(OPROTO[proto], ODT[dtype], 8, gen.SPARSE_MASK, 1 << 20)["chunk_elems"]


def _sparse_cases():
    return gen.sparse_sweep_cases(_chunk_elems_of, max_bytes=1 << 30)


@pytest.mark.parametrize("case", _sparse_cases(), ids=lambda c: c.name)
def test_sparse_mask_size_sweep(case):
    if case.count <= 1 << 20:
        x, got, _ = run_ring(case)
        assert_bit_exact(got, oracle_full(case, x))
        assert_naive_bound(x, got, case.dtype)
    else:
        _run_large(case)


# ---------------------------------------------------------------------------
# LL128: the bulk (TMA-staged) form for first-loop chunks of at least 960
# elements, the polling form below that; both must give the oracle's bytes
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,count,mask", [(2, 3840 * 3 + 5, 0b1), (3, 100003, 0b11), (5, 250001, 0b100101)])
def test_ll128_bulk_form(n, count, mask, dtype, in_place):
    case = gen.RingCase("ll128bulk", n, gen.ring_permutation(n, count % 97), mask, "LL128", count, dtype, "normal",
                        count % 1000, 0, 4)
    x = case.inputs()
    want = oracle_full(case, x)
    _, got, _ = run_ring(case, x=x, in_place=in_place)
    assert_bit_exact(got, want)


def test_ll128_forms_alternate_on_one_workspace():
    ws = B.Workspace(4, 0b11, "LL128", 0)
    for k, count in enumerate([1000, 200003, 777, 150000, 3, 300001]):
        dtype = "bf16" if k % 2 else "f32"
        case = gen.RingCase("alt", 4, gen.RING_0231, 0b11, "LL128", count, dtype, "normal", 70 + k, 0, 4)
        x, got, _ = run_ring(case, workspace=ws)
        assert_bit_exact(got, oracle_full(case, x))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("proto,thr", [("LL", 1024), ("LL128", 960)])
def test_line_forms_at_the_bulk_threshold(proto, thr, dtype):
    """First-loop chunks just below, at and above the bulk form's threshold
    (LL 1024, LL128 960 elements) on one workspace, so that the two forms
    alternate; odd calls end in a ragged chunk."""
    n = 3
    e = 4 if dtype == "f32" else 8
    ws = B.Workspace(n, 0b1, proto, 0)
    for k, chunk in enumerate([thr - e, thr, thr + e, thr - e, 4 * thr]):
        count = n * chunk - (k % 2)
        case = gen.RingCase("thr", n, [0, 2, 1], 0b1, proto, count, dtype, "normal", 80 + k, 0, 4)
        x, got, _ = run_ring(case, workspace=ws)
        assert_bit_exact(got, oracle_full(case, x))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("buff", [4 << 10, 64 << 10, 1 << 20])
def test_simple_sizes_follow_each_other_on_one_workspace(dtype, buff):
    """Simple calls of very different sizes on one workspace (the step counters
    carry over from call to call): first-loop chunks around 1024 elements,
    ragged chunks, empty slices, one loop and many; with 4 KiB buffers
    (512-element chunks) hundreds of loops."""
    n = 4
    e = 4 if dtype == "f32" else 8
    ws = B.Workspace(n, 0b1011, "Simple", buff)
    counts = [3 * n * 1024, 3 * n * (1024 + e), 5, 3 * n * (1024 - e) - 1, 300001, 4096, 2_000_003, 1000]
    for k, count in enumerate(counts):
        case = gen.RingCase("simple_alt", n, gen.RING_0231, 0b1011, "Simple", count, dtype, "normal", 90 + k, buff, 4)
        x, got, _ = run_ring(case, workspace=ws)
        assert_bit_exact(got, oracle_full(case, x))


def test_too_many_blocks_is_refused():
    """32 ranks x 8 channels = 256 blocks cannot all be resident on 152 SMs:
    the cooperative launch is refused with a status, nothing hangs."""
    n, mask, count = 32, 0xFF, 4096
    x = gen.draw("normal", n, count, 1)
    _, send = to_device(x, "f32")
    _, recv = guarded_outputs(n, count, "f32")
    ws = B.Workspace(n, mask, "Simple", 65536)
    with pytest.raises(B.RarError) as e:
        B.allreduce(send, recv, list(range(n)), mask, "Simple", ws, 65536, 4)
    assert e.value.status == B.Status.ERR_CORESIDENCY
    torch.cuda.synchronize()


@pytest.mark.parametrize("proto,count,bs", [("Simple", 200000, 65536), ("LL", 200000, 0), ("LL", 200000, 4096),
                                           ("LL128", 20000, 65536), ("LL128", 400000, 131072),
                                           ("Simple", 600000, 1 << 20), ("LL128", 300000, 524288)])
def test_dropped_head_times_out_and_recovers(proto, count, bs):
    """Failure detection without a GPU fault: with the receivers' head
    updates dropped, every sender runs out of credit after NCCL_STEPS steps;
    its bounded wait expires, the block raises the workspace's abort flag,
    every block leaves, the launch completes and the status reads TIMEOUT.
    Re-initialising the workspace restores normal, bit-exact operation. The
    sizes give every connection more than NCCL_STEPS steps; the two LL128
    cases use the polling and the bulk form, the LL case with a 4 KiB buffer
    the polling form whose block meets every NCCL_STEPS / 2 steps (the sender
    then waits for credit at a group boundary); the last Simple and LL128
    cases split every (rank, channel) over two blocks (first-loop chunks of
    75000 and 15360 elements), whose senders wait for both receiver parts."""
    case = gen.RingCase("fault", 4, gen.RING_0231, 0b11, proto, count, "f32", "normal", 8, bs, 4)
    x = case.inputs()
    _, send = to_device(x, "f32")
    _, recv = guarded_outputs(4, count, "f32")
    ws = B.Workspace(4, 0b11, proto, bs)
    B.set_spin_timeout_ns(200_000_000)
    try:
        B.debug_set_fault(1)
        B.allreduce(send, recv, case.ring, case.mask, proto, ws, bs, 4)
        assert B.get_status(ws) == B.Status.ERR_TIMEOUT
        B.debug_set_fault(0)
        # the workspace stays aborted until it is initialised again
        B.allreduce(send, recv, case.ring, case.mask, proto, ws, bs, 4)
        assert B.get_status(ws) == B.Status.ERR_ABORT
    finally:
        B.debug_set_fault(0)
        B.set_spin_timeout_ns(5_000_000_000)
    ws.init()
    x2, got, _ = run_ring(case, workspace=ws)
    assert_bit_exact(got, oracle_full(case, x2))


# ---------------------------------------------------------------------------
# many ranks: up to the library's 32, as many channels as still fit one
# block per SM (N x C <= 152)
# ---------------------------------------------------------------------------
def _many_rank_cases():
    rng = np.random.default_rng(4321)
    out = []
    for k, (n, mask) in enumerate([(32, 0b1111), (24, 0b111111), (16, 0x1FF), (9, 0xFFFF), (32, 0x1),
                                   (17, 0b101)]):
        for proto in ("Simple", "LL", "LL128"):
            dtype = "bf16" if (k + len(out)) % 2 else "f32"
            count = int(rng.integers(1, 400000))
            ring = rng.permutation(n).tolist()
            bs = 65536 if proto == "Simple" else 0
            out.append(gen.RingCase(f"many_n{n}_{proto}_{dtype}_m{mask:x}_c{count}", n, ring, mask, proto, count,
                                    dtype, "normal", 5000 + len(out), bs, 4))
    return out


@pytest.mark.parametrize("case", _many_rank_cases(), ids=lambda c: c.name)
def test_many_ranks(case):
    x, got, _ = run_ring(case)
    assert_bit_exact(got, oracle_full(case, x))


@pytest.mark.parametrize("proto", ["Simple", "LL", "LL128"])
def test_32_ranks_with_a_ring_per_channel(proto):
    n, mask, count = 32, 0b1111, 77777
    rings = [gen.ring_permutation(n, 60 + ch) for ch in range(4)]
    x = gen.draw("normal", n, count, 61, "f32")
    _, send = to_device(x, "f32")
    big_out, recv = guarded_outputs(n, count, "f32")
    bs = 65536 if proto == "Simple" else 0
    ws = B.Workspace(n, mask, proto, bs)
    B.allreduce_ex(send, recv, rings, mask, proto, ws, bs, 4)
    assert B.get_status(ws) == B.Status.OK
    check_guards(big_out, count, "f32")
    want = oracle.ring_allreduce_closed(list(x), rings, mask, OPROTO[proto], bs, 4)
    assert_bit_exact(device_rows_numpy(recv, "f32"), want)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("bs", [1 << 20, 4 << 20])
def test_ll_bulk_steps_of_several_tiles(bs, dtype):
    """LL buffers larger than the default: a step holds several 8192-element
    tiles (2 with 1 MiB, 8 with 4 MiB), paced once per step, with a ragged
    last loop."""
    n, mask = 4, 0b101
    count = 3 * n * (bs // 64) + 77
    case = gen.RingCase("llbig", n, [2, 0, 3, 1], mask, "LL", count, dtype, "normal", 31, bs, 4)
    x, got, _ = run_ring(case)
    assert_bit_exact(got, oracle_full(case, x))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("bs", [4096, 8192, 16384])
def test_ll_polling_groups_over_many_loops(bs, dtype):
    """LL with small buffers: every step fits one pass of the block, so the
    polling form's block meets only every NCCL_STEPS / 2 steps (heads
    published and credits taken there); many loops per channel, several calls
    on one workspace (step counters carry over), a ragged last loop, in place
    on the last call."""
    n, mask = 8, 0xFFF
    ring = gen.ring_permutation(n, 41)
    ws = B.Workspace(n, mask, "LL", bs)
    for k, count in enumerate([300007, 77777, 131072 + 5]):
        case = gen.RingCase("llgroups", n, ring, mask, "LL", count, dtype, "normal", 300 + k, bs, 4)
        x = case.inputs()
        want = oracle_full(case, x)
        _, got, _ = run_ring(case, x=x, workspace=ws, in_place=(k == 2))
        assert_bit_exact(got, want)
        assert_naive_bound(x, got, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_ll_polling_one_pass_of_1024_threads(dtype):
    """LL steps of 257..512 units (first-loop chunks of 514..1022 f32
    elements, below the bulk form's 1024): the polling form runs 1024 threads
    so that a step is one pass, with barrier groups; two calls on one
    workspace, the second ragged."""
    n, mask = 8, 0xFFF
    ring = gen.ring_permutation(n, 43)
    ws = B.Workspace(n, mask, "LL", 0)
    for k, count in enumerate([65536, 12 * 8 * 1000 + 7]):
        case = gen.RingCase("ll1024", n, ring, mask, "LL", count, dtype, "normal", 310 + k, 0, 4)
        x, got, _ = run_ring(case, workspace=ws)
        assert_bit_exact(got, oracle_full(case, x))
        assert_naive_bound(x, got, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n,mask,ring", [(4, 0b1, [0, 2, 3, 1]), (2, 0b10, [1, 0]), (8, 0b101101011011, None)])
@pytest.mark.parametrize("proto,chunk", [("LL128", 15360), ("LL", 8192)])
def test_line_bulk_steps_of_changing_size(proto, chunk, n, mask, ring, dtype):
    """LL128's bulk form split over two blocks per (rank, channel) (grids
    that fit the SMs twice): each half moves a fixed element range of every
    step, and the split point follows the step's size, so FIFO slots are
    reused by steps of different sizes (full chunks, the short last loop, the
    other calls') and a sender writes a slot only once both receiver halves
    released it. LL's bulk form (one block per pair) on the same calls. 512 KiB
    buffers (chunks of 15360 LL128 / 8192 LL elements): several loops per
    channel, each slot reused several times; calls of different sizes on one
    workspace, polling-form calls between them, the last in place."""
    ring = ring or gen.ring_permutation(n, 47)
    bs = 512 << 10
    ws = B.Workspace(n, mask, proto, bs)
    loop = n * chunk * bin(mask).count("1")
    for k, count in enumerate([3 * loop + 1234, 700, 2 * loop + 7, 25, loop - 5]):
        case = gen.RingCase("linesplit", n, ring, mask, proto, count, dtype, "normal", 320 + k, bs, 4)
        x = case.inputs()
        want = oracle_full(case, x)
        _, got, _ = run_ring(case, x=x, workspace=ws, in_place=(k == 4))
        assert_bit_exact(got, want)
        assert_naive_bound(x, got, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("cs", [4, 2])
@pytest.mark.parametrize("n,mask,ring", [(4, 0b1, [0, 2, 3, 1]), (3, 0b101, [2, 0, 1])])
def test_simple_split_slices_of_changing_size(n, mask, ring, cs, dtype):
    """The Simple kernel split over two blocks per (rank, channel) (grids
    that fit the SMs twice, first-loop chunks of at least 65536 elements):
    each part moves a fixed element range of every slice and publishes its
    own tail; the split point follows the slice's size, so FIFO slots are
    reused by slices of different sizes (full chunks, the short last loop)
    and a sender takes a slot only once both receiver parts released it.
    1 MiB buffers (131072- or 65536-element chunks, one or two steps per
    slice); split and unsplit calls alternate on one workspace (the step
    counters carry over), the last in place."""
    bs = 1 << 20
    ws = B.Workspace(n, mask, "Simple", bs)
    chunk = bs // 8 * cs // 4
    loop = n * chunk * bin(mask).count("1")
    for k, count in enumerate([3 * loop + 12345, 5000, 2 * loop + 7, 100, loop]):
        case = gen.RingCase("simplesplit", n, ring, mask, "Simple", count, dtype, "normal", 340 + k, bs, cs)
        x = case.inputs()
        want = oracle_full(case, x)
        _, got, _ = run_ring(case, x=x, workspace=ws, in_place=(k == 4))
        assert_bit_exact(got, want)
        assert_naive_bound(x, got, dtype)
