"""GPU parity for the two halves of the ring AllReduce run as collectives of
their own (rar_reduce_scatter, rar_all_gather), bit-exact against the oracle's
closed forms, with guard bands around every receive buffer."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_communication_gb300 import binding as B
from collective_communication_gb300 import inputs as gen
from gpu_util import check_guards, device_rows_numpy, guarded_outputs, to_device

pytestmark = pytest.mark.gpu
RS, AG = oracle.REDUCE_SCATTER, oracle.ALL_GATHER
OPROTO = {"LL": oracle.LL, "LL128": oracle.LL128, "Simple": oracle.SIMPLE}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    B.load_library()
    B.set_spin_timeout_ns(5_000_000_000)
    yield


def _compare(got, want):
    for r in range(len(want)):
        assert got[r].tobytes() == want[r].tobytes(), f"rank {r}"


def run_half(kind, n, rings, mask, count, dtype, bs=65536, cs=4, direct=False, seed=0, ws=None, in_place=False,
             proto="Simple"):
    """One call of `kind` with blocks of `count` elements; checks it against
    the oracle and returns the workspace."""
    ws = ws or B.Workspace(n, mask, proto, bs)
    big_count = n * count
    if kind == RS:
        x = gen.draw("normal", n, big_count, seed, dtype)
        big_in, send = to_device(x, dtype)
        if in_place:
            recv = [send[r][r * count:(r + 1) * count] for r in range(n)]
        else:
            big_out, recv = guarded_outputs(n, count, dtype)
        B.reduce_scatter(send, recv, rings, mask, proto, ws, bs, cs)
    else:
        x = gen.draw("normal", n, count, seed, dtype)
        if in_place:
            big_out, recv = guarded_outputs(n, big_count, dtype)
            _, src = to_device(x, dtype)
            send = [recv[r][r * count:(r + 1) * count] for r in range(n)]
            for r in range(n):
                send[r].copy_(src[r])
        else:
            big_in, send = to_device(x, dtype)
            big_out, recv = guarded_outputs(n, big_count, dtype)
        B.all_gather(send, recv, rings, mask, proto, ws, bs, cs, direct=direct)
    assert B.get_status(ws) == B.Status.OK
    if not (in_place and kind == RS):
        check_guards(big_out, count if kind == RS else big_count, dtype)
    got = device_rows_numpy(recv, dtype)
    want = oracle.ring_halves_closed(kind, list(x), rings, mask, OPROTO[proto], bs, cs)
    _compare(got, want)
    return ws


def _random_case(seed, counts):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 9))
    mask = int(rng.integers(1, 1 << 12))
    bs = 4096 * int(rng.integers(1, 65))
    cs = int(rng.choice([1, 2, 4]))
    count = counts[seed % len(counts)]
    nch = bin(mask).count("1")
    rings = [rng.permutation(n).tolist() for _ in range(nch)] if seed % 2 else rng.permutation(n).tolist()
    return n, mask, bs, cs, count, rings


# block sizes: one element, fewer than the channels, ragged (not a multiple
# of 16 bytes, so the blocks are not aligned), several chunks per channel
COUNTS = [1, 5, 1000, 4093, 65536, 250001, 1 << 20]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("seed", range(14))
def test_reduce_scatter_random(seed, dtype):
    n, mask, bs, cs, count, rings = _random_case(seed, COUNTS)
    run_half(RS, n, rings, mask, count, dtype, bs, cs, seed=seed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("direct", [False, True])
@pytest.mark.parametrize("seed", range(14))
def test_all_gather_random(seed, direct, dtype):
    n, mask, bs, cs, count, rings = _random_case(100 + seed, COUNTS)
    run_half(AG, n, rings, mask, count, dtype, bs, cs, direct=direct, seed=seed)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", [RS, AG])
def test_in_place(kind, dtype):
    for k, count in enumerate([8, 4096, 300000]):
        ring = gen.ring_permutation(5, k)
        run_half(kind, 5, ring, 0x0F0, count, dtype, 32768, [4, 2, 1][k], seed=k, in_place=True,
                 direct=(kind == AG and k % 2 == 1))


@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", [RS, AG])
def test_ll128_whole_tiles(kind, dtype, in_place):
    """LL128 with its default buffer and blocks of several whole 7680-element
    tiles (with and without a ragged tail): the bulk form's whole-tile path
    on the halves' own rows (recvReduceCopy, copySend)."""
    for k, (n, count, mask) in enumerate([(4, 40000, 0b1), (3, 7680 * 4, 0b10), (6, 7680 * 2 + 16, 0b1001)]):
        ring = gen.ring_permutation(n, 11 + k)
        run_half(kind, n, ring, mask, count, dtype, 0, 4, seed=k, in_place=in_place, proto="LL128")


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_allgather_of_reducescatter_is_allreduce_on_the_gpu(dtype):
    """Ring 0..n-1, one channel, one chunk per block: the two halves give the
    AllReduce bit for bit (the oracle pins the same identity)."""
    n, bs = 8, 1 << 20
    count = 8192  # elements per block; n blocks fit one AllReduce loop of 8 chunks of 32768
    ring = list(range(n))
    x = gen.draw("normal", n, n * count, 42, dtype)
    _, send = to_device(x, dtype)
    ws = B.Workspace(n, 0x1, "Simple", bs)
    _, mid = guarded_outputs(n, count, dtype)
    _, out = guarded_outputs(n, n * count, dtype)
    _, ar = guarded_outputs(n, n * count, dtype)
    B.reduce_scatter(send, mid, ring, 0x1, "Simple", ws, bs, 4)
    B.all_gather(mid, out, ring, 0x1, "Simple", ws, bs, 4)
    B.allreduce(send, ar, ring, 0x1, "Simple", ws, bs, 4)
    assert B.get_status(ws) == B.Status.OK
    _compare(device_rows_numpy(out, dtype), device_rows_numpy(ar, dtype))


def test_three_collectives_share_a_workspace():
    """AllReduce, ReduceScatter and AllGather calls alternate on one
    workspace: the step counters carry over and every call is exact."""
    n, mask, bs = 4, 0xFFF, 65536
    ws = B.Workspace(n, mask, "Simple", bs)
    for k in range(9):
        dtype = "f32" if k % 2 else "bf16"
        ring = gen.ring_permutation(n, k)
        count = 20011 + 997 * k
        if k % 3 == 0:
            x = gen.draw("normal", n, count, k, dtype)
            _, send = to_device(x, dtype)
            _, recv = guarded_outputs(n, count, dtype)
            B.allreduce_ex(send, recv, ring, mask, "Simple", ws, bs, 4, direct=(k % 2 == 0))
            assert B.get_status(ws) == B.Status.OK
            want = oracle.ring_allreduce_closed(list(x), ring, mask, oracle.SIMPLE, bs, 4)
            _compare(device_rows_numpy(recv, dtype), want)
        else:
            run_half(RS if k % 3 == 1 else AG, n, ring, mask, count, dtype, bs, [4, 2, 1][k % 3], seed=k, ws=ws,
                     direct=(k % 2 == 0))


@pytest.mark.parametrize("kind", [RS, AG])
def test_large_blocks(kind):
    """8 ranks, 12 channels, 4 MiB blocks (f32), the 1 MiB FIFO of the
    AllReduce headline: many chunk loops per channel."""
    n, mask, bs = 8, 0xFFF, 1 << 20
    count = 1 << 20
    run_half(kind, n, gen.ring_permutation(n, 3), mask, count, "f32", bs, 4, seed=9, direct=(kind == AG))


# LL and LL128 take blocks of whole 16-byte pieces
LINE_COUNTS = [8, 40, 1000, 4096, 65536, 250000, 1 << 20]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("kind", [RS, AG])
@pytest.mark.parametrize("proto", ["LL", "LL128"])
@pytest.mark.parametrize("seed", range(7))
def test_line_protocols(seed, proto, kind, dtype):
    n, mask, bs, cs, count, rings = _random_case(300 + seed, LINE_COUNTS)
    bs = 0 if seed % 2 else bs  # the protocol's default buffer, or a random one
    run_half(kind, n, rings, mask, count, dtype, bs, cs, seed=seed, proto=proto)


@pytest.mark.parametrize("proto", ["LL", "LL128"])
def test_line_protocols_share_a_workspace(proto):
    """The three collectives alternate on one LL / LL128 workspace (the step
    counters, and with them the line flags, carry over from call to call)."""
    n, mask = 5, 0x3F
    ws = B.Workspace(n, mask, proto, 0)
    for k in range(6):
        dtype = "bf16" if k % 2 else "f32"
        ring = gen.ring_permutation(n, 50 + k)
        count = [4000, 96000, 8, 200000, 1024, 77776][k]
        if k % 3 == 0:
            x = gen.draw("normal", n, count, k, dtype)
            _, send = to_device(x, dtype)
            _, recv = guarded_outputs(n, count, dtype)
            B.allreduce(send, recv, ring, mask, proto, ws, 0, 4)
            assert B.get_status(ws) == B.Status.OK
            _compare(device_rows_numpy(recv, dtype),
                     oracle.ring_allreduce_closed(list(x), ring, mask, OPROTO[proto], 0, 4))
        else:
            run_half(RS if k % 3 == 1 else AG, n, ring, mask, count, dtype, 0, 4, seed=k, ws=ws, proto=proto)
