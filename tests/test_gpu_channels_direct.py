"""GPU parity for per-channel ring orders (rar_allreduce_ex) and for the direct
all-gather mode of the Simple protocol, bit-exact against the oracle."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from naive_bound import violations
from collective_communication_gb300 import binding as B
from collective_communication_gb300 import inputs as gen
from golden_io import rows
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


def page_rings(n):
    return [[int(v) for v in ring.split("-")] for nr, _ch, ring in rows("channel_rings.txt") if int(nr) == n]


def run_ex(n, rings, mask, proto, count, dtype, bs=0, cs=4, direct=False, seed=0, ws=None, in_place=False):
    x = gen.draw("normal", n, count, seed, dtype)
    big_in, send = to_device(x, dtype)
    if in_place:
        big_out, recv = big_in, send
    else:
        big_out, recv = guarded_outputs(n, count, dtype)
    ws = ws or B.Workspace(n, mask, proto, bs)
    B.allreduce_ex(send, recv, rings, mask, proto, ws, bs, cs, direct=direct)
    assert B.get_status(ws) == B.Status.OK
    if not in_place:
        check_guards(big_out, count, dtype)
    got = device_rows_numpy(recv, dtype)
    want = oracle.ring_allreduce_closed(list(x), rings, mask, OPROTO[proto], bs, cs)
    for r in range(n):
        a, b = got[r], want[r]
        assert a.tobytes() == b.tobytes(), f"rank {r}"
    return ws


@pytest.mark.parametrize("proto", ["Simple", "LL", "LL128"])
@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("n", [2, 3, 4])
def test_page_channel_rings(n, dtype, proto):
    run_ex(n, page_rings(n), 0xFFF, proto, 300001, dtype, 65536 if proto == "Simple" else 0, seed=n)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("in_place", [False, True])
@pytest.mark.parametrize("case", range(6))
def test_direct_allgather(case, in_place, dtype):
    rng = np.random.default_rng(700 + case)
    n = int(rng.integers(2, 9))
    mask = int(rng.integers(1, 1 << 8))
    count = [5, 1000, 77777, 250001, 1 << 20, 3_000_017][case]
    bs = 4096 * int(rng.integers(1, 65))
    cs = int(rng.choice([1, 2, 4]))
    ring = rng.permutation(n).tolist()
    run_ex(n, ring, mask, "Simple", count, dtype, bs, cs, direct=True, seed=case, in_place=in_place)


def test_direct_and_fifo_calls_share_a_workspace():
    """Direct and FIFO calls, single and per-channel rings, alternate on one
    workspace: the step counters stay consistent and every call is exact."""
    n, mask, bs = 4, 0xFFF, 65536
    ws = B.Workspace(n, mask, "Simple", bs)
    for k in range(8):
        rings = page_rings(4) if k % 3 == 0 else gen.ring_permutation(4, k)
        run_ex(n, rings, mask, "Simple", 123457 + 1000 * k, "f32" if k % 2 else "bf16", bs,
               [4, 2, 1][k % 3], direct=(k % 2 == 0), seed=k, ws=ws)


def test_direct_64MiB_full():
    """Full headline size, direct mode with the page's per-channel rings:
    every rank identical, every element equal to the oracle's closed form
    (computed range by range) and within the naive-sum bound."""
    n, mask, count, bs = 8, 0xFFF, 16 << 20, 1 << 20
    rings = [gen.ring_permutation(8, 100 + ch) for ch in range(12)]
    g = torch.Generator(device="cuda")
    g.manual_seed(9)
    x = torch.randn((n, count), generator=g, device="cuda")
    y = torch.empty_like(x)
    ws = B.Workspace(n, mask, "Simple", bs)
    B.allreduce_ex([x[r] for r in range(n)], [y[r] for r in range(n)], rings, mask, "Simple", ws, bs, 4, direct=True)
    assert B.get_status(ws) == B.Status.OK
    raw = y.view(torch.int32)
    for r in range(1, n):
        assert bool(torch.equal(raw[r], raw[0]))
    span = 1 << 23
    for a in range(0, count, span):
        b = min(count, a + span)
        xs = x[:, a:b].cpu().numpy()
        want, _ = oracle.ring_closed_at(list(xs), rings, mask, oracle.SIMPLE, np.arange(a, b, dtype=np.int64),
                                        count, bs, 4)
        got = y[0, a:b].cpu().numpy()
        assert got.tobytes() == want.tobytes(), f"mismatch in [{a}, {b})"
        assert not violations(xs, got, "f32").bad.any()


def _random_default_buffer_case(seed):
    rng = np.random.default_rng(4000 + seed)
    n = int(rng.integers(2, 13))
    proto = ["LL", "LL128", "Simple"][seed % 3]
    dtype = "bf16" if seed % 2 else "f32"
    mask = int(rng.integers(1, 1 << 12))
    while n * bin(mask).count("1") > 152:  # one block per SM
        mask &= mask - 1
    nch = bin(mask).count("1")
    rings = [rng.permutation(n).tolist() for _ in range(nch)] if seed % 4 >= 2 else rng.permutation(n).tolist()
    count = int(rng.integers(1, 1 << int(rng.integers(1, 22))))
    return n, rings, mask, proto, count, dtype, bool(rng.integers(0, 2))


@pytest.mark.parametrize("seed", range(30))
def test_random_default_buffers(seed):
    """The protocols' default buffers (the forms and tile paths the bench
    uses) over random rank counts up to 12, masks over 12 channels, one ring
    or one per channel, sizes from 1 element to 2 Mi, in place or not."""
    n, rings, mask, proto, count, dtype, in_place = _random_default_buffer_case(seed)
    run_ex(n, rings, mask, proto, count, dtype, 0, 4, seed=seed, in_place=in_place)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_direct_split_over_two_blocks(dtype):
    """The direct all-gather mode with the Simple kernel split over two
    blocks per (rank, channel) (N=4, 2 channels, one ring per channel, 1 MiB
    FIFO: 131072-element chunks): calls of changing size on one workspace,
    direct and FIFO calls alternating, ragged last loops."""
    n, mask, bs = 4, 0b11, 1 << 20
    rings = [[0, 2, 3, 1], [0, 1, 2, 3]]
    loop = n * 131072 * 2
    ws = None
    for k, (count, direct) in enumerate([(2 * loop + 999, True), (loop, False), (3000, True), (3 * loop + 5, True)]):
        ws = run_ex(n, rings, mask, "Simple", count, dtype, bs, 4, direct=direct, seed=350 + k, ws=ws)
