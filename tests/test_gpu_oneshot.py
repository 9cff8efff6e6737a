"""GPU parity of the one-shot AllReduce against the CPU oracle: bit-exact on
every rank, guard bands intact. Calls go through the C ABI (librar.so)."""
import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle
from collective_communication_gb300 import binding as B
from collective_communication_gb300 import inputs as gen
from gpu_util import check_guards, device_rows_numpy, guarded_outputs, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    B.load_library()
    yield


def run_oneshot(n, count, dtype, kind="normal", seed=1):
    x = gen.draw(kind, n, count, seed, dtype)
    _, send = to_device(x, dtype)
    big_out, recv = guarded_outputs(n, count, dtype)
    B.oneshot(send, recv)
    torch.cuda.synchronize()
    check_guards(big_out, count, dtype)
    got = device_rows_numpy(recv, dtype)
    want = oracle.oneshot(list(x))
    for r in range(n):
        a = got[r].view(np.uint32 if dtype == "f32" else np.uint16)
        b = want[r].view(np.uint32 if dtype == "f32" else np.uint16)
        bad = np.nonzero(a != b)[0]
        assert bad.size == 0, f"rank {r}: {bad.size} mismatches at {bad[:8]}"


@pytest.mark.parametrize("case", gen.oneshot_cases(), ids=lambda c: c.name)
def test_oneshot_bf16_n8(case):
    run_oneshot(case.nranks, case.count, case.dtype, case.kind, case.seed)


@pytest.mark.parametrize("count", [1, 7, 8, 9, 1000, 2048, 4095, 123457])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("n", [2, 3, 8, 16])
def test_oneshot_ragged(n, count, dtype):
    run_oneshot(n, count, dtype, "normal", 10 + n)


def test_oneshot_integer_exact():
    run_oneshot(8, 50000, "bf16", "int8", 3)


@pytest.mark.parametrize("n", [2, 5, 8])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_oneshot_many_tiles(n, dtype):
    """Many grid-stride passes and a ragged end."""
    run_oneshot(n, 8192 * 40 + 4096 + 24 + 3, dtype, "normal", 40 + n)


@pytest.mark.parametrize("n", [1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 32])
@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_oneshot_every_rank_count(n, dtype):
    """Every rank count of the fixed-count kernels (1..8) and of the wide
    kernel (more than 8 ranks, peers read in batches of 8), with enough
    elements that every rank's blocks make several grid-stride passes (the
    grid holds at most 8 blocks per SM), and a ragged end."""
    run_oneshot(n, 1300007, dtype, "normal", 70 + n)
