"""The multi-GPU bench path runs independent replicas: its host-side
aggregation (slowest replica's time, bytes of all replicas) is checked with
world_size 2 gloo ranks on CPU."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    dist.barrier()
    local_ms = [10.0, 25.0][rank]  # rank 1 is the slow replica
    ms, value = bench.combine_replicas(local_ms, 5, 64 << 20, 8, world, dist, "cpu")
    out[rank] = (ms, value)
    dist.barrier()
    dist.destroy_process_group()


def test_replicas_take_the_slowest_time_and_sum_the_bytes():
    world = 2
    port = _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    import bench
    single_ms, single_value = bench.combine_replicas(25.0, 5, 64 << 20, 8, 1)
    for rank in range(world):
        ms, value = res[rank]
        assert ms == pytest.approx(5.0)  # 25 ms over 5 steps: the slow replica
        assert value == pytest.approx(2 * single_value)
    assert single_ms == pytest.approx(5.0)
    # busBW of one replica: S / t * 2(N-1)/N
    assert single_value == pytest.approx((64 << 20) / 5e-3 * 2 * 7 / 8 / 1e9)


def test_algorithmic_bytes_of_the_halves_add_up_to_the_allreduce():
    """ReduceScatter then AllGather move the AllReduce's bytes plus the
    intermediate block, written once and read once (2 blocks per rank)."""
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    from collective_communication_gb300 import inputs as gen
    for n, dtype, proto in ((8, "f32", "Simple"), (4, "bf16", "LL128"), (3, "f32", "LL")):
        block = 3000
        eb = 4 if dtype == "f32" else 2
        case = gen.RingCase("x", n, list(range(n)), 1, proto, n * block, dtype, "normal", 0, 0, 4)
        ar = bench.algorithmic_bytes(case)
        halves = (bench.half_algorithmic_bytes("rs", n, block, dtype, proto) +
                  bench.half_algorithmic_bytes("ag", n, block, dtype, proto))
        assert halves == pytest.approx(ar + 2 * n * block * eb)
    # direct AllGather: outputs written once, (n-2) blocks read back, one input block read
    assert bench.half_algorithmic_bytes("ag", 8, 10, "f32", "Simple", True) == 8 * (8 + 1 + 6) * 40
