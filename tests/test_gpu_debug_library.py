"""GPU runs of the debug library (RAR_LIBRARY=debug: every ring kernel checks
each slice's user ranges and FIFO footprint before using it). The parity
cases stay bit-exact with no bounds report, across every protocol, both
types, the two halves, in place, direct mode, one ring per channel and
uneven sizes; and with the check's view shifted (fault 3, which moves no
access) the first slice is refused with RAR_ERR_BOUNDS, after which a
re-initialised workspace works again."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np, torch, oracle
from collective_communication_gb300 import binding as B, inputs as gen
from gpu_util import to_device, device_rows_numpy, guarded_outputs, check_guards
assert B.library_path().endswith("librar_debug.so")
B.load_library()
B.set_spin_timeout_ns(5_000_000_000)
OP = {{"LL": oracle.LL, "LL128": oracle.LL128, "Simple": oracle.SIMPLE}}
rng = np.random.default_rng(11)
ncase = 0
for proto in ("Simple", "LL", "LL128"):
    for dtype in ("f32", "bf16"):
        for n, mask, count, bs in ((2, 0x1, 1, 0), (4, 0xF, 131072, 0), (5, 0b101101, 250001, 0),
                                   (8, 0xFFF, 1 << 20, 0), (3, 0x3, 77777, 65536 if proto == "Simple" else 0)):
            nch = bin(mask).count("1")
            rings = [rng.permutation(n).tolist() for _ in range(nch)] if count % 2 else rng.permutation(n).tolist()
            x = gen.draw("normal", n, count, ncase, dtype)
            _, send = to_device(x, dtype)
            in_place = ncase % 3 == 0
            if in_place:
                recv = send
            else:
                big_out, recv = guarded_outputs(n, count, dtype)
            ws = B.Workspace(n, mask, proto, bs)
            direct = proto == "Simple" and ncase % 2 == 1
            B.allreduce_ex(send, recv, rings, mask, proto, ws, bs, 4, direct=direct)
            st = B.get_status(ws)
            assert st == B.Status.OK, (proto, dtype, n, count, st)
            if not in_place:
                check_guards(big_out, count, dtype)
            want = oracle.ring_allreduce_closed(list(x), rings, mask, OP[proto], bs, 4)
            got = device_rows_numpy(recv, dtype)
            assert all(got[r].tobytes() == want[r].tobytes() for r in range(n)), (proto, dtype, n, count)
            ncase += 1
        # the two halves
        for kind in ("rs", "ag"):
            n, mask, block = 4, 0b11, 40000
            ring = [0, 2, 3, 1]
            ws = B.Workspace(n, mask, proto, 0)
            if kind == "rs":
                x = gen.draw("normal", n, n * block, 50 + ncase, dtype)
                _, send = to_device(x, dtype)
                _, recv = guarded_outputs(n, block, dtype)
                B.reduce_scatter(send, recv, ring, mask, proto, ws, 0, 4)
                want = oracle.ring_halves_closed(oracle.REDUCE_SCATTER, list(x), ring, mask, OP[proto], 0, 4)
            else:
                x = gen.draw("normal", n, block, 50 + ncase, dtype)
                _, send = to_device(x, dtype)
                _, recv = guarded_outputs(n, n * block, dtype)
                B.all_gather(send, recv, ring, mask, proto, ws, 0, 4)
                want = oracle.ring_halves_closed(oracle.ALL_GATHER, list(x), ring, mask, OP[proto], 0, 4)
            assert B.get_status(ws) == B.Status.OK, (kind, proto, dtype)
            got = device_rows_numpy(recv, dtype)
            assert all(got[r].tobytes() == want[r].tobytes() for r in range(n)), (kind, proto, dtype)
            ncase += 1
# fault 3: the check's view is shifted by one buffer; nothing moves, the call is refused
for proto in ("Simple", "LL", "LL128"):
    n, count = 4, 100000
    x = gen.draw("normal", n, count, 7, "f32")
    _, send = to_device(x, "f32")
    _, recv = guarded_outputs(n, count, "f32")
    ws = B.Workspace(n, 0x3, proto, 0)
    B.set_spin_timeout_ns(200_000_000)
    B.debug_set_fault(3)
    try:
        B.allreduce(send, recv, [0, 2, 3, 1], 0x3, proto, ws, 0, 4)
        assert B.get_status(ws) == B.Status.ERR_BOUNDS, proto
    finally:
        B.debug_set_fault(0)
        B.set_spin_timeout_ns(5_000_000_000)
    ws.init()
    B.allreduce(send, recv, [0, 2, 3, 1], 0x3, proto, ws, 0, 4)
    assert B.get_status(ws) == B.Status.OK
    want = oracle.ring_allreduce_closed(list(x), [0, 2, 3, 1], 0x3, OP[proto], 0, 4)
    got = device_rows_numpy(recv, "f32")
    assert all(got[r].tobytes() == want[r].tobytes() for r in range(n))
    ncase += 1
print("cases", ncase)
"""


def test_debug_library_parity_and_bounds_report():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    env = dict(os.environ, RAR_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"))],
                       env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stderr[-3000:]
    assert "cases" in r.stdout
