"""RAR_TRACE on the GPU: each call names the kernel form it launched, and the
form follows the first-loop chunk thresholds (LL bulk from 1024 elements,
LL128 bulk from 960, the polling forms below); the calls stay bit-exact.
LL128's bulk form and the Simple kernel (large chunks) split every (rank,
channel) over two blocks when twice the grid fits the SMs, and the trace says
so."""
import os
import re
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
from gpu_util import to_device, device_rows_numpy
OP = {{"LL": oracle.LL, "LL128": oracle.LL128, "Simple": oracle.SIMPLE}}
for case in {cases!r}:
    n, count, proto, dtype = case[:4]
    mask = case[4] if len(case) > 4 else 0x1
    x = gen.draw("normal", n, count, 3, dtype)
    _, send = to_device(x, dtype)
    _, recv = to_device(x, dtype)
    ring = list(range(n))
    ws = B.Workspace(n, mask, proto, 0)
    B.allreduce(send, recv, ring, mask, proto, ws, 0, 4)
    assert B.get_status(ws) == B.Status.OK
    want = oracle.ring_allreduce_closed(list(x), ring, mask, OP[proto], 0, 4)
    got = device_rows_numpy(recv, dtype)
    assert all(got[r].tobytes() == want[r].tobytes() for r in range(n))
    print("case done", file=sys.stderr, flush=True)
"""

# (nranks, count, proto, dtype): one channel, so the first chunk is ceil(count / n) aligned
CASES = [
    (4, 4 * 1020, "LL", "f32"), (4, 4 * 1024, "LL", "f32"),
    (4, 4 * 956, "LL128", "f32"), (4, 4 * 960, "LL128", "f32"),
    (4, 4 * 960, "LL128", "bf16"), (4, 1 << 16, "Simple", "f32"),
]
WANT = [r"ring_line_kernel<float, LL, \d+>", r"ring_line_bulk_kernel<float, LL>",
        r"ring_line_kernel<float, LL128, \d+>", r"ring_line_bulk_kernel<float, LL128>",
        r"ring_line_bulk_kernel<bf16, LL128>", r"ring_simple_kernel<float>"]


def _kernel_lines(cases):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    env = dict(os.environ, RAR_TRACE="1")
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                                                             cases=cases)],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    kernels = [l for l in r.stderr.splitlines() if "rar trace:   kernel" in l]
    assert len(kernels) == len(cases), r.stderr[-2000:]
    return kernels


def test_trace_names_the_kernel_form():
    for line, pat in zip(_kernel_lines(CASES), WANT):
        assert re.search(pat, line), (line, pat)


def test_trace_reports_the_split():
    """LL128's bulk form (first-loop chunks of 8000 elements, at least one
    whole tile): 4 ranks on 1 channel and 8 ranks on the sparse 8-channel mask
    (64 blocks) split; 8 ranks on 12 channels (96 blocks: 192 do not fit 152
    SMs) do not; 2000-element chunks do not. LL's bulk form never splits.
    Simple splits a grid that fits twice from first-loop chunks of 65536
    elements."""
    cases = [(4, 4 * 8000, "LL128", "f32", 0x1), (8, 8 * 8 * 8000 + 13, "LL128", "bf16", 0b101101011011),
             (8, 8 * 12 * 8000, "LL128", "f32", 0xFFF), (4, 4 * 2048, "LL", "f32", 0x1),
             (8, 8 * 12 * 2048, "LL", "bf16", 0xFFF), (4, 4 * 65536, "Simple", "f32", 0x1),
             (4, 4 * 65536 - 64, "Simple", "f32", 0x1), (8, 8 * 12 * 65536, "Simple", "bf16", 0xFFF),
             (4, 4 * 2000, "LL128", "f32", 0x1)]
    want = [("ring_line_bulk_kernel", r"grid 8 ", "split 2"), ("ring_line_bulk_kernel", r"grid 128 ", "split 2"),
            ("ring_line_bulk_kernel", r"grid 96 ", "split 1"), ("ring_line_bulk_kernel", r"grid 4 ", "split 1"),
            ("ring_line_bulk_kernel", r"grid 96 ", "split 1"), ("ring_simple_kernel", r"grid 8 ", "split 2"),
            ("ring_simple_kernel", r"grid 4 ", "split 1"), ("ring_simple_kernel", r"grid 96 ", "split 1"),
            ("ring_line_bulk_kernel", r"grid 4 ", "split 1")]
    for line, (kernel, grid, split) in zip(_kernel_lines(cases), want):
        assert kernel in line and re.search(grid, line) and line.rstrip().endswith(split), line
