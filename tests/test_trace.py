"""RAR_TRACE: with the variable set, a ring call prints its resolved geometry
to stderr (grid, block -> channel, per-channel range, loops, first chunk,
chunk and slice sizes) before it touches the device. The calls below fail the
workspace check right after the trace, so nothing is launched; the printed
values must equal the oracle's geometry (an implementation of its own)."""
import os
import re
import subprocess
import sys

import pytest

import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

# (nranks, count, dtype, mask, proto, buffSize); dtype 0 = f32, 1 = bf16;
# proto 0 = LL, 1 = LL128, 2 = Simple (the library's and the oracle's codes agree)
CASES = [
    (4, 1024, 0, 0x1, 2, 65536),
    (8, 16777216, 0, 0xFFF, 2, 1 << 20),
    (8, 8 * 131072 * 3 + 13, 1, 0b101101011011, 2, 0),
    (4, 131072, 0, 0xF, 0, 0),
    (5, 250001, 1, 0b100101, 1, 0),
    (3, 7, 0, 0xFF, 1, 0),
]

SCRIPT = r"""
import ctypes, sys
sys.path.insert(0, {root!r})
from collective_communication_gb300 import binding as B
L = B.load_library()
FAKE = 1 << 40  # never dereferenced: the calls stop at the workspace check
for n, count, dtype, mask, proto, bs in {cases!r}:
    send = (ctypes.c_void_p * n)(*[FAKE + (i << 28) for i in range(n)])
    recv = (ctypes.c_void_p * n)(*[FAKE + (1 << 35) + (i << 28) for i in range(n)])
    ring = (ctypes.c_int * n)(*range(n))
    st = L.rar_allreduce(send, recv, n, count, dtype, 0, ring, mask, proto, bs, 4, FAKE, 16, None)
    assert st == int(B.Status.ERR_WORKSPACE), st
"""


def _run(env_value):
    env = dict(os.environ)
    if env_value is None:
        env.pop("RAR_TRACE", None)
    else:
        env["RAR_TRACE"] = env_value
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT, cases=CASES)], env=env,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    return [l for l in r.stderr.splitlines() if l.startswith("rar trace:")]


def test_no_trace_by_default():
    assert _run(None) == []
    assert _run("0") == []


def test_trace_matches_the_oracle_geometry():
    lines = _run("1")
    heads = [i for i, l in enumerate(lines) if re.search(r"rar trace: allreduce ", l)]
    assert len(heads) == len(CASES)
    for k, (n, count, dtype, mask, proto, bs) in enumerate(CASES):
        head = dict(re.findall(r"(\w+)=(\S+)", lines[heads[k]]))
        want = oracle.geometry(proto, dtype, n, mask, count, bs, 4)
        assert int(head["nranks"]) == n and int(head["count"]) == count
        assert int(head["grid"]) == n * want["nchannels"]
        for key in ("step_bytes", "chunk_elems", "steps_per_slice", "slices_per_chunk", "per_channel"):
            assert int(head[key]) == want[key], (k, key)
        end = heads[k + 1] if k + 1 < len(heads) else len(lines)
        chans = [l for l in lines[heads[k] + 1:end] if "channel" in l]
        assert len(chans) == want["nchannels"]
        for c, line in enumerate(chans):
            m = re.search(r"channel (\d+) id (\d+) blocks (\d+)\+(\d+)\*rank offset (\d+) count (\d+) loops (\d+) "
                          r"first_chunk (\d+)", line)
            assert m, line
            dense, cid, b0, stride, off, cnt, loops, first = map(int, m.groups())
            assert dense == c and cid == want["channel_ids"][c]
            assert (b0, stride) == (c, want["nchannels"])  # block b serves rank b / C, dense channel b % C
            assert (off, cnt) == want["channels"][c]
            rows = oracle.channel_loops(proto, dtype, n, mask, count, c, bs, 4)
            assert loops == len(rows)
            assert first == (rows[0][2] if rows else 0)
