"""C-ABI checks that need no GPU: the library loads, exports every entry point
include/rar.h declares, rejects bad arguments before touching the device, and
computes the same geometry as the oracle (two independent implementations)."""
import ctypes
import os
import re

import numpy as np
import pytest

import oracle
from collective_communication_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from collective_communication_gb300 import build
    build.build()
    return B.load_library()


def declared_functions():
    text = open(os.path.join(ROOT, "include", "rar.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(rar_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert len(names) >= 9
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B.EXPORTED)


def test_strerror_covers_every_status(lib):
    for s in B.Status:
        assert B.strerror(s)


FAKE = 1 << 40  # never dereferenced: every call below fails its checks first


def call(n=4, count=1024, dtype=B.Dtype.F32, op=0, ring=None, mask=1, proto=B.Proto.SIMPLE, bs=65536, cs=4,
         send=None, recv=None, ws=FAKE, wsb=1 << 30):
    ring = list(range(n)) if ring is None else ring
    send = [FAKE + (i << 28) for i in range(n)] if send is None else send
    recv = [FAKE + (1 << 35) + (i << 28) for i in range(n)] if recv is None else recv
    L = B.load_library()
    sp = (ctypes.c_void_p * len(send))(*send)
    rp = (ctypes.c_void_p * len(recv))(*recv)
    rg = (ctypes.c_int * len(ring))(*ring)
    return L.rar_allreduce(sp, rp, n, count, int(dtype), op, rg, mask, int(proto), bs, cs, ws, wsb, None)


def test_argument_errors(lib):
    S = B.Status
    assert call(n=1, ring=[0]) == S.ERR_ARG
    assert call(n=33, ring=list(range(33))) == S.ERR_ARG
    assert call(op=1) == S.ERR_ARG
    assert call(dtype=7) == S.ERR_ARG
    assert call(proto=9) == S.ERR_ARG
    assert call(mask=0) == S.ERR_ARG
    assert call(cs=8) == S.ERR_ARG  # one chunk would fill the credit window: deadlock
    assert call(cs=3) == S.ERR_ARG
    assert call(bs=5000) == S.ERR_ARG
    assert call(proto=B.Proto.LL128, bs=1000) == S.ERR_ARG
    assert call(ring=[0, 1, 1, 2]) == S.ERR_RING
    assert call(ring=[0, 1, 2, 4]) == S.ERR_RING
    assert call(send=[FAKE + 4] + [FAKE + (i << 28) for i in range(1, 4)]) == S.ERR_ALIGN
    # a receive buffer overlapping another rank's send buffer
    assert call(recv=[FAKE + (1 << 28)] + [FAKE + (1 << 35) + (i << 28) for i in range(1, 4)]) == S.ERR_ARG
    # in place is allowed (fails later on the workspace size only)
    same = [FAKE + (i << 28) for i in range(4)]
    assert call(send=same, recv=same, wsb=16) == S.ERR_WORKSPACE
    assert call(ws=0) == S.ERR_WORKSPACE
    assert call(ws=FAKE + 16) == S.ERR_ALIGN
    assert call(wsb=16) == S.ERR_WORKSPACE
    # count 0: nothing is enqueued and nothing fails
    assert call(count=0) == S.OK


def call_static(n=4, count=1024, dtype=B.Dtype.F32, op=0, ring=None, mask=1, proto=B.Proto.SIMPLE, bs=65536,
                cs=4, send=None, recv=None):
    ring = list(range(n)) if ring is None else ring
    send = [FAKE + (i << 28) for i in range(n)] if send is None else send
    recv = [FAKE + (1 << 35) + (i << 28) for i in range(n)] if recv is None else recv
    L = B.load_library()
    sp = (ctypes.c_void_p * len(send))(*send)
    rp = (ctypes.c_void_p * len(recv))(*recv)
    rg = (ctypes.c_int * len(ring))(*ring)
    return L.rar_allreduce_static(sp, rp, n, count, int(dtype), op, rg, mask, int(proto), bs, cs, None)


def test_static_argument_errors_match_and_touch_nothing(lib):
    """rar_allreduce_static refuses bad arguments with rar_allreduce's codes
    before any CUDA call: without a GPU any CUDA call would fail, so a code
    other than ERR_CUDA shows that the refused call reached no CUDA call (and
    so enqueued nothing, cleared nothing)."""
    S = B.Status
    bad = [dict(n=1, ring=[0]), dict(op=1), dict(dtype=7), dict(proto=9), dict(mask=0), dict(cs=8), dict(cs=3),
           dict(bs=5000), dict(proto=B.Proto.LL128, bs=1000), dict(ring=[0, 1, 1, 2]), dict(ring=[0, 1, 2, 4]),
           dict(send=[FAKE + 4] + [FAKE + (i << 28) for i in range(1, 4)]),
           dict(recv=[FAKE + (1 << 28)] + [FAKE + (1 << 35) + (i << 28) for i in range(1, 4)])]
    for kw in bad:
        want = call(**kw)
        assert want != S.OK
        assert call_static(**kw) == want, kw
    # a valid call whose workspace exceeds the array: refused before any CUDA call
    n = 8
    assert B.workspace_bytes(n, 0xFFF, B.Proto.SIMPLE, 1 << 20) > (16 << 20)
    assert call_static(n=n, mask=0xFFF, bs=1 << 20) == S.ERR_WORKSPACE
    # an empty call: nothing to do, no CUDA call
    assert call_static(count=0) == S.OK


def test_oneshot_argument_errors(lib):
    L = B.load_library()
    S = B.Status
    n = 4
    send = (ctypes.c_void_p * n)(*[FAKE + (i << 28) for i in range(n)])
    recv = (ctypes.c_void_p * n)(*[FAKE + (1 << 35) + (i << 28) for i in range(n)])
    assert L.rar_oneshot(send, recv, n, 100, 1, 1, None) == S.ERR_ARG  # op
    assert L.rar_oneshot(send, recv, n, 100, 5, 0, None) == S.ERR_ARG  # dtype
    assert L.rar_oneshot(send, recv, 0, 100, 1, 0, None) == S.ERR_ARG
    assert L.rar_oneshot(send, send, n, 100, 1, 0, None) == S.ERR_ARG  # in place is a race here
    assert L.rar_oneshot(send, recv, n, 0, 1, 0, None) == S.OK


def test_workspace_bytes_formula(lib):
    for n, mask, proto, bs in [(4, 1, B.Proto.SIMPLE, 65536), (8, 0xFFF, B.Proto.SIMPLE, 1 << 20),
                               (8, 0b101101011011, B.Proto.LL128, 0), (2, 3, B.Proto.LL, 0)]:
        c = bin(mask).count("1")
        bs_eff = bs or oracle.default_buffsize(int(proto))
        conn = -(-(n * c * 256) // 4096) * 4096
        assert B.workspace_bytes(n, mask, proto, bs) == 4096 + conn + n * c * bs_eff
    assert B.workspace_bytes(1, 1, B.Proto.SIMPLE, 0) == 0


def _oracle_proto(p):
    return {B.Proto.LL: oracle.LL, B.Proto.LL128: oracle.LL128, B.Proto.SIMPLE: oracle.SIMPLE}[p]


@pytest.mark.parametrize("seed", range(25))
def test_library_geometry_matches_oracle(lib, seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(2, 9))
    proto = B.Proto(int(rng.integers(0, 3)))
    dtype = B.Dtype(int(rng.integers(0, 2)))
    mask = int(rng.integers(1, 1 << 63, dtype=np.uint64)) if seed % 3 == 0 else int(rng.integers(1, 1 << 12))
    count = int(rng.integers(0, 1 << 26))
    bs = {B.Proto.SIMPLE: 4096 * int(rng.integers(1, 1024)), B.Proto.LL: 4096 * int(rng.integers(1, 256)),
          B.Proto.LL128: 4096 * int(rng.integers(1, 2000))}[proto]
    cs = int(rng.choice([1, 2, 4]))
    got = B.describe_geometry(n, count, dtype, mask, proto, bs, cs)
    want = oracle.geometry(_oracle_proto(proto), int(dtype), n, mask, count, bs, cs)
    for k in ("step_bytes", "chunk_elems", "steps_per_slice", "slices_per_chunk", "nchannels", "per_channel",
              "channel_ids", "channels"):
        assert got[k] == want[k], k
    for ch in range(got["nchannels"]):
        loops = oracle.channel_loops(_oracle_proto(proto), int(dtype), n, mask, count, ch, bs, cs)
        assert got["loops"][ch] == len(loops)


def call_ex(n=4, rings=None, nrings=None, mask=0b11, proto=B.Proto.SIMPLE, flags=0, count=1024, ws=FAKE, wsb=1 << 30):
    rings = [list(range(n))] if rings is None else rings
    flat = [v for r in rings for v in r]
    nrings = len(rings) if nrings is None else nrings
    L = B.load_library()
    sp = (ctypes.c_void_p * n)(*[FAKE + (i << 28) for i in range(n)])
    rp = (ctypes.c_void_p * n)(*[FAKE + (1 << 35) + (i << 28) for i in range(n)])
    rg = (ctypes.c_int * len(flat))(*flat)
    return L.rar_allreduce_ex(sp, rp, n, count, 0, 0, rg, nrings, mask, int(proto), 65536, 4, flags, ws, wsb, None)


def test_allreduce_ex_argument_errors(lib):
    S = B.Status
    assert call_ex(count=0) == S.OK
    assert call_ex(rings=[[0, 1, 2, 3], [0, 2, 1, 3]], count=0) == S.OK  # one ring per channel
    assert call_ex(rings=[[0, 1, 2, 3]] * 3) == S.ERR_ARG  # 3 rings for 2 channels
    assert call_ex(rings=[[0, 1, 2, 3], [0, 1, 1, 3]]) == S.ERR_RING
    assert call_ex(flags=1, proto=B.Proto.LL) == S.ERR_ARG  # direct is Simple only
    assert call_ex(flags=1, count=0) == S.OK
    assert call_ex(flags=2) == S.ERR_ARG
    assert call_ex(wsb=16) == S.ERR_WORKSPACE


def call_half(kind, n=4, count=1024, mask=0b11, proto=B.Proto.SIMPLE, flags=0, send=None, recv=None, ws=FAKE,
              wsb=1 << 30, dtype=0, op=0, rings=None):
    rings = [list(range(n))] if rings is None else rings
    flat = [v for r in rings for v in r]
    send = [FAKE + (i << 28) for i in range(n)] if send is None else send
    recv = [FAKE + (1 << 35) + (i << 28) for i in range(n)] if recv is None else recv
    L = B.load_library()
    sp = (ctypes.c_void_p * n)(*send)
    rp = (ctypes.c_void_p * n)(*recv)
    rg = (ctypes.c_int * len(flat))(*flat)
    if kind == "rs":
        return L.rar_reduce_scatter(sp, rp, n, count, dtype, op, rg, len(rings), mask, int(proto), 65536, 4, flags,
                                    ws, wsb, None)
    return L.rar_all_gather(sp, rp, n, count, dtype, rg, len(rings), mask, int(proto), 65536, 4, flags, ws, wsb,
                            None)


@pytest.mark.parametrize("kind", ["rs", "ag"])
def test_halves_argument_errors(lib, kind):
    S = B.Status
    assert call_half(kind, count=0) == S.OK  # empty: nothing enqueued
    # LL and LL128 need 16-byte blocks; a valid call stops at the workspace size
    # here, before any launch (the pointers are not real)
    for proto in (B.Proto.LL, B.Proto.LL128):
        assert call_half(kind, proto=proto, count=1001) == S.ERR_ALIGN
        assert call_half(kind, proto=proto, count=1002, dtype=1) == S.ERR_ALIGN
        assert call_half(kind, proto=proto, wsb=16) == S.ERR_WORKSPACE
        assert call_half(kind, proto=proto, count=1000, wsb=16) == S.ERR_WORKSPACE
    assert call_half(kind, count=1001, wsb=16) == S.ERR_WORKSPACE  # Simple takes ragged blocks
    assert call_half(kind, n=1, rings=[[0]]) == S.ERR_ARG
    assert call_half(kind, rings=[[0, 1, 1, 3]]) == S.ERR_RING
    assert call_half(kind, dtype=7) == S.ERR_ARG
    assert call_half(kind, flags=2) == S.ERR_ARG
    assert call_half(kind, wsb=16) == S.ERR_WORKSPACE
    assert call_half(kind, ws=FAKE + 8) == S.ERR_ALIGN
    assert call_half(kind, send=[FAKE + 4] + [FAKE + (i << 28) for i in range(1, 4)]) == S.ERR_ALIGN
    assert call_half(kind, count=1 << 62) == S.ERR_ARG  # nranks blocks would overflow
    if kind == "rs":
        assert call_half(kind, op=1) == S.ERR_ARG
        assert call_half(kind, flags=1) == S.ERR_ARG  # no final value crosses a ReduceScatter hop
    else:
        assert call_half(kind, flags=1, count=0) == S.OK


@pytest.mark.parametrize("kind", ["rs", "ag"])
def test_halves_buffer_overlap_rules(lib, kind):
    S = B.Status
    n, count = 4, 1024
    blk = count * 4
    base = [FAKE + (i << 28) for i in range(n)]
    other = [FAKE + (1 << 35) + (i << 28) for i in range(n)]
    # in place: the one-block buffer is the rank's own block of the n-block one
    inplace = [b + r * blk for r, b in enumerate(base)]
    if kind == "rs":
        assert call_half(kind, send=base, recv=inplace, count=0) == S.OK
        assert call_half(kind, send=base, recv=inplace, wsb=16) == S.ERR_WORKSPACE  # passed the buffer checks
        # another rank's block, or rank r's recv inside another rank's input
        wrong = [b + ((r + 1) % n) * blk for r, b in enumerate(base)]
        assert call_half(kind, send=base, recv=wrong) == S.ERR_ARG
        assert call_half(kind, send=base, recv=[base[1]] + other[1:]) == S.ERR_ARG
    else:
        assert call_half(kind, send=inplace, recv=base, wsb=16) == S.ERR_WORKSPACE
        wrong = [b + ((r + 1) % n) * blk for r, b in enumerate(base)]
        assert call_half(kind, send=wrong, recv=base) == S.ERR_ARG
        assert call_half(kind, send=[base[1]] + other[1:], recv=base) == S.ERR_ARG
    # two receive buffers overlapping
    assert call_half(kind, send=other, recv=[base[0], base[0] + 16] + base[2:]) == S.ERR_ARG


def test_staged_oneshot_workspace_bytes_formula(lib):
    L = B.load_library()
    for n in (1, 2, 8, 32):
        for count, dt, eb in ((1, 0, 4), (7168 * 512, 1, 2), (1000, 1, 2), (4097, 0, 4)):
            slot = -(-count * eb // 256) * 256
            want = 4096 + -(-n * 640 // 4096) * 4096 + n * 4 * slot
            assert L.rar_oneshot_workspace_bytes(n, count, dt) == want
    assert L.rar_oneshot_workspace_bytes(0, 10, 0) == 0
    assert L.rar_oneshot_workspace_bytes(33, 10, 0) == 0
    assert L.rar_oneshot_workspace_bytes(4, 0, 0) == 0
    assert L.rar_oneshot_workspace_bytes(4, 10, 5) == 0


def call_staged(n=4, count=1024, dtype=0, op=0, send=None, recv=None, ws=FAKE, wsb=1 << 30):
    send = [FAKE + (i << 28) for i in range(n)] if send is None else send
    recv = [FAKE + (1 << 35) + (i << 28) for i in range(n)] if recv is None else recv
    L = B.load_library()
    sp = (ctypes.c_void_p * n)(*send)
    rp = (ctypes.c_void_p * n)(*recv)
    return L.rar_oneshot_staged(sp, rp, n, count, dtype, op, ws, wsb, None)


def test_staged_oneshot_argument_errors(lib):
    S = B.Status
    L = B.load_library()
    assert call_staged(count=0) == S.OK  # empty: nothing enqueued, nothing advanced
    assert call_staged(op=1) == S.ERR_ARG
    assert call_staged(dtype=3) == S.ERR_ARG
    assert call_staged(n=0, send=[], recv=[]) == S.ERR_ARG
    assert call_staged(send=[FAKE + 8] + [FAKE + (i << 28) for i in range(1, 4)]) == S.ERR_ALIGN
    assert call_staged(ws=0) == S.ERR_WORKSPACE
    assert call_staged(ws=FAKE + 16) == S.ERR_ALIGN
    assert call_staged(wsb=4096) == S.ERR_WORKSPACE  # too small for this count
    # in place is allowed (only staged copies are read); other overlaps are not
    base = [FAKE + (i << 28) for i in range(4)]
    assert call_staged(send=base, recv=base, wsb=4096) == S.ERR_WORKSPACE  # passed the buffer checks
    assert call_staged(send=base, recv=[base[1]] + base[1:]) == S.ERR_ARG
    # init: argument errors before any device work
    assert L.rar_oneshot_workspace_init(None, 1 << 30, 4, 1024, 0, None) == S.ERR_WORKSPACE
    assert L.rar_oneshot_workspace_init(FAKE + 16, 1 << 30, 4, 1024, 0, None) == S.ERR_ALIGN
    assert L.rar_oneshot_workspace_init(FAKE, 4096, 4, 1024, 0, None) == S.ERR_WORKSPACE
    assert L.rar_oneshot_workspace_init(FAKE, 1 << 30, 0, 1024, 0, None) == S.ERR_ARG


def test_ll_flag_wrap_setter(lib):
    L = B.load_library()
    S = B.Status
    for bad in (1, 63, 96, 255, 257, 1 << 32 - 1 | 1):
        assert L.rar_debug_set_ll_flag_wrap(bad) == S.ERR_ARG
    for good in (64, 256, 1 << 20, 1 << 31, 0):
        assert L.rar_debug_set_ll_flag_wrap(good) == S.OK
