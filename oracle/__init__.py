"""CPU oracle for the ring AllReduce over N virtual ranks, its two halves
(ReduceScatter, AllGather) as collectives of their own, and the one-shot
variant: a plain, slow, step-by-step C implementation plus the closed form of
each result.

TEST INFRASTRUCTURE. Only tests/, the smoke check in __graft_entry__ and the
CPU-baseline leg of bench.py may import this package. The product (the CUDA
library collective_communication_gb300 and its binding) never imports it and
shares no code with it.

Buffers are numpy arrays: float32 for f32, uint16 bit patterns for bf16.

Functions with no independent pin ("parity unpinned"): none. Each exported
function is checked in tests/test_oracle_*.py against values printed on the
pages, hand-derived values, brute force, closed forms or library routines.
"""
import ctypes
import os

import numpy as np

from . import build as _build

NSTEPS = 8
F32, BF16 = 0, 1
LL, LL128, SIMPLE = 0, 1, 2
PROTO_NAMES = {LL: "LL", LL128: "LL128", SIMPLE: "Simple"}
OK, EARG, ERING, EDEADLOCK, ECHECK, ENOMEM = range(6)
SEND, RECV_REDUCE_SEND, RECV_REDUCE_COPY_SEND, RECV_COPY_SEND, RECV, RECV_REDUCE_COPY, COPY_SEND = range(7)
PRIM_NAMES = {
    SEND: "send",
    RECV_REDUCE_SEND: "recvReduceSend",
    RECV_REDUCE_COPY_SEND: "directRecvReduceCopySend",
    RECV_COPY_SEND: "directRecvCopySend",
    RECV: "directRecv",
    RECV_REDUCE_COPY: "recvReduceCopy",
    COPY_SEND: "copySend",
}
ALLREDUCE, REDUCE_SCATTER, ALL_GATHER = 0, 1, 2
M_COMPLETE, M_STALL, M_CORRUPT = 0, 1, 2

_lib = None


class OracleError(RuntimeError):
    def __init__(self, code, what):
        super().__init__(f"oracle {what} failed with code {code}")
        self.code = code


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P, I, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
        L.orc_ring_setup.argtypes = [I, P, P, P, P, P]
        L.orc_schedule.argtypes = [I, I, P, P]
        L.orc_schedule_kind.argtypes = [I, I, I, P, P]
        L.orc_mask_channels.argtypes = [U64, P]
        L.orc_default_buffsize.argtypes = [I]
        L.orc_default_buffsize.restype = SZ
        L.orc_geometry.argtypes = [I, I, I, U64, SZ, SZ, I, P]
        L.orc_channel_loops.argtypes = [I, I, I, U64, SZ, SZ, I, I, P, ctypes.c_int64]
        L.orc_channel_loops.restype = ctypes.c_int64
        L.orc_ll_encode.argtypes = [P, SZ, ctypes.c_uint32, P]
        L.orc_ll_decode.argtypes = [P, SZ, ctypes.c_uint32, P]
        L.orc_ll_decode.restype = SZ
        L.orc_ll128_encode.argtypes = [P, SZ, U64, P]
        L.orc_ll128_decode.argtypes = [P, SZ, U64, P]
        L.orc_ll128_decode.restype = SZ
        L.orc_ring_allreduce_sim.argtypes = [P, P, I, SZ, I, P, I, U64, I, SZ, I, I, P, P, P]
        L.orc_ring_allreduce_closed.argtypes = [P, P, I, SZ, I, P, I, U64, I, SZ, I]
        L.orc_ring_collective_sim.argtypes = [I, P, P, I, SZ, I, P, I, U64, I, SZ, I, I, P, P, P]
        L.orc_ring_halves_closed.argtypes = [I, P, P, I, SZ, I, P, I, U64, I, SZ, I]
        L.orc_ll_session_sim.argtypes = [I, P, P, P, I, I, P, I, U64, SZ, ctypes.c_uint32, I, P, P]
        L.orc_ring_closed_at.argtypes = [P, I, SZ, I, P, I, U64, I, SZ, I, P, SZ, P, P]
        L.orc_oneshot.argtypes = [P, P, I, SZ, I]
        L.orc_state_model.argtypes = [I, I, I, I, P]
        L.orc_bf16_round.argtypes = [P, P, SZ]
        _lib = L
    return _lib


def _ptr(a):
    return a.ctypes.data_as(ctypes.c_void_p)


def _i32(seq):
    return np.ascontiguousarray(np.asarray(seq, dtype=np.int32))


def _rings(ring_order):
    """One ring (a list of ranks) or one ring per dense channel (a list of
    lists) -> (flat int32 array, number of rings)."""
    a = np.asarray(ring_order, dtype=np.int32)
    if a.ndim == 1:
        return np.ascontiguousarray(a), 1
    return np.ascontiguousarray(a.reshape(-1)), a.shape[0]


def _check(code, what):
    if code != OK:
        raise OracleError(code, what)


def _dtype_code(arr):
    if arr.dtype == np.float32:
        return F32
    if arr.dtype == np.uint16:
        return BF16
    raise TypeError("oracle buffers are float32 or uint16 (bf16 bit patterns)")


def _ptr_array(arrays):
    return (ctypes.c_void_p * len(arrays))(*[a.ctypes.data for a in arrays])


def ring_setup(ring_order):
    """Per user rank r: (index[r], prev[r], next[r], user_ranks[r][:])."""
    n = len(ring_order)
    idx, prv, nxt = (np.zeros(n, np.int32) for _ in range(3))
    ur = np.zeros((n, n), np.int32)
    _check(lib().orc_ring_setup(n, _ptr(_i32(ring_order)), _ptr(idx), _ptr(prv), _ptr(nxt), _ptr(ur)),
           "ring_setup")
    return idx, prv, nxt, ur


def ring_setup_status(ring_order):
    n = len(ring_order)
    return lib().orc_ring_setup(n, _ptr(_i32(ring_order)), None, None, None, None)


def schedule(n, ring_index):
    """The 2n-1 (primitive, chunk) rows of the rank with the given ring index."""
    prim = np.zeros(2 * n - 1, np.int32)
    chunk = np.zeros(2 * n - 1, np.int32)
    _check(lib().orc_schedule(n, ring_index, _ptr(prim), _ptr(chunk)), "schedule")
    return list(zip(prim.tolist(), chunk.tolist()))


def mask_channels(mask):
    ids = np.full(64, -1, np.int32)
    c = lib().orc_mask_channels(mask, _ptr(ids))
    return ids[:c].tolist()


def default_buffsize(proto):
    return lib().orc_default_buffsize(proto)


def geometry(proto, dtype, nranks, mask, count, buff_size=0, chunk_steps=4):
    out = np.zeros(6 + 3 * 64, np.int64)
    _check(lib().orc_geometry(proto, dtype, nranks, mask, count, buff_size, chunk_steps, _ptr(out)),
           "geometry")
    c = int(out[4])
    chans = []
    for n in range(c):
        chans.append((int(out[6 + c + 2 * n]), int(out[6 + c + 2 * n + 1])))
    return {
        "step_bytes": int(out[0]),
        "chunk_elems": int(out[1]),
        "steps_per_slice": int(out[2]),
        "slices_per_chunk": int(out[3]),
        "nchannels": c,
        "per_channel": int(out[5]),
        "channel_ids": out[6:6 + c].tolist(),
        "channels": chans,
    }


def channel_loops(proto, dtype, nranks, mask, count, channel, buff_size=0, chunk_steps=4):
    """[(elemOffset, remCount, chunkCount)] of one dense channel."""
    rows = np.zeros(3 * 4096, np.int64)
    k = lib().orc_channel_loops(proto, dtype, nranks, mask, count, buff_size, chunk_steps, channel,
                                _ptr(rows), 4096)
    if k < 0:
        raise OracleError(EARG, "channel_loops")
    return [tuple(int(v) for v in rows[3 * i:3 * i + 3]) for i in range(k)]


def ll_encode(payload: bytes, flag: int):
    p = np.frombuffer(payload, np.uint8).copy() if payload else np.zeros(1, np.uint8)
    nl = (len(payload) + 7) // 8
    lines = np.zeros(max(nl, 1) * 4, np.uint32)
    lib().orc_ll_encode(_ptr(p), len(payload), flag, _ptr(lines))
    return lines[:nl * 4]


def ll_decode(lines, nbytes, flag):
    lines = np.ascontiguousarray(lines, np.uint32)
    out = np.zeros(max(nbytes, 1), np.uint8)
    bad = lib().orc_ll_decode(_ptr(lines), nbytes, flag, _ptr(out))
    return (None if bad else out[:nbytes].tobytes()), int(bad)


def ll128_encode(payload: bytes, flag: int):
    p = np.frombuffer(payload, np.uint8).copy() if payload else np.zeros(1, np.uint8)
    nl = (len(payload) + 119) // 120
    lines = np.zeros(max(nl, 1) * 16, np.uint64)
    lib().orc_ll128_encode(_ptr(p), len(payload), flag, _ptr(lines))
    return lines[:nl * 16]


def ll128_decode(lines, nbytes, flag):
    lines = np.ascontiguousarray(lines, np.uint64)
    out = np.zeros(max(nbytes, 1), np.uint8)
    bad = lib().orc_ll128_decode(_ptr(lines), nbytes, flag, _ptr(out))
    return (None if bad else out[:nbytes].tobytes()), int(bad)


def _prep(inputs):
    ins = [np.ascontiguousarray(a) for a in inputs]
    dt = _dtype_code(ins[0])
    for a in ins:
        if a.dtype != ins[0].dtype or a.shape != ins[0].shape:
            raise ValueError("all ranks need inputs of one dtype and shape")
    return ins, dt


def ring_allreduce_sim(inputs, ring_order, mask, proto, buff_size=0, chunk_steps=4, outputs=None,
                       direct=False):
    """Step-by-step simulation. Returns (outputs, sends, recvs, loops per channel).

    ring_order: one ring, or one ring per dense channel. `outputs` may be given
    (e.g. the inputs themselves, for an in-place call). direct: Simple only,
    all-gather hops write the next rank's output instead of a FIFO slot."""
    ins, dt = _prep(inputs)
    n = len(ins)
    count = ins[0].size
    outs = outputs if outputs is not None else [np.zeros_like(a) for a in ins]
    sends = np.zeros(n, np.int64)
    recvs = np.zeros(n, np.int64)
    loops = np.zeros(64, np.int64)
    rings, nrings = _rings(ring_order)
    st = lib().orc_ring_allreduce_sim(_ptr_array(ins), _ptr_array(outs), n, count, dt, _ptr(rings), nrings,
                                      mask, proto, buff_size, chunk_steps, int(direct),
                                      _ptr(sends), _ptr(recvs), _ptr(loops))
    _check(st, "ring_allreduce_sim")
    return outs, sends, recvs, loops[:len(mask_channels(mask))]


def ring_allreduce_closed(inputs, ring_order, mask, proto, buff_size=0, chunk_steps=4):
    ins, dt = _prep(inputs)
    n = len(ins)
    outs = [np.zeros_like(a) for a in ins]
    rings, nrings = _rings(ring_order)
    st = lib().orc_ring_allreduce_closed(_ptr_array(ins), _ptr_array(outs), n, ins[0].size, dt,
                                         _ptr(rings), nrings, mask, proto, buff_size, chunk_steps)
    _check(st, "ring_allreduce_closed")
    return outs


def ring_closed_at(sampled, ring_order, mask, proto, idx, count, buff_size=0, chunk_steps=4):
    """Closed-form result at element indices idx of a call with `count`
    elements per rank. sampled[r][k] = input of rank r at element idx[k].
    Returns (values, chunk index of each element)."""
    ins, dt = _prep(sampled)
    n = len(ins)
    idx = np.ascontiguousarray(np.asarray(idx, np.int64))
    m = idx.size
    if ins[0].size != m:
        raise ValueError("one sampled value per index and rank")
    out = np.zeros(m, ins[0].dtype)
    chunks = np.zeros(m, np.int32)
    rings, nrings = _rings(ring_order)
    st = lib().orc_ring_closed_at(_ptr_array(ins), n, count, dt, _ptr(rings), nrings, mask,
                                  proto, buff_size, chunk_steps, _ptr(idx), m, _ptr(out),
                                  _ptr(chunks))
    _check(st, "ring_closed_at")
    return out, chunks


def schedule_kind(kind, n, ring_index):
    """Rows (primitive, chunk) of one collective kind for the rank at ring_index."""
    prim = np.zeros(2 * n, np.int32)
    chunk = np.zeros(2 * n, np.int32)
    rows = lib().orc_schedule_kind(kind, n, ring_index, _ptr(prim), _ptr(chunk))
    if rows < 0:
        raise OracleError(rows, "schedule_kind")
    return [(int(p), int(c)) for p, c in zip(prim[:rows], chunk[:rows])]


def _half_buffers(kind, inputs):
    ins, dt = _prep(inputs)
    n = len(ins)
    if kind == REDUCE_SCATTER:
        if ins[0].size % n:
            raise ValueError("a ReduceScatter input holds nranks blocks")
        count = ins[0].size // n
        outs = [np.zeros(count, ins[0].dtype) for _ in ins]
    elif kind == ALL_GATHER:
        count = ins[0].size
        outs = [np.zeros(n * count, ins[0].dtype) for _ in ins]
    else:
        raise ValueError("kind must be REDUCE_SCATTER or ALL_GATHER")
    return ins, dt, n, count, outs


def ring_halves_sim(kind, inputs, ring_order, mask, proto, buff_size=0, chunk_steps=4, direct=False):
    """Step-by-step simulation of a ReduceScatter (inputs of nranks*count
    elements, outputs of count) or an AllGather (inputs of count, outputs of
    nranks*count). Returns (outputs, sends, recvs, loops per channel)."""
    ins, dt, n, count, outs = _half_buffers(kind, inputs)
    sends = np.zeros(n, np.int64)
    recvs = np.zeros(n, np.int64)
    loops = np.zeros(64, np.int64)
    rings, nrings = _rings(ring_order)
    st = lib().orc_ring_collective_sim(kind, _ptr_array(ins), _ptr_array(outs), n, count, dt, _ptr(rings),
                                       nrings, mask, proto, buff_size, chunk_steps, int(direct),
                                       _ptr(sends), _ptr(recvs), _ptr(loops))
    _check(st, "ring_halves_sim")
    return outs, sends, recvs, loops[:len(mask_channels(mask))]


def ring_halves_closed(kind, inputs, ring_order, mask, proto, buff_size=0, chunk_steps=4):
    """Closed form of a ReduceScatter or an AllGather (shapes as in ring_halves_sim)."""
    ins, dt, n, count, outs = _half_buffers(kind, inputs)
    rings, nrings = _rings(ring_order)
    st = lib().orc_ring_halves_closed(kind, _ptr_array(ins), _ptr_array(outs), n, count, dt, _ptr(rings),
                                      nrings, mask, proto, buff_size, chunk_steps)
    _check(st, "ring_halves_closed")
    return outs


def ll_session_sim(calls, ring_order, mask, buff_size=0, flag_max=0, cleanup=True):
    """A sequence of LL ring AllReduce calls on one workspace (FIFOs and step
    counters persist). calls: list of per-rank input lists (one list per call,
    each of nranks equal-length arrays). flag_max 0: production flags, else the
    wrap period (a power of two >= 64). Returns (outputs per call,
    stale_accepts, max_stale_age)."""
    n = len(calls[0])
    ins, outs, counts = [], [], []
    for c in calls:
        arrs, dt = _prep(c)
        if len(arrs) != n:
            raise ValueError("every call needs nranks inputs")
        ins.extend(arrs)
        outs.extend(np.zeros_like(a) for a in arrs)
        counts.append(arrs[0].size)
    dts = {_dtype_code(a) for a in ins}
    if len(dts) != 1:
        raise ValueError("one dtype for the whole session")
    rings, nrings = _rings(ring_order)
    cnt = np.ascontiguousarray(np.asarray(counts, np.uint64))
    stale = np.zeros(1, np.int64)
    age = np.zeros(1, np.int64)
    st = lib().orc_ll_session_sim(len(calls), _ptr(cnt), _ptr_array(ins), _ptr_array(outs), n, dts.pop(),
                                  _ptr(rings), nrings, mask, buff_size, flag_max, int(cleanup), _ptr(stale),
                                  _ptr(age))
    _check(st, "ll_session_sim")
    return [outs[k * n:(k + 1) * n] for k in range(len(calls))], int(stale[0]), int(age[0])


def oneshot(inputs):
    ins, dt = _prep(inputs)
    n = len(ins)
    outs = [np.zeros_like(a) for a in ins]
    _check(lib().orc_oneshot(_ptr_array(ins), _ptr_array(outs), n, ins[0].size, dt), "oneshot")
    return outs


def state_model(proto, fault, slots, total=64):
    res = np.zeros(5, np.int64)
    _check(lib().orc_state_model(proto, fault, slots, total, _ptr(res)), "state_model")
    return {"outcome": int(res[0]), "corrupt_kinds": int(res[1]), "stall_producer": int(res[2]),
            "stall_consumer": int(res[3]), "states": int(res[4])}


def bf16_round(x):
    x = np.ascontiguousarray(x, np.float32)
    y = np.zeros(x.shape, np.uint16)
    lib().orc_bf16_round(_ptr(x), _ptr(y), x.size)
    return y
