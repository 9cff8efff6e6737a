"""Thin Python binding of librar.so (include/rar.h): argument marshalling only.

Every step of the collectives runs in the library's CUDA kernels. Torch
provides device memory (tensors) and streams; nothing here computes on data.
If the library is missing the binding raises -- there is no fallback path.
"""
import ctypes
import enum
import os
from typing import Optional, Sequence

HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_NAME = "librar.so"
_lib = None


class Status(enum.IntEnum):
    OK = 0
    ERR_ARG = 1
    ERR_RING = 2
    ERR_ALIGN = 3
    ERR_WORKSPACE = 4
    ERR_CORESIDENCY = 5
    ERR_CUDA = 6
    ERR_TIMEOUT = 7
    ERR_ABORT = 8
    ERR_BOUNDS = 9


class Dtype(enum.IntEnum):
    F32 = 0
    BF16 = 1


class Proto(enum.IntEnum):
    LL = 0
    LL128 = 1
    SIMPLE = 2


PROTO_BY_NAME = {"LL": Proto.LL, "LL128": Proto.LL128, "Simple": Proto.SIMPLE, "SIMPLE": Proto.SIMPLE}
EXPORTED = (
    "rar_workspace_bytes", "rar_workspace_init", "rar_allreduce", "rar_oneshot", "rar_get_status",
    "rar_strerror", "rar_set_spin_timeout_ns", "rar_debug_set_fault", "rar_describe_geometry",
    "rar_allreduce_static", "rar_allreduce_ex", "rar_reduce_scatter", "rar_all_gather",
    "rar_oneshot_workspace_bytes", "rar_oneshot_workspace_init", "rar_oneshot_staged",
    "rar_debug_set_ll_flag_wrap",
)


class RarError(RuntimeError):
    def __init__(self, status, what=""):
        self.status = Status(status)
        super().__init__(f"{what}: {self.status.name} ({strerror(self.status)})")


def library_path() -> str:
    """librar.so, or with RAR_LIBRARY=debug in the environment the debug build
    librar_debug.so (slice bounds checked on the device, RAR_ERR_BOUNDS)."""
    if os.environ.get("RAR_LIBRARY", "") == "debug":
        return os.path.join(HERE, "librar_debug.so")
    return os.path.join(HERE, _LIB_NAME)


def load_library():
    """Load librar.so (built in-tree by collective_communication_gb300/build.py)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python collective_communication_gb300/build.py` "
                           "(or __graft_entry__.build()); there is no fallback implementation")
    L = ctypes.CDLL(path)
    P, I, U64, SZ = ctypes.c_void_p, ctypes.c_int, ctypes.c_uint64, ctypes.c_size_t
    L.rar_workspace_bytes.argtypes = [I, U64, I, SZ]
    L.rar_workspace_bytes.restype = SZ
    L.rar_workspace_init.argtypes = [P, SZ, I, U64, I, SZ, P]
    L.rar_workspace_init.restype = I
    L.rar_allreduce.argtypes = [P, P, I, SZ, I, I, P, U64, I, SZ, I, P, SZ, P]
    L.rar_allreduce.restype = I
    L.rar_oneshot.argtypes = [P, P, I, SZ, I, I, P]
    L.rar_oneshot.restype = I
    L.rar_get_status.argtypes = [P, P]
    L.rar_get_status.restype = I
    L.rar_strerror.argtypes = [I]
    L.rar_strerror.restype = ctypes.c_char_p
    L.rar_set_spin_timeout_ns.argtypes = [U64]
    L.rar_set_spin_timeout_ns.restype = None
    L.rar_debug_set_fault.argtypes = [I]
    L.rar_debug_set_fault.restype = None
    L.rar_describe_geometry.argtypes = [I, SZ, I, U64, I, SZ, I, P]
    L.rar_describe_geometry.restype = I
    L.rar_allreduce_static.argtypes = [P, P, I, SZ, I, I, P, U64, I, SZ, I, P]
    L.rar_allreduce_static.restype = I
    L.rar_allreduce_ex.argtypes = [P, P, I, SZ, I, I, P, I, U64, I, SZ, I, ctypes.c_uint, P, SZ, P]
    L.rar_allreduce_ex.restype = I
    L.rar_reduce_scatter.argtypes = [P, P, I, SZ, I, I, P, I, U64, I, SZ, I, ctypes.c_uint, P, SZ, P]
    L.rar_reduce_scatter.restype = I
    L.rar_all_gather.argtypes = [P, P, I, SZ, I, P, I, U64, I, SZ, I, ctypes.c_uint, P, SZ, P]
    L.rar_all_gather.restype = I
    L.rar_oneshot_workspace_bytes.argtypes = [I, SZ, I]
    L.rar_oneshot_workspace_bytes.restype = SZ
    L.rar_oneshot_workspace_init.argtypes = [P, SZ, I, SZ, I, P]
    L.rar_oneshot_workspace_init.restype = I
    L.rar_oneshot_staged.argtypes = [P, P, I, SZ, I, I, P, SZ, P]
    L.rar_oneshot_staged.restype = I
    L.rar_debug_set_ll_flag_wrap.argtypes = [ctypes.c_uint32]
    L.rar_debug_set_ll_flag_wrap.restype = I
    _lib = L
    return L


def strerror(status) -> str:
    return load_library().rar_strerror(int(status)).decode()


def _check(st, what):
    if st != 0:
        raise RarError(st, what)


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _dtype_of(t) -> Dtype:
    import torch
    if t.dtype == torch.float32:
        return Dtype.F32
    if t.dtype == torch.bfloat16:
        return Dtype.BF16
    raise TypeError(f"unsupported dtype {t.dtype} (float32 or bfloat16)")


def _ptrs(tensors):
    return (ctypes.c_void_p * len(tensors))(*[t.data_ptr() for t in tensors])


def _proto(p) -> Proto:
    return PROTO_BY_NAME[p] if isinstance(p, str) else Proto(p)


def workspace_bytes(nranks: int, mask: int, proto, buff_size: int = 0) -> int:
    return int(load_library().rar_workspace_bytes(nranks, mask, int(_proto(proto)), buff_size))


class Workspace:
    """Device workspace (connector FIFOs and step counters) for one (nranks,
    channel mask, protocol, buffer size) configuration, held in a torch
    uint8 tensor and initialised through rar_workspace_init."""

    def __init__(self, nranks: int, mask: int, proto, buff_size: int = 0, device=None, stream=None):
        import torch
        self.nranks, self.mask, self.proto, self.buff_size = nranks, mask, _proto(proto), buff_size
        nbytes = workspace_bytes(nranks, mask, self.proto, buff_size)
        if nbytes == 0:
            raise RarError(Status.ERR_ARG, "rar_workspace_bytes")
        self.nbytes = nbytes
        self.tensor = torch.empty(nbytes, dtype=torch.uint8, device=device or "cuda")
        self.init(stream)

    @property
    def ptr(self) -> int:
        return self.tensor.data_ptr()

    def init(self, stream=None):
        _check(load_library().rar_workspace_init(self.ptr, self.nbytes, self.nranks, self.mask, int(self.proto),
                                                 self.buff_size, _stream_handle(stream)), "rar_workspace_init")


def allreduce(sendbufs: Sequence, recvbufs: Sequence, ring_order: Sequence[int], mask: int, proto,
              workspace: Workspace, buff_size: int = 0, chunk_steps: int = 4, stream=None) -> None:
    """Enqueue one ring AllReduce (sum) over len(sendbufs) virtual ranks."""
    n = len(sendbufs)
    count = sendbufs[0].numel()
    ring = (ctypes.c_int * n)(*ring_order)
    st = load_library().rar_allreduce(_ptrs(sendbufs), _ptrs(recvbufs), n, count, int(_dtype_of(sendbufs[0])), 0,
                                      ring, mask, int(_proto(proto)), buff_size, chunk_steps, workspace.ptr,
                                      workspace.nbytes, _stream_handle(stream))
    _check(st, "rar_allreduce")


FLAG_DIRECT = 1


def _ring_array(ring_orders):
    """(C array, nrings) for one ring order (a list of ranks) or one per channel."""
    rings = [list(r) for r in ring_orders] if isinstance(ring_orders[0], (list, tuple)) else [list(ring_orders)]
    flat = [int(v) for r in rings for v in r]
    return (ctypes.c_int * len(flat))(*flat), len(rings)


def allreduce_ex(sendbufs: Sequence, recvbufs: Sequence, ring_orders, mask: int, proto, workspace: Workspace,
                 buff_size: int = 0, chunk_steps: int = 4, direct: bool = False, stream=None) -> None:
    """Enqueue one ring AllReduce with one ring order (a list of ranks) or one
    per channel (a list of lists), optionally with direct all-gather writes."""
    n = len(sendbufs)
    ring_arr, nrings = _ring_array(ring_orders)
    st = load_library().rar_allreduce_ex(_ptrs(sendbufs), _ptrs(recvbufs), n, sendbufs[0].numel(),
                                         int(_dtype_of(sendbufs[0])), 0, ring_arr, nrings, mask,
                                         int(_proto(proto)), buff_size, chunk_steps, FLAG_DIRECT if direct else 0,
                                         workspace.ptr, workspace.nbytes, _stream_handle(stream))
    _check(st, "rar_allreduce_ex")


def reduce_scatter(sendbufs: Sequence, recvbufs: Sequence, ring_orders, mask: int, proto, workspace: Workspace,
                   buff_size: int = 0, chunk_steps: int = 4, stream=None) -> None:
    """Enqueue one ring ReduceScatter (sum): sendbufs[r] holds nranks blocks of
    recvbufs[r].numel() elements; recvbufs[r] receives block r reduced."""
    n = len(sendbufs)
    ring_arr, nrings = _ring_array(ring_orders)
    st = load_library().rar_reduce_scatter(_ptrs(sendbufs), _ptrs(recvbufs), n, recvbufs[0].numel(),
                                           int(_dtype_of(sendbufs[0])), 0, ring_arr, nrings, mask,
                                           int(_proto(proto)), buff_size, chunk_steps, 0,
                                           workspace.ptr, workspace.nbytes, _stream_handle(stream))
    _check(st, "rar_reduce_scatter")


def all_gather(sendbufs: Sequence, recvbufs: Sequence, ring_orders, mask: int, proto, workspace: Workspace,
               buff_size: int = 0, chunk_steps: int = 4, direct: bool = False, stream=None) -> None:
    """Enqueue one ring AllGather: recvbufs[r] (nranks blocks) receives every
    rank's sendbufs[b] as block b."""
    n = len(sendbufs)
    ring_arr, nrings = _ring_array(ring_orders)
    st = load_library().rar_all_gather(_ptrs(sendbufs), _ptrs(recvbufs), n, sendbufs[0].numel(),
                                       int(_dtype_of(sendbufs[0])), ring_arr, nrings, mask, int(_proto(proto)),
                                       buff_size, chunk_steps, FLAG_DIRECT if direct else 0,
                                       workspace.ptr, workspace.nbytes, _stream_handle(stream))
    _check(st, "rar_all_gather")


def allreduce_raw(send_ptrs, recv_ptrs, nranks, count, dtype, ring_order, mask, proto, buff_size, chunk_steps,
                  ws_ptr, ws_bytes, stream_handle) -> int:
    """Direct C-ABI call with raw pointers; returns the status code."""
    ring = (ctypes.c_int * len(ring_order))(*ring_order)
    sp = (ctypes.c_void_p * len(send_ptrs))(*send_ptrs)
    rp = (ctypes.c_void_p * len(recv_ptrs))(*recv_ptrs)
    return int(load_library().rar_allreduce(sp, rp, nranks, count, int(dtype), 0, ring, mask, int(_proto(proto)),
                                            buff_size, chunk_steps, ws_ptr, ws_bytes, stream_handle))


def oneshot(sendbufs: Sequence, recvbufs: Sequence, stream=None) -> None:
    """Enqueue one one-shot AllReduce (sum) over len(sendbufs) virtual ranks."""
    n = len(sendbufs)
    st = load_library().rar_oneshot(_ptrs(sendbufs), _ptrs(recvbufs), n, sendbufs[0].numel(),
                                    int(_dtype_of(sendbufs[0])), 0, _stream_handle(stream))
    _check(st, "rar_oneshot")


class OneShotWorkspace:
    """Device workspace of the staged one-shot (torch-allocated, 256-byte
    aligned), initialised for calls of up to max_count elements."""

    def __init__(self, nranks: int, max_count: int, dtype, device=None, stream=None):
        import torch
        if dtype in ("f32", "bf16"):
            dt = Dtype.F32 if dtype == "f32" else Dtype.BF16
        elif isinstance(dtype, torch.dtype):
            dt = Dtype.F32 if dtype == torch.float32 else Dtype.BF16 if dtype == torch.bfloat16 else None
        else:
            dt = Dtype(dtype)
        if dt is None:
            raise TypeError(f"unsupported dtype {dtype} (float32 or bfloat16)")
        self.nbytes = int(load_library().rar_oneshot_workspace_bytes(nranks, max_count, int(dt)))
        if self.nbytes == 0:
            raise RarError(Status.ERR_ARG, "rar_oneshot_workspace_bytes")
        self.buf = torch.empty(self.nbytes + 256, dtype=torch.uint8, device=device or "cuda")
        base = self.buf.data_ptr()
        self._ptr = (base + 255) // 256 * 256
        self.nranks, self.max_count, self.dtype = nranks, max_count, dt
        self.init(stream)

    def init(self, stream=None):
        """(Re-)initialise: zero the counters, record the configuration."""
        _check(load_library().rar_oneshot_workspace_init(self._ptr, self.nbytes, self.nranks, self.max_count,
                                                          int(self.dtype), _stream_handle(stream)),
               "rar_oneshot_workspace_init")

    @property
    def ptr(self) -> int:
        return self._ptr


def oneshot_staged(sendbufs: Sequence, recvbufs: Sequence, workspace: OneShotWorkspace, stream=None) -> None:
    """Enqueue one staged one-shot AllReduce (sum) over len(sendbufs) ranks."""
    n = len(sendbufs)
    st = load_library().rar_oneshot_staged(_ptrs(sendbufs), _ptrs(recvbufs), n, sendbufs[0].numel(),
                                           int(_dtype_of(sendbufs[0])), 0, workspace.ptr, workspace.nbytes,
                                           _stream_handle(stream))
    _check(st, "rar_oneshot_staged")


def get_status(workspace, stream=None) -> Status:
    return Status(load_library().rar_get_status(workspace.ptr, _stream_handle(stream)))


def set_spin_timeout_ns(ns: int) -> None:
    load_library().rar_set_spin_timeout_ns(ns)


def debug_set_fault(fault: int) -> None:
    load_library().rar_debug_set_fault(fault)


def debug_set_ll_flag_wrap(flag_max: int) -> None:
    """LL flag test mode: 0 = production flags, else the wrap period (a power
    of two >= 64) with the slot cleanup."""
    _check(load_library().rar_debug_set_ll_flag_wrap(flag_max), "rar_debug_set_ll_flag_wrap")


def describe_geometry(nranks, count, dtype, mask, proto, buff_size=0, chunk_steps=4):
    """The library's own geometry for a call (host computation, no device work)."""
    import numpy as np
    c = bin(mask).count("1")
    out = np.zeros(6 + 4 * max(c, 1), np.int64)
    st = load_library().rar_describe_geometry(nranks, count, int(dtype), mask, int(_proto(proto)), buff_size,
                                              chunk_steps, out.ctypes.data_as(ctypes.c_void_p))
    _check(st, "rar_describe_geometry")
    C = int(out[4])
    return {
        "step_bytes": int(out[0]),
        "chunk_elems": int(out[1]),
        "steps_per_slice": int(out[2]),
        "slices_per_chunk": int(out[3]),
        "nchannels": C,
        "per_channel": int(out[5]),
        "channel_ids": out[6:6 + C].tolist(),
        "channels": [(int(out[6 + C + 2 * i]), int(out[6 + C + 2 * i + 1])) for i in range(C)],
        "loops": out[6 + 3 * C:6 + 4 * C].tolist(),
    }
