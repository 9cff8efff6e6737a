"""Seeded synthetic inputs for the ring AllReduce and the one-shot AllReduce.

This module only draws random numbers and names the workloads; it holds none
of the collective's arithmetic. Tests and the benchmark feed the same arrays to
the CUDA library and to the CPU oracle.

Buffers are numpy arrays of shape [nranks, count]: float32 for f32 and uint16
bf16 bit patterns for bf16 (drawn in float32, then rounded to nearest-even by
torch's CPU conversion).
"""
from dataclasses import dataclass, field
from typing import List

import numpy as np

F32, BF16 = "f32", "bf16"
LL, LL128, SIMPLE = "LL", "LL128", "Simple"

KIB = 1024
MIB = 1024 * 1024


def ring_permutation(n: int, seed: int) -> List[int]:
    """A seeded random ring order over n ranks."""
    return [int(v) for v in np.random.default_rng(seed).permutation(n)]


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def draw(kind: str, nranks: int, count: int, seed: int, dtype: str = F32) -> np.ndarray:
    """[nranks, count] values.

    kind: "int8" -> integers uniform in [-8, 8] (both ends included),
          "uniform" -> uniform in [-1, 1), "normal" -> standard normal.
    """
    rng = np.random.default_rng(seed)
    shape = (nranks, count)
    if kind == "int8":
        x = rng.integers(-8, 9, size=shape).astype(np.float32)
    elif kind == "uniform":
        x = (rng.random(shape, dtype=np.float32) * np.float32(2.0) - np.float32(1.0)).astype(np.float32)
    elif kind == "normal":
        x = rng.standard_normal(shape, dtype=np.float32)
    else:
        raise ValueError(kind)
    if dtype == BF16:
        return _to_bf16_bits(x)
    return x


def elem_bytes(dtype: str) -> int:
    return 4 if dtype == F32 else 2


@dataclass
class RingCase:
    """One ring AllReduce workload."""
    name: str
    nranks: int
    ring: List[int]
    mask: int
    proto: str
    count: int
    dtype: str = F32
    kind: str = "normal"
    seed: int = 0
    buff_size: int = 0   # 0 = the protocol's default
    chunk_steps: int = 4

    def inputs(self) -> np.ndarray:
        return draw(self.kind, self.nranks, self.count, self.seed, self.dtype)

    @property
    def bytes_per_rank(self) -> int:
        return self.count * elem_bytes(self.dtype)


@dataclass
class OneShotCase:
    name: str
    nranks: int
    count: int
    dtype: str = BF16
    kind: str = "normal"
    seed: int = 1

    def inputs(self) -> np.ndarray:
        return draw(self.kind, self.nranks, self.count, self.seed, self.dtype)


RING_0231 = [0, 2, 3, 1]
SPARSE_MASK = 0b101101011011


def small_case() -> RingCase:
    """N=4, ring 0-2-3-1, one channel, Simple with a 64 KiB buffer and 4 chunk
    steps; 1024 f32 integers in [-8, 8] per rank (4 KiB), seed 0."""
    return RingCase("n4_ring0231_ch1_simple64k_4KiB_int", 4, RING_0231, 0b1, SIMPLE, 1024,
                    F32, "int8", 0, 64 * KIB, 4)


def sweep_512k_cases() -> List[RingCase]:
    """N=4, ring 0-2-3-1, f32, 512 KiB per rank of uniform(-1,1) values: every
    protocol x 1, 4 and 12 contiguous channels; Simple with a 1 MiB buffer."""
    out = []
    for proto in (LL, LL128, SIMPLE):
        for c in (1, 4, 12):
            out.append(RingCase(f"n4_{proto}_ch{c}_512KiB", 4, RING_0231, (1 << c) - 1, proto,
                                512 * KIB // 4, F32, "uniform", 2,
                                MIB if proto == SIMPLE else 0, 4))
    return out


def large_cases() -> List[RingCase]:
    """N=8, ring = seeded permutation (seed 3), f32, 64 MiB per rank of normal
    values, 12 channels: Simple with 64 KiB, 1 MiB and 4 MiB buffers at 4
    chunk steps, and LL128 with its default buffer."""
    ring = ring_permutation(8, 3)
    out = []
    for bs in (64 * KIB, MIB, 4 * MIB):
        out.append(RingCase(f"n8_simple{bs // KIB}k_ch12_64MiB", 8, ring, 0xFFF, SIMPLE,
                            64 * MIB // 4, F32, "normal", 3, bs, 4))
    out.append(RingCase("n8_ll128_ch12_64MiB", 8, ring, 0xFFF, LL128, 64 * MIB // 4, F32,
                        "normal", 3, 0, 4))
    return out


def oneshot_cases() -> List[OneShotCase]:
    """One-shot bf16, N=8: tensors of 7168 x {1, 8, 64, 512} normal values, seed 1."""
    return [OneShotCase(f"oneshot_bf16_n8_7168x{t}", 8, 7168 * t, BF16, "normal", 1)
            for t in (1, 8, 64, 512)]


def sparse_sweep_cases(chunk_elems_of, max_bytes: int = 1 << 30) -> List[RingCase]:
    """N=8, ring = seeded permutation (seed 5), channel mask 0b101101011011 (8
    channels), f32 and bf16, every protocol, sizes 1 KiB * 4^k up to 1 GiB per
    rank; count = 8*chunk*k + 13 with k = floor(size/(8*chunk)), or size + 13
    when that k is 0, so that the last chunk is ragged. chunk_elems_of(proto,
    dtype) gives the full-chunk element count (the caller's geometry)."""
    ring = ring_permutation(8, 5)
    out = []
    size = KIB
    while size <= max_bytes:
        for dtype in (F32, BF16):
            for proto in (LL, LL128, SIMPLE):
                se = size // elem_bytes(dtype)
                ch = chunk_elems_of(proto, dtype)
                k = se // (8 * ch)
                count = 8 * ch * k + 13 if k > 0 else se + 13
                out.append(RingCase(f"n8_sparse_{proto}_{dtype}_{size // KIB}KiB", 8, ring,
                                    SPARSE_MASK, proto, count, dtype, "normal", 5, 0, 4))
        size *= 4
    return out
