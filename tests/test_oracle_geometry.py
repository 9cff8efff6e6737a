"""Oracle pins: block -> channel mapping, chunk geometry, loop/tail chunking, slices."""
import numpy as np
import pytest

import oracle
from golden_io import rows


def test_simple_chunk_geometry_matches_page():
    for buf, step, chunk in rows("simple_chunk_geometry.txt"):
        g = oracle.geometry(oracle.SIMPLE, oracle.F32, 4, 1, 1 << 20, int(buf), 4)
        assert g["step_bytes"] == int(step)
        assert g["chunk_elems"] * 4 == int(chunk)
    # "default" is the 4 MiB row
    g = oracle.geometry(oracle.SIMPLE, oracle.F32, 4, 1, 1 << 20, 0, 4)
    assert g["chunk_elems"] * 4 == 2 * 1024 * 1024


def test_ll_ll128_default_chunks_match_page():
    want = {p: int(b) for p, b in rows("ll_chunk_geometry.txt")}
    g = oracle.geometry(oracle.LL, oracle.F32, 4, 1, 1 << 20)
    assert g["chunk_elems"] * 4 == want["LL"]
    assert g["step_bytes"] == oracle.default_buffsize(oracle.LL) // 8
    assert g["chunk_elems"] * 4 == oracle.default_buffsize(oracle.LL) // 8 // 2
    g = oracle.geometry(oracle.LL128, oracle.F32, 4, 1, 1 << 20)
    assert g["chunk_elems"] * 4 == want["LL128"]
    assert g["step_bytes"] // 128 * 120 == want["LL128"]


@pytest.mark.parametrize("mask", [0b1, 0xF, 0xFFF, 0b101101011011, 0x8000000000000001, (1 << 64) - 1])
def test_block_to_channel_by_popcount(mask):
    ids = oracle.mask_channels(mask)
    # gridX = popcount(mask); block n serves the n-th set bit (brute-force enumeration)
    assert len(ids) == bin(mask).count("1")
    assert ids == [b for b in range(64) if (mask >> b) & 1]


def test_sparse_mask_example():
    assert oracle.mask_channels(0b101101011011) == [0, 1, 3, 4, 6, 8, 9, 11]
    for c in (1, 4, 12):
        assert len(oracle.mask_channels((1 << c) - 1)) == c


def _chunk_ranges(proto, dtype, n, mask, count, bs, cs):
    g = oracle.geometry(proto, dtype, n, mask, count, bs, cs)
    out = []
    for ch, (go, cc) in enumerate(g["channels"]):
        for (eo, rem, cc_) in oracle.channel_loops(proto, dtype, n, mask, count, ch, bs, cs):
            for c in range(n):
                off = c * cc_
                ne = max(0, min(cc_, rem - off))
                out.append((go + eo + off, ne, cc_, rem, ch))
    return g, out


@pytest.mark.parametrize("seed", range(12))
def test_chunks_partition_the_buffer(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(2, 9))
    proto = int(rng.integers(0, 3))
    dtype = int(rng.integers(0, 2))
    mask = int(rng.integers(1, 1 << 12))
    count = int(rng.integers(0, 200000))
    bs = {oracle.SIMPLE: 4096 * int(rng.integers(1, 64)), oracle.LL: 4096 * int(rng.integers(1, 16)),
          oracle.LL128: 4096 * int(rng.integers(1, 16))}[proto]
    cs = int(rng.choice([1, 2, 4]))
    g, ranges = _chunk_ranges(proto, dtype, n, mask, count, bs, cs)
    E = 16 // (4 if dtype == oracle.F32 else 2)
    cover = np.zeros(count, np.int32)
    for start, ne, cc, rem, ch in ranges:
        assert start % E == 0  # every chunk starts 16-byte aligned
        assert cc % E == 0  # tail chunk counts are aligned to 16/sizeof(T)
        assert cc <= g["chunk_elems"]
        assert n * cc >= min(rem, n * g["chunk_elems"])  # the chunks of a loop cover it
        cover[start:start + ne] += 1
    assert (cover == 1).all()
    # channels are contiguous, in dense order
    starts = [go for go, _ in g["channels"]]
    assert starts == sorted(starts)


def test_config3_channel_split():
    g = oracle.geometry(oracle.SIMPLE, oracle.F32, 8, 0xFFF, 16777216, 1 << 20, 4)
    counts = [cc for _, cc in g["channels"]]
    assert counts[:11] == [1398104] * 11 and counts[11] == 1398072
    assert sum(counts) == 16777216


def test_tail_loop_example():
    # 16 elements, N=4: one short loop with chunks of alignUp(divUp(16,4),4) = 4
    loops = oracle.channel_loops(oracle.SIMPLE, oracle.F32, 4, 1, 16, 0, 65536, 4)
    assert loops == [(0, 16, 4)]
    # bf16 aligns the tail chunk to 8 elements
    loops = oracle.channel_loops(oracle.SIMPLE, oracle.BF16, 4, 1, 16, 0, 65536, 4)
    assert loops == [(0, 16, 8)]
