"""Oracle pins: LL (16-byte) and LL128 (128-byte) line layouts."""
import os

import numpy as np

import oracle


def test_ll_line_layout():
    payload = bytes(range(1, 9))
    lines = oracle.ll_encode(payload, 7)
    # one 16-byte line: data1 | flag1 | data2 | flag2, data1 = low 4 bytes
    assert lines.nbytes == 16
    assert lines.tolist() == [int.from_bytes(payload[:4], "little"), 7,
                              int.from_bytes(payload[4:], "little"), 7]


def test_ll_payload_efficiency_is_half():
    for nbytes in (8, 64, 4096):
        lines = oracle.ll_encode(os.urandom(nbytes), 3)
        assert lines.nbytes == 2 * nbytes


def test_ll_round_trip_and_missing_flags():
    rng = np.random.default_rng(0)
    for nbytes in (1, 7, 8, 9, 100, 1000):
        payload = rng.integers(0, 256, nbytes, dtype=np.uint8).tobytes()
        lines = oracle.ll_encode(payload, 42)
        got, bad = oracle.ll_decode(lines, nbytes, 42)
        assert bad == 0 and got == payload
        # an older generation is not accepted
        got, bad = oracle.ll_decode(lines, nbytes, 43)
        assert got is None and bad == 1
        # one missing second flag on the last line blocks the slice there
        broken = lines.copy()
        broken[-1] = 0
        got, bad = oracle.ll_decode(broken, nbytes, 42)
        assert got is None and bad == len(lines) // 4


def test_ll128_line_layout():
    payload = bytes(range(120))
    lines = oracle.ll128_encode(payload, 0x1234)
    assert lines.nbytes == 128
    assert int(lines[15]) == 0x1234  # word 15 is the flag
    assert lines[:15].tobytes() == payload


def test_ll128_payload_efficiency_is_15_16():
    lines = oracle.ll128_encode(os.urandom(120 * 40), 1)
    assert lines.nbytes * 15 == 120 * 40 * 16


def test_ll128_round_trip_and_missing_flag():
    rng = np.random.default_rng(1)
    for nbytes in (1, 119, 120, 121, 1000, 4800):
        payload = rng.integers(0, 256, nbytes, dtype=np.uint8).tobytes()
        lines = oracle.ll128_encode(payload, 99)
        got, bad = oracle.ll128_decode(lines, nbytes, 99)
        assert bad == 0 and got == payload
        broken = lines.copy()
        broken[15] = 98
        got, bad = oracle.ll128_decode(broken, nbytes, 99)
        assert got is None and bad == 1
