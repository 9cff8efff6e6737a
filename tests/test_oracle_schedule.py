"""Oracle pins: the per-rank ring schedule (primitive and chunk of each row)."""
import itertools

import numpy as np
import pytest

import oracle
from golden_io import rows

NAME = {v: k for k, v in oracle.PRIM_NAMES.items()}


def sched_for_rank(ring, r):
    index, prev, nextr, _ = oracle.ring_setup(ring)
    return oracle.schedule(len(ring), int(index[r])), prev[r], nextr[r]


def test_rank0_schedule_matches_page():
    ring = [0, 1, 2, 3]
    sched, prev, nextr = sched_for_rank(ring, 0)
    golden = rows("rank0_schedule.txt")
    assert len(sched) == len(golden) == 7
    for (prim, chunk), (seq, phase, pname, gchunk, rfrom, sto) in zip(sched, golden):
        assert prim == NAME[pname], seq
        assert chunk == int(gchunk), seq
        has_recv = prim != oracle.SEND
        has_send = prim != oracle.RECV
        assert (str(prev) if has_recv else "-") == rfrom
        assert (str(nextr) if has_send else "-") == sto


def test_first_send_table_matches_page():
    ring = [0, 1, 2, 3]
    for r, chunk, nxt in rows("first_send.txt"):
        sched, _, nextr = sched_for_rank(ring, int(r))
        assert sched[0] == (oracle.SEND, int(chunk))
        assert nextr == int(nxt)


def test_schedule_counts_match_page():
    g = {k: int(v) for k, v in rows("schedule_counts.txt")}
    n = g["nranks"]
    total = sends = 0
    for i in range(n):
        s = oracle.schedule(n, i)
        total += len(s)
        assert len(s) == g["rows_per_rank"]
        assert sum(p != oracle.RECV for p, _ in s) == g["sends_per_rank"]
        assert sum(p != oracle.SEND for p, _ in s) == g["receives_per_rank"]
        assert {c for _, c in s} == set(range(n))
    assert total == g["schedule_rows"]


@pytest.mark.parametrize("n", range(2, 9))
def test_schedule_brute_force(n):
    """Symbolic run of the schedule on every position of an n-ring.

    - the position form: position p handles chunk (p - s) mod n at step s,
      steps counted from 1;
    - every send of position p at row s is the receive of position p+1 at row
      s+1, for the same chunk;
    - in the reduce-scatter half each chunk's partial sum visits every position
      exactly once and ends at its owner (position c);
    - in the all-gather half every position writes every chunk exactly once;
    - 2(n-1) sends, 2(n-1) receives and 2n-1 rows per position."""
    S = [oracle.schedule(n, p) for p in range(n)]
    for p in range(n):
        assert len(S[p]) == 2 * n - 1
        for s1, (_, c) in enumerate(S[p], start=1):
            assert c == (p - s1) % n
        assert sum(pr != oracle.RECV for pr, _ in S[p]) == 2 * (n - 1)
        assert sum(pr != oracle.SEND for pr, _ in S[p]) == 2 * (n - 1)
    for p in range(n):
        q = (p + 1) % n
        for s in range(2 * n - 2):
            pr, c = S[p][s]
            if pr != oracle.RECV:
                pr2, c2 = S[q][s + 1]
                assert pr2 != oracle.SEND and c2 == c
    # reduce-scatter: follow each chunk's partial sum
    for c in range(n):
        contributors = []
        for s in range(n):
            holders = [p for p in range(n) if S[p][s][1] == c and S[p][s][0] in
                       (oracle.SEND, oracle.RECV_REDUCE_SEND, oracle.RECV_REDUCE_COPY_SEND)]
            assert len(holders) == 1
            contributors.append(holders[0])
        assert contributors == [(c + k) % n for k in range(1, n + 1)]
        assert S[c][n - 1] == (oracle.RECV_REDUCE_COPY_SEND, c)
    # all-gather: each position writes each chunk once
    for p in range(n):
        written = [c for pr, c in S[p] if pr in (oracle.RECV_REDUCE_COPY_SEND, oracle.RECV_COPY_SEND,
                                                 oracle.RECV)]
        assert sorted(written) == list(range(n))
