"""Oracle pins: ring setup (index / prev / next / rotated user ranks) and ring validation."""
import itertools

import numpy as np
import pytest

import oracle
from golden_io import rows


def test_ring_index_tables_match_page():
    for ring_s, r, idx, prv, nxt in rows("ring_index_tables.txt"):
        ring = [int(v) for v in ring_s.split("-")]
        index, prev, nextr, _ = oracle.ring_setup(ring)
        r = int(r)
        assert (index[r], prev[r], nextr[r]) == (int(idx), int(prv), int(nxt)), (ring_s, r)


def test_user_ranks_rotation():
    # userRanks of rank r lists the ring starting from r itself.
    for n in range(2, 7):
        for ring in itertools.islice(itertools.permutations(range(n)), 30):
            _, prev, nextr, ur = oracle.ring_setup(list(ring))
            for r in range(n):
                assert ur[r][0] == r
                assert ur[r][1] == nextr[r]
                assert ur[r][-1] == prev[r]
                assert sorted(ur[r].tolist()) == list(range(n))


def test_ring_index_is_distance_from_rank0_brute_force():
    # Walk `next` from rank 0: the k-th rank reached has ring index k.
    rng = np.random.default_rng(11)
    for n in range(2, 12):
        ring = rng.permutation(n).tolist()
        index, prev, nextr, _ = oracle.ring_setup(ring)
        cur = 0
        for k in range(n):
            assert index[cur] == k
            assert prev[nextr[cur]] == cur
            cur = nextr[cur]
        assert cur == 0


@pytest.mark.parametrize("ring", [[0, 1, 1, 2], [0, 1, 4, 2], [1, 2, 3, 5], [0, -1, 2, 3]])
def test_rejects_non_rings(ring):
    assert oracle.ring_setup_status(ring) == oracle.ERING
