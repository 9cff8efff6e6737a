"""Oracle pin: the 27-row credit/flag state model against the page's outcome table."""
import pytest

import oracle
from golden_io import rows

PROTO = {"Simple": oracle.SIMPLE, "LL": oracle.LL, "LL128": oracle.LL128}
FAULTS = {
    "Simple": ["normal", "drop_recv_head", "tail_before_payload"],
    "LL": ["normal", "second_flag_missing", "constant_flag"],
    "LL128": ["normal", "flag_word_missing", "flag_before_data"],
}


@pytest.mark.parametrize("slots", [2, 4, 8])
def test_state_model_table(slots):
    golden = rows("state_model.txt")
    assert len(golden) == 9
    for proto, fault, _wording, outcome, stall_after in golden:
        res = oracle.state_model(PROTO[proto], FAULTS[proto].index(fault), slots, 64)
        if outcome == "complete":
            assert res["outcome"] == oracle.M_COMPLETE, (proto, fault)
        elif outcome == "stall":
            assert res["outcome"] == oracle.M_STALL, (proto, fault)
            if stall_after == "slots":
                # the sender fills exactly the FIFO, then nothing moves
                assert res["stall_producer"] == slots and res["stall_consumer"] == slots
            else:
                assert res["stall_consumer"] == int(stall_after)
                assert res["stall_producer"] == slots
        elif outcome == "corrupt_stale":
            assert res["outcome"] == oracle.M_CORRUPT and res["corrupt_kinds"] == 1, (proto, fault)
        else:
            assert res["outcome"] == oracle.M_CORRUPT, (proto, fault)


def test_state_model_row_count():
    n = 0
    for slots in (2, 4, 8):
        for proto, faults in FAULTS.items():
            for f in range(len(faults)):
                oracle.state_model(PROTO[proto], f, slots, 64)
                n += 1
    assert n == 27
