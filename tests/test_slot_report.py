"""The binding's host-side debug check of a slot_mapping (counts of written,
padded, invalid and duplicated slots) and its opt-in use before a store.
Runs on the CPU: the check never reaches the library when it fails."""

import numpy as np
import pytest
import torch

from replication_token_warp_gb300 import kvpub


def test_counts():
    s = torch.tensor([5, -1, 7, 5, 300, -9, 255, 7, 7, -1], dtype=torch.int64)
    rep = kvpub.slot_report(s, num_blocks=4)                # 256 slots
    assert rep == {"written": 6, "padded": 2, "invalid": 2, "duplicates": 3}


def test_distinct_workload_slots_report_no_duplicates():
    from replication_token_warp_gb300 import inputs
    for i in range(5):
        w = inputs.make(i)
        rep = kvpub.slot_report(w.slot_mapping, w.num_blocks)
        assert rep["duplicates"] == 0 and rep["invalid"] == 0
        assert rep["written"] == w.num_valid


def test_opt_in_check_refuses_duplicates_before_any_launch():
    slots = torch.tensor([1, 2, 1], dtype=torch.int64)
    cache = torch.zeros(64 * 656, dtype=torch.uint8)
    with pytest.raises(ValueError, match="more than once"):
        kvpub.store_mla_fp8(None, None, None, slots, [cache], [cache], num_blocks=1,
                            check_slots=True)
