"""Pins for the oracle's unquantised (bf16) cache variant.

The variant stores each row's bf16 values as they arrive: Main slot s holds
latent[512] | rope[64] at byte s * 1152 and Indexer slot s holds index_k[128]
at byte s * 256, in every replica (the BF16 main/indexer cache cases of
"[Feature][KV Connector] Support QSA HiSparse in disaggregated serving",
Validation).  Checked here by independent numpy indexing and invariants:
the written bytes equal the inputs' little-endian bytes at those offsets,
exactly 1408 bytes per written row and replica change (two guard values),
and padded / invalid slots write nothing.
"""

import numpy as np
import pytest

import oracle
from replication_token_warp_gb300 import inputs


def run(w, guard):
    main, idx = oracle.new_caches_bf16(w.num_replicas, w.num_blocks, guard)
    n, inv = oracle.store_mla_bf16(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping, main, idx,
                                   w.num_blocks)
    return main, idx, n, inv


@pytest.mark.parametrize("index", [0, 1, 2])
def test_bytes_and_extents(index):
    w = inputs.make(index)
    a_main, a_idx, n, inv = run(w, 0xA5)
    b_main, b_idx, _, _ = run(w, 0x5A)
    assert n == w.num_valid and inv == 0
    cap = w.num_blocks * 64
    em = np.zeros(cap * 1152, bool)
    ei = np.zeros(cap * 256, bool)
    for t, s in enumerate(w.slot_mapping.tolist()):
        if 0 <= s < cap:
            em[s * 1152:(s + 1) * 1152] = True
            ei[s * 256:(s + 1) * 256] = True
            want_m = np.concatenate([w.kv_latent[t], w.k_rope[t]]).astype("<u2").tobytes()
            want_i = w.index_k[t].astype("<u2").tobytes()
            for r in range(w.num_replicas):
                assert a_main[r][s * 1152:(s + 1) * 1152].tobytes() == want_m
                assert a_idx[r][s * 256:(s + 1) * 256].tobytes() == want_i
    for r in range(w.num_replicas):
        changed_m = (a_main[r] != 0xA5) | (b_main[r] != 0x5A)
        changed_i = (a_idx[r] != 0xA5) | (b_idx[r] != 0x5A)
        assert np.array_equal(changed_m, em) and np.array_equal(changed_i, ei)
        assert changed_m.sum() + changed_i.sum() == 1408 * w.num_valid


def test_padding_and_invalid_slots():
    w = inputs.make(0)
    cap = w.num_blocks * 64
    w.slot_mapping = w.slot_mapping.copy()
    w.slot_mapping[[1, 4, 9]] = [cap, -7, cap + 99]
    main, idx, n, inv = run(w, 0xA5)
    assert inv == 3
    valid = [s for s in w.slot_mapping.tolist() if 0 <= s < cap]
    assert n == len(valid)
    mask = np.ones(cap * 1152, bool)
    for s in valid:
        mask[s * 1152:(s + 1) * 1152] = False
    assert np.all(main[0][mask] == 0xA5)
