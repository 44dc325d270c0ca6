"""Pins for the oracle's slot handling, byte placement and the gather path.

"[Kernel][PCP] Publish replicated KV updates through PyTorch symmetric
memory", Correctness and current-head validation: padded and invalid slots
and guard bytes are covered, and the direct path is byte-exact against
gather-then-insert.  Checked here on the host, by invariants:
  * exactly 656 + 128 + 4 bytes per written row and replica change, at the
    offsets of the slot layout, and nothing else (two runs with different
    guard bytes expose every written byte, even one equal to a guard);
  * padded (-1) and out-of-range slots write nothing and only the latter
    count as invalid;
  * every replica holds the same bytes;
  * strided input rows give the same bytes as contiguous rows;
  * the gather-then-insert path leaves the same bytes as direct publication.
"""

import numpy as np
import pytest

import oracle
from replication_token_warp_gb300 import inputs


def written_mask(w, guard):
    main, ixc = oracle.new_caches(w.num_replicas, w.num_blocks, guard)
    n, inv = oracle.store_mla_fp8(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping,
                                  main, ixc, w.num_blocks)
    return main, ixc, n, inv


def expected_extents(slots, num_blocks):
    cap = num_blocks * 64
    m = np.zeros(cap * 656, bool)
    ix = np.zeros(num_blocks * 8448, bool)
    for s in slots:
        s = int(s)
        if 0 <= s < cap:
            m[s * 656:(s + 1) * 656] = True
            blk, off = divmod(s, 64)
            ix[blk * 8448 + off * 128: blk * 8448 + (off + 1) * 128] = True
            ix[blk * 8448 + 8192 + 4 * off: blk * 8448 + 8196 + 4 * off] = True
    return m, ix


@pytest.mark.parametrize("index", [0, 1, 2])
def test_written_bytes_are_exactly_the_slot_rows(index):
    w = inputs.make(index)
    a_main, a_ix, n, inv = written_mask(w, 0xA5)
    b_main, b_ix, _, _ = written_mask(w, 0x5A)
    assert n == w.num_valid and inv == 0
    em, ei = expected_extents(w.slot_mapping, w.num_blocks)
    for r in range(w.num_replicas):
        changed_m = (a_main[r] != 0xA5) | (b_main[r] != 0x5A)
        changed_i = (a_ix[r] != 0xA5) | (b_ix[r] != 0x5A)
        assert np.array_equal(changed_m, em)
        assert np.array_equal(changed_i, ei)
        assert changed_m.sum() + changed_i.sum() == 788 * w.num_valid
        # written bytes do not depend on the guard
        assert np.array_equal(a_main[r][em], b_main[r][em])
        assert np.array_equal(a_ix[r][ei], b_ix[r][ei])
        assert np.array_equal(a_main[r], a_main[0]) and np.array_equal(a_ix[r], a_ix[0])


def test_padding_and_invalid_slots():
    w = inputs.make(0)
    cap = w.num_blocks * 64
    slots = w.slot_mapping.copy()
    bad = {1: cap, 4: -5, 9: cap + 1000, 12: 2 ** 40, 13: -(2 ** 62)}
    valid_before = [i for i in range(16) if slots[i] >= 0]
    for i, v in bad.items():
        slots[i] = v
    w.slot_mapping = slots
    main, ixc, n, inv = written_mask(w, 0xA5)
    assert inv == len(bad)
    expect_n = len([i for i in valid_before if i not in bad])
    assert n == expect_n
    em, ei = expected_extents(slots, w.num_blocks)
    assert np.all(main[0][~em] == 0xA5)
    assert np.all(ixc[0][~ei] == 0xA5)


def test_empty_batch_writes_nothing():
    w = inputs.make(0)
    main, ixc = oracle.new_caches(2, w.num_blocks)
    n, inv = oracle.store_mla_fp8(w.kv_latent[:0], w.k_rope[:0], w.index_k[:0],
                                  np.zeros(0, np.int64), main, ixc, w.num_blocks)
    assert (n, inv) == (0, 0)
    assert all(np.all(c == 0xA5) for c in main + ixc)


def test_all_padded_writes_nothing():
    w = inputs.make(1)
    main, ixc = oracle.new_caches(2, w.num_blocks)
    n, inv = oracle.store_mla_fp8(w.kv_latent, w.k_rope, w.index_k,
                                  np.full(w.num_tokens, -1, np.int64), main, ixc, w.num_blocks)
    assert (n, inv) == (0, 0)
    assert all(np.all(c == 0xA5) for c in main + ixc)


def test_strided_rows_match_contiguous_rows():
    w = inputs.make(1)
    T = w.num_tokens
    # latent and rope as views of one [T, 576] buffer; Indexer-K padded to 136
    kv = np.zeros((T, 576), np.uint16)
    kv[:, :512], kv[:, 512:] = w.kv_latent, w.k_rope
    ik = np.zeros((T, 136), np.uint16)
    ik[:, :128] = w.index_k
    a = oracle.new_caches(2, w.num_blocks)
    b = oracle.new_caches(2, w.num_blocks)
    oracle.store_mla_fp8(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping, *a, w.num_blocks)
    oracle.store_mla_fp8(kv[:, :512], kv[:, 512:], ik[:, :128], w.slot_mapping, *b,
                         w.num_blocks)
    for x, y in zip(a[0] + a[1], b[0] + b[1]):
        assert np.array_equal(x, y)


@pytest.mark.parametrize("index", [0, 1, 2])
def test_gather_insert_equals_direct_publication(index):
    w = inputs.make(index)
    a = oracle.new_caches(w.num_replicas, w.num_blocks)
    b = oracle.new_caches(w.num_replicas, w.num_blocks)
    ra = oracle.store_mla_fp8(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping, *a,
                              w.num_blocks)
    rb = oracle.gather_insert(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping, *b,
                              w.num_blocks)
    assert ra == rb
    for x, y in zip(a[0] + a[1], b[0] + b[1]):
        assert np.array_equal(x, y)


def test_rope_bytes_verbatim_and_scales_positive():
    w = inputs.make(2)
    main, ixc, n, _ = written_mask(w, 0xA5)
    for t in range(0, w.num_tokens, 251):
        s = int(w.slot_mapping[t])
        if s < 0:
            continue
        row = main[0][s * 656:(s + 1) * 656]
        assert row[528:].tobytes() == w.k_rope[t].astype("<u2").tobytes()
        scales = row[512:528].view("<f4")
        assert np.all(scales > 0) and np.all(np.isfinite(scales))
        blk, off = divmod(s, 64)
        iscale = ixc[0][blk * 8448 + 8192 + 4 * off: blk * 8448 + 8196 + 4 * off].view("<f4")
        assert iscale[0] > 0
