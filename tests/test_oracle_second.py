"""A second, independent statement of the store for small workloads, in
numpy: IEEE float32 division (numpy), the nearest-code search of e4m3_ref as
the encoder, and numpy indexing for the slot layout.  It shares nothing with
oracle/kvpub_oracle.c except the reading of the format, and must leave the
same bytes in every replica's whole buffer (tiny and decode workloads, the
hand rows).  Format: "[Kernel][PCP] Publish replicated KV updates through
PyTorch symmetric memory", Design, third bullet (final FP8 Main-KV and
Indexer-K bytes).
"""

import numpy as np
import pytest

import hand_rows
import oracle
from e4m3_ref import nearest_codes
from replication_token_warp_gb300 import inputs

F32 = np.float32


def quantize_tiles(x_bits: np.ndarray):
    """[n, 128] bf16 bit patterns -> (codes [n, 128] uint8, scales [n] float32)."""
    x = (x_bits.astype(np.uint32) << 16).view(np.float32)
    with np.errstate(invalid="ignore"):
        amax = np.max(np.abs(x), axis=1)                 # NaN propagates
    scale = np.maximum(amax, F32(1e-4)) / F32(448.0)      # np.maximum propagates NaN
    scale = scale.astype(np.float32)
    nan = np.isnan(scale)
    scale[nan] = np.uint32(0x7FFFFFFF).view(np.float32)
    with np.errstate(all="ignore"):
        q = (x / scale[:, None]).astype(np.float32)
        codes = nearest_codes(q.astype(np.float64).ravel()).reshape(q.shape)
    return codes, scale


def py_store(w):
    cap = w.num_blocks * 64
    main = [np.full(cap * 656, w.guard, np.uint8) for _ in range(w.num_replicas)]
    idx = [np.full(w.num_blocks * 8448, w.guard, np.uint8) for _ in range(w.num_replicas)]
    ok = (w.slot_mapping >= 0) & (w.slot_mapping < cap)
    t = np.nonzero(ok)[0]
    s = w.slot_mapping[t]
    lc, ls = quantize_tiles(w.kv_latent[t].reshape(-1, 128))
    ic, isc = quantize_tiles(w.index_k[t])
    rows = np.concatenate([
        lc.reshape(len(t), 512),
        ls.reshape(len(t), 4).astype("<f4").view(np.uint8).reshape(len(t), 16),
        w.k_rope[t].astype("<u2").view(np.uint8).reshape(len(t), 128)], axis=1)
    blk, off = s // 64, s % 64
    for r in range(w.num_replicas):
        m = main[r].reshape(cap, 656)
        m[s] = rows
        b = idx[r].reshape(w.num_blocks, 8448)
        for k in range(len(t)):
            b[blk[k], off[k] * 128:(off[k] + 1) * 128] = ic[k]
            b[blk[k], 8192 + 4 * off[k]:8196 + 4 * off[k]] = isc[k:k + 1].astype("<f4").view(np.uint8)
    return main, idx


def _hand_workload():
    rows = hand_rows.load()["rows"]
    return inputs.Workload(
        "hand", np.stack([hand_rows.build_bf16(r["latent"], 512) for r in rows]),
        np.stack([hand_rows.build_bf16(r["rope"], 64) for r in rows]),
        np.stack([hand_rows.build_bf16(r["index_k"], 128) for r in rows]),
        np.array([r["slot"] for r in rows], np.int64), 2, 4)


@pytest.mark.parametrize("make", [lambda: inputs.make(0), lambda: inputs.make(1), _hand_workload],
                         ids=["tiny", "decode", "hand_rows"])
def test_second_statement_equals_the_oracle(make):
    w = make()
    want_main, want_idx = py_store(w)
    main, idx = oracle.new_caches(w.num_replicas, w.num_blocks, w.guard)
    oracle.store_mla_fp8(w.kv_latent, w.k_rope, w.index_k, w.slot_mapping, main, idx,
                         w.num_blocks)
    for a, b in zip(main + idx, want_main + want_idx):
        assert np.array_equal(a, b)
