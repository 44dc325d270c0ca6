"""Pins for the oracle's per-row quantisation and the Main/Indexer row bytes.

Checked against things other than the oracle itself:
  * hand-derived bytes for three rows (tests/golden/hand_rows.json): exact
    scales, ties, saturation, subnormals, signed zero, NaN, Inf, the 1e-4
    floor and verbatim rope bytes;
  * exact rational arithmetic: every stored scale is RN32(max(amax, 1e-4f)
    / 448) and every code is the nearest E4M3 code of RN32(x / scale),
    computed with Python fractions and the brute-force nearest-code search;
  * invariants: the tile's largest element always codes to +-448, a tile is
    unaffected by its neighbours, and dequantised values stay within half an
    E4M3 spacing (plus the fp32 quotient's rounding) of the input.
The quantised rows are the "final FP8 Main-KV and Indexer-K bytes" of
"[Kernel][PCP] Publish replicated KV updates through PyTorch symmetric
memory", Design, third bullet.
"""

import struct
from fractions import Fraction

import numpy as np
import pytest
import torch

import hand_rows
import oracle
from e4m3_ref import DEC, nearest_code, rn_f32
from replication_token_warp_gb300 import inputs

F32_1EM4 = float(np.float32(1e-4))


def bits_f32(b: int) -> float:
    return struct.unpack("<f", struct.pack("<I", b))[0]


def f32_bits(x) -> int:
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


def bf16_value(bits: int) -> float:
    return bits_f32(int(bits) << 16)


def expected_scale(tile_bits: np.ndarray) -> float:
    """RN32(max(amax, fp32(1e-4)) / 448) for a finite tile, exactly."""
    amax = max(abs(bf16_value(b)) for b in tile_bits)
    m = amax if amax >= F32_1EM4 else F32_1EM4
    return rn_f32(Fraction(m) / 448)


@pytest.mark.parametrize("row", hand_rows.load()["rows"], ids=lambda r: r["name"])
def test_hand_rows(row):
    lat = hand_rows.build_bf16(row["latent"], 512)
    rope = hand_rows.build_bf16(row["rope"], 64)
    idx = hand_rows.build_bf16(row["index_k"], 128)
    ex = row["expect"]
    want_lat = hand_rows.build_codes(ex["latent_codes"], 512)
    want_idx = hand_rows.build_codes(ex["index_codes"], 128)
    want_scales = [int(b, 16) for b in ex["latent_scale_bits"]]
    want_iscale = int(ex["index_scale_bits"], 16)

    # the fixture's finite scales are themselves RN32(max(amax,1e-4)/448)
    for j in range(4):
        tile = lat[128 * j:128 * (j + 1)]
        vals = [bf16_value(b) for b in tile]
        if all(np.isfinite(vals)):
            assert f32_bits(expected_scale(tile)) == want_scales[j]
    if all(np.isfinite([bf16_value(b) for b in idx])):
        assert f32_bits(expected_scale(idx)) == want_iscale

    s = int(row["slot"])
    nb = 4
    main, ixc = oracle.new_caches(1, nb)
    n, inv = oracle.store_mla_fp8(lat[None], rope[None], idx[None], np.array([s]),
                                  main, ixc, nb)
    assert (n, inv) == (1, 0)
    m = main[0][s * 656:(s + 1) * 656]
    assert np.array_equal(m[:512], want_lat)
    got_scales = [int.from_bytes(m[512 + 4 * j:516 + 4 * j].tobytes(), "little") for j in range(4)]
    assert got_scales == want_scales
    assert m[528:656].tobytes() == rope.astype("<u2").tobytes()
    blk, off = divmod(s, 64)
    b = ixc[0][blk * 8448:(blk + 1) * 8448]
    assert np.array_equal(b[off * 128:(off + 1) * 128], want_idx)
    assert int.from_bytes(b[8192 + 4 * off:8196 + 4 * off].tobytes(), "little") == want_iscale
    # nothing else moved
    mask = np.ones(main[0].size, bool)
    mask[s * 656:(s + 1) * 656] = False
    assert np.all(main[0][mask] == 0xA5)
    mask = np.ones(ixc[0].size, bool)
    mask[blk * 8448 + off * 128: blk * 8448 + (off + 1) * 128] = False
    mask[blk * 8448 + 8192 + 4 * off: blk * 8448 + 8196 + 4 * off] = False
    assert np.all(ixc[0][mask] == 0xA5)


def _sample_tiles(n_tiles=48, seed=7):
    rng = np.random.default_rng(seed)
    w = inputs.make(4)                        # mixes N(0,1), zero and 6e4-sized rows
    lat = w.kv_latent.reshape(-1, 128)
    pick = rng.choice(lat.shape[0], n_tiles, replace=False)
    tiles = [lat[p] for p in pick]
    # plus tiles shaped to land near code boundaries and under the floor
    tiles.append(hand_rows.build_bf16({"fill": "0x1p-20", "set": {"0": "0x1p-15"}}, 128))
    tiles.append(hand_rows.build_bf16({"fill": "-0x1.8p-3", "set": {"7": "0x1.cp+1"}}, 128))
    return tiles


def test_scales_and_codes_are_exact_rational_results():
    for tile in _sample_tiles():
        q, scale = oracle.quantize_tile(tile)
        want_scale = expected_scale(tile)
        assert f32_bits(scale) == f32_bits(want_scale)
        fs = Fraction(float(scale))
        for x_bits, code in zip(tile.tolist(), q.tolist()):
            x = bf16_value(x_bits)
            quotient = rn_f32(Fraction(x) / fs)
            if quotient == 0.0 and (x < 0 or (x == 0 and np.signbit(x))):
                quotient = -0.0                # the quotient keeps the sign of x
            assert code == nearest_code(quotient), (x, float(scale), quotient, hex(code))


def test_largest_element_codes_to_448():
    w = inputs.make(2)
    for t in range(0, 2000, 37):
        for x_rows, tiles in ((w.kv_latent, 4), (w.index_k, 1)):
            for j in range(tiles):
                tile = x_rows[t, 128 * j:128 * (j + 1)]
                q, scale = oracle.quantize_tile(tile)
                mags = np.abs((tile.astype(np.uint32) << 16).view(np.float32))
                top = np.nonzero(mags == mags.max())[0]
                assert mags.max() >= F32_1EM4
                assert all((q[i] & 0x7F) == 0x7E for i in top)


def test_tiles_are_independent():
    w = inputs.make(1)
    row = w.kv_latent[5].copy()
    base = [oracle.quantize_tile(row[128 * j:128 * (j + 1)]) for j in range(4)]
    for j in range(4):
        pert = row.copy()
        pert[128 * j + 3] = hand_rows.bf16_bits_exact(1024.0)
        main, ixc = oracle.new_caches(1, 1)
        oracle.store_mla_fp8(pert[None], w.k_rope[5:6], w.index_k[5:6], np.array([0]),
                             main, ixc, 1)
        for k in range(4):
            codes = main[0][128 * k:128 * (k + 1)]
            if k == j:
                assert not np.array_equal(codes, base[k][0])
            else:
                assert np.array_equal(codes, base[k][0])
                got = int.from_bytes(main[0][512 + 4 * k:516 + 4 * k].tobytes(), "little")
                assert got == f32_bits(base[k][1])


def test_round_trip_error_bound():
    """|dec(q) * scale - x| <= (spacing(|x/scale|)/2 + 2^-24 |x/scale|) * scale."""
    w = inputs.make(2)
    for t in range(0, 16000, 997):
        for j in range(4):
            tile = w.kv_latent[t, 128 * j:128 * (j + 1)]
            q, scale = oracle.quantize_tile(tile)
            x = (tile.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
            y = np.abs(x) / float(scale)
            e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
            spacing = 2.0 ** (e - 3)
            deq = DEC[q] * float(scale)
            assert np.all(np.abs(DEC[q]) <= 448.0)
            err = np.abs(deq - x)
            bound = (spacing / 2 + 2.0 ** -24 * y) * float(scale) * (1 + 1e-12)
            assert np.all(err <= bound)


def _reciprocal_discriminating_pairs(limit=96):
    """(amax, x) bf16 pairs where multiplying by a rounded reciprocal of the
    scale gives a different E4M3 code from dividing by the scale (found by
    scanning; the expected codes below come from exact fractions)."""
    pos = (np.arange(0x0001, 0x7F80, dtype=np.uint32) << 16).view(np.float32)
    pairs = []
    for amax_bits in range(0x3800, 0x4400, 3):          # amax from 2^-15 to 2^9
        a = np.float32((np.uint32(amax_bits) << 16).view(np.float32))
        s = np.float32(max(a, np.float32(1e-4))) / np.float32(448)
        x = pos[pos <= a]
        with np.errstate(all="ignore"):
            q_div = x / s
            q_rcp = x * (np.float32(1) / s)
        differ = np.nonzero(q_div != q_rcp)[0]
        if differ.size == 0:
            continue
        c_div = torch.from_numpy(q_div[differ]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        c_rcp = torch.from_numpy(q_rcp[differ]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        for i in np.nonzero(c_div != c_rcp)[0]:
            pairs.append((amax_bits, int(pos.view(np.uint32)[pos <= a][differ[i]] >> 16)))
        if len(pairs) >= limit:
            break
    return pairs


def test_quotient_is_a_true_division():
    """Codes where x/scale and x*(1/scale) disagree must follow x/scale."""
    pairs = _reciprocal_discriminating_pairs()
    assert len(pairs) >= 8, "scan found too few discriminating pairs"
    for amax_bits, x_bits in pairs:
        tile = np.zeros(128, np.uint16)
        tile[0] = amax_bits
        tile[1] = x_bits
        tile[2] = x_bits | 0x8000
        q, scale = oracle.quantize_tile(tile)
        fs = Fraction(float(scale))
        for k in (1, 2):
            x = bf16_value(tile[k])
            assert q[k] == nearest_code(rn_f32(Fraction(x) / fs)), (hex(amax_bits), hex(x_bits))
