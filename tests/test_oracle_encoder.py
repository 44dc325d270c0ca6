"""Pins for the oracle's fp32 -> E4M3 encoder and its decode.

The encoder is checked against things other than itself:
  * the E4M3 ("fn") format definition of the OCP 8-bit floating point
    specification: the decode table is written here from that definition
    and compared with PyTorch's float8_e4m3fn decode (a library routine);
  * brute force: for every one of the 65,536 bf16 bit patterns (and for
    fp32 values on and next to every rounding midpoint) the oracle's code
    must be the nearest finite code of the same sign, ties to the even code;
  * PyTorch's fp32 -> float8_e4m3fn cast, which rounds to nearest even and
    agrees with a saturating conversion up to |v| <= 464;
  * hand-picked special values (zero, signed zero, ties, saturation, Inf,
    NaN).
The fp8 KV format itself is named on "[Kernel][PCP] Publish replicated KV
updates through PyTorch symmetric memory", Design, third bullet (final FP8
Main-KV and Indexer-K bytes).
"""

import numpy as np
import pytest
import torch

import oracle
from e4m3_ref import DEC, nearest_code, nearest_codes


def test_decode_table_matches_library():
    lib = torch.arange(256, dtype=torch.int32).to(torch.uint8).view(torch.float8_e4m3fn)
    lib = lib.to(torch.float32).double().numpy()
    both_nan = np.isnan(lib) & np.isnan(DEC)
    assert np.array_equal(np.isnan(lib), np.isnan(DEC))
    assert np.all((lib == DEC) | both_nan)
    # landmarks of the format
    assert DEC[0x7E] == 448.0 and DEC[0x01] == 2.0 ** -9 and DEC[0x08] == 2.0 ** -6
    assert DEC[0x38] == 1.0 and DEC[0xFE] == -448.0 and np.isnan(DEC[0x7F])


def test_oracle_decode_matches_definition():
    got = np.array([oracle.e4m3_decode(c) for c in range(256)])
    assert np.array_equal(np.isnan(got), np.isnan(DEC))
    ok = np.isnan(DEC) | (got == DEC)
    assert ok.all()


def _all_bf16_as_f32() -> np.ndarray:
    bits = np.arange(65536, dtype=np.uint32) << 16
    return bits.view(np.float32)


def test_encode_all_bf16_patterns_brute_force():
    v = _all_bf16_as_f32()
    got = oracle.e4m3_encode_array(v)
    with np.errstate(invalid="ignore"):      # signalling-NaN patterns widen quietly
        want = nearest_codes(v.astype(np.float64))
    bad = np.nonzero(got != want)[0]
    assert bad.size == 0, [(hex(int(b)), float(v[b]), hex(got[b]), hex(want[b])) for b in bad[:10]]


def _midpoints() -> np.ndarray:
    mags = DEC[:127]
    return (mags[:-1] + mags[1:]) / 2.0


def test_encode_around_every_midpoint():
    """fp32 values on each rounding midpoint and 1..3 fp32 ulps either side."""
    mids = _midpoints().astype(np.float32)   # exact: midpoints have <= 5 bits
    assert np.array_equal(mids.astype(np.float64), _midpoints())
    vals = [mids]
    for k in (1, 2, 3):
        up, dn = mids.copy(), mids.copy()
        for _ in range(k):
            up = np.nextafter(up, np.float32(np.inf))
            dn = np.nextafter(dn, np.float32(0))
        vals += [up, dn]
    vals.append(np.float32([448.0, np.nextafter(np.float32(448), np.float32(0)),
                            464.0, np.nextafter(np.float32(464), np.float32(0)),
                            np.nextafter(np.float32(464), np.float32(1e9)), 1e30]))
    v = np.concatenate(vals)
    v = np.concatenate([v, -v])
    got = oracle.e4m3_encode_array(v)
    want = nearest_codes(v.astype(np.float64))
    assert np.array_equal(got, want)


def test_encode_matches_library_cast_in_range():
    rng = np.random.default_rng(12345)
    mag = np.exp2(rng.uniform(-14.0, np.log2(464.0), size=200_000)).astype(np.float32)
    v = mag * np.where(rng.random(mag.shape) < 0.5, -1, 1).astype(np.float32)
    v = np.concatenate([v, _all_bf16_as_f32()])
    v = v[np.isfinite(v) & (np.abs(v) <= 464.0)]
    lib = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode_array(v)
    assert np.array_equal(got, lib)


@pytest.mark.parametrize("v,code", [
    (0.0, 0x00), (-0.0, 0x80), (448.0, 0x7E), (-448.0, 0xFE), (464.0, 0x7E),
    (480.0, 0x7E), (1e30, 0x7E), (float("inf"), 0x7E), (float("-inf"), 0xFE),
    (2.0 ** -9, 0x01), (2.0 ** -10, 0x00), (3 * 2.0 ** -10, 0x02),
    (2.0 ** -6, 0x08), (-(2.0 ** -11), 0x80), (1.0, 0x38), (1.0625, 0x38),
    (1.1875, 0x3A), (240.0, 0x77), (float("nan"), 0x7F),
])
def test_encode_special_values(v, code):
    assert oracle.e4m3_encode(v) == code
    if not np.isnan(v):
        assert nearest_code(v) == code


def test_no_nan_code_for_finite_inputs():
    v = _all_bf16_as_f32()
    v = v[np.isfinite(v)]
    got = oracle.e4m3_encode_array(v)
    assert not np.any((got & 0x7F) == 0x7F)
