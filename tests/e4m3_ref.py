"""Brute-force E4M3 references written from the format definition.

E4M3 ("fn") as defined by the OCP 8-bit floating point specification: bias
7, exponent field 0 holds subnormals m * 2^-9, the code with exponent field
15 and mantissa 7 is NaN, there are no infinities, the largest finite
magnitude is 448.  Also: exact round-to-nearest-even of a rational to fp32.
"""

from fractions import Fraction

import numpy as np


def decode_table_from_definition() -> np.ndarray:
    """E4M3 (fn): bias 7; exponent field 0 is subnormal m * 2^-9; the code
    with exponent field 15 and mantissa 7 is NaN; there is no infinity."""
    out = np.empty(256, dtype=np.float64)
    for c in range(256):
        s, e, m = c >> 7, (c >> 3) & 15, c & 7
        if e == 15 and m == 7:
            out[c] = np.nan
            continue
        mag = m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
        out[c] = -mag if s else mag
    return out


DEC = decode_table_from_definition()

# Every magnitude above 448 has 448 as its unique nearest finite value, so
# magnitudes are clipped to 1024 before distances are taken: that keeps the
# distances exact in double (|v| - 448 and |v| - 416 are indistinguishable in
# double once |v| is ~1e18) without changing the nearest code.
CLIP = 1024.0


def nearest_code(v: float) -> int:
    """Brute-force reference: nearest finite code of the same sign, ties to
    the even code; NaN -> 0x7F."""
    if np.isnan(v):
        return 0x7F
    sign = 0x80 if np.signbit(v) else 0x00
    a = min(abs(float(v)), CLIP)
    best, best_d = None, None
    for m in range(127):                     # 0x00..0x7E are the finite magnitudes
        d = abs(a - DEC[m])
        if best is None or d < best_d or (d == best_d and (m & 1) == 0 and (best & 1) == 1):
            best, best_d = m, d
    return sign | best


def nearest_codes(v: np.ndarray) -> np.ndarray:
    """Vectorised form of nearest_code for float arrays."""
    v = np.asarray(v, dtype=np.float64)
    mags = DEC[:127]
    a = np.minimum(np.abs(v), CLIP)
    a[np.isnan(a)] = 0.0                 # NaN inputs are coded below
    d = np.abs(a[:, None] - mags[None, :])
    dmin = d.min(axis=1, keepdims=True)
    cand = d == dmin
    # among the (at most two) nearest, take the even code
    even = cand & ((np.arange(127) & 1) == 0)[None, :]
    pick = np.where(even.any(axis=1), even.argmax(axis=1), cand.argmax(axis=1))
    code = pick.astype(np.uint8) | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    code[np.isnan(v)] = 0x7F
    return code


def rn_f32(q: Fraction) -> float:
    """Round the rational q to the nearest fp32 value, ties to even (exact,
    no intermediate double rounding).  Overflow is not handled (not needed)."""
    if q == 0:
        return 0.0
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                     # fp32 subnormals share 2^-149 spacing
    ulp = Fraction(2) ** (e - 23)
    n = round(a / ulp)                   # Fraction.__round__: ties to even
    return sign * float(n * ulp)
