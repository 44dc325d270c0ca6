"""The store kernel computes a tile's scale RN(max(amax, 1e-4f) / 448)
without an IEEE division: Markstein's correction with the constant
c = RN(1/448) (P. Markstein, IBM J. Res. Dev. 34(1), 1990),

    q0 = RN(m c),  r = RN(m - 448 q0),  s = RN(q0 + r c)

with the last two steps one fma each.  m is either 1e-4f or a finite bf16
magnitude above it, 18,095 values in all, so the claim that s is the
correctly rounded quotient can be proved by trying every one of them with
exact rational arithmetic.  (A GPU test compares the kernel's own device
function with CUDA's __fdiv_rn on the same inputs.)
"""

import struct
from fractions import Fraction

from e4m3_ref import rn_f32


def _f32(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", bits))[0]


FLOOR = _f32(struct.unpack("<I", struct.pack("<f", 1e-4))[0])


def _domain():
    ms = [FLOOR]
    for b in range(0x7F80):                      # every finite non-negative bf16
        v = _f32(b << 16)
        if v >= FLOOR:
            ms.append(v)
    return ms


def _markstein_by_448(m: float, c: float) -> float:
    q0 = rn_f32(Fraction(m) * Fraction(c))
    r = rn_f32(Fraction(m) - 448 * Fraction(q0))         # one fma: exact, then rounded
    return rn_f32(Fraction(r) * Fraction(c) + Fraction(q0))


def test_domain_is_the_floor_and_every_bf16_above_it():
    ms = _domain()
    assert len(ms) == 18095
    assert min(ms) == FLOOR and max(ms) == _f32(0x7F7F << 16)


def test_markstein_scale_is_correctly_rounded_on_the_whole_domain():
    c = rn_f32(Fraction(1, 448))
    bad = [m for m in _domain() if _markstein_by_448(m, c) != rn_f32(Fraction(m) / 448)]
    assert bad == []


def test_the_correction_step_is_needed():
    # A plain product by RN(1/448) is wrong for many maxima, so the two fma
    # steps are what make the scale exact.
    c = rn_f32(Fraction(1, 448))
    wrong = sum(rn_f32(Fraction(m) * Fraction(c)) != rn_f32(Fraction(m) / 448)
                for m in _domain()[:2000])
    assert wrong > 100
