"""Reader for tests/golden/hand_rows.json (hand-derived single-row bytes).

The fixture's mini-language: ``fill`` sets every element; ``set`` maps keys
to values in order, where a key is an index ``"k"``, a range ``"a..b"``
(inclusive), a range restricted to ``:even`` / ``:odd`` indices, or
``"a..b:iota1"`` with value ``"iota"`` (element k takes the value k + 1).
Values are hex floats (exact in bf16), ``"bits:0xHHHH"`` bf16 bit patterns,
or, for expected codes, hex bytes.
"""

import json
import os
import struct

import numpy as np

PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "hand_rows.json")


def load():
    with open(PATH) as f:
        return json.load(f)


def _f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]


def bf16_bits_exact(x: float) -> int:
    """bf16 bits of x; x must be exactly representable in bf16."""
    b = _f32_bits(x)
    if b & 0xFFFF:
        raise ValueError(f"{x!r} is not exact in bf16")
    if struct.unpack("<f", struct.pack("<I", b))[0] != x:
        raise ValueError(f"{x!r} is not exact in fp32")
    return b >> 16


def _indices(key: str, n: int):
    rng, _, sel = key.partition(":")
    if ".." in rng:
        a, b = (int(v) for v in rng.split(".."))
        idx = list(range(a, b + 1))
    else:
        idx = [int(rng)]
    if sel == "even":
        idx = [i for i in idx if i % 2 == 0]
    elif sel == "odd":
        idx = [i for i in idx if i % 2 == 1]
    assert all(0 <= i < n for i in idx), key
    return idx, sel


def _value_bits(v: str) -> int:
    if v.startswith("bits:"):
        return int(v[5:], 16)
    return bf16_bits_exact(float.fromhex(v))


def build_bf16(spec: dict, n: int) -> np.ndarray:
    out = np.full(n, _value_bits(spec["fill"]), dtype=np.uint16)
    for key, v in spec["set"].items():
        idx, sel = _indices(key, n)
        for i in idx:
            out[i] = bf16_bits_exact(float(i + 1)) if sel == "iota1" else _value_bits(v)
    return out


def build_codes(spec: dict, n: int) -> np.ndarray:
    out = np.full(n, int(spec["fill"], 16), dtype=np.uint8)
    for key, v in spec["set"].items():
        idx, _ = _indices(key, n)
        for i in idx:
            out[i] = int(v, 16)
    return out
