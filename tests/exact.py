"""Exact-rational helpers for pinning the oracle (independent of NumPy's float arithmetic)."""
from __future__ import annotations

import math
import struct
from fractions import Fraction


def f32_bits(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def half_value(bits: int) -> Fraction:
    """Exact value of an fp16 bit pattern (finite only), decoded from the IEEE 754 binary16 fields."""
    s = -1 if bits & 0x8000 else 1
    e = (bits >> 10) & 0x1F
    f = bits & 0x3FF
    assert e != 0x1F
    if e == 0:
        return s * Fraction(f, 1 << 24)
    return s * Fraction(1024 + f, 1 << 10) * (Fraction(2) ** (e - 15))


def round_to_f32(x: Fraction) -> float:
    """Correctly rounded (nearest, ties to even) binary32 value of an exact rational, as a Python float."""
    if x == 0:
        return 0.0
    sign = -1.0 if x < 0 else 1.0
    a = abs(x)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)                      # subnormals share the exponent of the smallest normal
    unit = Fraction(2) ** (e - 23)        # spacing of binary32 values at this exponent
    t = a / unit
    n = t.numerator // t.denominator
    rem = t - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = Fraction(n) * unit
    assert v < Fraction(2) ** 128, "binary32 overflow"
    return sign * float(v)


def all_finite_halves():
    """Every finite fp16 bit pattern."""
    return [b for b in range(0x10000) if ((b >> 10) & 0x1F) != 0x1F]
