"""Exact-arithmetic helpers for the oracle pins (test side, independent of oracle/).

``rne_bf16`` rounds an exact rational to bf16 straight from the textbook
definition of round-to-nearest, ties-to-even: scale by the quantum of the
value's binade (2^(e-7) for a normal bf16 with 8 significant bits, 2^-133
below 2^-126), round the quotient half-to-even (Python's ``round`` on a
Fraction does exactly that), and saturate to infinity past the largest finite
bf16, (2 - 2^-7) * 2^127.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction

import numpy as np

BF16_MAX = Fraction(2 ** 8 - 1, 2 ** 7) * Fraction(2) ** 127


def _bits_of_exact_bf16(v: Fraction) -> int:
    """bf16 bit pattern of a rational that is exactly a bf16 value."""
    f32 = struct.unpack("<I", struct.pack("<f", float(v)))[0]  # exact: v is a bf16
    assert (f32 & 0xFFFF) == 0
    return f32 >> 16


def rne_bf16(v) -> int:
    """bf16 bits of round-to-nearest-even(v) for an exact rational (or float) v."""
    v = Fraction(v)
    if v == 0:
        return 0
    sign = 0x8000 if v < 0 else 0
    a = -v if v < 0 else v
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # fix up floating log2 error: make 2^e <= a < 2^(e+1)
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    quantum = Fraction(2) ** (e - 7) if e >= -126 else Fraction(2) ** -133
    r = round(a / quantum) * quantum
    if r > BF16_MAX:
        return sign | 0x7F80
    return sign | _bits_of_exact_bf16(r)


def bf16_value(bits: int) -> Fraction:
    """Exact rational value of a finite bf16 bit pattern."""
    f = struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]
    return Fraction(f)


def bf16_ulp_distance(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """Distance in bf16 steps between two arrays of finite bf16 bit patterns
    (ordered-integer mapping of sign-magnitude codes)."""
    def ordered(x):
        x = np.asarray(x, dtype=np.int64)
        mag = x & 0x7FFF
        return np.where(x & 0x8000, -mag, mag)
    return np.abs(ordered(a_bits) - ordered(b_bits))
