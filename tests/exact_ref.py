"""Exact (rational) arithmetic used by the oracle pins.

Independent of the oracle's C code: binary floating-point values are turned
into ``fractions.Fraction`` and rounded back with Python integers, so a pin
that compares the oracle against these helpers checks it against the
mathematics, not against itself.
"""
from __future__ import annotations

import math
import struct
from fractions import Fraction


def bf16_value(bits: int) -> Fraction | float:
    """Exact value of a BF16 bit pattern (float('nan') / +-inf for specials)."""
    bits &= 0xFFFF
    sign = -1 if bits & 0x8000 else 1
    E = (bits >> 7) & 0xFF
    M = bits & 0x7F
    if E == 0xFF:
        return float("nan") if M else sign * math.inf
    if E == 0:
        return sign * Fraction(M, 2**133)
    return sign * Fraction(128 + M) * (Fraction(2) ** (E - 134))


def f32_value(x: float) -> Fraction:
    return Fraction(struct.unpack("<f", struct.pack("<f", x))[0])


def _round_half_even(q: Fraction) -> int:
    fl = math.floor(q)
    rem = q - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        return fl + 1
    return fl


def rne_bf16(q: Fraction, negative_zero: bool = False) -> int:
    """Round an exact rational to the nearest BF16 (ties to even)."""
    if q == 0:
        return 0x8000 if negative_zero else 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    assert Fraction(2) ** e <= a < Fraction(2) ** (e + 1)
    E = e + 127
    quantum_exp = (e - 7) if E >= 1 else -133
    k = _round_half_even(a / Fraction(2) ** quantum_exp)
    if k == 0:
        return sign
    # re-normalise (rounding may carry into the next binade)
    val_exp = quantum_exp
    while k >= 256:
        assert k % 2 == 0
        k //= 2
        val_exp += 1
    if k < 128:  # subnormal
        assert val_exp == -133
        return sign | k
    E = val_exp + 7 + 127
    if E >= 255:
        return sign | 0x7F80
    return sign | (E << 7) | (k - 128)


def rne_f32(q: Fraction) -> float:
    """Round an exact rational to the nearest binary32 (ties to even), normal range."""
    if q == 0:
        return 0.0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    qexp = max(e - 23, -149)
    k = _round_half_even(a / Fraction(2) ** qexp)
    v = math.ldexp(k, qexp)
    return -v if q < 0 else v


def murmur3_x86_32(data: bytes, seed: int = 0) -> int:
    """MurmurHash3_x86_32 over a byte string (Austin Appleby's published
    algorithm, public domain), with the tail bytes and the length mix."""
    c1, c2 = 0xCC9E2D51, 0x1B873593
    h = seed & 0xFFFFFFFF
    n = len(data)
    nblocks = n // 4
    rotl = lambda x, r: ((x << r) | (x >> (32 - r))) & 0xFFFFFFFF
    for i in range(nblocks):
        k = int.from_bytes(data[4 * i:4 * i + 4], "little")
        k = (k * c1) & 0xFFFFFFFF
        k = rotl(k, 15)
        k = (k * c2) & 0xFFFFFFFF
        h ^= k
        h = rotl(h, 13)
        h = (h * 5 + 0xE6546B64) & 0xFFFFFFFF
    tail = data[4 * nblocks:]
    k = 0
    if len(tail) >= 3:
        k ^= tail[2] << 16
    if len(tail) >= 2:
        k ^= tail[1] << 8
    if len(tail) >= 1:
        k ^= tail[0]
        k = (k * c1) & 0xFFFFFFFF
        k = rotl(k, 15)
        k = (k * c2) & 0xFFFFFFFF
        h ^= k
    h ^= n
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & 0xFFFFFFFF
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & 0xFFFFFFFF
    h ^= h >> 16
    return h
