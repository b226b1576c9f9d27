"""Exact-rational rounding helpers used to pin the oracle (independent of it).

``rne_bf16_exact`` rounds a Fraction to bfloat16 by searching the sorted table of
every positive finite bf16 value (built by decoding all bit patterns), so it
shares no rounding logic with the oracle's arithmetic. ``rne_f32_exact`` rounds
a Fraction to fp32 by comparing it exactly against the three fp32 neighbours of
a first guess.
"""
from __future__ import annotations

import bisect
import struct
from fractions import Fraction

import numpy as np


def _decode_bf16(bits: int) -> Fraction:
    f = struct.unpack("<f", struct.pack("<I", bits << 16))[0]
    return Fraction(f)


# every positive finite bf16 value, ascending; bits 0x0001 .. 0x7F7F
_POS_BITS = list(range(0x0001, 0x7F80))
_POS_VALS = [_decode_bf16(b) for b in _POS_BITS]
_TWO_128 = Fraction(2) ** 128


def rne_bf16_exact(v: Fraction) -> int:
    """bf16 bits nearest to v, ties to the even bit pattern, overflow to +-inf."""
    v = Fraction(v)
    sign = 0x8000 if v < 0 else 0
    a = -v if v < 0 else v
    if a == 0:
        return sign
    # candidates: 0, every finite value, and 2^128 (the overflow threshold stands for inf)
    vals = [Fraction(0)] + _POS_VALS + [_TWO_128]
    bits = [0x0000] + _POS_BITS + [0x7F80]
    i = bisect.bisect_left(vals, a)
    if i < len(vals) and vals[i] == a:
        return sign | bits[i]
    if i >= len(vals):
        return sign | 0x7F80
    lo, hi = i - 1, i
    dlo, dhi = a - vals[lo], vals[hi] - a
    if dlo < dhi:
        pick = lo
    elif dhi < dlo:
        pick = hi
    else:  # tie: the even significand (bit pattern even; 2^128 counts as even)
        pick = lo if bits[lo] % 2 == 0 else hi
    return sign | bits[pick]


def bf16_bits_to_fraction(bits: int) -> Fraction:
    bits &= 0xFFFF
    mag = _decode_bf16(bits & 0x7FFF)
    return -mag if bits & 0x8000 else mag


def rne_f32_exact(v: Fraction) -> np.float32:
    """fp32 nearest to v (ties to even), via exact comparison with neighbours."""
    v = Fraction(v)
    if v == 0:
        return np.float32(0.0)
    guess = np.float32(float(v)) if abs(float(v)) < 3.5e38 else np.float32(np.inf) * np.sign(float(v))
    cands = {guess, np.nextafter(guess, np.float32(np.inf)), np.nextafter(guess, np.float32(-np.inf))}
    best = None
    for c in cands:
        if not np.isfinite(c):
            continue
        d = abs(Fraction(float(c)) - v)
        key = (d, int(np.float32(c).view(np.uint32)) & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return np.float32(best[1])


def pow2(e: int) -> Fraction:
    return Fraction(2) ** e if e >= 0 else Fraction(1, 2 ** (-e))


def rne_f64_exact(v: Fraction) -> float:
    """fp64 nearest to v (ties to even; subnormals kept; overflow to +-inf). Python's
    int/Fraction to float conversion is correctly rounded; only its overflow needs care."""
    v = Fraction(v)
    if v == 0:
        return 0.0
    big = Fraction(2) ** 1024 - Fraction(2) ** (1024 - 54)  # halfway between max finite and 2^1024
    if abs(v) >= big:
        return float("inf") if v > 0 else float("-inf")
    return float(v)
