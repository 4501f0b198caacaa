"""Exact rational re-derivations used to pin the oracle (independent of numpy arithmetic)."""
from __future__ import annotations

import math
from fractions import Fraction as Fr


def fl32(x: Fr) -> Fr:
    """Round a rational to the nearest IEEE float32 value (ties to even), subnormals included."""
    if x == 0:
        return Fr(0)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fr(2) ** e > a:
        e -= 1
    if Fr(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    ulp = Fr(2) ** (e - 23)
    return sign * rne(a / ulp) * ulp


def rne(x: Fr) -> int:
    """Round a rational to the nearest integer, ties to even."""
    fl = math.floor(x)
    rem = x - fl
    if rem > Fr(1, 2) or (rem == Fr(1, 2) and fl % 2 == 1):
        fl += 1
    return fl


def quantize_block_exact(values) -> tuple[list[int], Fr]:
    """delta = fl32(max|x|/127); q = clamp(rne(fl32(x/delta)), -127, 127); zero block -> 0."""
    xs = [Fr(v) for v in values]
    mx = max((abs(v) for v in xs), default=Fr(0))
    delta = fl32(mx / 127)
    if delta == 0:
        return [0] * len(xs), Fr(0)
    return [max(-127, min(127, rne(fl32(v / delta)))) for v in xs], delta
