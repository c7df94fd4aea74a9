"""Exact rational arithmetic with explicit IEEE round-to-nearest-even, used to
check the oracle's floating-point sequences without using the hardware's own
fp32/fp64 operations."""
from fractions import Fraction
import struct

F32 = (24, -126)   # significand bits, minimum normal exponent
F64 = (53, -1022)


def _floor_log2(a: Fraction) -> int:
    n, d = a.numerator, a.denominator
    e = n.bit_length() - d.bit_length()
    # adjust so that 2^e <= a < 2^(e+1)
    if e >= 0:
        if n < d << e:
            e -= 1
    else:
        if n << -e < d:
            e -= 1
    return e


def rnd(x, fmt=F32) -> Fraction:
    """Round the exact value x to the nearest value of the format, ties to
    even (no overflow handling; the callers stay in range)."""
    x = Fraction(x)
    if x == 0:
        return Fraction(0)
    p, emin = fmt
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = max(_floor_log2(a), emin)
    quantum = Fraction(2) ** (e - p + 1)
    m = a / quantum
    fl = m.numerator // m.denominator
    rem = m - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * fl * quantum


def f32(x) -> float:
    """Python float holding the fp32 value nearest to x (ties to even)."""
    return float(rnd(Fraction(x), F32))


def f32_bits(v: float) -> int:
    return struct.unpack("<I", struct.pack("<f", v))[0]


def ulp32(v: float) -> float:
    a = abs(Fraction(v))
    e = max(_floor_log2(a), -126) if a else -126
    return float(Fraction(2) ** (e - 23))
