"""Exact reference arithmetic for pinning the oracle: rationals and the IEEE 754
round-to-nearest-even rule, written from the standard's definition and
independent of the oracle's C code and of the CPU's float unit."""
from fractions import Fraction


def half_value(bits):
    """Exact value of a binary16 bit pattern (finite only) as a Fraction."""
    s = -1 if bits & 0x8000 else 1
    e = (bits >> 10) & 0x1F
    m = bits & 0x3FF
    assert e != 31
    if e == 0:
        return s * Fraction(m, 2 ** 24)
    return s * Fraction(1024 + m, 1) * Fraction(2) ** (e - 25)


def rn(x, p=24, emin=-126):
    """Round a rational to the nearest binary floating-point number with a
    p-bit significand (ties to even), normal range only (no overflow)."""
    x = Fraction(x)
    if x == 0:
        return Fraction(0)
    s = -1 if x < 0 else 1
    a = abs(x)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    # normalise so that 2^e <= a < 2^(e+1)
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, emin)
    ulp = Fraction(2) ** (e - (p - 1))
    q, r = divmod(a, ulp)
    q = int(q)
    if r * 2 > ulp or (r * 2 == ulp and q % 2 == 1):
        q += 1
    return s * q * ulp


def rn32(x):
    return rn(x, 24, -126)


def round_half_even(x):
    x = Fraction(x)
    f = x.numerator // x.denominator
    r = x - f
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and f % 2 == 1):
        f += 1
    return f
