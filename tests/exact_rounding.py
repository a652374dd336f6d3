"""Exact-rational rounding used to pin the oracle (tests only).

Independent of numpy: values are ``fractions.Fraction`` objects and every
step is integer arithmetic, so it checks ``oracle.formats`` / ``oracle.codec``
from outside.  ``round_rational`` rounds to a binary format with ``frac_bits``
fraction bits and smallest normal exponent ``e_min``, ties to even.
"""

from __future__ import annotations

from fractions import Fraction


def floor_log2(x: Fraction) -> int:
    """floor(log2(x)) for x > 0, exactly."""
    n, d = x.numerator, x.denominator
    e = n.bit_length() - d.bit_length()
    # now 2**(e-1) < x < 2**(e+1); settle the exact exponent
    if e >= 0:
        if n < (d << e):
            e -= 1
    else:
        if (n << -e) < d:
            e -= 1
    return e


def round_rational(x: Fraction, frac_bits: int, e_min: int) -> Fraction:
    """Round x to the binary format (unbounded above), ties to even; the sign
    of zero is not tracked here (callers compare magnitudes and signs apart)."""
    if x == 0:
        return Fraction(0)
    s = -1 if x < 0 else 1
    a = abs(x)
    e = max(floor_log2(a), e_min)
    quantum = Fraction(2) ** (e - frac_bits)
    n = a / quantum
    r = round(n)          # Fraction.__round__ rounds half to even
    return s * r * quantum


def to_fp32(x: Fraction) -> Fraction:
    return round_rational(x, 23, -126)


def to_fp16(x: Fraction) -> Fraction | float:
    r = round_rational(x, 10, -14)
    if abs(r) > 65504:
        return float("inf") if r > 0 else float("-inf")
    return r


def e4m3_nearest_code(v: Fraction, negative: bool, table) -> int:
    """Exhaustive nearest E4M3FN code (satfinite), ties to the even code.
    ``table`` lists (code, Fraction value) for the 127 finite non-negative codes."""
    a = abs(v)
    best = None
    for code, val in table:
        dist = abs(a - val)
        key = (dist, code & 1)
        if best is None or key < best[0]:
            best = (key, code)
    return best[1] | (0x80 if negative else 0)


def e2m1_nearest_code(v: Fraction, negative: bool) -> int:
    vals = [Fraction(0), Fraction(1, 2), Fraction(1), Fraction(3, 2),
            Fraction(2), Fraction(3), Fraction(4), Fraction(6)]
    a = abs(v)
    best = None
    for code, val in enumerate(vals):
        key = (abs(a - val), code & 1)
        if best is None or key < best[0]:
            best = (key, code)
    return best[1] | (0x8 if negative else 0)
