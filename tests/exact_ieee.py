"""IEEE-754 rounding written from its definition, on exact rationals.

Used to pin the oracle: a binary32 sum is the exact sum rounded to the
nearest binary32 value, ties to the even significand; BF16 rounding is the
same rule with 7 stored fraction bits.  Nothing here uses hardware floating
point for the arithmetic being checked, so it is independent of the C
oracle's float adds and of its bias-and-truncate rounding.

Values are ``(Fraction, negative_zero)`` pairs so that the sign of zero is
tracked the way IEEE addition defines it.
"""
from __future__ import annotations

import struct
from fractions import Fraction

Value = tuple  # (Fraction, bool)


def _exponent(a: Fraction) -> int:
    """e with 2^e <= a < 2^(e+1), for a > 0."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def _round_to_format(x: Fraction, frac_bits: int, emin: int, emax: int):
    """Nearest value of a binary format with ``frac_bits`` stored fraction
    bits and normal exponent range [emin, emax]; ties go to the even
    significand; results beyond the largest finite value give +-inf."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    a = -x if x < 0 else x
    e = max(_exponent(a), emin)  # below the normal range the spacing stays fixed
    ulp = Fraction(2) ** (e - frac_bits)
    q = a / ulp
    n = q.numerator // q.denominator
    rem = q - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    r = n * ulp
    max_finite = (2 - Fraction(2) ** (-frac_bits)) * Fraction(2) ** emax
    if r > max_finite:
        return sign * float("inf")
    return sign * r


def round_binary32(x: Fraction):
    return _round_to_format(x, 23, -126, 127)


def round_bf16(x: Fraction):
    return _round_to_format(x, 7, -126, 127)


def bf16_bits_to_value(h: int) -> Value:
    """Decode a finite BF16 bit pattern exactly (raises on inf / NaN)."""
    sign = (h >> 15) & 1
    exp = (h >> 7) & 0xFF
    frac = h & 0x7F
    if exp == 0xFF:
        raise ValueError("inf/NaN are not finite rationals")
    if exp == 0:
        mag = Fraction(frac, 128) * Fraction(2) ** -126
    else:
        mag = (1 + Fraction(frac, 128)) * Fraction(2) ** (exp - 127)
    if mag == 0:
        return (Fraction(0), bool(sign))
    return (-mag if sign else mag, False)


def f32_bits_to_value(u: int) -> Value:
    """Decode a finite binary32 bit pattern exactly."""
    sign = (u >> 31) & 1
    exp = (u >> 23) & 0xFF
    frac = u & 0x7FFFFF
    if exp == 0xFF:
        raise ValueError("inf/NaN are not finite rationals")
    if exp == 0:
        mag = Fraction(frac, 1 << 23) * Fraction(2) ** -126
    else:
        mag = (1 + Fraction(frac, 1 << 23)) * Fraction(2) ** (exp - 127)
    if mag == 0:
        return (Fraction(0), bool(sign))
    return (-mag if sign else mag, False)


def value_to_bf16_bits(x) -> int:
    """Encode a value that is exactly a BF16 number (or +-inf) as bits;
    a zero is encoded as +0."""
    if isinstance(x, float):
        return 0x7F80 if x > 0 else 0xFF80
    if x == 0:
        return 0x0000
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    e = _exponent(a)
    if e < -126:  # subnormal: multiples of 2^-133
        frac = a / (Fraction(2) ** -133)
        assert frac.denominator == 1 and frac < 128, "not a BF16 subnormal"
        return sign | int(frac)
    m = (a / Fraction(2) ** e - 1) * 128
    assert m.denominator == 1, "value is not representable in BF16"
    return sign | ((e + 127) << 7) | int(m)


def add_binary32(a: Value, b: Value) -> Value:
    """IEEE binary32 addition, round to nearest even, from the definition.
    An exact zero sum is +0 unless both operands are -0."""
    xa, za = a
    xb, zb = b
    if isinstance(xa, float) or isinstance(xb, float):
        raise ValueError("infinite operands are outside this helper")
    s = xa + xb
    if s == 0:
        return (Fraction(0), bool(xa == 0 and za and xb == 0 and zb))
    return (round_binary32(s), False)


def fold_bf16_exact(column: list[int]) -> int:
    """The fixed-order reduction of one element, computed exactly:
    acc = x_0; acc = round32(acc + x_q) for q = 1..P-1; result = round_bf16(acc).
    Raises ValueError if a partial sum overflows before the last add."""
    acc = bf16_bits_to_value(column[0])
    for h in column[1:]:
        acc = add_binary32(acc, bf16_bits_to_value(h))
    x, negzero = acc
    if isinstance(x, float):
        return value_to_bf16_bits(x)
    if x == 0:
        return 0x8000 if negzero else 0x0000
    return value_to_bf16_bits(round_bf16(x))


def _signed(bits: int, x, width_sign: int) -> int:
    """A result that rounded to zero keeps the sign of the value rounded."""
    return (width_sign if x < 0 else 0) if bits == 0 else bits


def f32_to_bf16_exact(u: int) -> int:
    """Round a finite binary32 bit pattern to BF16 from the definition."""
    x, negzero = f32_bits_to_value(u)
    if x == 0:
        return 0x8000 if negzero else 0x0000
    return _signed(value_to_bf16_bits(round_bf16(x)), x, 0x8000)


def f32_bits(f: float) -> int:
    return struct.unpack("<I", struct.pack("<f", f))[0]


# ------------------------------------------------------ binary16 and orders ---

def round_f16(x: Fraction):
    return _round_to_format(x, 10, -14, 15)


def f16_bits_to_value(h: int) -> Value:
    """Decode a finite binary16 bit pattern exactly (raises on inf / NaN)."""
    sign = (h >> 15) & 1
    exp = (h >> 10) & 0x1F
    frac = h & 0x3FF
    if exp == 0x1F:
        raise ValueError("inf/NaN are not finite rationals")
    if exp == 0:
        mag = Fraction(frac, 1024) * Fraction(2) ** -14
    else:
        mag = (1 + Fraction(frac, 1024)) * Fraction(2) ** (exp - 15)
    if mag == 0:
        return (Fraction(0), bool(sign))
    return (-mag if sign else mag, False)


def value_to_f16_bits(x) -> int:
    """Encode a value that is exactly a binary16 number (or +-inf)."""
    if isinstance(x, float):
        return 0x7C00 if x > 0 else 0xFC00
    if x == 0:
        return 0x0000
    sign = 0x8000 if x < 0 else 0
    a = -x if x < 0 else x
    e = _exponent(a)
    if e < -14:  # subnormal: multiples of 2^-24
        frac = a / (Fraction(2) ** -24)
        assert frac.denominator == 1 and frac < 1024, "not a binary16 subnormal"
        return sign | int(frac)
    m = (a / Fraction(2) ** e - 1) * 1024
    assert m.denominator == 1, "value is not representable in binary16"
    return sign | ((e + 15) << 10) | int(m)


def value_to_f32_bits(x) -> int:
    """Encode a value that is exactly a binary32 number (or +-inf)."""
    if isinstance(x, float):
        return 0x7F800000 if x > 0 else 0xFF800000
    if x == 0:
        return 0
    sign = 0x80000000 if x < 0 else 0
    a = -x if x < 0 else x
    e = _exponent(a)
    if e < -126:
        frac = a / (Fraction(2) ** -149)
        assert frac.denominator == 1 and frac < (1 << 23)
        return sign | int(frac)
    m = (a / Fraction(2) ** e - 1) * (1 << 23)
    assert m.denominator == 1
    return sign | ((e + 127) << 23) | int(m)


DECODE = {"bf16": bf16_bits_to_value, "f16": f16_bits_to_value, "f32": f32_bits_to_value}


def fold_exact(column: list[int], dtype: str = "bf16", order: str = "linear") -> int:
    """The fixed-order reduction of one element, computed exactly, for
    element type `dtype` and summation order `order` ("linear": left to
    right; "tree": split at the largest power of two below the count, fold
    each side, add).  Raises ValueError if a partial sum overflows before the
    last add.  Returns the result's bit pattern."""
    vals = [DECODE[dtype](h) for h in column]

    def tree(lo, hi):
        n = hi - lo
        if n == 1:
            return vals[lo]
        m = 1
        while m * 2 < n:
            m *= 2
        return add_binary32(tree(lo, lo + m), tree(lo + m, hi))

    if order == "tree":
        acc = tree(0, len(vals))
    else:
        acc = vals[0]
        for v in vals[1:]:
            acc = add_binary32(acc, v)
    x, negzero = acc
    if dtype == "f32":
        if isinstance(x, float):
            return value_to_f32_bits(x)
        return (0x80000000 if negzero else 0) if x == 0 else value_to_f32_bits(x)
    if isinstance(x, float):
        return value_to_bf16_bits(x) if dtype == "bf16" else value_to_f16_bits(x)
    if x == 0:
        return 0x8000 if negzero else 0x0000
    if dtype == "bf16":
        return _signed(value_to_bf16_bits(round_bf16(x)), x, 0x8000)
    return _signed(value_to_f16_bits(round_f16(x)), x, 0x8000)


def f32_to_f16_exact(u: int) -> int:
    x, negzero = f32_bits_to_value(u)
    if x == 0:
        return 0x8000 if negzero else 0x0000
    return _signed(value_to_f16_bits(round_f16(x)), x, 0x8000)
