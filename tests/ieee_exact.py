"""Exact-rational emulation of IEEE 754 binary32 operations (test helper).

Every operation is computed exactly as a Fraction and then rounded to the
binary32 grid by hand (round to nearest, ties to even, gradual underflow,
overflow to infinity), with the sign-of-zero rules of IEEE 754-2008 section
6.3. Nothing here calls the platform's float arithmetic on the values being
rounded, so it is an independent check of the oracle's compiled C, which does.
"""
from __future__ import annotations

import math
from fractions import Fraction

import numpy as np

_EMIN = -126          # smallest normal exponent
_P = 24               # precision in bits
_MAXF = Fraction((2 ** _P - 1) * 2 ** (127 - _P + 1))   # FLT_MAX


def is_neg(x: np.float32) -> bool:
    return bool(np.signbit(np.float32(x)))


def to_frac(x) -> Fraction:
    x = np.float32(x)
    if not np.isfinite(x):
        raise ValueError("finite values only")
    return Fraction(float(x))   # float32 -> double is exact


def _floor_log2(a: Fraction) -> int:
    # 2^e <= a < 2^(e+1) for a > 0
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    elif Fraction(2) ** (e + 1) <= a:
        e += 1
    return e


def round_f32(q: Fraction, neg_zero: bool = False) -> np.float32:
    """Round an exact rational to binary32. A zero result takes the sign of q
    (underflow) or, when q == 0, the sign given by neg_zero."""
    if q == 0:
        return np.float32(-0.0) if neg_zero else np.float32(0.0)
    neg = q < 0
    a = -q if neg else q
    e = max(_floor_log2(a), _EMIN)
    ulp = Fraction(2) ** (e - (_P - 1))
    m = a / ulp
    n = m.numerator // m.denominator
    rem = m - n
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and n % 2 == 1):
        n += 1
    v = n * ulp
    if v > _MAXF:
        out = np.float32(np.inf)
    else:
        out = np.float32(float(v))        # v is on the binary32 grid: exact
    return np.float32(-out) if neg else out


def add(a, b) -> np.float32:
    a, b = np.float32(a), np.float32(b)
    q = to_frac(a) + to_frac(b)
    # exact zero: -0 only when both addends are -0
    return round_f32(q, neg_zero=(q == 0 and a == 0 and b == 0
                                  and is_neg(a) and is_neg(b)))


def sub(a, b) -> np.float32:
    return add(a, np.float32(-np.float32(b)))


def mul(a, b) -> np.float32:
    a, b = np.float32(a), np.float32(b)
    q = to_frac(a) * to_frac(b)
    return round_f32(q, neg_zero=(is_neg(a) != is_neg(b)))


def div(a, b) -> np.float32:
    a, b = np.float32(a), np.float32(b)
    if b == 0:
        raise ZeroDivisionError
    q = to_frac(a) / to_frac(b)
    return round_f32(q, neg_zero=(is_neg(a) != is_neg(b)))


def fma(a, b, c) -> np.float32:
    """a*b + c with a single rounding."""
    a, b, c = np.float32(a), np.float32(b), np.float32(c)
    prod = to_frac(a) * to_frac(b)
    q = prod + to_frac(c)
    prod_neg = is_neg(a) != is_neg(b)
    neg_zero = (q == 0 and prod == 0 and prod_neg and c == 0 and is_neg(c))
    return round_f32(q, neg_zero=neg_zero)


def sqrt(a) -> np.float32:
    """Correctly rounded square root (a >= 0). The exact root is bracketed to
    far below half an ulp; a binary32 square root never falls on a midpoint."""
    a = np.float32(a)
    if a == 0:
        return a
    if a < 0:
        raise ValueError
    q = to_frac(a)
    s = 200
    n = (q * Fraction(4) ** s)
    n = n.numerator // n.denominator
    r = math.isqrt(n)
    if r * r == n and Fraction(n) == q * Fraction(4) ** s:
        return round_f32(Fraction(r, 2 ** s))
    return round_f32(Fraction(2 * r + 1, 2 ** (s + 1)))


def bits(x) -> int:
    return int(np.float32(x).view(np.uint32))


def same_bits(x, y) -> bool:
    """Bitwise equality, with every NaN equal to every NaN."""
    x, y = np.float32(x), np.float32(y)
    if np.isnan(x) or np.isnan(y):
        return bool(np.isnan(x) and np.isnan(y))
    return bits(x) == bits(y)
