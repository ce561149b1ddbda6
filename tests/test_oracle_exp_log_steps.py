"""Step-exact pins for the oracle's exp and log.

The pages fix that the spellings of exp and log, and the tie rules, belong to
the frozen profile ("mojolearn" PyPI page, sections "What bitwise identity
means, and why it is not the default" and "The exact scope of the claim"); they
print no spelling. Profile v1's readings (R14 for exp, R15 for log) are
restated here step by step and evaluated in exact rational arithmetic with
round-to-nearest-even written by hand (ieee_exact), then compared bit for bit
with the oracle's compiled C:

* every constant is checked against its definition (the float nearest to
  1/ln 2, ln 2, 1/k!, 2/k, ...) with 200-bit arithmetic, independently of the
  oracle;
* exp: every tie of the round-to-integer step (where rint, round-half-away and
  an unrounded t part ways), a stratified sample of every binade of the
  argument, arguments whose reduced value sits on a rounding midpoint (where
  the split of ln 2 shows), the band whose results are subnormal, and the
  range ends;
* log: every binade of the argument (subnormals included), both sides of the
  sqrt 2 split of the mantissa, and the split's boundary values.

A plausible slip in the oracle -- roundf for rintf, another split of ln 2,
Horner terms in another order, a contracted multiply-add, a different
threshold -- changes some of these results.
"""
import math
from fractions import Fraction

import mpmath
import numpy as np

import ieee_exact as ie
import oracle
from exp_cases import binade_samples, exp_tie_arguments, reduction_sensitive_arguments

F = np.float32
mpmath.mp.prec = 200


def hexf(s: str) -> np.float32:
    return F(float.fromhex(s))


def nearest_f32(v) -> np.float32:
    """The float nearest to an mpmath value (exact rational rounding)."""
    m, e = mpmath.frexp(v)
    return ie.round_f32(Fraction(int(mpmath.ldexp(m, 120))) * Fraction(2) ** (e - 120))


# profile v1's constants (R14, R15), restated
LOG2E = hexf("0x1.715476p+0")
LN2_HI = hexf("0x1.62e430p-1")
LN2_LO = hexf("-0x1.05c610p-29")
EXPC = [hexf(h) for h in ("0x1p+0", "0x1p+0", "0x1p-1", "0x1.555556p-3", "0x1.555556p-5",
                           "0x1.111112p-7", "0x1.6c16c2p-10", "0x1.a01a02p-13")]
EXP_HI = hexf("0x1.62e42ep+6")
EXP_LO = F(-104.0)
LOGT = {3: hexf("0x1.555556p-1"), 5: hexf("0x1.99999ap-2"), 7: hexf("0x1.24924ap-2"),
        9: hexf("0x1.c71c72p-3"), 11: hexf("0x1.745d18p-3")}
SQRT2_BITS = 0x3FB504F3


def test_constants_are_the_floats_nearest_their_definitions():
    ln2 = mpmath.log(2)
    assert ie.bits(LOG2E) == ie.bits(nearest_f32(1 / ln2))
    assert ie.bits(LN2_HI) == ie.bits(nearest_f32(ln2))
    assert ie.bits(LN2_LO) == ie.bits(nearest_f32(ln2 - mpmath.mpf(float(LN2_HI))))
    for k, c in enumerate(EXPC):
        assert ie.bits(c) == ie.bits(ie.round_f32(Fraction(1, math.factorial(k)))), k
    for k, c in LOGT.items():
        assert ie.bits(c) == ie.bits(ie.round_f32(Fraction(2, k))), k
    s = np.array([SQRT2_BITS, SQRT2_BITS + 1], np.uint32).view(F)
    assert mpmath.mpf(float(s[0])) < mpmath.sqrt(2) < mpmath.mpf(float(s[1]))
    # EXP_HI: the largest float whose exp rounds to a finite float (below the
    # midpoint between FLT_MAX and 2^128); EXP_LO: exp(-104) is below half the
    # smallest subnormal, so every argument below it gives +0
    over = mpmath.mpf(2) ** 128 * (1 - mpmath.mpf(2) ** -25)
    nxt = np.array([ie.bits(EXP_HI) + 1], np.uint32).view(F)[0]
    assert mpmath.exp(float(EXP_HI)) < over <= mpmath.exp(float(nxt))
    assert mpmath.exp(float(EXP_LO)) < mpmath.mpf(2) ** -150


def rint_half_even(t: np.float32) -> np.float32:
    q = ie.to_frac(t)
    fl = q.numerator // q.denominator
    rem = q - fl
    n = fl + 1 if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1) else fl
    out = F(n)
    return F(-0.0) if n == 0 and ie.is_neg(t) else out


def pow2(e: int) -> np.float32:
    return F(2.0 ** e)


def exp_steps(x: np.float32) -> np.float32:
    """R14 step by step, each operation rounded by hand."""
    x = F(x)
    if np.isnan(x):
        return x
    if x > EXP_HI:
        return F(np.inf)
    if x < EXP_LO:
        return F(0.0)
    t = ie.mul(x, LOG2E)
    n = rint_half_even(t)
    mn = F(-n)
    r = ie.fma(mn, LN2_HI, x)
    r = ie.fma(mn, LN2_LO, r)
    p = EXPC[7]
    for k in range(6, -1, -1):
        p = ie.fma(p, r, EXPC[k])
    ni = int(n)
    if ni > 127:
        return ie.mul(ie.add(p, p), pow2(127))
    if ni < -126:
        return ie.mul(ie.mul(p, pow2(ni + 64)), pow2(-64))
    return ie.mul(p, pow2(ni))


def log_steps(x: np.float32) -> np.float32:
    """R15 step by step, each operation rounded by hand (positive finite x)."""
    x = F(x)
    e = 0
    if x < F(np.finfo(F).tiny):
        x = ie.mul(x, pow2(23))
        e = -23
    b = ie.bits(x)
    e += (b >> 23) - 127
    fb = (b & 0x7FFFFF) | 0x3F800000
    if fb > SQRT2_BITS:
        fb -= 0x800000
        e += 1
    f = np.array([fb], np.uint32).view(F)[0]
    u = ie.sub(f, F(1.0))
    s = ie.div(u, ie.add(F(2.0), u))
    z = ie.mul(s, s)
    R = LOGT[11]
    for k in (9, 7, 5, 3):
        R = ie.fma(R, z, LOGT[k])
    R = ie.mul(R, z)
    h = ie.mul(ie.mul(F(0.5), u), u)
    lf = ie.sub(u, ie.sub(h, ie.mul(s, ie.add(h, R))))
    ef = F(e)
    return ie.fma(ef, LN2_HI, ie.fma(ef, LN2_LO, lf))


def check(xs, steps, fn):
    xs = np.asarray(xs, F)
    got = fn(xs)
    bad = [(float(x), ie.bits(g), ie.bits(steps(x))) for x, g in zip(xs, got)
           if not ie.same_bits(g, steps(x))]
    assert not bad, f"{len(bad)} of {xs.size} differ, first {bad[:3]}"


def test_exp_ties_of_the_rounding_step():
    # every tie of rint(x LOG2E) over the whole finite range, both signs
    d = exp_tie_arguments(-151, 128)
    d = d[(d >= EXP_LO) & (d <= EXP_HI)]
    assert d.size > 600
    check(d, exp_steps, oracle.exp)


def test_exp_every_binade_stratified():
    # |x| from 2^-40 to 2^6, 200 random mantissas a binade and sign, plus the
    # top binade up to the ends of the range
    x = binade_samples(11, -40, 5, 200)
    x = np.concatenate([x, binade_samples(12, 6, 6, 400)])
    x = x[(x >= EXP_LO) & (x <= EXP_HI)]
    check(x, exp_steps, oracle.exp)


def test_exp_reduction_sensitive_arguments():
    # large |n|, reduced argument within 2^-10 ulp of a rounding midpoint: the
    # inputs where the bits of the ln 2 that the reduction subtracts, and the
    # order of its two steps, reach the result
    x = reduction_sensitive_arguments()
    assert x.size > 2000
    check(x, exp_steps, oracle.exp)


def test_exp_subnormal_results_and_range_ends():
    # results below FLT_MIN: x in [-104, -87.34]; n < -126 takes the two-step
    # scaling, which rounds once into the subnormals
    rng = np.random.default_rng(13)
    x = rng.uniform(-104.0, -87.3, 3000).astype(F)
    ends = np.array([EXP_LO, np.nextafter(EXP_LO, F(0)), EXP_HI,
                     np.nextafter(EXP_HI, F(0)), F(-87.33654), F(88.0), F(-0.0), F(0.0),
                     F(2.0 ** -149), F(-(2.0 ** -149))], F)
    check(np.concatenate([x, ends]), exp_steps, oracle.exp)


def test_log_every_binade_both_sides_of_the_split():
    rng = np.random.default_rng(14)
    out = []
    for e in range(-126, 128):
        # mantissa fields below and above the sqrt 2 split (0x3504f3)
        lo = rng.integers(0, 0x3504F4, 40, dtype=np.int64)
        hi = rng.integers(0x3504F4, 1 << 23, 40, dtype=np.int64)
        for m in (lo, hi):
            out.append((((e + 127) << 23) | m).astype(np.uint32).view(F))
    sub = rng.integers(1, 1 << 23, 2000, dtype=np.int64).astype(np.uint32).view(F)
    x = np.concatenate(out + [sub])
    check(x, log_steps, oracle.log)


def test_log_split_boundary_and_special_points():
    pts = []
    for e in range(-149, 128, 7):
        for m in (0, 1, 0x3504F2, 0x3504F3, 0x3504F4, 0x3504F5, 0x7FFFFF):
            if e >= -126:
                pts.append(((e + 127) << 23) | m)
    pts += [1, 2, 3, 0x7FFFFF, 0x3F800000, 0x3F800001, 0x3F7FFFFF, 0x7F7FFFFF,
            ie.bits(F(50257.0))]
    check(np.array(pts, np.uint32).view(F), log_steps, oracle.log)
