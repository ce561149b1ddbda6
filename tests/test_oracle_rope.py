"""Pins for the oracle's sin/cos spelling and rotary position embedding.

The model card ("MojoLearn 162M", table "Compared with GPT-3 Small") uses rotary
positions with theta = 10,000 over 12 heads of 64; the pages fix that the
transcendental spellings belong to the profile and print none. Readings:
  * sin/cos (R31): k = rint(x 2/pi), r = x - k pi/2 by three fmaf steps with
    pi/2 split in three floats, Taylor polynomials to degree 9 (sin) and 10
    (cos) in z = r^2 by fmaf Horner, the quadrant k mod 4;
  * rotary (R30): pairs (2i, 2i+1) of a head turn by pos * w_i,
    w_i = exp(-(2i/d) log(theta)); y0 = x0 c - x1 s, y1 = x0 s + x1 c.
Pinned by accuracy against the C library's double sin and cos (exhaustive on
[0, pi/4], strided to 4096), exact odd/even symmetry, special values, the
written steps re-evaluated in exact rationals, and for the rotation: the
identity at position 0, the pairing, norm preservation and a double bound.
"""
import math

import numpy as np

import ieee_exact as ie
import oracle
from bitcmp import assert_bitwise

F = np.float32
U = 2.0 ** -24


def fbits(x):
    return int(np.array([x], F).view(np.uint32)[0])


def test_accuracy_on_the_reduced_range():
    # every float in [0.5, pi/4] (the binade where the polynomials' error
    # peaks) and every 13th below: sin within 0.7 ulp, cos within 0.9 ulp
    top = fbits(math.pi / 4)
    for which, bound in ((0, 0.75), (1, 0.95)):
        m1, _ = oracle.sincos_ulp_scan(which, fbits(0.5), top + 1)
        m2, _ = oracle.sincos_ulp_scan(which, 0x00000000, fbits(0.5), 13)
        assert 0 <= m1 < bound and 0 <= m2 < bound


def test_accuracy_to_4096_strided():
    # every 101st float from pi/4 to 4096 (both signs): 1.5 ulp, or 1.5 ulps
    # of 2^-6 (an absolute 2^-28.4) nearer the zeros
    lo, hi = fbits(math.pi / 4), fbits(4096.0)
    for which in (0, 1):
        for base in (0, 0x80000000):
            m, _ = oracle.sincos_ulp_scan(which, base + lo, base + hi, 101)
            assert 0 <= m < 1.5


def test_symmetry_and_special_values():
    rng = np.random.default_rng(81)
    x = (rng.standard_normal(200000) * np.exp2(rng.integers(-20, 12, 200000))).astype(F)
    assert_bitwise(oracle.sin(-x), -oracle.sin(x), "sin is odd")
    assert_bitwise(oracle.cos(-x), oracle.cos(x), "cos is even")
    sp = np.array([0.0, -0.0, 2.0 ** -140, 2.0 ** 20, 2.0 ** 20 * 1.0000001, np.nan, np.inf], F)
    s, c = oracle.sin(sp), oracle.cos(sp)
    assert s.view(np.uint32)[0] == 0 and s.view(np.uint32)[1] == 0x80000000
    assert c[0] == F(1.0) and c[1] == F(1.0)
    assert s[2] == sp[2] and c[2] == F(1.0)             # sin x = x for tiny x
    assert np.isfinite(s[3]) and np.isnan(s[4]) and np.isnan(s[5]) and np.isnan(s[6])
    # pi/2 as a float lies 4.37e-8 above pi/2: cos is -4.37e-8 to within its
    # absolute accuracy, sin rounds to 1
    p = F(math.pi / 2)
    assert oracle.sin(np.array([p], F))[0] == F(1.0)
    assert abs(float(oracle.cos(np.array([p], F))[0]) - math.cos(float(p))) < 2.0 ** -48


def test_written_steps_in_exact_arithmetic():
    two_over_pi = F(float.fromhex('0x1.45f306p-1'))
    P = [F(float.fromhex(h)) for h in ('0x1.921fb6p+0', '-0x1.777a5cp-25', '-0x1.ee59dap-50')]
    S = [F(float.fromhex(h)) for h in ('0x1.71de3ap-19', '-0x1.a01a02p-13', '0x1.111112p-7',
                                         '-0x1.555556p-3')]
    C = [F(float.fromhex(h)) for h in ('-0x1.27e4fcp-22', '0x1.a01a02p-16', '-0x1.6c16c2p-10',
                                         '0x1.555556p-5', '-0x1p-1')]
    # each constant is the float nearest to its definition
    assert P[0] == F(math.pi / 2) and S[3] == F(-1 / 6) and C[4] == F(-0.5)
    assert S[0] == F(1 / math.factorial(9)) and C[0] == F(-1 / math.factorial(10))
    rng = np.random.default_rng(82)
    xs = (rng.uniform(-3000, 3000, 64)).astype(F)
    for x in xs:
        k = F(np.rint(ie.mul(x, two_over_pi)))
        r = x
        for pk in P:
            r = ie.fma(F(-k), pk, r)
        z = ie.mul(r, r)
        ps = S[0]
        for cst in S[1:]:
            ps = ie.fma(ps, z, cst)
        s = ie.fma(r, ie.mul(z, ps), r)
        pc = C[0]
        for cst in C[1:]:
            pc = ie.fma(pc, z, cst)
        c = ie.fma(pc, z, F(1.0))
        q = int(k) & 3
        sn = [s, c, -s, -c][q]
        cs = [c, -s, -c, s][q]
        assert ie.same_bits(oracle.sin(np.array([x], F))[0], F(sn)), x
        assert ie.same_bits(oracle.cos(np.array([x], F))[0], F(cs)), x


def test_rope_pairing_identity_and_norm():
    heads, d, T = 3, 64, 40
    # position 0 turns by 0: every value unchanged (signs of zero aside)
    rng = np.random.default_rng(83)
    x = rng.standard_normal((T, heads * d)).astype(F)
    y = oracle.rope(x, heads, d, seq_len=T)
    assert np.array_equal(y[0], x[0])
    # the pairs are (2i, 2i+1): a unit at 2i moves into (2i, 2i+1) only
    e = np.zeros((T, heads * d), F)
    e[:, 2 * 5] = 1.0
    ye = oracle.rope(e, heads, d, seq_len=T)
    nz = np.nonzero(ye[7])[0]
    assert set(nz.tolist()) <= {10, 11}
    a = F(F(7.0) * oracle.exp1(F(-(F(10.0) / F(64.0)) * oracle.log1(F(10000.0)))))
    assert ye[7, 10] == oracle.cos(np.array([a], F))[0]
    assert ye[7, 11] == oracle.sin(np.array([a], F))[0]
    # a rotation keeps the norm of every pair
    n0 = x[:, 0::2].astype(np.float64) ** 2 + x[:, 1::2].astype(np.float64) ** 2
    n1 = y[:, 0::2].astype(np.float64) ** 2 + y[:, 1::2].astype(np.float64) ** 2
    assert np.all(np.abs(n1 - n0) <= 8 * U * n0 + 1e-30)


def test_rope_double_bound():
    heads, d, T, seq = 2, 64, 4096, 2048
    rng = np.random.default_rng(84)
    x = rng.standard_normal((T, heads * d)).astype(F)
    y = oracle.rope(x, heads, d, seq_len=seq)
    pos = (np.arange(T) % seq).astype(np.float64)[:, None]
    i = np.arange(d // 2, dtype=np.float64)
    w = 10000.0 ** (-(2 * i) / d)
    ang = pos * w[None, :]
    c, s = np.cos(ang), np.sin(ang)
    for h in range(heads):
        x0 = x[:, h * d:(h + 1) * d:2].astype(np.float64)
        x1 = x[:, h * d + 1:(h + 1) * d:2].astype(np.float64)
        y0 = x0 * c - x1 * s
        y1 = x0 * s + x1 * c
        # the float angle pos * w carries the frequency's error (up to ~8 ulps:
        # exp magnifies the rounding of its argument -(2i/d) log(theta)) and
        # its own rounding, so at pos ~ 2048 the rotation is off by up to
        # ~ angle * 10 * 2^-24 radians
        tol = (np.abs(x0) + np.abs(x1)) * (6 * U + pos * w[None, :] * 10 * U)
        assert np.all(np.abs(y[:, h * d:(h + 1) * d:2] - y0) <= tol)
        assert np.all(np.abs(y[:, h * d + 1:(h + 1) * d:2] - y1) <= tol)
