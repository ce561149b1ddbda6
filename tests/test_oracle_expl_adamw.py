"""Pins for the oracle's exp and log spellings and its AdamW update.

exp/log (the "mojolearn" PyPI page, section "What bitwise identity means, and
why it is not the default": the spellings of exp and log are fixed by the
profile; the pages print none). v1 reading: exp by Cody-Waite reduction with
round-half-even n and a degree-7 Taylor polynomial, scaled by 2^n with one
rounding; log by exponent split and the atanh series. Their exact bits are the
reading's, not the pages' (parity unpinned by the pages); what pins them here is
accuracy against the C library's double exp/log over every float input, and
exact special values.

AdamW ("MojoLearn 162M" model card, table "Training": AdamW, beta (0.9, 0.95),
eps 1e-8, weight decay 0.1, no clipping) in its decoupled form
p <- p (1 - lr wd) - lr m_hat / (sqrt(v_hat) + eps): pinned by closed forms and
a double-precision bound.
"""
import math
import struct

import numpy as np
import pytest

import ieee_exact as ie
import oracle
from bitcmp import assert_bitwise

F = np.float32
U = 2.0 ** -24


def fbits(x):
    return struct.unpack("<I", struct.pack("<f", float(x)))[0]


# ----------------------------------------------------------------- exp
def test_exp_special_values():
    e = oracle.exp1
    assert e(0.0) == F(1.0) and ie.bits(e(-0.0)) == ie.bits(F(1.0))
    assert e(float("inf")) == F(np.inf)
    assert ie.bits(e(float("-inf"))) == 0
    assert np.isnan(e(float("nan")))
    assert e(89.0) == F(np.inf)
    assert e(88.72283172607422) < F(np.inf)          # largest finite input
    assert ie.bits(e(-104.5)) == 0
    # gradual underflow: results below FLT_MIN are nonzero subnormals
    for x in (-88.0, -95.0, -100.0, -103.0):
        y = e(x)
        assert 0 < y < F(np.finfo(F).tiny)
        # a subnormal result is within half a subnormal step of exp(x)
        assert abs(float(y) - math.exp(x)) <= 0.5 * 2.0 ** -149 + 2 * U * math.exp(x)


def test_exp_monotone_on_a_sweep():
    x = np.linspace(-103, 88.7, 2_000_001, dtype=F)
    y = oracle.exp(x)
    assert np.all(np.diff(y.astype(np.float64)) >= 0)


@pytest.mark.slow
def test_exp_accuracy_exhaustive():
    # every float in [-104, -0] and [+0, ln FLT_MAX): at most 1 ulp from the
    # exact value (the scan reports 0.94)
    neg, _ = oracle.ulp_scan("exp", 0x80000000, fbits(-104.0))
    pos, _ = oracle.ulp_scan("exp", 0x00000000, 0x42B17217)
    assert neg < 1.0 and pos < 1.0


# ----------------------------------------------------------------- log
def test_log_special_values():
    lg = oracle.log1
    assert ie.bits(lg(1.0)) == 0
    assert lg(0.0) == F(-np.inf) and lg(-0.0) == F(-np.inf)
    assert np.isnan(lg(-1.0)) and np.isnan(lg(float("nan")))
    assert lg(float("inf")) == F(np.inf)
    tiny = float(np.float32(2.0 ** -149))
    assert abs(float(lg(tiny)) - math.log(tiny)) <= float(np.spacing(F(103.3)))
    for k in range(-149, 128):
        y = float(lg(2.0 ** k))
        assert abs(y - k * math.log(2)) <= float(np.spacing(F(abs(k * math.log(2)) or 1e-30)))


def test_log_of_vocab_size():
    # the value a constant row's cross-entropy reduces to
    assert abs(float(oracle.log1(50257.0)) - math.log(50257)) <= float(np.spacing(F(10.8)))


@pytest.mark.slow
def test_log_accuracy_exhaustive():
    # every positive finite float, subnormals included (the scan reports 0.89)
    worst, _ = oracle.ulp_scan("log", 0x00000001, 0x7F7FFFFF)
    assert worst < 1.0


# ----------------------------------------------------------------- AdamW
HP = dict(lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def test_bias_correction_values():
    # step 1: 1 - beta exactly (Sterbenz: beta in [0.5, 1])
    b1, b2 = oracle.adamw_bias_correction(1, 0.9, 0.95)
    assert b1 == F(1) - F(0.9) and b2 == F(1) - F(0.95)
    # step 251: 0.9^251 = 3.3e-12 vanishes against 1; 0.95^251 = 2.6e-6
    b1, b2 = oracle.adamw_bias_correction(251, 0.9, 0.95)
    assert b1 == F(1.0)
    ref = 1.0 - float(F(0.95)) ** 251
    # 250 roundings of the power, relative 250 u on 2.6e-6, then one rounding
    assert abs(float(b2) - ref) <= 250 * U * 2.6e-6 + float(np.spacing(F(ref)))


def test_adamw_zero_gradient_is_pure_decay():
    rng = np.random.default_rng(41)
    p = (0.02 * rng.standard_normal(1000)).astype(F)
    z = np.zeros(1000, F)
    p2, m2, v2 = oracle.adamw(p, z, z, z, step=251, **HP)
    assert np.all(m2 == 0) and np.all(v2 == 0)
    decay = 1.0 - 6e-4 * 0.1
    assert np.all(np.abs(p2 - p.astype(np.float64) * decay)
                  <= 2 * np.spacing(np.abs(p2)) + 1e-45)


def test_adamw_first_step_is_sign_step():
    # step 1 from zero moments: m_hat = g, v_hat = g^2, u = g/(|g| + eps)
    rng = np.random.default_rng(42)
    g = rng.choice([-1, 1], size=1000).astype(F) * F(1e-2)
    p = np.zeros(1000, F)
    z = np.zeros(1000, F)
    p2, _, _ = oracle.adamw(p, g, z, z, step=1, **HP)
    assert np.allclose(p2, -6e-4 * np.sign(g), rtol=1e-5, atol=0)


def test_adamw_double_bound():
    rng = np.random.default_rng(43)
    n = 20000
    p = (0.02 * rng.standard_normal(n)).astype(F)
    g = (1e-3 * rng.standard_normal(n)).astype(F)
    m = (1e-3 * rng.standard_normal(n)).astype(F)
    v = ((1e-3 * rng.standard_normal(n)) ** 2).astype(F)
    p2, m2, v2 = oracle.adamw(p, g, m, v, step=251, **HP)
    d = lambda a: a.astype(np.float64)
    b1, b2 = float(F(0.9)), float(F(0.95))
    bc1 = 1 - b1 ** 251
    bc2 = 1 - b2 ** 251
    m64 = b1 * d(m) + (1 - b1) * d(g)
    v64 = b2 * d(v) + (1 - b2) * d(g) ** 2
    u64 = (m64 / bc1) / (np.sqrt(v64 / bc2) + float(F(1e-8)))
    lr = float(F(6e-4))
    p64 = d(p) * (1 - lr * float(F(0.1))) - lr * u64
    # m, v: two roundings each (and a tiny bias-correction difference);
    # u: ~8 roundings; p: two more
    assert np.all(np.abs(m2 - m64) <= 3 * U * (np.abs(d(m)) * b1 + np.abs(d(g)) * 0.1) + 1e-45)
    assert np.all(np.abs(v2 - v64) <= 4 * U * np.abs(v64) + 1e-45)
    assert np.all(np.abs(p2 - p64) <= 3 * U * np.abs(p64) + 12 * U * lr * np.abs(u64))


def test_adamw_exact_emulation_elementwise():
    # the written operation order, evaluated with exact rationals
    rng = np.random.default_rng(44)
    n = 64
    p = (0.02 * rng.standard_normal(n)).astype(F)
    g = (1e-3 * rng.standard_normal(n)).astype(F)
    m = (1e-3 * rng.standard_normal(n)).astype(F)
    v = ((1e-3 * rng.standard_normal(n)) ** 2).astype(F)
    p2, m2, v2 = oracle.adamw(p, g, m, v, step=7, **HP)
    lr, b1, b2, eps, wd = (F(HP[k]) for k in ("lr", "beta1", "beta2", "eps",
                                               "weight_decay"))
    pw1, pw2 = b1, b2
    for _ in range(6):
        pw1, pw2 = ie.mul(pw1, b1), ie.mul(pw2, b2)
    bc1, bc2 = ie.sub(F(1), pw1), ie.sub(F(1), pw2)
    omb1, omb2 = ie.sub(F(1), b1), ie.sub(F(1), b2)
    wdf = ie.sub(F(1), ie.mul(lr, wd))
    for i in range(n):
        mm = ie.fma(b1, m[i], ie.mul(omb1, g[i]))
        vv = ie.fma(b2, v[i], ie.mul(omb2, ie.mul(g[i], g[i])))
        u = ie.div(ie.div(mm, bc1), ie.add(ie.sqrt(ie.div(vv, bc2)), eps))
        pp = ie.fma(F(-lr), u, ie.mul(p[i], wdf))
        assert ie.same_bits(m2[i], mm) and ie.same_bits(v2[i], vv)
        assert ie.same_bits(p2[i], pp), i


def test_adamw_thread_invariance():
    rng = np.random.default_rng(45)
    n = 100003
    arrs = [(s * rng.standard_normal(n)).astype(F) for s in (0.02, 1e-3, 1e-3)]
    v = ((1e-3 * rng.standard_normal(n)) ** 2).astype(F)
    ref = oracle.adamw(arrs[0], arrs[1], arrs[2], v, step=251, nthreads=1, **HP)
    got = oracle.adamw(arrs[0], arrs[1], arrs[2], v, step=251, nthreads=6, **HP)
    for a, b in zip(got, ref):
        assert_bitwise(a, b)
