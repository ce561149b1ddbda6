"""Pins for the oracle's block operations: SwiGLU's gate, the residual add and
the causal softmax of attention scores.

Readings pinned here ("MojoLearn 162M" model card, table "Compared with GPT-3
Small": SwiGLU feed-forward, pre-norm residual blocks, causal attention; the
pages fix the profile's reduction order and exp spelling, "mojolearn" PyPI
page, section "What bitwise identity means, and why it is not the default",
but print no spelling of these operations):
  * silu(g) = g / (1 + exp(-g)) with the profile's exp, then times up;
  * the residual add is one rounded addition;
  * causal softmax: row r keeps columns j <= r + diag of s * scale; the
    cross-entropy's spelling: NaN-propagating max, e = exp(x - m), S the
    256-chain sum folded by the butterfly, p = e * (1 / S); masked columns +0.
"""
import math

import numpy as np

import ieee_exact as ie
import oracle
from bitcmp import assert_bitwise

F = np.float32
U = 2.0 ** -24


# ----------------------------------------------------------------- SwiGLU
def test_swiglu_exact_emulation():
    rng = np.random.default_rng(71)
    g = (rng.standard_normal(300) * np.exp2(rng.integers(-8, 7, 300))).astype(F)
    g[:6] = [0.0, -0.0, 100.0, -100.0, 88.0, -87.0]
    u = rng.standard_normal(300).astype(F)
    got = oracle.swiglu(g, u)
    want = np.empty(300, F)
    for i in range(300):
        ex = oracle.exp1(F(-g[i]))
        if np.isinf(ex):            # exp overflowed: g / inf is a zero of g's sign
            want[i] = F(np.copysign(0.0, g[i])) * u[i]
            continue
        den = ie.add(F(1.0), ex)
        want[i] = ie.mul(ie.div(g[i], den), u[i])
    assert_bitwise(got, want)


def test_swiglu_closed_forms():
    u = np.array([3.0, 3.0, 3.0, 3.0], F)
    got = oracle.swiglu(np.array([0.0, -0.0, 100.0, -100.0], F), u)
    assert got.view(np.uint32)[0] == 0                       # 0 / 2 * 3 = +0
    assert got.view(np.uint32)[1] == 0x80000000              # -0 / 2 * 3 = -0
    assert got[2] == F(300.0)                                # exp(-100) vanishes against 1
    assert got.view(np.uint32)[3] == 0x80000000              # -100 / inf = -0


def test_swiglu_double_bound():
    rng = np.random.default_rng(72)
    g = (3 * rng.standard_normal(100000)).astype(F)
    u = rng.standard_normal(100000).astype(F)
    got = oracle.swiglu(g, u).astype(np.float64)
    g64, u64 = g.astype(np.float64), u.astype(np.float64)
    want = g64 / (1.0 + np.exp(-g64)) * u64
    # exp within 1 ulp, then add, divide, multiply: a few ulps of the result
    assert np.all(np.abs(got - want) <= 6 * U * np.abs(want) + 1e-38)


def test_residual_add():
    rng = np.random.default_rng(73)
    a = rng.standard_normal(500).astype(F)
    b = rng.standard_normal(500).astype(F)
    b[0] = -a[0]
    got = oracle.add(a, b)
    assert_bitwise(got, np.array([ie.add(a[i], b[i]) for i in range(500)], F))
    assert got.view(np.uint32)[0] == 0                       # x + (-x) = +0


# ----------------------------------------------------------------- causal softmax
def emulate_softmax_row(s, scale, n, lanes=256, group=4):
    """One row, the first n columns kept, with exact rationals and hand rounding."""
    x = [ie.mul(F(s[j]), F(scale)) for j in range(n)]
    m = x[0]
    for j in range(1, n):
        if x[j] > m or x[j] != x[j]:
            m = x[j]
    e = [oracle.exp1(ie.sub(x[j], m)) for j in range(n)]
    acc = [F(0.0)] * lanes
    for j in range(n):
        l = (j // group) % lanes
        acc[l] = ie.add(acc[l], e[j])
    v = acc
    offs = [16, 8, 4, 2, 1] + [o for o in (32, 64, 128) if o < lanes]
    for off in offs:
        v = [ie.add(v[l], v[l ^ off]) for l in range(lanes)]
    inv = ie.div(F(1.0), v[0])
    return [ie.mul(e[j], inv) for j in range(n)]


def test_softmax_exact_emulation():
    rng = np.random.default_rng(74)
    rows, cols = 6, 1500          # more than one sweep of the 256 chains
    s = (4 * rng.standard_normal((rows, cols))).astype(F)
    for scale, diag in ((0.125, 0), (1.0 / 3.0, 1200)):
        got = oracle.softmax_causal(s, scale=scale, diag=diag)
        for r in range(rows):
            n = min(cols, r + diag + 1)
            want = emulate_softmax_row(s[r], scale, n)
            assert_bitwise(got[r, :n], np.array(want, F), f"row {r} scale {scale}")
            assert np.all(got[r, n:].view(np.uint32) == 0)


def test_softmax_closed_forms():
    # row 0 keeps one column: p = exp(0) / 1 = 1 exactly; constant rows give
    # fl(1 / n) everywhere (every e = 1, S = n exactly)
    s = np.full((300, 300), 2.5, F)
    p = oracle.softmax_causal(s, scale=0.125)
    assert p[0, 0] == F(1.0) and np.all(p[0, 1:].view(np.uint32) == 0)
    for r in (1, 2, 99, 255, 299):
        assert np.all(p[r, :r + 1] == F(1.0) / F(r + 1))
    # a row with no kept column is all +0
    q = oracle.softmax_causal(np.ones((3, 8), F), diag=-2)
    assert np.all(q[:2].view(np.uint32) == 0) and q[2, 0] == F(1.0)


def test_softmax_is_the_cross_entropy_spelling():
    # an unmasked row's probabilities are the cross-entropy's dlogits with
    # dscale 1 away from the label (e * (1/S) - 0)
    rng = np.random.default_rng(75)
    s = (2 * rng.standard_normal((1, 3000))).astype(F)
    p = oracle.softmax_causal(s, diag=3000)
    _, d, _ = oracle.xent(s, np.array([5], np.int32), with_dlogits=True, dscale=F(1.0))
    mask = np.arange(3000) != 5
    assert_bitwise(p[0, mask], d[0, mask])


def test_softmax_rows_sum_to_one():
    rng = np.random.default_rng(76)
    s = (8 * rng.standard_normal((512, 512))).astype(F)
    p = oracle.softmax_causal(s, scale=0.125).astype(np.float64)
    n = np.arange(1, 513)
    assert np.all(np.abs(p.sum(axis=1) - 1.0) <= (n + 10) * U)
