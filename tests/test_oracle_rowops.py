"""Pins for the oracle's RMSNorm, softmax cross-entropy and mean, against closed
forms, hand-derived crafted rows, double-precision bounds and an independent
restatement of the fixed reduction tree.

Profile readings pinned here (the "mojolearn" PyPI page, section "What bitwise
identity means, and why it is not the default", fixes the reduction order and
partitioning but prints none):
  * a row's sum is split over L chains; chain l owns the 4-element groups g of
    the row with g mod L == l and adds its elements in ascending index;
  * the L chain values are folded by an xor butterfly with offsets
    16, 8, 4, 2, 1, then 32, 64, ... (L = 32 for RMSNorm and the mean,
    L = 256 for the cross-entropy sum);
  * RMSNorm squares by fmaf; y = (x * r) * g with r = 1 / sqrt(ss / D + eps)
    ("MojoLearn 162M" model card, table "Compared with GPT-3 Small": RMSNorm,
    eps 1e-6);
  * cross-entropy: m = max, e = exp(x - m), loss = log(S) - (x_y - m),
    dlogits = (e / S - onehot) * dscale computed as e * (1/S).
"""
import math

import numpy as np
import pytest

import ieee_exact as ie
import oracle
from bitcmp import assert_bitwise

F = np.float32
U = 2.0 ** -24


# ----------------------------------------------------------------- RMSNorm
def test_rmsnorm_constant_row():
    # x = 1: every chain sums ones exactly, ss = D, ms = 1, r = 1/sqrt(1+eps)
    D = 768
    x = np.ones((3, D), F)
    g = np.ones(D, F)
    y, inv = oracle.rmsnorm(x, g, eps=1e-6)
    r64 = 1.0 / math.sqrt(1.0 + float(F(1e-6)))
    assert abs(float(inv[0]) - r64) <= 1.5 * float(np.spacing(F(r64)))
    assert np.all(inv == inv[0]) and np.all(y == inv[0])


def test_rmsnorm_chain_ownership_pinned():
    # D = 4096, 32 chains of 4-element groups: chain 0 owns j = 0..3,
    # 128..131, 256..259, ... With x_0 = 4096 (square 2^24) first and every
    # other element of chain 0 equal to 1, each +1 is a tie that rounds back to
    # 2^24, so ss = 2^24 exactly: ms = 4096, sqrt = 64, r = 1/64 exactly.
    # Contiguous per-chain blocks, or another order, give ss > 2^24.
    D = 4096
    x = np.zeros((1, D), F)
    for g in range(0, D // 4, 32):
        x[0, 4 * g: 4 * g + 4] = 1.0
    x[0, 0] = 4096.0
    y, inv = oracle.rmsnorm(x, np.ones(D, F), eps=1e-6)
    assert inv[0] == F(1.0 / 64.0)
    assert y[0, 0] == F(64.0) and y[0, 128] == F(1.0 / 64.0)


def test_rmsnorm_butterfly_pinned():
    # chain 0 holds 2^24 (x_0 = 4096); every odd chain l holds 1 (x_{4l} = 1).
    # Butterfly 16, 8, 4, 2, 1: the odd chains pair among themselves first
    # (1+1, 2+2, 4+4, 8+8 = 16, all exact) and meet chain 0 last:
    # ss = 2^24 + 16. A left-to-right sum of the chains loses each 1 to a tie
    # and gives 2^24. Then ms = 4096 + 2^-8, sqrt rounds to 64 + 2^-15 and
    # r = 2^-6 - 2^-27 (derivation: 1/(64(1 + 2^-21)) = 2^-6 (1 - 2^-21 + ...),
    # nearest binary32 2^-6 - 2^-27).
    D = 4096
    x = np.zeros((1, D), F)
    x[0, 0] = 4096.0
    for lane in range(1, 32, 2):
        x[0, 4 * lane] = 1.0
    _, inv = oracle.rmsnorm(x, np.ones(D, F), eps=1e-6)
    assert inv[0] == F(2.0 ** -6 - 2.0 ** -27)


@pytest.mark.parametrize("D,rows", [(37, 6), (3, 40), (5, 40), (7, 40)])
def test_rmsnorm_exact_emulation_tiny(D, rows):
    # the whole row computation with exact rationals and hand rounding; many
    # short rows, so that a one-ulp change anywhere in the row's chain of
    # operations (ss / D, the square root, 1 / sqrt) reaches inv_rms or y
    rng = np.random.default_rng(21 + D)
    x = rng.standard_normal((rows, D)).astype(F)
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    eps = F(1e-6)
    y, inv = oracle.rmsnorm(x, g, eps=eps)
    for i in range(rows):
        lanes = [F(0.0)] * 32
        for j in range(D):
            lanes[(j // 4) % 32] = ie.fma(x[i, j], x[i, j], lanes[(j // 4) % 32])
        v = lanes
        for off in (16, 8, 4, 2, 1):
            v = [ie.add(v[l], v[l ^ off]) for l in range(32)]
        ms = ie.div(v[0], F(D))
        r = ie.div(F(1.0), ie.sqrt(ie.add(ms, eps)))
        yexp = np.array([ie.mul(ie.mul(x[i, j], r), g[j]) for j in range(D)], F)
        assert ie.same_bits(inv[i], r), (D, i)
        assert_bitwise(y[i], yexp)


def test_rmsnorm_double_bound():
    rng = np.random.default_rng(22)
    rows, D = 64, 768
    x = rng.standard_normal((rows, D)).astype(F)
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    y, inv = oracle.rmsnorm(x, g, eps=1e-6)
    x64 = x.astype(np.float64)
    r64 = 1.0 / np.sqrt((x64 ** 2).mean(axis=1) + float(F(1e-6)))
    y64 = x64 * r64[:, None] * g.astype(np.float64)
    # error budget: chain of D/32 fmas + 5 tree adds on ss, div, add, sqrt,
    # div, two products
    rel = (D / 32 + 5 + 6) * U
    assert np.all(np.abs(inv - r64) <= rel * r64)
    assert np.all(np.abs(y - y64) <= rel * np.abs(y64) + 1e-30)


def test_rmsnorm_thread_invariance():
    rng = np.random.default_rng(23)
    x = rng.standard_normal((33, 500)).astype(F)
    g = np.ones(500, F)
    ref = oracle.rmsnorm(x, g, nthreads=1)
    for t in (2, 7):
        got = oracle.rmsnorm(x, g, nthreads=t)
        assert_bitwise(got[0], ref[0])
        assert_bitwise(got[1], ref[1])


# ----------------------------------------------------------------- mean
def test_mean_butterfly_pinned():
    # 32 chains, plain adds: chain 0 holds 2^24 then ties; odd chains hold 1.
    # ((odd chains pair up exactly to 16) + 2^24) = 2^24 + 16 over n = 128.
    n = 128
    x = np.zeros(n, F)
    x[0] = 2.0 ** 24
    for lane in range(1, 32, 2):
        x[4 * lane] = 1.0
    assert oracle.mean(x) == F((2.0 ** 24 + 16) / 128)


def test_mean_chain_order_pinned():
    # chain 0 owns i = 0..3, 128..131: 2^24 first, then ones lost to ties
    n = 256
    x = np.zeros(n, F)
    x[0] = 2.0 ** 24
    x[1:4] = 1.0
    x[128:132] = 1.0
    assert oracle.mean(x) == F(2.0 ** 24 / 256)


def test_mean_double_bound():
    x = np.random.default_rng(24).standard_normal(8192).astype(F) + F(10)
    assert abs(float(oracle.mean(x)) - x.astype(np.float64).mean()) <= 1e-5


# ----------------------------------------------------------------- xent
def fold_tree(v):
    """Independent restatement of the 256-chain tree: inside each 32-chain
    warp the butterfly 16, 8, 4, 2, 1 equals folding the upper half onto the
    lower half five times; across the 8 warp sums the levels 32, 64, 128 equal
    an adjacent-pairs tree ((w0+w1)+(w2+w3)) + ((w4+w5)+(w6+w7))."""
    v = np.asarray(v, F).reshape(8, 32)
    w = []
    for row in v:
        r = row
        while r.size > 1:
            h = r.size // 2
            r = (r[:h] + r[h:]).astype(F)     # numpy float32 add, RN
        w.append(r[0])
    w = np.array(w, F)
    while w.size > 1:
        w = (w[0::2] + w[1::2]).astype(F)
    return w[0]


def test_xent_tree_restated():
    # loss and dlogits of whole rows from the restated tree; dlogits carry S
    # through 1/S into every element, so a tree that sums in another shape
    # (other chains, another fold) shows there even where log S rounds alike
    rng = np.random.default_rng(31)
    V, rows = 3000, 6
    x = (2 * rng.standard_normal((rows, V))).astype(F)
    labels = rng.integers(0, V, rows).astype(np.int32)
    dscale = F(0.125)
    loss, d, bad = oracle.xent(x, labels, with_dlogits=True, dscale=dscale)
    assert bad == 0
    for r in range(rows):
        m = x[r].max()
        e = oracle.exp((x[r] - m).astype(F))
        lanes = np.zeros(256, F)
        for j in range(V):
            lanes[(j // 4) % 256] = F(lanes[(j // 4) % 256] + e[j])
        S = fold_tree(lanes)
        want = F(oracle.log1(S) - F(x[r, labels[r]] - m))
        assert ie.same_bits(loss[r], want)
        onehot = np.zeros(V, F)
        onehot[labels[r]] = 1.0
        dwant = ((e * (F(1.0) / S)).astype(F) - onehot).astype(F) * dscale
        assert_bitwise(d[r], dwant.astype(F))


def test_xent_constant_row():
    # all logits equal: every e_j = exp(0) = 1 exactly, S = V exactly,
    # loss = log(V); dlogits = (1/V - onehot) * dscale
    V = 50257
    x = np.full((2, V), 3.25, F)
    labels = np.array([0, 12345], np.int32)
    loss, d, bad = oracle.xent(x, labels, with_dlogits=True, dscale=F(0.5))
    assert bad == 0
    assert abs(float(loss[0]) - math.log(V)) <= 1.0 * float(np.spacing(F(math.log(V))))
    assert loss[0] == loss[1]
    inv = F(1) / F(V)
    assert d[0, 1] == F(inv * F(0.5))
    assert d[1, 12345] == F(F(inv - F(1)) * F(0.5))


def test_xent_double_bound_and_dlogits():
    rng = np.random.default_rng(32)
    rows, V = 16, 5000
    x = (2 * rng.standard_normal((rows, V))).astype(F)
    labels = rng.integers(0, V, size=rows, dtype=np.int32)
    loss, d, bad = oracle.xent(x, labels, with_dlogits=True,
                               dscale=F(1.0 / rows))
    assert bad == 0
    x64 = x.astype(np.float64)
    m = x64.max(axis=1, keepdims=True)
    lse = np.log(np.exp(x64 - m).sum(axis=1)) + m[:, 0]
    ref = lse - x64[np.arange(rows), labels]
    # S: V/256 sequential adds per chain + 8 tree levels, each exp <= 1 ulp;
    # log adds ~1 ulp; absolute error in loss ~ relative error of S
    tol = (V / 256 + 8 + 2) * U + 4 * U * np.abs(ref)
    assert np.all(np.abs(loss - ref) <= tol)
    p = np.exp(x64 - lse[:, None])
    onehot = np.zeros_like(p)
    onehot[np.arange(rows), labels] = 1
    dref = (p - onehot) / rows
    assert np.all(np.abs(d - dref) <= (V / 256 + 14) * U * (p + onehot) / rows + 1e-30)
    # softmax sums to one within the same budget
    assert np.all(np.abs(d.astype(np.float64).sum(axis=1)) <= 1e-5 / rows)


def test_xent_bad_label():
    x = np.zeros((3, 10), F)
    labels = np.array([0, 10, -1], np.int32)
    loss, d, bad = oracle.xent(x, labels, with_dlogits=True)
    assert bad == 2
    assert np.isfinite(loss[0]) and np.isnan(loss[1]) and np.isnan(loss[2])
    assert np.all(np.isnan(d[1])) and np.all(np.isfinite(d[0]))


def test_xent_max_sign_of_zero_inert():
    # the max is order-free: with +0 and -0 tied, x - m and x_y - m give the
    # same bits either way
    x = np.array([[0.0, -0.0, -1.0, -0.0]], F)
    x2 = np.array([[-0.0, 0.0, -1.0, 0.0]], F)
    for lab in range(4):
        l1, _, _ = oracle.xent(x, np.array([lab], np.int32))
        l2, _, _ = oracle.xent(x2, np.array([lab], np.int32))
        assert ie.same_bits(l1[0], l2[0])


def test_xent_thread_invariance():
    rng = np.random.default_rng(33)
    x = rng.standard_normal((37, 1111)).astype(F)
    lab = rng.integers(0, 1111, size=37, dtype=np.int32)
    ref = oracle.xent(x, lab, with_dlogits=True, nthreads=1)
    for t in (2, 5):
        got = oracle.xent(x, lab, with_dlogits=True, nthreads=t)
        assert_bitwise(got[0], ref[0])
        assert_bitwise(got[1], ref[1])
