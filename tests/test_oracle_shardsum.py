"""Pins for the oracle's fixed-order shard gradient sum and its beta = 1
(accumulating) GEMM.

Readings pinned here. The "MojoLearn 162M" model card, table "Training", sums
the 64 logical shard gradients (each a mean over 4 x 2,048 tokens) "in a fixed
order" and prints no order; the plainest is left to right over the shard
index, one rounding per addition, then one multiply by the caller's scale
(1/64 for the mean of 64 shards, an exact power of two). Gradient
accumulation adds a new profile GEMM result R to the old C once, C on the
left, so accumulating the shards one after another gives the same bits as the
shard sum.
"""
import numpy as np

import ieee_exact as ie
import oracle
from bitcmp import assert_bitwise

F = np.float32
U = 2.0 ** -24


def test_left_to_right_pinned():
    # 2^24 first: every +1 is a tie that rounds back to 2^24 (even)
    assert oracle.shardsum(np.array([[2.0 ** 24], [1], [1], [1]], F))[0] == F(2.0 ** 24)
    # the ones first: (1 + 1) + 2^24 = 2^24 + 2 exactly
    assert oracle.shardsum(np.array([[1], [1], [2.0 ** 24]], F))[0] == F(2.0 ** 24 + 2)
    # a pairwise tree would give (2^24 + 1) + (1 + 1) = 2^24 + 2 for the
    # first column; with the scale: one exact multiply after the sum
    assert oracle.shardsum(np.array([[2.0 ** 24], [1], [1], [1]], F), scale=2.0 ** -6)[0] \
        == F(2.0 ** 18)


def test_exact_emulation():
    rng = np.random.default_rng(51)
    S, n = 7, 40
    g = (rng.standard_normal((S, n)) * np.exp2(rng.integers(-30, 30, (S, n)))).astype(F)
    g[2, 5] = F(-0.0)
    g[:, 6] = F(-0.0)            # all -0: the sum stays -0
    for scale in (1.0, 1.0 / 3.0, 2.0 ** -6):
        got = oracle.shardsum(g, scale=scale)
        want = np.empty(n, F)
        for i in range(n):
            t = g[0, i]
            for s in range(1, S):
                t = ie.add(t, g[s, i])
            want[i] = ie.mul(t, F(scale))
        assert_bitwise(got, want, f"scale {scale}")
    assert np.signbit(oracle.shardsum(g)[6])


def test_mean_of_64_shards_and_double_bound():
    rng = np.random.default_rng(52)
    g = (1e-3 * rng.standard_normal((64, 5000))).astype(F)
    total = oracle.shardsum(g)
    mean = oracle.shardsum(g, scale=1.0 / 64)
    assert_bitwise(mean, (total * F(2.0 ** -6)).astype(F), "1/64 is an exact scaling")
    exact = g.astype(np.float64).sum(axis=0)
    bound = 63 * U * np.abs(g.astype(np.float64)).sum(axis=0)
    assert np.all(np.abs(total - exact) <= bound)


def test_accumulating_gemm_is_the_shard_sum_of_gemms():
    # four token shards of a weight gradient X_s^T dY_s, 300 tokens each (two
    # 256-wide chunks): accumulating them with beta = 1 in shard order gives
    # the same bits as gathering the four products and summing them in order
    rng = np.random.default_rng(53)
    X = [rng.standard_normal((300, 24)).astype(F) for _ in range(4)]
    dY = [(1e-3 * rng.standard_normal((300, 40))).astype(F) for _ in range(4)]
    parts = np.stack([oracle.gemm(X[s], dY[s], transA=True) for s in range(4)])
    C = parts[0].copy()
    for s in range(1, 4):
        C = oracle.gemm_acc(C, X[s], dY[s], transA=True)
    assert_bitwise(C, oracle.shardsum(parts), "beta = 1 accumulation vs shard sum")


def test_accumulate_adds_once_with_c_on_the_left():
    rng = np.random.default_rng(54)
    A = rng.standard_normal((9, 600)).astype(F)
    B = rng.standard_normal((600, 7)).astype(F)
    C = rng.standard_normal((9, 7)).astype(F)
    R = oracle.gemm(A, B)
    got = oracle.gemm_acc(C, A, B)
    want = np.array([[ie.add(C[i, j], R[i, j]) for j in range(7)] for i in range(9)], F)
    assert_bitwise(got, want, "C + R, one rounding")
    # signs of zero: R = -0 (a tiny negative product underflows); +0 + -0 = +0
    a = np.array([[-(2.0 ** -100)]], F)
    b = np.array([[2.0 ** -100]], F)
    assert oracle.gemm(a, b).view(np.uint32)[0, 0] == 0x80000000
    assert oracle.gemm_acc(np.zeros((1, 1), F), a, b).view(np.uint32)[0, 0] == 0
    assert oracle.gemm_acc(np.full((1, 1), -0.0, F), a, b).view(np.uint32)[0, 0] == 0x80000000
