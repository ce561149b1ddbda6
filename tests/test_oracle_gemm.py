"""Pins for the oracle's fixed-order GEMM, each against something other than the
oracle itself: exact-rational IEEE emulation on tiny inputs, integer closed
forms, identity and permutation matrices, and hand-derived crafted cases.

Profile (the "mojolearn" PyPI page, section "What bitwise identity means, and
why it is not the default": reduction order, partitioning and FMA policy are
fixed): C[i,j] is, for each 256-wide k-chunk in ascending order, a sequential
fmaf chain from +0 in ascending k; the chunk partials are summed left to right,
the first taken as is.
"""
import numpy as np
import pytest

import ieee_exact as ie
import oracle
from bitcmp import assert_bitwise

F = np.float32


def emulate_gemm(A, B, K_CHUNK=256):
    """The profile's definition evaluated with exact rationals and hand
    rounding (tiny sizes only). A is M x K, B is K x N (logical operands)."""
    M, K = A.shape
    N = B.shape[1]
    C = np.empty((M, N), F)
    for i in range(M):
        for j in range(N):
            total = F(0.0)
            for c0 in range(0, K, K_CHUNK):
                acc = F(0.0)
                for k in range(c0, min(c0 + K_CHUNK, K)):
                    acc = ie.fma(A[i, k], B[k, j], acc)
                total = acc if c0 == 0 else ie.add(total, acc)
            C[i, j] = total
    return C


def wide_random(rng, shape):
    """Random floats over a wide exponent range, both signs, some exact zeros
    and subnormals, so rounding, cancellation and underflow all occur."""
    mant = rng.uniform(1.0, 2.0, size=shape)
    exps = rng.integers(-40, 40, size=shape)
    sign = rng.choice([-1.0, 1.0], size=shape)
    x = (sign * mant * np.exp2(exps)).astype(F)
    mask = rng.random(shape)
    x[mask < 0.03] = F(0.0)
    x[(mask >= 0.03) & (mask < 0.05)] = F(-0.0)
    x[(mask >= 0.05) & (mask < 0.07)] *= F(2.0 ** -100)   # into subnormal products
    return x


@pytest.mark.parametrize("K", [1, 2, 7, 255, 256, 257, 513, 600])
def test_exact_rational_brute_force(K):
    rng = np.random.default_rng(1000 + K)
    M, N = 2, 3
    A = wide_random(rng, (M, K))
    B = wide_random(rng, (K, N))
    assert_bitwise(oracle.gemm(A, B), emulate_gemm(A, B), f"K={K}")


def test_exact_rational_cancellation_heavy():
    # values from a tiny set so partial sums cancel exactly and hit zero often
    rng = np.random.default_rng(7)
    vals = np.array([1.0, -1.0, 0.5, -0.5, 3.0, -3.0, 0.0, -0.0], F)
    A = rng.choice(vals, size=(3, 300)).astype(F)
    B = rng.choice(vals, size=(300, 3)).astype(F)
    assert_bitwise(oracle.gemm(A, B), emulate_gemm(A, B))


def test_integer_closed_form():
    # integer-valued operands with every partial sum below 2^24 are exact, so
    # the profile's result equals the integer product; a dropped, repeated or
    # transposed term changes it
    rng = np.random.default_rng(11)
    M, N, K = 37, 29, 700
    Ai = rng.integers(-8, 9, size=(M, K))
    Bi = rng.integers(-8, 9, size=(K, N))
    C = oracle.gemm(Ai.astype(F), Bi.astype(F))
    np.testing.assert_array_equal(C.astype(np.int64), Ai @ Bi)


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_transposed_storage_same_result(transA, transB):
    rng = np.random.default_rng(12)
    M, N, K = 19, 23, 300
    Ai = rng.integers(-8, 9, size=(M, K))
    Bi = rng.integers(-8, 9, size=(K, N))
    A = Ai.astype(F)
    B = Bi.astype(F)
    As = np.ascontiguousarray(A.T) if transA else A
    Bs = np.ascontiguousarray(B.T) if transB else B
    C = oracle.gemm(As, Bs, transA=bool(transA), transB=bool(transB))
    np.testing.assert_array_equal(C.astype(np.int64), Ai @ Bi)
    # and on random data the four storages agree bit for bit
    Ar = np.random.default_rng(13).standard_normal((M, K)).astype(F)
    Br = np.random.default_rng(14).standard_normal((K, N)).astype(F)
    ref = oracle.gemm(Ar, Br)
    got = oracle.gemm(np.ascontiguousarray(Ar.T) if transA else Ar,
                      np.ascontiguousarray(Br.T) if transB else Br,
                      transA=bool(transA), transB=bool(transB))
    assert_bitwise(got, ref)


@pytest.mark.parametrize("K", [5, 256, 300, 700])
def test_identity_and_permutation(K):
    rng = np.random.default_rng(15)
    B = rng.standard_normal((K, 9)).astype(F)
    B[0, 0] = F(-0.0)
    C = oracle.gemm(np.eye(K, dtype=F), B)
    expect = B.copy()
    expect[expect == 0] = F(0.0)    # -0 entries become +0 (chains start at +0)
    assert_bitwise(C, expect)
    perm = rng.permutation(K)
    P = np.eye(K, dtype=F)[perm]
    assert_bitwise(oracle.gemm(P, B), expect[perm])


def test_chain_starts_at_plus_zero():
    # product -1 * 0 = -0; +0 + -0 = +0, so C = +0 (a chain seeded with the
    # first product, or with -0, would give -0)
    C = oracle.gemm(np.array([[-1.0]], F), np.array([[0.0]], F))
    assert ie.bits(C[0, 0]) == 0x00000000


def test_first_partial_taken_as_is():
    # the product -2^-100 * 2^-100 underflows to -0: P_0 = -0, and C = P_0 = -0
    # (0 + P_0 would give +0)
    C = oracle.gemm(np.array([[-2.0 ** -100]], F), np.array([[2.0 ** -100]], F))
    assert ie.bits(C[0, 0]) == 0x80000000


def test_chunk_width_256():
    # K = 512: products 2^24 then 255 ones in chunk 0, 256 ones in chunk 1.
    # Each 1 added to 2^24 is a tie and rounds back to 2^24, so P_0 = 2^24,
    # P_1 = 256 exactly and C = 2^24 + 256. One unchunked chain gives 2^24;
    # 128-wide chunks give 2^24 + 384.
    K = 512
    a = np.ones((1, K), F)
    a[0, 0] = F(4096.0)
    b = np.ones((K, 1), F)
    b[0, 0] = F(4096.0)
    C = oracle.gemm(a, b)
    assert C[0, 0] == F(2.0 ** 24 + 256)
    # the K-tail chunk is partial: K = 300 -> P_0 = 2^24, P_1 = 44
    C = oracle.gemm(a[:, :300].copy(), b[:300].copy())
    assert C[0, 0] == F(2.0 ** 24 + 44)


def test_chunks_summed_left_to_right():
    # partials P_0 = 2^24, P_1 = 1, P_2 = 1: left to right (2^24 + 1) + 1
    # rounds back to 2^24 twice; right to left would give 2^24 + 2
    K = 768
    a = np.zeros((1, K), F)
    b = np.zeros((K, 1), F)
    a[0, 0], b[0, 0] = 4096.0, 4096.0
    a[0, 256], b[256, 0] = 1.0, 1.0
    a[0, 512], b[512, 0] = 1.0, 1.0
    assert oracle.gemm(a, b)[0, 0] == F(2.0 ** 24)


def test_k_zero_is_plus_zero():
    C = oracle.gemm(np.zeros((3, 0), F), np.zeros((0, 4), F))
    assert C.shape == (3, 4)
    assert np.all(C.view(np.uint32) == 0)


def test_thread_count_invariance():
    rng = np.random.default_rng(16)
    A = rng.standard_normal((61, 517)).astype(F)
    B = rng.standard_normal((517, 45)).astype(F)
    ref = oracle.gemm(A, B, nthreads=1)
    for t in (2, 3, 8):
        assert_bitwise(oracle.gemm(A, B, nthreads=t), ref, f"threads={t}")


def test_close_to_double_product():
    # accuracy sanity: within the classical bound |dC| <= (chain + chunks)
    # u sum |a||b| (u = 2^-24) of the float64 product
    rng = np.random.default_rng(17)
    M, N, K = 40, 50, 1000
    A = rng.standard_normal((M, K)).astype(F)
    B = rng.standard_normal((K, N)).astype(F)
    C = oracle.gemm(A, B).astype(np.float64)
    ref = A.astype(np.float64) @ B.astype(np.float64)
    absprod = np.abs(A.astype(np.float64)) @ np.abs(B.astype(np.float64))
    bound = (256 + 4 + 1) * 2.0 ** -24 * absprod
    assert np.all(np.abs(C - ref) <= bound)
