"""Pins for the oracle's RMSNorm backward against exact-rational emulation,
closed forms, crafted rows whose bits depend on the chain arrangement, the
profile's GEMM (the dgain contraction is its diagonal), the scale-invariance
identity of RMSNorm and a double-precision bound.

Readings pinned here (the pages fix the reduction order and partitioning of
the profile, "mojolearn" PyPI page, section "What bitwise identity means, and
why it is not the default", but print no backward spelling):
  * xhat = x * r, h = dy * g, with r the forward's inv_rms;
  * dot = sum of h * xhat by the forward's sum-of-squares arrangement (32
    chains of fmaf over 4-element groups, xor butterfly 16, 8, 4, 2, 1);
  * dx = (h - xhat * (dot / D)) * r;
  * dgain = the token contraction of dy * xhat in the GEMM's spelling (256-row
    chunks, fmaf chains from +0 in ascending row, partials added left to
    right).
"""
import numpy as np

import ieee_exact as ie
import oracle
from bitcmp import assert_bitwise

F = np.float32
U = 2.0 ** -24


def emulate(x, g, r, dy, k_chunk):
    """The whole backward with exact rationals and hand rounding."""
    rows, D = x.shape
    dx = np.empty((rows, D), F)
    for i in range(rows):
        lanes = [F(0.0)] * 32
        for j in range(D):
            xh = ie.mul(x[i, j], r[i])
            h = ie.mul(dy[i, j], g[j])
            lanes[(j // 4) % 32] = ie.fma(h, xh, lanes[(j // 4) % 32])
        v = lanes
        for off in (16, 8, 4, 2, 1):
            v = [ie.add(v[l], v[l ^ off]) for l in range(32)]
        q = ie.div(v[0], F(D))
        for j in range(D):
            xh = ie.mul(x[i, j], r[i])
            h = ie.mul(dy[i, j], g[j])
            dx[i, j] = ie.mul(ie.sub(h, ie.mul(xh, q)), r[i])
    dg = np.empty(D, F)
    for j in range(D):
        total = F(0.0)
        for c0 in range(0, rows, k_chunk):
            acc = F(0.0)
            for i in range(c0, min(c0 + k_chunk, rows)):
                acc = ie.fma(dy[i, j], ie.mul(x[i, j], r[i]), acc)
            total = acc if c0 == 0 else ie.add(total, acc)
        dg[j] = total
    return dx, dg


def test_exact_emulation_tiny():
    # 37 columns: every chain, a partial sweep and the butterfly; 5 rows with
    # 2-row chunks: three chunk partials, the last one short
    rng = np.random.default_rng(31)
    rows, D = 5, 37
    x = rng.standard_normal((rows, D)).astype(F)
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    _, r = oracle.rmsnorm(x, g)
    dy = rng.standard_normal((rows, D)).astype(F)
    dx, dg = oracle.rmsnorm_bwd(x, g, r, dy, k_chunk=2)
    dx_e, dg_e = emulate(x, g, r, dy, 2)
    assert_bitwise(dx, dx_e, "dx")
    assert_bitwise(dg, dg_e, "dgain")


def test_exact_emulation_subnormal_products():
    # tiny values: products and chain terms in the subnormal range, signed zeros
    rng = np.random.default_rng(32)
    rows, D = 3, 9
    x = (rng.standard_normal((rows, D)) * 2.0 ** -70).astype(F)
    x[0, 3] = F(-0.0)
    g = np.ones(D, F)
    r = np.array([2.0 ** 60, 2.0 ** 61, 1.0], F)
    dy = (rng.standard_normal((rows, D)) * 2.0 ** -60).astype(F)
    dy[1, 2] = F(-0.0)
    dx, dg = oracle.rmsnorm_bwd(x, g, r, dy, k_chunk=2)
    dx_e, dg_e = emulate(x, g, r, dy, 2)
    assert_bitwise(dx, dx_e, "dx")
    assert_bitwise(dg, dg_e, "dgain")


def test_dgain_is_the_gemm_diagonal():
    # dgain_j = (xhat^T dy)_jj under the profile's GEMM, xhat = x * r rounded
    rng = np.random.default_rng(33)
    rows, D = 700, 24          # three 256-row chunks, the last short
    x = rng.standard_normal((rows, D)).astype(F)
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    _, r = oracle.rmsnorm(x, g)
    dy = (1e-3 * rng.standard_normal((rows, D))).astype(F)
    _, dg = oracle.rmsnorm_bwd(x, g, r, dy)
    xhat = (x * r[:, None]).astype(F)          # float32 products, rounded once
    C = oracle.gemm(xhat, dy, transA=True)
    assert_bitwise(dg, np.ascontiguousarray(np.diagonal(C)), "dgain vs GEMM diagonal")


def test_zero_gradient_gives_positive_zeros():
    rng = np.random.default_rng(34)
    x = rng.standard_normal((300, 40)).astype(F)
    g = np.ones(40, F)
    _, r = oracle.rmsnorm(x, g)
    dx, dg = oracle.rmsnorm_bwd(x, g, r, np.zeros((300, 40), F))
    assert np.all(dx.view(np.uint32) == 0) and np.all(dg.view(np.uint32) == 0)


def test_unit_rows_closed_form():
    # x = 1, r = 1, g = 1, dy = 1: h = xhat = 1, dot = D, q = 1, dx = +0;
    # dgain = rows exactly (each 256-row chunk sums to 256)
    rows, D = 1000, 96
    x = np.ones((rows, D), F)
    dx, dg = oracle.rmsnorm_bwd(x, np.ones(D, F), np.ones(rows, F), np.ones((rows, D), F))
    assert np.all(dx.view(np.uint32) == 0)
    assert np.all(dg == F(rows))


def test_dot_chain_ownership_pinned():
    # r = 1, g = 1, dy = x, so h * xhat = x^2 and dot is the forward's ss of the
    # crafted row of the forward's ownership pin: 2^24 exactly (every +1 to
    # 2^24 is a tie that rounds back). Then q = 2^24 / 4096 = 4096 and
    # dx = x - 4096 x exactly: -16773120 at x = 4096, -4095 at x = 1.
    D = 4096
    x = np.zeros((1, D), F)
    for grp in range(0, D // 4, 32):
        x[0, 4 * grp: 4 * grp + 4] = 1.0
    x[0, 0] = 4096.0
    dx, _ = oracle.rmsnorm_bwd(x, np.ones(D, F), np.ones(1, F), x.copy())
    assert dx[0, 0] == F(4096.0 - 2.0 ** 24)
    assert dx[0, 1] == F(-4095.0) and dx[0, 128] == F(-4095.0)
    assert dx[0, 4].view(np.uint32) == 0


def test_dot_butterfly_pinned():
    # the forward's butterfly pin row: dot = 2^24 + 16 (the odd chains meet
    # chain 0 last), q = 4096 + 2^-8, and dx = x - x q exactly:
    # -(2^24 + 16 - 4096) at x = 4096, -(4095 + 2^-8) at x = 1. A left-to-right
    # fold of the chains gives dot = 2^24 and other bits.
    D = 4096
    x = np.zeros((1, D), F)
    x[0, 0] = 4096.0
    for lane in range(1, 32, 2):
        x[0, 4 * lane] = 1.0
    dx, _ = oracle.rmsnorm_bwd(x, np.ones(D, F), np.ones(1, F), x.copy())
    assert dx[0, 0] == F(-(2.0 ** 24 + 16 - 4096))
    assert dx[0, 4] == F(-(4095.0 + 2.0 ** -8))


def test_dgain_chunks_pinned():
    # one column, 512 rows, r = 1: dy * xhat = 2^24 at row 0 and 1 elsewhere.
    # Chunk 0 stays 2^24 (each +1 is a tie to even), chunk 1 sums to 256, so
    # dgain = 2^24 + 256; one chain over all rows would give 2^24.
    rows = 512
    x = np.ones((rows, 1), F)
    x[0, 0] = 4096.0
    _, dg = oracle.rmsnorm_bwd(x, np.ones(1, F), np.ones(rows, F), x.copy())
    assert dg[0] == F(2.0 ** 24 + 256)


def reference64(x, g, r, dy):
    x64, r64 = x.astype(np.float64), r.astype(np.float64)[:, None]
    h = dy.astype(np.float64) * g.astype(np.float64)
    xh = x64 * r64
    q = (h * xh).mean(axis=1, keepdims=True)
    return r64 * (h - xh * q), (dy.astype(np.float64) * xh).sum(axis=0), h, xh, q, r64


def test_double_bound():
    rng = np.random.default_rng(35)
    rows, D = 600, 768
    x = rng.standard_normal((rows, D)).astype(F)
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    _, r = oracle.rmsnorm(x, g)
    dy = (1e-3 * rng.standard_normal((rows, D))).astype(F)
    dx, dg = oracle.rmsnorm_bwd(x, g, r, dy)
    dx64, dg64, h, xh, q, r64 = reference64(x, g, r, dy)
    # dx: h, xhat, the D/32-long chains + 5 tree adds, the division, then
    # xhat q, the subtraction and the final product, on the scale of its terms
    scale = np.abs(r64 * h) + np.abs(r64 * xh) * np.abs(h * xh).mean(axis=1, keepdims=True)
    assert np.all(np.abs(dx - dx64) <= (D / 32 + 12) * U * scale + 1e-30)
    # dgain: 256-long chains, 2 chunk adds, the xhat product
    sc = (np.abs(dy.astype(np.float64)) * np.abs(xh)).sum(axis=0)
    assert np.all(np.abs(dg - dg64) <= (256 + 4) * U * sc)


def test_scale_invariance_identity():
    # With r the exact 1/rms (eps = 0), y(a x) = y(x), so x . dx = 0 in exact
    # arithmetic; a dropped term or a transposed factor breaks it by O(1).
    rng = np.random.default_rng(36)
    rows, D = 16, 512
    x = rng.standard_normal((rows, D)).astype(F)
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    _, r = oracle.rmsnorm(x, g, eps=0.0)
    dy = rng.standard_normal((rows, D)).astype(F)
    dx, _ = oracle.rmsnorm_bwd(x, g, r, dy)
    dot = (x.astype(np.float64) * dx).sum(axis=1)
    mag = (np.abs(x.astype(np.float64)) * np.abs(dx)).sum(axis=1)
    assert np.all(np.abs(dot) <= 1e-4 * mag)


def test_thread_invariance():
    rng = np.random.default_rng(37)
    x = rng.standard_normal((300, 130)).astype(F)
    g = np.ones(130, F)
    _, r = oracle.rmsnorm(x, g)
    dy = rng.standard_normal((300, 130)).astype(F)
    ref = oracle.rmsnorm_bwd(x, g, r, dy, nthreads=1)
    for t in (2, 5):
        got = oracle.rmsnorm_bwd(x, g, r, dy, nthreads=t)
        assert_bitwise(got[0], ref[0])
        assert_bitwise(got[1], ref[1])


def test_division_by_D_pinned():
    # q = dot / D, not dot * (1/D): for this row the two round apart
    # (dot = a^2 = 3.8043084, q = 1.2681028 vs 1.2681029) and so does dx_0
    a = np.array([1073326283], np.uint32).view(F)[0]
    x = np.array([[a, 0.0, 0.0]], F)
    dx, _ = oracle.rmsnorm_bwd(x, np.ones(3, F), np.ones(1, F), x.copy())
    t = ie.fma(a, a, F(0.0))
    q = ie.div(t, F(3.0))
    assert q != ie.mul(t, ie.div(F(1.0), F(3.0)))
    assert ie.same_bits(dx[0, 0], ie.sub(a, ie.mul(a, q)))
