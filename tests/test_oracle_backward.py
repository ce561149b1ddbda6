"""Pins for the oracle's backward operations of the byte-level LM step:
SwiGLU's backward, the causal softmax backward, the rotary backward and the
embedding backward.

Readings pinned here (the pages train the byte-level model's "embedding,
transformer forward and backward, cross entropy, and AdamW" bit-identically,
"mojolearn" PyPI page, section "Handing training off between vendors", and
print no spelling of any backward):
  * SwiGLU (R33): e = exp(-g), den = 1 + e, silu = g / den, sig = 1 / den;
    d_up = dh silu, d_gate = (dh u) (sig (1 + g (1 - sig)));
  * softmax (R34): dot = the 256-chain sum of fmaf(dP, P, .) over the kept
    columns, dS = (P (dP - dot)) scale, masked columns +0;
  * rotary (R35): the pair turns by -a: dx0 = dy0 c + dy1 s, dx1 = dy1 c - dy0 s;
  * embedding (R36): per id, its tokens' gradient rows added left to right in
    ascending token order; +0 for ids no token uses.
"""
import numpy as np

import ieee_exact as ie
import oracle
from bitcmp import assert_bitwise

F = np.float32
U = 2.0 ** -24


# ----------------------------------------------------------------- SwiGLU
def test_swiglu_bwd_exact_emulation():
    rng = np.random.default_rng(111)
    n = 300
    g = (3 * rng.standard_normal(n)).astype(F)
    g[:3] = [0.0, -0.0, 30.0]
    u = rng.standard_normal(n).astype(F)
    dh = rng.standard_normal(n).astype(F)
    dg, du = oracle.swiglu_bwd(g, u, dh)
    for i in range(n):
        den = ie.add(F(1.0), oracle.exp1(F(-g[i])))
        silu = ie.div(g[i], den)
        sig = ie.div(F(1.0), den)
        ds = ie.mul(sig, ie.add(F(1.0), ie.mul(g[i], ie.sub(F(1.0), sig))))
        assert ie.same_bits(du[i], ie.mul(dh[i], silu)), i
        assert ie.same_bits(dg[i], ie.mul(ie.mul(dh[i], u[i]), ds)), i


def test_swiglu_bwd_double_bound():
    rng = np.random.default_rng(112)
    g = (3 * rng.standard_normal(100000)).astype(F)
    u = rng.standard_normal(100000).astype(F)
    dh = rng.standard_normal(100000).astype(F)
    dg, du = oracle.swiglu_bwd(g, u, dh)
    g64, u64, d64 = (a.astype(np.float64) for a in (g, u, dh))
    sig = 1 / (1 + np.exp(-g64))
    assert np.all(np.abs(du - d64 * g64 * sig) <= 6 * U * np.abs(d64 * g64 * sig) + 1e-37)
    want = d64 * u64 * sig * (1 + g64 * (1 - sig))
    scale = np.abs(d64 * u64) * sig * (1 + np.abs(g64))
    assert np.all(np.abs(dg - want) <= 12 * U * scale + 1e-37)


# ----------------------------------------------------------------- softmax
def test_softmax_bwd_exact_emulation_and_masks():
    rng = np.random.default_rng(113)
    rows, cols = 5, 1100
    s = (3 * rng.standard_normal((rows, cols))).astype(F)
    p = oracle.softmax_causal(s, scale=0.125, diag=1000)
    dp = rng.standard_normal((rows, cols)).astype(F)
    ds = oracle.softmax_causal_bwd(p, dp, scale=0.125, diag=1000)
    for r in range(rows):
        n = min(cols, r + 1001)
        acc = [F(0.0)] * 256
        for j in range(n):
            l = (j // 4) % 256
            acc[l] = ie.fma(dp[r, j], p[r, j], acc[l])
        v = acc
        for off in (16, 8, 4, 2, 1, 32, 64, 128):
            v = [ie.add(v[l], v[l ^ off]) for l in range(256)]
        want = [ie.mul(ie.mul(p[r, j], ie.sub(dp[r, j], v[0])), F(0.125)) for j in range(n)]
        assert_bitwise(ds[r, :n], np.array(want, F), f"row {r}")
        assert np.all(ds[r, n:].view(np.uint32) == 0)


def test_softmax_bwd_double_bound_and_zero_sum():
    # the true gradient of a softmax row sums to zero (p is a probability
    # vector); a dropped dot term breaks it by O(1)
    rng = np.random.default_rng(114)
    s = (4 * rng.standard_normal((256, 256))).astype(F)
    p = oracle.softmax_causal(s, scale=0.125)
    dp = rng.standard_normal((256, 256)).astype(F)
    ds = oracle.softmax_causal_bwd(p, dp, scale=0.125)
    p64, dp64 = p.astype(np.float64), dp.astype(np.float64)
    mask = np.tril(np.ones((256, 256), bool))
    dot = (p64 * dp64 * mask).sum(axis=1, keepdims=True)
    want = 0.125 * p64 * (dp64 - dot) * mask
    scale = 0.125 * p64 * (np.abs(dp64) + np.abs(dp64 * p64).sum(axis=1, keepdims=True))
    assert np.all(np.abs(ds - want) <= 80 * U * scale + 1e-37)
    rowsum = ds.astype(np.float64).sum(axis=1)
    assert np.all(np.abs(rowsum) <= 1e-5 * np.abs(want).sum(axis=1) + 1e-30)


# ----------------------------------------------------------------- rotary
def test_rope_bwd_is_the_transpose():
    # <rope(x), y> = <x, rope_bwd(y)> for the same angles (a rotation's
    # transpose is its inverse); the wrong sign of the backward fails it
    rng = np.random.default_rng(115)
    heads, d, T = 3, 64, 300
    x = rng.standard_normal((T, heads * d)).astype(F)
    y = rng.standard_normal((T, heads * d)).astype(F)
    fx = oracle.rope(x, heads, d, seq_len=T).astype(np.float64)
    by = oracle.rope_bwd(y, heads, d, seq_len=T).astype(np.float64)
    lhs = (fx * y).sum(axis=1)
    rhs = (x.astype(np.float64) * by).sum(axis=1)
    mag = (np.abs(x) * np.abs(y)).astype(np.float64).sum(axis=1)
    assert np.all(np.abs(lhs - rhs) <= 16 * U * mag)
    back = oracle.rope_bwd(oracle.rope(x, heads, d, seq_len=T), heads, d, seq_len=T)
    assert np.all(np.abs(back - x) <= 8 * U * (np.abs(x) + 1e-30) + 4 * U * np.abs(x).max())
    # position 0 is untouched; a unit at 2i of position 7 goes to (c, -s)
    assert np.array_equal(oracle.rope_bwd(x, heads, d, seq_len=T)[0], x[0])
    e = np.zeros((T, heads * d), F)
    e[:, 10] = 1.0
    b = oracle.rope_bwd(e, heads, d, seq_len=T)
    f = oracle.rope(e, heads, d, seq_len=T)
    assert b[7, 10] == f[7, 10] and b[7, 11] == -f[7, 11]


# ----------------------------------------------------------------- embedding
def test_embedding_bwd_order_and_unused_ids():
    rng = np.random.default_rng(116)
    ntok, dim, vocab = 700, 9, 17
    tok = rng.integers(0, vocab - 2, size=ntok).astype(np.int32)   # ids 15, 16 unused
    dx = (rng.standard_normal((ntok, dim)) * np.exp2(rng.integers(-20, 20, (ntok, dim)))).astype(F)
    de = oracle.embedding_bwd(tok, dx, vocab)
    for v in range(vocab):
        idx = np.nonzero(tok == v)[0]
        for j in range(dim):
            if idx.size == 0:
                assert de[v, j].view(np.uint32) == 0
                continue
            t = dx[idx[0], j]
            for k in idx[1:]:
                t = ie.add(t, dx[k, j])
            assert ie.same_bits(de[v, j], t), (v, j)
    # order: 2^24 first, then ones (ties to even keep 2^24)
    tok2 = np.zeros(4, np.int32)
    dx2 = np.array([[2.0 ** 24], [1.0], [1.0], [1.0]], F)
    assert oracle.embedding_bwd(tok2, dx2, 1)[0, 0] == F(2.0 ** 24)
    assert oracle.embedding_bwd(tok2, dx2[::-1].copy(), 1)[0, 0] == F(2.0 ** 24 + 4)
