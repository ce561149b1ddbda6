"""GPU parity (0 ULP) of the backward operations against the oracle: SwiGLU's
backward, the causal softmax backward (square, batched by period, shifted
diagonals, in place), the rotary backward, the embedding backward (ids unused,
repeated, ragged widths), and the attention backward (small in full and at the
162M shape on sampled heads)."""
import numpy as np
import pytest

import oracle
from bitcmp import assert_bitwise
from bitwise_reproducible_fp32_gb300 import detlib
from gpu_util import host, need_gpu, to_dev, torch

pytestmark = pytest.mark.gpu
F = np.float32


@pytest.fixture(scope="module")
def dev():
    return need_gpu()


@pytest.mark.parametrize("n", [1, 7, 1000, (1 << 20) + 5])
def test_swiglu_bwd(dev, n):
    rng = np.random.default_rng(n)
    g = (3 * rng.standard_normal(n)).astype(F)
    u = rng.standard_normal(n).astype(F)
    dh = rng.standard_normal(n).astype(F)
    if n > 6:
        g[:6] = [0.0, -0.0, 100.0, -100.0, np.nan, 30.0]
    dg, du = detlib.detswiglu_bwd_f32(to_dev(g), to_dev(u), to_dev(dh))
    wg, wu = oracle.swiglu_bwd(g, u, dh)
    assert_bitwise(host(dg), wg, "d_gate")
    assert_bitwise(host(du), wu, "d_up")


@pytest.mark.parametrize("rows,cols,diag", [(1, 1, 0), (5, 5, 0), (300, 300, 0),
                                            (64, 2048, 1500), (257, 257, -3),
                                            (24, 2101, 2090)])
def test_softmax_bwd(dev, rows, cols, diag):
    rng = np.random.default_rng(rows + cols)
    s = (4 * rng.standard_normal((rows, cols))).astype(F)
    p = oracle.softmax_causal(s, scale=0.125, diag=diag)
    dp = rng.standard_normal((rows, cols)).astype(F)
    want = oracle.softmax_causal_bwd(p, dp, scale=0.125, diag=diag)
    got = detlib.detsoftmax_causal_bwd_f32(to_dev(p, "padded"), to_dev(dp, "padded"),
                                           scale=0.125, diag=diag)
    assert_bitwise(host(got), want)


def test_softmax_bwd_long_rows_offset_layout(dev):
    # past 1024 kept columns the backward reads P and dP again; unaligned rows
    rng = np.random.default_rng(202)
    s = (4 * rng.standard_normal((17, 1500))).astype(F)
    p = oracle.softmax_causal(s, scale=0.125, diag=1400)
    dp = rng.standard_normal((17, 1500)).astype(F)
    want = oracle.softmax_causal_bwd(p, dp, scale=0.125, diag=1400)
    got = detlib.detsoftmax_causal_bwd_f32(to_dev(p, "offset"), to_dev(dp, "offset"),
                                           scale=0.125, diag=1400)
    assert_bitwise(host(got), want)


def test_softmax_bwd_batched_in_place(dev):
    rng = np.random.default_rng(201)
    mats = [(3 * rng.standard_normal((130, 130))).astype(F) for _ in range(3)]
    ps = [oracle.softmax_causal(m, scale=0.25) for m in mats]
    dps = [rng.standard_normal((130, 130)).astype(F) for _ in range(3)]
    dpd = to_dev(np.concatenate(dps))
    detlib.detsoftmax_causal_bwd_f32(to_dev(np.concatenate(ps)), dpd, scale=0.25, period=130,
                                     ds=dpd)
    want = np.concatenate([oracle.softmax_causal_bwd(p, d, scale=0.25) for p, d in zip(ps, dps)])
    assert_bitwise(host(dpd), want)


def test_rope_bwd(dev):
    rng = np.random.default_rng(202)
    T, H, d = 600, 6, 64
    x = rng.standard_normal((T, 3 * H * d)).astype(F)
    xd = to_dev(x)
    detlib.detrope_bwd_f32(xd, heads=2 * H, head_dim=d, seq_len=300)
    got = host(xd)
    assert_bitwise(got[:, :2 * H * d], oracle.rope_bwd(x[:, :2 * H * d], 2 * H, d, seq_len=300))
    assert_bitwise(got[:, 2 * H * d:], x[:, 2 * H * d:])


@pytest.mark.parametrize("ntok,dim,vocab", [(1, 1, 1), (2048, 64, 256), (777, 9, 300),
                                            (5000, 33, 7),
                                            # one id for every token (full 256-token
                                            # lists), and columns beyond 1024 and 2048
                                            (600, 2100, 1), (300, 1030, 40)])
def test_embedding_bwd(dev, ntok, dim, vocab):
    rng = np.random.default_rng(ntok + dim)
    tok = rng.integers(0, max(vocab - 3, 1), size=ntok).astype(np.int32)
    dx = rng.standard_normal((ntok, dim)).astype(F)
    got = detlib.detembedding_bwd_f32(torch.from_numpy(tok).cuda(), to_dev(dx, "offset"), vocab)
    assert_bitwise(host(got), oracle.embedding_bwd(tok, dx, vocab))


def attention_bwd_oracle(qkv, dout, b, h, seq, heads, d, scale):
    hd = heads * d
    r = slice(b * seq, (b + 1) * seq)
    Q, K, V = (qkv[r, o + h * d:o + (h + 1) * d] for o in (0, hd, 2 * hd))
    dO = dout[r, h * d:(h + 1) * d]
    P = oracle.softmax_causal(oracle.gemm(Q, K, transB=True), scale=scale)
    dP = oracle.gemm(dO, V, transB=True)
    dV = oracle.gemm(P, dO, transA=True)
    dS = oracle.softmax_causal_bwd(P, dP, scale=scale)
    return oracle.gemm(dS, K), oracle.gemm(dS, Q, transA=True), dV


@pytest.mark.parametrize("B,T,H,d,checks,poison", [
    (2, 100, 3, 16, None, None), (4, 2048, 12, 64, [(0, 0), (3, 11)], None),
    # 3 chunks of k: dV, dQ and dK skip the +0 chunks of P and dS when dO, K and
    # Q are finite, and must take them all when one holds an inf or a NaN
    (1, 600, 2, 16, None, None), (1, 600, 2, 16, None, "dout"), (1, 600, 2, 16, None, "k"),
    (1, 600, 2, 16, None, "q"),
    # from 512 tokens the score products read Q and dO from transposed copies,
    # here with a ragged token count (the copies' row stride padded to 4)
    (3, 513, 2, 32, None, None)])
def test_attention_bwd(dev, B, T, H, d, checks, poison):
    rng = np.random.default_rng(T + H)
    qkv = rng.standard_normal((B * T, 3 * H * d)).astype(F)
    dout = rng.standard_normal((B * T, H * d)).astype(F)
    if poison == "dout":
        dout[500, 3] = np.inf
    elif poison == "k":
        qkv[520, H * d + 2] = np.nan
    elif poison == "q":
        qkv[10, 1] = -np.inf
    scale = 1.0 / np.sqrt(d)
    got = host(detlib.detattention_bwd_f32(to_dev(qkv), to_dev(dout), B, T, H, d))
    pairs = checks or [(b, h) for b in range(B) for h in range(H)]
    hd = H * d
    for b, h in pairs:
        dQ, dK, dV = attention_bwd_oracle(qkv, dout, b, h, T, H, d, float(F(scale)))
        r = slice(b * T, (b + 1) * T)
        assert_bitwise(got[r, h * d:(h + 1) * d], dQ, f"dQ b={b} h={h}")
        assert_bitwise(got[r, hd + h * d:hd + (h + 1) * d], dK, f"dK b={b} h={h}")
        assert_bitwise(got[r, 2 * hd + h * d:2 * hd + (h + 1) * d], dV, f"dV b={b} h={h}")


@pytest.mark.parametrize("B,T,H,d,poison", [
    (2, 100, 3, 16, None), (1, 600, 2, 16, None), (1, 600, 2, 16, "dout"),
    (1, 600, 2, 16, "v"), (1, 600, 2, 16, "k"), (3, 513, 2, 32, None),
    (4, 2048, 12, 64, None)])
def test_attention_bwd_with_the_forwards_p(dev, B, T, H, d, poison):
    # detattention_bwd_saved_f32 reads P from the forward's workspace instead
    # of recomputing it: the same bits as detattention_bwd_f32. A non-finite
    # dO makes dV take every chunk, so the rows' +0 columns past their chunk
    # (which the forward leaves unwritten when V is finite) are filled first;
    # a non-finite V makes the forward write them all
    rng = np.random.default_rng(T * 3 + H)
    qkv = rng.standard_normal((B * T, 3 * H * d)).astype(F)
    dout = rng.standard_normal((B * T, H * d)).astype(F)
    if poison == "dout":
        dout[500, 3] = np.inf
    elif poison == "v":
        qkv[300, 2 * H * d + 5] = np.inf
    elif poison == "k":
        qkv[520, H * d + 2] = np.nan
    qd, dod = to_dev(qkv), to_dev(dout)
    fws = torch.empty((detlib.detattention_workspace_bytes(B, T, H, d) + 3) // 4,
                      device="cuda").fill_(float("nan"))
    detlib.detattention_f32(qd, B, T, H, d, workspace=fws)
    got = host(detlib.detattention_bwd_saved_f32(qd, dod, B, T, H, d, fws))
    want = host(detlib.detattention_bwd_f32(qd, dod, B, T, H, d))
    assert_bitwise(got, want, "saved P against recomputed P")
    scale = 1.0 / np.sqrt(d)
    hd = H * d
    for b, h in ([(0, 0), (B - 1, H - 1)] if T >= 2048 else [(0, 0), (B - 1, H - 1), (0, H - 1)]):
        dQ, dK, dV = attention_bwd_oracle(qkv, dout, b, h, T, H, d, float(F(scale)))
        r = slice(b * T, (b + 1) * T)
        assert_bitwise(got[r, h * d:(h + 1) * d], dQ, f"dQ b={b} h={h}")
        assert_bitwise(got[r, hd + h * d:hd + (h + 1) * d], dK, f"dK b={b} h={h}")
        assert_bitwise(got[r, 2 * hd + h * d:2 * hd + (h + 1) * d], dV, f"dV b={b} h={h}")
    assert detlib.det_watchdog_status() == 0

