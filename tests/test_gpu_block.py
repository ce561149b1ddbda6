"""GPU parity (0 ULP) of the block-forward operations against the oracle:
SwiGLU's gate, the residual add, the causal softmax (square, batched by
period, shifted diagonals, special values), rotary embedding on the packed QKV
layout, the sin/cos spellings over dense float ranges, and causal attention,
small in full and at the 162M shape on sampled heads."""
import math

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


def flat_dev(a, offset):
    """1-D device copy, optionally one float past a 16-byte boundary."""
    buf = torch.full((a.size + 4,), float("nan"), device="cuda")
    buf[offset:offset + a.size] = torch.from_numpy(np.ascontiguousarray(a).ravel()).cuda()
    return buf[offset:offset + a.size]


@pytest.mark.parametrize("n", [1, 5, 1000, 1 << 20, (1 << 20) + 3])
@pytest.mark.parametrize("offset", [0, 1])
def test_swiglu_and_add(dev, n, offset):
    rng = np.random.default_rng(n + offset)
    g = (3 * rng.standard_normal(n)).astype(F)
    u = rng.standard_normal(n).astype(F)
    if n > 8:
        g[:8] = [0.0, -0.0, 100.0, -100.0, 88.0, -88.0, np.nan, np.inf]
    assert_bitwise(host(detlib.detswiglu_f32(flat_dev(g, offset), flat_dev(u, offset))),
                   oracle.swiglu(g, u), f"swiglu n={n}")
    assert_bitwise(host(detlib.detadd_f32(flat_dev(g, offset), flat_dev(u, offset))),
                   oracle.add(g, u), f"add n={n}")


@pytest.mark.parametrize("rows,cols", [(1, 1), (5, 5), (300, 300), (1030, 1030), (64, 2048)])
@pytest.mark.parametrize("scale,diag", [(0.125, 0), (1.0 / 3.0, 7), (1.0, -2)])
def test_softmax_causal(dev, rows, cols, scale, diag):
    rng = np.random.default_rng(rows * 31 + cols)
    s = (4 * rng.standard_normal((rows, cols))).astype(F)
    want = oracle.softmax_causal(s, scale=scale, diag=diag)
    got = detlib.detsoftmax_causal_f32(to_dev(s, "padded"), scale=scale, diag=diag)
    assert_bitwise(host(got), want, f"{rows}x{cols} scale={scale} diag={diag}")


@pytest.mark.parametrize("rows,cols,diag,layout", [(20, 3001, 2990, "offset"),
                                                   (33, 2500, 2400, "padded"),
                                                   (9, 4099, 4000, "dense")])
def test_softmax_causal_long_rows(dev, rows, cols, diag, layout):
    # rows past 2048 kept columns: the kernel reads those segments again
    rng = np.random.default_rng(rows + cols)
    s = (4 * rng.standard_normal((rows, cols))).astype(F)
    want = oracle.softmax_causal(s, scale=0.125, diag=diag)
    got = detlib.detsoftmax_causal_f32(to_dev(s, layout), scale=0.125, diag=diag)
    assert_bitwise(host(got), want, f"{rows}x{cols} diag={diag} {layout}")


def test_softmax_batched_by_period_in_place_and_specials(dev):
    rng = np.random.default_rng(91)
    mats = [(4 * rng.standard_normal((257, 257))).astype(F) for _ in range(3)]
    mats[1][10, 3] = F(np.nan)          # NaN row
    mats[1][11, :] = F(-np.inf)         # all -inf: -inf - (-inf) = NaN
    mats[2][12, 5] = F(np.inf)          # +inf max: inf - inf = NaN
    mats[2][13, 0] = F(-np.inf)         # one -inf: exp(-inf) = 0
    stack = np.concatenate(mats)
    sd = to_dev(stack)
    detlib.detsoftmax_causal_f32(sd, scale=0.125, period=257, p=sd)       # in place
    want = np.concatenate([oracle.softmax_causal(m, scale=0.125) for m in mats])
    assert_bitwise(host(sd), want)


@pytest.mark.parametrize("diag", [0, -3, 5])
def test_softmax_bulk_staged_rows_cycle_both_buffers(dev, diag):
    # 16-byte aligned rows of at most 2048 columns (a multiple of 4) take the
    # bulk-staged kernel; 6 x 512 rows are more than its warps, so each warp
    # runs several rows through both of its buffers, in place, with special
    # rows among them and (diag < 0) rows that keep no column
    rng = np.random.default_rng(1000 + diag)
    mats = [(4 * rng.standard_normal((512, 512))).astype(F) for _ in range(6)]
    mats[1][10, 3] = F(np.nan)
    mats[1][11, :] = F(-np.inf)
    mats[2][12, 5] = F(np.inf)
    mats[2][13, 0] = F(-np.inf)
    mats[4][300, :200] = F(88.0)
    stack = np.concatenate(mats)
    sd = to_dev(stack)
    detlib.detsoftmax_causal_f32(sd, scale=0.125, diag=diag, period=512, p=sd)
    want = np.concatenate([oracle.softmax_causal(m, scale=0.125, diag=diag) for m in mats])
    assert_bitwise(host(sd), want, f"diag={diag}")
    assert detlib.det_watchdog_status() == 0


@pytest.mark.parametrize("diag", [0, -1])
def test_softmax_bulk_staged_odd_period(dev, diag):
    # an odd period; cols (a multiple of 4) wider than the period
    rng = np.random.default_rng(31 - diag)
    mats = [(4 * rng.standard_normal((257, 260))).astype(F) for _ in range(3)]
    got = detlib.detsoftmax_causal_f32(to_dev(np.concatenate(mats)), scale=0.125, diag=diag,
                                       period=257)
    want = np.concatenate([oracle.softmax_causal(m, scale=0.125, diag=diag) for m in mats])
    assert_bitwise(host(got), want, f"diag={diag}")


def test_softmax_bulk_staged_out_of_place_padded(dev):
    rng = np.random.default_rng(77)
    s = (4 * rng.standard_normal((4000, 2048))).astype(F)
    want = np.concatenate([oracle.softmax_causal(s[:2000], scale=0.125),
                           oracle.softmax_causal(s[2000:], scale=0.125)])
    got = detlib.detsoftmax_causal_f32(to_dev(s, "padded"), scale=0.125, period=2000)
    assert_bitwise(host(got), want)


def test_rope_on_the_packed_qkv_layout(dev):
    # 2 sequences of 300 tokens, 6 heads of 64: Q and K (12 heads) turned in
    # place inside rows of [Q | K | V]; V untouched
    rng = np.random.default_rng(92)
    T, H, d = 600, 6, 64
    qkv = rng.standard_normal((T, 3 * H * d)).astype(F)
    xd = to_dev(qkv)
    detlib.detrope_f32(xd, heads=2 * H, head_dim=d, seq_len=300)
    got = host(xd)
    want_qk = oracle.rope(qkv[:, :2 * H * d], 2 * H, d, seq_len=300)
    assert_bitwise(got[:, :2 * H * d], want_qk, "Q and K")
    assert_bitwise(got[:, 2 * H * d:], qkv[:, 2 * H * d:], "V")


def test_rope_full_162m_qk(dev):
    # 8192 tokens = 4 x 2048, Q and K = 24 heads of 64, row stride 2304
    rng = np.random.default_rng(93)
    qkv = rng.standard_normal((8192, 2304)).astype(F)
    xd = to_dev(qkv)
    detlib.detrope_f32(xd, heads=24, head_dim=64, seq_len=2048)
    got = host(xd)
    want = oracle.rope(qkv[:, :1536], 24, 64, seq_len=2048)
    assert_bitwise(got[:, :1536], want)


@pytest.mark.parametrize("lo,hi,step", [(0.0, math.pi / 4, 1), (0.5, 4096.0, 7),
                                         (-4096.0, -0.5, 7), (2.0 ** -30, 0.5, 3)])
def test_sin_cos_dense_ranges(dev, lo, hi, step):
    a, b = sorted((np.array([lo], F).view(np.uint32)[0], np.array([hi], F).view(np.uint32)[0]))
    bits = np.arange(a, b, step, dtype=np.uint64).astype(np.uint32)
    if bits.size > 40_000_000:
        bits = bits[:: bits.size // 40_000_000 + 1]
    x = bits.view(F)
    xd = torch.from_numpy(x.copy()).cuda()
    assert_bitwise(host(detlib.detsin_f32(xd)), oracle.sin(x), "sin")
    assert_bitwise(host(detlib.detcos_f32(xd)), oracle.cos(x), "cos")
    sp = np.array([0.0, -0.0, np.nan, np.inf, 2.0 ** 21, -(2.0 ** 20)], F)
    assert_bitwise(host(detlib.detsin_f32(to_dev(sp))), oracle.sin(sp), "sin specials")
    assert_bitwise(host(detlib.detcos_f32(to_dev(sp))), oracle.cos(sp), "cos specials")


def attention_oracle(qkv, b, h, seq, heads, d, scale):
    hd = heads * d
    rows = slice(b * seq, (b + 1) * seq)
    Q = qkv[rows, h * d:(h + 1) * d]
    K = qkv[rows, hd + h * d:hd + (h + 1) * d]
    V = qkv[rows, 2 * hd + h * d:2 * hd + (h + 1) * d]
    S = oracle.gemm(Q, K, transB=True)
    P = oracle.softmax_causal(S, scale=scale)
    return oracle.gemm(P, V)


def test_attention_small_in_full(dev):
    rng = np.random.default_rng(94)
    B, T, H, d = 2, 300, 3, 16
    qkv = rng.standard_normal((B * T, 3 * H * d)).astype(F)
    out = host(detlib.detattention_f32(to_dev(qkv), B, T, H, d, scale=0.25))
    for b in range(B):
        for h in range(H):
            want = attention_oracle(qkv, b, h, T, H, d, 0.25)
            assert_bitwise(out[b * T:(b + 1) * T, h * d:(h + 1) * d], want, f"b={b} h={h}")


@pytest.mark.parametrize("poison", [False, True])
def test_attention_chunks_above_the_diagonal(dev, poison):
    # 600 tokens: 3 chunks of k, so P.V skips the +0 chunks past each row
    # block when V is finite. With an inf and a NaN in V (0 * inf = NaN) every
    # chunk must be taken, as in the oracle.
    rng = np.random.default_rng(95)
    B, T, H, d = 2, 600, 2, 16
    hd = H * d
    qkv = rng.standard_normal((B * T, 3 * H * d)).astype(F)
    if poison:
        qkv[550, 2 * hd + 3] = np.inf              # sequence 0, head 0
        qkv[T + 300, 2 * hd + d + 5] = np.nan      # sequence 1, head 1
    out = host(detlib.detattention_f32(to_dev(qkv), B, T, H, d, scale=0.25))
    for b in range(B):
        for h in range(H):
            want = attention_oracle(qkv, b, h, T, H, d, 0.25)
            assert_bitwise(out[b * T:(b + 1) * T, h * d:(h + 1) * d], want,
                           f"b={b} h={h} poison={poison}")
    if poison:
        assert np.isnan(out[:550, 3]).all()           # 0 * inf reached every row before it


@pytest.mark.parametrize("B,T,H,d", [(2, 512, 2, 64), (1, 777, 3, 32), (2, 513, 2, 16)])
def test_attention_score_product_from_the_q_copy(dev, B, T, H, d):
    # From 512 tokens the score product reads Q from a transposed copy of the
    # Q block (the GEMM's row-pair loop) instead of Q itself: the same bits.
    # 777 and 513 tokens put the sequences at column offsets that TMA cannot
    # take (plain loads); head widths of 16 and 32 leave part of a k-tile past
    # the head's last column.
    rng = np.random.default_rng(96 + T)
    qkv = rng.standard_normal((B * T, 3 * H * d)).astype(F)
    out = host(detlib.detattention_f32(to_dev(qkv), B, T, H, d, scale=0.25))
    for b in range(B):
        for h in range(H):
            want = attention_oracle(qkv, b, h, T, H, d, 0.25)
            assert_bitwise(out[b * T:(b + 1) * T, h * d:(h + 1) * d], want, f"b={b} h={h}")


def test_attention_162m_shape_sampled_heads(dev):
    # 4 sequences of 2048 tokens, 12 heads of 64, scale 1/8: two heads checked
    rng = np.random.default_rng(95)
    B, T, H, d = 4, 2048, 12, 64
    qkv = rng.standard_normal((B * T, 3 * H * d)).astype(F)
    out = host(detlib.detattention_f32(to_dev(qkv), B, T, H, d))
    for b, h in ((0, 0), (3, 11)):
        want = attention_oracle(qkv, b, h, T, H, d, 0.125)
        assert_bitwise(out[b * T:(b + 1) * T, h * d:(h + 1) * d], want, f"b={b} h={h}")
