"""GPU parity (0 ULP) of a whole pre-norm decoder block's forward, composed
from the library's calls, against the same composition of oracle functions:
a small block in full, and one 162M-shaped block (4 x 2048 tokens, 768 wide,
12 heads, SwiGLU 2048) in full."""
import numpy as np
import pytest

import oracle
from bitcmp import assert_bitwise
from bitwise_reproducible_fp32_gb300 import block, inputs
from gpu_util import host, need_gpu, to_dev, torch

pytestmark = pytest.mark.gpu
F = np.float32


@pytest.fixture(scope="module")
def dev():
    return need_gpu()


def oracle_block(c, heads):
    x = c["x"]
    B, T = c["batch"], c["seq"]
    D = x.shape[1]
    hd = D // heads
    h, _ = oracle.rmsnorm(x, c["g1"], eps=1e-6)
    qkv = oracle.gemm(h, c["W_qkv"])
    qk = oracle.rope(qkv[:, :2 * D], 2 * heads, hd, seq_len=T)
    qkv = np.concatenate([qk, qkv[:, 2 * D:]], axis=1)
    att = np.empty((B * T, D), F)
    for b in range(B):
        r = slice(b * T, (b + 1) * T)
        for hh in range(heads):
            Q = qkv[r, hh * hd:(hh + 1) * hd]
            K = qkv[r, D + hh * hd:D + (hh + 1) * hd]
            V = qkv[r, 2 * D + hh * hd:2 * D + (hh + 1) * hd]
            P = oracle.softmax_causal(oracle.gemm(Q, K, transB=True),
                                      scale=float(F(1.0 / np.sqrt(hd))))
            att[r, hh * hd:(hh + 1) * hd] = oracle.gemm(P, V)
    x1 = oracle.add(x, oracle.gemm(att, c["W_o"]))
    h2, _ = oracle.rmsnorm(x1, c["g2"], eps=1e-6)
    s = oracle.swiglu(oracle.gemm(h2, c["W_gate"]), oracle.gemm(h2, c["W_up"]))
    return oracle.add(x1, oracle.gemm(s, c["W_down"]))


def run(c, heads, dff):
    x = c["x"]
    blk = block.Block(c["batch"], c["seq"], x.shape[1], dff, heads, torch.device("cuda"))
    w = {k: to_dev(c[k]) for k in ("g1", "W_qkv", "W_o", "g2", "W_gate", "W_up", "W_down")}
    return host(blk.forward(to_dev(x), w))


def test_small_block(dev):
    c = inputs.block_cfg(batch=2, seq=96, d=64, dff=96)
    assert_bitwise(run(c, 4, 96), oracle_block(c, 4))


def test_162m_block(dev):
    c = inputs.block_cfg()
    assert_bitwise(run(c, 12, 2048), oracle_block(c, 12))
