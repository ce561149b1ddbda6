"""Seeded synthetic inputs for the four operations, shared by the library's
benchmark and the tests (the only code both sides share).

This module draws random numbers and nothing else: it holds none of the
method's arithmetic. Every tensor is float32 (labels int32), drawn from NumPy's
``default_rng(seed)`` (PCG64), the generator the "mojolearn" PyPI page uses in
its quick start and the "MojoLearn 162M" model card names for initialisation
(table "Training": ``default_rng(93261)``, N(0, 0.02), norm weights
1 + N(0, 0.02)). Shapes follow the model card's table "Compared with GPT-3
Small" (12 x 768, SwiGLU 2,048 wide, 50,257-id vocabulary, context 2,048,
162,147,840 parameters) and the five workload configurations of this library.

Draw order inside one seed is fixed and documented per function, so the same
seed always yields the same bytes on every host.
"""
from __future__ import annotations

import numpy as np

D_MODEL = 768
D_FF = 2048
VOCAB = 50257
TOKENS = 8192            # 4 sequences x 2,048 tokens
N_PARAMS = 162_147_840   # the 162M decoder's parameter count

SEED_CFG1, SEED_CFG2, SEED_CFG3, SEED_CFG4, SEED_CFG5 = 0, 1, 2, 3, 4
SEED_RMS_BWD = 5   # the backward row-op inputs (their own stream)
SEED_SHARDS = 6    # shard gradients for the fixed-order shard sum
N_SHARDS = 64      # the 162M model card's logical shards a step
SEED_BLOCK = 7     # one decoder block's input and weights
N_HEADS = 12


def uniform_pm1(rng: np.random.Generator, shape) -> np.ndarray:
    """Uniform on [-1, 1) in float32 (exact: a 24-bit grid scaled by 2, minus 1)."""
    return rng.random(shape, dtype=np.float32) * np.float32(2) - np.float32(1)


def normal(rng: np.random.Generator, shape, std: float = 1.0) -> np.ndarray:
    z = rng.standard_normal(shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    return z


# ------------------------------------------------------------------ GEMM
def gemm_cfg1(seed: int = SEED_CFG1, n: int = 256):
    """Fixed-order GEMM C = A B, M = N = K = 256, A and B uniform [-1, 1).
    Draw order: A, then B."""
    rng = np.random.default_rng(seed)
    A = uniform_pm1(rng, (n, n))
    B = uniform_pm1(rng, (n, n))
    return [dict(name="gemm256", A=A, B=B, transA=False, transB=False)]


def gemm_cfg2(seed: int = SEED_CFG2, tokens: int = 2048, d: int = 64,
              hidden: int = 172, vocab: int = 256):
    """Small byte-level LM step GEMMs: activations N(0, 1), weights N(0, 0.02).
    Weights are K x N (row-major) except the logits head, stored
    [vocab, d] = [out, in] and applied transposed.
    Draw order: X, W_qkv, W_o, W_gate, W_up, H, W_down, W_head."""
    rng = np.random.default_rng(seed)
    X = normal(rng, (tokens, d))
    W_qkv = normal(rng, (d, 3 * d), 0.02)
    W_o = normal(rng, (d, d), 0.02)
    W_gate = normal(rng, (d, hidden), 0.02)
    W_up = normal(rng, (d, hidden), 0.02)
    H = normal(rng, (tokens, hidden))
    W_down = normal(rng, (hidden, d), 0.02)
    W_head = normal(rng, (vocab, d), 0.02)
    return [
        dict(name="qkv", A=X, B=W_qkv, transA=False, transB=False),
        dict(name="attn_out", A=X, B=W_o, transA=False, transB=False),
        dict(name="swiglu_gate", A=X, B=W_gate, transA=False, transB=False),
        dict(name="swiglu_up", A=X, B=W_up, transA=False, transB=False),
        dict(name="swiglu_down", A=H, B=W_down, transA=False, transB=False),
        dict(name="logits", A=X, B=W_head, transA=False, transB=True),
    ]


def gemm_cfg3(seed: int = SEED_CFG3, tokens: int = TOKENS, d: int = D_MODEL,
              dff: int = D_FF, vocab: int = VOCAB):
    """162M-decoder forward GEMMs. X tokens x 768 and H tokens x 2048 are N(0, 1);
    weights N(0, 0.02), K x N row-major, except the LM head stored
    [50257, 768] = [out, in] (the model card's Linear layout) and applied
    transposed. Draw order: X, H, W_qkv, W_o, W_gate, W_up, W_down, W_head."""
    rng = np.random.default_rng(seed)
    X = normal(rng, (tokens, d))
    H = normal(rng, (tokens, dff))
    W_qkv = normal(rng, (d, 3 * d), 0.02)
    W_o = normal(rng, (d, d), 0.02)
    W_gate = normal(rng, (d, dff), 0.02)
    W_up = normal(rng, (d, dff), 0.02)
    W_down = normal(rng, (dff, d), 0.02)
    W_head = normal(rng, (vocab, d), 0.02)
    return [
        dict(name="qkv", A=X, B=W_qkv, transA=False, transB=False),
        dict(name="attn_out", A=X, B=W_o, transA=False, transB=False),
        dict(name="swiglu_gate", A=X, B=W_gate, transA=False, transB=False),
        dict(name="swiglu_up", A=X, B=W_up, transA=False, transB=False),
        dict(name="swiglu_down", A=H, B=W_down, transA=False, transB=False),
        dict(name="lm_head", A=X, B=W_head, transA=False, transB=True),
    ]


# ------------------------------------------------------------------ row ops
def rowops_cfg4(seed: int = SEED_CFG4, rows: int = TOKENS, d: int = D_MODEL,
                vocab: int = VOCAB, logit_std: float = 2.0):
    """RMSNorm input x rows x 768 ~ N(0, 1), gain 1 + N(0, 0.02), eps 1e-6;
    cross-entropy logits rows x 50257 ~ N(0, 2) (std 2), labels uniform int in
    [0, vocab). Draw order: x, gain noise, logits, labels."""
    rng = np.random.default_rng(seed)
    x = normal(rng, (rows, d))
    gain = np.float32(1) + normal(rng, (d,), 0.02)
    logits = normal(rng, (rows, vocab), logit_std)
    labels = rng.integers(0, vocab, size=rows, dtype=np.int32)
    return dict(x=x, gain=gain, eps=np.float32(1e-6), logits=logits,
                labels=labels)


def rmsnorm_cfg4(seed: int = SEED_CFG4, rows: int = TOKENS, d: int = D_MODEL):
    """The RMSNorm part of rowops_cfg4 alone (the same x and gain: the first
    two draws of the same stream), without the 1.6 GB of logits."""
    rng = np.random.default_rng(seed)
    x = normal(rng, (rows, d))
    gain = np.float32(1) + normal(rng, (d,), 0.02)
    return dict(x=x, gain=gain, eps=np.float32(1e-6))


# ------------------------------------------------------------------ backward
def rmsnorm_bwd_cfg4(seed: int = SEED_RMS_BWD, rows: int = TOKENS, d: int = D_MODEL):
    """RMSNorm backward at the cfg4 RMSNorm shape: x and gain of rmsnorm_cfg4,
    and the upstream gradient dy rows x 768 ~ N(0, 1e-3) from its own stream
    (the scale of the weight-gradient configuration's dY)."""
    f = rmsnorm_cfg4(rows=rows, d=d)
    rng = np.random.default_rng(seed)
    f["dy"] = normal(rng, (rows, d), 1e-3)
    return f


def dw_cfg5(seed: int = SEED_CFG5, tokens: int = TOKENS, d: int = D_MODEL,
            dff: int = D_FF):
    """Weight-gradient GEMMs dW = X^T dY contracting over the tokens:
    X N(0, 1), dY N(0, 1e-3). Draw order: X1 (tokens x 768),
    dY1 (tokens x 2304), X2 (tokens x 2048), dY2 (tokens x 768)."""
    rng = np.random.default_rng(seed)
    X1 = normal(rng, (tokens, d))
    dY1 = normal(rng, (tokens, 3 * d), 1e-3)
    X2 = normal(rng, (tokens, dff))
    dY2 = normal(rng, (tokens, d), 1e-3)
    return [
        dict(name="dW_qkv", A=X1, B=dY1, transA=True, transB=False),
        dict(name="dW_down", A=X2, B=dY2, transA=True, transB=False),
    ]


def shard_grads(seed: int = SEED_SHARDS, nshards: int = N_SHARDS,
                n: int = D_MODEL * 3 * D_MODEL):
    """nshards gathered shard gradients of one weight (default: the 768 x 2304
    QKV weight), each N(0, 1e-3) -- the scale of dY here, standing in for a
    per-shard mean gradient. One draw: an nshards x n array."""
    rng = np.random.default_rng(seed)
    return normal(rng, (nshards, n), 1e-3)


def block_cfg(seed: int = SEED_BLOCK, batch: int = 4, seq: int = 2048, d: int = D_MODEL,
              dff: int = D_FF):
    """One pre-norm decoder block at the 162M shape: x (batch*seq) x d ~ N(0, 1);
    gains 1 + N(0, 0.02); W_qkv d x 3d, W_o d x d, W_gate and W_up d x dff,
    W_down dff x d ~ N(0, 0.02) (the model card's initialisation), K x N
    row-major. Draw order: x, g1, W_qkv, W_o, g2, W_gate, W_up, W_down."""
    rng = np.random.default_rng(seed)
    x = normal(rng, (batch * seq, d))
    g1 = np.float32(1) + normal(rng, (d,), 0.02)
    W_qkv = normal(rng, (d, 3 * d), 0.02)
    W_o = normal(rng, (d, d), 0.02)
    g2 = np.float32(1) + normal(rng, (d,), 0.02)
    W_gate = normal(rng, (d, dff), 0.02)
    W_up = normal(rng, (d, dff), 0.02)
    W_down = normal(rng, (dff, d), 0.02)
    return dict(x=x, g1=g1, W_qkv=W_qkv, W_o=W_o, g2=g2, W_gate=W_gate, W_up=W_up,
                W_down=W_down, batch=batch, seq=seq)


def byte_lm_cfg2(seed: int = SEED_CFG2 + 100, batch: int = 16, seq: int = 128, d: int = 64,
                 dff: int = 172, vocab: int = 256, blocks: int = 2, heads: int = 4):
    """The small byte-level language model at the byte-LM GEMM shapes (16 x 128
    tokens, 64 wide, SwiGLU 172, 256 byte ids, two blocks): byte tokens uniform in
    [0, 256) for 129 positions a sequence (inputs: the first 128, labels: the
    last 128); embedding and LM head (the head stored [vocab, d]) N(0, 0.02);
    per block g1, W_qkv, W_o, g2, W_gate, W_up, W_down as block_cfg draws them.
    Draw order: tokens, embedding, each block's weights, the head."""
    rng = np.random.default_rng(seed)
    toks = rng.integers(0, vocab, size=(batch, seq + 1), dtype=np.int32)
    emb = normal(rng, (vocab, d), 0.02)
    blks = []
    for _ in range(blocks):
        g1 = np.float32(1) + normal(rng, (d,), 0.02)
        W_qkv = normal(rng, (d, 3 * d), 0.02)
        W_o = normal(rng, (d, d), 0.02)
        g2 = np.float32(1) + normal(rng, (d,), 0.02)
        W_gate = normal(rng, (d, dff), 0.02)
        W_up = normal(rng, (d, dff), 0.02)
        W_down = normal(rng, (dff, d), 0.02)
        blks.append(dict(g1=g1, W_qkv=W_qkv, W_o=W_o, g2=g2, W_gate=W_gate, W_up=W_up,
                         W_down=W_down))
    head = normal(rng, (vocab, d), 0.02)
    return dict(tokens=np.ascontiguousarray(toks[:, :seq]).reshape(-1),
                labels=np.ascontiguousarray(toks[:, 1:]).reshape(-1), emb=emb, blocks=blks,
                head=head, batch=batch, seq=seq, d=d, dff=dff, vocab=vocab, heads=heads)


def decoder_162m(layers: int = 12, batch: int = 4, seq: int = 2048, seed: int = 9):
    """The 162M decoder ("MojoLearn 162M" model card, table "Compared with GPT-3
    Small": 12 layers, 768 wide, 12 heads of 64, SwiGLU 2,048, context 2,048,
    RMSNorm pre-norm with no final norm, untied 50,257-id embeddings,
    162,147,840 parameters), drawn as byte_lm_cfg2 draws its model: token ids
    uniform in [0, 50257) for seq + 1 positions a sequence, weights N(0, 0.02),
    gains 1 + N(0, 0.02). `layers` and the token count can be cut for tests."""
    return byte_lm_cfg2(seed=seed, batch=batch, seq=seq, d=D_MODEL, dff=D_FF, vocab=VOCAB,
                        blocks=layers, heads=N_HEADS)


# the byte-level LM step's update: the 162M card's AdamW at the first step
BYTE_LM_HP = dict(lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1)

ADAMW_HP = dict(lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1,
                step=251)


def adamw_cfg5(seed: int = SEED_CFG5 + 100, n: int = N_PARAMS):
    """AdamW state for n parameters: p ~ N(0, 0.02), g ~ N(0, 1e-3),
    m ~ N(0, 1e-3), v = (N(0, 1e-3))^2 (warm moments, as step 251 implies).
    Draw order: p, g, m, v-root. Hyperparameters: ADAMW_HP."""
    rng = np.random.default_rng(seed)
    p = normal(rng, (n,), 0.02)
    g = normal(rng, (n,), 1e-3)
    m = normal(rng, (n,), 1e-3)
    v = normal(rng, (n,), 1e-3)
    np.multiply(v, v, out=v)
    return dict(p=p, g=g, m=m, v=v, **ADAMW_HP)


def flops_gemm(M: int, N: int, K: int) -> int:
    return 2 * M * N * K
