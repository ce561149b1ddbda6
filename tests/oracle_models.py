"""Compositions of oracle functions that mirror the library's block and the
byte-level LM forward stage by stage (test infrastructure: used by the GPU
parity tests and by the identity-card generator)."""
import numpy as np

import oracle

F = np.float32


def block(x, w, batch, seq, heads):
    """One pre-norm decoder block: RMSNorm, QKV, rotary on Q and K, causal
    attention (scale 1/sqrt(head_dim)), out projection, residual, RMSNorm,
    SwiGLU, down projection, residual."""
    D = x.shape[1]
    hd = D // heads
    h, _ = oracle.rmsnorm(x, w["g1"], eps=1e-6)
    qkv = oracle.gemm(h, w["W_qkv"])
    qk = oracle.rope(qkv[:, :2 * D], 2 * heads, hd, seq_len=seq)
    qkv = np.concatenate([qk, qkv[:, 2 * D:]], axis=1)
    att = np.empty((batch * seq, D), F)
    scale = float(F(1.0 / np.sqrt(hd)))
    for b in range(batch):
        r = slice(b * seq, (b + 1) * seq)
        for hh in range(heads):
            Q = qkv[r, hh * hd:(hh + 1) * hd]
            K = qkv[r, D + hh * hd:D + (hh + 1) * hd]
            V = qkv[r, 2 * D + hh * hd:2 * D + (hh + 1) * hd]
            P = oracle.softmax_causal(oracle.gemm(Q, K, transB=True), scale=scale)
            att[r, hh * hd:(hh + 1) * hd] = oracle.gemm(P, V)
    x1 = oracle.add(x, oracle.gemm(att, w["W_o"]))
    h2, _ = oracle.rmsnorm(x1, w["g2"], eps=1e-6)
    s = oracle.swiglu(oracle.gemm(h2, w["W_gate"]), oracle.gemm(h2, w["W_up"]))
    return oracle.add(x1, oracle.gemm(s, w["W_down"]))


def byte_lm_forward(c):
    """Stage outputs of the byte-level LM forward (inputs.byte_lm_cfg2)."""
    stages = {}
    x = c["emb"][c["tokens"]].astype(F)          # a gather: exact
    stages["embedding"] = x
    for i, w in enumerate(c["blocks"]):
        x = block(x, w, c["batch"], c["seq"], c["heads"])
        stages[f"block{i}"] = x
    logits = oracle.gemm(x, c["head"], transB=True)
    stages["logits"] = logits
    loss, _, bad = oracle.xent(logits, c["labels"])
    assert bad == 0
    stages["loss"] = loss
    stages["loss_mean"] = np.array([oracle.mean(loss)], F)
    return stages
