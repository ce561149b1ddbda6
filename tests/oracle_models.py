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


PARAMS = ("g1", "W_qkv", "W_o", "g2", "W_gate", "W_up", "W_down")


def block_with_activations(x, w, batch, seq, heads):
    """block(), keeping what the backward needs."""
    D = x.shape[1]
    hd = D // heads
    a = {}
    a["h"], a["inv1"] = oracle.rmsnorm(x, w["g1"], eps=1e-6)
    qkv = oracle.gemm(a["h"], w["W_qkv"])
    qk = oracle.rope(qkv[:, :2 * D], 2 * heads, hd, seq_len=seq)
    a["qkv"] = np.concatenate([qk, qkv[:, 2 * D:]], axis=1)
    att = np.empty((batch * seq, D), F)
    scale = float(F(1.0 / np.sqrt(hd)))
    for b in range(batch):
        r = slice(b * seq, (b + 1) * seq)
        for hh in range(heads):
            Q, K, V = (a["qkv"][r, o + hh * hd:o + (hh + 1) * hd] for o in (0, D, 2 * D))
            P = oracle.softmax_causal(oracle.gemm(Q, K, transB=True), scale=scale)
            att[r, hh * hd:(hh + 1) * hd] = oracle.gemm(P, V)
    a["att"] = att
    a["x1"] = oracle.add(x, oracle.gemm(att, w["W_o"]))
    a["h2"], a["inv2"] = oracle.rmsnorm(a["x1"], w["g2"], eps=1e-6)
    a["gate"] = oracle.gemm(a["h2"], w["W_gate"])
    a["up"] = oracle.gemm(a["h2"], w["W_up"])
    a["s"] = oracle.swiglu(a["gate"], a["up"])
    y = oracle.add(a["x1"], oracle.gemm(a["s"], w["W_down"]))
    return y, a


def block_backward(x, w, a, dy, batch, seq, heads):
    """The library's Block.backward, step for step, with oracle functions."""
    D = x.shape[1]
    hd = D // heads
    scale = float(F(1.0 / np.sqrt(hd)))
    g = {}
    ds = oracle.gemm(dy, w["W_down"], transB=True)
    g["W_down"] = oracle.gemm(a["s"], dy, transA=True)
    d_gate, d_up = oracle.swiglu_bwd(a["gate"], a["up"], ds)
    dh2 = oracle.gemm(d_gate, w["W_gate"], transB=True)
    dh2 = oracle.gemm_acc(dh2, d_up, w["W_up"], transB=True)
    g["W_gate"] = oracle.gemm(a["h2"], d_gate, transA=True)
    g["W_up"] = oracle.gemm(a["h2"], d_up, transA=True)
    dx1_b, g["g2"] = oracle.rmsnorm_bwd(a["x1"], w["g2"], a["inv2"], dh2)
    dx1 = oracle.add(dy, dx1_b)
    d_att = oracle.gemm(dx1, w["W_o"], transB=True)
    g["W_o"] = oracle.gemm(a["att"], dx1, transA=True)
    dqkv = np.empty_like(a["qkv"])
    for b in range(batch):
        r = slice(b * seq, (b + 1) * seq)
        for hh in range(heads):
            cols = [slice(o + hh * hd, o + (hh + 1) * hd) for o in (0, D, 2 * D)]
            Q, K, V = (a["qkv"][r, c] for c in cols)
            dO = d_att[r, hh * hd:(hh + 1) * hd]
            P = oracle.softmax_causal(oracle.gemm(Q, K, transB=True), scale=scale)
            dP = oracle.gemm(dO, V, transB=True)
            dqkv[r, cols[2]] = oracle.gemm(P, dO, transA=True)
            dS = oracle.softmax_causal_bwd(P, dP, scale=scale)
            dqkv[r, cols[0]] = oracle.gemm(dS, K)
            dqkv[r, cols[1]] = oracle.gemm(dS, Q, transA=True)
    dqk = oracle.rope_bwd(dqkv[:, :2 * D], 2 * heads, hd, seq_len=seq)
    dqkv = np.concatenate([dqk, dqkv[:, 2 * D:]], axis=1)
    dh = oracle.gemm(dqkv, w["W_qkv"], transB=True)
    g["W_qkv"] = oracle.gemm(a["h"], dqkv, transA=True)
    dx_b, g["g1"] = oracle.rmsnorm_bwd(x, w["g1"], a["inv1"], dh)
    return oracle.add(dx1, dx_b), g


def byte_lm_step(c, hp):
    """byte_lm.train_step with oracle functions: the same stage dict."""
    st = {}
    ntok = c["batch"] * c["seq"]
    x0 = c["emb"][c["tokens"]].astype(F)
    st["embedding"] = x0
    xs, acts = [x0], []
    for i, w in enumerate(c["blocks"]):
        y, a = block_with_activations(xs[-1], w, c["batch"], c["seq"], c["heads"])
        xs.append(y)
        acts.append(a)
        st[f"block{i}"] = y
    logits = oracle.gemm(xs[-1], c["head"], transB=True)
    st["logits"] = logits
    loss, dlogits, bad = oracle.xent(logits, c["labels"], with_dlogits=True,
                                     dscale=F(1.0 / ntok))
    assert bad == 0
    st["loss"], st["loss_mean"] = loss, np.array([oracle.mean(loss)], F)
    st["dlogits"] = dlogits
    grads = {"head": oracle.gemm(dlogits, xs[-1], transA=True)}
    dx = oracle.gemm(dlogits, c["head"])
    for i in reversed(range(len(c["blocks"]))):
        dx, g = block_backward(xs[i], c["blocks"][i], acts[i], dx, c["batch"], c["seq"],
                               c["heads"])
        for k in PARAMS:
            grads[f"block{i}.{k}"] = g[k]
        st[f"d_block{i}_input"] = dx
    grads["emb"] = oracle.embedding_bwd(c["tokens"], dx, c["vocab"])
    for k in sorted(grads):
        st[f"grad.{k}"] = grads[k]
    params = {"head": c["head"], "emb": c["emb"]}
    for i, w in enumerate(c["blocks"]):
        for k in PARAMS:
            params[f"block{i}.{k}"] = w[k]
    for k in sorted(params):
        z = np.zeros(params[k].size, F)
        p, m, v = oracle.adamw(params[k].ravel(), grads[k].ravel(), z, z.copy(), **hp)
        st[f"param.{k}"], st[f"m.{k}"], st[f"v.{k}"] = (t.reshape(params[k].shape)
                                                       for t in (p, m, v))
    return st
