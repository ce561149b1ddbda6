"""Pins the oracle's byte-level LM step composition (tests/oracle_models.py)
against an independent float64 model written with PyTorch's autograd on the
CPU: same weights, same structure (pre-norm RMSNorm, rotary pairs (2i, 2i+1),
causal softmax attention, SwiGLU, untied head, mean cross-entropy). The loss
and every gradient must agree to float32 accuracy; a transposed operand, a
missing residual or a wrong sign in any backward step would not."""
import numpy as np
import pytest

import oracle_models
from bitwise_reproducible_fp32_gb300 import inputs

torch = pytest.importorskip("torch")


def torch_model_grads(c):
    t = lambda a: torch.tensor(np.asarray(a, np.float64), requires_grad=True)  # noqa: E731
    emb, head = t(c["emb"]), t(c["head"])
    blocks = [{k: t(v) for k, v in w.items()} for w in c["blocks"]]
    B, T, H = c["batch"], c["seq"], c["heads"]
    D = c["emb"].shape[1]
    hd = D // H
    tok = torch.tensor(c["tokens"].astype(np.int64))
    lab = torch.tensor(c["labels"].astype(np.int64))
    pos = (torch.arange(B * T) % T).double()[:, None]
    w = 10000.0 ** (-(2 * torch.arange(hd // 2).double()) / hd)
    ang = pos * w[None, :]
    cos, sin = torch.cos(ang), torch.sin(ang)

    def rms(x, g):
        return x / torch.sqrt((x * x).mean(dim=1, keepdim=True) + 1e-6) * g

    def rope(x, nheads):
        x = x.view(B * T, nheads, hd // 2, 2)
        x0, x1 = x[..., 0], x[..., 1]
        c_, s_ = cos[:, None, :], sin[:, None, :]
        return torch.stack([x0 * c_ - x1 * s_, x0 * s_ + x1 * c_], dim=-1).view(B * T, -1)

    x = emb[tok]
    mask = torch.tril(torch.ones(T, T, dtype=torch.bool))
    for wb in blocks:
        h = rms(x, wb["g1"])
        qkv = h @ wb["W_qkv"]
        qk = rope(qkv[:, :2 * D], 2 * H)
        q = qk[:, :D].view(B, T, H, hd).transpose(1, 2)
        k = qk[:, D:].view(B, T, H, hd).transpose(1, 2)
        v = qkv[:, 2 * D:].view(B, T, H, hd).transpose(1, 2)
        s = (q @ k.transpose(-1, -2)) / np.sqrt(hd)
        s = s.masked_fill(~mask, float("-inf"))
        att = (torch.softmax(s, dim=-1) @ v).transpose(1, 2).reshape(B * T, D)
        x1 = x + att @ wb["W_o"]
        h2 = rms(x1, wb["g2"])
        g = h2 @ wb["W_gate"]
        x = x1 + (g * torch.sigmoid(g) * (h2 @ wb["W_up"])) @ wb["W_down"]
    logits = x @ head.T
    loss = torch.nn.functional.cross_entropy(logits, lab)
    loss.backward()
    grads = {"head": head.grad.detach().numpy(), "emb": emb.grad.detach().numpy()}
    for i, wb in enumerate(blocks):
        for k2, v2 in wb.items():
            grads[f"block{i}.{k2}"] = v2.grad.detach().numpy()
    return float(loss.detach()), grads


def test_step_gradients_match_float64_autograd():
    c = inputs.byte_lm_cfg2(batch=4, seq=32)
    hp = dict(lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=1)
    st = oracle_models.byte_lm_step(c, hp)
    loss64, g64 = torch_model_grads(c)
    assert abs(float(st["loss_mean"][0]) - loss64) <= 1e-5 * abs(loss64)
    for k, ref in g64.items():
        got = st[f"grad.{k}"].astype(np.float64)
        err = np.abs(got - ref).max()
        assert err <= 5e-6 * np.abs(ref).max() + 1e-12, (k, err, np.abs(ref).max())
