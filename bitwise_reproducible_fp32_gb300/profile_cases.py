"""Runs one operation of the path on a fixed, seeded case, a few times, so a
profiler can capture a chosen launch (ncu -k ... -s ... -c ...).

  python -m bitwise_reproducible_fp32_gb300.profile_cases CASE [--reps R]

Cases keep the device footprint at a few hundred MB, above the 129 MB L2 so
DRAM counters mean something:
  lm_head   GEMM 1024 x 50257 x 768, weight [50257, 768] transposed (with its
            workspace: X is copied transposed first, as in the benchmark);
            --tokens 8192 gives the benchmark's full size (about 1.9 GB)
  qkv       GEMM 8192 x 2304 x 768 (likewise)
  dw_qkv    GEMM X^T dY, 768 x 2304 over 8192 tokens
  dw_pair   the two weight-gradient GEMMs (768 x 2304 and 2048 x 768 over 8192
            tokens) as one group, as the benchmark runs them
  gate_up   the gate and up projections of one 8192 x 768 input (768 x 2048
            each) as one group: one transposed copy, one grid
  xent      cross-entropy 1024 x 50257 with dlogits and mean; --tokens 8192
            gives the benchmark's full size (about 3.3 GB)
  rmsnorm   RMSNorm 8192 x 768
  rms_bwd   RMSNorm backward 8192 x 768 (dx, dgain)
  shardsum  fixed-order sum of 64 shard gradients of 768 x 2304
  adamw     AdamW over 32 Mi parameters; --params 162147840 gives the 162M
            model's full size (about 2.6 GB)
  softmax   causal softmax of 48 stacked 2048 x 2048 score matrices (the 162M
            block's attention, 4 x 2048 tokens x 12 heads), in place
  attention causal attention of 4 x 2048 tokens, 12 heads of 64 (the 162M
            block's), from a packed QKV activation
  attention_bwd  the backward of that attention (S and P again, dP, dV, dS, dQ, dK)
  block     one decoder block forward at 4 x 2048 tokens (the 162M shape)
Each run is one warm-up launch followed by R launches (default 2).
"""
from __future__ import annotations

import argparse
import sys

import numpy as np


def main(argv=None):
    import torch

    from bitwise_reproducible_fp32_gb300 import build, detlib, inputs

    ap = argparse.ArgumentParser()
    ap.add_argument("case", choices=["lm_head", "qkv", "dw_qkv", "dw_pair", "gate_up", "xent",
                                    "rmsnorm", "rms_bwd", "shardsum", "adamw", "softmax",
                                    "attention", "attention_bwd", "block"])
    ap.add_argument("--reps", type=int, default=2)
    ap.add_argument("--tokens", type=int, default=None,
                    help="rows of the lm_head / qkv / xent cases (defaults 1024 / 8192 / 1024)")
    ap.add_argument("--params", type=int, default=32 * 1024 * 1024,
                    help="parameters of the adamw case")
    a = ap.parse_args(argv)
    build.build()
    detlib.load()
    dev = torch.device("cuda", 0)
    up = lambda x: torch.from_numpy(np.ascontiguousarray(x)).to(dev)

    if a.case in ("lm_head", "qkv"):
        tokens = a.tokens or (1024 if a.case == "lm_head" else 8192)
        probs = {p["name"]: p for p in inputs.gemm_cfg3(tokens=tokens)}
        p = probs[a.case]
        A, B = up(p["A"]), up(p["B"])
        M = p["A"].shape[0]
        N = p["B"].shape[0] if p["transB"] else p["B"].shape[1]
        C = torch.empty((M, N), dtype=torch.float32, device=dev)
        K = p["A"].shape[1]
        ws = detlib.gemm_workspace(M, N, K, p["transA"], p["transB"])
        run = lambda: detlib.detgemm_f32(A, B, C, transA=p["transA"], transB=p["transB"],
                                         workspace=ws)
    elif a.case == "dw_qkv":
        p = inputs.dw_cfg5()[0]
        A, B = up(p["A"]), up(p["B"])
        C = torch.empty((p["A"].shape[1], p["B"].shape[1]), dtype=torch.float32, device=dev)
        ws = detlib.gemm_workspace(C.shape[0], C.shape[1], p["A"].shape[0], True, False)
        run = lambda: detlib.detgemm_f32(A, B, C, transA=True, workspace=ws)
    elif a.case == "dw_pair":
        probs = []
        for p in inputs.dw_cfg5():
            A, B = up(p["A"]), up(p["B"])
            C = torch.empty((p["A"].shape[1], p["B"].shape[1]), dtype=torch.float32, device=dev)
            probs.append(dict(A=A, B=B, C=C, transA=True))
        ws = detlib.gemm_group_workspace(probs)
        run = lambda: detlib.detgemm_group_f32(probs, workspace=ws)
    elif a.case == "gate_up":
        fw = {p["name"]: p for p in inputs.gemm_cfg3()}
        X = up(fw["swiglu_gate"]["A"])
        probs = [dict(A=X, B=up(fw[n]["B"]), C=torch.empty((X.shape[0], fw[n]["B"].shape[1]),
                                                             dtype=torch.float32, device=dev))
                 for n in ("swiglu_gate", "swiglu_up")]
        ws = detlib.gemm_group_workspace(probs)
        run = lambda: detlib.detgemm_group_f32(probs, workspace=ws)
    elif a.case in ("xent", "rmsnorm"):
        r = inputs.rowops_cfg4(rows=(a.tokens or 1024) if a.case == "xent" else 8192)
        if a.case == "xent":
            X, L = up(r["logits"]), up(r["labels"])
            D = torch.empty_like(X)
            loss = torch.empty(X.shape[0], dtype=torch.float32, device=dev)
            mean = torch.empty(1, dtype=torch.float32, device=dev)
            run = lambda: detlib.detxent_f32(X, L, loss=loss, loss_mean=mean, dlogits=D)
        else:
            x, g = up(r["x"]), up(r["gain"])
            y = torch.empty_like(x)
            inv = torch.empty(x.shape[0], dtype=torch.float32, device=dev)
            run = lambda: detlib.detrmsnorm_f32(x, g, float(r["eps"]), y=y, inv_rms=inv)
    elif a.case == "rms_bwd":
        f = inputs.rmsnorm_bwd_cfg4()
        x, g, dy = up(f["x"]), up(f["gain"]), up(f["dy"])
        _, inv = detlib.detrmsnorm_f32(x, g, float(f["eps"]))
        dx = torch.empty_like(x)
        dgain = torch.empty(x.shape[1], dtype=torch.float32, device=dev)
        ws = torch.empty((detlib.detrmsnorm_bwd_workspace_bytes(*x.shape) + 3) // 4,
                         dtype=torch.float32, device=dev)
        run = lambda: detlib.detrmsnorm_bwd_f32(x, g, inv, dy, dx=dx, dgain=dgain, workspace=ws)
    elif a.case == "shardsum":
        g = up(inputs.shard_grads())
        out = torch.empty(g.shape[1], dtype=torch.float32, device=dev)
        run = lambda: detlib.detshardsum_f32(g, scale=1.0 / g.shape[0], out=out)
    elif a.case == "softmax":
        g = torch.Generator(device=dev).manual_seed(5)
        S = torch.randn((48 * 2048, 2048), generator=g, device=dev) * 4
        run = lambda: detlib.detsoftmax_causal_f32(S, scale=0.125, period=2048, p=S)
    elif a.case == "attention":
        g = torch.Generator(device=dev).manual_seed(6)
        B, T, H, d = 4, 2048, 12, 64
        qkv = torch.randn((B * T, 3 * H * d), generator=g, device=dev)
        out = torch.empty((B * T, H * d), dtype=torch.float32, device=dev)
        ws = torch.empty((detlib.detattention_workspace_bytes(B, T, H, d) + 3) // 4,
                         dtype=torch.float32, device=dev)
        run = lambda: detlib.detattention_f32(qkv, B, T, H, d, out=out, workspace=ws)
    elif a.case == "attention_bwd":
        g = torch.Generator(device=dev).manual_seed(6)
        B, T, H, d = 4, 2048, 12, 64
        qkv = torch.randn((B * T, 3 * H * d), generator=g, device=dev)
        dout = torch.randn((B * T, H * d), generator=g, device=dev)
        dqkv = torch.empty_like(qkv)
        ws = torch.empty((detlib.detattention_bwd_workspace_bytes(B, T, H, d) + 3) // 4,
                         dtype=torch.float32, device=dev)
        run = lambda: detlib.detattention_bwd_f32(qkv, dout, B, T, H, d, dqkv=dqkv, workspace=ws)
    elif a.case == "block":
        from bitwise_reproducible_fp32_gb300 import block as blockmod
        bc = inputs.block_cfg()
        blk = blockmod.Block(bc["batch"], bc["seq"], bc["x"].shape[1], bc["W_gate"].shape[1],
                             inputs.N_HEADS, dev)
        x = up(bc["x"])
        w = {k: up(bc[k]) for k in ("g1", "W_qkv", "W_o", "g2", "W_gate", "W_up", "W_down")}
        run = lambda: blk.forward(x, w)
    else:
        w = inputs.adamw_cfg5(n=a.params)
        P, G, M_, V_ = (up(w[k]) for k in ("p", "g", "m", "v"))
        hp = {k: w[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "step")}
        run = lambda: detlib.detadamw_f32(P, G, M_, V_, **hp)

    for _ in range(1 + a.reps):
        run()
    torch.cuda.synchronize()
    print(f"{a.case}: {1 + a.reps} launches done")


if __name__ == "__main__":
    sys.exit(main())
