"""The forward of one pre-norm decoder block through the library's operations
("MojoLearn 162M" model card, table "Compared with GPT-3 Small": 768 wide,
12 heads of 64, rotary positions with theta = 10,000, RMSNorm eps 1e-6,
pre-norm, SwiGLU 2,048 wide, no biases):

    h   = RMSNorm(x, g1)
    qkv = h W_qkv;  Q, K turned by the rotary embedding
    a   = causal attention(Q, K, V), scale 1/sqrt(64)
    x1  = x + a W_o
    h2  = RMSNorm(x1, g2)
    y   = x1 + (silu(h2 W_gate) * (h2 W_up)) W_down

Every step is one call of the C ABI (detlib); this module only sequences them
and owns the intermediate buffers. Weights are K x N row-major, as the
GEMMs take them.
"""
from __future__ import annotations


class Block:
    """Buffers and workspaces for one block's forward at a fixed shape."""

    def __init__(self, batch, seq, d_model, d_ff, heads, device, eps=1e-6, theta=10000.0):
        import torch

        from bitwise_reproducible_fp32_gb300 import detlib
        self.B, self.T, self.D, self.Fd, self.H = batch, seq, d_model, d_ff, heads
        self.hd = d_model // heads
        self.eps, self.theta = eps, theta
        n = batch * seq
        e = lambda *s: torch.empty(s, dtype=torch.float32, device=device)  # noqa: E731
        self.h, self.inv1 = e(n, d_model), e(n)
        self.qkv, self.att, self.o = e(n, 3 * d_model), e(n, d_model), e(n, d_model)
        self.x1, self.h2, self.inv2 = e(n, d_model), e(n, d_model), e(n)
        self.gate, self.up, self.s, self.dn = e(n, d_ff), e(n, d_ff), e(n, d_ff), e(n, d_model)
        self.y = e(n, d_model)
        ws = lambda M, N, K: detlib.gemm_workspace(M, N, K, False, False, device=device)  # noqa: E731
        self.ws = {"qkv": ws(n, 3 * d_model, d_model), "o": ws(n, d_model, d_model),
                   "down": ws(n, d_model, d_ff)}
        # the gate and up projections of h2 run as one group (one transposed
        # copy of h2, one grid for both); the plan needs only shapes and that
        # both read the same h2, so a stand-in weight serves for the query
        wq = e(d_model, d_ff)
        self.ws["gate_up"] = detlib.gemm_group_workspace(
            [dict(A=self.h2, B=wq, C=self.gate), dict(A=self.h2, B=wq, C=self.up)])
        del wq
        self.att_ws = e((detlib.detattention_workspace_bytes(batch, seq, heads, self.hd) + 3)
                        // 4)
        self.ws_bwd = {}       # weight-gradient GEMM workspaces, by output shape

    def flops(self):
        """The forward's algorithmic FLOPs: 2 per multiply-add of the six
        projections, and of the causal attention's two products counted over
        the kept scores only (query i against keys 0..i: T(T+1)/2 pairs a
        head, hd multiply-adds each, for Q K^T and again for P V). Work the
        kernels do on tiles that straddle the diagonal is not counted."""
        n, D, Fd = self.B * self.T, self.D, self.Fd
        gemm = 2 * n * (D * 3 * D + D * D + 2 * D * Fd + Fd * D)
        kept = self.T * (self.T + 1) // 2
        attn = 2 * 2 * self.B * self.H * kept * self.hd
        return gemm + attn

    def forward(self, x, w, residual=None, defer_add=False):
        """x: (batch * seq) x d_model; w: g1, W_qkv, W_o, g2, W_gate, W_up,
        W_down (device tensors). Returns y (this object's buffer).
        residual: (x1, dn) of the block before, which deferred its last add:
        x is then that block's y buffer, and this block forms x = x1 + dn
        there together with its first RMSNorm (one kernel, the same bits).
        defer_add: leave y = x1 + dn to the next block (its residual)."""
        from bitwise_reproducible_fp32_gb300 import detlib as L
        if residual is not None:
            L.detadd_rmsnorm_f32(residual[0], residual[1], w["g1"], self.eps, x=x, y=self.h,
                                 inv_rms=self.inv1)
        else:
            L.detrmsnorm_f32(x, w["g1"], self.eps, y=self.h, inv_rms=self.inv1)
        L.detgemm_f32(self.h, w["W_qkv"], self.qkv, workspace=self.ws["qkv"])
        L.detrope_f32(self.qkv, heads=2 * self.H, head_dim=self.hd, seq_len=self.T,
                      theta=self.theta)
        L.detattention_f32(self.qkv, self.B, self.T, self.H, self.hd, out=self.att,
                           workspace=self.att_ws)
        L.detgemm_f32(self.att, w["W_o"], self.o, workspace=self.ws["o"])
        # x1 = x + o and h2 = RMSNorm(x1), one kernel
        L.detadd_rmsnorm_f32(x, self.o, w["g2"], self.eps, x=self.x1, y=self.h2,
                             inv_rms=self.inv2)
        L.detgemm_group_f32([dict(A=self.h2, B=w["W_gate"], C=self.gate),
                             dict(A=self.h2, B=w["W_up"], C=self.up)],
                            workspace=self.ws["gate_up"])
        L.detswiglu_f32(self.gate, self.up, out=self.s)
        L.detgemm_f32(self.s, w["W_down"], self.dn, workspace=self.ws["down"])
        if not defer_add:
            L.detadd_f32(self.x1, self.dn, out=self.y)
        return self.y

    def residual(self):
        """The pair whose sum is y, for a next block given defer_add."""
        return self.x1, self.dn

    def backward(self, x, w, dy):
        """Gradients of the block's forward from dy (the gradient of its
        output), with the activations this object kept. Returns (dx, grads)
        with grads named as the weights (g1, W_qkv, W_o, g2, W_gate, W_up,
        W_down). Readings: a residual's gradient first in every sum of
        gradients; the gate's contribution to dh2 first, then up's (as the
        forward used them)."""
        import torch

        from bitwise_reproducible_fp32_gb300 import detlib as L
        n, D, Fd = self.B * self.T, self.D, self.Fd
        e = lambda *s: torch.empty(s, dtype=torch.float32, device=dy.device)  # noqa: E731
        g = {}
        def tA(A, B):
            # weight gradients contract over the tokens: K = batch * seq, few
            # output tiles, so the GEMM splits K through a workspace
            M, N = A.shape[1], B.shape[1]
            if (M, N) not in self.ws_bwd:
                self.ws_bwd[(M, N)] = L.gemm_workspace(M, N, n, True, False, device=dy.device)
            return L.detgemm_f32(A, B, transA=True, workspace=self.ws_bwd[(M, N)])

        def tB_ws(A, B):
            # the input gradients: A k-contiguous, so the GEMM reads a
            # transposed copy of it where its plan takes one
            M, N, K = A.shape[0], B.shape[0], A.shape[1]
            key = ("tB", M, N, K)
            if key not in self.ws_bwd:
                self.ws_bwd[key] = L.gemm_workspace(M, N, K, False, True, device=dy.device)
            return self.ws_bwd[key]
        tB = lambda A, B, C=None: L.detgemm_f32(A, B, C, transB=True,          # noqa: E731
                                                workspace=tB_ws(A, B))

        def tA2(A, B1, B2):
            # two weight gradients of one input, as one group
            M, N1, N2 = A.shape[1], B1.shape[1], B2.shape[1]
            probs = [dict(A=A, B=B1, C=e(M, N1), transA=True),
                     dict(A=A, B=B2, C=e(M, N2), transA=True)]
            key = ("pair", M, N1, N2)
            if key not in self.ws_bwd:
                self.ws_bwd[key] = L.gemm_group_workspace(probs)
            L.detgemm_group_f32(probs, workspace=self.ws_bwd[key])
            return probs[0]["C"], probs[1]["C"]
        # y = x1 + s W_down
        ds = tB(dy, w["W_down"])
        g["W_down"] = tA(self.s, dy)
        d_gate, d_up = L.detswiglu_bwd_f32(self.gate, self.up, ds)
        dh2 = tB(d_gate, w["W_gate"])
        L.detgemm_acc_f32(d_up, w["W_up"], dh2, transB=True, workspace=tB_ws(d_up, w["W_up"]))
        g["W_gate"], g["W_up"] = tA2(self.h2, d_gate, d_up)
        dx1_b, g["g2"] = L.detrmsnorm_bwd_f32(self.x1, w["g2"], self.inv2, dh2)
        dx1 = L.detadd_f32(dy, dx1_b)
        # x1 = x + att W_o
        d_att = tB(dx1, w["W_o"])
        g["W_o"] = tA(self.att, dx1)
        # P from the forward (still in this block's attention workspace)
        dqkv = L.detattention_bwd_saved_f32(self.qkv, d_att, self.B, self.T, self.H, self.hd,
                                            self.att_ws)
        L.detrope_bwd_f32(dqkv, heads=2 * self.H, head_dim=self.hd, seq_len=self.T,
                          theta=self.theta)
        dh = tB(dqkv, w["W_qkv"])
        g["W_qkv"] = tA(self.h, dqkv)
        dx_b, g["g1"] = L.detrmsnorm_bwd_f32(x, w["g1"], self.inv1, dh)
        dx = L.detadd_f32(dx1, dx_b)
        return dx, g
