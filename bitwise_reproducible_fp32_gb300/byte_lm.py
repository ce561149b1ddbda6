"""Forward, backward and AdamW update of the small byte-level language model
(the pages' "two transformer blocks, byte level", trained with "embedding,
transformer forward and backward, cross entropy, and AdamW"; "mojolearn" PyPI
page, section "Handing training off between vendors"), at the byte-LM GEMM
shapes: 16 x 128 tokens, 64 wide, 4 heads of 16, SwiGLU 172, 256 byte ids.
Pre-norm blocks, no final norm, an untied LM head stored [vocab, d].

Every stage is a C-ABI call; the returned stage dict names each stage's output
so identity cards (raw-bit hashes per stage) can be compared with the
oracle's.
"""
from __future__ import annotations

PARAMS = ("g1", "W_qkv", "W_o", "g2", "W_gate", "W_up", "W_down")


def head_workspaces(c, device):
    """The three head GEMMs' workspaces of a training step (logits = X W^T,
    dW = dlogits^T X, dX = dlogits W): the transposed copies and split-K
    partials their plans use (None where a plan uses none)."""
    from bitwise_reproducible_fp32_gb300 import detlib as L
    ntok, d, V = c["batch"] * c["seq"], c["d"], c["vocab"]
    return {"logits": L.gemm_workspace(ntok, V, d, False, True, device=device),
            "head_dw": L.gemm_workspace(V, d, ntok, True, False, device=device),
            "head_dx": L.gemm_workspace(ntok, d, V, False, False, device=device)}


def train_step(c, device, hp, status=None, blocks=None, ws=None):
    """One training step. c: the byte_lm_cfg2 tensors on the device; hp: AdamW
    hyperparameters (lr, beta1, beta2, eps, weight_decay, step). The moments
    start at zero. Returns the ordered stage dict: the forward's outputs, the
    gradients, then every parameter and moment after the update.
    status: an int32 device word of one element for the out-of-range token and
    label flag; when given, the step issues no host synchronisation (the
    caller reads the word), so it can be captured in a CUDA graph. Without it
    the step checks the flag itself and raises.
    blocks / ws: prebuilt make_blocks() and head_workspaces() for repeated
    steps (built here when omitted; the bits are the same either way)."""
    import torch

    from bitwise_reproducible_fp32_gb300 import detlib as L
    ntok = c["batch"] * c["seq"]
    check = status is None
    if check:
        status = torch.zeros(1, dtype=torch.int32, device=device)
    if blocks is None:
        blocks = make_blocks(c, device)
    if ws is None:
        ws = {"logits": None, "head_dw": None, "head_dx": None}
    st = {}
    # forward
    x0 = L.detembedding_f32(c["emb"], c["tokens"], dev_status=status)
    st["embedding"] = x0
    xs = [x0]
    # each block but the last leaves its last residual add to the next block,
    # which forms it together with its first RMSNorm (the same bits)
    pending = None
    for i, (blk, w) in enumerate(zip(blocks, c["blocks"])):
        last = i == len(blocks) - 1
        xs.append(blk.forward(xs[-1], w, residual=pending, defer_add=not last))
        pending = None if last else blk.residual()
        st[f"block{i}"] = xs[-1]
    logits = L.detgemm_f32(xs[-1], c["head"], transB=True, workspace=ws["logits"])
    st["logits"] = logits
    # dlogits rows padded to a multiple of 4 floats: the head's two backward
    # GEMMs read them through TMA, which wants 16-byte row strides
    vpad = (c["vocab"] + 3) // 4 * 4
    dl = torch.empty((ntok, vpad), dtype=torch.float32, device=device)[:, :c["vocab"]]
    loss, mean, dlogits = L.detxent_f32(logits, c["labels"], want_mean=True, dlogits=dl,
                                        dscale=1.0 / ntok, dev_status=status)
    st["loss"], st["loss_mean"], st["dlogits"] = loss, mean, dlogits
    # backward
    head_ws = ws["head_dw"]
    if head_ws is None:
        head_ws = L.gemm_workspace(c["vocab"], c["d"], ntok, True, False, device=device)
    grads = {"head": L.detgemm_f32(dlogits, xs[-1], transA=True, workspace=head_ws)}
    dx = L.detgemm_f32(dlogits, c["head"], workspace=ws["head_dx"])
    for i in reversed(range(len(blocks))):
        dx, g = blocks[i].backward(xs[i], c["blocks"][i], dx)
        for k in PARAMS:
            grads[f"block{i}.{k}"] = g[k]
        st[f"d_block{i}_input"] = dx
    grads["emb"] = L.detembedding_bwd_f32(c["tokens"], dx, c["vocab"])
    for k in sorted(grads):
        st[f"grad.{k}"] = grads[k]
    # AdamW on every parameter (decay on all, no mask), moments from zero
    params = {"head": c["head"], "emb": c["emb"]}
    for i, w in enumerate(c["blocks"]):
        for k in PARAMS:
            params[f"block{i}.{k}"] = w[k]
    for k in sorted(params):
        p = params[k].clone()
        m = torch.zeros_like(p)
        v = torch.zeros_like(p)
        L.detadamw_f32(p.view(-1), grads[k].contiguous().view(-1), m.view(-1), v.view(-1), **hp)
        st[f"param.{k}"], st[f"m.{k}"], st[f"v.{k}"] = p, m, v
    if check and int(status.item()) != 0:
        raise ValueError("a token or label outside the vocabulary")
    return st


def make_blocks(c, device):
    """The Block objects (activation buffers and GEMM workspaces) of a model
    configuration, one a layer; built once, they serve every forward call."""
    from bitwise_reproducible_fp32_gb300 import block
    return [block.Block(c["batch"], c["seq"], c["d"], c["dff"], c["heads"], device)
            for _ in c["blocks"]]


def forward(c, device, blocks=None, head_ws=None):
    """The forward stages alone (embedding, blocks, logits, loss, mean). The
    same code runs the byte-level LM and the 12-layer 162M decoder (the two
    share the architecture: pre-norm blocks, no final norm, untied head).
    blocks / head_ws: prebuilt make_blocks() and the head GEMM's workspace
    (built here when omitted)."""
    import torch

    from bitwise_reproducible_fp32_gb300 import detlib as L
    status = torch.zeros(1, dtype=torch.int32, device=device)
    st = {}
    x = L.detembedding_f32(c["emb"], c["tokens"], dev_status=status)
    st["embedding"] = x
    if blocks is None:
        blocks = make_blocks(c, device)
    if head_ws is None:
        head_ws = L.gemm_workspace(c["batch"] * c["seq"], c["vocab"], c["d"], False, True,
                                   device=device)
    pending = None
    for i, (blk, w) in enumerate(zip(blocks, c["blocks"])):
        # each block owns its output buffer; all but the last leave their last
        # residual add to the next block's first kernel
        last = i == len(blocks) - 1
        x = blk.forward(x, w, residual=pending, defer_add=not last)
        pending = None if last else blk.residual()
        st[f"block{i}"] = x
    logits = L.detgemm_f32(x, c["head"], transB=True, workspace=head_ws)
    st["logits"] = logits
    loss, mean, _ = L.detxent_f32(logits, c["labels"], want_mean=True, dev_status=status)
    st["loss"], st["loss_mean"] = loss, mean
    if int(status.item()) != 0:
        raise ValueError("a token or label outside the vocabulary")
    return st
