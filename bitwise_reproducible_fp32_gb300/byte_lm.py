"""Forward and loss of the small byte-level language model (the pages' "two
transformer blocks, byte level"; "mojolearn" PyPI page, section "Handing
training off between vendors"), at the byte-LM GEMM shapes: 16 x 128 tokens,
64 wide, 4 heads of 16, SwiGLU 172, 256 byte ids. Pre-norm blocks, no final
norm, an untied LM head stored [vocab, d] (the 162M model card's layout).
Every stage is a C-ABI call; `stages` names each stage's output so identity
cards (raw-bit hashes per stage) can be compared with the oracle's.
"""
from __future__ import annotations


def forward(cfg_dev, device):
    """cfg_dev: the byte_lm_cfg2 tensors on the device (tokens, labels int32;
    emb, head and each block's weights float32). Returns the ordered stage
    dict: embedding, block0, block1, ..., logits, loss, loss_mean."""
    import torch

    from bitwise_reproducible_fp32_gb300 import block, detlib
    B, T, d = cfg_dev["batch"], cfg_dev["seq"], cfg_dev["d"]
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stages = {}
    x = detlib.detembedding_f32(cfg_dev["emb"], cfg_dev["tokens"], dev_status=status)
    stages["embedding"] = x
    blocks = [block.Block(B, T, d, cfg_dev["dff"], cfg_dev["heads"], device)
              for _ in cfg_dev["blocks"]]
    for i, (blk, w) in enumerate(zip(blocks, cfg_dev["blocks"])):
        x = blk.forward(x, w)          # each block owns its output buffer
        stages[f"block{i}"] = x
    logits = detlib.detgemm_f32(x, cfg_dev["head"], transB=True)
    stages["logits"] = logits
    loss, mean, _ = detlib.detxent_f32(logits, cfg_dev["labels"], want_mean=True,
                                       dev_status=status)
    stages["loss"] = loss
    stages["loss_mean"] = mean
    if int(status.item()) != 0:
        raise ValueError("a token or label outside the vocabulary")
    return stages
