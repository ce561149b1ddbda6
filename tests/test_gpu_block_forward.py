"""GPU parity (0 ULP) of a whole pre-norm decoder block's forward, composed
from the library's calls, against the same composition of oracle functions:
a small block in full, and one 162M-shaped block (4 x 2048 tokens, 768 wide,
12 heads, SwiGLU 2048) in full."""
import numpy as np
import pytest

import oracle
import oracle_models
from bitcmp import assert_bitwise
from bitwise_reproducible_fp32_gb300 import block, inputs
from gpu_util import host, need_gpu, to_dev, torch

pytestmark = pytest.mark.gpu
F = np.float32


@pytest.fixture(scope="module")
def dev():
    return need_gpu()


def oracle_block(c, heads):
    return oracle_models.block(c["x"], c, c["batch"], c["seq"], heads)


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
