"""Every non-positive float through the row reductions' own exp.

The cross-entropy and the causal softmax do not call the general exp: their
hot loops use a branch-free form for arguments d = x - max <= 0 (rounding t =
d log2(e) to an integer by the 1.5 * 2^23 addition, scaling on the exponent
bits, packed FP32 pairs), which must give the profile's exp bits ("mojolearn"
PyPI page, section "What bitwise identity means, and why it is not the
default": the spellings of exp and log are fixed). This test feeds every float
d <= 0 -- all 2^31 - 2^23 + 1 of them from -0 to -inf, NaNs excluded -- through
those kernels in chunks of 2^28, each chunk as rows [0, d_0, ..., d_{V-2}]
(row max +0, label 0, so the row's exp arguments are exactly the d), and
compares loss, dlogits and probabilities bit for bit with the oracle:
  * detxent_f32 with rows of 4096 (the shared-memory kernel);
  * detxent_f32 with rows of 60,001 (the kernel for rows longer than shared
    memory);
  * detsoftmax_causal_f32 with every column kept.
Rows whose d are all below -28 have S = 1 exactly, so their dlogits and
probabilities are the exp values themselves.
"""
import numpy as np
import pytest

import oracle
from bitcmp import assert_bitwise
from bitwise_reproducible_fp32_gb300 import detlib
from gpu_util import host, need_gpu, torch

pytestmark = pytest.mark.gpu
F = np.float32

FIRST, LAST = 0x80000000, 0xFF800000        # -0 ... -inf, by bit pattern
CHUNK = 1 << 28


def chunk_rows(lo_bits: int, hi_bits: int, V: int) -> np.ndarray:
    """Rows [0, d...] covering the bit patterns lo_bits .. hi_bits - 1; the
    last row is padded with -inf (exp gives +0 there)."""
    d = np.arange(lo_bits, hi_bits, dtype=np.uint64).astype(np.uint32).view(F)
    per = V - 1
    rows = -(-d.size // per)
    body = np.full(rows * per, -np.inf, F)
    body[:d.size] = d
    x = np.empty((rows, V), F)
    x[:, 0] = 0.0
    x[:, 1:] = body.reshape(rows, per)
    return x


def check_xent(x: np.ndarray, what: str):
    lab = np.zeros(x.shape[0], np.int32)
    loss_w, d_w, bad = oracle.xent(x, lab, with_dlogits=True, dscale=F(1.0))
    assert bad == 0
    xd = torch.from_numpy(x).cuda()
    loss, _, dl = detlib.detxent_f32(xd, torch.from_numpy(lab).cuda(), want_dlogits=True,
                                     dscale=1.0)
    assert_bitwise(host(loss), loss_w, f"{what} loss")
    assert_bitwise(host(dl), d_w, f"{what} dlogits")
    del xd, dl, loss


def check_softmax(x: np.ndarray, what: str):
    rows, cols = x.shape
    p_w = oracle.softmax_causal(x, scale=1.0, diag=cols)
    xd = torch.from_numpy(x).cuda()
    p = detlib.detsoftmax_causal_f32(xd, scale=1.0, diag=cols)
    assert_bitwise(host(p), p_w, f"{what} probabilities")
    del xd, p


def ranges():
    lo = FIRST
    while lo <= LAST:
        hi = min(lo + CHUNK, LAST + 1)
        yield lo, hi
        lo = hi


def test_every_nonpositive_float_through_the_cross_entropy():
    need_gpu()
    n = 0
    for lo, hi in ranges():
        check_xent(chunk_rows(lo, hi, 4096), f"bits {lo:#x}..{hi - 1:#x}, rows of 4096")
        n += hi - lo
    assert n == LAST - FIRST + 1


def test_every_nonpositive_float_through_the_long_row_cross_entropy():
    need_gpu()
    for lo, hi in ranges():
        check_xent(chunk_rows(lo, hi, 60001), f"bits {lo:#x}..{hi - 1:#x}, rows of 60001")


def test_every_nonpositive_float_through_the_causal_softmax():
    need_gpu()
    for lo, hi in ranges():
        check_softmax(chunk_rows(lo, hi, 4096), f"bits {lo:#x}..{hi - 1:#x}")
