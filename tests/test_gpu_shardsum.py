"""GPU parity (0 ULP) of the fixed-order shard gradient sum and the
accumulating (beta = 1) GEMM against the oracle: shard counts up to 64,
ragged lengths, strided and unaligned shard buffers, special values, in-place
output, the split-K path of the accumulating GEMM, and the identity between
accumulating shard after shard and summing the shards' products."""
import numpy as np
import pytest

import oracle
from bitcmp import assert_bitwise
from bitwise_reproducible_fp32_gb300 import detlib, inputs
from gpu_util import host, need_gpu, to_dev, torch

pytestmark = pytest.mark.gpu
F = np.float32


@pytest.fixture(scope="module")
def dev():
    return need_gpu()


def shards(S, n, seed):
    rng = np.random.default_rng(seed)
    g = (rng.standard_normal((S, n)) * np.exp2(rng.integers(-20, 20, (S, n)))).astype(F)
    return g


@pytest.mark.parametrize("S", [1, 2, 7, 9, 64])
@pytest.mark.parametrize("n", [1, 5, 1000, 4099, 100004])
@pytest.mark.parametrize("layout", ["dense", "padded", "offset"])
def test_shard_sum(dev, S, n, layout):
    g = shards(S, n, S * 1000 + n)
    for scale in (1.0, 1.0 / 64, 1.0 / 3):
        want = oracle.shardsum(g, scale=scale)
        got = detlib.detshardsum_f32(to_dev(g, layout), scale=scale)
        assert_bitwise(host(got), want, f"S={S} n={n} {layout} scale={scale}")


def test_shard_sum_special_values_and_in_place(dev):
    g = shards(5, 1003, 61)
    g[:, 0] = F(-0.0)                 # stays -0
    g[1, 1] = F(np.nan)
    g[2, 2] = F(np.inf)
    g[3, 2] = F(-np.inf)              # inf - inf = NaN
    g[:, 3] = F(2.0 ** -140)          # subnormal sums
    g[0, 4], g[1:, 4] = F(2.0 ** 24), F(1.0)     # order: ties to even keep 2^24
    want = oracle.shardsum(g, scale=1.0 / 64)
    gd = to_dev(g)
    got = detlib.detshardsum_f32(gd, scale=1.0 / 64, out=gd[0])   # in place over shard 0
    assert_bitwise(host(got), want)
    assert host(got)[4] == F(2.0 ** 24 / 64)


def test_shard_sum_64_shards_of_a_weight_gradient(dev):
    # the pages' 64 logical shards, at the 768 x 2304 QKV weight-gradient size
    rng = np.random.default_rng(62)
    g = (1e-3 * rng.standard_normal((64, 768 * 2304))).astype(F)
    want = oracle.shardsum(g, scale=1.0 / 64)
    got = detlib.detshardsum_f32(to_dev(g), scale=1.0 / 64)
    assert_bitwise(host(got), want)


@pytest.mark.parametrize("M,N,K", [(1, 1, 1), (70, 90, 777), (300, 200, 1300), (33, 1000, 2049)])
@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_accumulating_gemm(dev, M, N, K, transA, transB):
    rng = np.random.default_rng(M * 7 + N + K)
    A = rng.standard_normal((K, M) if transA else (M, K)).astype(F)
    B = rng.standard_normal((N, K) if transB else (K, N)).astype(F)
    C = rng.standard_normal((M, N)).astype(F)
    C[0, 0] = F(-0.0)
    want = oracle.gemm_acc(C, A, B, transA=bool(transA), transB=bool(transB))
    for use_ws in (False, True):
        ws = detlib.gemm_workspace(M, N, K, transA, transB) if use_ws else None
        Cd = to_dev(C, "padded")
        detlib.detgemm_acc_f32(to_dev(A), to_dev(B), Cd, transA=bool(transA),
                               transB=bool(transB), workspace=ws)
        assert_bitwise(host(Cd), want, f"{M}x{N}x{K} tA={transA} tB={transB} ws={use_ws}")


def test_accumulating_gemm_k_zero(dev):
    C = np.array([[-0.0, 1.0, np.nan]], F)
    Cd = to_dev(C)
    detlib.detgemm_acc_f32(torch.zeros((1, 0), device="cuda"), torch.zeros((0, 3), device="cuda"),
                           Cd)
    got = host(Cd)
    assert got.view(np.uint32)[0, 0] == 0 and got[0, 1] == F(1.0) and np.isnan(got[0, 2])


def test_accumulation_over_token_shards_is_the_shard_sum(dev):
    # dW = X^T dY over 8192 tokens cut into 4 shards of 2048 (8 chunks each):
    # accumulating the shards in order equals the shard sum of their products
    p = inputs.dw_cfg5(tokens=8192)[0]
    X, dY = p["A"], p["B"]
    parts = []
    Cacc = None
    for s in range(4):
        Xs, dYs = to_dev(X[2048 * s:2048 * (s + 1)]), to_dev(dY[2048 * s:2048 * (s + 1)])
        Ps = detlib.detgemm_f32(Xs, dYs, transA=True)
        parts.append(Ps)
        if Cacc is None:
            Cacc = Ps.clone()
        else:
            detlib.detgemm_acc_f32(Xs, dYs, Cacc, transA=True)
    stacked = torch.stack(parts).reshape(4, -1)
    total = detlib.detshardsum_f32(stacked)
    assert_bitwise(host(Cacc).reshape(-1), host(total), "accumulate vs shard sum on the GPU")
    rows = [0, 1, 383, 767]
    want = oracle.shardsum(np.stack([oracle.gemm(X[2048 * s:2048 * (s + 1), :][:, rows], dY[2048 * s:2048 * (s + 1)], True, False)
                                     for s in range(4)]))
    assert_bitwise(host(Cacc)[rows], want, "against the oracle on sampled rows")
