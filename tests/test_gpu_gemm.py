"""GPU parity of the fixed-order GEMM: every output bit-identical (0 ULP) to the
oracle, over ragged shapes, all four operand layouts, both operand staging
paths (TMA for 16-byte aligned operands, plain loads otherwise), the small
configurations in full, and the full-size 162M-decoder and weight-gradient
GEMMs on sampled rows, in the launch configuration the benchmark uses."""
import numpy as np
import pytest

import oracle
from bitcmp import assert_bitwise
from bitwise_reproducible_fp32_gb300 import detlib, inputs
from gpu_util import empty_dev, host, need_gpu, to_dev, torch

pytestmark = pytest.mark.gpu
F = np.float32


@pytest.fixture(scope="module")
def dev():
    return need_gpu()


def wide_random(rng, shape):
    mant = rng.uniform(1.0, 2.0, size=shape)
    exps = rng.integers(-30, 30, size=shape)
    sign = rng.choice([-1.0, 1.0], size=shape)
    x = (sign * mant * np.exp2(exps)).astype(F)
    mask = rng.random(shape)
    x[mask < 0.03] = F(0.0)
    x[(mask >= 0.03) & (mask < 0.05)] = F(-0.0)
    x[(mask >= 0.05) & (mask < 0.06)] *= F(2.0 ** -110)   # subnormal products
    return x


def run_case(M, N, K, transA, transB, layout_a, layout_b, layout_c, seed, wide=False,
             workspaces=(False, True)):
    """Checks every layout/workspace combination against the oracle; the
    workspace (split-K over whole chunks) must not change a bit."""
    rng = np.random.default_rng(seed)
    gen = (lambda s: wide_random(rng, s)) if wide else (
        lambda s: rng.standard_normal(s).astype(F))
    A = gen((K, M) if transA else (M, K))
    B = gen((N, K) if transB else (K, N))
    want = oracle.gemm(A, B, transA=transA, transB=transB)
    Ad, Bd = to_dev(A, layout_a), to_dev(B, layout_b)
    for use_ws in workspaces:
        ws = detlib.gemm_workspace(M, N, K, transA, transB) if use_ws else None
        C = empty_dev(M, N, layout_c)
        detlib.detgemm_f32(Ad, Bd, C, transA=transA, transB=transB, workspace=ws)
        torch.cuda.synchronize()
        assert_bitwise(host(C), want,
                       f"M={M} N={N} K={K} tA={transA} tB={transB} "
                       f"{layout_a}/{layout_b}/{layout_c} workspace={ws is not None}")


SHAPES = [
    (1, 1, 1), (3, 5, 7), (31, 33, 31), (1, 300, 257), (129, 1, 300),
    (128, 128, 32), (128, 128, 256), (127, 129, 255), (129, 127, 257),
    (255, 257, 513), (256, 256, 767), (300, 200, 600), (257, 384, 1000),
    (100, 131, 2049),
]


@pytest.mark.parametrize("M,N,K", SHAPES)
@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_ragged_shapes_all_layouts(dev, M, N, K, transA, transB):
    seed = hash((M, N, K, transA, transB)) % 2 ** 31
    # TMA staging (padded strides keep rows 16-byte aligned)
    run_case(M, N, K, bool(transA), bool(transB), "padded", "padded", "padded", seed)
    # plain-load staging (dense odd strides or an offset base)
    run_case(M, N, K, bool(transA), bool(transB), "dense", "offset", "offset", seed + 1)


@pytest.mark.parametrize("transA,transB", [(0, 0), (0, 1), (1, 0), (1, 1)])
def test_signed_zero_underflow_and_wide_exponents(dev, transA, transB):
    for layout in ("padded", "offset"):
        run_case(70, 90, 777, bool(transA), bool(transB), layout, layout, layout, 5,
                 wide=True)


def test_split_plan_is_used_where_it_helps(dev):
    # few tiles and many chunks: the weight-gradient shapes split K
    assert detlib.detgemm_workspace_bytes(768, 2304, 8192, True, False) > 0
    assert detlib.detgemm_workspace_bytes(2048, 768, 8192, True, False) > 0
    # plenty of tiles: the LM head does not split, but reads a transposed copy
    # of its k-contiguous W (768 x 50,260 floats, 256-byte rounded, first) and
    # of X (768 x 8192 floats) from the workspace
    wcopy = (768 * 50260 * 4 + 255) // 256 * 256
    assert detlib.detgemm_workspace_bytes(8192, 50257, 768, False, True) == wcopy + 768 * 8192 * 4
    # ... of which an m-contiguous A needs only the first
    assert detlib.detgemm_workspace_bytes(8192, 50257, 768, True, True) == wcopy
    # and an n-contiguous B neither
    assert detlib.detgemm_workspace_bytes(8192, 50257, 768, True, False) == 0
    # one chunk and a small product: neither
    assert detlib.detgemm_workspace_bytes(64, 64, 256) == 0


@pytest.mark.parametrize("M,N,K", [(517, 6000, 700), (1000, 4000, 600)])
@pytest.mark.parametrize("transB", [0, 1])
def test_transposed_a_copy_same_bits(dev, M, N, K, transB):
    # large enough that a k-contiguous A is copied transposed into the
    # workspace (row stride M rounded up to 4 floats); ragged M and K
    assert detlib.detgemm_workspace_bytes(M, N, K, False, transB) == K * ((M + 3) // 4 * 4) * 4
    run_case(M, N, K, False, bool(transB), "padded", "padded", "padded", M + K + transB)
    run_case(M, N, K, False, bool(transB), "dense", "offset", "offset", M + K + transB + 1,
             wide=True)
    # an A whose rows are not 16-byte aligned: the copy moves it element by
    # element, and the GEMM then stages the aligned copy by TMA
    run_case(M, N, K, False, bool(transB), "offset", "padded", "padded", M + K + transB + 2)


@pytest.mark.parametrize("M,N,K,transA", [(8192, 2047, 768, 0), (4099, 1537, 2304, 1),
                                           (8192, 770, 2048, 0)])
def test_transposed_b_copy_same_bits(dev, M, N, K, transA):
    # a k-contiguous B (transB) of a product large enough is copied transposed
    # (K x N, row stride N rounded up to 4) into the workspace first; the bits
    # equal those of the product read in place (no workspace) and the oracle
    wsn = detlib.detgemm_workspace_bytes(M, N, K, bool(transA), True)
    assert wsn >= K * ((N + 3) // 4 * 4) * 4
    rng = np.random.default_rng(M + N + K)
    A = rng.standard_normal((K, M) if transA else (M, K)).astype(F)
    B = rng.standard_normal((N, K)).astype(F)
    Ad, Bd = to_dev(A, "padded"), to_dev(B, "offset")
    ws = detlib.gemm_workspace(M, N, K, bool(transA), True)
    C = detlib.detgemm_f32(Ad, Bd, transA=bool(transA), transB=True, workspace=ws)
    C2 = detlib.detgemm_f32(Ad, Bd, transA=bool(transA), transB=True)
    assert_bitwise(host(C2), host(C), "with vs without workspace")
    rows = sampled_rows(M, 16, 9)
    Asub = np.ascontiguousarray(A[:, rows] if transA else A[rows])
    assert_bitwise(host(C[torch.as_tensor(rows, device="cuda")]),
                   oracle.gemm(Asub, B, transA=bool(transA), transB=True), "sampled rows")


@pytest.mark.parametrize("M,N,K", [(300, 200, 1300), (129, 77, 2049), (512, 384, 4096),
                                   (33, 1000, 777)])
@pytest.mark.parametrize("transA,transB", [(0, 0), (1, 0), (0, 1), (1, 1)])
def test_split_k_same_bits(dev, M, N, K, transA, transB):
    assert detlib.detgemm_workspace_bytes(M, N, K, transA, transB) > 0
    run_case(M, N, K, bool(transA), bool(transB), "padded", "padded", "padded",
             M * 31 + K)
    run_case(M, N, K, bool(transA), bool(transB), "offset", "dense", "offset",
             M * 37 + K, wide=True)


def test_crafted_profile_cases(dev):
    # +0 chain start: -1 * 0 -> C = +0
    a = to_dev(np.array([[-1.0]], F))
    b = to_dev(np.array([[0.0]], F))
    assert host(detlib.detgemm_f32(a, b)).view(np.uint32)[0, 0] == 0
    # first partial as is: -2^-100 * 2^-100 underflows to -0 -> C = -0
    a = to_dev(np.array([[-(2.0 ** -100)]], F))
    b = to_dev(np.array([[2.0 ** -100]], F))
    assert host(detlib.detgemm_f32(a, b)).view(np.uint32)[0, 0] == 0x80000000
    # chunk width 256 and left-to-right combine
    K = 768
    a = np.zeros((1, K), F)
    b = np.zeros((K, 1), F)
    a[0, 0] = b[0, 0] = 4096.0
    a[0, 256] = b[256, 0] = 1.0
    a[0, 512] = b[512, 0] = 1.0
    assert host(detlib.detgemm_f32(to_dev(a), to_dev(b)))[0, 0] == F(2.0 ** 24)
    a = np.ones((1, 512), F)
    b = np.ones((512, 1), F)
    a[0, 0] = b[0, 0] = 4096.0
    assert host(detlib.detgemm_f32(to_dev(a), to_dev(b)))[0, 0] == F(2.0 ** 24 + 256)


def test_k_zero_and_empty(dev):
    C = empty_dev(5, 7)
    detlib.detgemm_f32(torch.zeros((5, 0), device="cuda"),
                       torch.zeros((0, 7), device="cuda"), C)
    assert np.all(host(C).view(np.uint32) == 0)
    detlib.detgemm_f32(torch.zeros((0, 3), device="cuda"),
                       torch.zeros((3, 4), device="cuda"))


@pytest.mark.parametrize("cfg", ["cfg1", "cfg2"])
def test_small_configs_in_full(dev, cfg):
    probs = inputs.gemm_cfg1() if cfg == "cfg1" else inputs.gemm_cfg2()
    for p in probs:
        C = detlib.detgemm_f32(to_dev(p["A"]), to_dev(p["B"]), transA=p["transA"],
                               transB=p["transB"])
        want = oracle.gemm(p["A"], p["B"], p["transA"], p["transB"])
        assert_bitwise(host(C), want, f"{cfg}/{p['name']}")


def sampled_rows(M, n, seed):
    rng = np.random.default_rng(seed)
    base = {0, 1, 127, 128, M - 129, M - 1}
    return np.array(sorted(base | set(rng.choice(M, n, replace=False).tolist())))


def check_rows(p, C_dev, rows):
    A, B = p["A"], p["B"]
    Asub = np.ascontiguousarray(A[:, rows] if p["transA"] else A[rows])
    want = oracle.gemm(Asub, B, p["transA"], p["transB"])
    got = host(C_dev[torch.as_tensor(rows, device="cuda")])
    assert_bitwise(got, want, f"{p['name']} rows {rows[:4]}...")


def test_cfg3_full_size_sampled(dev):
    probs = inputs.gemm_cfg3()
    for p in probs:
        M = p["A"].shape[0]
        K = p["A"].shape[1]
        N = p["B"].shape[0] if p["transB"] else p["B"].shape[1]
        ws = detlib.gemm_workspace(M, N, K, p["transA"], p["transB"])
        C = detlib.detgemm_f32(to_dev(p["A"]), to_dev(p["B"]), transA=p["transA"],
                               transB=p["transB"], workspace=ws)
        n = 10 if p["name"] == "lm_head" else 26
        check_rows(p, C, sampled_rows(C.shape[0], n, 3))
        del C


@pytest.mark.parametrize("M,K,transA,transB", [(8000, 2048, 0, 1), (8192, 768, 0, 0),
                                             (7937, 2304, 1, 1)])
def test_unsplit_head_rows_and_split_tail(dev, M, K, transA, transB):
    # 768-wide outputs over 8,000-odd rows fill the 152 SMs once and a little
    # more: the first row blocks that make one round run unsplit in a launch
    # of their own and only the rest is split (only its partials cross HBM);
    # every output keeps detgemm_f32's bits, with or without the workspace,
    # and with beta = 1
    N = 768
    rng = np.random.default_rng(M + K)
    A = rng.standard_normal((K, M) if transA else (M, K)).astype(F)
    B = rng.standard_normal((N, K) if transB else (K, N)).astype(F)
    wsn = detlib.detgemm_workspace_bytes(M, N, K, bool(transA), bool(transB))
    split_alone = detlib.detgemm_launches(M, N, K, bool(transA), bool(transB), wsn)
    assert split_alone >= 3                  # head, tail and its split pass
    ws = detlib.gemm_workspace(M, N, K, bool(transA), bool(transB))
    Ad, Bd = to_dev(A, "padded"), to_dev(B, "padded")
    C = detlib.detgemm_f32(Ad, Bd, transA=bool(transA), transB=bool(transB), workspace=ws)
    C2 = detlib.detgemm_f32(Ad, Bd, transA=bool(transA), transB=bool(transB))
    assert_bitwise(host(C2), host(C), "with vs without workspace")
    rows = np.array(sorted({0, 255, 256, 6143, 6144, 6399, 6400, 6401, 7423, M - 257, M - 1} |
                           set(np.random.default_rng(5).choice(M, 12, replace=False).tolist())))
    Asub = np.ascontiguousarray(A[:, rows] if transA else A[rows])
    want = oracle.gemm(Asub, B, transA=bool(transA), transB=bool(transB))
    assert_bitwise(host(C[torch.as_tensor(rows, device="cuda")]), want, "sampled rows")
    C0 = rng.standard_normal((M, N)).astype(F)
    Cacc = to_dev(C0)
    detlib.detgemm_acc_f32(Ad, Bd, Cacc, transA=bool(transA), transB=bool(transB), workspace=ws)
    assert_bitwise(host(Cacc)[rows], oracle.add(C0[rows], want), "accumulate")


def test_cfg5_dw_full_size_sampled(dev):
    for p in inputs.dw_cfg5():
        M, N, K = p["A"].shape[1], p["B"].shape[1], p["A"].shape[0]
        ws = detlib.gemm_workspace(M, N, K, True, False)
        assert ws is not None
        A, B = to_dev(p["A"]), to_dev(p["B"])
        C = detlib.detgemm_f32(A, B, transA=True, workspace=ws)
        rows = sampled_rows(C.shape[0], 18, 4)
        check_rows(p, C, rows)
        C2 = detlib.detgemm_f32(A, B, transA=True)          # no workspace
        assert_bitwise(host(C2), host(C), p["name"] + " with vs without workspace")


def test_repeatable_across_runs_and_streams(dev):
    rng = np.random.default_rng(9)
    A = to_dev(rng.standard_normal((1000, 1500)).astype(F))
    B = to_dev(rng.standard_normal((1500, 700)).astype(F))
    ref = host(detlib.detgemm_f32(A, B))
    s = torch.cuda.Stream()
    for i in range(4):
        with torch.cuda.stream(s):
            C = detlib.detgemm_f32(A, B)
        s.synchronize()
        assert_bitwise(host(C), ref, f"run {i}")


def test_watchdog_clean(dev):
    torch.cuda.synchronize()
    assert detlib.det_watchdog_status() == 0


# ---------------------------------------------------------------- groups of products
def group_case(shapes, seed, layouts=None):
    """Host operands for products (M, N, K, transA, transB)."""
    rng = np.random.default_rng(seed)
    out = []
    for i, (M, N, K, tA, tB) in enumerate(shapes):
        A = rng.standard_normal((K, M) if tA else (M, K)).astype(F)
        B = rng.standard_normal((N, K) if tB else (K, N)).astype(F)
        la = layouts[i] if layouts else "dense"
        out.append(dict(A=A, B=B, transA=tA, transB=tB, layout=la, M=M, N=N))
    return out


def run_group(case, workspace=True):
    probs = [dict(A=to_dev(c["A"], c["layout"]), B=to_dev(c["B"], c["layout"]),
                  C=empty_dev(c["M"], c["N"], c["layout"]), transA=c["transA"],
                  transB=c["transB"]) for c in case]
    ws = detlib.gemm_group_workspace(probs) if workspace else None
    detlib.detgemm_group_f32(probs, workspace=ws)
    torch.cuda.synchronize()
    return [host(p["C"]) for p in probs]


@pytest.mark.parametrize("shapes", [
    # split pairs (weight-gradient form and plain), an unsplit pair, ragged
    [(300, 200, 1300, True, False), (129, 77, 2049, True, False)],
    [(300, 200, 1300, False, False), (129, 77, 2049, False, False)],
    [(600, 500, 300, True, True), (257, 900, 300, True, True)],
    [(64, 192, 2048, True, False), (64, 64, 2048, True, False), (172, 64, 2048, True, False)],
    # layouts differ: run one after the other
    [(200, 300, 700, True, False), (200, 300, 700, False, True)],
    # an empty product in the middle, and K = 0
    [(100, 0, 300, False, False), (130, 90, 600, False, False), (40, 50, 0, False, False)],
])
def test_group_equals_the_oracle(dev, shapes):
    case = group_case(shapes, 77)
    for use_ws in (True, False):
        got = run_group(case, workspace=use_ws)
        for c, g in zip(case, got):
            want = oracle.gemm(c["A"], c["B"], transA=c["transA"], transB=c["transB"])
            assert_bitwise(g, want, f"{shapes} workspace={use_ws}")


def test_group_plain_load_staging(dev):
    # operands TMA cannot describe (rows one float off a 16-byte boundary)
    case = group_case([(300, 200, 1300, True, False), (129, 77, 2049, True, False)], 78,
                      layouts=["offset", "offset"])
    for c, g in zip(case, run_group(case)):
        assert_bitwise(g, oracle.gemm(c["A"], c["B"], transA=True), "offset layout")


def test_group_cfg5_dw_pair_full_size(dev):
    # the two weight-gradient GEMMs of the 162M step in one call, as the
    # benchmark runs them: sampled rows against the oracle, every bit against
    # detgemm_f32
    ps = inputs.dw_cfg5()
    probs = []
    for p in ps:
        A, B = to_dev(p["A"]), to_dev(p["B"])
        probs.append(dict(A=A, B=B, transA=True, C=torch.empty((p["A"].shape[1], p["B"].shape[1]),
                                                             dtype=torch.float32, device="cuda")))
    ws = detlib.gemm_group_workspace(probs)
    assert ws is not None
    detlib.detgemm_group_f32(probs, workspace=ws)
    for p, q in zip(ps, probs):
        check_rows(p, q["C"], sampled_rows(q["C"].shape[0], 18, 5))
        alone = detlib.detgemm_f32(q["A"], q["B"], transA=True,
                                   workspace=detlib.gemm_workspace(*q["C"].shape,
                                                                   p["A"].shape[0], True, False))
        assert_bitwise(host(q["C"]), host(alone), p["name"] + ": group vs alone")


def test_group_shared_input_takes_one_transposed_copy(dev):
    # two products of one A (the gate and up projections of one input) large
    # enough that each alone would read a transposed copy of A: the group
    # makes one copy for both, and each result is the oracle's
    rng = np.random.default_rng(79)
    M, N, K = 8192, 2048, 768          # the 162M block's gate and up projections
    A = rng.standard_normal((M, K)).astype(F)
    B1 = (0.02 * rng.standard_normal((K, N))).astype(F)
    B2 = (0.02 * rng.standard_normal((K, N))).astype(F)
    Ad = to_dev(A)
    probs = [dict(A=Ad, B=to_dev(B1), C=empty_dev(M, N)), dict(A=Ad, B=to_dev(B2), C=empty_dev(M, N))]
    ws = detlib.gemm_group_workspace(probs)
    assert ws is not None and ws.numel() * 4 >= K * M * 4      # one copy of A
    assert detlib.detgemm_group_launches(probs, ws) == 2       # the copy, one GEMM
    detlib.detgemm_group_f32(probs, workspace=ws)
    torch.cuda.synchronize()
    rows = sampled_rows(M, 24, 6)
    for B, q in zip((B1, B2), probs):
        want = oracle.gemm(np.ascontiguousarray(A[rows]), B)
        assert_bitwise(host(q["C"][torch.as_tensor(rows, device="cuda")]), want, "shared A")
