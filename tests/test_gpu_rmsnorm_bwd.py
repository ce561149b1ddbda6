"""GPU parity (0 ULP) of the RMSNorm backward against the oracle: ragged row
counts around the 256-row chunk grid, widths on both sides of the register
path, every storage layout (TMA tiles and vector rows when aligned, scalar
loads otherwise), in-place dx, crafted rows whose bits fix the chain
arrangement and the chunking, special values, and the full 8192 x 768 shape
in the launch configuration the benchmark uses."""
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


def case(rows, D, seed, scale_dy=1.0):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, D)).astype(F)
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    _, r = oracle.rmsnorm(x, g)
    dy = (scale_dy * rng.standard_normal((rows, D))).astype(F)
    return x, g, r, dy


def run(x, g, r, dy, layout="dense", in_place=False):
    rows, D = x.shape
    xd, dyd = to_dev(x, layout), to_dev(dy, layout)
    dx = dyd if in_place else empty_dev(rows, D, layout)
    dgain = torch.full((D,), float("nan"), device="cuda")
    detlib.detrmsnorm_bwd_f32(xd, to_dev(g), to_dev(r), dyd, dx=dx, dgain=dgain)
    torch.cuda.synchronize()
    return host(dx), host(dgain)


SHAPES = [(1, 1), (3, 5), (7, 37), (256, 128), (257, 768), (300, 130), (513, 1),
          (100, 1024), (65, 1030), (1000, 96), (31, 4100)]


@pytest.mark.parametrize("rows,D", SHAPES)
@pytest.mark.parametrize("layout", ["dense", "padded", "offset"])
def test_shapes_and_layouts(dev, rows, D, layout):
    x, g, r, dy = case(rows, D, rows * 7 + D)
    dx_w, dg_w = oracle.rmsnorm_bwd(x, g, r, dy)
    dx, dg = run(x, g, r, dy, layout)
    assert_bitwise(dx, dx_w, f"dx {rows}x{D} {layout}")
    assert_bitwise(dg, dg_w, f"dgain {rows}x{D} {layout}")


@pytest.mark.parametrize("layout", ["dense", "offset"])
def test_dx_in_place_over_dy(dev, layout):
    x, g, r, dy = case(600, 256, 41)
    dx_w, dg_w = oracle.rmsnorm_bwd(x, g, r, dy)
    dx, dg = run(x, g, r, dy, layout, in_place=True)
    assert_bitwise(dx, dx_w, "dx in place")
    assert_bitwise(dg, dg_w, "dgain")


def test_crafted_chain_butterfly_division_and_chunks(dev):
    # the oracle pins' crafted rows: dot's chain ownership (row 0), its
    # butterfly (row 1), and a column whose chunking decides dgain
    D = 4096
    x = np.zeros((512, D), F)
    for grp in range(0, D // 4, 32):
        x[0, 4 * grp: 4 * grp + 4] = 1.0
    x[0, 0] = 4096.0
    x[1, 0] = 4096.0
    for lane in range(1, 32, 2):
        x[1, 4 * lane] = 1.0
    x[2:, 7] = 1.0
    x[2, 7] = 4096.0
    r = np.ones(512, F)
    g = np.ones(D, F)
    dx_w, dg_w = oracle.rmsnorm_bwd(x, g, r, x.copy())
    dx, dg = run(x, g, r, x.copy(), "padded")
    assert dx[0, 0] == F(4096.0 - 2.0 ** 24) and dx[1, 4] == F(-(4095.0 + 2.0 ** -8))
    assert_bitwise(dx, dx_w, "dx")
    assert_bitwise(dg, dg_w, "dgain")


def test_subnormals_signed_zeros_and_specials(dev):
    x, g, r, dy = case(520, 40, 43)
    x[3] *= F(2.0 ** -100)
    r[3] = F(2.0 ** 90)
    dy[5] *= F(2.0 ** -120)
    x[7, 2] = F(-0.0)
    dy[8, 3] = F(-0.0)
    x[9, 4] = F(np.nan)          # NaN row 9 and column 4's dgain
    dy[10, 5] = F(np.inf)        # inf in row 10 and column 5
    dx_w, dg_w = oracle.rmsnorm_bwd(x, g, r, dy)
    for layout in ("padded", "offset"):
        dx, dg = run(x, g, r, dy, layout)
        assert_bitwise(dx, dx_w, f"dx {layout}")
        assert_bitwise(dg, dg_w, f"dgain {layout}")


def test_zero_rows_write_positive_zero_dgain(dev):
    dgain = torch.full((9,), float("nan"), device="cuda")
    e = torch.empty((0, 9), device="cuda")
    detlib.detrmsnorm_bwd_f32(e, torch.ones(9, device="cuda"),
                              torch.ones(0, device="cuda"), e, dx=e, dgain=dgain)
    assert np.all(host(dgain).view(np.uint32) == 0)


def test_workspace_is_required_past_one_chunk(dev):
    x, g, r, dy = case(300, 8, 44)
    with pytest.raises(detlib.DetError):
        detlib.detrmsnorm_bwd_f32(to_dev(x), to_dev(g), to_dev(r), to_dev(dy),
                                  workspace=torch.empty(3, device="cuda"))


def test_full_size_8192x768(dev):
    f = inputs.rmsnorm_bwd_cfg4()
    y, r = oracle.rmsnorm(f["x"], f["gain"], eps=f["eps"])
    dx_w, dg_w = oracle.rmsnorm_bwd(f["x"], f["gain"], r, f["dy"])
    dx, dg = run(f["x"], f["gain"], r, f["dy"])
    assert_bitwise(dx, dx_w, "dx 8192x768")
    assert_bitwise(dg, dg_w, "dgain 768")
    # the forward's inv_rms from the library gives the same result
    xd = to_dev(f["x"])
    _, rd = detlib.detrmsnorm_f32(xd, to_dev(f["gain"]), float(f["eps"]))
    dx2, dg2 = detlib.detrmsnorm_bwd_f32(xd, to_dev(f["gain"]), rd, to_dev(f["dy"]))
    assert_bitwise(host(dx2), dx_w, "dx from the library's inv_rms")
    assert_bitwise(host(dg2), dg_w, "dgain from the library's inv_rms")


def test_dependent_launches_in_a_chain(dev):
    """Both kernels of the backward launch as programmatic dependents. Here
    each backward takes the previous one's dx as its dy, they share one
    workspace, and the last overwrites the first one's x, with nothing
    synchronised in between: every result must still be the oracle's."""
    rows, D = 8192, 768
    x, g, r, dy = case(rows, D, 91, scale_dy=1e-3)
    w = np.random.default_rng(92).standard_normal((rows, D)).astype(F)
    xd, gd, rd, dyd, wd = to_dev(x), to_dev(g), to_dev(r), to_dev(dy), to_dev(w)
    ws = torch.empty((detlib.detrmsnorm_bwd_workspace_bytes(rows, D) + 3) // 4,
                     dtype=torch.float32, device=xd.device)
    dxs = [torch.empty_like(xd) for _ in range(3)]
    dgs = [torch.empty(D, dtype=torch.float32, device=xd.device) for _ in range(4)]
    src = dyd
    for dx, dg in zip(dxs, dgs):
        detlib.detrmsnorm_bwd_f32(xd, gd, rd, src, dx=dx, dgain=dg, workspace=ws)
        src = dx
    # the last one writes its dx over x, which every launch before it read
    detlib.detrmsnorm_bwd_f32(wd, gd, rd, dyd, dx=xd, dgain=dgs[3], workspace=ws)
    want = dy
    for dx, dg in zip(dxs, dgs):
        want, dg_w = oracle.rmsnorm_bwd(x, g, r, want)
        assert_bitwise(host(dx), want, "dx")
        assert_bitwise(host(dg), dg_w, "dgain")
    dx_w, dg_w = oracle.rmsnorm_bwd(w, g, r, dy)
    assert_bitwise(host(xd), dx_w, "dx over x")
    assert_bitwise(host(dgs[3]), dg_w, "dgain")


def test_repeatable_and_watchdog_clean(dev):
    x, g, r, dy = case(1024, 768, 45, 1e-3)
    ref = run(x, g, r, dy)
    for _ in range(3):
        got = run(x, g, r, dy)
        assert_bitwise(got[0], ref[0])
        assert_bitwise(got[1], ref[1])
    assert detlib.det_watchdog_status() == 0
