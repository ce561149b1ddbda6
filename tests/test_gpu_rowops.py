"""GPU parity (0 ULP) of RMSNorm, softmax cross-entropy (+ dlogits, + mean),
AdamW and the exp/log spellings against the oracle: ragged and misaligned
rows, edge cases, the full-size workloads, and every float32 input for
exp/log."""
import numpy as np
import pytest

import oracle
from exp_cases import exp_tie_arguments
from bitcmp import assert_bitwise
from bitwise_reproducible_fp32_gb300 import detlib, inputs
from gpu_util import empty_dev, host, need_gpu, to_dev, torch

pytestmark = pytest.mark.gpu
F = np.float32


@pytest.fixture(scope="module")
def dev():
    return need_gpu()


# ----------------------------------------------------------------- RMSNorm
@pytest.mark.parametrize("rows,D", [(1, 1), (3, 3), (5, 4), (7, 127), (64, 768),
                                    (9, 769), (4, 1024), (3, 4096), (2, 5000)])
@pytest.mark.parametrize("layout", ["dense", "padded", "offset"])
def test_rmsnorm_shapes(dev, rows, D, layout):
    rng = np.random.default_rng(rows * 10007 + D)
    x = rng.standard_normal((rows, D)).astype(F)
    x[0, 0] = F(-0.0)
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    y_want, inv_want = oracle.rmsnorm(x, g, eps=1e-6)
    y = empty_dev(rows, D, layout)
    _, inv = detlib.detrmsnorm_f32(to_dev(x, layout), to_dev(g), 1e-6, y=y)
    assert_bitwise(host(y), y_want)
    assert_bitwise(host(inv), inv_want)


def test_rmsnorm_crafted_rows_and_in_place(dev):
    D = 4096
    x = np.zeros((2, D), F)
    for grp in range(0, D // 4, 32):
        x[0, 4 * grp: 4 * grp + 4] = 1.0
    x[0, 0] = 4096.0
    x[1, 0] = 4096.0
    for lane in range(1, 32, 2):
        x[1, 4 * lane] = 1.0
    xd = to_dev(x)
    _, inv = detlib.detrmsnorm_f32(xd, to_dev(np.ones(D, F)), 1e-6, y=xd)  # in place
    inv = host(inv)
    assert inv[0] == F(1 / 64) and inv[1] == F(2.0 ** -6 - 2.0 ** -27)
    y_want, _ = oracle.rmsnorm(x, np.ones(D, F), eps=1e-6)
    assert_bitwise(host(xd), y_want)


def test_streamed_rmsnorm_repeats_bit_for_bit(dev):
    # The streamed RMSNorm (plain and with the fused add) at 8192 x 768, 200
    # launches each on the same inputs: every repeat gives the first one's
    # bits, and the first matches the oracle. A consumer warp that read a ring
    # slot before its copy landed would show here as a repeat that differs.
    rng = np.random.default_rng(77)
    a = rng.standard_normal((8192, 768)).astype(F)
    b = rng.standard_normal((8192, 768)).astype(F)
    g = (1 + 0.02 * rng.standard_normal(768)).astype(F)
    ad, bd, gd = to_dev(a), to_dev(b), to_dev(g)
    y0, _ = detlib.detrmsnorm_f32(ad, gd, 1e-6)
    x1, y1, _ = detlib.detadd_rmsnorm_f32(ad, bd, gd, 1e-6)
    y0, x1, y1 = y0.clone(), x1.clone(), y1.clone()
    y, xs, ys = torch.empty_like(y0), torch.empty_like(x1), torch.empty_like(y1)
    bad = torch.zeros((), dtype=torch.int64, device="cuda")
    for _ in range(200):
        detlib.detrmsnorm_f32(ad, gd, 1e-6, y=y)
        detlib.detadd_rmsnorm_f32(ad, bd, gd, 1e-6, x=xs, y=ys)
        bad += (y.view(torch.int32) != y0.view(torch.int32)).sum()
        bad += (xs.view(torch.int32) != x1.view(torch.int32)).sum()
        bad += (ys.view(torch.int32) != y1.view(torch.int32)).sum()
    assert int(bad) == 0
    assert_bitwise(host(y0), oracle.rmsnorm(a, g, eps=1e-6)[0])
    x_want = oracle.add(a, b)
    assert_bitwise(host(x1), x_want)
    assert_bitwise(host(y1), oracle.rmsnorm(x_want, g, eps=1e-6)[0])


@pytest.mark.parametrize("rows,D,offset", [(8192, 768, 0), (1000, 768, 0), (7, 4096, 0),
                                           (33, 130, 0), (64, 768, 1), (3, 4, 0)])
def test_add_rmsnorm_equals_add_then_rmsnorm(dev, rows, D, offset):
    # x = a + b and y = RMSNorm(x) in one call: the fused streamed kernel for
    # aligned rows with D a multiple of 4, the two operations apart otherwise
    # (D = 130, or rows one float past a 16-byte boundary); the bits of
    # detadd_f32 then detrmsnorm_f32
    rng = np.random.default_rng(rows + D + offset)
    a = rng.standard_normal((rows, D)).astype(F)
    b = rng.standard_normal((rows, D)).astype(F)
    a[0, :3] = [np.inf, -np.inf, 0.0]
    b[0, :3] = [1.0, 2.0, -0.0]
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    x_want = oracle.add(a, b)
    y_want, inv_want = oracle.rmsnorm(x_want, g, eps=1e-6)

    def dense(m):
        buf = torch.full((m.size + 4,), float("nan"), device="cuda")
        buf[offset:offset + m.size] = torch.from_numpy(m.ravel()).cuda()
        return buf[offset:offset + m.size].view(rows, D)
    x, y, inv = detlib.detadd_rmsnorm_f32(dense(a), dense(b), to_dev(g), 1e-6,
                                          x=dense(np.zeros_like(a)))
    assert_bitwise(host(x), x_want)
    assert_bitwise(host(y), y_want)
    assert_bitwise(host(inv), inv_want)


def test_rmsnorm_cfg4_full(dev):
    r = inputs.rowops_cfg4(vocab=8)   # x and gain as in the full config
    y, inv = detlib.detrmsnorm_f32(to_dev(r["x"]), to_dev(r["gain"]), float(r["eps"]))
    y_want, inv_want = oracle.rmsnorm(r["x"], r["gain"], eps=r["eps"])
    assert_bitwise(host(y), y_want)
    assert_bitwise(host(inv), inv_want)


def test_rmsnorm_dependent_launches_in_a_chain(dev):
    """RMSNorm launches as a programmatic dependent of the launch before it.
    Each of these reads what the one before wrote (y1 = RMSNorm(x), y2 =
    RMSNorm(y1), ...), and the last overwrites the first one's input while
    nothing is synchronised in between: every result must still be the
    oracle's, which holds only if each launch waits for the previous grid
    before it reads or writes."""
    rows, D = 8192, 768            # the streamed kernel: one CTA an SM
    rng = np.random.default_rng(77)
    x = rng.standard_normal((rows, D)).astype(F)
    g = (1 + 0.02 * rng.standard_normal(D)).astype(F)
    w = rng.standard_normal((rows, D)).astype(F)
    xd, gd, wd = to_dev(x), to_dev(g), to_dev(w)
    ys = [torch.empty_like(xd) for _ in range(4)]
    invs = [torch.empty(rows, dtype=torch.float32, device=xd.device) for _ in range(5)]
    src = xd
    for y, inv in zip(ys, invs):
        detlib.detrmsnorm_f32(src, gd, 1e-6, y=y, inv_rms=inv)
        src = y
    detlib.detrmsnorm_f32(wd, gd, 1e-6, y=xd, inv_rms=invs[4])   # overwrites x
    want = x
    for y, inv in zip(ys, invs):
        want, inv_want = oracle.rmsnorm(want, g, eps=1e-6)
        assert_bitwise(host(y), want)
        assert_bitwise(host(inv), inv_want)
    wy, winv = oracle.rmsnorm(w, g, eps=1e-6)
    assert_bitwise(host(xd), wy)
    assert_bitwise(host(invs[4]), winv)


# ----------------------------------------------------------------- cross-entropy
@pytest.mark.parametrize("rows,V", [(1, 1), (3, 2), (5, 5), (4, 255), (7, 1024),
                                    (6, 1025), (5, 1601), (3, 7777), (3, 50257)])
@pytest.mark.parametrize("layout", ["dense", "offset"])
def test_xent_shapes(dev, rows, V, layout):
    rng = np.random.default_rng(rows * 7919 + V)
    x = (2 * rng.standard_normal((rows, V))).astype(F)
    lab = rng.integers(0, V, size=rows, dtype=np.int32)
    loss_w, d_w, bad = oracle.xent(x, lab, with_dlogits=True, dscale=F(1 / rows))
    assert bad == 0
    d = empty_dev(rows, V, layout)
    loss, mean, _ = detlib.detxent_f32(to_dev(x, layout), to_dev(lab), want_mean=True,
                                       dlogits=d, dscale=float(F(1 / rows)))
    assert_bitwise(host(loss), loss_w)
    assert_bitwise(host(d), d_w)
    assert_bitwise(host(mean), np.array([oracle.mean(loss_w)], F))


def test_xent_bad_labels_nan_inf_rows_and_status(dev):
    rng = np.random.default_rng(77)
    rows, V = 6, 3000
    x = rng.standard_normal((rows, V)).astype(F)
    x[2, 17] = F(np.nan)        # NaN row -> NaN loss and dlogits
    x[3, 5] = F(np.inf)         # +Inf -> inf - inf = NaN
    x[4, :] = F(-np.inf)
    x[4, 9] = F(1.0)            # -Inf logits give e = 0
    lab = rng.integers(0, V, size=rows, dtype=np.int32)
    lab[1] = V                  # out of range
    lab[5] = -3
    loss_w, d_w, bad = oracle.xent(x, lab, with_dlogits=True)
    assert bad == 2
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    loss, _, d = detlib.detxent_f32(to_dev(x), to_dev(lab), want_dlogits=True,
                                    dev_status=status)
    assert_bitwise(host(loss), loss_w)
    assert_bitwise(host(d), d_w)
    assert int(host(status)[0]) == 1
    # a clean call leaves the caller's status word as it was
    lab2 = np.clip(lab, 0, V - 1).astype(np.int32)
    status.zero_()
    detlib.detxent_f32(to_dev(x), to_dev(lab2), dev_status=status)
    assert int(host(status)[0]) == 0


@pytest.mark.parametrize("lx,ld_", [("dense", "offset"), ("offset", "dense"),
                                     ("padded", "offset")])
def test_xent_logits_and_dlogits_aligned_differently(dev, lx, ld_):
    rng = np.random.default_rng(79)
    rows, V = 9, 2051
    x = (2 * rng.standard_normal((rows, V))).astype(F)
    lab = rng.integers(0, V, size=rows, dtype=np.int32)
    loss_w, d_w, _ = oracle.xent(x, lab, with_dlogits=True, dscale=F(0.25))
    d = empty_dev(rows, V, ld_)
    loss, _, _ = detlib.detxent_f32(to_dev(x, lx), to_dev(lab), dlogits=d, dscale=0.25)
    assert_bitwise(host(loss), loss_w)
    assert_bitwise(host(d), d_w)


def test_xent_deep_underflow_row(dev):
    # logits spread so that x - m runs through the subnormal and zero range
    V = 4099
    x = np.linspace(0.0, -120.0, V, dtype=F)[None, :].repeat(3, axis=0)
    x[1] = x[1][::-1]
    x[2, ::7] = F(-np.inf)
    x[2, 1] = F(0.0)
    lab = np.array([0, V - 1, 1], np.int32)
    loss_w, d_w, _ = oracle.xent(x, lab, with_dlogits=True)
    loss, _, d = detlib.detxent_f32(to_dev(x), to_dev(lab), want_dlogits=True)
    assert_bitwise(host(loss), loss_w)
    assert_bitwise(host(d), d_w)


def test_xent_exp_rounding_ties(dev):
    d = exp_tie_arguments()
    assert d.size > 100
    # known inputs where one spelling of the packed exp went one ulp off
    # (row max 0, and row max 7.25)
    extra = np.array([0xc2a70c69, 0xc2490340, 0xc283013c, 0xc14214ca, 0xc25f3183,
                      0xc0d2b77c, 0xc158430d, 0xc16e7150], np.uint32).view(F)
    extra2 = np.array([0xc29463bc, 0xc29300d8, 0xc0f4e2a0, 0xc0f4e2a1, 0xc0f4e29f,
                       0xc2988c69, 0xc22c0340, 0xc09c2994], np.uint32).view(F)
    V = d.size + extra.size + 1
    x = np.zeros((2, V), F)
    x[0, 1:] = np.concatenate([d, extra])
    x[1, 0] = F(7.25)
    x[1, 1:] = np.concatenate([d + F(7.25), extra2, np.full(extra.size - extra2.size, -1.0, F)])
    lab = np.array([0, 3], np.int32)
    loss_w, d_w, _ = oracle.xent(x, lab, with_dlogits=True)
    for dscale in (1.0, 0.375):
        loss, _, dl = detlib.detxent_f32(to_dev(x), to_dev(lab), want_dlogits=True,
                                         dscale=dscale)
        loss_w, d_w, _ = oracle.xent(x, lab, with_dlogits=True, dscale=F(dscale))
        assert_bitwise(host(loss), loss_w, f"loss dscale={dscale}")
        assert_bitwise(host(dl), d_w, f"dlogits dscale={dscale}")


def test_xent_exp_ties_rows_without_underflow(dev):
    # the ties of rint(d LOG2E) in rows whose every x - m is >= -86 (no element
    # near underflow), max 0 and max 7.25
    d = exp_tie_arguments()
    d = d[d >= F(-85.9)]
    assert d.size > 100
    V = d.size + 1
    x = np.zeros((2, V), F)
    x[0, 1:] = d
    x[1, 0] = F(7.25)
    x[1, 1:] = d + F(7.25)
    assert (x[1, 1:] - x[1, 0]).min() >= -86.0
    lab = np.array([0, 5], np.int32)
    loss_w, d_w, _ = oracle.xent(x, lab, with_dlogits=True, dscale=F(1.0))
    loss, _, dl = detlib.detxent_f32(to_dev(x), to_dev(lab), want_dlogits=True, dscale=1.0)
    assert_bitwise(host(loss), loss_w)
    assert_bitwise(host(dl), d_w)


@pytest.mark.parametrize("layout", ["dense", "offset"])
def test_xent_rows_longer_than_shared_memory(dev, layout):
    # rows of more than ~57,600 floats take the register/L2 kernel
    rng = np.random.default_rng(81)
    rows, V = 3, 60001
    x = (2 * rng.standard_normal((rows, V))).astype(F)
    x[1, 7] = F(-np.inf)
    lab = np.array([0, V - 1, 31337], np.int32)
    loss_w, d_w, _ = oracle.xent(x, lab, with_dlogits=True)
    d = empty_dev(rows, V, layout)
    loss, _, _ = detlib.detxent_f32(to_dev(x, layout), to_dev(lab), dlogits=d,
                                    dscale=float(F(1 / rows)))
    assert_bitwise(host(loss), loss_w)
    assert_bitwise(host(d), d_w)


def test_xent_dlogits_in_place(dev):
    rng = np.random.default_rng(78)
    x = (2 * rng.standard_normal((4, 777))).astype(F)
    lab = rng.integers(0, 777, size=4, dtype=np.int32)
    loss_w, d_w, _ = oracle.xent(x, lab, with_dlogits=True)
    xd = to_dev(x)
    loss, _, _ = detlib.detxent_f32(xd, to_dev(lab), dlogits=xd)
    assert_bitwise(host(loss), loss_w)
    assert_bitwise(host(xd), d_w)


def test_xent_cfg4_full(dev):
    r = inputs.rowops_cfg4()
    loss, mean, d = detlib.detxent_f32(to_dev(r["logits"]), to_dev(r["labels"]),
                                       want_mean=True, want_dlogits=True)
    loss_w, d_w, bad = oracle.xent(r["logits"], r["labels"], with_dlogits=True)
    assert bad == 0
    assert_bitwise(host(loss), loss_w, "loss")
    assert_bitwise(host(mean), np.array([oracle.mean(loss_w)], F), "mean")
    assert_bitwise(host(d), d_w, "dlogits")


# ----------------------------------------------------------------- AdamW
@pytest.mark.parametrize("n", [1, 3, 4, 5, 1000, 1001, (1 << 20) + 3])
@pytest.mark.parametrize("step", [1, 2, 251, 20000])
def test_adamw_shapes(dev, n, step):
    rng = np.random.default_rng(n + step)
    p = (0.02 * rng.standard_normal(n)).astype(F)
    g = (1e-3 * rng.standard_normal(n)).astype(F)
    m = (1e-3 * rng.standard_normal(n)).astype(F)
    v = ((1e-3 * rng.standard_normal(n)) ** 2).astype(F)
    g[0] = F(0.0)
    hp = dict(lr=6e-4, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1, step=step)
    pw, mw, vw = oracle.adamw(p, g, m, v, **hp)
    for offset in (0, 1):
        def put(a):
            buf = torch.empty(n + offset, dtype=torch.float32, device="cuda")
            buf[offset:] = torch.from_numpy(a).cuda()
            return buf[offset:]
        pd, gd, md, vd = put(p), put(g), put(m), put(v)
        detlib.detadamw_f32(pd, gd, md, vd, **hp)
        assert_bitwise(host(pd), pw, f"p offset={offset}")
        assert_bitwise(host(md), mw, f"m offset={offset}")
        assert_bitwise(host(vd), vw, f"v offset={offset}")


def test_adamw_cfg5_full(dev):
    a = inputs.adamw_cfg5()
    hp = {k: a[k] for k in ("lr", "beta1", "beta2", "eps", "weight_decay", "step")}
    pd, gd, md, vd = (to_dev(a[k]) for k in ("p", "g", "m", "v"))
    detlib.detadamw_f32(pd, gd, md, vd, **hp)
    pw, mw, vw = oracle.adamw(a["p"], a["g"], a["m"], a["v"], **hp)
    assert_bitwise(host(pd), pw, "p")
    assert_bitwise(host(md), mw, "m")
    assert_bitwise(host(vd), vw, "v")


# ----------------------------------------------------------------- exp / log
def test_exp_log_every_float(dev):
    chunk = 1 << 26
    for start in range(0, 1 << 32, chunk):
        bits = np.arange(start, start + chunk, dtype=np.uint64).astype(np.uint32)
        x = bits.view(F)
        xd = torch.from_numpy(x).cuda()
        ye = host(detlib.detexp_f32(xd))
        assert_bitwise(ye, oracle.exp(x), f"exp chunk {start:#x}")
        yl = host(detlib.detlog_f32(xd))
        assert_bitwise(yl, oracle.log(x), f"log chunk {start:#x}")


# ----------------------------------------------------------------- identity cards
def test_identity_cards_on_this_host_and_gpu(dev):
    """The frozen cards reproduce with the oracle built on this host, and the
    GPU's outputs for the same workloads carry the same cards."""
    import json, os, sys
    from bitcmp import card
    golden = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
    sys.path.insert(0, golden)
    import make_identity_cards as mk
    want = json.load(open(os.path.join(golden, "identity_cards_v1.json")))["cards"]
    assert mk.cards() == want
    got = {}
    for p in inputs.gemm_cfg1():
        got[f"cfg1/{p['name']}"] = card(host(detlib.detgemm_f32(to_dev(p["A"]), to_dev(p["B"]))))
    for p in inputs.gemm_cfg2():
        got[f"cfg2/{p['name']}"] = card(host(detlib.detgemm_f32(
            to_dev(p["A"]), to_dev(p["B"]), transA=p["transA"], transB=p["transB"])))
    for p in inputs.gemm_cfg3(tokens=64, d=96, dff=128, vocab=1000):
        got[f"cfg3_small/{p['name']}"] = card(host(detlib.detgemm_f32(
            to_dev(p["A"]), to_dev(p["B"]), transA=p["transA"], transB=p["transB"])))
    r = inputs.rowops_cfg4(rows=32, d=768, vocab=5003)
    y, inv = detlib.detrmsnorm_f32(to_dev(r["x"]), to_dev(r["gain"]), float(r["eps"]))
    got["cfg4_small/rmsnorm_y"] = card(host(y))
    got["cfg4_small/rmsnorm_inv_rms"] = card(host(inv))
    loss, mean, d = detlib.detxent_f32(to_dev(r["logits"]), to_dev(r["labels"]),
                                       want_mean=True, want_dlogits=True)
    got["cfg4_small/xent_loss"] = card(host(loss))
    got["cfg4_small/xent_dlogits"] = card(host(d))
    got["cfg4_small/xent_loss_mean"] = card(host(mean)[0])
    for p in inputs.dw_cfg5(tokens=600, d=64, dff=96):
        got[f"cfg5_small/{p['name']}"] = card(host(detlib.detgemm_f32(
            to_dev(p["A"]), to_dev(p["B"]), transA=True)))
    a = inputs.adamw_cfg5(n=100_003)
    pd, gd, md, vd = (to_dev(a[k]) for k in ("p", "g", "m", "v"))
    detlib.detadamw_f32(pd, gd, md, vd, a["lr"], a["beta1"], a["beta2"], a["eps"],
                        a["weight_decay"], a["step"])
    got["cfg5_small/adamw_p"] = card(host(pd))
    got["cfg5_small/adamw_m"] = card(host(md))
    got["cfg5_small/adamw_v"] = card(host(vd))
    # the cfg cards; the byte-level LM's stage cards are checked in its own test
    mine = [k for k in want if k.startswith("cfg")]
    assert set(mine) == set(got)
    diff = sorted(k for k in mine if got[k] != want[k])
    assert not diff, diff
