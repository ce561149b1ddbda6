"""Input generators for the exp and log tests (no expected values here).

exp_tie_arguments: floats x whose t = fl(x * LOG2E) lands exactly on a tie
k + 1/2 of the round-to-integer step of the profile's exp, and their
neighbours. At those inputs a spelling that rounds t differently (ties away
from zero, no rounding of t, another LOG2E) picks the other n, and the result
moves by an ulp, so they separate the tie rule from its look-alikes.
"""
import numpy as np

F = np.float32
LOG2E = F(1.4426950408889634)


def exp_tie_arguments(kmin: int = -151, kmax: int = 0) -> np.ndarray:
    out = []
    for k in range(kmin, kmax):
        c = F((k + 0.5) / 1.4426950408889634)
        if c == 0:
            continue
        bits = c.view(np.int32) + np.arange(-400, 401, dtype=np.int32)
        d = bits.view(F)
        with np.errstate(over="ignore", invalid="ignore"):
            t = d * LOG2E                  # float32 product, rounded once
        ties = np.nonzero(t == F(k + 0.5))[0]
        for i in ties:
            out.extend(d[max(i - 1, 0):i + 2])
    return np.unique(np.array(out, F))


def binade_samples(seed: int, emin: int, emax: int, per: int, signs=(1, -1)) -> np.ndarray:
    """per random floats in each binade [2^e, 2^(e+1)) for emin <= e <= emax,
    for each sign (normal binades only)."""
    rng = np.random.default_rng(seed)
    out = []
    for e in range(emin, emax + 1):
        mant = rng.integers(0, 1 << 23, per, dtype=np.int64)
        bits = ((e + 127) << 23) | mant
        v = bits.astype(np.uint32).view(F)
        for s in signs:
            out.append(v * F(s))
    return np.concatenate(out)


def reduction_sensitive_arguments(window: float = 2.0 ** -10, per_range: int = 1 << 21,
                                  seed: int = 5) -> np.ndarray:
    """Floats x (far from 0, where |n| is large) whose reduced argument
    r = x - n ln 2, n = rint(fl(x LOG2E)), lies within `window` ulps of a
    rounding midpoint of the float grid. There the rounded r depends on the
    last bits of the ln 2 that the reduction subtracts, so these inputs
    separate the profile's reduction constants and steps from nearby ones.

    r is formed in double with ln 2 split into a 30-bit head (n * head is
    exact) and a double tail: accurate to ~2^-70, far inside the window."""
    rng = np.random.default_rng(seed)
    ln2_hi, ln2_lo = 0.6931471805599453, 2.3190468138462996e-17   # double-double ln 2
    l1 = (np.array([ln2_hi]).view(np.int64) & ~np.int64((1 << 23) - 1)).view(np.float64)[0]
    l2 = (ln2_hi - l1) + ln2_lo
    out = []
    for lo, hi in ((40.0, 88.72), (-103.0, -40.0)):
        x = rng.uniform(lo, hi, per_range).astype(F)
        t = (x * LOG2E).astype(F)
        n = np.rint(t).astype(np.float64)           # half to even
        r = (x.astype(np.float64) - n * l1) - n * l2
        a = np.maximum(np.abs(r), 2.0 ** -140)
        e = np.floor(np.log2(a))
        ulp = np.exp2(np.maximum(e, -126.0) - 23.0)
        frac = a / ulp - np.floor(a / ulp)
        keep = np.abs(frac - 0.5) < window
        out.append(x[keep])
    return np.unique(np.concatenate(out))
