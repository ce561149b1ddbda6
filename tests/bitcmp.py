"""Bitwise comparison of float32 results (test helper).

Two results agree when every element has the same 32-bit pattern; the only
exception is NaN, where any NaN equals any NaN (NaN payloads are not part of the
profile: hosts and GPUs produce different canonical NaNs). On a mismatch the
report names the first differing element, as a stage-level identity card would.
"""
import hashlib

import numpy as np


def mismatch(a, b):
    """None when a and b agree bitwise (NaN class-equal), else a description
    of the first differing element and the count of differing elements."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32))
    b = np.ascontiguousarray(np.asarray(b, dtype=np.float32))
    if a.shape != b.shape:
        return f"shape {a.shape} != {b.shape}"
    ua = a.view(np.uint32)
    ub = b.view(np.uint32)
    nan_a = np.isnan(a)
    nan_b = np.isnan(b)
    diff = (ua != ub) & ~(nan_a & nan_b)
    n = int(np.count_nonzero(diff))
    if n == 0:
        return None
    idx = np.unravel_index(int(np.flatnonzero(diff)[0]), a.shape)
    return (f"{n} of {a.size} elements differ; first at {tuple(int(i) for i in idx)}: "
            f"{a[idx]!r} (0x{int(ua[idx]):08x}) vs {b[idx]!r} (0x{int(ub[idx]):08x})")


def assert_bitwise(a, b, what=""):
    m = mismatch(a, b)
    assert m is None, f"{what}: {m}"


def card(a) -> str:
    """SHA-256 of the raw bits with every NaN canonicalised."""
    a = np.ascontiguousarray(np.asarray(a, dtype=np.float32)).copy()
    a[np.isnan(a)] = np.float32(np.nan)
    return hashlib.sha256(a.view(np.uint32).tobytes()).hexdigest()
