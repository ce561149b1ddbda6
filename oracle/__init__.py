"""The CPU oracle for the frozen FP32 numerical profile v1 (test infrastructure).

This package is test infrastructure. Only the test suite, the smoke check in
``__graft_entry__`` and the CPU-baseline / reference legs of ``bench.py`` may
import it. The library under ``bitwise_reproducible_fp32_gb300`` never does,
and it shares no code with it.

The arithmetic lives in ``det_oracle.c`` (plain C11, ``fmaf`` and explicit
ordered loops). This module builds it with the host C compiler and marshals
numpy arrays through ctypes. Each function names the page passage it follows in
``det_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "det_oracle.c")
_LIB = os.path.join(_HERE, "libdetoracle.so")

# The profile v1 constants the oracle is driven with. They restate the profile
# (256-wide k-chunks, 32 RMSNorm chains, 256 cross-entropy chains, groups of 4);
# the library receives the same values through its own profile struct.
K_CHUNK = 256
RMS_LANES = 32
XENT_LANES = 256
LANE_GROUP = 4

CFLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
          "-shared", "-Wall"]

_lock = threading.Lock()
_lib = None


def build_variant(defines, out_path: str) -> str:
    """Compile det_oracle.c with extra -D flags into out_path (the test suite's
    separating arms, which plant one mistake each). Never the shipped oracle."""
    cc = os.environ.get("CC", "cc")
    subprocess.run([cc, *CFLAGS, *[f"-D{d}" for d in defines], _SRC, "-o", str(out_path),
                    "-lm", "-lpthread"], check=True)
    return str(out_path)


def build(force: bool = False) -> str:
    """Compile det_oracle.c into libdetoracle.so next to it; return the path."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)
            and os.path.getmtime(_LIB) >= os.path.getmtime(
                os.path.join(_HERE, "det_oracle.h"))):
        return _LIB
    cc = os.environ.get("CC", "cc")
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run([cc, *CFLAGS, _SRC, "-o", tmp, "-lm", "-lpthread"],
                   check=True)
    os.replace(tmp, _LIB)
    return _LIB


def nthreads_default() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        # DET_ORACLE_LIB: load another build of det_oracle.c (a separating arm
        # of the test suite) in place of the shipped one
        lib = ctypes.CDLL(os.environ.get("DET_ORACLE_LIB") or build())
        f32p = ctypes.POINTER(ctypes.c_float)
        i32p = ctypes.POINTER(ctypes.c_int32)
        i64 = ctypes.c_int64
        c_int = ctypes.c_int
        lib.detor_fp_env_ok.restype = c_int
        lib.detor_exp.restype = ctypes.c_float
        lib.detor_exp.argtypes = [ctypes.c_float]
        lib.detor_log.restype = ctypes.c_float
        lib.detor_log.argtypes = [ctypes.c_float]
        lib.detor_exp_n.argtypes = [i64, f32p, f32p, c_int]
        lib.detor_log_n.argtypes = [i64, f32p, f32p, c_int]
        lib.detor_gemm.argtypes = [c_int, c_int, i64, i64, i64, f32p, i64, f32p,
                                   i64, f32p, i64, i64, c_int]
        lib.detor_rmsnorm.argtypes = [i64, i64, f32p, i64, f32p, ctypes.c_float,
                                      f32p, i64, f32p, c_int, c_int, c_int]
        for name in ("detor_sin", "detor_cos"):
            getattr(lib, name).restype = ctypes.c_float
            getattr(lib, name).argtypes = [ctypes.c_float]
        lib.detor_sin_n.argtypes = [i64, f32p, f32p, c_int]
        lib.detor_cos_n.argtypes = [i64, f32p, f32p, c_int]
        lib.detor_rope.argtypes = [i64, i64, i64, f32p, i64, i64, ctypes.c_float, c_int]
        lib.detor_sincos_ulp_scan.restype = ctypes.c_double
        lib.detor_sincos_ulp_scan.argtypes = [c_int, ctypes.c_uint32, ctypes.c_uint32,
                                              ctypes.c_uint32, c_int,
                                              ctypes.POINTER(ctypes.c_uint32)]
        lib.detor_swiglu_bwd.argtypes = [i64, f32p, f32p, f32p, f32p, f32p, c_int]
        lib.detor_softmax_causal_bwd.argtypes = [i64, i64, f32p, f32p, i64, ctypes.c_float,
                                                 i64, f32p, c_int, c_int, c_int]
        lib.detor_rope_bwd.argtypes = [i64, i64, i64, f32p, i64, i64, ctypes.c_float, c_int]
        lib.detor_embedding_bwd.argtypes = [i64, i64, i32p, f32p, i64, f32p, c_int]
        lib.detor_swiglu.argtypes = [i64, f32p, f32p, f32p, c_int]
        lib.detor_add.argtypes = [i64, f32p, f32p, f32p, c_int]
        lib.detor_softmax_causal.argtypes = [i64, i64, f32p, i64, ctypes.c_float, i64, f32p,
                                             i64, c_int, c_int, c_int]
        lib.detor_gemm_acc.argtypes = [c_int, c_int, i64, i64, i64, f32p, i64, f32p,
                                       i64, f32p, i64, i64, c_int]
        lib.detor_shardsum.argtypes = [i64, i64, f32p, i64, ctypes.c_float, f32p, c_int]
        lib.detor_rmsnorm_bwd.argtypes = [i64, i64, f32p, i64, f32p, f32p, f32p, i64,
                                          f32p, i64, f32p, c_int, c_int, i64, c_int]
        lib.detor_xent.restype = i64
        lib.detor_xent.argtypes = [i64, i64, f32p, i64, i32p, f32p, f32p, i64,
                                   ctypes.c_float, c_int, c_int, c_int]
        lib.detor_mean.restype = ctypes.c_float
        lib.detor_mean.argtypes = [i64, f32p, c_int, c_int]
        lib.detor_adamw_bias_correction.argtypes = [
            i64, ctypes.c_float, ctypes.c_float, f32p, f32p]
        lib.detor_adamw.argtypes = [i64, f32p, f32p, f32p, f32p, ctypes.c_float,
                                    ctypes.c_float, ctypes.c_float, ctypes.c_float,
                                    ctypes.c_float, i64, c_int]
        for name in ("detor_exp_ulp_scan", "detor_log_ulp_scan"):
            getattr(lib, name).argtypes = [
                ctypes.c_uint32, ctypes.c_uint32, c_int,
                ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_uint32)]
        if not lib.detor_fp_env_ok():
            raise RuntimeError("host FP environment flushes subnormals or "
                               "widens float evaluation; the oracle refuses")
        _lib = lib
        return lib


def _fp(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_float))


def _f32(a) -> np.ndarray:
    a = np.asarray(a)
    if a.dtype != np.float32:
        raise TypeError(f"oracle takes float32 only, got {a.dtype}")
    return a


def _threads(nthreads):
    return nthreads_default() if nthreads is None else int(nthreads)


# ---------------------------------------------------------------- exp / log
def exp(x, nthreads=None) -> np.ndarray:
    x = np.ascontiguousarray(_f32(x))
    y = np.empty_like(x)
    _load().detor_exp_n(x.size, _fp(x), _fp(y), _threads(nthreads))
    return y


def log(x, nthreads=None) -> np.ndarray:
    x = np.ascontiguousarray(_f32(x))
    y = np.empty_like(x)
    _load().detor_log_n(x.size, _fp(x), _fp(y), _threads(nthreads))
    return y


def exp1(x: float) -> np.float32:
    return np.float32(_load().detor_exp(np.float32(x)))


def log1(x: float) -> np.float32:
    return np.float32(_load().detor_log(np.float32(x)))


def ulp_scan(fn: str, lo_bits: int, hi_bits: int, nthreads=None):
    """(max error in float ulps of the exact result, bit pattern of the worst
    input) of the oracle's exp or log over the given bit-pattern range."""
    lib = _load()
    mx = ctypes.c_double()
    wb = ctypes.c_uint32()
    getattr(lib, f"detor_{fn}_ulp_scan")(lo_bits, hi_bits, _threads(nthreads),
                                          ctypes.byref(mx), ctypes.byref(wb))
    return mx.value, wb.value


# ---------------------------------------------------------------- GEMM
def gemm(A, B, transA=False, transB=False, k_chunk=K_CHUNK, nthreads=None,
         out=None) -> np.ndarray:
    """C = op(A) @ op(B) under the profile; A, B row-major float32 2-D arrays
    (row stride may exceed the row length). op(X) = X.T when trans is set."""
    A = _f32(A)
    B = _f32(B)
    if A.ndim != 2 or B.ndim != 2:
        raise ValueError("2-D operands expected")
    if A.strides[1] != 4 or B.strides[1] != 4:
        A = np.ascontiguousarray(A)
        B = np.ascontiguousarray(B)
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    K2, N = (B.shape[1], B.shape[0]) if transB else B.shape
    if K != K2:
        raise ValueError(f"inner dims differ: {K} vs {K2}")
    C = np.empty((M, N), np.float32) if out is None else out
    _load().detor_gemm(int(transA), int(transB), M, N, K, _fp(A),
                       A.strides[0] // 4, _fp(B), B.strides[0] // 4, _fp(C),
                       C.strides[0] // 4, int(k_chunk), _threads(nthreads))
    return C


def gemm_acc(C, A, B, transA=False, transB=False, k_chunk=K_CHUNK, nthreads=None):
    """C + op(A) op(B) under the profile (beta = 1): a new array."""
    A = np.ascontiguousarray(_f32(A))
    B = np.ascontiguousarray(_f32(B))
    M, K = (A.shape[1], A.shape[0]) if transA else A.shape
    Kb, N = (B.shape[1], B.shape[0]) if transB else B.shape
    assert K == Kb
    out = np.array(_f32(C), dtype=np.float32, order="C", copy=True)
    assert out.shape == (M, N)
    _load().detor_gemm_acc(int(transA), int(transB), M, N, K, _fp(A), A.strides[0] // 4,
                           _fp(B), B.strides[0] // 4, _fp(out), N, int(k_chunk),
                           _threads(nthreads))
    return out


def sin(x, nthreads=None) -> np.ndarray:
    x = np.ascontiguousarray(_f32(x))
    y = np.empty_like(x)
    _load().detor_sin_n(x.size, _fp(x), _fp(y), _threads(nthreads))
    return y


def cos(x, nthreads=None) -> np.ndarray:
    x = np.ascontiguousarray(_f32(x))
    y = np.empty_like(x)
    _load().detor_cos_n(x.size, _fp(x), _fp(y), _threads(nthreads))
    return y


def sincos_ulp_scan(which, lo_bits, hi_bits, step=1, nthreads=None):
    """(max error, worst input bits) of sin (which 0) or cos (1) over the bit
    patterns [lo, hi) stepping by step; ulps of the true value where it is at
    least 2^-6, ulps of 2^-6 nearer the zeros."""
    w = ctypes.c_uint32()
    m = _load().detor_sincos_ulp_scan(which, lo_bits, hi_bits, step, _threads(nthreads),
                                      ctypes.byref(w))
    return m, w.value


def rope(x, heads, head_dim, seq_len, theta=10000.0, nthreads=None):
    """Rotary embedding of the rows of x (rows x heads*head_dim), row t at
    position t mod seq_len: a new array."""
    out = np.array(_f32(x), dtype=np.float32, order="C", copy=True)
    rows = out.shape[0]
    _load().detor_rope(rows, heads, head_dim, _fp(out), out.shape[1], seq_len,
                       np.float32(theta), _threads(nthreads))
    return out


def swiglu(gate, up, nthreads=None):
    """(gate / (1 + exp(-gate))) * up element-wise under the profile."""
    g = np.ascontiguousarray(_f32(gate))
    u = np.ascontiguousarray(_f32(up))
    assert g.shape == u.shape
    out = np.empty_like(g)
    _load().detor_swiglu(g.size, _fp(g), _fp(u), _fp(out), _threads(nthreads))
    return out


def swiglu_bwd(gate, up, dh, nthreads=None):
    """(d_gate, d_up) of h = (g / (1 + exp(-g))) * u under the profile."""
    g = np.ascontiguousarray(_f32(gate))
    u = np.ascontiguousarray(_f32(up))
    d = np.ascontiguousarray(_f32(dh))
    dg, du = np.empty_like(g), np.empty_like(g)
    _load().detor_swiglu_bwd(g.size, _fp(g), _fp(u), _fp(d), _fp(dg), _fp(du),
                             _threads(nthreads))
    return dg, du


def softmax_causal_bwd(p, dp, scale=1.0, diag=0, lanes=XENT_LANES, group=LANE_GROUP,
                       nthreads=None):
    """dS from P and dP (row r keeps columns j <= r + diag)."""
    p = np.ascontiguousarray(_f32(p))
    dp = np.ascontiguousarray(_f32(dp))
    rows, cols = p.shape
    ds = np.empty_like(p)
    _load().detor_softmax_causal_bwd(rows, cols, _fp(p), _fp(dp), cols, np.float32(scale),
                                     int(diag), _fp(ds), lanes, group, _threads(nthreads))
    return ds


def rope_bwd(dy, heads, head_dim, seq_len, theta=10000.0, nthreads=None):
    """The rotary embedding's backward: each pair turned by -a. A new array."""
    out = np.array(_f32(dy), dtype=np.float32, order="C", copy=True)
    _load().detor_rope_bwd(out.shape[0], heads, head_dim, _fp(out), out.shape[1], seq_len,
                           np.float32(theta), _threads(nthreads))
    return out


def embedding_bwd(tokens, dx, vocab, nthreads=None):
    """dE: per id, the left-to-right sum of its tokens' gradient rows."""
    t = np.ascontiguousarray(np.asarray(tokens, np.int32))
    d = np.ascontiguousarray(_f32(dx))
    de = np.empty((vocab, d.shape[1]), np.float32)
    _load().detor_embedding_bwd(t.size, d.shape[1],
                                t.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), _fp(d),
                                vocab, _fp(de), _threads(nthreads))
    return de


def add(a, b, nthreads=None):
    """a + b element-wise, one rounding."""
    a = np.ascontiguousarray(_f32(a))
    b = np.ascontiguousarray(_f32(b))
    assert a.shape == b.shape
    out = np.empty_like(a)
    _load().detor_add(a.size, _fp(a), _fp(b), _fp(out), _threads(nthreads))
    return out


def softmax_causal(s, scale=1.0, diag=0, lanes=XENT_LANES, group=LANE_GROUP, nthreads=None):
    """Row r keeps columns j <= r + diag of s * scale; the profile's softmax
    over them (the cross-entropy's 256-chain sum); masked columns +0."""
    s = np.ascontiguousarray(_f32(s))
    rows, cols = s.shape
    p = np.empty_like(s)
    _load().detor_softmax_causal(rows, cols, _fp(s), cols, np.float32(scale), int(diag),
                                 _fp(p), cols, lanes, group, _threads(nthreads))
    return p


def shardsum(shards, scale=1.0, nthreads=None):
    """scale * (((g_0 + g_1) + g_2) + ...) over the first axis of shards
    (S x n), left to right."""
    g = np.ascontiguousarray(_f32(shards))
    S = g.shape[0]
    flat = g.reshape(S, -1)
    out = np.empty(flat.shape[1], np.float32)
    _load().detor_shardsum(S, flat.shape[1], _fp(flat), flat.shape[1], np.float32(scale),
                           _fp(out), _threads(nthreads))
    return out.reshape(g.shape[1:])


# ---------------------------------------------------------------- RMSNorm
def rmsnorm(x, gain, eps=1e-6, lanes=RMS_LANES, group=LANE_GROUP,
            nthreads=None):
    """(y, inv_rms) for each row of x under the profile."""
    x = _f32(x)
    if x.strides[1] != 4:
        x = np.ascontiguousarray(x)
    gain = np.ascontiguousarray(_f32(gain))
    rows, D = x.shape
    y = np.empty((rows, D), np.float32)
    inv = np.empty(rows, np.float32)
    _load().detor_rmsnorm(rows, D, _fp(x), x.strides[0] // 4, _fp(gain),
                          np.float32(eps), _fp(y), D, _fp(inv), lanes, group,
                          _threads(nthreads))
    return y, inv


def rmsnorm_bwd(x, gain, inv_rms, dy, lanes=RMS_LANES, group=LANE_GROUP,
                k_chunk=K_CHUNK, nthreads=None):
    """(dx, dgain) of RMSNorm under the profile, from the forward's inv_rms
    (det_oracle.c: dx = (h - xhat q) r with h = dy g, xhat = x r and q the
    lane-chain mean of h xhat; dgain = the chunked contraction of dy xhat over
    the rows)."""
    x = np.ascontiguousarray(_f32(x))
    dy = np.ascontiguousarray(_f32(dy))
    gain = np.ascontiguousarray(_f32(gain))
    inv = np.ascontiguousarray(_f32(inv_rms))
    rows, D = x.shape
    assert dy.shape == (rows, D) and gain.shape == (D,) and inv.shape == (rows,)
    dx = np.empty((rows, D), np.float32)
    dgain = np.empty(D, np.float32)
    _load().detor_rmsnorm_bwd(rows, D, _fp(x), D, _fp(gain), _fp(inv), _fp(dy), D,
                              _fp(dx), D, _fp(dgain), lanes, group, int(k_chunk),
                              _threads(nthreads))
    return dx, dgain


# ---------------------------------------------------------------- xent
def xent(logits, labels, with_dlogits=False, dscale=None, lanes=XENT_LANES,
         group=LANE_GROUP, nthreads=None):
    """(loss[rows], dlogits or None, bad_label_count)."""
    x = _f32(logits)
    if x.strides[1] != 4:
        x = np.ascontiguousarray(x)
    labels = np.ascontiguousarray(np.asarray(labels, dtype=np.int32))
    rows, V = x.shape
    loss = np.empty(rows, np.float32)
    d = np.empty((rows, V), np.float32) if with_dlogits else None
    if dscale is None:
        dscale = np.float32(1.0) / np.float32(max(rows, 1))
    dptr = _fp(d) if d is not None else ctypes.POINTER(ctypes.c_float)()
    bad = _load().detor_xent(rows, V, _fp(x), x.strides[0] // 4,
                             labels.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)),
                             _fp(loss), dptr, V, np.float32(dscale), lanes, group,
                             _threads(nthreads))
    return loss, d, int(bad)


def mean(x, lanes=RMS_LANES, group=LANE_GROUP) -> np.float32:
    x = np.ascontiguousarray(_f32(x))
    return np.float32(_load().detor_mean(x.size, _fp(x), lanes, group))


# ---------------------------------------------------------------- AdamW
def adamw_bias_correction(step, beta1, beta2):
    b1 = ctypes.c_float()
    b2 = ctypes.c_float()
    _load().detor_adamw_bias_correction(
        int(step), np.float32(beta1), np.float32(beta2), ctypes.byref(b1),
        ctypes.byref(b2))
    return np.float32(b1.value), np.float32(b2.value)


def adamw(p, g, m, v, lr, beta1, beta2, eps, weight_decay, step,
          nthreads=None):
    """Returns updated copies (p, m, v); the inputs are left untouched."""
    p = np.array(_f32(p), copy=True, order="C")
    m = np.array(_f32(m), copy=True, order="C")
    v = np.array(_f32(v), copy=True, order="C")
    g = np.ascontiguousarray(_f32(g))
    _load().detor_adamw(p.size, _fp(p), _fp(g), _fp(m), _fp(v), np.float32(lr),
                        np.float32(beta1), np.float32(beta2), np.float32(eps),
                        np.float32(weight_decay), int(step), _threads(nthreads))
    return p, m, v
