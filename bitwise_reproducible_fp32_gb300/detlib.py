"""ctypes binding over libdetfp32.so (include/detfp32.h).

Argument marshalling only: each function takes torch CUDA tensors, reads their
shapes, strides, data pointers and the current stream, and calls the C entry
point of the same name. All arithmetic runs in the library's kernels. A missing
library, a CPU tensor or a non-OK status raises; nothing falls back to another
implementation.
"""
from __future__ import annotations

import ctypes
import os
import threading

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libdetfp32.so")

DET_OK = 0
STATUS_NAMES = {0: "DET_OK", 1: "DET_ERR_INVALID_ARG", 2: "DET_ERR_PROFILE",
                3: "DET_ERR_UNSUPPORTED_DEVICE", 4: "DET_ERR_ALIGNMENT",
                5: "DET_ERR_WORKSPACE", 6: "DET_ERR_TIMEOUT", 7: "DET_ERR_CUDA"}


class DetError(RuntimeError):
    def __init__(self, fn, status, msg):
        super().__init__(f"{fn}: {msg}")
        self.status = status


class Profile(ctypes.Structure):
    """det_profile_v1."""
    _fields_ = [("version", ctypes.c_uint32), ("k_chunk", ctypes.c_uint32),
                ("rms_lanes", ctypes.c_uint32), ("xent_lanes", ctypes.c_uint32),
                ("lane_group", ctypes.c_uint32), ("flags", ctypes.c_uint32)]


class GemmProblem(ctypes.Structure):
    """det_gemm_problem."""
    _fields_ = [("transA", ctypes.c_int), ("transB", ctypes.c_int),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64),
                ("A", ctypes.c_void_p), ("lda", ctypes.c_int64),
                ("B", ctypes.c_void_p), ("ldb", ctypes.c_int64),
                ("C", ctypes.c_void_p), ("ldc", ctypes.c_int64)]


class AdamWHP(ctypes.Structure):
    """det_adamw_hp."""
    _fields_ = [("lr", ctypes.c_float), ("beta1", ctypes.c_float),
                ("beta2", ctypes.c_float), ("eps", ctypes.c_float),
                ("weight_decay", ctypes.c_float), ("step", ctypes.c_int64)]


_lock = threading.Lock()
_lib = None

# (name, restype, argtypes) of every exported function
_vp, _i64, _int, _f = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
_PROF = ctypes.POINTER(Profile)
SIGNATURES = [
    ("det_profile_default", None, [_PROF]),
    ("det_status_string", ctypes.c_char_p, [_int]),
    ("detgemm_f32", _int, [_PROF, _int, _int, _i64, _i64, _i64, _vp, _i64, _vp, _i64,
                           _vp, _i64, _vp, ctypes.c_size_t, _vp]),
    ("detgemm_acc_f32", _int, [_PROF, _int, _int, _i64, _i64, _i64, _vp, _i64, _vp, _i64,
                               _vp, _i64, _vp, ctypes.c_size_t, _vp]),
    ("detshardsum_f32", _int, [_PROF, _i64, _i64, _vp, _i64, _f, _vp, _vp]),
    ("detgemm_workspace_bytes", _int, [_PROF, _int, _int, _i64, _i64, _i64,
                                       ctypes.POINTER(ctypes.c_size_t)]),
    ("detgemm_group_f32", _int, [_PROF, _i64, ctypes.POINTER(GemmProblem), _vp,
                                 ctypes.c_size_t, _vp]),
    ("detgemm_group_workspace_bytes", _int, [_PROF, _i64, ctypes.POINTER(GemmProblem),
                                             ctypes.POINTER(ctypes.c_size_t)]),
    ("detgemm_launches", _int, [_PROF, _int, _int, _i64, _i64, _i64, ctypes.c_size_t,
                                ctypes.POINTER(ctypes.c_int64)]),
    ("detgemm_group_launches", _int, [_PROF, _i64, ctypes.POINTER(GemmProblem),
                                      ctypes.c_size_t, ctypes.POINTER(ctypes.c_int64)]),
    ("detgemm_f32_noalloc", _int, [_PROF, _int, _int, _i64, _i64, _i64, _vp, _i64, _vp,
                                   _i64, _vp, _i64, _vp]),
    ("detrmsnorm_f32", _int, [_PROF, _i64, _i64, _vp, _i64, _vp, _f, _vp, _i64, _vp,
                              _vp]),
    ("detrmsnorm_bwd_f32", _int, [_PROF, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _i64, _vp,
                                  _i64, _vp, _vp, ctypes.c_size_t, _vp]),
    ("detrmsnorm_bwd_workspace_bytes", _int, [_PROF, _i64, _i64,
                                              ctypes.POINTER(ctypes.c_size_t)]),
    ("detxent_f32", _int, [_PROF, _i64, _i64, _vp, _i64, _vp, _vp, _vp, _vp, _i64, _f,
                           _vp, _vp]),
    ("det_adamw_bias_correction", _int, [_i64, _f, _f, ctypes.POINTER(_f),
                                         ctypes.POINTER(_f)]),
    ("detadamw_f32", _int, [_PROF, _i64, _vp, _vp, _vp, _vp, ctypes.POINTER(AdamWHP),
                            _vp]),
    ("detexp_f32", _int, [_PROF, _i64, _vp, _vp, _vp]),
    ("detlog_f32", _int, [_PROF, _i64, _vp, _vp, _vp]),
    ("detswiglu_f32", _int, [_PROF, _i64, _vp, _vp, _vp, _vp]),
    ("detadd_f32", _int, [_PROF, _i64, _vp, _vp, _vp, _vp]),
    ("detadd_rmsnorm_f32", _int, [_PROF, _i64, _i64, _vp, _vp, _vp, _vp, _f, _vp, _i64, _vp,
                                  _vp]),
    ("detsoftmax_causal_f32", _int, [_PROF, _i64, _i64, _vp, _i64, _f, _i64, _i64, _vp, _i64,
                                     _vp]),
    ("detrope_f32", _int, [_PROF, _i64, _i64, _i64, _vp, _i64, _i64, _f, _vp]),
    ("detembedding_f32", _int, [_PROF, _i64, _i64, _vp, _i64, _i64, _vp, _vp, _i64, _vp, _vp]),
    ("detsin_f32", _int, [_PROF, _i64, _vp, _vp, _vp]),
    ("detcos_f32", _int, [_PROF, _i64, _vp, _vp, _vp]),
    ("detattention_f32", _int, [_PROF, _i64, _i64, _i64, _i64, _vp, _i64, _f, _vp, _i64, _vp,
                                ctypes.c_size_t, _vp]),
    ("detattention_workspace_bytes", _int, [_PROF, _i64, _i64, _i64, _i64,
                                            ctypes.POINTER(ctypes.c_size_t)]),
    ("detattention_launches", _int, [_PROF, _i64, _i64, _i64, _i64, ctypes.c_int,
                                     ctypes.POINTER(ctypes.c_int64)]),
    ("detswiglu_bwd_f32", _int, [_PROF, _i64, _vp, _vp, _vp, _vp, _vp, _vp]),
    ("detsoftmax_causal_bwd_f32", _int, [_PROF, _i64, _i64, _vp, _vp, _i64, _f, _i64, _i64,
                                         _vp, _i64, _vp]),
    ("detrope_bwd_f32", _int, [_PROF, _i64, _i64, _i64, _vp, _i64, _i64, _f, _vp]),
    ("detembedding_bwd_f32", _int, [_PROF, _i64, _i64, _vp, _vp, _i64, _i64, _vp, _i64, _vp]),
    ("detattention_bwd_f32", _int, [_PROF, _i64, _i64, _i64, _i64, _vp, _i64, _vp, _i64, _f,
                                    _vp, _i64, _vp, ctypes.c_size_t, _vp]),
    ("detattention_bwd_workspace_bytes", _int, [_PROF, _i64, _i64, _i64, _i64,
                                                ctypes.POINTER(ctypes.c_size_t)]),
    ("detattention_bwd_saved_f32", _int, [_PROF, _i64, _i64, _i64, _i64, _vp, _i64, _vp,
                                          _i64, _f, _vp, ctypes.c_size_t, _vp, _i64, _vp,
                                          ctypes.c_size_t, _vp]),
    ("det_watchdog_status", _int, [ctypes.POINTER(ctypes.c_int32), _int]),
]


def load(path: str = LIB_PATH):
    """Loads the library (once). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with "
                "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(path)
        for name, res, args in SIGNATURES:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def det_profile_default() -> Profile:
    p = Profile()
    load().det_profile_default(ctypes.byref(p))
    return p


def det_status_string(status: int) -> str:
    return load().det_status_string(int(status)).decode()


def _check(fn: str, status: int):
    if status != DET_OK:
        raise DetError(fn, status, det_status_string(status))


def _prof(profile):
    return ctypes.byref(profile if profile is not None else det_profile_default())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p()


def _cuda_f32(t, name, ndim=None):
    import torch
    if not isinstance(t, torch.Tensor) or t.device.type != "cuda":
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.float32:
        raise TypeError(f"{name} must be float32 (the profile is FP32 only), got {t.dtype}")
    if ndim is not None and t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D")
    if ndim == 2 and t.numel() > 0 and t.stride(1) != 1:
        raise ValueError(f"{name} rows must be contiguous (stride(1) == 1)")
    if ndim in (None, 1) and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def _ld(t):
    # an empty matrix has no row stride to speak of: report its row length
    return t.stride(0) if t.dim() == 2 and t.numel() > 0 else max(t.shape[-1], 1)


# ---------------------------------------------------------------- GEMM
def detgemm_workspace_bytes(M, N, K, transA=False, transB=False, profile=None) -> int:
    n = ctypes.c_size_t()
    _check("detgemm_workspace_bytes",
           load().detgemm_workspace_bytes(_prof(profile), int(bool(transA)),
                                          int(bool(transB)), int(M), int(N), int(K),
                                          ctypes.byref(n)))
    return n.value


def detgemm_launches(M, N, K, transA=False, transB=False, workspace=None,
                     profile=None) -> int:
    """Kernel launches detgemm_f32 makes for this shape with this workspace (a
    tensor, a size in bytes, or None)."""
    n = ctypes.c_int64()
    if workspace is None:
        wsn = 0
    elif isinstance(workspace, int):
        wsn = workspace
    else:
        wsn = workspace.numel() * 4
    _check("detgemm_launches",
           load().detgemm_launches(_prof(profile), int(bool(transA)), int(bool(transB)),
                                   int(M), int(N), int(K), wsn, ctypes.byref(n)))
    return n.value


def gemm_workspace(M, N, K, transA=False, transB=False, device="cuda"):
    """A caller-owned workspace tensor of the size detgemm_f32 can use for
    this shape (None when it needs none)."""
    import torch
    n = detgemm_workspace_bytes(M, N, K, transA, transB)
    if n == 0:
        return None
    return torch.empty((n + 3) // 4, dtype=torch.float32, device=device)


def detgemm_f32(A, B, C=None, transA=False, transB=False, workspace=None, profile=None,
                stream=None):
    """C = op(A) @ op(B) under the profile. A, B row-major 2-D float32 CUDA
    tensors (transA: A is K x M; transB: B is N x K). workspace: optional
    float32 CUDA tensor (see gemm_workspace); the bits do not depend on it.
    Returns C."""
    import torch
    _cuda_f32(A, "A", 2)
    _cuda_f32(B, "B", 2)
    M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
    Kb, N = (B.shape[1], B.shape[0]) if transB else (B.shape[0], B.shape[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
    _cuda_f32(C, "C", 2)
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {M} x {N}")
    ws_ptr, ws_bytes = ctypes.c_void_p(), 0
    if workspace is not None:
        _cuda_f32(workspace, "workspace")
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * 4
    st = load().detgemm_f32(_prof(profile), int(bool(transA)), int(bool(transB)), M, N,
                            K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C),
                            ws_ptr, ws_bytes, _stream(stream))
    _check("detgemm_f32", st)
    return C


def detgemm_acc_f32(A, B, C, transA=False, transB=False, workspace=None, profile=None,
                    stream=None):
    """C = C + op(A) @ op(B) (beta = 1) under the profile, in place. Returns C."""
    _cuda_f32(A, "A", 2)
    _cuda_f32(B, "B", 2)
    _cuda_f32(C, "C", 2)
    M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
    Kb, N = (B.shape[1], B.shape[0]) if transB else (B.shape[0], B.shape[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {M} x {N}")
    ws_ptr, ws_bytes = ctypes.c_void_p(), 0
    if workspace is not None:
        _cuda_f32(workspace, "workspace")
        ws_ptr, ws_bytes = _ptr(workspace), workspace.numel() * 4
    st = load().detgemm_acc_f32(_prof(profile), int(bool(transA)), int(bool(transB)), M, N,
                                K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C), _ld(C),
                                ws_ptr, ws_bytes, _stream(stream))
    _check("detgemm_acc_f32", st)
    return C


def detshardsum_f32(shards, scale=1.0, out=None, profile=None, stream=None):
    """scale * (((g_0 + g_1) + g_2) + ...) over the rows of shards (S x n, a
    2-D float32 CUDA tensor: one gathered shard gradient a row). Returns out
    (n floats; it may be shards[0])."""
    import torch
    _cuda_f32(shards, "shards", 2)
    S, n = shards.shape
    if out is None:
        out = torch.empty(n, dtype=torch.float32, device=shards.device)
    _cuda_f32(out, "out")
    if out.numel() != n or (out.dim() > 1 and not out.is_contiguous()):
        raise ValueError(f"out must hold {n} contiguous floats")
    st = load().detshardsum_f32(_prof(profile), S, n, _ptr(shards), _ld(shards),
                                ctypes.c_float(scale), _ptr(out), _stream(stream))
    _check("detshardsum_f32", st)
    return out


def detgemm_f32_noalloc(A, B, C, transA=False, transB=False, profile=None, stream=None):
    """detgemm_f32 without any device allocation, for callers that cannot
    allocate when they multiply (inside another framework's memory pool, or
    in a loop that must not synchronise on cudaMalloc). C must be given; the
    split-K scratch is the library's built-in 64 MiB array, shared by every
    call on the device, so calls must not overlap on the GPU. Shapes that
    would need more scratch raise DetError (DET_ERR_WORKSPACE)."""
    _cuda_f32(A, "A", 2)
    _cuda_f32(B, "B", 2)
    _cuda_f32(C, "C", 2)
    M, K = (A.shape[1], A.shape[0]) if transA else (A.shape[0], A.shape[1])
    Kb, N = (B.shape[1], B.shape[0]) if transB else (B.shape[0], B.shape[1])
    if K != Kb:
        raise ValueError(f"inner dimensions differ: {K} vs {Kb}")
    if tuple(C.shape) != (M, N):
        raise ValueError(f"C must be {M} x {N}")
    st = load().detgemm_f32_noalloc(_prof(profile), int(bool(transA)), int(bool(transB)),
                                    M, N, K, _ptr(A), _ld(A), _ptr(B), _ld(B), _ptr(C),
                                    _ld(C), _stream(stream))
    _check("detgemm_f32_noalloc", st)
    return C


def _problems(problems):
    """det_gemm_problem array from dicts with A, B, C (2-D float32 CUDA
    tensors) and optional transA / transB."""
    arr = (GemmProblem * len(problems))()
    for i, q in enumerate(problems):
        A, B, C = q["A"], q["B"], q["C"]
        tA, tB = bool(q.get("transA", False)), bool(q.get("transB", False))
        for t, name in ((A, "A"), (B, "B"), (C, "C")):
            _cuda_f32(t, name, 2)
        M, K = (A.shape[1], A.shape[0]) if tA else (A.shape[0], A.shape[1])
        Kb, N = (B.shape[1], B.shape[0]) if tB else (B.shape[0], B.shape[1])
        if K != Kb:
            raise ValueError(f"problem {i}: inner dimensions differ: {K} vs {Kb}")
        if tuple(C.shape) != (M, N):
            raise ValueError(f"problem {i}: C must be {M} x {N}")
        arr[i] = GemmProblem(int(tA), int(tB), M, N, K, A.data_ptr(), _ld(A), B.data_ptr(),
                             _ld(B), C.data_ptr(), _ld(C))
    return arr


def detgemm_group_workspace_bytes(problems, profile=None) -> int:
    n = ctypes.c_size_t()
    arr = _problems(problems)
    _check("detgemm_group_workspace_bytes",
           load().detgemm_group_workspace_bytes(_prof(profile), len(problems), arr,
                                                ctypes.byref(n)))
    return n.value


def detgemm_group_launches(problems, workspace=None, profile=None) -> int:
    """Kernel launches detgemm_group_f32 makes for these problems with this
    workspace (a tensor or None)."""
    n = ctypes.c_int64()
    arr = _problems(problems)
    wsn = 0 if workspace is None else workspace.numel() * 4
    _check("detgemm_group_launches",
           load().detgemm_group_launches(_prof(profile), len(problems), arr, wsn,
                                         ctypes.byref(n)))
    return n.value


def gemm_group_workspace(problems, device=None):
    """A workspace tensor for detgemm_group_f32 on these problems (None when
    none helps)."""
    import torch
    n = detgemm_group_workspace_bytes(problems)
    if n == 0:
        return None
    return torch.empty((n + 3) // 4, dtype=torch.float32,
                       device=device if device is not None else problems[0]["C"].device)


def detgemm_group_f32(problems, workspace=None, profile=None, stream=None):
    """Independent products C_i = op(A_i) op(B_i), each with detgemm_f32's
    bits; consecutive pairs may share a launch. problems: dicts with A, B, C
    (and optional transA, transB). Returns the list of C."""
    arr = _problems(problems)
    wsp, wsn = ctypes.c_void_p(), 0
    if workspace is not None:
        _cuda_f32(workspace, "workspace")
        wsp, wsn = _ptr(workspace), workspace.numel() * 4
    st = load().detgemm_group_f32(_prof(profile), len(problems), arr, wsp, wsn,
                                  _stream(stream))
    _check("detgemm_group_f32", st)
    return [q["C"] for q in problems]


# ---------------------------------------------------------------- RMSNorm
def detrmsnorm_f32(x, gain, eps=1e-6, y=None, inv_rms=None, want_inv_rms=True,
                   profile=None, stream=None):
    """Returns (y, inv_rms or None)."""
    import torch
    _cuda_f32(x, "x", 2)
    _cuda_f32(gain, "gain", 1)
    rows, D = x.shape
    if y is None:
        y = torch.empty((rows, D), dtype=torch.float32, device=x.device)
    _cuda_f32(y, "y", 2)
    if inv_rms is None and want_inv_rms:
        inv_rms = torch.empty(rows, dtype=torch.float32, device=x.device)
    st = load().detrmsnorm_f32(_prof(profile), rows, D, _ptr(x), _ld(x), _ptr(gain),
                               ctypes.c_float(eps), _ptr(y), _ld(y), _ptr(inv_rms),
                               _stream(stream))
    _check("detrmsnorm_f32", st)
    return y, inv_rms


def detadd_rmsnorm_f32(a, b, gain, eps=1e-6, x=None, y=None, inv_rms=None, want_inv_rms=True,
                       profile=None, stream=None):
    """x = a + b, then (y, inv_rms) = the RMSNorm of x, as detadd_f32 and
    detrmsnorm_f32 give them (a, b, x dense rows x D). Returns (x, y, inv_rms
    or None)."""
    import torch
    _cuda_f32(a, "a", 2)
    _cuda_f32(b, "b", 2)
    _cuda_f32(gain, "gain", 1)
    rows, D = a.shape
    if tuple(b.shape) != (rows, D) or _ld(a) != D or _ld(b) != D:
        raise ValueError("a and b must be dense rows of the same shape")
    if x is None:
        x = torch.empty((rows, D), dtype=torch.float32, device=a.device)
    _cuda_f32(x, "x", 2)
    if _ld(x) != D:
        raise ValueError("x must be dense")
    if y is None:
        y = torch.empty((rows, D), dtype=torch.float32, device=a.device)
    _cuda_f32(y, "y", 2)
    if inv_rms is None and want_inv_rms:
        inv_rms = torch.empty(rows, dtype=torch.float32, device=a.device)
    st = load().detadd_rmsnorm_f32(_prof(profile), rows, D, _ptr(a), _ptr(b), _ptr(x),
                                   _ptr(gain), ctypes.c_float(eps), _ptr(y), _ld(y),
                                   _ptr(inv_rms), _stream(stream))
    _check("detadd_rmsnorm_f32", st)
    return x, y, inv_rms


def detrmsnorm_bwd_workspace_bytes(rows, D, profile=None) -> int:
    n = ctypes.c_size_t(0)
    _check("detrmsnorm_bwd_workspace_bytes",
           load().detrmsnorm_bwd_workspace_bytes(_prof(profile), rows, D, ctypes.byref(n)))
    return n.value


def detrmsnorm_bwd_f32(x, gain, inv_rms, dy, dx=None, dgain=None, workspace=None,
                       profile=None, stream=None):
    """RMSNorm backward from the forward's inv_rms. Returns (dx, dgain).
    workspace: float32 CUDA tensor of at least detrmsnorm_bwd_workspace_bytes
    bytes; allocated here when needed and not given."""
    import torch
    _cuda_f32(x, "x", 2)
    _cuda_f32(dy, "dy", 2)
    _cuda_f32(gain, "gain", 1)
    _cuda_f32(inv_rms, "inv_rms", 1)
    rows, D = x.shape
    if dx is None:
        dx = torch.empty((rows, D), dtype=torch.float32, device=x.device)
    if dgain is None:
        dgain = torch.empty(D, dtype=torch.float32, device=x.device)
    _cuda_f32(dx, "dx", 2)
    _cuda_f32(dgain, "dgain", 1)
    need = detrmsnorm_bwd_workspace_bytes(rows, D, profile)
    if workspace is None and need > 0:
        workspace = torch.empty((need + 3) // 4, dtype=torch.float32, device=x.device)
    wbytes = workspace.numel() * 4 if workspace is not None else 0
    st = load().detrmsnorm_bwd_f32(_prof(profile), rows, D, _ptr(x), _ld(x), _ptr(gain),
                                   _ptr(inv_rms), _ptr(dy), _ld(dy), _ptr(dx), _ld(dx),
                                   _ptr(dgain), _ptr(workspace), wbytes, _stream(stream))
    _check("detrmsnorm_bwd_f32", st)
    return dx, dgain


# ---------------------------------------------------------------- block forward
def _flat(t, name):
    _cuda_f32(t, name)
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t


def detswiglu_f32(gate, up, out=None, profile=None, stream=None):
    """(gate / (1 + exp(-gate))) * up element-wise. Returns out."""
    import torch
    _flat(gate, "gate")
    _flat(up, "up")
    if gate.shape != up.shape:
        raise ValueError("gate and up differ in shape")
    if out is None:
        out = torch.empty_like(gate)
    _flat(out, "out")
    _check("detswiglu_f32", load().detswiglu_f32(_prof(profile), gate.numel(), _ptr(gate),
                                                 _ptr(up), _ptr(out), _stream(stream)))
    return out


def detadd_f32(a, b, out=None, profile=None, stream=None):
    """a + b element-wise, one rounding. Returns out."""
    import torch
    _flat(a, "a")
    _flat(b, "b")
    if a.shape != b.shape:
        raise ValueError("a and b differ in shape")
    if out is None:
        out = torch.empty_like(a)
    _flat(out, "out")
    _check("detadd_f32", load().detadd_f32(_prof(profile), a.numel(), _ptr(a), _ptr(b),
                                           _ptr(out), _stream(stream)))
    return out


def detsoftmax_causal_f32(scores, scale=1.0, diag=0, period=None, p=None, profile=None,
                          stream=None):
    """Causal softmax of a 2-D score tensor; row r keeps columns
    j <= (r mod period) + diag. Returns p (may be scores, in place)."""
    import torch
    _cuda_f32(scores, "scores", 2)
    rows, cols = scores.shape
    if p is None:
        p = torch.empty_like(scores)
    _cuda_f32(p, "p", 2)
    period = rows if period is None else period
    st = load().detsoftmax_causal_f32(_prof(profile), rows, cols, _ptr(scores), _ld(scores),
                                      ctypes.c_float(scale), int(diag), max(int(period), 1),
                                      _ptr(p), _ld(p), _stream(stream))
    _check("detsoftmax_causal_f32", st)
    return p


def detrope_f32(x, heads, head_dim, seq_len, theta=10000.0, profile=None, stream=None):
    """Rotary embedding in place on the first heads * head_dim columns of the
    rows of x (row t at position t mod seq_len). Returns x."""
    _cuda_f32(x, "x", 2)
    st = load().detrope_f32(_prof(profile), x.shape[0], heads, head_dim, _ptr(x), _ld(x),
                            seq_len, ctypes.c_float(theta), _stream(stream))
    _check("detrope_f32", st)
    return x


def detembedding_f32(table, tokens, out=None, dev_status=None, profile=None, stream=None):
    """Rows of table (vocab x dim) picked by the int32 tokens. Returns out."""
    import torch
    _cuda_f32(table, "table", 2)
    if tokens.dtype != torch.int32 or tokens.device.type != "cuda" or not tokens.is_contiguous():
        raise TypeError("tokens must be a contiguous int32 CUDA tensor")
    vocab, dim = table.shape
    n = tokens.numel()
    if out is None:
        out = torch.empty((n, dim), dtype=torch.float32, device=table.device)
    _cuda_f32(out, "out", 2)
    st = load().detembedding_f32(_prof(profile), n, dim, _ptr(table), _ld(table), vocab,
                                 _ptr(tokens), _ptr(out), _ld(out), _ptr(dev_status),
                                 _stream(stream))
    _check("detembedding_f32", st)
    return out


def detsin_f32(x, y=None, profile=None, stream=None):
    return _sincos(x, y, profile, stream, "detsin_f32")


def detcos_f32(x, y=None, profile=None, stream=None):
    return _sincos(x, y, profile, stream, "detcos_f32")


def _sincos(x, y, profile, stream, fn):
    import torch
    _flat(x, "x")
    if y is None:
        y = torch.empty_like(x)
    _flat(y, "y")
    _check(fn, getattr(load(), fn)(_prof(profile), x.numel(), _ptr(x), _ptr(y),
                                   _stream(stream)))
    return y


def detattention_workspace_bytes(batch, seq, heads, head_dim, profile=None) -> int:
    n = ctypes.c_size_t(0)
    _check("detattention_workspace_bytes",
           load().detattention_workspace_bytes(_prof(profile), batch, seq, heads, head_dim,
                                               ctypes.byref(n)))
    return n.value


def detattention_launches(batch, seq, heads, head_dim, backward=False, saved=False,
                          profile=None) -> int:
    """Kernel launches detattention_f32 (or, backward=True, detattention_bwd_f32;
    with saved=True as well, detattention_bwd_saved_f32) makes for these sizes."""
    n = ctypes.c_int64()
    mode = (2 if saved else 1) if backward else 0
    _check("detattention_launches",
           load().detattention_launches(_prof(profile), batch, seq, heads, head_dim,
                                        mode, ctypes.byref(n)))
    return n.value


def detattention_f32(qkv, batch, seq, heads, head_dim, scale=None, out=None, workspace=None,
                     profile=None, stream=None):
    """Causal attention over packed QKV rows (batch * seq rows of [Q | K | V]).
    Returns out (batch * seq rows of heads * head_dim)."""
    import torch
    _cuda_f32(qkv, "qkv", 2)
    if qkv.shape[0] != batch * seq:
        raise ValueError("qkv must hold batch * seq rows")
    if out is None:
        out = torch.empty((batch * seq, heads * head_dim), dtype=torch.float32,
                          device=qkv.device)
    _cuda_f32(out, "out", 2)
    if scale is None:
        scale = 1.0 / float(head_dim) ** 0.5
    if workspace is None:
        workspace = torch.empty(
            (detattention_workspace_bytes(batch, seq, heads, head_dim, profile) + 3) // 4,
            dtype=torch.float32, device=qkv.device)
    st = load().detattention_f32(_prof(profile), batch, seq, heads, head_dim, _ptr(qkv),
                                 _ld(qkv), ctypes.c_float(scale), _ptr(out), _ld(out),
                                 _ptr(workspace), workspace.numel() * 4, _stream(stream))
    _check("detattention_f32", st)
    return out


# ---------------------------------------------------------------- block backward
def detswiglu_bwd_f32(gate, up, dh, d_gate=None, d_up=None, profile=None, stream=None):
    """Returns (d_gate, d_up) of h = silu(gate) * up."""
    import torch
    for t, n in ((gate, "gate"), (up, "up"), (dh, "dh")):
        _flat(t, n)
    d_gate = torch.empty_like(gate) if d_gate is None else _flat(d_gate, "d_gate")
    d_up = torch.empty_like(gate) if d_up is None else _flat(d_up, "d_up")
    st = load().detswiglu_bwd_f32(_prof(profile), gate.numel(), _ptr(gate), _ptr(up), _ptr(dh),
                                  _ptr(d_gate), _ptr(d_up), _stream(stream))
    _check("detswiglu_bwd_f32", st)
    return d_gate, d_up


def detsoftmax_causal_bwd_f32(p, dp, scale=1.0, diag=0, period=None, ds=None, profile=None,
                              stream=None):
    """dS of the causal softmax from P and dP (same layout). Returns ds."""
    import torch
    _cuda_f32(p, "p", 2)
    _cuda_f32(dp, "dp", 2)
    rows, cols = p.shape
    if _ld(p) != _ld(dp):
        raise ValueError("p and dp must share a row stride")
    ds = torch.empty_like(p) if ds is None else ds
    _cuda_f32(ds, "ds", 2)
    period = rows if period is None else period
    st = load().detsoftmax_causal_bwd_f32(_prof(profile), rows, cols, _ptr(p), _ptr(dp), _ld(p),
                                          ctypes.c_float(scale), int(diag),
                                          max(int(period), 1), _ptr(ds), _ld(ds),
                                          _stream(stream))
    _check("detsoftmax_causal_bwd_f32", st)
    return ds


def detrope_bwd_f32(dx, heads, head_dim, seq_len, theta=10000.0, profile=None, stream=None):
    """The rotary backward in place on dx's first heads * head_dim columns."""
    _cuda_f32(dx, "dx", 2)
    st = load().detrope_bwd_f32(_prof(profile), dx.shape[0], heads, head_dim, _ptr(dx),
                                _ld(dx), seq_len, ctypes.c_float(theta), _stream(stream))
    _check("detrope_bwd_f32", st)
    return dx


def detembedding_bwd_f32(tokens, dx, vocab, de=None, profile=None, stream=None):
    """Per-id ordered sums of the tokens' gradient rows. Returns de."""
    import torch
    _cuda_f32(dx, "dx", 2)
    if tokens.dtype != torch.int32 or tokens.device.type != "cuda" or not tokens.is_contiguous():
        raise TypeError("tokens must be a contiguous int32 CUDA tensor")
    dim = dx.shape[1]
    de = torch.empty((vocab, dim), dtype=torch.float32, device=dx.device) if de is None else de
    _cuda_f32(de, "de", 2)
    st = load().detembedding_bwd_f32(_prof(profile), tokens.numel(), dim, _ptr(tokens),
                                     _ptr(dx), _ld(dx), vocab, _ptr(de), _ld(de),
                                     _stream(stream))
    _check("detembedding_bwd_f32", st)
    return de


def detattention_bwd_workspace_bytes(batch, seq, heads, head_dim, profile=None) -> int:
    n = ctypes.c_size_t(0)
    _check("detattention_bwd_workspace_bytes",
           load().detattention_bwd_workspace_bytes(_prof(profile), batch, seq, heads, head_dim,
                                                   ctypes.byref(n)))
    return n.value


def detattention_bwd_f32(qkv, dout, batch, seq, heads, head_dim, scale=None, dqkv=None,
                         workspace=None, profile=None, stream=None):
    """Gradients of the packed Q, K, V (the forward's input). Returns dqkv."""
    import torch
    _cuda_f32(qkv, "qkv", 2)
    _cuda_f32(dout, "dout", 2)
    dqkv = torch.empty_like(qkv) if dqkv is None else dqkv
    _cuda_f32(dqkv, "dqkv", 2)
    if scale is None:
        scale = 1.0 / float(head_dim) ** 0.5
    if workspace is None:
        workspace = torch.empty(
            (detattention_bwd_workspace_bytes(batch, seq, heads, head_dim, profile) + 3) // 4,
            dtype=torch.float32, device=qkv.device)
    st = load().detattention_bwd_f32(_prof(profile), batch, seq, heads, head_dim, _ptr(qkv),
                                     _ld(qkv), _ptr(dout), _ld(dout), ctypes.c_float(scale),
                                     _ptr(dqkv), _ld(dqkv), _ptr(workspace),
                                     workspace.numel() * 4, _stream(stream))
    _check("detattention_bwd_f32", st)
    return dqkv


def detattention_bwd_saved_f32(qkv, dout, batch, seq, heads, head_dim, fwd_workspace,
                               scale=None, dqkv=None, workspace=None, profile=None,
                               stream=None):
    """detattention_bwd_f32 reading P from fwd_workspace, the workspace of the
    detattention_f32 call on the same qkv (unchanged since). Returns dqkv."""
    import torch
    _cuda_f32(qkv, "qkv", 2)
    _cuda_f32(dout, "dout", 2)
    dqkv = torch.empty_like(qkv) if dqkv is None else dqkv
    _cuda_f32(dqkv, "dqkv", 2)
    if scale is None:
        scale = 1.0 / float(head_dim) ** 0.5
    if workspace is None:
        workspace = torch.empty(
            (detattention_bwd_workspace_bytes(batch, seq, heads, head_dim, profile) + 3) // 4,
            dtype=torch.float32, device=qkv.device)
    st = load().detattention_bwd_saved_f32(_prof(profile), batch, seq, heads, head_dim,
                                           _ptr(qkv), _ld(qkv), _ptr(dout), _ld(dout),
                                           ctypes.c_float(scale), _ptr(fwd_workspace),
                                           fwd_workspace.numel() * fwd_workspace.element_size(),
                                           _ptr(dqkv), _ld(dqkv), _ptr(workspace),
                                           workspace.numel() * 4, _stream(stream))
    _check("detattention_bwd_saved_f32", st)
    return dqkv


# ---------------------------------------------------------------- cross-entropy
def detxent_f32(logits, labels, loss=None, want_mean=False, loss_mean=None,
                dlogits=None, want_dlogits=False, dscale=None, dev_status=None,
                profile=None, stream=None):
    """Returns (loss, loss_mean or None, dlogits or None). dscale defaults to
    1/rows. dev_status: optional int32 CUDA tensor of one element."""
    import torch
    _cuda_f32(logits, "logits", 2)
    if labels.dtype != torch.int32 or labels.device.type != "cuda":
        raise TypeError("labels must be an int32 CUDA tensor")
    rows, V = logits.shape
    if loss is None:
        loss = torch.empty(rows, dtype=torch.float32, device=logits.device)
    if loss_mean is None and want_mean:
        loss_mean = torch.empty(1, dtype=torch.float32, device=logits.device)
    if dlogits is None and want_dlogits:
        dlogits = torch.empty((rows, V), dtype=torch.float32, device=logits.device)
    if dscale is None:
        dscale = 1.0 / max(rows, 1)
    if dev_status is not None and (dev_status.dtype != torch.int32
                                   or dev_status.device.type != "cuda"):
        raise TypeError("dev_status must be an int32 CUDA tensor")
    st = load().detxent_f32(_prof(profile), rows, V, _ptr(logits), _ld(logits),
                            _ptr(labels), _ptr(loss), _ptr(loss_mean), _ptr(dlogits),
                            _ld(dlogits) if dlogits is not None else V,
                            ctypes.c_float(dscale), _ptr(dev_status), _stream(stream))
    _check("detxent_f32", st)
    return loss, loss_mean, dlogits


# ---------------------------------------------------------------- AdamW
def det_adamw_bias_correction(step, beta1, beta2):
    """(bc1, bc2) = (1 - beta1^t, 1 - beta2^t) as float32 bits, the values
    detadamw_f32 divides by at step t. Host-only: needs no GPU."""
    import numpy as np
    bc1, bc2 = ctypes.c_float(), ctypes.c_float()
    st = load().det_adamw_bias_correction(int(step), ctypes.c_float(beta1),
                                          ctypes.c_float(beta2), ctypes.byref(bc1),
                                          ctypes.byref(bc2))
    _check("det_adamw_bias_correction", st)
    return np.float32(bc1.value), np.float32(bc2.value)


def detadamw_f32(p, g, m, v, lr, beta1, beta2, eps, weight_decay, step,
                 profile=None, stream=None):
    """In-place AdamW update of p, m, v (1-D float32 CUDA tensors)."""
    for t, name in ((p, "p"), (g, "g"), (m, "m"), (v, "v")):
        _cuda_f32(t, name, 1)
    n = p.numel()
    if not (g.numel() == m.numel() == v.numel() == n):
        raise ValueError("p, g, m, v must have the same length")
    hp = AdamWHP(lr, beta1, beta2, eps, weight_decay, int(step))
    st = load().detadamw_f32(_prof(profile), n, _ptr(p), _ptr(g), _ptr(m), _ptr(v),
                             ctypes.byref(hp), _stream(stream))
    _check("detadamw_f32", st)
    return p, m, v


# ---------------------------------------------------------------- exp / log
def detexp_f32(x, y=None, profile=None, stream=None):
    import torch
    _cuda_f32(x, "x")
    if y is None:
        y = torch.empty_like(x)
    st = load().detexp_f32(_prof(profile), x.numel(), _ptr(x), _ptr(y), _stream(stream))
    _check("detexp_f32", st)
    return y


def detlog_f32(x, y=None, profile=None, stream=None):
    import torch
    _cuda_f32(x, "x")
    if y is None:
        y = torch.empty_like(x)
    st = load().detlog_f32(_prof(profile), x.numel(), _ptr(x), _ptr(y), _stream(stream))
    _check("detlog_f32", st)
    return y


def det_watchdog_status(clear: bool = False) -> int:
    code = ctypes.c_int32()
    _check("det_watchdog_status",
           load().det_watchdog_status(ctypes.byref(code), int(bool(clear))))
    return code.value
