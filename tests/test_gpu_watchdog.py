"""The GEMM's give-up path, run on a GPU without a fault.

Every device wait of the library is bounded. When a wait runs out, the CTA
records a watchdog bit, lets the copies it issued land, skips its stores and
returns, so the context stays usable. To run that path on healthy copies, the
test builds a separate copy of the library (never the shipped one) whose GEMM
consumers use a wait limit of 0: they give up at the first operand wait that
is not already complete. The drain of copies in flight keeps its normal bound.
Then:
  * that copy's det_watchdog_status reports bit 0 (GEMM operand staging);
  * every output the aborted call left is either unwritten or correct;
  * the next call through the shipped library, on the same device and
    context, gives the oracle's bits, and its own watchdog word is clean.
"""
import ctypes
import os

import numpy as np
import pytest

import oracle
from bitcmp import assert_bitwise
from bitwise_reproducible_fp32_gb300 import build, detlib
from gpu_util import host, need_gpu, to_dev, torch

pytestmark = pytest.mark.gpu
F = np.float32


@pytest.fixture(scope="module")
def short_wait_lib(tmp_path_factory):
    need_gpu()
    path = os.path.join(str(tmp_path_factory.mktemp("wd")), "libdetfp32_shortwait.so")
    build.build_variant(["DET_TEST_GEMM_WAIT_NS=0"], path)
    lib = ctypes.CDLL(path)
    for name, res, args in detlib.SIGNATURES:
        if name in ("detgemm_f32", "det_watchdog_status", "det_profile_default"):
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
    return lib


def test_gemm_wait_that_runs_out_sets_the_watchdog_and_leaves_the_device_usable(
        short_wait_lib):
    lib = short_wait_lib
    rng = np.random.default_rng(606)
    M = N = K = 256
    A = rng.standard_normal((M, K)).astype(F)
    B = rng.standard_normal((K, N)).astype(F)
    want = oracle.gemm(A, B)
    Ad, Bd = to_dev(A), to_dev(B)
    C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
    prof = detlib.Profile()
    lib.det_profile_default(ctypes.byref(prof))
    code = ctypes.c_int32(-1)
    assert lib.det_watchdog_status(ctypes.byref(code), 1) == 0     # start clean
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = lib.detgemm_f32(ctypes.byref(prof), 0, 0, M, N, K,
                         ctypes.c_void_p(Ad.data_ptr()), K, ctypes.c_void_p(Bd.data_ptr()), N,
                         ctypes.c_void_p(C.data_ptr()), N, None, 0, stream)
    assert st == 0
    torch.cuda.synchronize()                  # returns: no hang, no fault
    assert lib.det_watchdog_status(ctypes.byref(code), 1) == 0
    assert code.value & 1, f"watchdog word {code.value}: the GEMM's wait did not give up"
    # the aborted units skipped their stores: every output is untouched or right
    got = host(C)
    left = np.isnan(got)
    assert left.any()
    assert_bitwise(got[~left], want[~left], "outputs the aborted call did write")
    assert lib.det_watchdog_status(ctypes.byref(code), 0) == 0 and code.value == 0
    # the shipped library, same device and context: the oracle's bits
    C2 = detlib.detgemm_f32(Ad, Bd)
    torch.cuda.synchronize()
    assert_bitwise(host(C2), want, "shipped GEMM after the give-up")
    assert detlib.det_watchdog_status() == 0
