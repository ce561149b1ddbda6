"""detgemm_f32_noalloc: the GEMM for callers that cannot allocate device
memory when they multiply (inside another framework's memory pool, or in a loop
that must not synchronise on cudaMalloc). It must give the same bits as
detgemm_f32 and refuse shapes whose split-K scratch exceeds its built-in
64 MiB array. This file is collected last on purpose."""
import numpy as np
import pytest

from bitcmp import assert_bitwise
from bitwise_reproducible_fp32_gb300 import detlib
from gpu_util import empty_dev, host, need_gpu, to_dev, torch

pytestmark = pytest.mark.gpu
F = np.float32

CASES = [
    # (M, N, K, transA, transB): the first three split K through the scratch
    (300, 200, 1300, False, False),
    (512, 384, 4096, True, False),
    (129, 77, 2049, False, True),
    (64, 64, 256, False, False),     # one chunk: no scratch needed
    (517, 6000, 700, False, True),   # A copied transposed into the scratch
]


def test_noalloc_same_bits_as_detgemm_f32_two_calls_in_a_row():
    need_gpu()
    rng = np.random.default_rng(2024)
    for M, N, K, tA, tB in CASES:
        A = rng.standard_normal((K, M) if tA else (M, K)).astype(F)
        B = rng.standard_normal((N, K) if tB else (K, N)).astype(F)
        Ad, Bd = to_dev(A), to_dev(B)
        ws = detlib.gemm_workspace(M, N, K, tA, tB)
        ref = host(detlib.detgemm_f32(Ad, Bd, transA=tA, transB=tB, workspace=ws))
        for call in range(2):
            C = empty_dev(M, N)
            detlib.detgemm_f32_noalloc(Ad, Bd, C, transA=tA, transB=tB)
            torch.cuda.synchronize()
            assert_bitwise(host(C), ref, f"M={M} N={N} K={K} call {call}")


def test_noalloc_refuses_shapes_beyond_its_scratch():
    need_gpu()
    M, N, K = 768, 2304, 8192      # needs ~221 MB of split-K scratch
    assert detlib.detgemm_workspace_bytes(M, N, K, True, False) > 64 * 2 ** 20
    A = torch.zeros((K, M), dtype=torch.float32, device="cuda")
    B = torch.zeros((K, N), dtype=torch.float32, device="cuda")
    C = torch.zeros((M, N), dtype=torch.float32, device="cuda")
    with pytest.raises(detlib.DetError) as err:
        detlib.detgemm_f32_noalloc(A, B, C, transA=True)
    assert err.value.status == 5      # DET_ERR_WORKSPACE


def test_noalloc_skips_a_transposed_copy_beyond_its_scratch():
    need_gpu()
    # the copy of A would take 24,576 x 768 floats (75 MB): A is read in place
    M, N, K = 24576, 2048, 768
    assert detlib.detgemm_workspace_bytes(M, N, K, False, False) > 64 * 2 ** 20
    rng = np.random.default_rng(77)
    A = rng.standard_normal((M, K)).astype(F)
    B = rng.standard_normal((K, N)).astype(F)
    Ad, Bd = to_dev(A), to_dev(B)
    ref = host(detlib.detgemm_f32(Ad, Bd, workspace=detlib.gemm_workspace(M, N, K)))
    C = empty_dev(M, N)
    detlib.detgemm_f32_noalloc(Ad, Bd, C)
    torch.cuda.synchronize()
    assert_bitwise(host(C), ref, "no-alloc without the transposed copy")


def test_noalloc_empty_contraction_and_argument_checks():
    need_gpu()
    # K == 0: the empty sum, +0 in every output, as detgemm_f32 gives
    A = torch.zeros((5, 0), dtype=torch.float32, device="cuda")
    B = torch.zeros((0, 7), dtype=torch.float32, device="cuda")
    C = torch.full((5, 7), float("nan"), dtype=torch.float32, device="cuda")
    detlib.detgemm_f32_noalloc(A, B, C)
    torch.cuda.synchronize()
    assert np.all(host(C).view(np.uint32) == 0)
    # a row stride below the row length is refused on the host, before any launch
    import ctypes
    lib = detlib.load()
    prof = ctypes.byref(detlib.det_profile_default())
    Ad = torch.zeros((4, 8), dtype=torch.float32, device="cuda")
    Bd = torch.zeros((8, 4), dtype=torch.float32, device="cuda")
    Cd = torch.zeros((4, 4), dtype=torch.float32, device="cuda")
    ptr = lambda t: ctypes.c_void_p(t.data_ptr())
    assert lib.detgemm_f32_noalloc(prof, 0, 0, 4, 4, 8, ptr(Ad), 7, ptr(Bd), 4, ptr(Cd), 4,
                                   None) == 1       # lda < K
    assert lib.detgemm_f32_noalloc(prof, 0, 0, 4, 4, 8, ptr(Ad), 8, ptr(Bd), 4, None, 4,
                                   None) == 1       # null C


def test_noalloc_on_a_side_stream_after_a_first_call():
    need_gpu()
    # the first call (address look-up) happened on the current stream in the
    # tests above, or happens here; a later call on another stream must give
    # detgemm_f32's bits
    rng = np.random.default_rng(2025)
    M, N, K = 300, 200, 1300          # split K through the scratch
    A = rng.standard_normal((M, K)).astype(F)
    B = rng.standard_normal((K, N)).astype(F)
    Ad, Bd = to_dev(A), to_dev(B)
    ref = host(detlib.detgemm_f32(Ad, Bd, workspace=detlib.gemm_workspace(M, N, K)))
    detlib.detgemm_f32_noalloc(Ad, Bd, empty_dev(M, N))
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    C = empty_dev(M, N)
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        detlib.detgemm_f32_noalloc(Ad, Bd, C, stream=side)
    side.synchronize()
    assert_bitwise(host(C), ref, "no-alloc GEMM on a side stream")
