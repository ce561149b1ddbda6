"""The C-ABI library builds, loads without a GPU, exports every function that
include/detfp32.h declares, and refuses bad profiles and arguments on the host
before touching any device."""
import ctypes
import os
import re

import pytest

from bitwise_reproducible_fp32_gb300 import build, detlib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "detfp32.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return detlib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(det\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for want in ("detgemm_f32", "detgemm_workspace_bytes", "detrmsnorm_f32", "detxent_f32", "detadamw_f32",
                 "detrmsnorm_bwd_f32", "detrmsnorm_bwd_workspace_bytes",
                 "detgemm_acc_f32", "detshardsum_f32", "detswiglu_f32", "detadd_f32",
                 "detsoftmax_causal_f32", "detrope_f32", "detsin_f32", "detcos_f32",
                 "detattention_f32", "detattention_workspace_bytes", "detembedding_f32",
                 "detswiglu_bwd_f32", "detsoftmax_causal_bwd_f32", "detrope_bwd_f32",
                 "detembedding_bwd_f32", "detattention_bwd_f32", "detadd_rmsnorm_f32",
                 "detattention_bwd_workspace_bytes", "detattention_bwd_saved_f32",
                 "detexp_f32", "detlog_f32", "det_adamw_bias_correction",
                 "det_profile_default",
                 "det_status_string", "det_watchdog_status"):
        assert want in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding wraps each of them under the same name
    wrapped = {n for n, _, _ in detlib.SIGNATURES}
    assert set(declared_functions()) <= wrapped


def test_only_the_boundary_is_exported(lib):
    # internal C++ symbols are hidden (-fvisibility=hidden); only det* is public
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", detlib.LIB_PATH],
                         capture_output=True, text=True).stdout
    public = [l.split()[-1] for l in out.splitlines() if " T " in l]
    assert public and all(n.startswith("det") for n in public), public


def test_profile_default_and_strings(lib):
    p = detlib.det_profile_default()
    assert (p.version, p.k_chunk, p.rms_lanes, p.xent_lanes, p.lane_group, p.flags) == (
        1, 256, 32, 256, 4, 0)
    assert detlib.det_status_string(0) == "DET_OK"
    assert "PROFILE" in detlib.det_status_string(2)
    assert detlib.det_status_string(99) == "unknown det_status"


@pytest.mark.parametrize("field,value", [("version", 2), ("k_chunk", 128),
                                         ("rms_lanes", 64), ("xent_lanes", 32),
                                         ("lane_group", 1), ("flags", 1)])
def test_unknown_profile_is_refused_by_name(lib, field, value):
    p = detlib.det_profile_default()
    setattr(p, field, value)
    null = ctypes.c_void_p()
    st = lib.detgemm_f32(ctypes.byref(p), 0, 0, 4, 4, 4, null, 4, null, 4, null, 4,
                         null, 0, null)
    assert st == 2
    hp = detlib.AdamWHP(1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    assert lib.detadamw_f32(ctypes.byref(p), 4, null, null, null, null,
                            ctypes.byref(hp), null) == 2
    assert lib.detexp_f32(ctypes.byref(p), 4, null, null, null) == 2
    assert lib.detxent_f32(ctypes.byref(p), 1, 4, null, 4, null, null, null, null, 4,
                           ctypes.c_float(1.0), null, null) == 2
    assert lib.detrmsnorm_f32(ctypes.byref(p), 1, 4, null, 4, null,
                              ctypes.c_float(1e-6), null, 4, null, null) == 2
    assert lib.detrmsnorm_bwd_f32(ctypes.byref(p), 1, 4, null, 4, null, null, null, 4,
                                  null, 4, null, null, 0, null) == 2
    n = ctypes.c_size_t(7)
    assert lib.detrmsnorm_bwd_workspace_bytes(ctypes.byref(p), 1000, 8, ctypes.byref(n)) == 2
    assert lib.detgemm_acc_f32(ctypes.byref(p), 0, 0, 4, 4, 4, null, 4, null, 4, null, 4,
                               null, 0, null) == 2
    assert lib.detshardsum_f32(ctypes.byref(p), 2, 4, null, 4, ctypes.c_float(1.0), null,
                               null) == 2
    assert lib.detswiglu_f32(ctypes.byref(p), 4, null, null, null, null) == 2
    assert lib.detrope_f32(ctypes.byref(p), 4, 2, 64, null, 128, 4, ctypes.c_float(1e4),
                           null) == 2


def test_bad_arguments_are_refused_on_the_host(lib):
    p = ctypes.byref(detlib.det_profile_default())
    null = ctypes.c_void_p()
    dummy = ctypes.c_void_p(0x1000)
    # negative sizes, ld below the row length, null pointers, >= 2^31 dims
    assert lib.detgemm_f32(p, 0, 0, -1, 4, 4, dummy, 4, dummy, 4, dummy, 4, null, 0, null) == 1
    assert lib.detgemm_f32(p, 0, 0, 4, 4, 8, dummy, 7, dummy, 4, dummy, 4, null, 0, null) == 1
    assert lib.detgemm_f32(p, 1, 0, 9, 4, 8, dummy, 8, dummy, 4, dummy, 4, null, 0, null) == 1
    assert lib.detgemm_f32(p, 0, 1, 4, 4, 8, dummy, 8, dummy, 7, dummy, 4, null, 0, null) == 1
    assert lib.detgemm_f32(p, 0, 0, 4, 4, 8, null, 8, dummy, 4, dummy, 4, null, 0, null) == 1
    assert lib.detgemm_f32(p, 0, 0, 2 ** 31, 4, 8, dummy, 8, dummy, 4, dummy, 4, null, 0,
                           null) == 1
    # empty problems are a successful no-op without any device call
    assert lib.detgemm_f32(p, 0, 0, 0, 4, 8, null, 8, null, 4, null, 4, null, 0, null) == 0
    assert lib.detrmsnorm_f32(p, 3, 0, dummy, 4, dummy, ctypes.c_float(1e-6), dummy, 4,
                              null, null) == 1
    assert lib.detrmsnorm_f32(p, 0, 8, null, 8, null, ctypes.c_float(1e-6), null, 8, null,
                              null) == 0
    assert lib.detxent_f32(p, 2, 0, dummy, 4, dummy, dummy, null, null, 4,
                           ctypes.c_float(1.0), null, null) == 1
    assert lib.detxent_f32(p, 2, 8, dummy, 8, dummy, dummy, null, dummy, 7,
                           ctypes.c_float(1.0), null, null) == 1
    # RMSNorm backward: D < 1, stride below D, null gain, dx == dy with other
    # strides, a missing or short workspace past one 256-row chunk
    rb = lib.detrmsnorm_bwd_f32
    assert rb(p, 4, 0, dummy, 4, dummy, dummy, dummy, 4, dummy, 4, dummy, null, 0, null) == 1
    assert rb(p, 4, 8, dummy, 7, dummy, dummy, dummy, 8, dummy, 8, dummy, null, 0, null) == 1
    assert rb(p, 4, 8, dummy, 8, null, dummy, dummy, 8, dummy, 8, dummy, null, 0, null) == 1
    assert rb(p, 4, 8, dummy, 8, dummy, dummy, dummy, 8, dummy, 12, dummy, null, 0, null) == 1
    assert rb(p, 4, 8, dummy, 8, dummy, dummy, dummy, 8, dummy, 8, null, null, 0, null) == 1
    assert rb(p, 300, 8, dummy, 8, dummy, dummy, dummy, 8, dummy, 8, dummy, null, 0, null) == 5
    assert rb(p, 300, 8, dummy, 8, dummy, dummy, dummy, 8, dummy, 8, dummy, dummy, 63,
              null) == 5
    n = ctypes.c_size_t(7)
    assert lib.detrmsnorm_bwd_workspace_bytes(p, 256, 768, ctypes.byref(n)) == 0 and n.value == 0
    assert lib.detrmsnorm_bwd_workspace_bytes(p, 8192, 768, ctypes.byref(n)) == 0
    assert n.value == 32 * 768 * 4
    # accumulating GEMM: the GEMM's rules; shard sum: counts, strides, overlap
    assert lib.detgemm_acc_f32(p, 0, 0, 4, 4, 8, dummy, 7, dummy, 4, dummy, 4, null, 0,
                               null) == 1
    assert lib.detgemm_acc_f32(p, 0, 0, 0, 4, 8, null, 8, null, 4, null, 4, null, 0, null) == 0
    ss = lib.detshardsum_f32
    one = ctypes.c_float(1.0)
    assert ss(p, 0, 8, dummy, 8, one, dummy, null) == 1
    assert ss(p, 2, -1, dummy, 8, one, dummy, null) == 1
    assert ss(p, 2, 8, dummy, 7, one, dummy, null) == 1
    assert ss(p, 2, 8, null, 8, one, dummy, null) == 1
    assert ss(p, 2, 8, ctypes.c_void_p(0x1000), 8, one, ctypes.c_void_p(0x1000 + 4 * 8),
              null) == 1                                   # out over shard 1
    assert ss(p, 2, 0, null, 0, one, null, null) == 0
    # block forward: sizes, strides, periods, head shapes, overlaps, workspace
    d0 = ctypes.c_void_p(0x1000)
    assert lib.detswiglu_f32(p, -1, dummy, dummy, dummy, null) == 1
    assert lib.detswiglu_f32(p, 8, d0, dummy, ctypes.c_void_p(0x1000 + 4), null) == 1
    assert lib.detswiglu_f32(p, 0, null, null, null, null) == 0
    assert lib.detadd_f32(p, 8, null, dummy, dummy, null) == 1
    sm = lib.detsoftmax_causal_f32
    assert sm(p, 4, 0, dummy, 4, one, 0, 4, dummy, 4, null) == 1
    assert sm(p, 4, 8, dummy, 7, one, 0, 4, dummy, 8, null) == 1
    assert sm(p, 4, 8, dummy, 8, one, 0, 0, dummy, 8, null) == 1
    assert sm(p, 4, 8, dummy, 8, one, 0, 4, dummy, 12, null) == 1      # p == scores, ld differ
    rp = lib.detrope_f32
    assert rp(p, 4, 2, 63, dummy, 200, 4, ctypes.c_float(1e4), null) == 1   # odd head_dim
    assert rp(p, 4, 2, 64, dummy, 127, 4, ctypes.c_float(1e4), null) == 1   # ld < heads*d
    assert rp(p, 4, 2, 64, dummy, 128, 0, ctypes.c_float(1e4), null) == 1   # seq_len 0
    assert lib.detsin_f32(p, -1, dummy, dummy, null) == 1
    at = lib.detattention_f32
    assert at(p, 1, 16, 2, 8, dummy, 47, one, dummy, 16, dummy, 1 << 20, null) == 1
    assert at(p, 1, 16, 2, 8, dummy, 48, one, dummy, 15, dummy, 1 << 20, null) == 1
    assert at(p, 0, 16, 2, 8, null, 48, one, null, 16, null, 0, null) == 0
    # workspace queries (host only): the score buffers of one group of heads,
    # all 48 heads of 4 x 2048 tokens fitting the 1 GiB cap, 16 x 128 tokens
    # too, and from 512 tokens a transposed copy of the Q and K blocks (2 x
    # heads x head_dim rows of batch x seq floats); the backward's copies of
    # the Q, dO and V blocks
    n = ctypes.c_size_t(0)
    assert lib.detattention_workspace_bytes(p, 4, 2048, 12, 64, ctypes.byref(n)) == 0
    assert n.value == 48 * 2048 * 2048 * 4 + 256 + 2 * 768 * 8192 * 4   # + counts, Q/K copy
    assert lib.detattention_bwd_workspace_bytes(p, 4, 2048, 12, 64, ctypes.byref(n)) == 0
    assert n.value == 2 * 48 * 2048 * 2048 * 4 + 256 + 3 * 768 * 8192 * 4   # + Q, dO, V copies
    assert lib.detattention_workspace_bytes(p, 16, 128, 4, 16, ctypes.byref(n)) == 0
    assert n.value == 64 * 128 * 128 * 4 + 256
    # 8 sequences of 8192 tokens x 12 heads (3 GiB of scores) go 4 heads at a time
    assert lib.detattention_workspace_bytes(p, 8, 8192, 12, 64, ctypes.byref(n)) == 0
    assert n.value == 4 * 8192 * 8192 * 4 + 256 + 2 * 768 * 65536 * 4
    assert lib.detattention_workspace_bytes(p, 1, 0, 12, 64, ctypes.byref(n)) == 1
    # launches: 4 a group forward (+ the Q/K copy from 512 tokens), 10 backward
    # (+ the Q, dO and V copies from 512 tokens)
    k = ctypes.c_int64(0)
    assert lib.detattention_launches(p, 4, 2048, 12, 64, 0, ctypes.byref(k)) == 0
    assert k.value == 5
    assert lib.detattention_launches(p, 4, 2048, 12, 64, 1, ctypes.byref(k)) == 0
    assert k.value == 13
    assert lib.detattention_launches(p, 16, 128, 4, 16, 1, ctypes.byref(k)) == 0
    assert k.value == 10
    # the backward with the forward's P (one group): no S, no softmax, one +0
    # fill; the dO and V copies from 512 tokens
    assert lib.detattention_launches(p, 4, 2048, 12, 64, 2, ctypes.byref(k)) == 0
    assert k.value == 11
    assert lib.detattention_launches(p, 16, 128, 4, 16, 2, ctypes.byref(k)) == 0
    assert k.value == 9
    # several groups: P is not all in the forward's workspace, so it recomputes
    assert lib.detattention_launches(p, 8, 8192, 12, 64, 2, ctypes.byref(k)) == 0
    assert k.value == 8 * 3 * 10 + 3
    assert lib.detattention_launches(p, 16, 128, 4, 16, 0, ctypes.byref(k)) == 0
    assert k.value == 4
    assert lib.detattention_launches(p, 8, 8192, 12, 64, 0, ctypes.byref(k)) == 0
    assert k.value == 8 * 3 * 4 + 1
    assert lib.detattention_launches(p, 8, 8192, 12, 64, 1, ctypes.byref(k)) == 0
    assert k.value == 8 * 3 * 10 + 3
    assert lib.detattention_launches(p, 0, 2048, 12, 64, 0, ctypes.byref(k)) == 0
    assert k.value == 0
    assert lib.detattention_launches(p, 1, 0, 12, 64, 0, ctypes.byref(k)) == 1
    # backward ops and the embedding
    assert lib.detswiglu_bwd_f32(p, 8, d0, dummy, dummy, ctypes.c_void_p(0x1000 + 16), dummy,
                                 null) == 1                      # d_gate over gate
    assert lib.detsoftmax_causal_bwd_f32(p, 4, 8, dummy, dummy, 8, one, 0, 4, dummy, 12,
                                         null) == 1
    assert lib.detrope_bwd_f32(p, 4, 2, 63, dummy, 200, 4, ctypes.c_float(1e4), null) == 1
    assert lib.detembedding_f32(p, 4, 8, dummy, 7, 10, dummy, dummy, 8, null, null) == 1
    assert lib.detembedding_bwd_f32(p, 4, 8, dummy, dummy, 8, 10, dummy, 7, null) == 1
    assert lib.detattention_bwd_f32(p, 1, 16, 2, 8, dummy, 48, dummy, 16, one, dummy, 47,
                                    dummy, 1 << 20, null) == 1
    assert lib.detattention_bwd_saved_f32(p, 1, 16, 2, 8, dummy, 48, dummy, 16, one, null,
                                          1 << 20, dummy, 48, dummy, 1 << 20, null) == 5
    assert lib.detattention_bwd_saved_f32(p, 1, 16, 2, 8, dummy, 48, dummy, 16, one, dummy,
                                          16, dummy, 48, dummy, 1 << 20, null) == 5
    hp = detlib.AdamWHP(1e-3, 0.9, 0.95, 1e-8, 0.1, 0)
    assert lib.detadamw_f32(p, 4, dummy, dummy, dummy, dummy, ctypes.byref(hp), null) == 1
    hp = detlib.AdamWHP(1e-3, 1.25, 0.95, 1e-8, 0.1, 3)              # beta outside [0, 1]
    assert lib.detadamw_f32(p, 4, dummy, dummy, dummy, dummy, ctypes.byref(hp), null) == 1
    assert lib.detexp_f32(p, -1, dummy, dummy, null) == 1
    assert lib.detexp_f32(p, 0, null, null, null) == 0


def test_adamw_bias_correction_matches_the_oracle(lib):
    # a host-only entry point: called here without a GPU, compared bit for bit
    # with the oracle's own product loop ("MojoLearn 162M" model card, table
    # "Training": beta (0.9, 0.95))
    import numpy as np

    import oracle
    for step in (1, 2, 7, 251, 20000, 5_000_000):
        for b1, b2 in ((0.9, 0.95), (0.5, 0.999), (0.0, 1.0), (1.0, 0.99999994)):
            got = detlib.det_adamw_bias_correction(step, b1, b2)
            want = oracle.adamw_bias_correction(step, b1, b2)
            assert np.asarray(got, np.float32).view(np.uint32).tolist() == \
                np.asarray(want, np.float32).view(np.uint32).tolist(), (step, b1, b2)
    bc1, bc2 = ctypes.c_float(), ctypes.c_float()
    f = lib.det_adamw_bias_correction
    assert f(0, ctypes.c_float(0.9), ctypes.c_float(0.95), ctypes.byref(bc1),
             ctypes.byref(bc2)) == 1                                   # step < 1
    assert f(3, ctypes.c_float(1.5), ctypes.c_float(0.95), ctypes.byref(bc1),
             ctypes.byref(bc2)) == 1                                   # beta > 1
    assert f(3, ctypes.c_float(float("nan")), ctypes.c_float(0.95), ctypes.byref(bc1),
             ctypes.byref(bc2)) == 1                                   # NaN beta
    assert f(3, ctypes.c_float(0.9), ctypes.c_float(0.95), None, ctypes.byref(bc2)) == 1


def test_binding_refuses_cpu_tensors(lib):
    import torch
    with pytest.raises(TypeError):
        detlib.detgemm_f32(torch.zeros(2, 2), torch.zeros(2, 2))
