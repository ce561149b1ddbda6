"""Builds libdetfp32.so in-tree from csrc/*.cu for sm_103a.

The numerics flags are part of the profile: no FMA contraction of separate
multiply/add (-fmad=false on the device, -ffp-contract=off for the host code
that forms AdamW's bias corrections), no flush-to-zero (-ftz=false), IEEE
division and square root (-prec-div=true -prec-sqrt=true), never
--use_fast_math.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
LIB = os.path.join(HERE, "libdetfp32.so")
BUILD_DIR = os.path.join(HERE, "_build")
SOURCES = ["gemm.cu", "gemm_n64.cu", "gemm_m128.cu", "rowops.cu", "rmsbwd.cu", "shardsum.cu", "block.cu",
           "adamw.cu", "api.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NUMERICS = ["-fmad=false", "-ftz=false", "-prec-div=true", "-prec-sqrt=true"]


def nvcc() -> str:
    cand = os.environ.get("NVCC") or shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return cand


def common_flags(extra=()):
    return [*ARCH, "-O3", "-lineinfo", "-std=c++17", *NUMERICS,
            "-Xcompiler", "-fPIC,-fvisibility=hidden,-ffp-contract=off",
            "-I", os.path.join(ROOT, "include"), "-I", CSRC, *extra]


def _stale() -> bool:
    if not os.path.exists(LIB):
        return True
    t = os.path.getmtime(LIB)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(ROOT, "include", "detfp32.h"))
    deps.append(os.path.abspath(__file__))
    return any(os.path.getmtime(d) > t for d in deps)


def build_variant(defines, out_path: str) -> str:
    """Compile a separate copy of the library with extra -D flags into out_path
    (the test suite's copy with a shortened GEMM wait). Never the shipped
    library: LIB is not touched."""
    work = out_path + ".build"
    os.makedirs(work, exist_ok=True)
    dflags = [f"-D{d}" for d in defines]

    def compile_one(src):
        obj = os.path.join(work, src.replace(".cu", ".o"))
        cmd = [nvcc(), *common_flags(dflags), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-Xlinker", "--no-undefined",
           "-o", out_path, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    return out_path


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every translation unit in parallel and link the shared library.
    Returns the library path."""
    if not force and not _stale():
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc(), *common_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stdout + r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log.strip():
                print(log, file=sys.stderr)
    tmp = LIB + f".tmp{os.getpid()}"
    # --no-undefined: an unresolved symbol fails the build, not the first load
    cmd = [nvcc(), *ARCH, "-shared", "-Xcompiler", "-fPIC", "-Xlinker", "--no-undefined",
           "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                ptxas_info="--ptxas-info" in sys.argv))
