"""Builds the C-ABI shared library ``_build/libpwsgemm.so`` for sm_103a with nvcc,
and the measurement kernels bench.py uses (``_build/libpwspeaks.so``).

Each translation unit compiles in parallel; the objects are linked into one
shared library (CUDA runtime linked statically, no libcuda link: the driver's
tensor-map encoder is fetched through the runtime's entry-point query).

    python -m pipelined_warp_specialized_gb300.build [--force] [--ptxas-verbose]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libpwsgemm.so")
PEAKS_PATH = os.path.join(OUT_DIR, "libpwspeaks.so")

SOURCES = ["runtime.cu", "gemm_s32_nn.cu", "gemm_f16_nt.cu"]
PEAKS_SOURCES = ["peaks.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("ptx.cuh", "internal.h")] + [os.path.join(INCLUDE, "pwsgemm.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")
    return cand


def _flags(verbose: bool) -> list:
    # Hidden visibility: only what a header declares with default visibility
    # is exported, so two copies of a library in one process keep separate
    # function-local statics (the compiler would otherwise bind those of
    # templates process-wide).
    f = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-fvisibility=hidden", "-I", INCLUDE,
                "-I", CSRC, "--expt-relaxed-constexpr"]
    if verbose:
        f += ["-Xptxas", "-v"]
    return f


def _stale() -> bool:
    if not os.path.exists(LIB_PATH) or not os.path.exists(PEAKS_PATH):
        return True
    t = min(os.path.getmtime(LIB_PATH), os.path.getmtime(PEAKS_PATH))
    deps = [os.path.join(CSRC, s) for s in SOURCES + PEAKS_SOURCES] + HEADERS + [os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    flags = _flags(verbose)

    def compile_one(src: str):
        obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [cc] + flags + ["-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        return src, obj, r

    with cf.ThreadPoolExecutor(max_workers=len(SOURCES + PEAKS_SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES + PEAKS_SOURCES))
    failed = [(s, r) for s, _, r in results if r.returncode != 0]
    for s, _, r in results:
        if verbose or r.returncode != 0:
            sys.stderr.write(f"--- {s}\n{r.stdout}{r.stderr}")
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(s for s, _ in failed))
    for path, srcs in ((LIB_PATH, SOURCES), (PEAKS_PATH, PEAKS_SOURCES)):
        tmp = path + f".tmp{os.getpid()}"
        cmd = [cc] + ARCH + ["-shared", "-o", tmp] + [o for s, o, _ in results if s in srcs]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            sys.stderr.write(r.stdout + r.stderr)
            raise RuntimeError("link failed")
        os.replace(tmp, path)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--ptxas-verbose" in sys.argv))
