"""Build libqcodec.so in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled to an object file in parallel, then the
objects are linked into a shared library next to this file.  The CUDA runtime
is linked statically, so the library depends only on the driver at run time.
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
ROOT = os.path.dirname(PKG)
BUILD_DIR = os.path.join(ROOT, "_build")
LIB_NAME = "libqcodec.so"
LIB_PATH = os.path.join(PKG, LIB_NAME)
SOURCES = ["qc_api.cu", "qc_encode.cu", "qc_encode_tma.cu", "qc_encode_clip.cu",
           "qc_encode_clip_bf16.cu", "qc_encode_bf16.cu", "qc_encode_bf16_fast.cu", "qc_decode.cu", "qc_decode_tma.cu",
           "qc_reencode.cu", "qc_reencode_other.cu", "qc_topk.cu", "qc_fp8.cu",
           "qc_encode_log.cu", "qc_reencode_log.cu", "qc_selftest.cu", "qc_encode_direct_log.cu"]
HEADERS = ["qc_device.cuh", "qc_internal.h", "qc_encode_math.cuh", "qc_encode_tma.cuh",
           "qc_encode_direct.cuh",
           "qc_reencode.cuh", "qc_pipeline.cuh", "qc_decode_math.cuh", "qc_exact_norm.cuh"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fmad=false: no multiply-add contraction; every fused op is an explicit
# __fmaf_rn.  Division and square root stay IEEE (no fast math).
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-fmad=false", "-Xcompiler", "-fPIC",
              "-Xcompiler", "-ffp-contract=off"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libqcodec")


def _inputs():
    files = [os.path.join(CSRC, s) for s in SOURCES + HEADERS]
    files.append(os.path.join(ROOT, "include", "qcodec.h"))
    files.append(os.path.abspath(__file__))
    return files


def up_to_date() -> bool:
    if not os.path.exists(LIB_PATH):
        return False
    t = os.path.getmtime(LIB_PATH)
    return all(os.path.getmtime(f) <= t for f in _inputs())


def build_library(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile and link libqcodec.so; returns its path."""
    if not force and up_to_date():
        return LIB_PATH
    os.makedirs(BUILD_DIR, exist_ok=True)
    cc = nvcc()
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, log in results:
            if log:
                print(log)
    tmp = LIB_PATH + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *[o for o, _ in results], "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    import sys
    print(build_library(force="--force" in sys.argv, verbose=True,
                        ptxas_info="--ptxas-info" in sys.argv))
