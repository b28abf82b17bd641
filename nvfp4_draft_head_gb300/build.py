"""Compile libdrafthead.so (the CUDA kernels and the C ABI) for sm_103a.

Each translation unit is compiled by its own nvcc process in parallel, then
linked into ``nvfp4_draft_head_gb300/_build/libdrafthead.so``. Usage:
``python -m nvfp4_draft_head_gb300.build`` (or ``build()`` from Python).
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(os.path.dirname(HERE), "include")
OUT_DIR = os.path.join(HERE, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libdrafthead.so")

SOURCES = ["dh_abi.cu", "dh_quantize.cu", "dh_gemv.cu", "dh_gemv_nvfp4.cu", "dh_gemv_fp8.cu",
           "dh_gemv_bf16.cu", "dh_static_ws.cu", "dh_gemv_nvfp4p.cu", "dh_gemv_nvfp4p_ldg.cu", "dh_pack.cu",
           "dh_gemv_w8a8.cu", "dh_gemv_linear.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# -fno-gnu-unique: the launchers' per-device caches (function-local statics of
# templates) stay private to each loaded copy of the library instead of being
# merged process-wide, so two builds loaded side by side do not share them.
NVCC_FLAGS = ["-std=c++17", "-O3", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fno-gnu-unique",
              "-I", INCLUDE, "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libdrafthead.so")


def _inputs():
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(INCLUDE, "drafthead.h"))
    return deps


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    return any(os.path.getmtime(p) > t for p in _inputs())


def build(force: bool = False, verbose: bool = False) -> str:
    """Build the library if any source is newer than it; returns its path."""
    if not force and not _stale():
        return LIB_PATH
    os.makedirs(OUT_DIR, exist_ok=True)
    cc = nvcc()
    objs = []

    def compile_one(src):
        obj = os.path.join(OUT_DIR, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        return obj, r.stderr

    with ThreadPoolExecutor(len(SOURCES)) as ex:
        for obj, log in ex.map(compile_one, SOURCES):
            objs.append(obj)
            if verbose and log:
                sys.stderr.write(log)
    tmp = LIB_PATH + f".{os.getpid()}.tmp"
    cmd = [cc, *ARCH, "-shared", "--cudart", "shared", "-o", tmp, *objs,
           "-Xlinker", "-rpath", "-Xlinker", "/usr/local/cuda/lib64"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, LIB_PATH)
    return LIB_PATH


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
