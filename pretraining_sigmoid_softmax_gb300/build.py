"""Builds the in-tree shared library ``libmoe_gb300.so`` from ``csrc/*.cu`` with nvcc.

Every translation unit is compiled for sm_103a only, in parallel, then linked into one
shared object next to this file (the CUDA runtime is linked statically). Run as a module
(``python -m pretraining_sigmoid_softmax_gb300.build``) or call ``build_library()``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(HERE, "csrc")
LIB_NAME = "libmoe_gb300.so"
LIB_PATH = os.path.join(HERE, LIB_NAME)
BUILD_DIR = os.path.join(HERE, "_build")
GENCODE = "-gencode=arch=compute_103a,code=sm_103a"
SOURCES = ["status.cu", "route.cu", "route_tc.cu", "permute.cu", "grouped_gemm.cu", "fp8.cu"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the MoE library needs the CUDA toolkit to build")


def _compile(nvcc: str, src: str, extra: list[str]) -> str:
    obj = os.path.join(BUILD_DIR, os.path.splitext(os.path.basename(src))[0] + ".o")
    cmd = [nvcc, GENCODE, "-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
           "-diag-suppress", "177", "-c", os.path.join(CSRC, src), "-o", obj] + extra
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"nvcc failed on {src}:\n{res.stdout}\n{res.stderr}")
    return obj


def _stale() -> bool:
    if not os.path.exists(LIB_PATH):
        return True
    t = os.path.getmtime(LIB_PATH)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    deps.append(os.path.join(HERE, "..", "include", "moe_gb300.h"))
    deps.append(__file__)
    return any(os.path.getmtime(p) > t for p in deps if os.path.exists(p))


def build_library(force: bool = False, extra: list[str] | None = None, verbose: bool = False) -> str:
    """Compile and link the library if any source is newer; returns its path."""
    if not force and not _stale():
        return LIB_PATH
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = list(extra or [])
    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(lambda s: _compile(nvcc, s, extra), SOURCES))
    tmp = LIB_PATH + ".tmp"
    cmd = [nvcc, GENCODE, "-shared", "-o", tmp] + objs
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"link failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIB_PATH)
    if verbose:
        print(f"built {LIB_PATH}")
    return LIB_PATH


if __name__ == "__main__":
    build_library(force="--force" in sys.argv, verbose=True)
