"""Builds libkvgqa.so in-tree with nvcc for sm_103a.

Each .cu translation unit compiles in its own nvcc process (in parallel), then
one nvcc call links the shared library next to this file.  No cmake, no torch
extension machinery: the library has a plain C ABI.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG_DIR)
CSRC = os.path.join(PKG_DIR, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG_DIR, "_build")
LIB_PATH = os.path.join(PKG_DIR, "libkvgqa.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["api.cu", "rope_kv_store.cu", "flash_decode.cu", "flash_decode_f16.cu", "prefill_attention.cu",
           "wait_check.cu"]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def common_flags(extra=()):
    return ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-I", INCLUDE, "-I", CSRC,
                   "--expt-relaxed-constexpr", *extra]


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build_library(verbose: bool = False, ptxas_info: bool = False, force: bool = False) -> str:
    """Compile and link libkvgqa.so; returns its path.  Rebuilds when a source
    or header is newer than the library (or when forced)."""
    nvcc = nvcc_path()
    os.makedirs(BUILD_DIR, exist_ok=True)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "kvgqa.h")]
    if (not force and os.path.exists(LIB_PATH)
            and os.path.getmtime(LIB_PATH) >= max(os.path.getmtime(d) for d in deps)):
        return LIB_PATH
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        out = _run([nvcc, *common_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj])
        return obj, out

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    logs = "".join(out for _, out in results)
    tmp = LIB_PATH + ".tmp"
    _run([nvcc, *ARCH, "-shared", "-o", tmp, *[obj for obj, _ in results]])
    os.replace(tmp, LIB_PATH)
    if verbose or ptxas_info:
        sys.stdout.write(logs)
    return LIB_PATH


if __name__ == "__main__":
    build_library(verbose=True, ptxas_info="-v" in sys.argv, force="-f" in sys.argv)
    print(LIB_PATH)
