"""Builds libtern.so (the C-ABI library) in-tree with nvcc for sm_103a.

Each CUDA translation unit is compiled in parallel, then linked into
``ternary_weight_linear_block_gb300/libtern.so``.  No cmake, no torch
extension machinery: the library has a plain C ABI (include/tern.h).
"""

from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
OUT_DIR = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libtern.so")
SOURCES = ["tern_abi.cu", "fwht.cu", "pack.cu", "gemv.cu", "gemm.cu", "noalloc.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
CFLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
          "--expt-relaxed-constexpr", "-I", os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return p.returncode, p.stdout


def _inputs():
    """Every file the library is built from."""
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    inc = os.path.join(ROOT, "include")
    files += [os.path.join(inc, f) for f in os.listdir(inc)]
    files.append(os.path.abspath(__file__))
    return [f for f in files if os.path.isfile(f)]


def is_stale() -> bool:
    """True when libtern.so is missing or older than any of its sources."""
    if not os.path.exists(LIB):
        return True
    built = os.path.getmtime(LIB)
    return any(os.path.getmtime(f) > built for f in _inputs())


def ensure_built() -> str:
    """Build libtern.so if it is missing or stale; returns its path."""
    if is_stale():
        build()
    return LIB


def build(verbose: bool = False, ptxas_info: bool = False) -> str:
    """Compile every translation unit and link libtern.so; returns its path."""
    nvcc = _nvcc()
    os.makedirs(OUT_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if ptxas_info else []

    def compile_one(src):
        obj = os.path.join(OUT_DIR, src.replace(".cu", ".o"))
        cmd = [nvcc, *ARCH, *CFLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        rc, out = _run(cmd)
        return src, obj, rc, out

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    failed = [r for r in results if r[2] != 0]
    for src, _, rc, out in results:
        if verbose or rc != 0 or ptxas_info:
            sys.stderr.write(f"--- {src} (rc={rc})\n{out}")
    if failed:
        raise RuntimeError("nvcc failed for: " + ", ".join(r[0] for r in failed))
    tmp = LIB + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *[r[1] for r in results]]
    rc, out = _run(cmd)
    if rc != 0:
        sys.stderr.write(out)
        raise RuntimeError("link failed")
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv, ptxas_info="--ptxas" in sys.argv))
