"""Build the C-ABI shared library ``libfa_gb300.so`` in-tree with nvcc.

One translation unit per kernel family, compiled in parallel for sm_103a
only, then linked into a shared library next to this file.  No cmake, no
torch extension machinery: the library has a plain C ABI (include/fa.h).
"""
from __future__ import annotations

import os
import shutil
import subprocess
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = PKG / "libfa_gb300.so"
SOURCES = ["api.cu", "fwd_tc.cu", "fwd_tc1.cu", "bwd_tc.cu", "bwd_tc128.cu", "simt_f32.cu", "aux_kernels.cu",
           "noalloc.cu", "fwd_fp8.cu", "fp8_quant.cu"]
HEADERS = ["common.cuh", "bwd_items.cuh", "fa_internal.h", "fwd_plan.cuh", "fp8.cuh"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
         "-Xptxas", "-warn-spills"]


def _nvcc():
    n = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(n):
        raise RuntimeError("nvcc not found; the CUDA toolkit is required to build libfa_gb300.so")
    return n


def _stale():
    if not LIB.exists():
        return True
    t = LIB.stat().st_mtime
    deps = [CSRC / s for s in SOURCES + HEADERS] + [PKG.parent / "include" / "fa.h", Path(__file__)]
    return any(d.stat().st_mtime > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile (if needed) and return the path of libfa_gb300.so."""
    if not force and not _stale():
        return LIB
    nvcc = _nvcc()
    BUILD.mkdir(exist_ok=True)
    inc = ["-I", str(CSRC), "-I", str(PKG.parent / "include")]

    def compile_one(src):
        obj = BUILD / (Path(src).stem + ".o")
        cmd = [nvcc, *ARCH, *FLAGS, *inc, "-c", str(CSRC / src), "-o", str(obj)]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, " ".join(cmd), r.stderr))
        if verbose and r.stderr:
            print(r.stderr)
        return obj

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        objs = list(ex.map(compile_one, SOURCES))
    tmp = LIB.with_suffix(".so.tmp")
    cmd = [nvcc, *ARCH, "-shared", "-o", str(tmp), *map(str, objs)]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (" ".join(cmd), r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    import sys
    print(build(force="--force" in sys.argv, verbose=True))
