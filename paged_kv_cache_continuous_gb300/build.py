"""In-tree build of libpagedattn.so for GB300 (sm_103a) with nvcc.

Each translation unit is compiled in parallel to an object file under
``_build/``; the shared library links the CUDA runtime statically, so it
needs nothing but the driver at run time.  No cmake, no torch extension
machinery: ``python -m paged_kv_cache_continuous_gb300.build``.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

PKG = Path(__file__).resolve().parent
ROOT = PKG.parent
CSRC = PKG / "csrc"
BUILD = PKG / "_build"
LIB = BUILD / "libpagedattn.so"

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
              "-I", str(ROOT / "include")]
CXX_FLAGS = ["-O2", "-std=c++17", "-fPIC", "-Wall", "-I", str(ROOT / "include")]

CU_SOURCES = ["pa_api.cu", "kv_append.cu", "decode.cu", "prefill_tc.cu", "prefill_tc2.cu", "block_copy.cu", "rope.cu"]
CXX_SOURCES = ["block_alloc.cpp", "scheduler.cpp"]


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not Path(cand).exists():
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libpagedattn")
    return cand


def _deps_mtime() -> float:
    files = list(CSRC.glob("*")) + list((ROOT / "include").glob("*.h")) + [Path(__file__)]
    return max(f.stat().st_mtime for f in files if f.is_file())


def _run(cmd):
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"build step failed: {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    return r.stdout + r.stderr


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False) -> Path:
    """Compile every CUDA/C++ source and link libpagedattn.so; returns its path."""
    if not force and LIB.exists() and LIB.stat().st_mtime >= _deps_mtime():
        return LIB
    BUILD.mkdir(exist_ok=True)
    nv = nvcc()
    jobs = []
    for src in CU_SOURCES:
        obj = BUILD / (src + ".o")
        extra = ["-Xptxas", "-v"] if ptxas_info else []
        jobs.append([nv, *ARCH, *NVCC_FLAGS, *extra, "-c", str(CSRC / src), "-o", str(obj)])
    for src in CXX_SOURCES:
        obj = BUILD / (src + ".o")
        jobs.append(["g++", *CXX_FLAGS, "-c", str(CSRC / src), "-o", str(obj)])
    with ThreadPoolExecutor(max_workers=min(len(jobs), os.cpu_count() or 4)) as ex:
        outs = list(ex.map(_run, jobs))
    if verbose or ptxas_info:
        for o in outs:
            if o.strip():
                print(o, file=sys.stderr)
    tmp = BUILD / f"libpagedattn.{os.getpid()}.so"
    objs = [str(BUILD / (s + ".o")) for s in CU_SOURCES + CXX_SOURCES]
    _run([nv, *ARCH, "-shared", "-o", str(tmp), *objs, "-ldl"])
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="--ptxas" in sys.argv))
