"""Builds the CUDA library ``libfp8gemm.so`` in-tree for sm_103a.

The translation units compile in parallel (one nvcc per file), then link
into one shared library with the CUDA runtime linked statically.  The C ABI
is ``include/fp8gemm.h``.
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
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libfp8gemm.so")
SOURCES = ["api.cu", "gemm_nt.cu", "gemm_nt_acc.cu", "gemm_contiguous.cu", "gemm_masked.cu",
           "gemm_pair.cu", "gemm_pair256.cu", "gemm_ue8m0.cu", "gemm_ue8m0_pair.cu",
           "gemm_share.cu", "gemm_narrow.cu"]

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
                     "--expt-relaxed-constexpr", "-Xptxas", "-v", "-I", os.path.join(ROOT, "include")]
PTXAS_LOG = os.path.join(BUILD, "ptxas.log")


def nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found")
    return cand


def _deps_mtime() -> float:
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(ROOT, "include", "fp8gemm.h"))
    return max(os.path.getmtime(f) for f in files)


# the bounds-checking build: every kernel checks the invariants its accesses
# rely on and records FP8G_ERR_BOUNDS instead of faulting (see ptx.cuh)
DEBUG_LIB = os.path.join(PKG, "libfp8gemm_debug.so")
DEBUG_FLAGS = ["-DFP8G_DEBUG_BOUNDS=1"]


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Builds libfp8gemm.so and its bounds-checking twin libfp8gemm_debug.so
    (all translation units of both compiled in parallel); returns the path of
    the first."""
    deps = _deps_mtime()
    if (not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= deps and os.path.exists(DEBUG_LIB)
            and os.path.getmtime(DEBUG_LIB) >= deps):
        return LIB
    cc = nvcc()
    jobs = [(src, BUILD, list(extra_flags)) for src in SOURCES] + \
           [(src, os.path.join(BUILD, "debug"), DEBUG_FLAGS + list(extra_flags)) for src in SOURCES]
    for d in {j[1] for j in jobs}:
        os.makedirs(d, exist_ok=True)

    def compile_one(job):
        src, outdir, flags = job
        obj = os.path.join(outdir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *NVCC_FLAGS, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src} ({' '.join(flags)}):\n{r.stdout}\n{r.stderr}")
        if verbose:
            sys.stderr.write(r.stdout + r.stderr)
        return obj, r.stderr

    with ThreadPoolExecutor(min(len(jobs), max(4, os.cpu_count() or 4))) as ex:
        done = list(ex.map(compile_one, jobs))
    n = len(SOURCES)
    # the register report of every kernel of the normal build (checked by tests/test_build.py)
    with open(PTXAS_LOG, "w") as f:
        f.write("".join(log for _, log in done[:n]))
    for lib, objs in ((LIB, [o for o, _ in done[:n]]), (DEBUG_LIB, [o for o, _ in done[n:]])):
        tmp = lib + f".tmp{os.getpid()}"
        r = subprocess.run([cc, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
        os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
