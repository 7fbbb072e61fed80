"""Build libcoda.so in-tree: one nvcc per translation unit in parallel, for
sm_103a only, then a shared-library link with the static CUDA runtime.
``--checked`` builds the same sources with CODA_CHECKED=1 into
libcoda_checked.so: every direct global access of the fused epilogues tests
its index against the tensor's extent first (CODA_DEVST_BOUNDS on a miss).

Usage: ``python -m gemm_epilogue_transformer_gb300.build_lib [--force] [--checked] [-v]``
"""
from __future__ import annotations

import argparse
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(PKG, "libcoda.so")
LIB_CHECKED = os.path.join(PKG, "libcoda_checked.so")

SOURCES = ["runtime.cu", "aux.cu", "unfused.cu", "gemm_fwd.cu", "gemm_bwd.cu", "gemm_chain.cu", "block.cu",
           "gemm_fp8.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: libcoda needs the CUDA 13 toolkit to build")


def _deps():
    out = [os.path.join(INCLUDE, "coda.h")]
    for f in os.listdir(CSRC):
        if f.endswith((".cuh", ".h", ".cu")):
            out.append(os.path.join(CSRC, f))
    return out


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, checked: bool = False) -> str:
    """Compile every translation unit for sm_103a and link libcoda.so (or, with
    checked, libcoda_checked.so); return its path."""
    lib = LIB_CHECKED if checked else LIB
    if not force and up_to_date(lib):
        return lib
    bdir = os.path.join(BUILD, "checked") if checked else BUILD
    os.makedirs(bdir, exist_ok=True)
    cc = nvcc()
    flags = ["-std=c++17", "-O3", "-lineinfo", *ARCH, "-Xcompiler", "-fPIC", "-I", INCLUDE,
             "--expt-relaxed-constexpr", "-diag-suppress", "177"]
    if checked:
        flags += ["-DCODA_CHECKED=1"]
    if ptxas_verbose:
        flags += ["-Xptxas", "-v"]
    procs = []
    objs = []
    for src in SOURCES:
        obj = os.path.join(bdir, src.replace(".cu", ".o"))
        objs.append(obj)
        cmd = [cc, *flags, "-c", os.path.join(CSRC, src), "-o", obj]
        if verbose:
            print(" ".join(cmd), flush=True)
        procs.append((src, subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)))
    failed = []
    for src, p in procs:
        out, _ = p.communicate()
        if out and (verbose or ptxas_verbose or p.returncode):
            print(f"--- {src}\n{out}", flush=True)
        if p.returncode:
            failed.append(src)
    if failed:
        raise RuntimeError(f"nvcc failed for {failed}")
    tmp = lib + ".tmp"
    cmd = [cc, "-shared", *ARCH, "-o", tmp, *objs]
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    if r.returncode:
        raise RuntimeError(f"link failed:\n{r.stdout}")
    os.replace(tmp, lib)
    return lib


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--force", action="store_true")
    ap.add_argument("-v", "--verbose", action="store_true")
    ap.add_argument("--ptxas-verbose", action="store_true")
    ap.add_argument("--checked", action="store_true", help="build libcoda_checked.so (bounds-tested epilogues)")
    a = ap.parse_args(argv)
    print(build(force=a.force, verbose=a.verbose, ptxas_verbose=a.ptxas_verbose, checked=a.checked))


if __name__ == "__main__":
    sys.exit(main())
