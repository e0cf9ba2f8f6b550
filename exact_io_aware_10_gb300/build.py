"""Builds the C-ABI shared library ``lib/libfa_gb300.so`` for sm_103a.

Each CUDA translation unit is compiled by its own ``nvcc`` process (in
parallel), then the objects are linked with the static CUDA runtime.  The
output is rebuilt only when a source or header is newer than the library.
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
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(PKG, "_build")
LIB_DIR = os.path.join(PKG, "lib")
LIB_NAME = "libfa_gb300.so"
LIB_PATH = os.path.join(LIB_DIR, LIB_NAME)
# the same sources built with FA_DEBUG: device bounds checks on every global
# access the kernels' threads issue (load it with FA_GB300_LIB=<this path>)
DEBUG_BUILD_DIR = os.path.join(PKG, "_build_debug")
DEBUG_LIB_PATH = os.path.join(LIB_DIR, "libfa_gb300_debug.so")

SOURCES = ["fa_api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_decode.cu", "fa_graph.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "--expt-relaxed-constexpr", "-Xcompiler", "-fPIC,-O2",
              "-I" + INCLUDE, "-I" + CSRC]


def nvcc_path() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise FileNotFoundError("nvcc not found (set NVCC or put the CUDA toolkit on PATH)")


def _deps():
    files = [os.path.join(CSRC, f) for f in os.listdir(CSRC)]
    files.append(os.path.join(INCLUDE, "fa.h"))
    files.append(os.path.abspath(__file__))
    return files


def _stale(path) -> bool:
    if not os.path.exists(path):
        return True
    t = os.path.getmtime(path)
    return any(os.path.getmtime(f) > t for f in _deps())


def _run(cmd):
    p = subprocess.run(cmd, stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    return p.returncode, p.stdout


def build(force: bool = False, verbose: bool = False, ptxas_verbose: bool = False, debug: bool = False) -> str:
    """Compile every translation unit for sm_103a and link the shared library
    (``debug``: the FA_DEBUG variant with device bounds checks, a separate
    library).  Returns the library path; raises RuntimeError with the
    compiler output on failure."""
    lib_path = DEBUG_LIB_PATH if debug else LIB_PATH
    build_dir = DEBUG_BUILD_DIR if debug else BUILD_DIR
    if not force and not _stale(lib_path):
        return lib_path
    os.makedirs(build_dir, exist_ok=True)
    os.makedirs(LIB_DIR, exist_ok=True)
    nvcc = nvcc_path()
    extra = ["-Xptxas", "-v"] if ptxas_verbose else []
    if debug:
        extra.append("-DFA_DEBUG")
    jobs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        jobs.append((src, [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj], obj))
    with ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        results = list(ex.map(lambda j: (j[0], *_run(j[1])), jobs))
    log = []
    for src, rc, out in results:
        if out.strip() and (verbose or ptxas_verbose or rc != 0):
            log.append(f"--- {src}\n{out}")
        if rc != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{out}")
    tmp = lib_path + ".tmp"
    rc, out = _run([nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp,
                    *[j[2] for j in jobs], "-ldl"])
    if rc != 0:
        raise RuntimeError(f"link failed:\n{out}")
    os.replace(tmp, lib_path)
    if log:
        sys.stderr.write("\n".join(log) + "\n")
    return lib_path


if __name__ == "__main__":
    force = "--force" in sys.argv
    print(build(force=force, verbose="-v" in sys.argv, ptxas_verbose="--ptxas" in sys.argv,
                debug="--debug" in sys.argv))
