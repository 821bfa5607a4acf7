"""Build the C-ABI library ``lib/libmvp.so`` for sm_103a with nvcc.

Each ``csrc/*.cu`` translation unit is compiled in parallel, then linked into
one shared library (static CUDA runtime) next to this file.  Run as
``python -m masked_varlen_prefill_gb300._build`` or through
``__graft_entry__.build()``.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(PKG, "csrc")
LIBDIR = os.path.join(PKG, "lib")
LIB = os.path.join(LIBDIR, "libmvp.so")
OBJDIR = os.path.join(PKG, "_build")
# The bounds-checked build: the same sources with MVP_DEBUG_BOUNDS, linked
# into a second library that tests load next to the product one.
DEBUG_LIB = os.path.join(LIBDIR, "libmvp_debug.so")
DEBUG_OBJDIR = os.path.join(PKG, "_build_debug")
DEBUG_FLAGS = ["-DMVP_DEBUG_BOUNDS"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-O2",
                     "--expt-relaxed-constexpr", "-Xptxas", "-v"]


def _nvcc():
    nvcc = shutil.which("nvcc")
    if nvcc is None:
        cand = "/usr/local/cuda/bin/nvcc"
        if os.path.exists(cand):
            return cand
        raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libmvp.so")
    return nvcc


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _compile(nvcc, src, objdir, extra):
    obj = os.path.join(objdir, os.path.basename(src)[:-3] + ".o")
    cmd = [nvcc, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
    r = subprocess.run(cmd, capture_output=True, text=True)
    log = r.stdout + r.stderr
    if r.returncode != 0:
        raise RuntimeError(f"nvcc failed for {src}:\n{log}")
    return obj, log


def _link(nvcc, objs, lib):
    tmp = lib + ".tmp"
    cmd = [nvcc, *ARCH, "-shared", "-o", tmp, *sorted(objs), "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}{r.stderr}")
    os.replace(tmp, lib)


def build(verbose: bool = False, jobs: int | None = None, debug_bounds: bool = True) -> str:
    """Compile every translation unit (and, with debug_bounds, again with
    MVP_DEBUG_BOUNDS) in parallel and link libmvp.so (and libmvp_debug.so)."""
    nvcc = _nvcc()
    variants = [(OBJDIR, LIB, [])] + ([(DEBUG_OBJDIR, DEBUG_LIB, DEBUG_FLAGS)] if debug_bounds else [])
    for objdir, _, _ in variants:
        os.makedirs(objdir, exist_ok=True)
    os.makedirs(LIBDIR, exist_ok=True)
    srcs = sources()
    jobs = jobs or min(len(srcs) * len(variants), os.cpu_count() or 4)
    logs = {}
    objs = {objdir: [] for objdir, _, _ in variants}
    with cf.ThreadPoolExecutor(max_workers=jobs) as ex:
        futs = {ex.submit(_compile, nvcc, s, objdir, extra): (s, objdir) for s in srcs for objdir, _, extra in variants}
        for f in cf.as_completed(futs):
            src, objdir = futs[f]
            obj, log = f.result()
            objs[objdir].append(obj)
            if objdir == OBJDIR:
                logs[src] = log
    for objdir, lib, _ in variants:
        _link(nvcc, objs[objdir], lib)
    with open(os.path.join(OBJDIR, "ptxas.log"), "w") as f:
        for s in srcs:
            f.write(f"==== {os.path.basename(s)}\n{logs.get(s, '')}\n")
    if verbose:
        for s in srcs:
            print(f"==== {os.path.basename(s)}\n{logs.get(s, '')}")
    return LIB


if __name__ == "__main__":
    print(build(verbose="-v" in sys.argv))
