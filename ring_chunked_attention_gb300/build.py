"""Build libringattn.so in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` compiles to an object in parallel, then one link step.
The result lands beside this file (git-ignored).  Run as a script or call
:func:`build`.  ``--debug`` (``build(debug=True)``) builds the bounds-checked
flavour instead, ``libringattn_debug.so`` (compiled with ``RA_DEBUG``: every
global address a kernel computes is checked against its buffer; see
``include/ringattn.h``), which the binding loads when the environment variable
``RA_DEBUG`` is ``1``; ``--trace`` builds ``libringattn_trace.so`` (``RA_TRACE``:
per-role cycle counters in the forward kernel), loaded when ``RA_TRACE`` is ``1``.
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libringattn.so")
DEBUG_LIB = os.path.join(HERE, "libringattn_debug.so")
TRACE_LIB = os.path.join(HERE, "libringattn_trace.so")
SOURCES = ["ra_api.cu", "ra_fwd.cu", "ra_bwd.cu", "ra_merge.cu", "ra_ceil.cu"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _flags(extra=()):
    return ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                   "-I", INCLUDE, "-I", CSRC, "--expt-relaxed-constexpr", *extra]


def _stale(lib: str) -> bool:
    if not os.path.exists(lib):
        return True
    t = os.path.getmtime(lib)
    deps = [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "ringattn.h"),
                                                               os.path.abspath(__file__)]
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False, ptxas_info: bool = False,
          debug: bool = False, trace: bool = False) -> str:
    if debug and trace:
        raise ValueError("one flavour at a time: debug or trace")
    lib = DEBUG_LIB if debug else TRACE_LIB if trace else LIB
    if not force and not _stale(lib):
        return lib
    nvcc = _nvcc()
    build_dir = BUILD_DIR + ("_debug" if debug else "_trace" if trace else "")
    os.makedirs(build_dir, exist_ok=True)
    extra = ((["-Xptxas", "-v"] if ptxas_info else []) + (["-DRA_DEBUG"] if debug else [])
             + (["-DRA_TRACE"] if trace else []))

    def compile_one(src):
        obj = os.path.join(build_dir, src.replace(".cu", ".o"))
        cmd = [nvcc, *_flags(extra), "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed for {src}:\n{r.stderr}")
        return obj, r.stderr

    with cf.ThreadPoolExecutor(len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if verbose or ptxas_info:
        for _, err in results:
            if err:
                sys.stderr.write(err)
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-o", tmp, *[o for o, _ in results]]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, ptxas_info="-v" in sys.argv,
                debug="--debug" in sys.argv, trace="--trace" in sys.argv))
