"""Build libcp.so (the C-ABI CUDA library) in-tree with nvcc for sm_103a.

Each ``csrc/*.cu`` is compiled in parallel to an object file, then linked
into ``context_parallelism_02_gb300/_build/libcp.so`` with the CUDA runtime
linked statically, so the library needs only the driver at load time.

Usage: ``python -m context_parallelism_02_gb300.build`` (or ``build()``).

``build(debug_bounds=True)`` (``--debug-bounds``) builds the checking variant
``_build/debug_bounds/libcp.so`` with ``-DCP_DEBUG_BOUNDS``: the tensor-core
kernels check every TMA tile coordinate and output row index against the
tensor extents and record CP_EBOUNDS in the error word instead of going out
of range (no trap).  Tests select it with ``_lib.variant("debug_bounds")``.
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
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD, "libcp.so")
LIB_DEBUG_BOUNDS = os.path.join(BUILD, "debug_bounds", "libcp.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2", "-I", INCLUDE, "-I", CSRC,
              "--expt-relaxed-constexpr"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libcp")


def _sources():
    return sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))


def _deps():
    return [os.path.join(CSRC, f) for f in os.listdir(CSRC)] + [os.path.join(INCLUDE, "cp.h")]


def up_to_date(lib: str = LIB) -> bool:
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=(),
          debug_bounds: bool = False) -> str:
    """Compile and link libcp.so (or its debug-bounds variant); returns its path."""
    lib = LIB_DEBUG_BOUNDS if debug_bounds else LIB
    if not force and up_to_date(lib):
        return lib
    out_dir = os.path.dirname(lib)
    os.makedirs(out_dir, exist_ok=True)
    cc = nvcc()
    if debug_bounds:
        extra_flags = (*extra_flags, "-DCP_DEBUG_BOUNDS")

    def compile_one(src):
        obj = os.path.join(out_dir, src[:-3] + ".o")
        cmd = [cc, *ARCH, *NVCC_FLAGS, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    srcs = _sources()
    with cf.ThreadPoolExecutor(max_workers=min(len(srcs), os.cpu_count() or 4)) as ex:
        objs = list(ex.map(compile_one, srcs))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [cc, *ARCH, "-shared", "-o", tmp, *objs, "-cudart", "static"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True,
                extra_flags=("-Xptxas", "-v") if "--ptxas-v" in sys.argv else (),
                debug_bounds="--debug-bounds" in sys.argv))
