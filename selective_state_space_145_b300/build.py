"""Build libssm.so (the CUDA kernels and the C ABI) in-tree with nvcc for sm_103a.

Every .cu file under csrc/ is compiled to an object in _build/ (in parallel) and the
objects are linked into selective_state_space_145_b300/libssm.so. A rebuild happens when
any source or header is newer than the library.

The debug variant, libssm_debug.so (objects in _build/debug/), is the same sources compiled
with SSM_DEBUG_BOUNDS: every checked global access is range-tested against its tensor and a
violation sets a device error word (ssm_debug_bounds_status) instead of touching memory.
"""

from __future__ import annotations

import concurrent.futures as cf
import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(ROOT, "_build")
LIB = os.path.join(HERE, "libssm.so")
DEBUG_LIB = os.path.join(HERE, "libssm_debug.so")
VARIANTS = {"release": (LIB, BUILD, []), "debug": (DEBUG_LIB, os.path.join(BUILD, "debug"), ["-DSSM_DEBUG_BOUNDS"])}

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-fvisibility=hidden",
              "--expt-relaxed-constexpr", "-I", INCLUDE, "-I", CSRC]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")))


def _deps():
    return sources() + glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) + \
        glob.glob(os.path.join(INCLUDE, "*.h")) + [os.path.abspath(__file__)]


def up_to_date(variant: str = "release") -> bool:
    lib = VARIANTS[variant][0]
    if not os.path.exists(lib):
        return False
    t = os.path.getmtime(lib)
    return all(os.path.getmtime(p) <= t for p in _deps())


def build(force: bool = False, verbose: bool = False, extra_flags=None, variant: str = "release") -> str:
    """Compile and link libssm.so (variant "release") or libssm_debug.so (variant "debug") if
    needed; return its path. Raises on a compiler error."""
    lib, bdir, vflags = VARIANTS[variant]
    if not force and up_to_date(variant):
        return lib
    os.makedirs(bdir, exist_ok=True)
    nvcc = _nvcc()
    flags = NVCC_FLAGS + vflags + list(extra_flags or [])

    def compile_one(src):
        obj = os.path.join(bdir, os.path.basename(src) + ".o")
        cmd = [nvcc] + ARCH + flags + ["-c", src, "-o", obj]
        if verbose:
            print(" ".join(cmd), file=sys.stderr)
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        objs = list(ex.map(compile_one, sources()))
    tmp = lib + f".tmp{os.getpid()}"
    cmd = [nvcc] + ARCH + ["-shared", "-o", tmp] + objs
    if verbose:
        print(" ".join(cmd), file=sys.stderr)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv,
                extra_flags=["-Xptxas", "-v"] if "--ptxas-v" in sys.argv else None,
                variant="debug" if "--debug" in sys.argv else "release"))
