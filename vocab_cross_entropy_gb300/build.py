"""Build libvce.so in-tree from csrc/*.cu for sm_103a (nvcc, one translation unit per file,
compiled in parallel, then linked with the static CUDA runtime).

    python -m vocab_cross_entropy_gb300.build [--force] [--verbose] [--debug-checks]

--debug-checks builds libvce_debug.so instead: the same library with device-side index
checks (csrc/vce_check.cuh) compiled in.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libvce.so")
# the debug build: the same sources with device-side index checks (csrc/vce_check.cuh)
BUILD_DEBUG = os.path.join(PKG, "_build_debug")
LIB_DEBUG = os.path.join(PKG, "libvce_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Hidden symbol visibility: only the C ABI (VCE_API in include/*.h) is exported, so two builds
# loaded in one process (the release and the debug-check library) share no internal symbol.
NVCC_FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC,-O2,-fvisibility=hidden", "-I", INCLUDE,
              "-I", CSRC, "--expt-relaxed-constexpr"]


def _nvcc():
    for c in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if c and (os.path.isabs(c) and os.path.exists(c) or not os.path.isabs(c)):
            return c
    return "nvcc"


def _deps():
    return sorted(glob.glob(os.path.join(CSRC, "*.cuh")) + glob.glob(os.path.join(CSRC, "*.h")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def _stale(target, sources):
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(s) > t for s in sources)


def build(force: bool = False, verbose: bool = False, debug_checks: bool = False) -> str:
    """Compile libvce.so (or, with debug_checks, libvce_debug.so with -DVCE_DEBUG_CHECKS)."""
    build_dir, lib = (BUILD_DEBUG, LIB_DEBUG) if debug_checks else (BUILD, LIB)
    flags = NVCC_FLAGS + (["-DVCE_DEBUG_CHECKS"] if debug_checks else [])
    os.makedirs(build_dir, exist_ok=True)
    srcs = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    deps = _deps()
    nvcc = _nvcc()
    objs = []
    jobs = []
    for s in srcs:
        o = os.path.join(build_dir, os.path.basename(s)[:-3] + ".o")
        objs.append(o)
        if force or _stale(o, [s] + deps):
            jobs.append([nvcc, *ARCH, *flags, "-c", s, "-o", o] + (["-Xptxas", "-v"] if verbose else []))

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed ({' '.join(cmd)}):\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)

    if jobs:
        with ThreadPoolExecutor(max(1, min(len(jobs), os.cpu_count() or 1))) as ex:
            list(ex.map(run, jobs))
    if force or jobs or _stale(lib, objs):
        tmp = lib + f".tmp{os.getpid()}"
        run([nvcc, *ARCH, "-shared", "-o", tmp, *objs])
        os.replace(tmp, lib)
    return lib


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="--verbose" in sys.argv,
                debug_checks="--debug-checks" in sys.argv))
