"""Build the C-ABI library ``libddpreducer.so`` in-tree with nvcc for sm_103a.

    python -m reduction_reducer_gb300.build [-v] [--all | --trace]

Translation units are compiled in parallel into ``_build/`` next to this
file and linked (static CUDA runtime) into ``libddpreducer.so`` beside the
package.  No fast-math: the reduction must round exactly like IEEE fp32.
"""

from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(PKG, "libddpreducer.so")
# Bounds-checking variant of the same sources (-DDDP_DEBUG): every kernel
# checks the ranges it walks and the bulk copies it issues, and records the
# first failure instead of touching memory out of range.
DEBUG_BUILD = os.path.join(PKG, "_build_debug")
DEBUG_LIB = os.path.join(PKG, "libddpreducer_debug.so")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
# Size of the static device scratch of ddp_reduce_all_noalloc (256 KiB).
NOALLOC_SCRATCH_BYTES = 256 * 1024
COMMON = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC,-Wall", "-I" + INCLUDE, "-I" + CSRC,
          f"-DDDP_NOALLOC_SCRATCH_BYTES={NOALLOC_SCRATCH_BYTES}"]
SOURCES = ["ddp_host.cpp", "ddp_kernels.cu", "ddp_kernels_tma.cu", "ddp_noalloc.cu", "ddp_shard.cpp"]


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libddpreducer.so")


def _run(cmd, verbose):
    if verbose:
        print(" ".join(cmd), flush=True)
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"command failed ({r.returncode}): {' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
    if verbose and (r.stdout or r.stderr):
        print(r.stdout + r.stderr, flush=True)
    return r


def build(verbose: bool = False, extra_flags=(), lib_path: str = LIB, build_dir: str = BUILD) -> str:
    """Compile and link; returns the library path.  ``extra_flags`` are passed
    to every nvcc compile (e.g. a -D tuning constant for a variant built at
    ``lib_path`` in ``build_dir``)."""
    os.makedirs(build_dir, exist_ok=True)
    cc = nvcc()
    jobs = []
    for src in SOURCES:
        obj = os.path.join(build_dir, os.path.splitext(src)[0] + ".o")
        cmd = [cc, *ARCH, *COMMON, *extra_flags, "-c", os.path.join(CSRC, src), "-o", obj]
        jobs.append((cmd, obj))
    with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
        list(ex.map(lambda j: _run(j[0], verbose), jobs))
    tmp = lib_path + ".tmp"
    _run([cc, *ARCH, "-shared", "-o", tmp, *[o for _, o in jobs], "-cudart", "static",
          "-Xlinker", "-z,defs", "-lpthread", "-ldl", "-lrt"], verbose)
    os.replace(tmp, lib_path)
    return lib_path


def build_debug(verbose: bool = False) -> str:
    """The bounds-checking variant at ``DEBUG_LIB``."""
    return build(verbose, extra_flags=("-DDDP_DEBUG=1",), lib_path=DEBUG_LIB, build_dir=DEBUG_BUILD)


# Launch-trace variant (-DDDP_TRACE): the bulk-copy kernel records
# %globaltimer stamps per CTA (ddp_read_launch_trace); a diagnostics build.
TRACE_BUILD = os.path.join(PKG, "_build_trace")
TRACE_LIB = os.path.join(PKG, "libddpreducer_trace.so")


def build_trace(verbose: bool = False) -> str:
    """The launch-trace variant at ``TRACE_LIB``."""
    return build(verbose, extra_flags=("-DDDP_TRACE=1",), lib_path=TRACE_LIB, build_dir=TRACE_BUILD)


def build_all(verbose: bool = False):
    """Release, bounds-checking and launch-trace builds, compiled side by side."""
    with cf.ThreadPoolExecutor(max_workers=3) as ex:
        rel = ex.submit(build, verbose)
        dbg = ex.submit(build_debug, verbose)
        trc = ex.submit(build_trace, verbose)
        return rel.result(), dbg.result(), trc.result()


if __name__ == "__main__":
    if "--trace" in sys.argv:
        print(build_trace(verbose="-v" in sys.argv))
    else:
        print(build_all(verbose="-v" in sys.argv) if "--all" in sys.argv else build(verbose="-v" in sys.argv))
