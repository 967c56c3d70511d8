"""Build libzero_gb300.so in-tree for sm_103a.

One nvcc per translation unit, run in parallel, then one shared-library link.
Float contraction is off (-fmad=false) on top of the explicit round-to-nearest
intrinsics in the kernels, so every fp32 operation of the step is one IEEE
rounding.  Set ZERO_PTXAS_VERBOSE=1 to print register and spill counts.
"""
import os
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
BUILD_DIR = os.path.join(HERE, "_build")
LIB = os.path.join(BUILD_DIR, "libzero_gb300.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
SOURCES = ["zero_host.cu", "k_fused.cu", "k_twopass.cu", "k_update.cu", "k_gather.cu", "k_noalloc.cu", "zero_fetch.cu", "k_async.cu", "zero_pa.cu"]
HEADERS = ["zero_internal.h", "dev_common.cuh", "dev_state.cuh", "nvtx_ranges.h", "host_ptrs.h"]
FLAGS = ["-O3", "-lineinfo", "-std=c++17", "-fmad=false", "-Xcompiler", "-fPIC,-Wall",
         "-I" + INCLUDE, "-I" + CSRC]


def _deps():
    return ([os.path.join(CSRC, s) for s in SOURCES + HEADERS] + [os.path.join(INCLUDE, "zero_gb300.h")])


def _stale(out):
    return not os.path.exists(out) or any(os.path.getmtime(d) > os.path.getmtime(out) for d in _deps())


def build(force: bool = False, verbose: bool = False) -> str:
    if not force and not _stale(LIB):
        return LIB
    os.makedirs(BUILD_DIR, exist_ok=True)
    extra = ["-Xptxas", "-v"] if (verbose or os.environ.get("ZERO_PTXAS_VERBOSE")) else []

    def compile_one(src):
        obj = os.path.join(BUILD_DIR, src.replace(".cu", ".o"))
        cmd = [NVCC, *ARCH, *FLAGS, *extra, "-c", os.path.join(CSRC, src), "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError("nvcc failed for %s:\n%s\n%s" % (src, r.stdout, r.stderr))
        return obj, r.stderr

    with ThreadPoolExecutor(max_workers=len(SOURCES)) as ex:
        results = list(ex.map(compile_one, SOURCES))
    if extra:
        for _, log in results:
            sys.stderr.write(log)
    objs = [o for o, _ in results]
    tmp = LIB + ".tmp.%d" % os.getpid()
    r = subprocess.run([NVCC, *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError("link failed:\n%s\n%s" % (r.stdout, r.stderr))
    os.replace(tmp, LIB)
    return LIB


if __name__ == "__main__":
    print(build(force=True, verbose="-v" in sys.argv))
