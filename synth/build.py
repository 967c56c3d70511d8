"""Build the seeded input generator: a host library (gcc) and a device library
(nvcc, sm_103a).  Harness code for tests and the benchmark."""
import os
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
BUILD_DIR = os.path.join(HERE, "_build")
HOST_LIB = os.path.join(BUILD_DIR, "libzsynth_host.so")
DEV_LIB = os.path.join(BUILD_DIR, "libzsynth_dev.so")
NVCC = os.environ.get("NVCC", "/usr/local/cuda/bin/nvcc")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _stale(out, srcs):
    return not os.path.exists(out) or any(os.path.getmtime(s) > os.path.getmtime(out) for s in srcs)


def build_host(force=False):
    os.makedirs(BUILD_DIR, exist_ok=True)
    src = os.path.join(HERE, "synth_host.c")
    hdr = os.path.join(HERE, "zsynth.h")
    if force or _stale(HOST_LIB, [src, hdr]):
        tmp = HOST_LIB + ".tmp.%d" % os.getpid()
        subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-Wall",
                        "-o", tmp, src], check=True)
        os.replace(tmp, HOST_LIB)
    return HOST_LIB


def build_dev(force=False):
    os.makedirs(BUILD_DIR, exist_ok=True)
    src = os.path.join(HERE, "synth_gpu.cu")
    hdr = os.path.join(HERE, "zsynth.h")
    if force or _stale(DEV_LIB, [src, hdr]):
        tmp = DEV_LIB + ".tmp.%d" % os.getpid()
        subprocess.run([NVCC, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "-shared",
                        "-o", tmp, src], check=True)
        os.replace(tmp, DEV_LIB)
    return DEV_LIB


def build(force=False):
    return build_host(force), build_dev(force)


if __name__ == "__main__":
    print(build(force=True))
