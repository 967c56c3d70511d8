"""Seeded synthetic inputs for the ZeRO step: gradients, master weights.

Harness code shared by the tests and the benchmark.  It holds none of the
optimizer's arithmetic: it only draws numbers.  The generator is defined in
zsynth.h (Philox4x32-10 counters, an Irwin-Hall(4) normal, one fp32 rounding,
round-to-nearest-even into 16 bits); the host library and the device library
implement it separately and agree bit for bit (tested on the GPU).

Streams: GRAD gradients (per rank and step), WEIGHT initial master weights.
"""
import ctypes
import math

import numpy as np

from . import build as _build

FP16, BF16, FP32 = 0, 1, 2
STREAM_GRAD = 1
STREAM_WEIGHT = 2
STREAM_INJECT = 3

_host = None
_dev = None


def k_for(sigma: float) -> float:
    """fp32 factor that gives the Irwin-Hall(4) sum standard deviation sigma."""
    return float(np.float32(sigma / (65536.0 * math.sqrt(4.0 / 3.0))))


def host():
    global _host
    if _host is None:
        L = ctypes.CDLL(_build.build_host())
        vp, i64, i32, u32, u64, f = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                                     ctypes.c_uint64, ctypes.c_float)
        L.zsynth_host_normal16.argtypes = [vp, i64, i32, u64, u32, u32, u32, i64, f]
        L.zsynth_host_normal32.argtypes = [vp, i64, u64, u32, u32, u32, i64, f]
        L.zsynth_host_normal16_at.argtypes = [vp, i64, vp, i32, u64, u32, u32, u32, f]
        L.zsynth_host_normal32_at.argtypes = [vp, i64, vp, u64, u32, u32, u32, f]
        L.zsynth_host_philox4x32_10.argtypes = [vp, vp, vp]
        _host = L
    return _host


def dev():
    global _dev
    if _dev is None:
        L = ctypes.CDLL(_build.build_dev())
        vp, i64, i32, u32, u64, f = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                                     ctypes.c_uint64, ctypes.c_float)
        L.zsynth_dev_normal16.argtypes = [vp, i64, i32, u64, u32, u32, u32, i64, f, vp]
        L.zsynth_dev_normal16.restype = ctypes.c_int
        L.zsynth_dev_normal32.argtypes = [vp, i64, u64, u32, u32, u32, i64, f, vp]
        L.zsynth_dev_normal32.restype = ctypes.c_int
        _dev = L
    return _dev


def philox(ctr, key):
    c = (ctypes.c_uint32 * 4)(*ctr)
    k = (ctypes.c_uint32 * 2)(*key)
    o = (ctypes.c_uint32 * 4)()
    host().zsynth_host_philox4x32_10(c, k, o)
    return list(o)


def host_normal16(n, dtype, sigma, *, seed, stream, step=0, rank=0, offset=0):
    out = np.empty(n, np.uint16)
    host().zsynth_host_normal16(out.ctypes.data, n, dtype, seed, stream, step, rank, offset, k_for(sigma))
    return out


def host_normal32(n, sigma, *, seed, stream, step=0, rank=0, offset=0):
    out = np.empty(n, np.float32)
    host().zsynth_host_normal32(out.ctypes.data, n, seed, stream, step, rank, offset, k_for(sigma))
    return out


def host_normal16_at(idx, dtype, sigma, *, seed, stream, step=0, rank=0):
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.uint16)
    host().zsynth_host_normal16_at(out.ctypes.data, idx.size, idx.ctypes.data, dtype, seed, stream, step,
                                   rank, k_for(sigma))
    return out


def host_normal32_at(idx, sigma, *, seed, stream, step=0, rank=0):
    idx = np.ascontiguousarray(idx, np.int64)
    out = np.empty(idx.size, np.float32)
    host().zsynth_host_normal32_at(out.ctypes.data, idx.size, idx.ctypes.data, seed, stream, step, rank,
                                   k_for(sigma))
    return out


def dev_normal16(ptr, n, dtype, sigma, *, seed, stream, step=0, rank=0, offset=0, cuda_stream=0):
    rc = dev().zsynth_dev_normal16(ptr, n, dtype, seed, stream, step, rank, offset, k_for(sigma), cuda_stream)
    if rc:
        raise RuntimeError("zsynth_dev_normal16 failed with CUDA error %d" % rc)


def dev_normal32(ptr, n, sigma, *, seed, stream, step=0, rank=0, offset=0, cuda_stream=0):
    rc = dev().zsynth_dev_normal32(ptr, n, seed, stream, step, rank, offset, k_for(sigma), cuda_stream)
    if rc:
        raise RuntimeError("zsynth_dev_normal32 failed with CUDA error %d" % rc)


def inf_positions(n_params, n_ranks, *, seed, step, period=10 ** 9):
    """(rank, element) pairs where a gradient element is set to +inf: flat
    positions k*period + off over the rank-major index space [rank][element],
    off drawn from (seed, step).  'One inf per 1e9 elements.'"""
    o = philox([step, 0, 0xFFFFFFFF, 0], [seed & 0xFFFFFFFF, STREAM_INJECT])
    off = ((o[1] << 32) | o[0]) % period
    total = n_params * n_ranks
    return [(f // n_params, f % n_params) for f in range(off, total, period)]


def inf_bits(dtype):
    return {FP16: 0x7C00, BF16: 0x7F80, FP32: 0x7F800000}[dtype]


# Gradients of any model precision, as bit patterns (uint16, or uint32 for
# FP32, whose values are the fp32 draws themselves).
def host_grad(n, dtype, sigma, *, seed, stream, step=0, rank=0, offset=0):
    if dtype == FP32:
        return host_normal32(n, sigma, seed=seed, stream=stream, step=step, rank=rank, offset=offset).view(np.uint32)
    return host_normal16(n, dtype, sigma, seed=seed, stream=stream, step=step, rank=rank, offset=offset)


def host_grad_at(idx, dtype, sigma, *, seed, stream, step=0, rank=0):
    if dtype == FP32:
        return host_normal32_at(idx, sigma, seed=seed, stream=stream, step=step, rank=rank).view(np.uint32)
    return host_normal16_at(idx, dtype, sigma, seed=seed, stream=stream, step=step, rank=rank)


def dev_grad(ptr, n, dtype, sigma, *, seed, stream, step=0, rank=0, offset=0, cuda_stream=0):
    if dtype == FP32:
        dev_normal32(ptr, n, sigma, seed=seed, stream=stream, step=step, rank=rank, offset=offset,
                     cuda_stream=cuda_stream)
    else:
        dev_normal16(ptr, n, dtype, sigma, seed=seed, stream=stream, step=step, rank=rank, offset=offset,
                     cuda_stream=cuda_stream)
