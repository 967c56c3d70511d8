"""Python binding of libzero_gb300 (the ZeRO sharded mixed-precision Adam step
on one GB300).

Argument marshalling only: every step of the computation runs in the CUDA
library.  The functions carry the C names (``zero_plan``, ``zero_step_stage2``
...) and raise :class:`ZeroError` when the library returns a status other
than ZERO_OK.  PyTorch is used by :class:`DeviceBuffers` for device memory
only.

The library must have been built (``zero_sharded_mixed_bucket_gb300.build``
or ``__graft_entry__.build()``); importing this module without it raises
ImportError -- there is no fallback implementation.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = [
    "ZERO_OK", "ZERO_EINVAL", "ZERO_EALIGN", "ZERO_ENOMEM", "ZERO_ECUDA", "ZERO_ETIMEOUT", "ZERO_EUNSUPPORTED",
    "ZERO_FP16", "ZERO_BF16", "ZERO_FP32", "ZERO_ADAM", "ZERO_SGD_MOMENTUM", "ZERO_SGD", "ZeroError", "zero_config_t", "zero_plan_t", "zero_adam_t", "zero_state_t",
    "zero_buffers_t", "zero_step_result_t", "Config", "lib", "lib_path",
    "zero_plan", "zero_plan_bucket", "zero_plan_layer", "zero_model_state_bytes", "zero_comm_bytes",
    "zero_step", "zero_step_stage0", "zero_step_stage1", "zero_step_stage2", "zero_step_stage3",
    "zero_step_stage2_noalloc", "zero_dev_state_init", "zero_step_async", "zero_dev_state_read",
    "DEV_STATE_BYTES", "zero_step_begin_async", "zero_step_bucket_async", "zero_step_end_async",
    "zero_pa_plan_t", "zero_pa_plan", "zero_pa_partition", "zero_pa_gather",
    "zero_step_begin", "zero_step_bucket", "zero_step_end", "zero_gather_layer", "zero_last_error",
    "zero_step_buckets", "zero_step_buckets_async",
    "zero_version", "zero_set_profile_events", "zero_fetch_schedule", "Fetcher", "DeviceBuffers", "ptr_array",
]

ZERO_OK, ZERO_EINVAL, ZERO_EALIGN, ZERO_ENOMEM, ZERO_ECUDA, ZERO_ETIMEOUT, ZERO_EUNSUPPORTED = range(7)
ZERO_FP16, ZERO_BF16, ZERO_FP32 = 0, 1, 2
ZERO_ADAM, ZERO_SGD_MOMENTUM, ZERO_SGD = 0, 1, 2

c_i64, c_i32, c_u32, c_f, c_d, c_vp = (ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_float,
                                       ctypes.c_double, ctypes.c_void_p)


class zero_config_t(ctypes.Structure):
    _fields_ = [("n_params", c_i64), ("bucket_elems", c_i64), ("align_elems", c_i64),
                ("layer_sizes", ctypes.POINTER(c_i64)), ("n_layers", c_i32), ("stage", c_i32),
                ("n_ranks", c_i32), ("dtype", c_i32), ("optimizer", c_i32), ("reserved", c_i32)]


class zero_plan_t(ctypes.Structure):
    _fields_ = [(n, c_i64) for n in ("shard_elems", "padded_elems", "n_buckets", "n_layers", "max_layer_elems",
                                      "state_elems", "param16_elems", "grad16_elems", "reduced_elems",
                                      "workspace_bytes", "hbm_bytes_fused", "hbm_bytes_two_pass",
                                      "comm_counted_bytes")] + \
               [("comm_paper_bytes", c_d), ("mem_total_bytes", c_d), ("reserved", c_d)]


class zero_adam_t(ctypes.Structure):
    _fields_ = [("lr", c_f), ("beta1", c_f), ("beta2", c_f), ("eps", c_f), ("max_grad_norm", c_f),
                ("momentum", c_f)]


class zero_state_t(ctypes.Structure):
    _fields_ = [("t", c_i64), ("loss_scale", c_f), ("min_loss_scale", c_f), ("dynamic", c_i32),
                ("growth_interval", c_i32), ("good_steps", c_i32), ("reserved", c_i32)]


class zero_buffers_t(ctypes.Structure):
    _fields_ = [("grads", ctypes.POINTER(c_vp)), ("params16", ctypes.POINTER(c_vp)),
                ("w", c_vp * 2), ("m", c_vp * 2), ("v", c_vp * 2), ("reduced", c_vp), ("workspace", c_vp),
                ("cur", c_i32), ("reserved", c_i32)]


class zero_step_result_t(ctypes.Structure):
    _fields_ = [("t", c_i64), ("hbm_bytes", c_i64), ("comm_counted_bytes", c_i64), ("grad_norm", c_d),
                ("overflow", c_u32), ("skipped", c_i32), ("clip_coef", c_f), ("loss_scale_used", c_f),
                ("new_loss_scale", c_f), ("kernel_launches", c_i32), ("path", c_i32), ("reserved", c_i32)]


class zero_pa_plan_t(ctypes.Structure):
    _fields_ = [("act_elems", c_i64), ("shard_elems", c_i64), ("align_elems", c_i64), ("n_mp", c_i32),
                ("dtype", c_i32), ("mem_per_rank_bytes", c_i64), ("mem_per_rank_pa_bytes", c_i64),
                ("gather_bytes", c_i64), ("reserved", c_i64 * 2)]


class ZeroError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__("zero status %d: %s" % (status, message))
        self.status = status


_lib = None


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded CUDA library (ctypes).  Raises ImportError if it was not built."""
    global _lib
    if _lib is None:
        if not os.path.exists(_build.LIB):
            raise ImportError("libzero_gb300.so is not built; run zero_sharded_mixed_bucket_gb300.build.build() "
                              "(or __graft_entry__.build()) first")
        L = ctypes.CDLL(_build.LIB)
        P = ctypes.POINTER
        cfg, plan, bufs = P(zero_config_t), P(zero_plan_t), P(zero_buffers_t)
        adam, state, res = P(zero_adam_t), P(zero_state_t), P(zero_step_result_t)
        sigs = {
            "zero_plan": [cfg, plan],
            "zero_plan_bucket": [cfg, c_i64, P(c_i64), P(c_i32)],
            "zero_plan_layer": [cfg, c_i32, P(c_i64), P(c_i64)],
            "zero_model_state_bytes": [c_i64, c_i32, c_i32, c_i32, c_i32, P(c_d)],
            "zero_comm_bytes": [c_i64, c_i32, c_i32, c_i32, P(c_d), P(c_i64)],
            "zero_step": [cfg, plan, bufs, adam, state, c_vp, res],
            "zero_step_stage0": [cfg, plan, bufs, adam, state, c_vp, res],
            "zero_step_stage1": [cfg, plan, bufs, adam, state, c_vp, res],
            "zero_step_stage2": [cfg, plan, bufs, adam, state, c_vp, res],
            "zero_step_stage3": [cfg, plan, bufs, adam, state, c_vp, res],
            "zero_step_stage2_noalloc": [cfg, plan, bufs, adam, state, c_vp, res],
            "zero_dev_state_init": [c_vp, adam, state, c_vp],
            "zero_step_async": [cfg, plan, bufs, adam, c_vp, c_vp, P(c_i32)],
            "zero_dev_state_read": [c_vp, state, res, c_vp],
            "zero_step_begin_async": [cfg, plan, bufs, adam, c_vp, c_vp],
            "zero_step_bucket_async": [cfg, plan, bufs, adam, c_i64, P(c_vp), c_vp],
            "zero_step_end_async": [cfg, plan, bufs, adam, c_vp, c_vp, P(c_i32)],
            "zero_step_buckets": [cfg, plan, bufs, adam, state, P(c_i64), c_i32, P(c_vp), c_vp],
            "zero_step_buckets_async": [cfg, plan, bufs, adam, P(c_i64), c_i32, P(c_vp), c_vp],
            "zero_pa_plan": [c_i64, c_i32, c_i32, c_i64, P(zero_pa_plan_t)],
            "zero_pa_partition": [P(zero_pa_plan_t), P(c_vp), P(c_vp), c_vp],
            "zero_pa_gather": [P(zero_pa_plan_t), P(c_vp), P(c_vp), c_i32, c_vp],
            "zero_step_begin": [cfg, plan, bufs, adam, state, c_vp],
            "zero_step_bucket": [cfg, plan, bufs, adam, state, c_i64, P(c_vp), c_vp],
            "zero_step_end": [cfg, plan, bufs, adam, state, c_vp, res],
            "zero_gather_layer": [cfg, plan, c_i32, P(c_vp), P(c_vp), c_i32, c_vp],
            "zero_fetcher_init": [c_vp, cfg, plan, P(c_vp), P(c_vp), c_i32, c_i64, P(c_i32), c_i32, c_i32, c_vp,
                                  P(c_vp), c_i32],
            "zero_fetch_layer": [c_vp, c_i32, c_vp, P(c_i64)],
            "zero_release_layer": [c_vp, c_i32, c_vp],
            "zero_fetcher_stats": [c_vp, P(c_i64), P(c_i32)],
            "zero_fetch_schedule": [P(c_i64), c_i32, P(c_i32), c_i32, c_i64, c_i32, P(c_i32), P(c_i64), P(c_i64)],
        }
        for name, args in sigs.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        L.zero_set_profile_events.argtypes = [c_vp, c_vp]
        L.zero_set_profile_events.restype = ctypes.c_int
        L.zero_last_error.restype = ctypes.c_char_p
        L.zero_last_error.argtypes = []
        L.zero_version.restype = c_i32
        L.zero_version.argtypes = []
        _lib = L
    return _lib


def _check(status: int):
    if status != ZERO_OK:
        raise ZeroError(status, zero_last_error())


def zero_set_profile_events(start_event=None, end_event=None):
    """Record two CUDA events around the kernels of every later step call on
    this thread (torch.cuda.Event objects or raw cudaEvent_t ints; None, None
    to stop)."""
    def raw(e):
        if e is None:
            return None
        return int(e) if isinstance(e, int) else int(e.cuda_event)
    _check(lib().zero_set_profile_events(raw(start_event), raw(end_event)))


def zero_last_error() -> str:
    return lib().zero_last_error().decode()


def zero_version() -> int:
    return int(lib().zero_version())


class Config:
    """A zero_config_t that keeps its layer-size array alive."""

    def __init__(self, n_params: int, n_ranks: int, stage: int, bucket_elems: int, align_elems: int = 0,
                 layer_sizes=None, dtype: int = ZERO_FP16, optimizer: int = ZERO_ADAM):
        self._layers = None
        self.c = zero_config_t(n_params=n_params, bucket_elems=bucket_elems, align_elems=align_elems,
                               n_layers=0, stage=stage, n_ranks=n_ranks, dtype=dtype, optimizer=optimizer)
        if layer_sizes is not None:
            self._layers = (c_i64 * len(layer_sizes))(*[int(x) for x in layer_sizes])
            self.c.layer_sizes = ctypes.cast(self._layers, ctypes.POINTER(c_i64))
            self.c.n_layers = len(layer_sizes)

    def __getattr__(self, name):
        return getattr(self.c, name)


def _cfg(cfg):
    return ctypes.byref(cfg.c if isinstance(cfg, Config) else cfg)


def zero_plan(cfg) -> zero_plan_t:
    p = zero_plan_t()
    _check(lib().zero_plan(_cfg(cfg), ctypes.byref(p)))
    return p


def zero_plan_bucket(cfg, bucket: int) -> list[tuple[int, int, int]]:
    n = (cfg.c if isinstance(cfg, Config) else cfg).n_ranks
    seg = (c_i64 * (3 * n))()
    cnt = c_i32()
    _check(lib().zero_plan_bucket(_cfg(cfg), bucket, seg, ctypes.byref(cnt)))
    return [(seg[3 * k], seg[3 * k + 1], seg[3 * k + 2]) for k in range(cnt.value)]


def zero_plan_layer(cfg, layer: int) -> tuple[int, int]:
    s, n = c_i64(), c_i64()
    _check(lib().zero_plan_layer(_cfg(cfg), layer, ctypes.byref(s), ctypes.byref(n)))
    return s.value, n.value


def zero_model_state_bytes(n_params: int, n_ranks: int, stage: int, param_bytes: int = 2, optim_K: int = 12):
    out = (c_d * 4)()
    _check(lib().zero_model_state_bytes(n_params, n_ranks, stage, param_bytes, optim_K, out))
    return tuple(out)


def zero_comm_bytes(n_params: int, n_ranks: int, stage: int, param_bytes: int = 2):
    paper, counted = c_d(), c_i64()
    _check(lib().zero_comm_bytes(n_params, n_ranks, stage, param_bytes, ctypes.byref(paper), ctypes.byref(counted)))
    return paper.value, counted.value


def _stream(stream) -> int:
    if stream is None:
        return 0
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)   # torch.cuda.Stream


def _step(fn, cfg, plan, bufs, adam, state, stream):
    res = zero_step_result_t()
    b = bufs.b if isinstance(bufs, DeviceBuffers) else bufs
    _check(fn(_cfg(cfg), ctypes.byref(plan), ctypes.byref(b), ctypes.byref(adam), ctypes.byref(state),
              _stream(stream), ctypes.byref(res)))
    return res


def zero_step(cfg, plan, bufs, adam, state, stream=None) -> zero_step_result_t:
    return _step(lib().zero_step, cfg, plan, bufs, adam, state, stream)


def zero_step_stage0(cfg, plan, bufs, adam, state, stream=None) -> zero_step_result_t:
    return _step(lib().zero_step_stage0, cfg, plan, bufs, adam, state, stream)


def zero_step_stage1(cfg, plan, bufs, adam, state, stream=None) -> zero_step_result_t:
    return _step(lib().zero_step_stage1, cfg, plan, bufs, adam, state, stream)


def zero_step_stage2(cfg, plan, bufs, adam, state, stream=None) -> zero_step_result_t:
    return _step(lib().zero_step_stage2, cfg, plan, bufs, adam, state, stream)


def zero_step_stage3(cfg, plan, bufs, adam, state, stream=None) -> zero_step_result_t:
    return _step(lib().zero_step_stage3, cfg, plan, bufs, adam, state, stream)


def zero_step_stage2_noalloc(cfg, plan, bufs, adam, state, stream=None) -> zero_step_result_t:
    """Stage-2 step whose scratch comes from a static array in the library
    (for callers that cannot allocate device memory); see the header."""
    return _step(lib().zero_step_stage2_noalloc, cfg, plan, bufs, adam, state, stream)


DEV_STATE_BYTES = 64


def _dptr(x) -> int:
    return x if isinstance(x, int) else int(x.data_ptr())


def zero_dev_state_init(dev_state, adam, state, stream=None):
    """Upload `state` into a 64-byte device block (a pointer or a tensor)."""
    _check(lib().zero_dev_state_init(_dptr(dev_state), ctypes.byref(adam), ctypes.byref(state), _stream(stream)))


def zero_step_async(cfg, plan, bufs, adam, dev_state, stream=None) -> int:
    """Enqueue one step whose step state lives in `dev_state`; no host
    synchronisation.  Returns the number of kernels launched."""
    b = bufs.b if isinstance(bufs, DeviceBuffers) else bufs
    n = c_i32(0)
    _check(lib().zero_step_async(_cfg(cfg), ctypes.byref(plan), ctypes.byref(b), ctypes.byref(adam),
                                 _dptr(dev_state), _stream(stream), ctypes.byref(n)))
    return n.value


def zero_step_begin_async(cfg, plan, bufs, adam, dev_state, stream=None):
    b = bufs.b if isinstance(bufs, DeviceBuffers) else bufs
    _check(lib().zero_step_begin_async(_cfg(cfg), ctypes.byref(plan), ctypes.byref(b), ctypes.byref(adam),
                                       _dptr(dev_state), _stream(stream)))


def zero_step_bucket_async(cfg, plan, bufs, adam, bucket: int, bucket_grads=None, stream=None):
    b = bufs.b if isinstance(bufs, DeviceBuffers) else bufs
    _check(lib().zero_step_bucket_async(_cfg(cfg), ctypes.byref(plan), ctypes.byref(b), ctypes.byref(adam), bucket,
                                        _ptr_array(bucket_grads), _stream(stream)))


def zero_step_end_async(cfg, plan, bufs, adam, dev_state, stream=None) -> int:
    b = bufs.b if isinstance(bufs, DeviceBuffers) else bufs
    n = c_i32(0)
    _check(lib().zero_step_end_async(_cfg(cfg), ctypes.byref(plan), ctypes.byref(b), ctypes.byref(adam),
                                     _dptr(dev_state), _stream(stream), ctypes.byref(n)))
    return n.value


def zero_dev_state_read(dev_state, stream=None):
    """(zero_state_t, zero_step_result_t of the last step) from the device block."""
    st, res = zero_state_t(), zero_step_result_t()
    _check(lib().zero_dev_state_read(_dptr(dev_state), ctypes.byref(st), ctypes.byref(res), _stream(stream)))
    return st, res


def zero_pa_plan(act_elems: int, n_mp: int, dtype: int = ZERO_FP16, align_elems: int = 0) -> zero_pa_plan_t:
    """Partition of one activation checkpoint across N_m model-parallel ranks (P_a)."""
    p = zero_pa_plan_t()
    _check(lib().zero_pa_plan(act_elems, n_mp, dtype, align_elems, ctypes.byref(p)))
    return p


def zero_pa_partition(plan: zero_pa_plan_t, replicas, shards, stream=None):
    """Rank r keeps its slice of replicas[r] in shards[r] (pointers or tensors)."""
    _check(lib().zero_pa_partition(ctypes.byref(plan), _ptr_array([_dptr(x) for x in replicas]),
                                   _ptr_array([_dptr(x) for x in shards]), _stream(stream)))


def zero_pa_gather(plan: zero_pa_plan_t, shards, dst, stream=None):
    """All-gather: the checkpoint rebuilt from the slices into every dst."""
    _check(lib().zero_pa_gather(ctypes.byref(plan), _ptr_array([_dptr(x) for x in shards]),
                                _ptr_array([_dptr(x) for x in dst]), len(dst), _stream(stream)))


def zero_step_begin(cfg, plan, bufs, adam, state, stream=None):
    b = bufs.b if isinstance(bufs, DeviceBuffers) else bufs
    _check(lib().zero_step_begin(_cfg(cfg), ctypes.byref(plan), ctypes.byref(b), ctypes.byref(adam),
                                 ctypes.byref(state), _stream(stream)))


def _ptr_array(ptrs):
    """A host array of pointers: None, a ctypes array of c_void_p (passed as
    it is, so callers can build one once and reuse it), or a sequence of ints."""
    if ptrs is None:
        return None
    if isinstance(ptrs, ctypes.Array) and ptrs._type_ is c_vp:
        return ptrs
    return (c_vp * len(ptrs))(*[int(p) for p in ptrs])


def ptr_array(ptrs):
    """A reusable host array of device pointers for the calls that take one."""
    return (c_vp * len(ptrs))(*[int(p) for p in ptrs])


def zero_step_bucket(cfg, plan, bufs, adam, state, bucket: int, bucket_grads=None, stream=None):
    """bucket_grads: None, or N device pointers (ints) to this bucket's gradient windows."""
    b = bufs.b if isinstance(bufs, DeviceBuffers) else bufs
    _check(lib().zero_step_bucket(_cfg(cfg), ctypes.byref(plan), ctypes.byref(b), ctypes.byref(adam),
                                  ctypes.byref(state), bucket, _ptr_array(bucket_grads), _stream(stream)))


def _bucket_run(buckets, bucket_grads):
    """(int64 array of indices, count, flat pointer array or None) of a run of buckets;
    bucket_grads: None, a prebuilt ctypes pointer array (count*N), or one pointer list per bucket."""
    idx = buckets if isinstance(buckets, ctypes.Array) else (c_i64 * len(buckets))(*[int(x) for x in buckets])
    if bucket_grads is None or isinstance(bucket_grads, ctypes.Array):
        g = bucket_grads
    else:
        g = _ptr_array([int(p) for ptrs in bucket_grads for p in ptrs])
    return idx, len(idx), g


def zero_step_buckets(cfg, plan, bufs, adam, state, buckets, bucket_grads=None, stream=None):
    """Several buckets of one step in one call, consecutive kernels overlapping their edges."""
    b = bufs.b if isinstance(bufs, DeviceBuffers) else bufs
    idx, n, g = _bucket_run(buckets, bucket_grads)
    _check(lib().zero_step_buckets(_cfg(cfg), ctypes.byref(plan), ctypes.byref(b), ctypes.byref(adam),
                                   ctypes.byref(state), idx, n, g, _stream(stream)))


def zero_step_buckets_async(cfg, plan, bufs, adam, buckets, bucket_grads=None, stream=None):
    """zero_step_buckets between zero_step_begin_async and zero_step_end_async."""
    b = bufs.b if isinstance(bufs, DeviceBuffers) else bufs
    idx, n, g = _bucket_run(buckets, bucket_grads)
    _check(lib().zero_step_buckets_async(_cfg(cfg), ctypes.byref(plan), ctypes.byref(b), ctypes.byref(adam), idx,
                                         n, g, _stream(stream)))


def zero_step_end(cfg, plan, bufs, adam, state, stream=None) -> zero_step_result_t:
    return _step(lib().zero_step_end, cfg, plan, bufs, adam, state, stream)


def zero_gather_layer(cfg, plan, layer: int, param_shards, dst, stream=None):
    """param_shards: N device pointers; dst: n_dst device pointers."""
    _check(lib().zero_gather_layer(_cfg(cfg), ctypes.byref(plan), layer, _ptr_array(param_shards),
                                   _ptr_array(dst), len(dst), _stream(stream)))


def zero_fetch_schedule(layer_sizes, order, capacity: int, depth: int):
    """The fetcher's decisions without a GPU: (issue_at, offsets, max_live)."""
    n, L = len(order), len(layer_sizes)
    sizes = (c_i64 * L)(*[int(x) for x in layer_sizes])
    ordr = (c_i32 * n)(*[int(x) for x in order])
    issue = (c_i32 * n)()
    offs = (c_i64 * n)()
    ml = c_i64()
    _check(lib().zero_fetch_schedule(sizes, L, ordr, n, capacity, depth, issue, offs, ctypes.byref(ml)))
    return list(issue), list(offs), ml.value


class Fetcher:
    """Stage-3 layer fetches ahead of use under a live-parameter budget (see
    the header).  pool: n_dst device buffers (int16 tensors) of `capacity`
    elements; order: layer sequence of one pass; events are created here
    with torch (the library allocates nothing)."""

    FETCHER_BYTES = 8192

    def __init__(self, cfg, plan, param_shards, pool, capacity: int, order, depth: int, side_stream):
        import torch
        self._state = (ctypes.c_byte * self.FETCHER_BYTES)()
        self._order = (c_i32 * len(order))(*[int(x) for x in order])
        self._shards = _ptr_array([int(p) for p in param_shards])
        self._pool = _ptr_array([t.data_ptr() for t in pool])
        self.pool = pool
        self.events = [torch.cuda.Event() for _ in range(2 * (depth + 1))]
        side = torch.cuda.current_stream() if side_stream is None else side_stream
        for e in self.events:          # materialise the events (the library records them by handle)
            e.record(side)
        self._events = _ptr_array([int(e.cuda_event) for e in self.events])
        self.side = side
        _check(lib().zero_fetcher_init(ctypes.addressof(self._state), _cfg(cfg), ctypes.byref(plan), self._shards,
                                       self._pool, len(pool), capacity, self._order, len(order), depth,
                                       _stream(side), self._events, len(self.events)))

    def fetch(self, pos: int, stream=None) -> int:
        off = c_i64()
        _check(lib().zero_fetch_layer(ctypes.addressof(self._state), pos, _stream(stream), ctypes.byref(off)))
        return off.value

    def release(self, pos: int, stream=None):
        _check(lib().zero_release_layer(ctypes.addressof(self._state), pos, _stream(stream)))

    def stats(self):
        ml, g = c_i64(), c_i32()
        _check(lib().zero_fetcher_stats(ctypes.addressof(self._state), ctypes.byref(ml), ctypes.byref(g)))
        return ml.value, g.value


class DeviceBuffers:
    """Device memory for one job, allocated with PyTorch to the plan's sizes.

    grads[r], params16[r]: int16 tensors (16-bit bit patterns; int32 tensors
    of binary32 patterns for ZERO_FP32); w/m/v[k]: float32 tensors (k = 0
    current, 1 shadow when shadow=True); reduced (stages 2-3, same element
    type as the gradients); workspace.  ``b`` is the zero_buffers_t that
    points at them.
    """

    def __init__(self, cfg, plan: zero_plan_t, device="cuda", shadow: bool = True, reduced: bool = True,
                 grads: bool = True):
        import torch
        c = cfg.c if isinstance(cfg, Config) else cfg
        N = c.n_ranks
        z = lambda n, dt: torch.zeros(max(int(n), 1), dtype=dt, device=device)
        vt = torch.int32 if c.dtype == ZERO_FP32 else torch.int16
        self.value_dtype = vt
        self.grads = [z(plan.grad16_elems, vt) for _ in range(N)] if grads else []
        self.params16 = [z(plan.param16_elems, vt) for _ in range(N)]
        ncopy = 2 if shadow else 1
        self.w = [z(plan.state_elems, torch.float32) for _ in range(ncopy)]
        self.m = [z(plan.state_elems, torch.float32) for _ in range(ncopy)]
        self.v = [z(plan.state_elems, torch.float32) for _ in range(ncopy)]
        self.reduced = z(plan.reduced_elems, vt) if (reduced and plan.reduced_elems) else None
        self.workspace = torch.zeros(plan.workspace_bytes, dtype=torch.uint8, device=device)
        self._gp = (c_vp * N)(*[t.data_ptr() for t in self.grads]) if grads else None
        self._pp = (c_vp * N)(*[t.data_ptr() for t in self.params16])
        self.b = zero_buffers_t()
        if self._gp is not None:
            self.b.grads = ctypes.cast(self._gp, ctypes.POINTER(c_vp))
        self.b.params16 = ctypes.cast(self._pp, ctypes.POINTER(c_vp))
        for k in range(ncopy):
            self.b.w[k] = self.w[k].data_ptr()
            self.b.m[k] = self.m[k].data_ptr()
            self.b.v[k] = self.v[k].data_ptr()
        self.b.reduced = self.reduced.data_ptr() if self.reduced is not None else None
        self.b.workspace = self.workspace.data_ptr()
        self.b.cur = 0

    @property
    def cur(self) -> int:
        return self.b.cur

    def state(self):
        """(w, m, v) tensors of the current state copy."""
        k = self.b.cur
        return self.w[k], self.m[k], self.v[k]
