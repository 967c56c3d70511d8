"""CPU oracle for the ZeRO sharded mixed-precision Adam step.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this package.  The
GPU library (``zero_sharded_mixed_bucket_gb300``) never imports it and shares
no code with it; the two meet only in the seeded input generator (``synth``),
which holds none of the step's arithmetic.

Sources (page titles as published):

* [P1] "AI论文陪读·ZeRO：分布式训练的第一篇论文（中英双语）" (reading notes)
* [P2] "ZeRO：大模型训练的内存优化革命" (summary)
* [P3] ZeRO visual reading (blog.vllbc.top, zero-deepspeed) -- memory
  accounting, worked examples A/B/C, communication accounting, Table 1 and
  Table 2 as transcribed there
* [P4] "SC-2020 ZeRO：Memory Optimizations Toward Training Trillion Parameter
  Models" (paper notes)

What is here
------------
``plan`` / ``bucket_segments`` / ``owner``
    ZeRO-DP partitioning: rank r owns the r-th contiguous 1/N_d slice of the
    flat parameter vector ([P3] stage list; [P2] 3.1.1-3.1.3), padded to an
    alignment, and the constant-size fusion buckets ([P2] 3.2.2 C_B; [P4]
    "Deep Dive into ZeRO-R / C_B").
``model_state_bytes`` / ``comm_bytes`` / ``display_gb`` / ``max_model_size``
    The memory and communication accounting of [P3] (stage formulas, worked
    examples, display rule, Table 1, Table 2) and [P1] section 04.
``step``
    The unpartitioned mixed-precision Adam step (see zero_oracle.c for the
    elementwise part); with dtype FP32 the fp32-training variant of the
    pages' fp32 SGD examples (binary32 parameters and gradients).  The exact gradient norm for clipping uses
    ``math.fsum`` (a correctly rounded sum) of the squares, which are exact
    in fp64 for 16-bit inputs.

Parity pins live in tests/test_oracle_*.py.  Every function here is pinned
there against printed page values, closed forms, library routines or brute
force, except where its docstring says "parity unpinned".
"""
from __future__ import annotations

import ctypes
import math
from fractions import Fraction

import numpy as np

from . import build as _build

FP16 = 0
BF16 = 1
FP32 = 2        # fp32 training: parameters and gradients in binary32 (b = 4)

_lib = None


class Hyper(ctypes.Structure):
    _fields_ = [
        ("inv_scale", ctypes.c_float),
        ("use_clip", ctypes.c_int32),
        ("clip", ctypes.c_float),
        ("lr", ctypes.c_float),
        ("beta1", ctypes.c_float),
        ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("one_minus_beta1", ctypes.c_float),
        ("one_minus_beta2", ctypes.c_float),
        ("bc1", ctypes.c_float),
        ("bc2", ctypes.c_float),
    ]


def lib():
    """Load (building if needed) the oracle's C library."""
    global _lib
    if _lib is None:
        L = ctypes.CDLL(_build.build())
        vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32
        L.oracle_f16_to_f32.restype = ctypes.c_float
        L.oracle_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_bf16_to_f32.restype = ctypes.c_float
        L.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.oracle_f32_to_f16.restype = ctypes.c_uint16
        L.oracle_f32_to_f16.argtypes = [ctypes.c_float]
        L.oracle_f32_to_bf16.restype = ctypes.c_uint16
        L.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
        L.oracle_to_f32_array.argtypes = [i64, vp, i32, vp]
        L.oracle_from_f32_array.argtypes = [i64, vp, i32, vp]
        L.oracle_reduce.restype = ctypes.c_uint32
        L.oracle_reduce.argtypes = [i32, i64, vp, i32, vp]
        L.oracle_sumsq_bins.argtypes = [i64, vp, i32, vp]
        L.oracle_adam.argtypes = [i64, vp, i32, ctypes.POINTER(Hyper), vp, vp, vp, vp]
        L.oracle_cast.argtypes = [i64, vp, i32, vp]
        L.oracle_sgd.argtypes = [i64, vp, i32, ctypes.POINTER(Hyper), vp, vp, vp]
        _lib = L
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("16-bit values are passed as uint16 bit patterns")
    return a


def bits_dtype(dtype: int):
    """numpy type of the bit patterns of model-precision values."""
    return np.uint32 if dtype == FP32 else np.uint16


def _bits(a, dtype: int) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != bits_dtype(dtype):
        raise TypeError("values are passed as %s bit patterns" % np.dtype(bits_dtype(dtype)).name)
    return a


def _f32arr(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.float32:
        raise TypeError("expected float32")
    return a


def f32(x: float) -> float:
    """Round a Python float (fp64) to the nearest fp32 value."""
    return float(np.float32(x))


# ---------------------------------------------------------------------------
# 16-bit formats
# ---------------------------------------------------------------------------
def to_f32(bits, dtype: int) -> np.ndarray:
    bits = _bits(bits, dtype)
    out = np.empty(bits.shape, np.float32)
    lib().oracle_to_f32_array(bits.size, _ptr(bits), dtype, _ptr(out))
    return out


def from_f32(x, dtype: int) -> np.ndarray:
    x = _f32arr(x)
    out = np.empty(x.shape, bits_dtype(dtype))
    lib().oracle_from_f32_array(x.size, _ptr(x), dtype, _ptr(out))
    return out


def is_nonfinite16(bits, dtype: int) -> np.ndarray:
    return ~np.isfinite(to_f32(bits, dtype))


# ---------------------------------------------------------------------------
# Scalars of the step
# ---------------------------------------------------------------------------
def inv_scale(loss_scale: float, n_ranks: int) -> float:
    """1/(S*N_d) rounded once to fp32: removes the loss scale S and turns the
    rank sum into the data-parallel mean.  Exact whenever S*N_d is a power of
    two."""
    return f32(1.0 / (f32(loss_scale) * n_ranks))


def bias_corrections(beta1: float, beta2: float, t: int) -> tuple[float, float]:
    """(1 - beta1^t, 1 - beta2^t) of Adam step t (Kingma & Ba, Algorithm 1).

    beta^t is formed in fp64 by t repeated multiplications of the fp32 value
    of beta, then 1 - beta^t is rounded once to fp32."""
    if t < 1:
        raise ValueError("Adam steps count from t = 1")
    b1, b2 = f32(beta1), f32(beta2)
    p1 = p2 = 1.0
    for _ in range(t):
        p1 *= b1
        p2 *= b2
    return f32(1.0 - p1), f32(1.0 - p2)


def exact_sumsq(h, dtype: int) -> float:
    """sum_i h_i^2 over the finite elements, correctly rounded to fp64.

    Each square of a 16-bit or binary32 value is exact in fp64 (at most 48
    significant bits, exponents well inside fp64's range); math.fsum returns
    the correctly rounded value of their exact sum."""
    x = to_f32(h, dtype).astype(np.float64)
    x = x[np.isfinite(x)]
    return math.fsum((x * x).tolist())


def sumsq_fraction(h, dtype: int) -> Fraction:
    """The exact sum of squares as a rational, from the C oracle's exponent
    bins (used to pin exact_sumsq and the GPU's integer accumulator); for
    binary32 values, the sum of the exact rational squares."""
    if dtype == FP32:
        x = to_f32(h, dtype)
        return sum((Fraction(float(v)) ** 2 for v in x[np.isfinite(x)]), Fraction(0))
    h = _u16(h)
    bins = np.zeros(256, np.uint64)
    lib().oracle_sumsq_bins(h.size, _ptr(h), dtype, _ptr(bins))
    total = Fraction(0)
    for k in range(256):
        if bins[k] == 0:
            continue
        if dtype == BF16:
            E = (max(k, 1) - 134)     # value = M * 2^(e - 127 - 7)
        else:
            E = (max(k, 1) - 25)      # value = M * 2^(e - 15 - 10)
        total += Fraction(int(bins[k])) * (Fraction(2) ** (2 * E))
    return total


def grad_norm(sumsq: float, inv: float) -> float:
    """||g||_2 of the unscaled mean gradient g = h * inv: sqrt in fp64 of the
    correctly rounded sum of squares, times inv."""
    return math.sqrt(sumsq) * inv


def clip_coef(norm: float, max_norm: float) -> float:
    """min(1, max_norm/(norm + 1e-6)) in fp64, rounded once to fp32."""
    return f32(min(1.0, f32(max_norm) / (norm + 1e-6)))


# ---------------------------------------------------------------------------
# Loss scaler (dynamic: halve and skip on overflow)
# ---------------------------------------------------------------------------
def scaler_update(scale: float, good_steps: int, overflow: bool, dynamic: bool,
                  min_scale: float = 1.0, growth_interval: int = 0) -> tuple[float, int]:
    """Next (loss scale, consecutive clean steps).

    On overflow the step is skipped; a dynamic scaler halves S (not below
    min_scale).  After growth_interval consecutive clean steps (0: never) a
    dynamic scaler doubles S.  A static scaler never changes S."""
    if overflow:
        if dynamic:
            scale = max(f32(scale * 0.5), f32(min_scale))
        return scale, 0
    good_steps += 1
    if dynamic and growth_interval > 0 and good_steps >= growth_interval:
        return f32(scale * 2.0), 0
    return scale, good_steps


# ---------------------------------------------------------------------------
# Elementwise parts (C)
# ---------------------------------------------------------------------------
def reduce(grads, dtype: int) -> tuple[np.ndarray, int]:
    """Rank-order fp32 sum of the N_d ranks' 16-bit gradients, rounded once to
    the 16-bit type (FP32: the fp32 sum itself), and the overflow flag (any
    inf/NaN)."""
    grads = [_bits(g, dtype) for g in grads]
    n = grads[0].size
    if any(g.size != n for g in grads):
        raise ValueError("all ranks hold the same number of gradient elements")
    ptrs = (ctypes.c_void_p * len(grads))(*[_ptr(g) for g in grads])
    h = np.empty(n, bits_dtype(dtype))
    flag = lib().oracle_reduce(len(grads), n, ptrs, dtype, _ptr(h))
    return h, int(flag)


def make_hyper(*, inv: float, clip: float | None, lr: float, beta1: float, beta2: float,
               eps: float, t: int) -> Hyper:
    bc1, bc2 = bias_corrections(beta1, beta2, t)
    return Hyper(
        inv_scale=inv,
        use_clip=0 if clip is None else 1,
        clip=1.0 if clip is None else clip,
        lr=f32(lr), beta1=f32(beta1), beta2=f32(beta2), eps=f32(eps),
        one_minus_beta1=f32(f32(1.0) - f32(beta1)),
        one_minus_beta2=f32(f32(1.0) - f32(beta2)),
        bc1=bc1, bc2=bc2,
    )


def adam(h, dtype: int, hyper: Hyper, w: np.ndarray, m: np.ndarray, v: np.ndarray) -> np.ndarray:
    """Adam on the fp32 master state (in place) and the 16-bit cast."""
    h = _bits(h, dtype)
    for a in (w, m, v):
        if a.dtype != np.float32 or not a.flags.c_contiguous or a.size != h.size:
            raise ValueError("state arrays are contiguous float32 of the gradient's length")
    p16 = np.empty(h.size, bits_dtype(dtype))
    lib().oracle_adam(h.size, _ptr(h), dtype, ctypes.byref(hyper), _ptr(w), _ptr(m), _ptr(v), _ptr(p16))
    return p16


def sgd(h, dtype: int, hyper: Hyper, w: np.ndarray, m=None) -> np.ndarray:
    """SGD (with momentum when m is given, mu = hyper.beta1) on the fp32
    master weights (in place) and the 16-bit cast."""
    h = _bits(h, dtype)
    for a in (w,) + ((m,) if m is not None else ()):
        if a.dtype != np.float32 or not a.flags.c_contiguous or a.size != h.size:
            raise ValueError("state arrays are contiguous float32 of the gradient's length")
    p16 = np.empty(h.size, bits_dtype(dtype))
    lib().oracle_sgd(h.size, _ptr(h), dtype, ctypes.byref(hyper), _ptr(w), _ptr(m) if m is not None else None,
                     _ptr(p16))
    return p16


OPTIMIZERS = ("adam", "sgdm", "sgd")
OPTIM_K = {"adam": 12, "sgdm": 8, "sgd": 4}   # fp32 bytes per parameter incl. the fp32 master copy


def cast16(w: np.ndarray, dtype: int) -> np.ndarray:
    """The model-precision copy of w (16-bit patterns; FP32: w's own bits)."""
    w = _f32arr(w)
    p = np.empty(w.size, bits_dtype(dtype))
    lib().oracle_cast(w.size, _ptr(w), dtype, _ptr(p))
    return p


def step(grads, w, m, v, *, dtype: int, lr: float, beta1: float, beta2: float, eps: float,
         t: int, loss_scale: float, max_grad_norm: float = 0.0, dynamic: bool = False,
         min_scale: float = 1.0, growth_interval: int = 0, good_steps: int = 0, optimizer: str = "adam",
         momentum: float = 0.0) -> dict:
    """One unpartitioned mixed-precision optimizer step (Adam by default;
    optimizer="sgdm" -- SGD with momentum `momentum`, state w, m -- or "sgd",
    state w only).

    grads: list of N_d uint16 arrays (each rank's 16-bit gradient, loss-scaled;
    uint32 binary32 patterns for dtype FP32, whose outputs h and p16 are
    binary32 patterns too)
    w, m, v: fp32 master weights, momentum, variance (updated in place unless
    the step is skipped).  t: number of steps applied so far; this step
    applies Adam step t+1.

    Returns h (reduced 16-bit gradient), overflow, skipped, grad_norm
    (+inf when overflowed, None when clipping is off), clip, p16 (the 16-bit
    cast of the resulting master weights), t, loss_scale, good_steps."""
    n_ranks = len(grads)
    h, overflow = reduce(grads, dtype)
    inv = inv_scale(loss_scale, n_ranks)
    norm = None
    clip = None
    if overflow:
        norm = math.inf if max_grad_norm > 0 else None
        p16 = cast16(w, dtype)
        t_new = t
    else:
        if max_grad_norm > 0:
            norm = grad_norm(exact_sumsq(h, dtype), inv)
            clip = clip_coef(norm, max_grad_norm)
        if optimizer == "adam":
            hyper = make_hyper(inv=inv, clip=clip, lr=lr, beta1=beta1, beta2=beta2, eps=eps, t=t + 1)
            p16 = adam(h, dtype, hyper, w, m, v)
        elif optimizer in ("sgdm", "sgd"):
            hyper = make_hyper(inv=inv, clip=clip, lr=lr, beta1=momentum, beta2=0.0, eps=0.0, t=1)
            p16 = sgd(h, dtype, hyper, w, m if optimizer == "sgdm" else None)
        else:
            raise ValueError(optimizer)
        t_new = t + 1
    new_scale, good = scaler_update(loss_scale, good_steps, bool(overflow), dynamic,
                                    min_scale, growth_interval)
    return dict(h=h, overflow=int(overflow), skipped=int(bool(overflow)), grad_norm=norm,
                clip=clip, inv=inv, p16=p16, t=t_new, loss_scale=new_scale, good_steps=good)


# ---------------------------------------------------------------------------
# Partitioning and buckets
# ---------------------------------------------------------------------------
DEFAULT_ALIGN = 2048


# ---------------------------------------------------------------------------
# P_a: partitioned activation checkpoints ([P2] 3.2.1; [P4] "P_a:
# Partitioned Activation Checkpointing")
# ---------------------------------------------------------------------------
def pa_plan(act_elems: int, n_mp: int, value_bytes: int = 2, align_elems: int = 0) -> dict:
    """Partition of one activation checkpoint of act_elems values across the
    N_m model-parallel ranks.  Without P_a every rank holds the whole
    checkpoint (model parallelism replicates a layer's input on every rank);
    with P_a rank r keeps only the contiguous slice [rP, (r+1)P), P =
    ceil(act_elems / N_m) rounded up to the alignment, and the slices are
    all-gathered when backward recomputes the layer; with P_a+cpu the slices
    live in host memory.  Bytes per rank, and the bytes a rank receives in
    one all-gather (the other ranks' slices)."""
    A = align_elems or DEFAULT_ALIGN
    P = -(-act_elems // n_mp)
    P = -(-P // A) * A
    own = [max(0, min(P, act_elems - r * P)) for r in range(n_mp)]
    return dict(act_elems=act_elems, n_mp=n_mp, shard=P, own=own,
                mem_per_rank=act_elems * value_bytes,
                mem_per_rank_pa=P * value_bytes,
                mem_per_rank_pa_cpu=0,
                gather_recv_per_rank=[(act_elems - own[r]) * value_bytes for r in range(n_mp)])


def pa_partition(replicas, n_mp: int, shard: int):
    """Rank r keeps the slice [r*shard, (r+1)*shard) of its own replica."""
    return [np.array(replicas[r][r * shard:(r + 1) * shard]) for r in range(n_mp)]


def pa_gather(shards, act_elems: int):
    """The full checkpoint: the ranks' slices concatenated in rank order."""
    return np.concatenate(shards)[:act_elems]


def plan(n_params: int, n_ranks: int, bucket_elems: int, align_elems: int = 0,
         layer_sizes=None) -> dict:
    """ZeRO-DP partition of a flat parameter vector of n_params elements.

    Shard P = ceil(n_params / N_d) rounded up to the alignment A; rank r owns
    flat indices [rP, (r+1)P) ([P3] stage list: each rank keeps 1/N_d).
    Buckets are consecutive windows of bucket_elems elements over
    [0, n_params) in parameter order (constant-size fusion buffers, [P2]
    3.2.2).  Layers (gather units for stage 3) are consecutive runs of the
    parameter list."""
    A = align_elems or DEFAULT_ALIGN
    shard = -(-n_params // n_ranks)
    shard = -(-shard // A) * A
    nb = -(-n_params // bucket_elems) if n_params else 0
    buckets = [(b * bucket_elems, min((b + 1) * bucket_elems, n_params)) for b in range(nb)]
    if layer_sizes is None:
        layer_sizes = [n_params] if n_params else []
    layer_sizes = [int(x) for x in layer_sizes]
    if sum(layer_sizes) != n_params:
        raise ValueError("layer sizes must add up to n_params")
    starts = [0]
    for s in layer_sizes:
        starts.append(starts[-1] + s)
    return dict(n_params=n_params, n_ranks=n_ranks, shard=shard, padded=shard * n_ranks,
                bucket_elems=bucket_elems, n_buckets=nb, buckets=buckets,
                layer_sizes=layer_sizes, layer_starts=starts[:-1],
                max_layer=max(layer_sizes) if layer_sizes else 0)


def owner(p: dict, i: int) -> int:
    return i // p["shard"]


def bucket_segments(p: dict, b: int) -> list[tuple[int, int, int]]:
    """(rank, offset within the rank's shard, length) for each rank that owns
    part of bucket b, in rank order."""
    lo, hi = p["buckets"][b]
    P = p["shard"]
    segs = []
    for r in range(p["n_ranks"]):
        a, z = max(lo, r * P), min(hi, (r + 1) * P)
        if a < z:
            segs.append((r, a - r * P, z - a))
    return segs


# ---------------------------------------------------------------------------
# Memory and communication accounting ([P3] stage formulas, examples, tables)
# ---------------------------------------------------------------------------
def model_state_bytes(psi, n_ranks: int, stage: int, b: int = 2, K: int = 12) -> dict:
    """Per-rank model-state bytes as exact rationals.

    b: bytes per parameter of the model copy (and of the gradient): 2 in
    mixed precision, 4 in fp32.  K: optimizer-state bytes per parameter: 12
    for mixed-precision Adam (fp32 master + momentum + variance), and for
    other optimizers the multiplier of [P3]'s calculator (Adam 8, SGD with
    momentum 4, SGD 0, plus 4 for an fp32 master copy in mixed precision).
    Stage 0 keeps everything, stage 1 partitions the optimizer state, stage 2
    also the gradients, stage 3 also the parameters ([P3] stage formulas;
    [P2] 3.1.1-3.1.3)."""
    psi = Fraction(psi)
    N = Fraction(n_ranks)
    params = b * psi
    grads = b * psi
    optim = K * psi
    if stage >= 1:
        optim /= N
    if stage >= 2:
        grads /= N
    if stage >= 3:
        params /= N
    return dict(params=params, grads=grads, optim=optim, total=params + grads + optim)


COLLECTIVE_PASSES = {0: 2, 1: 3, 2: 2, 3: 3}   # RS+AG, AR+AG, RS+AG, RS+2*AG (in units of psi)


def comm_bytes(psi: int, n_ranks: int, stage: int, b: int = 2) -> dict:
    """Communication per step.

    paper: the per-rank volume of [P3]'s communication accounting and [P1]
    section 04 -- 2*psi elements for stages 0-2 (all-reduce = reduce-scatter
    + all-gather, or the stage-2 reduce-scatter + all-gather) and 3*psi for
    stage 3 (an extra parameter all-gather, forward and backward) -- times b.
    counted: bytes that cross simulated rank boundaries, all ranks together:
    each reduce-scatter or all-gather pass over psi elements moves
    (N_d - 1) * psi elements; stage 1 counts its end-of-step parameter
    all-gather as a third pass ([P3], "Stage 1 with the step-end gather")."""
    paper_passes = 3 if stage == 3 else 2
    return dict(paper=Fraction(paper_passes * psi * b),
                counted=COLLECTIVE_PASSES[stage] * (n_ranks - 1) * psi * b,
                counted_passes=COLLECTIVE_PASSES[stage])


def hbm_bytes_per_param(n_ranks: int, stage: int, mode: str, state_bytes: int = 12, value_bytes: int = 2) -> int:
    """Algorithmic HBM bytes per parameter of one step with N_d simulated
    ranks in one memory.  mode 'fused': one pass, new state written beside the
    old; 'two_pass': reduced gradient materialised, then read back.
    Gradient and parameter values are value_bytes each (2 for 16-bit, 4 for
    fp32 training); state_bytes = fp32 state per parameter (12 for Adam's w,
    m, v; 8 for SGD with momentum; 4 for SGD), read and written."""
    N, sb, e = n_ranks, state_bytes, value_bytes
    if mode == "fused":
        return {0: N * (3 * e + 2 * sb), 1: 3 * e * N + 2 * sb, 2: 2 * e * N + 2 * sb, 3: e * N + 2 * sb + e}[stage]
    if mode == "two_pass":
        return {0: N * (4 * e + 2 * sb), 1: 3 * e * N + e + 2 * sb, 2: 2 * e * N + 2 * e + 2 * sb,
                3: e * N + 3 * e + 2 * sb}[stage]
    if mode == "restore":   # after an overflowed fused step: read w, write each model-precision copy
        return {0: (4 + e) * N, 1: 4 + e * N, 2: 4 + e * N, 3: 4 + e}[stage]
    raise ValueError(mode)


GB = Fraction(10 ** 9)   # [P3]: GB means 10^9 bytes, not GiB


def display_gb(x) -> str:
    """[P3]'s display rule: at or above 100 GB the integer part; 10-100 GB at
    most one decimal; below 10 GB at most two decimals; no trailing zeros.
    Rounding below 100 GB is half-up (Table 1 prints 41.25 as 41.3); the
    integer part at or above 100 GB is a floor (4187.5 prints as 4187)."""
    x = Fraction(x)
    if x >= 100:
        return str(math.floor(x))
    digits = 1 if x >= 10 else 2
    q = Fraction(10) ** digits
    r = Fraction(math.floor(x * q + Fraction(1, 2)), q)
    s = f"{float(r):.{digits}f}"
    s = s.rstrip("0").rstrip(".")
    return s


def max_model_size(mem_bytes, n_ranks: int, stage: int, mp: int = 1) -> Fraction:
    """Largest parameter count whose model states fit in mem_bytes per GPU
    with N_d-way ZeRO-DP and mp-way model parallelism (Table 2's theoretical
    columns)."""
    per_param = model_state_bytes(1, n_ranks, stage)["total"]
    return Fraction(mem_bytes) * mp / per_param
