"""Benchmark: ZeRO sharded mixed-precision Adam step on GB300.

Workload (default, the largest single-GPU configuration): ZeRO stage 3 on
the parameter list of a 32-layer d=4096 transformer (embedding 50257 x
4096, per layer 4 d^2 attention + 8 d^2 MLP + 4 d LayerNorm vectors:
6,648,827,904 parameters), N_d = 64 simulated data-parallel ranks, bucket
2^24 elements, fp16 gradients N(0, 1e-3) x 1024 (static loss scale 1024),
Adam (lr 1e-4, betas 0.9/0.999, eps 1e-8).  A step is one pass of the whole
hot path: every layer gathered from the 64 owners' shards into 64
constant-size buffers for the forward pass, and again, in reverse order,
for the backward pass, where each bucket's 64 gradient copies are
reduce-scattered, checked, unscaled, applied by Adam to the owned fp32
shard and cast back into the owner's 16-bit shard; then the commit.  Each
bucket's gradients come from a ring of pre-generated gradient sets in HBM
(generation is not part of the step).  Also reported, each with its own
roofline: the stage-2 step on a 12-layer d=768 list (N_d = 8) and the
clipped stage-2 steps at 2^31 parameters (N_d = 2 and 32, bf16).

Output: one JSON line (rank 0).  `value` is parameters updated per second
over all GPUs with inputs resident in HBM; `e2e` is the same through the C
ABI with every bucket's gradients copied in from pinned host memory inside
the timed region; `roofline` is the dominant kernel's (the layer gather's)
algorithmic bytes per launch over its CUDA-event duration against the
measured HBM copy bandwidth, with the other kernel and the whole step
beside it.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
  python bench.py --config K          the other workloads (bench_workloads.py)

With --gpus N > 1 (under torchrun) each rank runs an independent replica of
the job on its own GPU: the simulated ranks live inside one GPU, so there is
no data-path collective between GPUs; timing is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "Gparams/s per sharded Adam step; achieved HBM GB/s vs GB300 peak"
UNIT = "Gparams/s"
VOCAB, D_MODEL, N_LAYERS = 50257, 768, 12
N_RANKS = 8
BUCKET = 1 << 24
STAGE = 2
SIGMA = 1e-3
ADAM = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8)
GRAD_RING = 10          # distinct per-step gradient sets ("10 steps, fresh seeds per step")
FALLBACK_HBM_GBS = 6800.0
# GB300's nominal HBM3e bandwidth: NVIDIA's GB300 NVL72 specification gives
# 576 TB/s over its 72 GPUs, 8 TB/s per GPU.  Reported beside the fraction of
# the measured copy bandwidth, which is the roofline's denominator.
CHIP_HBM_GBS = 8000.0
CHIP_HBM_SOURCE = "NVIDIA GB300 NVL72 specification: 576 TB/s HBM3e over 72 GPUs = 8 TB/s per GPU (nominal)"
KERNEL_SOURCES = ["zero_sharded_mixed_bucket_gb300/csrc/k_fused.cu",
                  "zero_sharded_mixed_bucket_gb300/csrc/dev_common.cuh",
                  "zero_sharded_mixed_bucket_gb300/csrc/zero_internal.h"]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "k_fused_stage2_fp16_n8.md")
GATHER_SOURCES = ["zero_sharded_mixed_bucket_gb300/csrc/k_gather.cu",
                  "zero_sharded_mixed_bucket_gb300/csrc/dev_common.cuh",
                  "zero_sharded_mixed_bucket_gb300/csrc/zero_internal.h"]
GATHER_SUMMARY = os.path.join(ROOT, "profiles", "k_gather_stage3_n64.md")
S3_LAYERS, S3_D, S3_RANKS, S3_SCALE = 32, 4096, 64, 1024.0


def bytes_per_param(stage, n=N_RANKS, sb=12, e=2):
    """Algorithmic HBM bytes per parameter of the fused step (gradient and
    parameter values e bytes -- 2 for 16-bit, 4 for fp32 training -- and sb
    bytes of fp32 state -- 12 for Adam's w, m, v): N gradient reads, the
    all-reduce write-back in stages 0/1, the state read and written, the
    parameter writes."""
    return {0: n * (3 * e + 2 * sb), 1: 3 * e * n + 2 * sb, 2: 2 * e * n + 2 * sb, 3: e * n + 2 * sb + e}[stage]


DTYPES = {"fp16": 0, "bf16": 1, "fp32": 2}


def layer_sizes(vocab=VOCAB, d=D_MODEL, layers=N_LAYERS):
    return [vocab * d] + [12 * d * d + 4 * d] * layers


N_PARAMS = sum(layer_sizes())
S3_N_PARAMS = sum(layer_sizes(VOCAB, S3_D, S3_LAYERS))
S3_WORKLOAD = ("ZeRO stage 3, 32-layer d=4096 transformer parameter list (%d params), N_d=64 simulated ranks, "
               "bucket 2^24 elements, two all-gathers per layer into 64 constant-size buffers, fp16 gradients "
               "N(0,1e-3) x 1024 static loss scale, Adam" % S3_N_PARAMS)
WORKLOAD = ("12-layer d=768 transformer parameter list (%d params), N_d=%d simulated ranks, ZeRO stage %d, "
            "bucket 2^24 elements, fp16 gradients N(0,1e-3), Adam" % (N_PARAMS, N_RANKS, STAGE))


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def kernel_source_hash(sources=None) -> str:
    """First 16 hex digits of the SHA-256 of a kernel's source files: an ncu
    summary records it, and its counters are used only while it matches."""
    h = hashlib.sha256()
    for p in sources or KERNEL_SOURCES:
        with open(os.path.join(ROOT, p), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_peak_hbm():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profiled_value(key, summary=PROFILE_SUMMARY, sources=None):
    """A number recorded as `key: value` in a committed ncu summary, if the
    summary's kernel_source_hash matches the current kernel source (counters
    taken on other code do not count); else None."""
    try:
        text = open(summary, encoding="utf-8").read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_val = re.search(re.escape(key) + r":\s*([0-9.eE+]+)", text)
    if not m_hash or not m_val or m_hash.group(1) != kernel_source_hash(sources):
        return None
    return float(m_val.group(1))


def profiled_traffic():
    """dram bytes per full-bucket launch of the stage-2 fused kernel from its
    committed ncu summary (None when it was taken on other code)."""
    return profiled_value("dram_bytes_per_full_launch")


def traffic_source(summary, sources):
    return {"summary": os.path.relpath(summary, ROOT), "kernel_source_hash": kernel_source_hash(sources),
            "note": "dram__bytes_read.sum + dram__bytes_write.sum of one ncu capture of a smaller launch, scaled "
                    "to the average launch by its elements; writes read below the algorithmic count when dirty "
                    "L2 lines are written back after the captured kernel ends"}


class ClockSampler:
    """nvidia-smi samples (with their own timestamps) while the GPU works."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.f = tempfile.NamedTemporaryFile("w", prefix="clocks_", suffix=".csv", delete=False)
        self.path = self.f.name
        self.proc = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits",
                                          "-i", str(gpu), "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        rows = []
        if self.proc is None:
            return rows
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                rows.append(dict(t=ts, sm=float(parts[2]), max=float(parts[3]),
                                 power=float(parts[4]) if parts[4] not in ("[N/A]", "N/A") else None,
                                 hw=parts[6], hwt=parts[7], swt=parts[8], pcap=parts[9]))
            except (ValueError, IndexError):
                continue
        os.unlink(self.path)
        return rows


def clocks_summary(rows, t0, t1):
    inside = [r for r in rows if t0 - 0.05 <= r["t"] <= t1 + 0.05]
    window = "timed"
    if not inside:
        # the timed region is shorter than the sampling interval: nearest samples
        inside = sorted(rows, key=lambda r: abs(r["t"] - (t0 + t1) / 2))[:3]
        window = "nearest samples to the timed region"
    if not inside:
        return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
    reasons = set()
    for r in inside:
        for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"), ("swt", "sw_thermal_slowdown"),
                          ("pcap", "sw_power_cap")):
            if r[key].lower().startswith("active"):
                reasons.add(name)
    return {"sm_mhz": statistics.median(r["sm"] for r in inside), "sm_max_mhz": max(r["max"] for r in inside),
            "reasons": sorted(reasons), "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------
def oracle_sample_step(n_sample, seed_step, ranks=S3_RANKS, scale=S3_SCALE):
    """Inputs of the oracle on the first n_sample parameters: every rank's
    fp16 gradients N(0, 1e-3) x scale, master weights N(0, 0.02), m = v = 0."""
    import numpy as np

    import synth
    grads = [synth.host_normal16(n_sample, synth.FP16, SIGMA * scale, seed=0, stream=synth.STREAM_GRAD,
                                 step=seed_step, rank=r) for r in range(ranks)]
    w = synth.host_normal32(n_sample, 0.02, seed=0, stream=synth.STREAM_WEIGHT)
    m = np.zeros(n_sample, np.float32)
    v = np.zeros(n_sample, np.float32)
    return grads, w, m, v


def run_oracle_steps(n_sample, steps, warmup, ranks=S3_RANKS, scale=S3_SCALE):
    import oracle
    grads, w, m, v = oracle_sample_step(n_sample, 1, ranks, scale)
    t = 0
    times = []
    for k in range(warmup + steps):
        t0 = time.perf_counter()
        r = oracle.step(grads, w, m, v, dtype=oracle.FP16, t=t, loss_scale=scale, **ADAM)
        dt = time.perf_counter() - t0
        t = r["t"]
        if k >= warmup:
            times.append(dt)
    return times


def host_cores() -> int:
    return len(os.sched_getaffinity(0))


def cpu_baseline(n_sample=1 << 22, steps=3, ranks=S3_RANKS, scale=S3_SCALE):
    """The oracle as it is (single-threaded C: one of the host's cores) on
    the first n_sample parameters of the workload."""
    times = run_oracle_steps(n_sample, steps, 0, ranks, scale)
    sec = sum(times) / len(times)
    return {"value": n_sample / sec / 1e9, "unit": UNIT, "cores": 1, "host_cores": host_cores(), "kind": "oracle",
            "sample": "%d contiguous parameters of the workload, N_d=%d ranks, loss scale %g, %d steps, "
                      "single-threaded C oracle (the unpartitioned step: every stage computes the same numbers; "
                      "the stage-3 gathers are copies of its 16-bit result)" % (n_sample, ranks, scale, steps),
            "seconds": sum(times)}


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    n_sample = 1 << 19
    times = run_oracle_steps(n_sample, args.steps, args.warmup)
    sec = sum(times) / len(times)
    value = n_sample / sec / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": S3_WORKLOAD, "n_params": S3_N_PARAMS, "n_ranks": S3_RANKS, "stage": 3,
                       "bucket_elems": BUCKET, "sample_params": n_sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "host_cores": host_cores(), "kind": "oracle",
                             "sample": "%d parameters of the workload per step, N_d=%d, loss scale %g, "
                                       "single-threaded C oracle" % (n_sample, S3_RANKS, S3_SCALE)},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


# ---------------------------------------------------------------------------
# GPU legs
# ---------------------------------------------------------------------------
OPTIMIZERS = {"adam": 0, "sgdm": 1, "sgd": 2}
STATE_BYTES = {0: 12, 1: 8, 2: 4}


class GpuJob:
    def __init__(self, stage, device, ring=GRAD_RING, n_params=None, optimizer=0, dtype=0):
        import torch

        import synth
        import zero_sharded_mixed_bucket_gb300 as zg
        self.zg, self.torch = zg, torch
        self.stage = stage
        self.n = n_params or N_PARAMS
        self.optimizer = optimizer
        self.dtype = dtype
        self.e = 4 if dtype == zg.ZERO_FP32 else 2          # bytes per gradient / parameter value
        self.cfg = zg.Config(self.n, N_RANKS, stage, BUCKET, 0, layer_sizes() if self.n == N_PARAMS else None,
                             dtype, optimizer)
        self.plan = zg.zero_plan(self.cfg)
        self.bufs = zg.DeviceBuffers(self.cfg, self.plan, device=device, grads=True)
        self.stream = torch.cuda.current_stream(device)
        s = self.stream.cuda_stream
        reps = N_RANKS if stage == 0 else 1
        for r in range(reps):
            synth.dev_normal32(self.bufs.w[0].data_ptr() + 4 * r * self.plan.padded_elems, self.n, 0.02, seed=0,
                               stream=synth.STREAM_WEIGHT, cuda_stream=s)
        # gradient ring: GRAD_RING steps' worth of fresh gradients, each set N_d buffers
        self.ring = []
        self.ring_ptrs = []
        import ctypes
        for k in range(ring):
            vt = torch.int32 if self.e == 4 else torch.int16
            bufs = [torch.empty(self.plan.grad16_elems, dtype=vt, device=device) for _ in range(N_RANKS)]
            for r in range(N_RANKS):
                synth.dev_grad(bufs[r].data_ptr(), self.n, dtype, SIGMA, seed=0, stream=synth.STREAM_GRAD,
                               step=k + 1, rank=r, cuda_stream=s)
            self.ring.append(bufs)
            self.ring_ptrs.append((ctypes.c_void_p * N_RANKS)(*[b.data_ptr() for b in bufs]))
        self.adam = zg.zero_adam_t(max_grad_norm=0.0, momentum=0.9, **ADAM)
        self.state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
        torch.cuda.synchronize(device)

    def set_ring(self, k):
        import ctypes
        self.bufs.b.grads = ctypes.cast(self.ring_ptrs[k % len(self.ring_ptrs)], ctypes.POINTER(ctypes.c_void_p))

    def step(self, k):
        """One optimizer step with gradient set k: one call into the library,
        which launches every bucket's kernel and reads the overflow flag."""
        zg = self.zg
        self.set_ring(k)
        fn = [zg.zero_step_stage0, zg.zero_step_stage1, zg.zero_step_stage2, zg.zero_step_stage3][self.stage]
        return fn(self.cfg, self.plan, self.bufs, self.adam, self.state, self.stream)

    def init_dev_state(self):
        """A device-resident copy of the step state for zero_step_async."""
        torch, zg = self.torch, self.zg
        self.dev = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device=self.bufs.workspace.device)
        zg.zero_dev_state_init(self.dev, self.adam, self.state, self.stream)

    def step_async(self, k):
        """One optimizer step with gradient set k, enqueued without any host
        synchronisation (step state on the device).  Returns the kernels launched."""
        self.set_ring(k)
        return self.zg.zero_step_async(self.cfg, self.plan, self.bufs, self.adam, self.dev, self.stream)

    def bucket_len(self, b):
        lo = b * BUCKET
        return min(lo + BUCKET, self.n) - lo


def dist_setup(args):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest of every rank's x (the slowest rank's time)."""
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    device = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate(ms_local: float, n_params: int, steps: int, world: int):
    """Whole-job figures: every rank runs its own replica of the job, so the
    job processes world * n_params parameters per step in the slowest rank's
    time.  Returns (ms_per_step, Gparams/s)."""
    ms_per_step = max_over_ranks(ms_local, world) / steps
    return ms_per_step, world * n_params / (ms_per_step * 1e-3) / 1e9


def timed_steps(job, steps, warmup, world, api="sync"):
    """Time `steps` steps after `warmup` untimed ones.  Returns the elapsed
    milliseconds (CUDA events on the job's stream around all timed steps),
    the kernels launched, the kernel span per step (events the library records
    before the first and after the last bucket kernel of each step) and the
    host wall-clock window of the timed region.

    api="sync": zero_step_stage*, which reads the overflow flag at the end of
    every step; api="async": zero_step_async, step state on the device, steps
    enqueued back to back and the state read once after the timed region."""
    import torch
    zg = job.zg
    if api == "async":
        return _timed_steps_async(job, steps, warmup, world)
    for k in range(warmup):
        job.step(k)
    span_start, span_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    span_start.record(job.stream)
    span_end.record(job.stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    spans = []
    zg.zero_set_profile_events(span_start, span_end)
    try:
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        start.record(job.stream)
        for k in range(steps):
            res = job.step(warmup + k)      # returns after the step's flag read (stream synchronised)
            spans.append(span_start.elapsed_time(span_end))
            launches += res.kernel_launches
            assert res.overflow == 0
        end.record(job.stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
    finally:
        zg.zero_set_profile_events(None, None)
    ms = start.elapsed_time(end)
    nb = job.plan.n_buckets
    step_bytes = sum(job.bucket_len(b) for b in range(nb)) * bytes_per_param(job.stage, N_RANKS,
                                                                              STATE_BYTES[job.optimizer], job.e)
    kernel = dict(total_ms=sum(spans), bytes=steps * step_bytes, launches=steps * nb,
                  span_ms_per_step=sum(spans) / steps, launches_per_step=nb)
    return ms, launches, kernel, (t0, t1)


# Profile events (library-recorded around a step's bucket kernels) go on every
# PROFILE_EVERY-th timed step only: an event recorded between two kernels breaks
# the programmatic-dependent launch chain of the device-state step, and events
# on every step measured 1.0186 against 1.0098 ms per headline step.
PROFILE_EVERY = 4


def _timed_steps_async(job, steps, warmup, world):
    import torch
    zg = job.zg
    job.init_dev_state()
    for k in range(warmup):
        job.step_async(k)
    evs = {k: (torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for k in range(0, steps, PROFILE_EVERY)}
    for a, b in evs.values():              # recorded once so that the library may re-record them
        a.record(job.stream)
        b.record(job.stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    try:
        barrier(world)
        torch.cuda.synchronize()
        t0 = time.time()
        start.record(job.stream)
        for k in range(steps):
            zg.zero_set_profile_events(*evs.get(k, (None, None)))
            launches += job.step_async(warmup + k)
        end.record(job.stream)
        torch.cuda.synchronize()
        t1 = time.time()
        barrier(world)
    finally:
        zg.zero_set_profile_events(None, None)
    st, last = zg.zero_dev_state_read(job.dev, job.stream)
    assert st.t == warmup + steps and last.overflow == 0, "a step overflowed"
    ms = start.elapsed_time(end)
    spans = [a.elapsed_time(b) for a, b in evs.values()]
    nb = job.plan.n_buckets
    step_bytes = sum(job.bucket_len(b) for b in range(nb)) * bytes_per_param(job.stage, N_RANKS,
                                                                              STATE_BYTES[job.optimizer], job.e)
    kernel = dict(total_ms=sum(spans), bytes=len(spans) * step_bytes, launches=len(spans) * nb,
                  span_ms_per_step=sum(spans) / len(spans), launches_per_step=nb, profiled_steps=len(spans))
    return ms, launches, kernel, (t0, t1)


def e2e_leg(job, steps, warmup, device, world=1):
    """Same step through the C ABI with each step's gradients copied in from
    pinned host memory (bucket by bucket on a copy stream, overlapped with the
    previous bucket's kernel) and the step result read back by the library.
    With several ranks all run at once (each GPU has its own host link); the
    time is the slowest rank's and the value counts every rank's parameters."""
    import torch
    zg = job.zg
    n = N_PARAMS
    host = []
    for k in range(2):
        hb = [torch.empty(n, dtype=torch.int16, pin_memory=True) for _ in range(N_RANKS)]
        for r in range(N_RANKS):
            hb[r].copy_(job.ring[k][r][:n])
        host.append(hb)
    dev = job.ring[0]
    job.set_ring(0)
    copy_stream = torch.cuda.Stream(device)
    nb = job.plan.n_buckets

    def one(k):
        hb = host[k % 2]
        done = []
        for b in range(nb):
            lo, hi = b * BUCKET, min((b + 1) * BUCKET, n)
            with torch.cuda.stream(copy_stream):
                for r in range(N_RANKS):
                    dev[r][lo:hi].copy_(hb[r][lo:hi], non_blocking=True)
                e = torch.cuda.Event()
                e.record(copy_stream)
            done.append(e)
        zg.zero_step_begin(job.cfg, job.plan, job.bufs, job.adam, job.state, job.stream)
        for b in range(nb):
            job.stream.wait_event(done[b])
            zg.zero_step_bucket(job.cfg, job.plan, job.bufs, job.adam, job.state, b, None, job.stream)
        res = zg.zero_step_end(job.cfg, job.plan, job.bufs, job.adam, job.state, job.stream)
        # the next step's copies must not overwrite gradients still being read
        copy_stream.wait_stream(job.stream)
        return res

    def timed(fn):
        for k in range(warmup):
            fn(k)
        torch.cuda.synchronize()
        barrier(world)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(job.stream)
        for k in range(steps):
            res = fn(warmup + k)
            assert res.overflow == 0
        end.record(job.stream)
        torch.cuda.synchronize()
        ms = max_over_ranks(start.elapsed_time(end) / steps, world)
        barrier(world)
        return ms

    import ctypes
    host_ptrs = [(ctypes.c_void_p * N_RANKS)(*[t.data_ptr() for t in hb]) for hb in host]

    def direct(k):
        # the fused kernel loads each rank's gradient straight from pinned host
        # memory over NVLink-C2C: no copy engine, no device staging
        job.bufs.b.grads = ctypes.cast(host_ptrs[k % 2], ctypes.POINTER(ctypes.c_void_p))
        return zg.zero_step_stage2(job.cfg, job.plan, job.bufs, job.adam, job.state, job.stream)

    ms_copy = timed(one)
    ms_direct = timed(direct)
    job.set_ring(0)
    h2d = N_RANKS * n * 2
    ms = min(ms_copy, ms_direct)
    mode = "direct" if ms_direct <= ms_copy else "copy"
    return dict(value=world * n / (ms * 1e-3) / 1e9, unit=UNIT, h2d_bytes_per_step=world * h2d,
                d2h_bytes_per_step=world * 32, ms_per_step=ms, mode=mode,
                host_link_gbs_per_gpu=h2d / (ms * 1e-3) / 1e9,
                modes={"copy": {"ms_per_step": ms_copy, "value": world * n / (ms_copy * 1e-3) / 1e9,
                                "note": "per-bucket cudaMemcpyAsync from pinned host memory on a second stream, "
                                        "overlapped with the previous bucket's kernel"},
                       "direct": {"ms_per_step": ms_direct, "value": world * n / (ms_direct * 1e-3) / 1e9,
                                  "note": "the fused kernel reads the gradients from pinned host memory over "
                                          "NVLink-C2C"}},
                note="every step moves the step's 16-bit gradients of all ranks from pinned host memory to the "
                     "GPU and reads the 32-byte step result back")


def gpu_arm(args):
    global BUCKET
    BUCKET = args.bucket
    import torch
    world, rank, local = dist_setup(args)
    device = torch.device("cuda", local)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()      # one builder: concurrent builds would write the same object files
    barrier(world)
    dt_name = args.dtype or "fp16"
    stage = args.stage
    job = GpuJob(stage, device, ring=args.ring, n_params=args.n_params, optimizer=OPTIMIZERS[args.optimizer],
                 dtype=DTYPES[dt_name])
    n_params = job.n
    sampler = ClockSampler(local)
    ms, launches, kernel, (t0, t1) = timed_steps(job, args.steps, args.warmup, world, api=args.step_api)
    rows = sampler.stop()
    ms_per_step, value = aggregate(ms, n_params, args.steps, world)
    peak, peak_kind = measured_peak_hbm()
    achieved = kernel["bytes"] / (kernel["total_ms"] * 1e-3) / 1e9
    per_launch = kernel["bytes"] / kernel["launches"]
    # the committed capture is of the fp16 Adam kernel: no counters for the other variants
    traffic_full = profiled_traffic() if (stage, dt_name, args.optimizer) == (2, "fp16", "adam") else None
    # the capture is of a full 2^24-element bucket: scale to the average launch
    traffic = None if traffic_full is None else traffic_full * (n_params / kernel["launches_per_step"]) / (1 << 24)
    step_bytes = job.plan.hbm_bytes_fused
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "io_dtype": dt_name, "data": "synthetic",
        "config": {"workload": (WORKLOAD if n_params == N_PARAMS else
                                "flat parameter vector of %d params, N_d=%d simulated ranks, ZeRO stage 2, bucket "
                                "2^24 elements, fp16 gradients N(0,1e-3), Adam" % (n_params, N_RANKS))
                   .replace("ZeRO stage 2", "ZeRO stage %d" % stage)
                   .replace("fp16 gradients", "%s gradients" % dt_name)
                   .replace("Adam", {"adam": "Adam", "sgdm": "SGD with momentum 0.9", "sgd": "SGD"}[args.optimizer]),
                   "n_params": n_params, "n_ranks": N_RANKS, "stage": stage,
                   "bucket_elems": BUCKET, "parallelism": "replicas only (simulated ranks inside each GPU)",
                   "l2": "inputs larger than L2: %.2f GB moved per step, %d-step gradient ring of %.1f GB"
                         % (step_bytes / 1e9, args.ring, args.ring * N_RANKS * n_params * 2 / 1e9)},
        "hbm_gbs_step": step_bytes / (ms_per_step * 1e-3) / 1e9,
        "roofline": {"bound": "hbm",
                     "kernel": "%s<stage %d, %s, %s>" % (
                         "k_fused_tiled" if stage == 1 or (stage == 2 and (args.optimizer != "adam" or
                                                                           dt_name == "fp32")) else "k_fused",
                         stage, dt_name, args.optimizer),
                     "achieved": achieved, "peak": peak,
                     "peak_kind": peak_kind, "unit": "GB/s", "frac": achieved / peak,
                     "traffic": traffic, "algorithmic_bytes_per_launch": per_launch,
                     "bytes_per_param": bytes_per_param(stage, N_RANKS, STATE_BYTES[job.optimizer], job.e),
                     "launches": kernel["launches"],
                     "avg_launch_ms": kernel["total_ms"] / kernel["launches"],
                     "kernel_span_ms_per_step": kernel["span_ms_per_step"],
                     "timing": "library-recorded CUDA events around a step's bucket kernels on the step's "
                               "stream (%s); consecutive bucket kernels overlap their edges, so a launch's "
                               "duration is the step's kernel span over its launches"
                               % ("every step" if args.step_api == "sync" else
                                  "every %dth timed step: %d of %d" % (PROFILE_EVERY, kernel.get("profiled_steps", 0),
                                                                       args.steps))},
        "gpu_launches": launches,
    }
    out["optimizer"] = args.optimizer
    out["step_api"] = {"async": "zero_step_async (step state in device memory, no host synchronisation between "
                                "steps)", "sync": "zero_step_stage%d (overflow flag read by the host every step)" % stage
                       }[args.step_api]
    out["clocks"] = clocks_summary(rows, t0, t1)
    if args.headline_only:
        if rank == 0:
            print(json.dumps(out))
    elif args.optimizer != "adam" or dt_name != "fp16":
        raise SystemExit("--optimizer other than adam or --dtype other than fp16 needs --headline-only")
    else:
        if rank == 0:
            # the other step entry point on the same job (reported, not the headline)
            other = "sync" if args.step_api == "async" else "async"
            try:
                k = max(5, args.steps // 4)
                oms, _, ok, _ = timed_steps(job, k, 3, 1, api=other)
                out["other_step_api"] = {"api": other, "steps": k, "ms_per_step": oms / k,
                                         "value": n_params / (oms / k * 1e-3) / 1e9,
                                         "kernel_span_ms_per_step": ok["span_ms_per_step"]}
            except Exception as e:    # reported, never hides the headline
                out["other_step_api"] = {"api": other, "error": repr(e)}
        del job
        torch.cuda.empty_cache()
        # end to end on every rank at once: each GPU has its own host link
        barrier(world)
        if world == 1:
            try:
                j2 = GpuJob(STAGE, device, ring=2)
                e2e = e2e_leg(j2, max(3, args.steps // 2), 3, device, world)
                del j2
            except Exception as e:   # reported, never hides the headline
                e2e = {"error": repr(e)}
        else:
            j2 = GpuJob(STAGE, device, ring=2)
            e2e = e2e_leg(j2, max(3, args.steps // 2), 3, device, world)
            del j2
        torch.cuda.empty_cache()
        if rank == 0:
            out["e2e"] = e2e
            # stages 0 and 1 on the same workload (reported, not the headline).
            # Stages 0/1 overwrite each rank's gradient with the all-reduce result,
            # so every step gets a gradient set of its own.
            stages = {}
            st_steps, st_warm = 5, 3
            for st in (1, 0):
                try:
                    j = GpuJob(st, device, ring=st_steps + st_warm)
                    sms, _, sk, _ = timed_steps(j, st_steps, st_warm, 1, api=args.step_api)
                    stages["stage%d" % st] = {"ms_per_step": sms / st_steps,
                                              "value": N_PARAMS / (sms / st_steps * 1e-3) / 1e9,
                                              "kernel_gbs": sk["bytes"] / (sk["total_ms"] * 1e-3) / 1e9,
                                              "bytes_per_param": bytes_per_param(st), "steps": st_steps}
                    del j
                except Exception as e:   # reported, never hides the headline
                    stages["stage%d" % st] = {"error": repr(e)}
                torch.cuda.empty_cache()
            out["stages"] = stages
            if world == 1:
                out["cpu_baseline"] = cpu_baseline(1 << 26, 2, N_RANKS, 1.0)
            print(json.dumps(out))
        barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


# ---------------------------------------------------------------------------
# the default line: the stage-3 step at 6.65B parameters
# ---------------------------------------------------------------------------
def stage3_e2e(job, steps, warmup, device, world=1, mode="direct"):
    """The stage-3 step through the C ABI with every bucket's 64 gradient
    copies crossing from pinned host memory to the GPU inside the timed
    region, and the step's result read back by the host after every step
    (zero_dev_state_read, 64 bytes).  Two pinned host sets of N_d x 2^24
    values serve the buckets alternately.

    mode "direct": each bucket kernel loads its 64 gradient windows straight
    from pinned host memory over NVLink-C2C (the library accepts any pointer
    the GPU can load from).  mode "copy": one cudaMemcpyAsync per bucket (the
    whole 2.1 GB set) on a second stream into one of two device sets,
    double-buffered against the bucket kernels.  Measured on GB300: direct
    199 GB/s on the host link; copy 140-160 GB/s, single 2.1 GB copies taking
    10 to 94 ms."""
    import torch
    zg = job.zg
    assert len(job.ring) >= 2
    host = [torch.empty(job.N * job.B, dtype=torch.int16).pin_memory() for _ in range(2)]
    for k in range(2):
        host[k].copy_(job.ring[k])
    host_ptrs = [zg.ptr_array([h.data_ptr() + 2 * r * job.B for r in range(job.N)]) for h in host]
    copy_stream = torch.cuda.Stream(device)
    free = [None, None]            # per device set: event after the bucket kernel that last read it

    def before(b):
        k = b % 2
        with torch.cuda.stream(copy_stream):
            if free[k] is not None:
                copy_stream.wait_event(free[k])
            job.ring[k].copy_(host[k], non_blocking=True)
            e = torch.cuda.Event()
            e.record(copy_stream)
        job.stream.wait_event(e)

    def after(b):
        e = torch.cuda.Event()
        e.record(job.stream)
        free[b % 2] = e

    def one():
        if mode == "direct":
            job.step(grad_ptrs=lambda b: host_ptrs[b % 2])
        else:
            job.step(grad_ptrs=lambda b: job.ring_ptrs[b % 2], before_bucket=before, after_bucket=after)
        st, last = zg.zero_dev_state_read(job.dev_state, job.stream)       # the step's result, to the host
        assert last.overflow == 0
        return st

    for _ in range(warmup):
        one()
    torch.cuda.synchronize()
    barrier(world)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record(job.stream)
    copy_stream.wait_event(start)
    for _ in range(steps):
        one()
    end.record(job.stream)
    torch.cuda.synchronize()
    ms = max_over_ranks(start.elapsed_time(end) / steps, world)
    barrier(world)
    nb = job.plan.n_buckets
    # bytes that cross the host link per step: direct, each bucket's windows
    # (N_d x bucket length); copy, the whole set per bucket
    h2d = job.N * job.n * 2 if mode == "direct" else nb * job.N * job.B * 2
    return dict(value=world * job.n / (ms * 1e-3) / 1e9, unit=UNIT, h2d_bytes_per_step=world * h2d,
                d2h_bytes_per_step=world * zg.DEV_STATE_BYTES, ms_per_step=ms, steps=steps, warmup=warmup,
                mode=mode, host_link_gbs_per_gpu=h2d / (ms * 1e-3) / 1e9,
                note="every step's 64 x 6.65e9 fp16 gradient values cross from pinned host memory to the GPU "
                     + ("(the bucket kernels load them over NVLink-C2C)" if mode == "direct" else
                        "(one cudaMemcpyAsync per bucket on a second stream, double-buffered)")
                     + "; the step's result block is read back after every step; the host link sets the pace")


def stage3_arm(args):
    import torch
    world, rank, local = dist_setup(args)
    device = torch.device("cuda", local)
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()      # one builder: concurrent builds would write the same object files
    barrier(world)
    import bench_workloads as bw
    import zero_sharded_mixed_bucket_gb300 as zg
    job = bw.Stage3Job(device, ring=args.ring3, n_layers=args.s3_layers, d=args.s3_d)
    n = job.n
    for _ in range(args.warmup):
        job.step()
    nsched = len(job.schedule)
    prof = {k: [torch.cuda.Event(enable_timing=True) for _ in range(nsched + 1)]
            for k in range(0, args.steps, PROFILE_EVERY)}
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.time()
    start.record(job.stream)
    for k in range(args.steps):
        job.step(events=prof.get(k))
    end.record(job.stream)
    torch.cuda.synchronize()
    t1 = time.time()
    barrier(world)
    rows = sampler.stop()
    st, last = zg.zero_dev_state_read(job.dev_state, job.stream)
    assert st.t == args.warmup + args.steps and last.overflow == 0, "a step overflowed"
    ms = start.elapsed_time(end)
    ms_per_step, value = aggregate(ms, n, args.steps, world)
    peak, peak_kind = measured_peak_hbm()
    # per-kernel durations from the profiled steps' events
    g_ms = b_ms = 0.0
    for evs in prof.values():
        g, b = job.kernel_times(evs)
        g_ms += g
        b_ms += b
    n_prof = len(prof)
    n_gathers = sum(1 for kind, _ in job.schedule if kind == "gather")
    g_bytes = n_prof * 2 * n * (2 + 2 * job.N)
    f_bytes = n_prof * n * bench_bytes(3, job.N)    # every bucket kernel of a profiled step
    g_launch = g_bytes / (n_prof * n_gathers)
    g_ach = g_bytes / (g_ms * 1e-3) / 1e9
    f_ach = f_bytes / (b_ms * 1e-3) / 1e9
    step_bytes = n * job.bytes_per_param()
    g_units = profiled_value("dram_bytes_per_gathered_element", GATHER_SUMMARY, GATHER_SOURCES)
    g_traffic = None if g_units is None else g_units * (2 * n / n_gathers)
    layers = "%d-layer d=%d" % (args.s3_layers, args.s3_d)
    workload = S3_WORKLOAD if (args.s3_layers, args.s3_d) == (S3_LAYERS, S3_D) else \
        S3_WORKLOAD.replace("32-layer d=4096", layers).replace("(%d params)" % S3_N_PARAMS, "(%d params)" % n)
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "io_dtype": "fp16", "data": "synthetic",
        "config": {"workload": workload, "n_params": n, "n_ranks": job.N, "stage": 3, "bucket_elems": job.B,
                   "n_layers": len(job.layers), "gather_capacity_elems": job.plan.max_layer_elems,
                   "loss_scale": job.S, "parallelism": "replicas only (simulated ranks inside each GPU)",
                   "gradients": "each bucket's %d gradient copies read from a ring of %d pre-generated bucket-sized "
                                "gradient sets in HBM (bucket b reads set b mod %d; %.1f GB); generated before the "
                                "timed region, so no generation is inside a step" % (
                                    job.N, len(job.ring), len(job.ring), len(job.ring) * job.N * job.B * 2 / 1e9),
                   "l2": "inputs larger than L2: %.0f GB moved per step; each gradient set 2.1 GB"
                         % (step_bytes / 1e9)},
        "hbm_gbs_step": step_bytes / (ms_per_step * 1e-3) / 1e9,
        "step_roofline": {"bytes_per_param": job.bytes_per_param(), "bytes_per_step": step_bytes,
                          "achieved": step_bytes / (ms_per_step * 1e-3) / 1e9, "peak": peak,
                          "frac": step_bytes / (ms_per_step * 1e-3) / 1e9 / peak,
                          "frac_of_chip_nominal": step_bytes / (ms_per_step * 1e-3) / 1e9 / CHIP_HBM_GBS},
        "roofline": {"bound": "hbm", "kernel": "k_gather (stage-3 layer all-gather, 64 destinations)",
                     "achieved": g_ach, "peak": peak, "peak_kind": peak_kind, "unit": "GB/s", "frac": g_ach / peak,
                     "traffic": g_traffic,
                     "traffic_source": traffic_source(GATHER_SUMMARY, GATHER_SOURCES) if g_traffic else None,
                     "algorithmic_bytes_per_launch": g_launch, "bytes_per_element": 2 + 2 * job.N,
                     "launches": n_prof * n_gathers, "avg_launch_ms": g_ms / (n_prof * n_gathers),
                     "share_of_step_bytes": 2 * (2 + 2 * job.N) / job.bytes_per_param(),
                     "frac_of_chip_nominal": g_ach / CHIP_HBM_GBS, "chip_nominal_gbs": CHIP_HBM_GBS,
                     "chip_nominal_source": CHIP_HBM_SOURCE,
                     "timing": "CUDA events recorded on the step's stream between consecutive library calls on "
                               "every %dth timed step (%d of %d); each gather interval holds one gather kernel, each "
                               "run interval one layer's bucket kernels" % (PROFILE_EVERY, n_prof, args.steps)},
        "kernels": {"k_fused<stage 3, fp16, adam>": {
            "achieved": f_ach, "frac": f_ach / peak, "bytes_per_param": bench_bytes(3, job.N),
            "launches": n_prof * job.plan.n_buckets, "avg_launch_ms": b_ms / (n_prof * job.plan.n_buckets),
            "algorithmic_bytes_per_launch": f_bytes / (n_prof * job.plan.n_buckets)}},
        "gpu_launches": args.steps * job.launches_per_step(),
        "step_api": "zero_step_begin_async / zero_gather_layer / zero_step_buckets_async (one run of buckets per "
                    "layer) / zero_step_end_async (step state in device memory, steps enqueued back to back)",
    }
    out["clocks"] = clocks_summary(rows, t0, t1)
    if args.headline_only:
        if rank == 0:
            print(json.dumps(out))
        return _finish(world)
    # end to end on every rank at once: each GPU has its own host link
    try:
        out["e2e"] = stage3_e2e(job, args.e2e_steps, 1, device, world, args.e2e_mode)
    except Exception as e:         # reported, never hides the headline
        if world > 1:
            raise
        out["e2e"] = {"error": repr(e)}
    del job
    torch.cuda.empty_cache()
    if rank == 0:
        # the gather writes 64 of every 65 bytes it moves: beside the copy
        # bandwidth (half read, half written), the write-only ceiling
        w = bw.write_ceiling_gbs()
        out["roofline"]["write_only_ceiling"] = {
            "gbs": w, "frac": g_ach / w,
            "how": "torch fill_ of one 8 GiB fp32 buffer on this GPU after the timed steps, median of 5"}
        out["legs"] = other_legs(args, device)
        if world == 1:
            out["cpu_baseline"] = cpu_baseline()
        print(json.dumps(out))
    barrier(world)
    return _finish(world)


def bench_bytes(stage, n_ranks):
    return bytes_per_param(stage, n_ranks)


def _finish(world):
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def other_legs(args, device):
    """The stage-2 step on the 12-layer d=768 list (N_d = 8) and the clipped
    stage-2 steps at 2^31 parameters (N_d = 2 and 32, bf16), each with its
    own roofline; reported beside the headline, never hiding it."""
    import torch

    import bench_workloads as bw
    legs = {}
    try:
        job = GpuJob(2, device, ring=GRAD_RING)
        k = max(10, args.steps)
        ms, launches, kernel, _ = timed_steps(job, k, args.warmup, 1, api="async")
        peak, kind = measured_peak_hbm()
        ach = kernel["bytes"] / (kernel["total_ms"] * 1e-3) / 1e9
        tr = profiled_traffic()
        legs["workload2_stage2"] = {
            "workload": WORKLOAD, "n_params": N_PARAMS, "steps": k, "ms_per_step": ms / k,
            "value": N_PARAMS / (ms / k * 1e-3) / 1e9,
            "roofline": {"bound": "hbm", "kernel": "k_fused<stage 2, fp16, adam>", "achieved": ach, "peak": peak,
                         "peak_kind": kind, "unit": "GB/s", "frac": ach / peak,
                         "traffic": None if tr is None else tr * (N_PARAMS / job.plan.n_buckets) / (1 << 24),
                         "traffic_source": traffic_source(PROFILE_SUMMARY, KERNEL_SOURCES) if tr else None,
                         "bytes_per_param": bytes_per_param(2), "launches": kernel["launches"],
                         "avg_launch_ms": kernel["total_ms"] / kernel["launches"],
                         "timing": "library-recorded events around a step's bucket kernels (kernel span) on every "
                                   "%dth step" % PROFILE_EVERY}}
        del job
    except Exception as e:
        legs["workload2_stage2"] = {"error": repr(e)}
    torch.cuda.empty_cache()
    peak, kind = measured_peak_hbm()
    for n_ranks, dt in ((2, "bf16"), (32, "bf16")):
        name = "clip_2p31_n%d_%s" % (n_ranks, dt)
        try:
            r = bw.sweep_point(1 << 31, n_ranks, dt, max(2, min(args.steps, 4)), 1)
            r["roofline"] = {"bound": "hbm", "kernel": "k_reduce + k_finalize + k_update (two-pass, clipping)",
                             "achieved": r["hbm_gbs"], "peak": peak, "peak_kind": kind, "unit": "GB/s",
                             "frac": r["hbm_gbs"] / peak, "traffic": None,
                             "timing": "whole clipped step (CUDA events); generation of staged gradients "
                                       "subtracted where gradients are staged"}
            legs[name] = r
        except Exception as e:
            legs[name] = {"error": repr(e)}
        torch.cuda.empty_cache()
    return legs


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--n-params", type=int, default=None,
                    help="flat parameter vector of this size instead of the transformer list (smaller cases, "
                         "e.g. for profiling captures)")
    ap.add_argument("--ring", type=int, default=GRAD_RING, help="distinct per-step gradient sets kept in HBM")
    ap.add_argument("--bucket", type=int, default=BUCKET, help="gradient bucket size in elements")
    ap.add_argument("--config", type=int, default=4, choices=[1, 2, 3, 4, 5, 6, 7, 8, 9],
                    help="workload: 4 (default) the stage-3 step at 6.65B parameters; 2 the stage-2 step on the "
                         "12-layer d=768 list (the options --stage, --optimizer, --dtype, --step-api, --n-params "
                         "apply to it); 1, 3, 5 the others, 6 the optimizer state in host memory, 7 the P_a "
                         "activation-checkpoint partition and all-gather, 8 stage-3 layer gathers alone, 9 the "
                         "clipped step split into its passes (bench_workloads.py)")
    ap.add_argument("--ring3", type=int, default=4, help="--config 4: pre-generated bucket gradient sets in HBM")
    ap.add_argument("--s3-layers", type=int, default=S3_LAYERS, help="--config 4: transformer layers")
    ap.add_argument("--s3-d", type=int, default=S3_D, help="--config 4: model width d")
    ap.add_argument("--e2e-steps", type=int, default=2, help="--config 4: timed steps of the end-to-end leg")
    ap.add_argument("--e2e-mode", default="direct", choices=["direct", "copy"],
                    help="--config 4: gradients read by the kernels from pinned host memory, or copied per bucket")
    ap.add_argument("--with-generation", action="store_true",
                    help="--config 4: instead, the step with each bucket's gradients generated into a staging "
                         "area right before its kernel (generation timed and subtracted), and the prefetching "
                         "fetcher run")
    ap.add_argument("--layer-elems", type=int, default=1 << 24, help="--config 8: elements per layer")
    ap.add_argument("--n-layers", type=int, default=2, help="--config 8: layers")
    ap.add_argument("--ranks", type=int, default=None, help="--config 5, 9: N_d of a single point; --config 8: N_d")
    ap.add_argument("--optimizer", default="adam", choices=sorted(OPTIMIZERS),
                    help="optimizer of the headline step (with --headline-only)")
    ap.add_argument("--dtype", default=None, choices=["fp16", "bf16", "fp32"],
                    help="--config 5: dtype of a single point (fp16/bf16); --config 2 with --headline-only: the "
                         "value type of the headline step (fp32: fp32 training)")
    ap.add_argument("--step-api", default="async", choices=["async", "sync"],
                    help="entry point of the timed steps: zero_step_async (default) or the synchronising "
                         "zero_step_stage2")
    ap.add_argument("--headline-only", action="store_true",
                    help="time the workload's step only (no other legs, end-to-end or CPU legs)")
    ap.add_argument("--stage", type=int, default=2, choices=[0, 1, 2, 3],
                    help="ZeRO stage of the timed step (other than 2: with --headline-only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.stage != 2 and not (args.headline_only and args.config == 2):
        ap.error("--stage other than 2 needs --config 2 --headline-only")
    if args.stage in (0, 1) and args.ring < args.steps + args.warmup:
        ap.error("stages 0 and 1 write the all-reduced gradient back into every rank's buffer: give each step "
                 "a gradient set of its own (--ring >= steps + warmup)")
    if args.impl == "reference":
        return reference_arm(args)
    if args.config == 4 and not args.with_generation:
        return stage3_arm(args)
    if args.config != 2:
        import torch

        import __graft_entry__
        import bench_workloads
        __graft_entry__.build()
        torch.cuda.set_device(0)
        print(json.dumps(bench_workloads.LEGS[args.config](args)))
        return 0
    return gpu_arm(args)


if __name__ == "__main__":
    sys.exit(main())
