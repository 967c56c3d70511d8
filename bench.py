"""Benchmark: ZeRO sharded mixed-precision Adam step on GB300.

Workload (default): the parameter list of a 12-layer d=768 transformer
(embedding 50257 x 768, per layer 4 d^2 attention + 8 d^2 MLP + 4 d
LayerNorm vectors: 123,568,896 parameters), N_d = 8 simulated data-parallel
ranks, ZeRO stage 2, gradient bucket 2^24 elements, fp16 gradients
N(0, 1e-3), loss scale 1, Adam (lr 1e-4, betas 0.9/0.999, eps 1e-8).  A
step is one pass of the whole hot path: every bucket's fused
reduce-scatter + overflow check + unscale + Adam + cast + all-gather kernel,
then the flag read and commit.  Stages 0 and 1 on the same workload are
timed after the headline and reported under "stages".

Output: one JSON line (rank 0).  `value` is parameters updated per second
over all GPUs with inputs resident in HBM; `e2e` is the same through the C
ABI with gradients arriving from pinned host memory every step; `roofline`
is the fused kernel's algorithmic bytes per launch over its CUDA-event
duration against the measured HBM copy bandwidth.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]

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
KERNEL_SOURCES = ["zero_sharded_mixed_bucket_gb300/csrc/k_fused.cu",
                  "zero_sharded_mixed_bucket_gb300/csrc/dev_common.cuh",
                  "zero_sharded_mixed_bucket_gb300/csrc/zero_internal.h"]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "k_fused_stage2_fp16_n8.md")


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
WORKLOAD = ("12-layer d=768 transformer parameter list (%d params), N_d=%d simulated ranks, ZeRO stage %d, "
            "bucket 2^24 elements, fp16 gradients N(0,1e-3), Adam" % (N_PARAMS, N_RANKS, STAGE))


# ---------------------------------------------------------------------------
# helpers
# ---------------------------------------------------------------------------
def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for p in KERNEL_SOURCES:
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


def profiled_traffic():
    """dram bytes per launch of the fused kernel from the committed ncu
    summary, if it was taken on the current kernel source (else None)."""
    try:
        text = open(PROFILE_SUMMARY, encoding="utf-8").read()
    except OSError:
        return None
    m_hash = re.search(r"kernel_source_hash:\s*([0-9a-f]+)", text)
    m_bytes = re.search(r"dram_bytes_per_full_launch:\s*([0-9.eE+]+)", text)
    if not m_hash or not m_bytes or m_hash.group(1) != kernel_source_hash():
        return None
    return float(m_bytes.group(1))


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
def oracle_sample_step(n_sample, seed_step):
    import numpy as np

    import oracle
    import synth
    grads = [synth.host_normal16(n_sample, synth.FP16, SIGMA, seed=0, stream=synth.STREAM_GRAD, step=seed_step,
                                 rank=r) for r in range(N_RANKS)]
    w = synth.host_normal32(n_sample, 0.02, seed=0, stream=synth.STREAM_WEIGHT)
    m = np.zeros(n_sample, np.float32)
    v = np.zeros(n_sample, np.float32)
    return grads, w, m, v


def run_oracle_steps(n_sample, steps, warmup):
    import oracle
    grads, w, m, v = oracle_sample_step(n_sample, 1)
    t = 0
    times = []
    for k in range(warmup + steps):
        t0 = time.perf_counter()
        r = oracle.step(grads, w, m, v, dtype=oracle.FP16, t=t, loss_scale=1.0, **ADAM)
        dt = time.perf_counter() - t0
        t = r["t"]
        if k >= warmup:
            times.append(dt)
    return times


def cpu_baseline(n_sample=1 << 26, steps=2):
    times = run_oracle_steps(n_sample, steps, 0)
    sec = sum(times) / len(times)
    return {"value": n_sample / sec / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": "%d contiguous parameters of the workload, N_d=%d ranks, %d steps, single-threaded C oracle "
                      "(unpartitioned step; stage 2 computes the same numbers)" % (n_sample, N_RANKS, steps),
            "seconds": sum(times)}


def reference_arm(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    n_sample = 1 << 22
    times = run_oracle_steps(n_sample, args.steps, args.warmup)
    sec = sum(times) / len(times)
    value = n_sample / sec / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": WORKLOAD, "n_params": N_PARAMS, "n_ranks": N_RANKS, "stage": STAGE,
                       "bucket_elems": BUCKET, "sample_params": n_sample},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "%d parameters of the workload per step, N_d=%d, single-threaded C oracle"
                                       % (n_sample, N_RANKS)},
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
                out["cpu_baseline"] = cpu_baseline()
            print(json.dumps(out))
        barrier(world)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=500)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--n-params", type=int, default=None,
                    help="flat parameter vector of this size instead of the transformer list (smaller cases, "
                         "e.g. for profiling captures)")
    ap.add_argument("--ring", type=int, default=GRAD_RING, help="distinct per-step gradient sets kept in HBM")
    ap.add_argument("--bucket", type=int, default=BUCKET, help="gradient bucket size in elements")
    ap.add_argument("--config", type=int, default=2, choices=[1, 2, 3, 4, 5, 6, 7],
                    help="workload: 2 (default) the headline; 1, 3, 4, 5 the others, 6 the optimizer state in host "
                         "memory, 7 the P_a activation-checkpoint partition and all-gather (bench_workloads.py)")
    ap.add_argument("--ranks", type=int, default=None, help="--config 5: N_d of a single sweep point")
    ap.add_argument("--optimizer", default="adam", choices=sorted(OPTIMIZERS),
                    help="optimizer of the headline step (with --headline-only)")
    ap.add_argument("--dtype", default=None, choices=["fp16", "bf16", "fp32"],
                    help="--config 5: dtype of a single point (fp16/bf16); --config 2 with --headline-only: the "
                         "value type of the headline step (fp32: fp32 training)")
    ap.add_argument("--step-api", default="async", choices=["async", "sync"],
                    help="entry point of the timed steps: zero_step_async (default) or the synchronising "
                         "zero_step_stage2")
    ap.add_argument("--headline-only", action="store_true",
                    help="time the stage-2 step only (no stage 0/1, end-to-end or CPU legs)")
    ap.add_argument("--stage", type=int, default=2, choices=[0, 1, 2, 3],
                    help="ZeRO stage of the timed step (other than 2: with --headline-only)")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("at least 3 warm-up steps")
    if args.stage != 2 and not args.headline_only:
        ap.error("--stage other than 2 needs --headline-only")
    if args.stage in (0, 1) and args.ring < args.steps + args.warmup:
        ap.error("stages 0 and 1 write the all-reduced gradient back into every rank's buffer: give each step "
                 "a gradient set of its own (--ring >= steps + warmup)")
    if args.impl == "reference":
        return reference_arm(args)
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
