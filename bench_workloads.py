"""The other workloads of the ZeRO step, run by ``bench.py --config K``.

  1  stage 2, flat 2^20 parameters, N_d = 4, grads N(0,1e-3) x 1024 loss
     scale (static), one bucket; L2-resident, so L2 is flushed between steps.
  3  stage 2, 48-layer d=1600 parameter list (1,555,278,400 params), N_d = 8,
     constant 5e8-element bucket, fp16 grads N(0,1e-3) x S with one +inf per
     1e9 gradient elements, dynamic loss scale (halve and skip), S0 = 1024.
     Two runs: the literal injection (every step overflows) and a companion
     run with injection on odd steps only.
  4  stage 3, 32-layer d=4096 parameter list (6,648,827,904 params), N_d = 64,
     bucket 2^24: per step every layer is gathered into 64 constant-size
     buffers for the forward and again for the backward, and each bucket's 64
     gradient copies are generated into a staging area right before its
     kernel (generation time is excluded).
  5  stage 2 sweep, flat 2^20 .. 2^31 parameters, N_d in {2, 8, 32}, fp16 or
     bf16 grads N(0,1e-3), bias correction, global-norm clipping at 1.0
     (two-pass path); gradients resident in HBM when all ranks' gradients
     and parameters fit in 160 GB, else generated per bucket (excluded).
  6  the headline workload with the fp32 optimizer state in pinned host
     (Grace) memory, updated by the fused kernel over NVLink-C2C.

Each leg prints one JSON line with the same keys as the headline.  Times are
CUDA events on the step's stream; input generation on the same stream is
bracketed by its own events and subtracted.
"""
from __future__ import annotations

import bench

ADAM = bench.ADAM


def transformer_layers(vocab, d, layers):
    return [vocab * d] + [12 * d * d + 4 * d] * layers


def _ev():
    import torch
    return torch.cuda.Event(enable_timing=True)


def _base(metric_value, ms_per_step, steps, warmup, workload, extra_config, dtype="f32"):
    return {"metric": bench.METRIC, "value": metric_value, "unit": bench.UNIT, "n_gpus": 1, "steps": steps,
            "warmup": warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": dtype, "data": "synthetic",
            "config": dict({"workload": workload}, **extra_config)}


def _roofline(bytes_per_step, kernel_ms_per_step, kernel_name):
    peak, kind = bench.measured_peak_hbm()
    achieved = bytes_per_step / (kernel_ms_per_step * 1e-3) / 1e9
    return {"bound": "hbm", "kernel": kernel_name, "achieved": achieved, "peak": peak, "peak_kind": kind,
            "unit": "GB/s", "frac": achieved / peak, "traffic": None, "algorithmic_bytes_per_step": bytes_per_step}


class StagedGrads:
    """Per-bucket gradient staging: N buffers of one bucket each, filled by
    the device generator right before the bucket's kernel, on the step's
    stream, between a pair of events (so the fill can be subtracted)."""

    def __init__(self, n_ranks, bucket, dtype, device):
        import torch
        self.bufs = [torch.empty(bucket, dtype=torch.int16, device=device) for _ in range(n_ranks)]
        self.ptrs = [b.data_ptr() for b in self.bufs]
        self.dtype = dtype
        self.events = []

    def fill(self, lo, hi, sigma, seed, step, stream, inject=()):
        import synth
        e0, e1 = _ev(), _ev()
        e0.record(stream)
        for r, b in enumerate(self.bufs):
            synth.dev_normal16(b.data_ptr(), hi - lo, self.dtype, sigma, seed=seed, stream=synth.STREAM_GRAD,
                               step=step, rank=r, offset=lo, cuda_stream=stream.cuda_stream)
        for r, e in inject:
            if lo <= e < hi:
                self.bufs[r][e - lo] = synth.inf_bits(self.dtype)      # 0x7C00 / 0x7F80 fit int16
        e1.record(stream)
        self.events.append((e0, e1))

    def take_ms(self):
        ms = sum(a.elapsed_time(b) for a, b in self.events)
        self.events = []
        return ms


def write_ceiling_gbs(nbytes=8 << 30, reps=5):
    """GB/s of a write-only stream on this GPU: a fill of one fp32 buffer of
    `nbytes` (median of `reps`).  The measured copy bandwidth moves half its
    bytes each way; a kernel that mostly writes (the stage-3 gather writes
    64 bytes for every one it reads) is bounded by this instead."""
    import torch
    dev = torch.device("cuda", 0)
    s = torch.cuda.current_stream(dev)
    buf = torch.empty(nbytes // 4, dtype=torch.float32, device=dev)
    buf.fill_(0.0)
    torch.cuda.synchronize()
    times = []
    for k in range(reps):
        e0, e1 = _ev(), _ev()
        e0.record(s)
        buf.fill_(float(k + 1))
        e1.record(s)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    times.sort()
    del buf
    torch.cuda.empty_cache()
    return nbytes / (times[len(times) // 2] * 1e-3) / 1e9


def copy_ceiling(nbytes, reps=20, flush=None, graph=False):
    """Milliseconds of one device copy moving `nbytes` in all (nbytes/2 read,
    nbytes/2 written) -- the floor of any kernel with that traffic, measured
    the way the step beside it is: back to back (one pair of events around
    `reps` copies), or, given a flush buffer, one copy per flush with events
    around the copy alone; graph=True replays the copy from a captured CUDA
    graph, as the step it is compared with is."""
    import torch
    dev = torch.device("cuda", 0)
    s = torch.cuda.current_stream(dev)
    half = max(16, (nbytes // 2) // 16 * 16)
    src = torch.empty(half, dtype=torch.uint8, device=dev)
    dst = torch.empty(half, dtype=torch.uint8, device=dev)
    src.fill_(1)
    run = lambda: dst.copy_(src)
    if graph:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(dev)
        cap.wait_stream(s)
        with torch.cuda.graph(g, stream=cap):
            dst.copy_(src)
        s.wait_stream(cap)
        run = g.replay
    for _ in range(3):
        run()
    torch.cuda.synchronize()
    if flush is None:
        e0, e1 = _ev(), _ev()
        e0.record(s)
        for _ in range(reps):
            run()
        e1.record(s)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / reps
    times = []
    for k in range(reps):
        flush.fill_(k & 0xff)
        e0, e1 = _ev(), _ev()
        e0.record(s)
        run()
        e1.record(s)
        torch.cuda.synchronize()
        times.append(e0.elapsed_time(e1))
    return sum(times) / reps


# ---------------------------------------------------------------------------
class Stage3Job:
    """ZeRO stage 3 on a transformer parameter list (default: 32 layers,
    d = 4096, 6,648,827,904 parameters), N_d = 64 simulated ranks, bucket
    2^24, fp16 gradients N(0, 1e-3) x 1024 (static loss scale 1024), Adam,
    step state in device memory.

    One step, as a stage-3 data-parallel step runs it: the forward pass
    gathers every layer's 16-bit parameters from the owners' shards into 64
    constant-size buffers (one per rank, each the size of the largest
    layer); the backward pass, in reverse layer order, gathers the layer
    again, then reduces, updates and writes back to the owners' shards every
    bucket whose lowest element lies in that layer.  Each bucket's 64
    gradient copies come from a ring of `ring` bucket-sized gradient sets
    generated in HBM when the job is built (bucket b reads set b mod ring):
    no input is generated inside a step, and every set (N_d x 2^24 x 2 B =
    2.1 GB) is far larger than L2.  Set k holds the generator's gradients of
    step k+1 at offsets 0..2^24 of each rank's stream."""

    def __init__(self, device, ring=4, n_layers=32, d=4096, vocab=50257, ranks=64, bucket=1 << 24, scale=1024.0):
        import torch

        import synth
        import zero_sharded_mixed_bucket_gb300 as zg
        self.zg, self.torch = zg, torch
        self.layers = transformer_layers(vocab, d, n_layers)
        self.n = sum(self.layers)
        self.N, self.B, self.S = ranks, bucket, scale
        self.cfg = zg.Config(self.n, ranks, 3, bucket, 0, self.layers)
        self.plan = zg.zero_plan(self.cfg)
        self.bufs = zg.DeviceBuffers(self.cfg, self.plan, device=device, grads=False, reduced=False)
        self.stream = torch.cuda.current_stream(device)
        s = self.stream.cuda_stream
        synth.dev_normal32(self.bufs.w[0].data_ptr(), self.n, 0.02, seed=0, stream=synth.STREAM_WEIGHT, cuda_stream=s)
        self.ring = [torch.empty(ranks * bucket, dtype=torch.int16, device=device) for _ in range(ring)]
        for k, t in enumerate(self.ring):
            for r in range(ranks):
                synth.dev_normal16(t.data_ptr() + 2 * r * bucket, bucket, synth.FP16, bench.SIGMA * scale, seed=0,
                                   stream=synth.STREAM_GRAD, step=k + 1, rank=r, cuda_stream=s)
        self.ring_ptrs = [zg.ptr_array([t.data_ptr() + 2 * r * bucket for r in range(ranks)]) for t in self.ring]
        self.dst = [torch.empty(self.plan.max_layer_elems, dtype=torch.int16, device=device) for _ in range(ranks)]
        self.dst_ptrs = zg.ptr_array([t.data_ptr() for t in self.dst])
        self.shard_ptrs = zg.ptr_array([t.data_ptr() for t in self.bufs.params16])
        self.adam = zg.zero_adam_t(max_grad_norm=0.0, **ADAM)
        self.state = zg.zero_state_t(t=0, loss_scale=scale, min_loss_scale=1.0)
        self.dev_state = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device=device)
        zg.zero_dev_state_init(self.dev_state, self.adam, self.state, self.stream)
        starts = [0]
        for ln in self.layers:
            starts.append(starts[-1] + ln)
        self.starts = starts
        # the step's library calls in order: forward gathers, then per layer
        # (reversed) its gather and one run of the buckets that start inside it
        sched = [("gather", l) for l in range(len(self.layers))]
        nxt = self.plan.n_buckets - 1
        for l in reversed(range(len(self.layers))):
            sched.append(("gather", l))
            run = []
            while nxt >= 0 and nxt * bucket >= starts[l]:
                run.append(nxt)
                nxt -= 1
            if run:
                sched.append(("buckets", run))
        assert nxt == -1
        self.schedule = sched
        self.n_bucket_kernels = self.plan.n_buckets
        self._runs = {}           # run index -> (indices, flat gradient pointers) for the ring
        for k, (kind, x) in enumerate(sched):
            if kind == "buckets":
                self._runs[k] = self._run_arrays(x, lambda b: self.ring_ptrs[b % len(self.ring_ptrs)])
        torch.cuda.synchronize(device)

    def _run_arrays(self, run, grad_ptrs):
        import ctypes
        idx = (ctypes.c_int64 * len(run))(*run)
        flat = self.zg.ptr_array([p for b in run for p in list(grad_ptrs(b))])
        return idx, flat

    def bucket_len(self, b):
        lo = b * self.B
        return min(lo + self.B, self.n) - lo

    def bytes_per_param(self):
        """Algorithmic HBM bytes per parameter of one step: two gathers (the
        shard read once, 64 destinations written: 2 + 2 N_d each) and the
        fused stage-3 update (N_d gradient reads, 12 B of state read and
        written, the owner's 16-bit parameter written: 2 N_d + 24 + 2)."""
        return 2 * (2 + 2 * self.N) + bench.bytes_per_param(3, self.N)

    def launches_per_step(self):
        # prepare, the gathers, the bucket kernels, restore/commit
        return 2 + sum(1 for kind, _ in self.schedule if kind == "gather") + self.n_bucket_kernels

    def step(self, events=None, grad_ptrs=None, before_bucket=None, after_bucket=None):
        """Enqueue one step on the job's stream; never synchronises.
        events: None, or len(schedule)+1 CUDA events recorded between the
        library calls (event k before schedule entry k).  grad_ptrs(b): the
        64 gradient pointers of bucket b (default: ring set b mod ring).
        Each layer's buckets go to the library as one run
        (zero_step_buckets_async: consecutive kernels overlap their edges),
        unless before_bucket(b) / after_bucket(b) stream hooks are given
        (end-to-end copies): then one call per bucket, in plain stream order."""
        zg, s = self.zg, self.stream
        zg.zero_step_begin_async(self.cfg, self.plan, self.bufs, self.adam, self.dev_state, s)
        for k, (kind, x) in enumerate(self.schedule):
            if events is not None:
                events[k].record(s)
            if kind == "gather":
                zg.zero_gather_layer(self.cfg, self.plan, x, self.shard_ptrs, self.dst_ptrs, s)
            elif before_bucket or after_bucket:
                for b in x:
                    if before_bucket:
                        before_bucket(b)
                    ptrs = grad_ptrs(b) if grad_ptrs else self.ring_ptrs[b % len(self.ring_ptrs)]
                    zg.zero_step_bucket_async(self.cfg, self.plan, self.bufs, self.adam, b, ptrs, s)
                    if after_bucket:
                        after_bucket(b)
            else:
                idx, flat = self._runs[k] if grad_ptrs is None else self._run_arrays(x, grad_ptrs)
                zg.zero_step_buckets_async(self.cfg, self.plan, self.bufs, self.adam, idx, flat, s)
        if events is not None:
            events[len(self.schedule)].record(s)
        zg.zero_step_end_async(self.cfg, self.plan, self.bufs, self.adam, self.dev_state, s)

    def kernel_times(self, events):
        """(gather ms, bucket ms) of one profiled step from its events."""
        g = b = 0.0
        for k, (kind, _) in enumerate(self.schedule):
            ms = events[k].elapsed_time(events[k + 1])
            if kind == "gather":
                g += ms
            else:
                b += ms
        return g, b


# ---------------------------------------------------------------------------
def leg_cfg1(args):
    import torch

    import synth
    import zero_sharded_mixed_bucket_gb300 as zg
    n, N, S = 1 << 20, 4, 1024.0
    dev = torch.device("cuda", 0)
    cfg = zg.Config(n, N, 2, 1 << 24)
    plan = zg.zero_plan(cfg)
    bufs = zg.DeviceBuffers(cfg, plan, device=dev)
    s = torch.cuda.current_stream(dev)
    synth.dev_normal32(bufs.w[0].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT, cuda_stream=s.cuda_stream)
    for r in range(N):
        synth.dev_normal16(bufs.grads[r].data_ptr(), n, synth.FP16, 1e-3 * S, seed=0, stream=synth.STREAM_GRAD,
                           step=1, rank=r, cuda_stream=s.cuda_stream)
    adam = zg.zero_adam_t(max_grad_norm=0.0, **ADAM)
    state = zg.zero_state_t(t=0, loss_scale=S, min_loss_scale=1.0)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    e0, e1 = _ev(), _ev()
    e0.record(s)        # materialise the events (the library records them by handle)
    e1.record(s)
    zg.zero_set_profile_events(e0, e1)
    spans, walls = [], []
    try:
        for k in range(args.warmup + args.steps):
            flush.fill_(k & 0xff)                      # evict the step's working set from L2
            w0, w1 = _ev(), _ev()
            w0.record(s)
            res = zg.zero_step_stage2(cfg, plan, bufs, adam, state, s)
            w1.record(s)
            torch.cuda.synchronize()
            if k >= args.warmup:
                spans.append(e0.elapsed_time(e1))
                walls.append(w0.elapsed_time(w1))
            assert res.overflow == 0
    finally:
        zg.zero_set_profile_events(None, None)
    ms_sync = sum(walls) / len(walls)
    # the same step with the step state on the device, replayed from two
    # captured CUDA graphs (one per state copy): no host round trip per step
    dev_state = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device=dev)
    zg.zero_dev_state_init(dev_state, adam, state, s)
    zg.zero_step_async(cfg, plan, bufs, adam, dev_state, s)       # warms the launch-shape cache
    torch.cuda.synchronize()
    graphs = []
    cap = torch.cuda.Stream(dev)
    for _ in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            zg.zero_step_async(cfg, plan, bufs, adam, dev_state, torch.cuda.current_stream(dev))
        graphs.append(g)
    gwalls = []
    for k in range(args.warmup + args.steps):
        flush.fill_(k & 0xff)
        w0, w1 = _ev(), _ev()
        w0.record(s)
        graphs[k % 2].replay()
        w1.record(s)
        torch.cuda.synchronize()
        if k >= args.warmup:
            gwalls.append(w0.elapsed_time(w1))
    st, last = zg.zero_dev_state_read(dev_state, s)
    assert last.overflow == 0 and st.t == state.t + 1 + args.warmup + args.steps
    ms_graph = sum(gwalls) / len(gwalls)
    ms = min(ms_sync, ms_graph)
    ceil_ms = copy_ceiling(plan.hbm_bytes_fused, reps=args.steps, flush=flush, graph=True)
    out = _base(n / (ms * 1e-3) / 1e9, ms, args.steps, args.warmup,
                "stage 2, flat 2^20 params, N_d=4, fp16 grads N(0,1e-3) x 1024 static loss scale, one bucket",
                {"n_params": n, "n_ranks": N, "stage": 2, "l2": "flushed before every step (256 MB write)"})
    out["modes"] = {"zero_step_stage2": {"ms_per_step": ms_sync, "value": n / (ms_sync * 1e-3) / 1e9},
                    "graph of zero_step_async": {"ms_per_step": ms_graph, "value": n / (ms_graph * 1e-3) / 1e9}}
    out["mode"] = "graph of zero_step_async" if ms_graph <= ms_sync else "zero_step_stage2"
    out["roofline"] = _roofline(plan.hbm_bytes_fused, sum(spans) / len(spans), "k_fused<stage 2, fp16>")
    out["copy_ceiling"] = {"ms": ceil_ms, "step_over_copy": ms / ceil_ms,
                           "note": "one device copy of the step's %d bytes (half read, half written), replayed from a "
                                   "CUDA graph after the same 256 MB flush" % plan.hbm_bytes_fused}
    out["note"] = "42 MB per step: launch latency dominates; a parity case, not a bandwidth one"
    return out


# ---------------------------------------------------------------------------
def leg_cfg3(args):
    import torch

    import synth
    import zero_sharded_mixed_bucket_gb300 as zg
    layers = transformer_layers(50257, 1600, 48)
    n, N, B = sum(layers), 8, 500_000_000
    dev = torch.device("cuda", 0)
    s = torch.cuda.current_stream(dev)
    cfg = zg.Config(n, N, 2, B, 0, layers)
    plan = zg.zero_plan(cfg)
    bufs = zg.DeviceBuffers(cfg, plan, device=dev)
    runs = {}
    steps = max(args.steps, 4)
    for run in ("literal", "odd_steps"):
        # both runs start from the same master weights (m = v = 0)
        synth.dev_normal32(bufs.w[bufs.cur].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT,
                           cuda_stream=s.cuda_stream)
        adam = zg.zero_adam_t(max_grad_norm=0.0, **ADAM)
        state = zg.zero_state_t(t=0, loss_scale=1024.0, min_loss_scale=1.0, dynamic=1, growth_interval=0)
        walls, skipped, scales, skipped_bytes, moved = [], 0, [], [], []
        for k in range(steps):
            step_no = k + 1
            S = state.loss_scale
            for r in range(N):
                synth.dev_normal16(bufs.grads[r].data_ptr(), n, synth.FP16, 1e-3 * S, seed=0,
                                   stream=synth.STREAM_GRAD, step=step_no, rank=r, cuda_stream=s.cuda_stream)
            if run == "literal" or step_no % 2 == 1:
                for r, e in synth.inf_positions(n, N, seed=0, step=step_no):
                    bufs.grads[r][e] = synth.inf_bits(synth.FP16)
            w0, w1 = _ev(), _ev()
            w0.record(s)
            res = zg.zero_step_stage2(cfg, plan, bufs, adam, state, s)
            w1.record(s)
            torch.cuda.synchronize()
            walls.append(w0.elapsed_time(w1))
            skipped += res.skipped
            scales.append(res.new_loss_scale)
            moved.append(res.hbm_bytes)
            if res.skipped:
                skipped_bytes.append(res.hbm_bytes)
        ms = sum(walls) / len(walls)
        runs[run] = {"ms_per_step": ms, "value": n / (ms * 1e-3) / 1e9, "steps": steps, "skipped": skipped,
                     "hbm_gbs": sum(moved) / (sum(walls) * 1e-3) / 1e9,
                     "loss_scales": scales, "t": state.t,
                     "hbm_bytes_per_clean_step": plan.hbm_bytes_fused,
                     "hbm_bytes_per_skipped_step": (sum(skipped_bytes) / len(skipped_bytes)) if skipped_bytes
                     else None,
                     "hbm_bytes_per_skipped_step_without_skipping": plan.hbm_bytes_fused + n * (4 + 2 * N)}
    main = runs["odd_steps"]
    out = _base(main["value"], main["ms_per_step"], steps, 0,
                "stage 2, 48-layer d=1600 parameter list (%d params), N_d=8, bucket 5e8, fp16 grads N(0,1e-3) x S, "
                "one +inf per 1e9 gradient elements, dynamic loss scale (halve and skip), S0=1024" % n,
                {"n_params": n, "n_ranks": N, "stage": 2, "bucket_elems": B, "injection": "value: odd steps only; "
                 "runs.literal: every step (12 infs over 1.24e10 gradient elements)"})
    out["runs"] = runs
    peak, kind = bench.measured_peak_hbm()
    out["roofline"] = {"bound": "hbm", "kernel": "k_fused<stage 2, fp16, adam> + k_restore (skipped steps)",
                       "achieved": main["hbm_gbs"], "peak": peak, "peak_kind": kind, "unit": "GB/s",
                       "frac": main["hbm_gbs"] / peak, "traffic": None,
                       "bytes": "the library's count of what each step moved (hbm_bytes), over the steps' time"}
    out["note"] = ("bucket kernels that start after the step's flag is raised do nothing; a skipped step then "
                   "restores the parameters of the window the other kernels wrote (cast of the unchanged master "
                   "weights to every rank); hbm_bytes_per_skipped_step is the library's count of what moved; step "
                   "times are CUDA events around the whole library call")
    return out


# ---------------------------------------------------------------------------
def leg_cfg4(args):
    """Stage 3 at 6.65B parameters, N_d = 64.  Two runs: (a) every gather on
    the step's stream into 64 constant-size buffers of the largest layer;
    (b) a fetcher prefetching one layer ahead on a side stream into a pool of
    two largest layers (the live-parameter budget)."""
    import torch

    import synth
    import zero_sharded_mixed_bucket_gb300 as zg
    layers = transformer_layers(50257, 4096, 32)
    n, N, B = sum(layers), 64, 1 << 24
    dev = torch.device("cuda", 0)
    s = torch.cuda.current_stream(dev)
    cfg = zg.Config(n, N, 3, B, 0, layers)
    plan = zg.zero_plan(cfg)
    bufs = zg.DeviceBuffers(cfg, plan, device=dev, grads=False, reduced=False)
    S = 1024.0
    synth.dev_normal32(bufs.w[0].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT, cuda_stream=s.cuda_stream)
    staging = StagedGrads(N, B, synth.FP16, dev)
    shard_ptrs = [t.data_ptr() for t in bufs.params16]
    adam = zg.zero_adam_t(max_grad_norm=0.0, **ADAM)
    state = zg.zero_state_t(t=0, loss_scale=S, min_loss_scale=1.0)
    starts = [0]
    for l in layers:
        starts.append(starts[-1] + l)
    nb = plan.n_buckets
    L = len(layers)

    def run_buckets(layer, step_no, done):
        while done[0] > 0 and (done[0] - 1) * B >= starts[layer]:
            b = done[0] - 1
            lo, hi = b * B, min((b + 1) * B, n)
            staging.fill(lo, hi, 1e-3 * S, 0, step_no, s)
            zg.zero_step_bucket(cfg, plan, bufs, adam, state, b, staging.ptrs, s)
            done[0] -= 1

    def step_plain(step_no, dst_ptrs):
        zg.zero_step_begin(cfg, plan, bufs, adam, state, s)
        for l in range(L):
            zg.zero_gather_layer(cfg, plan, l, shard_ptrs, dst_ptrs, s)
        done = [nb]
        for l in reversed(range(L)):
            zg.zero_gather_layer(cfg, plan, l, shard_ptrs, dst_ptrs, s)
            run_buckets(l, step_no, done)
        return zg.zero_step_end(cfg, plan, bufs, adam, state, s)

    def step_prefetch(step_no, pool, cap, side):
        zg.zero_step_begin(cfg, plan, bufs, adam, state, s)
        f = zg.Fetcher(cfg, plan, shard_ptrs, pool, cap, list(range(L)), 1, side)
        for pos in range(L):
            f.fetch(pos, s)
            f.release(pos, s)
        f = zg.Fetcher(cfg, plan, shard_ptrs, pool, cap, list(reversed(range(L))), 1, side)
        done = [nb]
        for pos, l in enumerate(reversed(range(L))):
            f.fetch(pos, s)
            run_buckets(l, step_no, done)
            f.release(pos, s)
        return zg.zero_step_end(cfg, plan, bufs, adam, state, s)

    def timed(fn, steps, warm):
        for k in range(warm):
            fn(k + 1)
        torch.cuda.synchronize()
        staging.take_ms()
        walls, gens = [], []
        for k in range(steps):
            w0, w1 = _ev(), _ev()
            w0.record(s)
            res = fn(warm + k + 1)
            w1.record(s)
            torch.cuda.synchronize()
            assert res.overflow == 0
            walls.append(w0.elapsed_time(w1))
            gens.append(staging.take_ms())
        return sum(w - g for w, g in zip(walls, gens)) / steps, sum(gens) / steps, sum(walls) / steps

    steps = max(1, min(args.steps, 3))
    dst = [torch.empty(plan.max_layer_elems, dtype=torch.int16, device=dev) for _ in range(N)]
    ms_plain, gen_ms, wall_plain = timed(lambda k: step_plain(k, [d.data_ptr() for d in dst]), steps, 1)
    del dst
    torch.cuda.empty_cache()
    cap = 2 * ((plan.max_layer_elems + 7) // 8 * 8)
    pool = [torch.empty(cap, dtype=torch.int16, device=dev) for _ in range(N)]
    side = torch.cuda.Stream(dev)
    ms_pf, _, wall_pf = timed(lambda k: step_prefetch(k, pool, cap, side), steps, 1)
    ms = ms_plain       # the prefetch run overlaps the excluded generation: reported, not the value
    bpp_gather = 2 + 2 * N
    bytes_step = n * (2 * bpp_gather + bench.bytes_per_param(3, N))
    out = _base(n / (ms * 1e-3) / 1e9, ms, steps, 1,
                "stage 3, 32-layer d=4096 parameter list (%d params), N_d=64, bucket 2^24; two gathers per layer "
                "for 64 destinations; 64 gradient copies generated per bucket (excluded)" % n,
                {"n_params": n, "n_ranks": N, "stage": 3, "bucket_elems": B, "n_layers": L,
                 "gather_capacity_elems": plan.max_layer_elems})
    out["runs"] = {"gathers_in_stream": {"ms_per_step": ms_plain, "value": n / (ms_plain * 1e-3) / 1e9,
                                         "ms_per_step_with_generation": wall_plain,
                                         "buffers": "64 x the largest layer"},
                   "prefetch_depth_1": {"ms_per_step": ms_pf, "value": n / (ms_pf * 1e-3) / 1e9,
                                        "ms_per_step_with_generation": wall_pf,
                                        "buffers": "pool of 64 x 2 largest layers (live budget)",
                                        "note": "gathers overlap the bucket kernels and the excluded gradient "
                                                "generation, so subtracting the generation time overstates "
                                                "this run's speed by up to the overlap; the times with the "
                                                "generation included compare the two runs like for like"}}
    out["roofline"] = _roofline(bytes_step, ms_plain, "k_gather + k_fused<stage 3, fp16> (gathers in stream)")
    out["bytes_per_param"] = 2 * bpp_gather + bench.bytes_per_param(3, N)
    out["generation_ms_per_step"] = gen_ms
    out["device_memory_gb"] = torch.cuda.max_memory_allocated(dev) / 1e9
    return out


# ---------------------------------------------------------------------------
SWEEP_DEFAULT = [(1 << 20, 8, "fp16"), (1 << 24, 8, "fp16"), (1 << 28, 2, "fp16"), (1 << 28, 8, "bf16"),
                 (1 << 28, 32, "fp16"), (1 << 31, 2, "bf16"), (1 << 31, 8, "fp16"), (1 << 31, 32, "bf16")]


def sweep_point(n, N, dtype_name, steps, warm):
    import torch

    import synth
    import zero_sharded_mixed_bucket_gb300 as zg
    dtype = zg.ZERO_BF16 if dtype_name == "bf16" else zg.ZERO_FP16
    B = 1 << 24
    dev = torch.device("cuda", 0)
    s = torch.cuda.current_stream(dev)
    cfg = zg.Config(n, N, 2, B, 0, None, dtype)
    plan = zg.zero_plan(cfg)
    resident = 2 * N * n * 2 <= 160e9          # all ranks' gradients and parameters in HBM
    bufs = zg.DeviceBuffers(cfg, plan, device=dev, grads=resident, shadow=False)
    synth.dev_normal32(bufs.w[0].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT, cuda_stream=s.cuda_stream)
    if resident:
        for r in range(N):
            synth.dev_normal16(bufs.grads[r].data_ptr(), n, dtype, 1e-3, seed=0, stream=synth.STREAM_GRAD, step=1,
                               rank=r, cuda_stream=s.cuda_stream)
    staging = None if resident else StagedGrads(N, min(B, n), dtype, dev)
    adam = zg.zero_adam_t(max_grad_norm=1.0, **ADAM)
    state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)

    def one_step(step_no):
        if resident:            # stage 2 leaves the gradients unchanged: the same set serves every step
            return zg.zero_step_stage2(cfg, plan, bufs, adam, state, s)
        zg.zero_step_begin(cfg, plan, bufs, adam, state, s)
        for b in range(plan.n_buckets):
            lo, hi = b * B, min((b + 1) * B, n)
            staging.fill(lo, hi, 1e-3, 0, step_no, s)
            zg.zero_step_bucket(cfg, plan, bufs, adam, state, b, staging.ptrs, s)
        return zg.zero_step_end(cfg, plan, bufs, adam, state, s)

    for k in range(warm):
        one_step(k + 1)
    if staging:
        staging.take_ms()
    walls, gens, norms = [], [], []
    for k in range(steps):
        w0, w1 = _ev(), _ev()
        w0.record(s)
        res = one_step(warm + k + 1)
        w1.record(s)
        torch.cuda.synchronize()
        walls.append(w0.elapsed_time(w1))
        gens.append(staging.take_ms() if staging else 0.0)
        norms.append(res.grad_norm)
        assert res.overflow == 0
    ms_sync = sum(w - g for w, g in zip(walls, gens)) / steps
    ms, api = ms_sync, "zero_step_stage2"
    if resident:
        # the same step with the step state on the device: steps enqueued back
        # to back, one pair of events around them all, the state read after
        dev_state = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device=dev)
        zg.zero_dev_state_init(dev_state, adam, state, s)
        zg.zero_step_async(cfg, plan, bufs, adam, dev_state, s)
        k_async = max(steps, 10)
        w0, w1 = _ev(), _ev()
        w0.record(s)
        for _ in range(k_async):
            zg.zero_step_async(cfg, plan, bufs, adam, dev_state, s)
        w1.record(s)
        torch.cuda.synchronize()
        st, last = zg.zero_dev_state_read(dev_state, s)
        assert st.t == state.t + 1 + k_async and last.overflow == 0
        assert last.grad_norm == norms[-1]          # the gradients, hence the norm, are the same every step
        ms_async = w0.elapsed_time(w1) / k_async
        if ms_async < ms:
            ms, api = ms_async, "zero_step_async"
        if n * (28 + 4 * N) <= 4 << 30:
            # a small step is bound by launches: the same step captured once in
            # a CUDA graph (the two-pass path keeps one state copy, so one
            # graph serves every step) and replayed back to back
            t_before = zg.zero_dev_state_read(dev_state, s)[0].t
            g = torch.cuda.CUDAGraph()
            cap = torch.cuda.Stream(dev)
            cap.wait_stream(s)
            with torch.cuda.graph(g, stream=cap):
                zg.zero_step_async(cfg, plan, bufs, adam, dev_state, torch.cuda.current_stream(dev))
            s.wait_stream(cap)
            for _ in range(3):
                g.replay()
            w0, w1 = _ev(), _ev()
            w0.record(s)
            for _ in range(k_async):
                g.replay()
            w1.record(s)
            torch.cuda.synchronize()
            st, last = zg.zero_dev_state_read(dev_state, s)
            assert st.t == t_before + 3 + k_async and last.overflow == 0 and last.grad_norm == norms[-1]
            ms_graph = w0.elapsed_time(w1) / k_async
            if ms_graph < ms:
                ms, api = ms_graph, "graph of zero_step_async"
    bpp = 28 + 4 * N
    out = {"n_params": n, "n_ranks": N, "dtype": dtype_name, "ms_per_step": ms, "value": n / (ms * 1e-3) / 1e9,
           "hbm_gbs": n * bpp / (ms * 1e-3) / 1e9, "bytes_per_param": bpp, "grad_norm": norms[-1],
           "clip_coef": res.clip_coef, "t": state.t, "step_api": api, "ms_per_step_sync": ms_sync,
           "gradients": "resident in HBM" if resident else "generated per bucket into staging (excluded)"}
    if resident and n * bpp <= 4 << 30:
        # the same bytes as one device copy, back to back like the steps above
        c = copy_ceiling(n * bpp, reps=20)
        out["copy_ceiling"] = {"ms": c, "step_over_copy": ms / c,
                               "note": "one device copy moving the step's %d bytes (half read, half written), "
                                       "timed back to back like the steps" % (n * bpp)}
    del bufs, staging
    torch.cuda.empty_cache()
    return out


def leg_cfg5(args):
    points = SWEEP_DEFAULT
    if args.n_params:
        points = [(args.n_params, args.ranks or 8, args.dtype or "fp16")]
    steps = max(1, min(args.steps, 3))
    res = [sweep_point(n, N, d, steps, 1) for n, N, d in points]
    peak, kind = bench.measured_peak_hbm()
    for r in res:
        r["frac"] = r["hbm_gbs"] / peak
    best = max(res, key=lambda r: r["n_params"] * 1000 + r["n_ranks"])
    out = _base(best["value"], best["ms_per_step"], steps, 1,
                "stage 2 sweep, flat 2^20..2^31 params, N_d in {2,8,32}, fp16/bf16 grads N(0,1e-3), clipping at 1.0, "
                "bias correction; gradients resident when they fit, else generated per bucket (excluded)",
                {"stage": 2, "bucket_elems": 1 << 24, "value_point": {k: best[k] for k in ("n_params", "n_ranks",
                                                                                            "dtype")}})
    out["points"] = res
    out["roofline"] = {"bound": "hbm", "kernel": "k_reduce + k_finalize + k_update (two-pass, clipping)",
                       "achieved": best["hbm_gbs"], "peak": peak, "peak_kind": kind, "unit": "GB/s",
                       "frac": best["hbm_gbs"] / peak, "traffic": None}
    return out


def leg_pass_split(args):
    """The clipped two-pass stage-2 step split into its passes by CUDA
    events: pass 1 (the buckets' reduce, flag and exact sum of squares, sent
    as one run through zero_step_buckets) and pass 2 (the norm finalize and
    the update kernels, up to the library's end event), each against its
    algorithmic bytes (pass 1: 2 N + 2 B per parameter; pass 2: 2 + 24 + 2 N
    B).  Points: --n-params/--ranks/--dtype, else 2^28 and 2^31 parameters,
    two ranks, fp16 and bf16."""
    import torch

    import synth
    import zero_sharded_mixed_bucket_gb300 as zg
    dev = torch.device("cuda", 0)
    s = torch.cuda.current_stream(dev)
    peak, kind = bench.measured_peak_hbm()
    if args.n_params:
        points = [(args.n_params, args.ranks or 2, args.dtype or "bf16")]
    else:
        points = [(1 << 28, 2, "fp16"), (1 << 28, 2, "bf16"), (1 << 31, 2, "bf16"), (1 << 31, 2, "fp16")]
    steps = max(args.steps, 3)
    res = []
    for n, N, dt in points:
        dtype = zg.ZERO_BF16 if dt == "bf16" else zg.ZERO_FP16
        cfg = zg.Config(n, N, 2, 1 << 24, 0, None, dtype)
        plan = zg.zero_plan(cfg)
        bufs = zg.DeviceBuffers(cfg, plan, device=dev, shadow=False)
        synth.dev_normal32(bufs.w[0].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT,
                           cuda_stream=s.cuda_stream)
        for r in range(N):
            synth.dev_normal16(bufs.grads[r].data_ptr(), n, dtype, 1e-3, seed=0, stream=synth.STREAM_GRAD, step=1,
                               rank=r, cuda_stream=s.cuda_stream)
        adam = zg.zero_adam_t(max_grad_norm=1.0, **ADAM)
        state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
        p1 = p2 = 0.0
        for k in range(args.warmup + steps):
            c0, c1, mid = _ev(), _ev(), _ev()
            c0.record(s)
            c1.record(s)            # materialised: the library records them by handle
            zg.zero_set_profile_events(c0, c1)    # c0 after the workspace clear, c1 after the update kernels
            try:
                zg.zero_step_begin(cfg, plan, bufs, adam, state, s)
                zg.zero_step_buckets(cfg, plan, bufs, adam, state, list(range(plan.n_buckets)), None, s)
                mid.record(s)
                zg.zero_step_end(cfg, plan, bufs, adam, state, s)
            finally:
                zg.zero_set_profile_events(None, None)
            torch.cuda.synchronize()
            if k >= args.warmup:
                p1 += c0.elapsed_time(mid)
                p2 += mid.elapsed_time(c1)
        p1 /= steps
        p2 /= steps
        b1, b2 = n * (2 * N + 2), n * (2 + 24 + 2 * N)
        res.append({"n_params": n, "n_ranks": N, "dtype": dt, "pass1_ms": p1, "pass1_frac": b1 / (p1 * 1e-3) / 1e9 / peak,
                    "pass2_ms": p2, "pass2_frac": b2 / (p2 * 1e-3) / 1e9 / peak, "step_ms": p1 + p2,
                    "step_frac": (b1 + b2) / ((p1 + p2) * 1e-3) / 1e9 / peak})
        del bufs
        torch.cuda.empty_cache()
    last = res[-1]
    out = _base(last["n_params"] / (last["step_ms"] * 1e-3) / 1e9, last["step_ms"], steps, args.warmup,
                "clipped stage-2 step split into its two passes (CUDA events), flat parameters, grads N(0,1e-3)",
                {"stage": 2, "bucket_elems": 1 << 24})
    out["points"] = res
    out["roofline"] = {"bound": "hbm", "kernel": "k_reduce_staged (pass 1) / k_finalize + k_update (pass 2)",
                       "achieved": last["step_frac"] * peak, "peak": peak, "peak_kind": kind, "unit": "GB/s",
                       "frac": last["step_frac"], "traffic": None}
    return out


# ---------------------------------------------------------------------------
def leg_offload(args):
    """The headline workload with the fp32 optimizer state (w, m, v and their
    shadow copies: 2 x 12 B per parameter) in pinned host memory; the fused
    kernel reads and writes it over NVLink-C2C, gradients and 16-bit
    parameters stay in HBM."""
    import ctypes

    import torch
    dev = torch.device("cuda", 0)
    job = bench.GpuJob(2, dev, ring=2)
    n = job.n
    keep = []
    for name in ("w", "m", "v"):
        for k in range(2):
            h = torch.zeros(job.plan.state_elems, dtype=torch.float32).pin_memory()
            h.copy_(getattr(job.bufs, name)[k].cpu())
            getattr(job.bufs.b, name)[k] = h.data_ptr()
            keep.append(h)
    for name in ("w", "m", "v"):
        setattr(job.bufs, name, None)
    torch.cuda.empty_cache()
    ms, launches, kernel, _ = bench.timed_steps(job, max(3, min(args.steps, 20)), args.warmup, 1)
    steps = max(3, min(args.steps, 20))
    ms_step = ms / steps
    out = _base(n / (ms_step * 1e-3) / 1e9, ms_step, steps, args.warmup,
                "headline workload (12-layer d=768 list, N_d=8, stage 2, bucket 2^24) with the fp32 optimizer "
                "state in pinned host memory", {"n_params": n, "n_ranks": 8, "stage": 2,
                                                "state_location": "pinned host memory (Grace), via NVLink-C2C"})
    out["host_link_bytes_per_step"] = n * 24
    out["host_link_gbs"] = n * 24 / (kernel["span_ms_per_step"] * 1e-3) / 1e9
    out["hbm_bytes_per_step"] = n * (4 * 8)
    out["gpu_launches"] = launches
    return out


# ---------------------------------------------------------------------------
def leg_pa(args):
    """P_a, partitioned activation checkpoints: one layer checkpoint of the
    1.5B GPT-2 example (batch 32, sequence 1024, hidden 1600; fp16), N_m = 16
    model-parallel ranks.  Partition (each rank keeps its 1/16 slice) and the
    all-gather that rebuilds the checkpoint in all 16 ranks' buffers, with
    the slices in HBM (P_a) and in pinned host memory (P_a+cpu)."""
    import torch

    import zero_sharded_mixed_bucket_gb300 as zg
    A, N = 32 * 1024 * 1600, 16
    dev = torch.device("cuda", 0)
    s = torch.cuda.current_stream(dev)
    p = zg.zero_pa_plan(A, N, zg.ZERO_FP16)
    x = torch.randint(-2 ** 15, 2 ** 15, (A,), dtype=torch.int16, device=dev)
    replicas = [x.clone() for _ in range(N)]          # model parallelism: the same checkpoint on every rank
    dst = [torch.empty(A, dtype=torch.int16, device=dev) for _ in range(N)]
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    steps = max(3, min(args.steps, 20))
    runs = {}
    for where in ("hbm", "host"):
        if where == "hbm":
            shards = [torch.empty(p.shard_elems, dtype=torch.int16, device=dev) for _ in range(N)]
        else:
            shards = [torch.empty(p.shard_elems, dtype=torch.int16).pin_memory() for _ in range(N)]
        tp, tg = [], []
        for k in range(args.warmup + steps):
            flush.fill_(k & 0xff)
            e0, e1, e2 = _ev(), _ev(), _ev()
            e0.record(s)
            zg.zero_pa_partition(p, replicas, shards, s)
            e1.record(s)
            flush.fill_((k + 1) & 0xff)
            e2.record(s)
            zg.zero_pa_gather(p, shards, dst, s)
            e3 = _ev()
            e3.record(s)
            torch.cuda.synchronize()
            if k >= args.warmup:
                tp.append(e0.elapsed_time(e1))
                tg.append(e2.elapsed_time(e3))
        assert torch.equal(dst[N - 1], x) and torch.equal(dst[0], x)
        ms_p, ms_g = sum(tp) / steps, sum(tg) / steps
        b = 2 * A
        runs["slices_in_" + where] = {
            "partition_ms": ms_p, "partition_gbs": 2 * b / (ms_p * 1e-3) / 1e9,
            "gather_ms": ms_g, "gather_gbs": (1 + N) * b / (ms_g * 1e-3) / 1e9,
            "note": "partition: each rank reads and writes its slice (2 x 2A bytes in all); gather: the slices "
                    "read once (2A bytes), the checkpoint written to 16 buffers (16 x 2A)"
                    + (" -- the slices cross the host link both ways" if where == "host" else "")}
        del shards
    hb = runs["slices_in_hbm"]
    # a copy of the all-gather's bytes after the same flush, for the ceiling
    hb["gather_copy_ceiling_ms"] = copy_ceiling((1 + N) * 2 * A, reps=steps, flush=flush)
    hb["gather_over_copy"] = hb["gather_ms"] / hb["gather_copy_ceiling_ms"]
    out = _base(A / (hb["gather_ms"] * 1e-3) / 1e9, hb["gather_ms"], steps, args.warmup,
                "P_a: one activation checkpoint of the 1.5B GPT-2 example (batch 32 x sequence 1024 x hidden 1600, "
                "fp16), N_m = 16 model-parallel ranks simulated; value = checkpoint values rebuilt per second by the "
                "all-gather into all 16 ranks",
                {"act_elems": A, "n_mp": N, "l2": "flushed before each partition and gather (256 MB write)"},
                dtype="u16")
    out["unit"] = "Gvalues/s"
    out["metric"] = "P_a all-gather: checkpoint values rebuilt per second (all 16 ranks)"
    out["runs"] = runs
    out["memory_per_rank_bytes"] = {"without_pa": p.mem_per_rank_bytes, "pa": p.mem_per_rank_pa_bytes,
                                    "pa_cpu_on_gpu": 0}
    out["gather_bytes_across_ranks"] = p.gather_bytes
    out["roofline"] = _roofline((1 + N) * 2 * A, hb["gather_ms"], "k_gather (chunk by chunk, destination by destination), P_a all-gather")
    return out


# ---------------------------------------------------------------------------
def leg_gather(args):
    """Stage-3 layer gathers alone: a model of --n-layers layers of
    --layer-elems elements each, N_d = 64 owner shards (--ranks: another
    N_d), every call gathering one layer (in turn) into N_d destination
    buffers.  The case the k_gather ncu summary captures (small enough for a
    profiler: 2 x 2^24 elements hold about 4.4 GB of device memory)."""
    import torch

    import zero_sharded_mixed_bucket_gb300 as zg
    N, le, nl = args.ranks or 64, args.layer_elems, args.n_layers
    layers = [le] * nl
    n = le * nl
    dev = torch.device("cuda", 0)
    s = torch.cuda.current_stream(dev)
    cfg = zg.Config(n, N, 3, 1 << 24, 0, layers)
    plan = zg.zero_plan(cfg)
    P = plan.shard_elems
    flat = torch.randint(-2 ** 15, 2 ** 15, (N * P,), dtype=torch.int16, device=dev)
    shards = [flat[r * P:(r + 1) * P] for r in range(N)]
    dst = [torch.empty(plan.max_layer_elems, dtype=torch.int16, device=dev) for _ in range(N)]
    sp = zg.ptr_array([t.data_ptr() for t in shards])
    dp = zg.ptr_array([t.data_ptr() for t in dst])
    steps = max(1, args.steps)
    times = []
    for k in range(args.warmup + steps):
        e0, e1 = _ev(), _ev()
        e0.record(s)
        zg.zero_gather_layer(cfg, plan, k % nl, sp, dp, s)
        e1.record(s)
        torch.cuda.synchronize()
        if k >= args.warmup:
            times.append(e0.elapsed_time(e1))
    last = (args.warmup + steps - 1) % nl
    assert torch.equal(dst[N - 1][:le], flat[last * le:(last + 1) * le])
    assert torch.equal(dst[0][:le], flat[last * le:(last + 1) * le])
    ms = sum(times) / steps
    bpe = 2 + 2 * N
    out = _base(le / (ms * 1e-3) / 1e9, ms, steps, args.warmup,
                "stage-3 layer gather alone: %d layers of %d elements, N_d=%d owner shards, %d destination buffers"
                % (nl, le, N, N), {"n_params": n, "n_ranks": N, "stage": 3, "layer_elems": le}, dtype="u16")
    out["unit"] = "Gelements/s"
    out["metric"] = "stage-3 layer gather: elements gathered per second into all %d destinations" % N
    out["roofline"] = _roofline(le * bpe, ms, "k_gather (chunk by chunk, destination by destination, %d destinations)"
                                % N)
    out["bytes_per_element"] = bpe
    out["l2"] = "each call writes %.1f GB: far larger than L2" % (le * 2 * N / 1e9)
    return out


LEGS = {1: leg_cfg1, 3: leg_cfg3, 4: leg_cfg4, 5: leg_cfg5, 6: leg_offload, 7: leg_pa, 8: leg_gather,
        9: leg_pass_split}
