"""Steps whose step state lives in device memory (zero_step_async): equal to
the oracle bit for bit across stages, paths, optimizers and 16-bit types,
through an overflowed step, loss-scale growth and a resumed step count; and
two CUDA graphs captured from it (one per value of the state-copy index)
replayed alternately with new gradients between replays."""
import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_mixed_bucket_gb300 as zg
from tests.gpu_harness import Job

pytestmark = pytest.mark.gpu


class AsyncJob(Job):
    def __init__(self, *args, shadow=True, t0=0, **kw):
        super().__init__(*args, shadow=shadow, **kw)
        if t0:
            self.state.t = t0
            self.o["t"] = t0
        self.dev = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device="cuda")
        zg.zero_dev_state_init(self.dev, self.adam, self.state, torch.cuda.current_stream())
        self.two_pass = self.max_norm > 0 or not shadow

    def launch(self, stream=None):
        return zg.zero_step_async(self.cfg, self.plan, self.bufs, self.adam, self.dev,
                                  stream or torch.cuda.current_stream())

    def read(self):
        st, res = zg.zero_dev_state_read(self.dev, torch.cuda.current_stream())
        assert res.path == -1
        res.path = 1 if self.two_pass else 0
        self.state = st
        return res

    def two_kernels(self):
        """The library's rule: a two-pass step (clipping, or no shadow state)
        of a model that is one bucket, in stages 2-3, whose gradients,
        reduced gradient, state and parameters (n x (2 N e + 2 e + 24) bytes)
        fit in 64 MiB, runs as two kernels."""
        e = 4 if self.dtype == oracle.FP32 else 2
        return (self.two_pass and self.plan.n_buckets == 1 and self.stage >= 2
                and self.n * (2 * self.N * e + 2 * e + 24) <= 64 << 20)

    def step(self, grads):
        self.load_grads(grads)
        n = self.launch()
        per_bucket = 2 if self.two_pass else 1
        # prepare, the bucket kernels (and the finalize and updates), then the
        # commit (joined with the restore on the fused path); or pass 1 and pass 2
        if self.two_kernels():
            assert n == 2
        else:
            assert n == 2 + per_bucket * self.plan.n_buckets + (1 if self.max_norm > 0 else 0)
        return self.read(), self.oracle_step(grads)


def inf_at(job, r, i):
    return (r, i, synth.inf_bits(job.dtype))


CASES = [
    # stage, N, n, B, dtype, shadow, max_norm, optimizer
    (2, 8, 5 * 1024 + 3, 1024, oracle.FP16, True, 0.0, zg.ZERO_ADAM),
    (2, 4, 5 * 1024 + 3, 1024, oracle.FP16, True, 1e-3, zg.ZERO_ADAM),
    (2, 4, 5 * 1024 + 3, 1024, oracle.BF16, False, 0.0, zg.ZERO_ADAM),
    (0, 3, 3 * 1024 + 5, 1024, oracle.FP16, True, 0.0, zg.ZERO_ADAM),
    (0, 3, 3 * 1024 + 5, 1024, oracle.BF16, False, 5e-3, zg.ZERO_ADAM),
    (1, 4, 4 * 512 + 9, 512, oracle.FP16, True, 0.0, zg.ZERO_SGD_MOMENTUM),
    (1, 4, 4 * 512 + 9, 512, oracle.FP16, False, 0.0, zg.ZERO_SGD),
    (3, 5, 7 * 256 + 1, 256, oracle.FP16, True, 0.0, zg.ZERO_SGD),
    (3, 5, 7 * 256 + 1, 256, oracle.BF16, True, 0.0, zg.ZERO_ADAM),
    (3, 5, 7 * 256 + 1, 256, oracle.FP16, True, 2e-3, zg.ZERO_SGD_MOMENTUM),
]


@pytest.mark.parametrize("case", CASES)
def test_async_steps_match_oracle(case):
    stage, N, n, B, dtype, shadow, max_norm, opt = case
    job = AsyncJob(n, N, stage, B, 8, None, dtype, shadow=shadow, loss_scale=256.0, dynamic=True, growth=2,
                   max_norm=max_norm, optimizer=opt)
    plan = [(), (), (inf_at(job, N - 1, n - 1),), (), (), (), (inf_at(job, 0, B + 1),), ()]
    for step, inject in enumerate(plan, start=1):
        res, ref = job.step(job.make_grads(step, inject))
        job.check(res, ref)
        assert res.overflow == (1 if inject else 0)
    # two overflows, two growth doublings (growth interval 2) from 256
    assert job.state.t == 6 and job.state.loss_scale == ref["loss_scale"]


def test_async_resumes_at_a_later_step_count():
    job = AsyncJob(3000, 4, 2, 1024, 8, None, oracle.FP16, t0=37, loss_scale=64.0)
    for step in (1, 2):
        res, ref = job.step(job.make_grads(step))
        job.check(res, ref)
    assert job.state.t == 39


def test_async_state_round_trip():
    dev = torch.zeros(8, dtype=torch.int64, device="cuda")
    adam = zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8)
    st = zg.zero_state_t(t=12, loss_scale=512.0, min_loss_scale=2.0, dynamic=1, growth_interval=7, good_steps=3)
    zg.zero_dev_state_init(dev, adam, st)
    got, last = zg.zero_dev_state_read(dev)
    assert (got.t, got.loss_scale, got.min_loss_scale, got.dynamic, got.growth_interval, got.good_steps) == \
        (12, 512.0, 2.0, 1, 7, 3)
    assert last.overflow == 0 and last.grad_norm == -1.0 and last.clip_coef == 1.0


@pytest.mark.parametrize("max_norm,N,B", [(0.0, 8, 2048), (1e-3, 8, 2048), (1e-3, 16, 2048), (0.0, 8, 1 << 16),
                                         (1e-3, 8, 1 << 16)])
def test_two_captured_graphs_replayed_alternately(max_norm, N, B):
    """(16 ranks, clipped: the update pass captured is the one that writes
    the parameters by bulk copies from shared-memory tiles.  One bucket of
    2^16: the model is a single bucket; clipped, the step captured is two
    kernels.)"""
    n = 6 * 2048 + 17
    job = AsyncJob(n, N, 2, B, 8, None, oracle.FP16, loss_scale=1024.0, dynamic=True, growth=3, max_norm=max_norm)
    s = torch.cuda.Stream()
    # one eager step first: it warms the library's launch-shape cache
    res, ref = job.step(job.make_grads(1))
    job.check(res, ref)
    graphs = []
    torch.cuda.synchronize()
    cur0 = job.bufs.cur
    for _ in range(2):                       # one graph per value of the copy index
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            job.launch(torch.cuda.current_stream())
        graphs.append(g)
    assert job.bufs.cur == cur0              # two captures flipped it twice (fused) or never (two-pass)
    inject = {4: (inf_at(job, 3, 5),), 7: (inf_at(job, N - 1, n - 1),)}
    for step in range(2, 12):
        grads = job.make_grads(step, inject.get(step, ()))
        job.load_grads(grads)
        graphs[(step - 2) % 2].replay()
        torch.cuda.synchronize()
        res, ref = job.read(), job.oracle_step(grads)
        if not job.two_pass:
            job.bufs.b.cur = 1 - job.bufs.b.cur   # what the call does on the host, replayed by hand
        job.check(res, ref)
        assert res.overflow == (1 if step in inject else 0)


# --- a model that is one bucket ---------------------------------------------------
ONE = [
    # stage, N, n, dtype, optimizer
    (2, 4, 1 << 20, oracle.FP16, zg.ZERO_ADAM),            # the 2^20-parameter, 4-rank workload
    (2, 1, 1, oracle.FP16, zg.ZERO_ADAM),
    (2, 3, 1005, oracle.BF16, zg.ZERO_SGD_MOMENTUM),
    (2, 2, 1_200_003, oracle.FP16, zg.ZERO_ADAM),          # more groups than one wave of blocks
    (2, 4, 300_001, oracle.FP32, zg.ZERO_ADAM),
    (3, 5, 12_345, oracle.FP16, zg.ZERO_SGD),
    (3, 8, 70_001, oracle.BF16, zg.ZERO_ADAM),
    (3, 64, 65_536, oracle.FP16, zg.ZERO_ADAM),
]


@pytest.mark.parametrize("case", ONE, ids=lambda c: "s%d-N%d-n%d-dt%d-o%d" % c)
def test_one_bucket_steps_match_oracle(case):
    """Stages 2-3, the model one bucket (sizes up to more groups than one
    wave of blocks): equal to the oracle bit for bit through overflows at the
    first and the last element and loss-scale growth."""
    stage, N, n, dtype, opt = case
    job = AsyncJob(n, N, stage, 1 << 22, 8, None, dtype, loss_scale=256.0, dynamic=True, growth=2, optimizer=opt)
    assert job.plan.n_buckets == 1
    plan = [(), (), (inf_at(job, 0, 0),), (), (), (inf_at(job, N - 1, n - 1),), (), ()]
    for step, inject in enumerate(plan, start=1):
        res, ref = job.step(job.make_grads(step, inject))
        job.check(res, ref)
        assert res.overflow == (1 if inject else 0)
    assert job.state.t == 6 and job.state.loss_scale == ref["loss_scale"]


TWO = [
    # stage, N, n, dtype, max_norm, optimizer, shadow
    (2, 8, 1 << 20, oracle.FP16, 1.0, zg.ZERO_ADAM, False),      # the 2^20-parameter point of the clipping sweep
    (2, 2, 300_001, oracle.BF16, 1e-2, zg.ZERO_ADAM, False),
    (2, 1, 1, oracle.FP16, 1e-2, zg.ZERO_SGD_MOMENTUM, False),
    (3, 5, 70_001, oracle.BF16, 1e-3, zg.ZERO_ADAM, False),
    (3, 64, 65_536, oracle.FP16, 1e-2, zg.ZERO_SGD, False),
    (2, 4, 100_003, oracle.FP32, 0.0, zg.ZERO_ADAM, False),      # binary32 without a shadow: two-pass, no clipping
    (2, 3, 1005, oracle.FP16, 0.0, zg.ZERO_ADAM, False),
    (2, 8, 1 << 20, oracle.FP16, 1.0, zg.ZERO_ADAM, True),       # clipping with the shadow state given
    (2, 32, 1 << 20, oracle.FP16, 1.0, zg.ZERO_ADAM, False),     # one bucket above 64 MiB: five kernels
]


@pytest.mark.parametrize("case", TWO, ids=lambda c: "s%d-N%d-n%d-dt%d-c%g-o%d-sh%d" % c)
def test_one_bucket_two_pass_steps_match_oracle(case):
    """Two-pass device-state steps of a model that is one bucket: when small,
    pass 1 (whose last block derives the step's scalars and finishes the
    norm) and pass 2 (whose last block commits) are the whole step.  Equal to
    the oracle bit for bit, norm and clip coefficient included, through
    overflows at the first and the last element and loss-scale growth."""
    stage, N, n, dtype, max_norm, opt, shadow = case
    job = AsyncJob(n, N, stage, 1 << 22, 8, None, dtype, shadow=shadow, loss_scale=256.0, dynamic=True, growth=2,
                   max_norm=max_norm, optimizer=opt, sigma=0.03 if max_norm >= 1.0 else 1e-3)
    assert job.plan.n_buckets == 1 and job.two_pass
    plan = [(), (), (inf_at(job, 0, 0),), (), (), (inf_at(job, N - 1, n - 1),), (), ()]
    for step, inject in enumerate(plan, start=1):
        res, ref = job.step(job.make_grads(step, inject))
        job.check(res, ref)
        assert res.overflow == (1 if inject else 0)
    assert job.state.t == 6 and job.state.loss_scale == ref["loss_scale"]


# --- the same step one bucket at a time -----------------------------------------
@pytest.mark.parametrize("stage,shadow,max_norm,staged", [(2, True, 0.0, False), (2, True, 0.0, True),
                                                          (2, False, 1e-3, True), (3, True, 0.0, True),
                                                          (3, False, 0.0, False), (1, True, 0.0, False)])
def test_per_bucket_async_matches_oracle(stage, shadow, max_norm, staged):
    """begin_async, the buckets in backward (reverse) order -- from per-rank
    staging buffers that are refilled for every bucket when `staged` --, then
    end_async: the oracle's step, bit for bit, through an overflowed step."""
    n, N, B = 4 * 1024 + 37, 4, 1024
    job = AsyncJob(n, N, stage, B, 8, None, oracle.FP16, shadow=shadow, loss_scale=64.0, dynamic=True,
                   max_norm=max_norm)
    s = torch.cuda.current_stream()
    staging = [torch.zeros(B, dtype=torch.int16, device="cuda") for _ in range(N)]
    for step, inject in ((1, ()), (2, ((2, 3 * B + 5, synth.inf_bits(oracle.FP16)),)), (3, ())):
        grads = job.make_grads(step, inject)
        job.load_grads(grads)
        zg.zero_step_begin_async(job.cfg, job.plan, job.bufs, job.adam, job.dev, s)
        for b in reversed(range(job.plan.n_buckets)):
            if staged:
                lo, hi = b * B, min((b + 1) * B, n)
                for r in range(N):
                    staging[r][:hi - lo].copy_(torch.from_numpy(grads[r][lo:hi].view(np.int16)))
            zg.zero_step_bucket_async(job.cfg, job.plan, job.bufs, job.adam, b,
                                      [t.data_ptr() for t in staging] if staged else None, s)
        zg.zero_step_end_async(job.cfg, job.plan, job.bufs, job.adam, job.dev, s)
        res, ref = job.read(), job.oracle_step(grads)
        job.check(res, ref)
        assert res.overflow == (1 if inject else 0)


def test_per_bucket_async_captured_in_graphs():
    n, N, B = 3 * 2048 + 11, 4, 2048
    job = AsyncJob(n, N, 2, B, 8, None, oracle.FP16, loss_scale=32.0, dynamic=True)
    cap = torch.cuda.Stream()

    def sequence(stream):
        zg.zero_step_begin_async(job.cfg, job.plan, job.bufs, job.adam, job.dev, stream)
        for b in reversed(range(job.plan.n_buckets)):
            zg.zero_step_bucket_async(job.cfg, job.plan, job.bufs, job.adam, b, None, stream)
        zg.zero_step_end_async(job.cfg, job.plan, job.bufs, job.adam, job.dev, stream)

    grads = job.make_grads(1)
    job.load_grads(grads)
    sequence(torch.cuda.current_stream())
    res, ref = job.read(), job.oracle_step(grads)
    job.check(res, ref)
    torch.cuda.synchronize()
    graphs = []
    for _ in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cap):
            sequence(torch.cuda.current_stream())
        graphs.append(g)
    for step in range(2, 7):
        grads = job.make_grads(step, ((1, 17, synth.inf_bits(oracle.FP16)),) if step == 4 else ())
        job.load_grads(grads)
        graphs[step % 2].replay()
        torch.cuda.synchronize()
        res, ref = job.read(), job.oracle_step(grads)
        job.bufs.b.cur = 1 - job.bufs.b.cur
        job.check(res, ref)


@pytest.mark.parametrize("shadow", [True, False])
def test_async_empty_model(shadow):
    """Zero parameters: the device-state step still commits (t advances), as
    the synchronising step does.  (The two-pass path still wants a reduced
    buffer, even an empty one: a 16-byte placeholder.)"""
    job = AsyncJob(0, 4, 2, 64, 8, None, oracle.FP16, shadow=shadow)
    placeholder = torch.zeros(8, dtype=torch.int16, device="cuda")
    if not shadow:
        job.bufs.b.reduced = placeholder.data_ptr()
    for step in (1, 2):
        job.load_grads(job.make_grads(step))
        assert job.launch() == 2
        st, last = zg.zero_dev_state_read(job.dev)
        assert st.t == step and last.overflow == 0
