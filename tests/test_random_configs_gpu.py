"""Random combinations of everything the step takes -- stage, N_d, sizes,
bucket and alignment, value type, optimizer, shadow state or not, clipping,
loss scaling, staged per-bucket gradients, and the entry point (one call,
begin/bucket/end, the device-state step, its per-bucket form, and runs of
buckets in a random order, plain and device-state) -- each run for three
steps (the second overflowed by an inf at a random rank and element, so
the buckets after it may skip) against the oracle, bit for bit.
The combinations come from a fixed seed, so a failure names a reproducible
case; ZG_RANDOM_SEED and ZG_RANDOM_CASES draw another set (a longer soak)."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_mixed_bucket_gb300 as zg
from tests.gpu_harness import Job, as_signed

pytestmark = pytest.mark.gpu

APIS = ("step", "per_bucket", "async", "per_bucket_async", "runs", "runs_async")


def _cases(k=96, seed=2024):
    rng = np.random.default_rng(seed)
    out = []
    while len(out) < k:
        stage = int(rng.integers(0, 4))
        N = int(rng.choice([1, 2, 3, 5, 8, 9, 16, 17, 33]))
        B = int(rng.choice([8, 64, 512, 2048, 4096]))
        n = int(rng.integers(1, 6 * B + 50)) if B < 4096 else int(rng.integers(1, 20_000))
        A = int(rng.choice([8, 64, 2048]))
        dtype = int(rng.choice([oracle.FP16, oracle.BF16, oracle.FP32]))
        opt = int(rng.choice([zg.ZERO_ADAM, zg.ZERO_SGD_MOMENTUM, zg.ZERO_SGD]))
        shadow = bool(rng.integers(0, 2))
        clip = dtype != oracle.FP32 and bool(rng.integers(0, 3) == 0)
        api = APIS[int(rng.integers(0, len(APIS)))]
        staged = api != "step" and api != "async" and stage >= 2 and bool(rng.integers(0, 2))
        scale = float(rng.choice([1.0, 8.0, 1024.0]))
        inj = (int(rng.integers(0, N)), int(rng.integers(0, n)))
        order = int(rng.integers(0, 2 ** 31))       # seed of the bucket order and runs
        out.append((stage, N, n, B, A, dtype, opt, shadow, clip, api, staged, scale, inj, order))
    return out


def _runs(nb, seed):
    """The buckets in a random order, cut into runs of 1 to 4."""
    rng = np.random.default_rng(seed)
    perm = [int(b) for b in rng.permutation(nb)]
    runs = []
    while perm:
        k = int(rng.integers(1, 5))
        runs.append(perm[:k])
        perm = perm[k:]
    return runs


@pytest.mark.parametrize("case", _cases(int(os.environ.get("ZG_RANDOM_CASES", "96")),
                                         int(os.environ.get("ZG_RANDOM_SEED", "2024"))), ids=lambda c: "s%d-N%d-n%d-B%d-A%d-dt%d-o%d-sh%d-c%d-%s-st%d-i%d.%d" % (
    c[0], c[1], c[2], c[3], c[4], c[5], c[6], c[7], c[8], c[9], c[10], c[12][0], c[12][1]))
def test_random_combination(case):
    stage, N, n, B, A, dtype, opt, shadow, clip, api, staged, scale, inj, order = case
    job = Job(n, N, stage, B, A, dtype=dtype, shadow=shadow, optimizer=opt, max_norm=1e-2 if clip else 0.0,
              loss_scale=scale, dynamic=True, growth=2, sigma=1e-3)
    dev = None
    if api in ("async", "per_bucket_async", "runs_async"):
        dev = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device="cuda")
        zg.zero_dev_state_init(dev, job.adam, job.state)
    s = torch.cuda.current_stream()
    vt = torch.int32 if dtype == oracle.FP32 else torch.int16
    staging = [torch.zeros(B, dtype=vt, device="cuda") for _ in range(N)] if staged else None
    for step in (1, 2, 3):
        inject = ((inj[0], inj[1], synth.inf_bits(dtype)),) if step == 2 else ()
        grads = job.make_grads(step, inject)
        job.load_grads(grads)
        two_pass = clip or not shadow
        if api == "step":
            fn = [zg.zero_step_stage0, zg.zero_step_stage1, zg.zero_step_stage2, zg.zero_step_stage3][stage]
            res = fn(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
        elif api == "async":
            zg.zero_step_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
        elif api in ("runs", "runs_async"):
            is_async = api == "runs_async"
            if is_async:
                zg.zero_step_begin_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
            else:
                zg.zero_step_begin(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
            windows = []                       # every bucket its own windows: a run's kernels overlap
            for run in _runs(job.plan.n_buckets, order + step):
                table = None
                if staged:
                    table = []
                    for b in run:
                        lo, hi = b * B, min((b + 1) * B, n)
                        w = [torch.from_numpy(as_signed(grads[r][lo:hi]).copy()).cuda() for r in range(N)]
                        windows.append(w)
                        table.append([t.data_ptr() for t in w])
                if is_async:
                    zg.zero_step_buckets_async(job.cfg, job.plan, job.bufs, job.adam, run, table, s)
                else:
                    zg.zero_step_buckets(job.cfg, job.plan, job.bufs, job.adam, job.state, run, table, s)
            if is_async:
                zg.zero_step_end_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
            else:
                res = zg.zero_step_end(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
        else:
            is_async = api == "per_bucket_async"
            if is_async:
                zg.zero_step_begin_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
            else:
                zg.zero_step_begin(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
            for b in reversed(range(job.plan.n_buckets)):
                ptrs = None
                if staged:
                    lo, hi = b * B, min((b + 1) * B, n)
                    for r in range(N):
                        staging[r][:hi - lo].copy_(torch.from_numpy(as_signed(grads[r][lo:hi])))
                    ptrs = [t.data_ptr() for t in staging]
                if is_async:
                    zg.zero_step_bucket_async(job.cfg, job.plan, job.bufs, job.adam, b, ptrs, s)
                else:
                    zg.zero_step_bucket(job.cfg, job.plan, job.bufs, job.adam, job.state, b, ptrs, s)
            if is_async:
                zg.zero_step_end_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
            else:
                res = zg.zero_step_end(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
        torch.cuda.synchronize()
        if dev is not None:
            st, res = zg.zero_dev_state_read(dev, s)
            job.state = st
            res.path = 1 if two_pass else 0
        ref = job.oracle_step(grads)
        job.check(res, ref)
        assert res.overflow == (1 if step == 2 else 0)
