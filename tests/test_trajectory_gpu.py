"""Long trajectories: 100 consecutive steps against the oracle, bit for bit
at every step, so that anything that drifts with the step count (the bias
corrections from the repeated-product beta powers, the moment buffers, the
loss scale) is caught where it first differs.

The clipped runs have the shape of the stage-2 clipping sweep (clipping at
1.0, bias correction, S = 1, N_d in {2, 8, 32}, both 16-bit types), scaled
down: the gradient spread is set so that the norm of the mean gradient sits
near 1.0 and about half of the steps are clipped.  The device-state runs take
the fused path (speculative, with shadow state) and the clipped two-pass path
through 100 steps with a dynamic loss scale, overflows injected every 17th
step and growth every 10 clean steps (two ranks: pass 1 staged through
shared memory; and a model that is one bucket)."""
import math

import numpy as np
import pytest

import oracle
import synth
import zero_sharded_mixed_bucket_gb300 as zg
from tests.gpu_harness import Job
from tests.test_async_gpu import AsyncJob

pytestmark = pytest.mark.gpu

STEPS = 100


@pytest.mark.parametrize("N", [2, 8, 32])
@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
def test_clipped_trajectory(N, dtype):
    n, B = (1 << 14) + 13, 4096
    sigma = math.sqrt(N / n)          # ||mean gradient|| ~ sqrt(n) * sigma / sqrt(N) = 1
    job = Job(n, N, 2, B, 8, dtype=dtype, shadow=False, max_norm=1.0, sigma=sigma, loss_scale=1.0)
    clipped = 0
    for t in range(1, STEPS + 1):
        res, ref = job.step(job.make_grads(t))
        job.check(res, ref)
        clipped += ref["clip"] < 1.0
    assert job.state.t == STEPS
    assert 0 < clipped < STEPS, clipped


@pytest.mark.parametrize("shadow,max_norm,dtype,N,B", [(True, 0.0, oracle.FP16, 8, 2048), (False, 1.0, oracle.BF16, 8, 2048),
                                                       (False, 1.0, oracle.FP16, 2, 2048),
                                                       (True, 0.0, oracle.BF16, 4, 1 << 14),
                                                       (False, 1.0, oracle.FP16, 8, 1 << 14)])
def test_device_state_trajectory(shadow, max_norm, dtype, N, B):
    n = 5 * 2048 + 19
    job = AsyncJob(n, N, 2, B, 8, None, dtype, shadow=shadow, loss_scale=1024.0, dynamic=True, growth=10,
                   max_norm=max_norm, sigma=0.03 if max_norm else 1e-3)
    skipped = 0
    for step in range(1, STEPS + 1):
        inject = ((step % N, (step * 7919) % n, synth.inf_bits(dtype)),) if step % 17 == 0 else ()
        res, ref = job.step(job.make_grads(step, inject))
        job.check(res, ref)
        assert res.overflow == (1 if inject else 0)
        skipped += res.skipped
    assert skipped == STEPS // 17
    assert job.state.t == STEPS - skipped
    assert job.state.loss_scale == ref["loss_scale"]
