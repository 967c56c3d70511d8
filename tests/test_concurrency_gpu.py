"""Two host threads drive two independent jobs at once, each on its own CUDA
stream, through the same library: the host-side state the library keeps
(thread-local error text and profile events, the launch-shape cache, the
per-thread table of pointer kinds) must not mix them up.  Each job's steps
equal the oracle's bit for bit."""
import threading

import pytest
import torch

import oracle
import zero_sharded_mixed_bucket_gb300 as zg
from tests.gpu_harness import Job

pytestmark = pytest.mark.gpu


def _run(job, steps, errors, name):
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            for t in range(1, steps + 1):
                res, ref = job.step(job.make_grads(t))
                job.check(res, ref)
    except Exception as e:          # reported by the main thread
        errors.append((name, repr(e)))


def test_two_jobs_from_two_threads():
    jobs = {
        "stage 2 fp16 fused": Job(6 * 1024 + 5, 4, 2, 1024, 8, dtype=oracle.FP16, loss_scale=64.0),
        "stage 3 bf16 clipped": Job(5 * 512 + 3, 3, 3, 512, 8, dtype=oracle.BF16, shadow=False, max_norm=0.05,
                                    sigma=1e-2),
        "stage 1 fp16 many ranks": Job(3 * 2048 + 1, 16, 1, 2048, 8, dtype=oracle.FP16,
                                       optimizer=zg.ZERO_SGD_MOMENTUM),
    }
    errors = []
    threads = [threading.Thread(target=_run, args=(job, 6, errors, name)) for name, job in jobs.items()]
    for th in threads:
        th.start()
    for th in threads:
        th.join(timeout=300)
        assert not th.is_alive()
    assert not errors, errors
    for job in jobs.values():
        assert job.state.t == 6
