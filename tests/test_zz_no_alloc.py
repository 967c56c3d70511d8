"""zero_step_stage2_noalloc: the stage-2 step for callers that cannot
allocate device memory (for example code running inside another runtime that
owns the GPU's memory pool, or code that must not allocate after start-up).
Its scratch comes from a static array inside the library, so the caller
passes no workspace and no reduced-gradient buffer.

The GPU test runs the new entry point and the regular zero_step_stage2 on
identical inputs, several calls in a row (clean and overflowed steps, with
and without clipping), and requires identical results; every call is also
compared with the CPU oracle's unpartitioned step on the same inputs, at
the parity tests' bar (bit-exact 16-bit parameters, flag, norm, clip
coefficient and loss scale; the fp32 state here bit-identical too).  The
file is collected last so that a run stopping at the first failure has
already run every other test.
"""
import ctypes

import numpy as np
import pytest

import zero_sharded_mixed_bucket_gb300 as zg


def _fake_buffers(N):
    """zero_buffers_t with made-up device addresses; only the host-side
    checks ever see them."""
    gp = (ctypes.c_void_p * N)(*[0x10000000 + 0x100000 * r for r in range(N)])
    pp = (ctypes.c_void_p * N)(*[0x20000000 + 0x100000 * r for r in range(N)])
    b = zg.zero_buffers_t()
    b.grads = ctypes.cast(gp, ctypes.POINTER(ctypes.c_void_p))
    b.params16 = ctypes.cast(pp, ctypes.POINTER(ctypes.c_void_p))
    b.w[0], b.m[0], b.v[0] = 0x30000000, 0x40000000, 0x50000000
    return b, (gp, pp)


def _call(cfg, b):
    plan = zg.zero_plan_t()
    zg.lib().zero_plan(ctypes.byref(cfg.c), ctypes.byref(plan))
    adam = zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8)
    state = zg.zero_state_t(loss_scale=1.0, min_loss_scale=1.0)
    res = zg.zero_step_result_t()
    return zg.lib().zero_step_stage2_noalloc(ctypes.byref(cfg.c), ctypes.byref(plan), ctypes.byref(b),
                                             ctypes.byref(adam), ctypes.byref(state), None, ctypes.byref(res))


def test_noalloc_rejects_what_does_not_fit():
    """Checked on the host before any CUDA call: too large for the static
    scratch, or not a stage-2 config."""
    b, keep = _fake_buffers(1)
    st = _call(zg.Config(8 * 1024 * 1024 + 1, 1, 2, 1 << 20), b)
    assert st == zg.ZERO_EUNSUPPORTED
    assert "static scratch" in zg.zero_last_error()
    b, keep = _fake_buffers(4)
    assert _call(zg.Config(1000, 4, 3, 64), b) == zg.ZERO_EINVAL
    assert "stage-2" in zg.zero_last_error()


@pytest.mark.gpu
@pytest.mark.parametrize("max_norm", [0.0, 1.0])
def test_noalloc_matches_regular_step(max_norm):
    import torch

    from tests.gpu_harness import Job, as_u16, as_u32

    n, N, B = 3 * 65536 + 123, 4, 65536
    kw = dict(shadow=False, max_norm=max_norm, sigma=0.05, loss_scale=64.0, dynamic=True)
    ref = Job(n, N, 2, B, **kw)     # regular entry point, its own workspace and reduced buffer
    job = Job(n, N, 2, B, **kw)     # same seeded inputs; no scratch handed over
    job.bufs.b.workspace = None
    job.bufs.b.reduced = None
    s = torch.cuda.current_stream()
    inf = 0x7C00
    # clean, overflowed, clean, clean: the static scratch must start each call clear
    for t, inject in ((1, []), (2, [(2, 77, inf)]), (3, []), (4, [])):
        grads = ref.make_grads(t, inject=inject)
        ref.load_grads(grads)
        job.load_grads(grads)
        ra = zg.zero_step_stage2(ref.cfg, ref.plan, ref.bufs, ref.adam, ref.state, s)
        rb = zg.zero_step_stage2_noalloc(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
        torch.cuda.synchronize()
        # against the oracle: the job's reduced-gradient buffer is not used
        # (that scratch is the library's static array), everything else is
        job.check(rb, job.oracle_step(grads), reduced=False)
        assert (rb.overflow, rb.skipped, rb.t, rb.path) == (ra.overflow, ra.skipped, ra.t, ra.path)
        assert rb.overflow == (1 if inject else 0)
        assert rb.new_loss_scale == ra.new_loss_scale
        assert rb.grad_norm == ra.grad_norm and rb.clip_coef == ra.clip_coef
        if max_norm > 0 and not inject:
            assert rb.clip_coef < 1.0
        for a, b in zip(ref.bufs.state(), job.bufs.state()):
            assert np.array_equal(as_u32(a[:n]), as_u32(b[:n]))
        for r in range(N):
            assert np.array_equal(as_u16(ref.bufs.params16[r][:n]), as_u16(job.bufs.params16[r][:n]))
