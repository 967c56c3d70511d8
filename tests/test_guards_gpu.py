"""Out-of-bounds writes, checked without a sanitizer: every buffer the
library is given sits between two guard regions filled with a pattern, and
after steps across stages, paths, optimizers, value types (16-bit and
binary32) and ragged sizes (plus stage-3 gathers and fetches) every guard
must still hold its pattern."""
import ctypes

import pytest
import torch

import synth
import zero_sharded_mixed_bucket_gb300 as zg

pytestmark = pytest.mark.gpu

GUARD = 4096                     # elements on each side (a multiple of 8: interiors stay 16-byte aligned)
PAT16 = 0x7DA5                   # an int16 pattern (a NaN bit pattern in binary16)
PAT32 = 0x7FC0DEAD               # an int32 pattern (a NaN bit pattern in binary32)


class Guarded:
    """A tensor with guard regions; .t is the interior."""

    def __init__(self, n, dtype):
        self.full = torch.empty(n + 2 * GUARD, dtype=dtype, device="cuda")
        if dtype in (torch.float32, torch.int32):
            self.full.view(torch.int32).fill_(PAT32)
        else:
            self.full.fill_(PAT16 if dtype == torch.int16 else 0xA5)
        self.n = n
        self.t = self.full[GUARD:GUARD + n]
        self.pattern = self.full.clone()

    def ptr(self):
        return self.t.data_ptr()

    def intact(self):
        a = self.full.view(torch.int8)
        b = self.pattern.view(torch.int8)
        k = GUARD * self.full.element_size()
        return torch.equal(a[:k], b[:k]) and torch.equal(a[-k:], b[-k:])


def _buffers(cfg, plan, shadow, reduced):
    N = cfg.c.n_ranks
    vt = torch.int32 if cfg.c.dtype == zg.ZERO_FP32 else torch.int16    # binary32 values, or 16-bit
    g = [Guarded(plan.grad16_elems, vt) for _ in range(N)]
    p = [Guarded(plan.param16_elems, vt) for _ in range(N)]
    st = {k: [Guarded(plan.state_elems, torch.float32) for _ in range(2 if shadow else 1)] for k in "wmv"}
    red = Guarded(max(plan.reduced_elems, 1), vt) if reduced else None
    ws = Guarded(plan.workspace_bytes, torch.uint8)
    for k in "wmv":
        for x in st[k]:
            x.t.zero_()
    for x in g + p:
        x.t.zero_()
    b = zg.zero_buffers_t()
    gp = (ctypes.c_void_p * N)(*[x.ptr() for x in g])
    pp = (ctypes.c_void_p * N)(*[x.ptr() for x in p])
    b.grads = ctypes.cast(gp, ctypes.POINTER(ctypes.c_void_p))
    b.params16 = ctypes.cast(pp, ctypes.POINTER(ctypes.c_void_p))
    for k in "wmv":
        for c, x in enumerate(st[k]):
            getattr(b, k)[c] = x.ptr()
    b.reduced = red.ptr() if red else None
    b.workspace = ws.ptr()
    every = g + p + [x for k in "wmv" for x in st[k]] + ([red] if red else []) + [ws]
    return b, (gp, pp), g, st, every


CASES = [
    # stage, n_ranks, n, bucket, align, dtype, shadow, max_norm, optimizer
    (0, 3, 3 * 1024 + 5, 1024, 8, 0, True, 0.0, zg.ZERO_ADAM),
    (1, 3, 2 * 1024 + 7, 1024, 16, 1, False, 1.0, zg.ZERO_ADAM),
    (2, 4, 5 * 512 + 3, 512, 8, 0, True, 0.0, zg.ZERO_SGD_MOMENTUM),
    (2, 4, 5 * 512 + 3, 512, 8, 1, False, 1.0, zg.ZERO_ADAM),
    (3, 5, 7 * 256 + 1, 256, 8, 0, True, 0.0, zg.ZERO_SGD),
    (3, 5, 7 * 256 + 1, 256, 64, 0, False, 1.0, zg.ZERO_ADAM),
    (0, 1, 7, 8, 8, 0, True, 0.0, zg.ZERO_ADAM),
    (0, 3, 3 * 1024 + 5, 1024, 8, 2, True, 0.0, zg.ZERO_ADAM),
    (1, 3, 2 * 1024 + 7, 1024, 16, 2, False, 0.0, zg.ZERO_SGD_MOMENTUM),
    (2, 4, 5 * 512 + 3, 512, 8, 2, True, 0.0, zg.ZERO_SGD_MOMENTUM),
    (3, 5, 7 * 256 + 1, 256, 8, 2, False, 0.0, zg.ZERO_SGD),
    # two-pass with 2 or more ranks: parameters written by bulk copies from tiles
    (2, 17, 5 * 512 + 3, 512, 8, 0, False, 1.0, zg.ZERO_ADAM),
    (1, 16, 2 * 1024 + 7, 1024, 16, 2, False, 0.0, zg.ZERO_SGD_MOMENTUM),
    (2, 8, 3 * 4096 + 11, 4096, 8, 1, False, 1.0, zg.ZERO_ADAM),
    (1, 8, 2 * 4096 + 5, 8192, 8, 0, False, 0.0, zg.ZERO_SGD),
]


@pytest.mark.parametrize("case", CASES)
def test_steps_write_only_inside_their_buffers(case):
    stage, N, n, B, A, dtype, shadow, max_norm, opt = case
    cfg = zg.Config(n, N, stage, B, A, None, dtype, opt)
    plan = zg.zero_plan(cfg)
    b, keep, grads, st, every = _buffers(cfg, plan, shadow, reduced=stage >= 2)
    reps = N if stage == 0 else 1
    for r in range(reps):
        synth.dev_normal32(st["w"][0].ptr() + 4 * r * plan.padded_elems, n, 0.02, seed=0,
                           stream=synth.STREAM_WEIGHT)
    adam = zg.zero_adam_t(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, max_grad_norm=max_norm, momentum=0.9)
    state = zg.zero_state_t(t=0, loss_scale=8.0, min_loss_scale=1.0, dynamic=1)
    s = torch.cuda.current_stream()
    for step in (1, 2, 3):
        for r in range(N):
            synth.dev_grad(grads[r].ptr(), n, dtype, 8e-3, seed=0, stream=synth.STREAM_GRAD, step=step, rank=r)
        if step == 2:
            grads[N - 1].t[n - 1] = synth.inf_bits(dtype)       # an overflowed step (restore path)
        res = zg.zero_step(cfg, plan, b, adam, state, s)
        torch.cuda.synchronize()
        assert res.overflow == (1 if step == 2 else 0)
    bad = [i for i, x in enumerate(every) if not x.intact()]
    assert not bad, "guard regions overwritten: %s" % bad


def test_bucket_staging_gather_and_fetch_stay_inside():
    layers = [1003, 2048, 17, 4001]
    n, N, B = sum(layers), 3, 1024
    cfg = zg.Config(n, N, 3, B, 8, layers)
    plan = zg.zero_plan(cfg)
    b, keep, grads, st, every = _buffers(cfg, plan, shadow=True, reduced=False)
    staging = [Guarded(B, torch.int16) for _ in range(N)]
    s = torch.cuda.current_stream()
    adam = zg.zero_adam_t(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8)
    state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
    zg.zero_step_begin(cfg, plan, b, adam, state, s)
    for bk in range(plan.n_buckets):
        lo, hi = bk * B, min((bk + 1) * B, n)
        for r in range(N):
            synth.dev_normal16(staging[r].ptr(), hi - lo, 0, 1e-3, seed=0, stream=synth.STREAM_GRAD, step=1, rank=r,
                               offset=lo)
        zg.zero_step_bucket(cfg, plan, b, adam, state, bk, [x.ptr() for x in staging], s)
    zg.zero_step_end(cfg, plan, b, adam, state, s)
    shards = [x.ptr() for x in every[N:2 * N]]
    dst = [Guarded(plan.max_layer_elems, torch.int16) for _ in range(9)]
    for l in range(len(layers)):
        zg.zero_gather_layer(cfg, plan, l, shards, [d.ptr() for d in dst[:2]], s)   # chunked, 2 destinations
        zg.zero_gather_layer(cfg, plan, l, shards, [d.ptr() for d in dst], s)       # chunked, destination by destination
    cap = 4008 + 2056
    pool = [Guarded(cap, torch.int16) for _ in range(2)]
    side = torch.cuda.Stream()
    f = zg.Fetcher(cfg, plan, shards, [x.t for x in pool], cap, list(reversed(range(len(layers)))), 2, side)
    for pos in range(len(layers)):
        f.fetch(pos, s)
        f.release(pos, s)
    torch.cuda.synchronize()
    for x in every + staging + dst + pool:
        assert x.intact()
