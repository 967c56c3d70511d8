"""Helpers for the GPU parity tests: a job on the device driven through the
C ABI, mirrored step by step by the CPU oracle on the same seeded inputs."""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import synth
import zero_sharded_mixed_bucket_gb300 as zg

ADAM = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8)


def as_u16(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def as_bits(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a value buffer: uint16 (16-bit types) or uint32
    (binary32 values, held in int32 tensors)."""
    return t.cpu().numpy().view(np.uint32 if t.dtype == torch.int32 else np.uint16)


def as_signed(a: np.ndarray) -> np.ndarray:
    """Host bit patterns in the signed type of the device tensors."""
    return a.view(np.int32 if a.dtype == np.uint32 else np.int16)


def as_u32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.cpu().numpy()
    return np.ascontiguousarray(a).view(np.uint32)


def same16(a: np.ndarray, b: np.ndarray, dtype: int) -> bool:
    """Bit-equal 16-bit arrays, treating any two NaNs as equal (payloads of
    NaN are not part of the result)."""
    if a.shape != b.shape:
        return False
    na = oracle.is_nonfinite16(a, dtype) & np.isnan(oracle.to_f32(a, dtype))
    nb = oracle.is_nonfinite16(b, dtype) & np.isnan(oracle.to_f32(b, dtype))
    return bool(np.array_equal(na, nb) and np.array_equal(a[~na], b[~nb]))


def max_rel(a: np.ndarray, b: np.ndarray) -> float:
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    d = np.abs(a - b) / np.maximum(np.abs(b), 1e-30)
    return float(d.max()) if d.size else 0.0


class Job:
    """One simulated ZeRO job on the GPU plus the oracle's unpartitioned copy."""

    OPT_NAMES = {zg.ZERO_ADAM: "adam", zg.ZERO_SGD_MOMENTUM: "sgdm", zg.ZERO_SGD: "sgd"}

    def __init__(self, n, N, stage, B, A=0, layers=None, dtype=oracle.FP16, shadow=True, seed=0,
                 loss_scale=1.0, dynamic=False, min_scale=1.0, growth=0, max_norm=0.0, sigma=1e-3, adam=None,
                 optimizer=zg.ZERO_ADAM, momentum=0.9):
        self.n, self.N, self.stage, self.dtype = n, N, stage, dtype
        self.seed, self.sigma = seed, sigma
        self.optimizer, self.momentum = optimizer, momentum
        self.cfg = zg.Config(n, N, stage, B, A, layers, dtype, optimizer)
        self.plan = zg.zero_plan(self.cfg)
        self.bufs = zg.DeviceBuffers(self.cfg, self.plan, device="cuda", shadow=shadow)
        if optimizer != zg.ZERO_ADAM:          # arrays the optimizer does not use are not handed over
            for k in range(2):
                self.bufs.b.v[k] = None
                if optimizer == zg.ZERO_SGD:
                    self.bufs.b.m[k] = None
        self.hp = dict(ADAM if adam is None else adam)
        self.adam = zg.zero_adam_t(max_grad_norm=max_norm, momentum=momentum, **self.hp)
        self.max_norm = max_norm
        self.state = zg.zero_state_t(t=0, loss_scale=loss_scale, min_loss_scale=min_scale, dynamic=int(dynamic),
                                     growth_interval=growth)
        self.o = dict(t=0, loss_scale=loss_scale, good_steps=0)
        self.dynamic, self.min_scale, self.growth = dynamic, min_scale, growth
        # master weights and their 16-bit cast on every rank
        self.w = synth.host_normal32(n, 0.02, seed=seed, stream=synth.STREAM_WEIGHT)
        self.m = np.zeros(n, np.float32)
        self.v = np.zeros(n, np.float32)
        p0 = oracle.cast16(self.w, dtype)
        P = self.plan.shard_elems
        reps = N if stage == 0 else 1
        for r in range(reps):
            off = r * self.plan.padded_elems
            self.bufs.w[0][off:off + n].copy_(torch.from_numpy(self.w))
        for r in range(N):
            if stage == 3:
                lo, hi = r * P, min((r + 1) * P, n)
                if hi > lo:
                    self.bufs.params16[r][:hi - lo].copy_(torch.from_numpy(as_signed(p0[lo:hi])))
            else:
                self.bufs.params16[r][:n].copy_(torch.from_numpy(as_signed(p0)))
        self.p16 = p0
        self.h = None
        self.last_ref = None
        torch.cuda.synchronize()

    # -- inputs -------------------------------------------------------------
    def make_grads(self, step, inject=()):
        S = self.o["loss_scale"]
        grads = [synth.host_grad(self.n, self.dtype, self.sigma * S, seed=self.seed, stream=synth.STREAM_GRAD,
                                     step=step, rank=r) for r in range(self.N)]
        for r, i, bits in inject:
            grads[r][i] = bits
        return grads

    def load_grads(self, grads):
        for r in range(self.N):
            self.bufs.grads[r][:self.n].copy_(torch.from_numpy(as_signed(grads[r])))

    # -- one step on both sides ------------------------------------------------
    def step(self, grads, per_bucket=False):
        self.load_grads(grads)
        s = torch.cuda.current_stream()
        if per_bucket:
            zg.zero_step_begin(self.cfg, self.plan, self.bufs, self.adam, self.state, s)
            for b in range(self.plan.n_buckets):
                zg.zero_step_bucket(self.cfg, self.plan, self.bufs, self.adam, self.state, b, None, s)
            res = zg.zero_step_end(self.cfg, self.plan, self.bufs, self.adam, self.state, s)
        else:
            fn = [zg.zero_step_stage0, zg.zero_step_stage1, zg.zero_step_stage2, zg.zero_step_stage3][self.stage]
            res = fn(self.cfg, self.plan, self.bufs, self.adam, self.state, s)
        torch.cuda.synchronize()
        return res, self.oracle_step(grads)

    def oracle_step(self, grads):
        """The same step on the oracle's copy; updates the expected state."""
        ref = oracle.step(grads, self.w, self.m, self.v, dtype=self.dtype, t=self.o["t"],
                          loss_scale=self.o["loss_scale"], max_grad_norm=self.max_norm, dynamic=self.dynamic,
                          min_scale=self.min_scale, growth_interval=self.growth, good_steps=self.o["good_steps"],
                          optimizer=self.OPT_NAMES[self.optimizer], momentum=self.momentum, **self.hp)
        self.o.update(t=ref["t"], loss_scale=ref["loss_scale"], good_steps=ref["good_steps"])
        self.p16 = ref["p16"]
        self.h = ref["h"]
        self.last_ref = ref
        return ref

    # -- comparisons ---------------------------------------------------------
    def check(self, res, ref, reduced=True):
        """Compare the step's outputs with the oracle's.  reduced=False skips
        the two-pass path's reduced-gradient buffer (for a step whose scratch
        is not the job's buffer)."""
        n, N, P = self.n, self.N, self.plan.shard_elems
        assert res.overflow == ref["overflow"], (res.overflow, ref["overflow"])
        assert res.skipped == ref["skipped"]
        assert res.t == ref["t"] == self.state.t
        assert res.new_loss_scale == ref["loss_scale"] == self.state.loss_scale
        if self.max_norm > 0:
            if ref["overflow"]:
                assert math.isinf(res.grad_norm)
            else:
                assert res.grad_norm == ref["grad_norm"], (res.grad_norm, ref["grad_norm"])
                assert res.clip_coef == ref["clip"], (res.clip_coef, ref["clip"])
        w, m, v = self.bufs.state()
        reps = N if self.stage == 0 else 1
        for r in range(reps):
            off = r * self.plan.padded_elems
            gw, gm, gv = (as_u32(t[off:off + n]) for t in (w, m, v))
            for g, o, name in ((gw, self.w, "w"), (gm, self.m, "m"), (gv, self.v, "v")):
                same = np.array_equal(g, as_u32(o))
                assert same, "%s differs (replica %d): max rel %.3g, %d elements" % (
                    name, r, max_rel(g.view(np.float32), o), int((g != as_u32(o)).sum()))
            # padding never touched
            pad = (self.plan.padded_elems - n)
            if pad:
                assert not w[off + n:off + self.plan.padded_elems].any().item()
        for r in range(N):
            if self.stage == 3:
                lo, hi = r * P, min((r + 1) * P, n)
                got = as_bits(self.bufs.params16[r][:max(hi - lo, 0)])
                assert np.array_equal(got, self.p16[lo:hi]), "param shard of rank %d differs" % r
                assert not self.bufs.params16[r][max(hi - lo, 0):].any().item()
            else:
                got = as_bits(self.bufs.params16[r][:n])
                bad = int((got != self.p16).sum())
                assert bad == 0, "params16 of rank %d: %d elements differ" % (r, bad)
                assert not self.bufs.params16[r][n:].any().item()
        if self.stage <= 1:
            for r in range(N):
                assert same16(as_bits(self.bufs.grads[r][:n]), self.h, self.dtype), "all-reduce result, rank %d" % r
        elif res.path == 1 and reduced:
            assert same16(as_bits(self.bufs.reduced[:n]), self.h, self.dtype), "reduced gradient"
