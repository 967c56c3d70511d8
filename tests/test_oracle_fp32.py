"""Pins for the oracle's fp32-training variant (CPU only): parameters and
gradients in binary32 (b = 4 bytes, the pages' fp32 SGD / SGD-with-momentum
worked examples), the same step otherwise.

What fixes it: numpy's own binary32 bit patterns (the values pass through
unchanged), sums that must or must not round (a 16-bit rounding, or another
summation order, fails them), torch.optim.SGD / torch.optim.Adam on fp32
parameters, exact rational sums of squares, and byte counts per array."""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests.test_oracle_step import ADAM, _close, _close_w, _torch_adam

FP32 = oracle.FP32


def _bits(x):
    return np.ascontiguousarray(x, np.float32).view(np.uint32)


def _grads32(rng, n_ranks, n, sigma, scale):
    return [_bits(rng.standard_normal(n) * sigma * scale) for _ in range(n_ranks)]


def test_values_pass_through_unchanged():
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2 ** 32, 100_000, dtype=np.uint64).astype(np.uint32)
    f = oracle.to_f32(u, FP32)
    assert np.array_equal(f.view(np.uint32), u)        # NaN payloads included
    assert np.array_equal(oracle.from_f32(f, FP32), u)
    x = rng.standard_normal(1000).astype(np.float32)
    assert np.array_equal(oracle.cast16(x, FP32), x.view(np.uint32))
    with pytest.raises(TypeError):
        oracle.to_f32(u.astype(np.uint16), FP32)


def test_reduce_keeps_fp32_and_rank_order():
    """2^-24 + 2^-24 + 1 = 1 + 2^-23 exactly in rank order (a binary32 value,
    which neither 16-bit format holds); 1 + 2^-24 + 2^-24 rounds twice to even
    and gives 1."""
    up = [_bits([2.0 ** -24]), _bits([2.0 ** -24]), _bits([1.0])]
    h, flag = oracle.reduce(up, FP32)
    assert flag == 0 and h.dtype == np.uint32
    assert h.view(np.float32)[0] == np.float32(1.0 + 2.0 ** -23)
    h, _ = oracle.reduce(up[::-1], FP32)
    assert h.view(np.float32)[0] == np.float32(1.0)


@pytest.mark.parametrize("n_ranks", [1, 3, 64])
def test_reduce_exact_on_a_grid(n_ranks):
    rng = np.random.default_rng(5 + n_ranks)
    ints = rng.integers(-(2 ** 14), 2 ** 14, (n_ranks, 4000))
    vals = ints * 2.0 ** -20                      # partial sums stay below 2^24 units: exact in fp32
    h, flag = oracle.reduce([_bits(v) for v in vals], FP32)
    assert flag == 0
    assert np.array_equal(h.view(np.float32).astype(np.float64), ints.sum(axis=0) * 2.0 ** -20)


def test_overflow_flag():
    n = 100
    g = [_bits(np.full(n, 3.0e38)) for _ in range(2)]
    _, flag = oracle.reduce(g, FP32)
    assert flag == 1
    g = [_bits(np.zeros(n)) for _ in range(3)]
    g[1][17] = 0x7F800000
    h, flag = oracle.reduce(g, FP32)
    assert flag == 1 and np.isinf(h.view(np.float32)[17])
    g[1][17] = 0x7FC00000
    h, flag = oracle.reduce(g, FP32)
    assert flag == 1 and np.isnan(h.view(np.float32)[17])
    g[1][17] = 0
    assert oracle.reduce(g, FP32)[1] == 0
    # an overflowed step leaves every state array and the model copy as they were
    rng = np.random.default_rng(2)
    w0 = rng.standard_normal(n).astype(np.float32)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    g[2][5] = 0x7F800000
    r = oracle.step(g, w, m, v, dtype=FP32, t=3, loss_scale=64.0, dynamic=True, optimizer="sgdm", momentum=0.9,
                    **ADAM)
    assert r["overflow"] == 1 and r["t"] == 3 and r["loss_scale"] == 32.0
    assert np.array_equal(w, w0) and not m.any() and np.array_equal(r["p16"], w0.view(np.uint32))


def _torch_grads(steps, n_ranks, loss_scale):
    out = []
    for grads in steps:
        s = np.zeros(grads[0].size, np.float32)
        for g in grads:
            s = s + g.view(np.float32)
        out.append((s.astype(np.float64) / (loss_scale * n_ranks)).astype(np.float32))
    return out


@pytest.mark.parametrize("momentum", [0.0, 0.9])
@pytest.mark.parametrize("n_ranks,loss_scale", [(1, 1.0), (4, 1024.0)])
def test_sgd_matches_torch(momentum, n_ranks, loss_scale):
    rng = np.random.default_rng(60 + n_ranks)
    n = 3000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    steps = [_grads32(rng, n_ranks, n, 1e-3, loss_scale) for _ in range(5)]
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    t = 0
    for grads in steps:
        r = oracle.step(grads, w, m, v, dtype=FP32, t=t, loss_scale=loss_scale,
                        optimizer="sgdm" if momentum else "sgd", momentum=momentum, **ADAM)
        t = r["t"]
        assert np.array_equal(r["p16"], w.view(np.uint32))     # the model copy is the master itself
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.SGD([p], lr=ADAM["lr"], momentum=float(np.float32(momentum)), foreach=False)
    for g in _torch_grads(steps, n_ranks, loss_scale):
        p.grad = torch.from_numpy(g)
        opt.step()
    assert _close_w(w, p.detach().numpy(), w0, len(steps))
    if momentum:
        assert np.allclose(m, opt.state[p]["momentum_buffer"].numpy(), rtol=1e-6, atol=1e-12)


@pytest.mark.parametrize("n_ranks,loss_scale", [(1, 1.0), (8, 256.0)])
def test_adam_matches_torch(n_ranks, loss_scale):
    rng = np.random.default_rng(70 + n_ranks)
    n = 3000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    steps = [_grads32(rng, n_ranks, n, 1e-3, loss_scale) for _ in range(4)]
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    t = 0
    for grads in steps:
        r = oracle.step(grads, w, m, v, dtype=FP32, t=t, loss_scale=loss_scale, **ADAM)
        t = r["t"]
    tg = _torch_grads(steps, n_ranks, loss_scale)
    tw, tm, tv = _torch_adam(tg, w0, **ADAM)
    assert _close_w(w, tw, w0, len(steps))
    assert _close(m, tm, 1e-6, floor=np.max(np.abs(np.stack(tg)), axis=0))
    assert _close(v, tv, 1e-6, floor=1e-30)


def test_exact_sumsq_brute_force():
    rng = np.random.default_rng(9)
    x = np.concatenate([rng.standard_normal(3000) * 10.0 ** rng.integers(-30, 30, 3000),
                        [2.0 ** -149, -(2.0 ** -149), 3.0e38, 0.0]]).astype(np.float32)
    h = _bits(x).copy()
    exact = sum((Fraction(float(v)) ** 2 for v in x), Fraction(0))
    assert oracle.sumsq_fraction(h, FP32) == exact
    assert oracle.exact_sumsq(h, FP32) == float(exact)        # correctly rounded
    h[7] = 0x7F800000                                          # non-finite elements are left out
    assert oracle.sumsq_fraction(h, FP32) == exact - Fraction(float(x[7])) ** 2


def test_hbm_bytes_with_fp32_values():
    """Counting each access once, with 4-byte gradients and parameters."""
    for N in (1, 8, 64):
        # stage 2 fused: read N grads, read and write the state, write N params
        assert oracle.hbm_bytes_per_param(N, 2, "fused", 12, 4) == 4 * N + 24 + 4 * N
        # stage 0 fused: grads read and written back on every rank, N replicas updated
        assert oracle.hbm_bytes_per_param(N, 0, "fused", 8, 4) == N * (4 + 4 + 16 + 4)
        # stage 3 two-pass: grads, reduced written and read twice over two passes, owner's param
        assert oracle.hbm_bytes_per_param(N, 3, "two_pass", 4, 4) == 4 * N + 4 + 4 + 8 + 4
        assert oracle.hbm_bytes_per_param(N, 1, "restore", 12, 4) == 4 + 4 * N
        for stage in range(4):
            for mode in ("fused", "two_pass", "restore"):
                # 16-bit defaults unchanged
                assert oracle.hbm_bytes_per_param(N, stage, mode, 12) == \
                    oracle.hbm_bytes_per_param(N, stage, mode, 12, 2)
