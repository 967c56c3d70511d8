"""Pins for the oracle's step arithmetic (CPU only).

Each check compares the oracle with something other than itself: library
routines (numpy's binary16 conversion, torch's bfloat16 conversion,
torch.optim.Adam, torch.nn.utils.clip_grad_norm_, math.fsum), exact integer
or rational arithmetic, closed forms, and brute force on tiny inputs.  The
last group plants mistakes into copies of the oracle's inputs and checks that
the pins catch them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle

FP16, BF16 = oracle.FP16, oracle.BF16


def _f32_from_bits(u32):
    return np.asarray(u32, np.uint32).view(np.float32)


def _interesting_floats(rng, n=400_000):
    """Random fp32 bit patterns over every exponent, plus the boundary cases
    of both 16-bit formats (ties, subnormal edges, overflow thresholds)."""
    xs = [rng.integers(0, 2 ** 32, n, dtype=np.uint64).astype(np.uint32).view(np.float32)]
    xs.append((rng.standard_normal(n) * 10.0 ** rng.integers(-9, 6, n)).astype(np.float32))
    edge = []
    # binary16 halfway points and their neighbours: (k + 0.5) ulps in every binade
    for e in range(-24, 16):
        for k in (0, 1, 2, 3, 1022, 1023, 1024, 2046, 2047):
            v = (k + 0.5) * 2.0 ** (e - 10)
            edge += [v, np.nextafter(np.float32(v), np.float32(0)), np.nextafter(np.float32(v), np.float32(np.inf))]
    edge += [65504.0, 65519.0, 65520.0, 65536.0, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26, 2.0 ** -14, 0.0, -0.0]
    # bfloat16 halfway points
    for e in range(-133, 128, 7):
        for k in (0, 1, 127, 128, 255):
            edge.append((k + 0.5) * 2.0 ** (e - 7))
    edge += [3.3895313892515355e38, 3.3961775292304086e38, float(np.finfo(np.float32).max)]
    e = np.array(edge, np.float64).astype(np.float32)
    xs += [e, -e]
    xs.append(np.array([np.inf, -np.inf, np.nan], np.float32))
    return np.concatenate(xs)


# --- 16-bit formats vs library conversions -------------------------------
def test_fp16_round_matches_numpy():
    rng = np.random.default_rng(1)
    x = _interesting_floats(rng)
    got = oracle.from_f32(x, FP16)
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(oracle.to_f32(got[nan], FP16)))


def test_bf16_round_matches_torch():
    rng = np.random.default_rng(2)
    x = _interesting_floats(rng)
    got = oracle.from_f32(x, BF16)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    nan = np.isnan(x)
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.all(np.isnan(oracle.to_f32(got[nan], BF16)))


def test_16bit_to_f32_exhaustive():
    allbits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = oracle.to_f32(allbits, FP16)
    ref = allbits.view(np.float16).astype(np.float32)
    same = (f.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(f) & np.isnan(ref))
    assert same.all()
    b = oracle.to_f32(allbits, BF16)
    refb = torch.from_numpy(allbits.view(np.int16)).view(torch.bfloat16).float().numpy()
    same = (b.view(np.uint32) == refb.view(np.uint32)) | (np.isnan(b) & np.isnan(refb))
    assert same.all()


# --- Reduction ---------------------------------------------------------------
@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("n_ranks", [1, 2, 3, 8, 64])
def test_reduce_exact_when_representable(dtype, n_ranks):
    """Gradients on a coarse grid sum exactly in fp32, so the rank-order sum
    must equal the integer sum; h must be its nearest-even 16-bit value
    (numpy/torch conversion of the exact value)."""
    rng = np.random.default_rng(3 + n_ranks)
    n = 5000
    ints = rng.integers(-200, 201, (n_ranks, n))
    vals = (ints * 2.0 ** -6).astype(np.float32)          # exactly representable in both formats
    grads = [oracle.from_f32(vals[r], dtype) for r in range(n_ranks)]
    assert all(np.array_equal(oracle.to_f32(g, dtype), vals[r]) for r, g in enumerate(grads))
    h, flag = oracle.reduce(grads, dtype)
    exact = ints.sum(axis=0) * 2.0 ** -6                   # exact in fp64 and fp32
    if dtype == FP16:
        ref = exact.astype(np.float16).view(np.uint16)
    else:
        ref = torch.from_numpy(exact).float().to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert flag == 0
    assert np.array_equal(h, ref)


def test_reduce_is_in_rank_order():
    """32768 - 32768 + 0.0002 is 0.0002 in rank order, but 0 if summed in
    reverse (0.0002 is below half an fp32 ulp of 32768)."""
    vals = [32768.0, -32768.0, 0.0002, 0.0]
    grads = [oracle.from_f32(np.array([v], np.float32), FP16) for v in vals]
    h, _ = oracle.reduce(grads, FP16)
    assert oracle.to_f32(h, FP16)[0] == np.float16(0.0002).astype(np.float32)
    h_rev, _ = oracle.reduce(grads[::-1], FP16)
    assert oracle.to_f32(h_rev, FP16)[0] == 0.0


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_overflow_flag(dtype):
    n = 1000
    big = 60000.0 if dtype == FP16 else 3.0e38
    g = [oracle.from_f32(np.full(n, big, np.float32), dtype) for _ in range(2)]
    _, flag = oracle.reduce(g, dtype)
    assert flag == 1            # the sum overflows the 16-bit range
    g = [oracle.from_f32(np.zeros(n, np.float32), dtype) for _ in range(3)]
    g[2][777] = 0x7C00 if dtype == FP16 else 0x7F80   # +inf in one rank
    h, flag = oracle.reduce(g, dtype)
    assert flag == 1 and np.isinf(oracle.to_f32(h, dtype)[777])
    g[2][777] = 0x7E00 if dtype == FP16 else 0x7FC0   # NaN
    h, flag = oracle.reduce(g, dtype)
    assert flag == 1 and np.isnan(oracle.to_f32(h, dtype)[777])
    g[2][777] = 0
    _, flag = oracle.reduce(g, dtype)
    assert flag == 0


# --- Scalars -------------------------------------------------------------
def test_bias_corrections_against_closed_form():
    for t in (1, 2, 10, 100, 1000, 20000):
        bc1, bc2 = oracle.bias_corrections(0.9, 0.999, t)
        b1, b2 = float(np.float32(0.9)), float(np.float32(0.999))
        assert abs(bc1 - (1 - b1 ** t)) <= 2e-7 * (1 - b1 ** t) + 1e-12
        assert abs(bc2 - (1 - b2 ** t)) <= 2e-7 * (1 - b2 ** t) + 1e-12
    with pytest.raises(ValueError):
        oracle.bias_corrections(0.9, 0.999, 0)


def test_inv_scale_is_mean_and_unscale():
    assert oracle.inv_scale(1024.0, 4) == 2.0 ** -12
    assert oracle.inv_scale(1.0, 8) == 0.125
    assert oracle.inv_scale(1.0, 3) == float(np.float32(1 / 3))


def test_loss_scaler_sequence():
    # dynamic: halve and skip on overflow, floor at min_scale, grow after 3 clean steps
    s, good = 1024.0, 0
    seq = []
    for ov in [1, 0, 0, 0, 0, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1, 1]:
        s, good = oracle.scaler_update(s, good, bool(ov), True, min_scale=2.0, growth_interval=3)
        seq.append(s)
    assert seq[:5] == [512.0, 512.0, 512.0, 1024.0, 1024.0]
    assert seq[5:10] == [512.0, 256.0, 128.0, 64.0, 32.0]
    assert seq[-1] == 2.0
    # static scale never changes
    assert oracle.scaler_update(8.0, 0, True, False) == (8.0, 0)
    assert oracle.scaler_update(8.0, 5, False, False, growth_interval=1) == (8.0, 6)


# --- Exact norm ------------------------------------------------------------
def _bits_random(rng, n, dtype, spread=True):
    if spread:
        x = (rng.standard_normal(n) * 10.0 ** rng.integers(-7, 4, n)).astype(np.float32)
    else:
        x = (rng.standard_normal(n) * 1e-3).astype(np.float32)
    return oracle.from_f32(x, dtype)


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_exact_sumsq_brute_force(dtype):
    rng = np.random.default_rng(5)
    for n in (1, 2, 17, 300):
        h = _bits_random(rng, n, dtype)
        if dtype == FP16:
            h[0] = 0x0001            # smallest subnormal
            h[-1] = 0x7BFF           # largest finite
        ref = sum(Fraction(float(x)) ** 2 for x in oracle.to_f32(h, dtype))
        assert oracle.sumsq_fraction(h, dtype) == ref
        assert oracle.exact_sumsq(h, dtype) == float(ref)   # correctly rounded


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_exact_sumsq_large(dtype):
    rng = np.random.default_rng(6)
    h = _bits_random(rng, 200_000, dtype)
    assert oracle.exact_sumsq(h, dtype) == float(oracle.sumsq_fraction(h, dtype))
    h[5] = 0x7C00 if dtype == FP16 else 0x7F80
    assert math.isfinite(oracle.exact_sumsq(h, dtype))    # non-finite elements skipped


def test_clip_coefficient_matches_torch():
    rng = np.random.default_rng(7)
    for scale in (1e-3, 1e-1, 1.0, 10.0):
        h = _bits_random(rng, 5000, FP16, spread=False)
        inv = oracle.inv_scale(1.0, 4)
        g = oracle.to_f32(h, FP16).astype(np.float64) * inv * scale
        h2 = oracle.from_f32(g.astype(np.float32) / np.float32(inv), FP16)
        norm = oracle.grad_norm(oracle.exact_sumsq(h2, FP16), inv)
        c = oracle.clip_coef(norm, 1.0)
        t = torch.from_numpy(oracle.to_f32(h2, FP16).astype(np.float64) * inv).requires_grad_()
        t.grad = t.detach().clone()
        before = t.grad.clone()
        tn = torch.nn.utils.clip_grad_norm_([t], 1.0)
        assert abs(float(tn) - norm) <= 1e-12 * norm
        ratio = (t.grad / before)[before != 0]
        assert abs(float(ratio.mean()) - c) <= 1e-6 * c


# --- Adam ----------------------------------------------------------------
def _run_oracle_steps(grads_per_step, w0, *, lr, beta1, beta2, eps, loss_scale, dtype=FP16, max_norm=0.0):
    w = w0.copy()
    m = np.zeros_like(w)
    v = np.zeros_like(w)
    t = 0
    outs = []
    for grads in grads_per_step:
        r = oracle.step(grads, w, m, v, dtype=dtype, lr=lr, beta1=beta1, beta2=beta2, eps=eps,
                        t=t, loss_scale=loss_scale, max_grad_norm=max_norm)
        t = r["t"]
        outs.append(r)
    return w, m, v, outs


def _torch_adam(grad_list, w0, *, lr, beta1, beta2, eps):
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.Adam([p], lr=lr, betas=(beta1, beta2), eps=eps, foreach=False, fused=False)
    for g in grad_list:
        p.grad = torch.from_numpy(np.ascontiguousarray(g, np.float32))
        opt.step()
    st = opt.state[p]
    return p.detach().numpy(), st["exp_avg"].numpy(), st["exp_avg_sq"].numpy()


def _close(a, b, rel=1e-6, floor=0.0):
    a = a.astype(np.float64)
    b = b.astype(np.float64)
    return np.all(np.abs(a - b) <= rel * np.maximum(np.abs(b), floor))


def _close_w(w, ref, w0, steps, rel=1e-6):
    """Weights: relative to the operands' magnitude.  w' = w - lr*u may cancel
    towards zero, so rounding differences are a few ulps of the operands, not
    of the result; an Adam step moves a weight by about lr, so the operands
    stay below |w0| + steps*lr."""
    w, ref, w0 = (x.astype(np.float64) for x in (w, ref, w0))
    scale = np.maximum(np.abs(ref), np.abs(w0) + steps * ADAM["lr"])
    return np.all(np.abs(w - ref) <= rel * scale)


ADAM = dict(lr=1e-4, beta1=float(np.float32(0.9)), beta2=float(np.float32(0.999)), eps=1e-8)


def _grads(rng, n_ranks, n, sigma, scale, dtype=FP16):
    return [oracle.from_f32((rng.standard_normal(n) * sigma * scale).astype(np.float32), dtype)
            for _ in range(n_ranks)]


@pytest.mark.parametrize("n_ranks,loss_scale", [(1, 1.0), (1, 1024.0), (4, 1024.0), (8, 1.0)])
def test_adam_matches_torch(n_ranks, loss_scale):
    """Five steps against torch.optim.Adam fed the mean unscaled gradient
    h/(S*N) of each step (h recomputed here in numpy: fp32 rank-order sum,
    numpy's binary16 rounding)."""
    rng = np.random.default_rng(10 + n_ranks)
    n = 4000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    steps = [_grads(rng, n_ranks, n, 1e-3, loss_scale) for _ in range(5)]
    # include gradients comparable to eps, where a dropped eps shows
    steps[0][0][:50] = oracle.from_f32(np.full(50, 3e-9 * loss_scale, np.float32), FP16)
    w, m, v, _ = _run_oracle_steps(steps, w0, loss_scale=loss_scale, **ADAM)
    tg = []
    for grads in steps:
        s = np.zeros(n, np.float32)
        for g in grads:
            s = s + g.view(np.float16).astype(np.float32)
        h = s.astype(np.float16).astype(np.float64)
        tg.append((h / (loss_scale * n_ranks)).astype(np.float32))
    tw, tm, tv = _torch_adam(tg, w0, **ADAM)
    assert _close_w(w, tw, w0, len(steps))
    # m averages signed gradients and may cancel: scale by max |g| seen
    gmax = np.max(np.abs(np.stack(tg)), axis=0)
    assert _close(m, tm, 1e-6, floor=gmax)
    assert _close(v, tv, 1e-6, floor=1e-30)


def test_adam_first_step_closed_form():
    """t = 1 from m = v = 0: m' = (1-b1) g, v' = (1-b2) g^2, and the update is
    lr * g / (|g| + eps)."""
    rng = np.random.default_rng(20)
    n = 3000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = _grads(rng, 4, n, 1e-3, 1024.0)
    w, m, v, outs = _run_oracle_steps([grads], w0, loss_scale=1024.0, **ADAM)
    g = oracle.to_f32(outs[0]["h"], FP16).astype(np.float64) / (1024.0 * 4)
    assert _close(m, (1 - ADAM["beta1"]) * g, 1e-6, floor=1e-15)
    assert _close(v, (1 - ADAM["beta2"]) * g * g, 1e-6, floor=1e-25)
    expect = w0.astype(np.float64) - ADAM["lr"] * g / (np.abs(g) + ADAM["eps"])
    assert _close_w(w, expect, w0, 1)
    assert np.array_equal(outs[0]["p16"], w.astype(np.float16).view(np.uint16))


def test_zero_gradient_leaves_weights():
    rng = np.random.default_rng(21)
    w0 = (rng.standard_normal(500) * 0.02).astype(np.float32)
    zeros = [np.zeros(500, np.uint16) for _ in range(3)]
    w, m, v, outs = _run_oracle_steps([zeros, zeros], w0, loss_scale=1.0, **ADAM)
    assert np.array_equal(w, w0) and not m.any() and not v.any()
    assert outs[-1]["t"] == 2


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_overflow_leaves_state_bit_identical(dtype):
    rng = np.random.default_rng(22)
    n = 1000
    w = (rng.standard_normal(n) * 0.02).astype(np.float32)
    m = (rng.standard_normal(n) * 1e-4).astype(np.float32)
    v = (rng.standard_normal(n) * 1e-4).astype(np.float32) ** 2
    w0, m0, v0 = w.copy(), m.copy(), v.copy()
    grads = _grads(rng, 2, n, 1e-3, 1.0, dtype)
    grads[1][10] = 0x7C00 if dtype == FP16 else 0x7F80
    r = oracle.step(grads, w, m, v, dtype=dtype, t=7, loss_scale=1024.0, dynamic=True, max_grad_norm=1.0, **ADAM)
    assert r["overflow"] == 1 and r["skipped"] == 1 and r["t"] == 7
    assert r["loss_scale"] == 512.0 and r["grad_norm"] == math.inf
    assert np.array_equal(w, w0) and np.array_equal(m, m0) and np.array_equal(v, v0)
    assert np.array_equal(r["p16"], oracle.from_f32(w0, dtype))


def test_clipped_step_matches_torch():
    """Clipping at 1.0 with gradients whose norm is far above 1: torch's
    clip_grad_norm_ followed by torch.optim.Adam."""
    rng = np.random.default_rng(23)
    n = 4000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    steps = [_grads(rng, 2, n, 0.05, 1.0) for _ in range(3)]
    w, m, v, outs = _run_oracle_steps(steps, w0, loss_scale=1.0, max_norm=1.0, **ADAM)
    assert all(r["clip"] < 1.0 for r in outs)
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.Adam([p], lr=ADAM["lr"], betas=(ADAM["beta1"], ADAM["beta2"]), eps=ADAM["eps"], foreach=False)
    for grads in steps:
        s = np.zeros(n, np.float32)
        for g in grads:
            s = s + g.view(np.float16).astype(np.float32)
        h = s.astype(np.float16).astype(np.float64)
        p.grad = torch.from_numpy(h / 2.0).float()
        torch.nn.utils.clip_grad_norm_([p], 1.0)
        opt.step()
    assert _close_w(w, p.detach().numpy(), w0, len(steps))


# --- Planted mistakes: each must be caught by a pin above --------------------
def _adam_vs_torch_error(mutate):
    """Run one oracle step with a mutated hyper-parameter record and return
    the max relative error against torch.optim.Adam."""
    rng = np.random.default_rng(30)
    n = 2000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = _grads(rng, 4, n, 1e-3, 1024.0)
    h, _ = oracle.reduce(grads, FP16)
    errs = []
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    gl = []
    for t in (1, 2, 3):
        hyper = oracle.make_hyper(inv=oracle.inv_scale(1024.0, 4), clip=None, t=t, **ADAM)
        mutate(hyper, t)
        oracle.adam(h, FP16, hyper, w, m, v)
        gl.append((oracle.to_f32(h, FP16).astype(np.float64) / 4096.0).astype(np.float32))
    tw, tm, tv = _torch_adam(gl, w0, **ADAM)
    gmax = np.max(np.abs(np.stack(gl)), axis=0)
    for a, b, s in ((w, tw, np.abs(w0) + 3 * ADAM["lr"]), (m, tm, gmax), (v, tv, 0)):
        d = np.abs(a.astype(np.float64) - b) / np.maximum(np.maximum(np.abs(b), s), 1e-30)
        errs.append(float(d.max()))
    return max(errs)


def test_planted_mistakes_are_caught():
    assert _adam_vs_torch_error(lambda h, t: None) <= 1e-6

    def swap_betas(h, t):
        h.beta1, h.beta2 = h.beta2, h.beta1
        h.one_minus_beta1, h.one_minus_beta2 = h.one_minus_beta2, h.one_minus_beta1

    def stale_bias_correction(h, t):
        if t > 1:
            h.bc1, h.bc2 = oracle.bias_corrections(ADAM["beta1"], ADAM["beta2"], t - 1)

    def sum_not_mean(h, t):
        h.inv_scale = np.float32(1 / 1024.0)

    def no_bias_correction(h, t):
        h.bc1 = h.bc2 = 1.0

    def wrong_sign(h, t):
        h.lr = -h.lr

    for mutate in (swap_betas, stale_bias_correction, sum_not_mean, no_bias_correction, wrong_sign):
        assert _adam_vs_torch_error(mutate) > 1e-4, mutate.__name__


def test_planted_reduce_mistakes_are_caught():
    """Dropping or duplicating a rank's contribution breaks the exact-sum pin."""
    rng = np.random.default_rng(31)
    ints = rng.integers(-100, 101, (4, 3000))
    vals = (ints * 2.0 ** -6).astype(np.float32)
    grads = [oracle.from_f32(vals[r], FP16) for r in range(4)]
    ref = (ints.sum(axis=0) * 2.0 ** -6).astype(np.float16).view(np.uint16)
    assert np.array_equal(oracle.reduce(grads, FP16)[0], ref)
    dropped = oracle.reduce(grads[:3], FP16)[0]
    duplicated = oracle.reduce(grads + grads[:1], FP16)[0]
    assert not np.array_equal(dropped, ref)
    assert not np.array_equal(duplicated, ref)


# --- SGD variants (the other optimizers of the (2b+K) accounting) -----------
@pytest.mark.parametrize("momentum", [0.0, 0.9])
@pytest.mark.parametrize("n_ranks,loss_scale", [(1, 1.0), (4, 1024.0)])
def test_sgd_matches_torch(momentum, n_ranks, loss_scale):
    rng = np.random.default_rng(40 + n_ranks)
    n = 3000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    steps = [_grads(rng, n_ranks, n, 1e-3, loss_scale) for _ in range(5)]
    w, m = w0.copy(), np.zeros(n, np.float32)
    v = np.zeros(n, np.float32)
    opt_name = "sgdm" if momentum else "sgd"
    t = 0
    for grads in steps:
        r = oracle.step(grads, w, m, v, dtype=FP16, t=t, loss_scale=loss_scale, optimizer=opt_name,
                        momentum=momentum, **ADAM)
        t = r["t"]
    assert not v.any()                                   # SGD keeps no variance
    if not momentum:
        assert not m.any()
    p = torch.nn.Parameter(torch.from_numpy(w0.copy()))
    opt = torch.optim.SGD([p], lr=ADAM["lr"], momentum=float(np.float32(momentum)), foreach=False)
    for grads in steps:
        s = np.zeros(n, np.float32)
        for g in grads:
            s = s + g.view(np.float16).astype(np.float32)
        h = s.astype(np.float16).astype(np.float64)
        p.grad = torch.from_numpy((h / (loss_scale * n_ranks)).astype(np.float32))
        opt.step()
    assert _close_w(w, p.detach().numpy(), w0, len(steps))
    if momentum:
        buf = opt.state[p]["momentum_buffer"].numpy()
        assert np.allclose(m, buf, rtol=1e-6, atol=1e-12)


def test_sgd_closed_form_and_planted_mistakes():
    """Plain SGD: w' = w - lr*g in one step; a wrong sign or a dropped
    unscale is caught."""
    rng = np.random.default_rng(44)
    n = 2000
    w0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    grads = _grads(rng, 2, n, 1e-3, 8.0)
    w, m, v = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    r = oracle.step(grads, w, m, v, dtype=FP16, t=0, loss_scale=8.0, optimizer="sgd", **ADAM)
    g = oracle.to_f32(r["h"], FP16).astype(np.float64) / 16.0
    assert _close_w(w, w0 - ADAM["lr"] * g, w0, 1)
    h, _ = oracle.reduce(grads, FP16)
    for mutate in (lambda hp: setattr(hp, "lr", -hp.lr), lambda hp: setattr(hp, "inv_scale", 1.0)):
        hp = oracle.make_hyper(inv=oracle.inv_scale(8.0, 2), clip=None, lr=ADAM["lr"], beta1=0.0, beta2=0.0,
                               eps=0.0, t=1)
        mutate(hp)
        wm = w0.copy()
        oracle.sgd(h, FP16, hp, wm)
        assert not _close_w(wm, w0 - ADAM["lr"] * g, w0, 1)
