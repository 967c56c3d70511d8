"""GPU parity at the workloads' full sizes, in the launch configurations that
bench.py times, on about 2^20 sampled elements per test that the oracle
recomputes from the host generator (plus properties that hold at any size).

  * 48-layer d=1600 list (1,555,278,400 params), N_d = 8, bucket 5e8, dynamic
    loss scale: an overflowed step (one inf per 1e9 gradient elements), then a
    clean one.
  * 32-layer d=4096 list (6,648,827,904 params), stage 3, N_d = 64, bucket
    2^24, gradients staged per bucket, layer gathers; and the same step as
    the default benchmark runs it (gradients from the ring of pre-generated
    sets, device-state protocol, two gathers per layer).
  * 2^31 flat params, N_d = 32, bf16, clipping path with c < 1, staged
    gradients; the exact norm over all 2^31 reduced values.
  * 2^28 flat params, N_d = 2, fp16 and bf16, clipping: pass 1 on the
    staged kernel (packed sums, the bfloat16 window tested two values per
    word); the exact norm over all 2^28 reduced values.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_mixed_bucket_gb300 as zg
from tests.gpu_harness import as_u16, as_u32

pytestmark = pytest.mark.gpu

ADAM = dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8)


def transformer_layers(vocab, d, layers):
    return [vocab * d] + [12 * d * d + 4 * d] * layers


def _samples(n, extra, k=1 << 20, seed=7):
    rng = np.random.default_rng(seed)
    idx = np.concatenate([rng.integers(0, n, k), np.array([i for i in extra if 0 <= i < n], np.int64)])
    return np.unique(idx)


def _at(t, idx):
    return t.index_select(0, torch.from_numpy(idx).to(t.device))


@pytest.fixture(autouse=True)
def _free_memory():
    torch.cuda.empty_cache()
    yield
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


def test_cfg3_overflow_then_clean():
    layers = transformer_layers(50257, 1600, 48)
    n, N, B = sum(layers), 8, 500_000_000
    assert n == 1_555_278_400
    s = torch.cuda.current_stream()
    cfg = zg.Config(n, N, 2, B, 0, layers)
    plan = zg.zero_plan(cfg)
    bufs = zg.DeviceBuffers(cfg, plan, device="cuda")
    synth.dev_normal32(bufs.w[0].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT, cuda_stream=s.cuda_stream)
    # every rank's 16-bit parameters start as the cast of the master weights
    # (torch's binary32 -> binary16 conversion rounds to nearest even)
    p16 = bufs.w[0][:n].to(torch.float16).view(torch.int16)
    for r in range(N):
        bufs.params16[r][:n].copy_(p16)
    del p16
    adam = zg.zero_adam_t(max_grad_norm=0.0, **ADAM)
    state = zg.zero_state_t(t=0, loss_scale=1024.0, min_loss_scale=1.0, dynamic=1)
    inj = synth.inf_positions(n, N, seed=0, step=1)
    assert len(inj) >= 12
    idx = _samples(n, [e for _, e in inj] + [0, n - 1, B - 1, B, 3 * B])
    w0 = synth.host_normal32_at(idx, 0.02, seed=0, stream=synth.STREAM_WEIGHT)
    # step 1: gradients x 1024 with the injected infs -> skipped
    for r in range(N):
        synth.dev_normal16(bufs.grads[r].data_ptr(), n, synth.FP16, 1e-3 * 1024.0, seed=0, stream=synth.STREAM_GRAD,
                           step=1, rank=r, cuda_stream=s.cuda_stream)
    for r, e in inj:
        bufs.grads[r][e] = synth.inf_bits(synth.FP16)
    res = zg.zero_step_stage2(cfg, plan, bufs, adam, state, s)
    torch.cuda.synchronize()
    assert res.overflow == 1 and res.skipped == 1 and res.t == 0 and res.new_loss_scale == 512.0
    w, m, v = bufs.state()
    assert np.array_equal(as_u32(_at(w, idx)), as_u32(w0))
    assert not _at(m, idx).any().item() and not _at(v, idx).any().item()
    p_restored = oracle.cast16(w0, oracle.FP16)
    for r in (0, 5, 7):
        assert np.array_equal(as_u16(_at(bufs.params16[r], idx)), p_restored)
    # step 2: clean gradients at the halved scale
    for r in range(N):
        synth.dev_normal16(bufs.grads[r].data_ptr(), n, synth.FP16, 1e-3 * 512.0, seed=0, stream=synth.STREAM_GRAD,
                           step=2, rank=r, cuda_stream=s.cuda_stream)
    res = zg.zero_step_stage2(cfg, plan, bufs, adam, state, s)
    torch.cuda.synchronize()
    assert res.overflow == 0 and res.t == 1
    grads = [synth.host_normal16_at(idx, synth.FP16, 1e-3 * 512.0, seed=0, stream=synth.STREAM_GRAD, step=2, rank=r)
             for r in range(N)]
    wr, mr, vr = w0.copy(), np.zeros_like(w0), np.zeros_like(w0)
    ref = oracle.step(grads, wr, mr, vr, dtype=oracle.FP16, t=0, loss_scale=512.0, dynamic=True, **ADAM)
    assert ref["overflow"] == 0
    w, m, v = bufs.state()
    assert np.array_equal(as_u32(_at(w, idx)), as_u32(wr))
    assert np.array_equal(as_u32(_at(m, idx)), as_u32(mr))
    assert np.array_equal(as_u32(_at(v, idx)), as_u32(vr))
    for r in range(N):
        assert np.array_equal(as_u16(_at(bufs.params16[r], idx)), ref["p16"])


def test_cfg4_stage3_staged_with_gathers():
    layers = transformer_layers(50257, 4096, 32)
    n, N, B = sum(layers), 64, 1 << 24
    assert n == 6_648_827_904
    s = torch.cuda.current_stream()
    cfg = zg.Config(n, N, 3, B, 0, layers)
    plan = zg.zero_plan(cfg)
    bufs = zg.DeviceBuffers(cfg, plan, device="cuda", grads=False, reduced=False)
    synth.dev_normal32(bufs.w[0].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT, cuda_stream=s.cuda_stream)
    staging = [torch.empty(B, dtype=torch.int16, device="cuda") for _ in range(N)]
    S = 1024.0
    adam = zg.zero_adam_t(max_grad_norm=0.0, **ADAM)
    state = zg.zero_state_t(t=0, loss_scale=S, min_loss_scale=1.0)
    zg.zero_step_begin(cfg, plan, bufs, adam, state, s)
    for b in reversed(range(plan.n_buckets)):          # backward order
        lo, hi = b * B, min((b + 1) * B, n)
        for r in range(N):
            synth.dev_normal16(staging[r].data_ptr(), hi - lo, synth.FP16, 1e-3 * S, seed=0,
                               stream=synth.STREAM_GRAD, step=1, rank=r, offset=lo, cuda_stream=s.cuda_stream)
        zg.zero_step_bucket(cfg, plan, bufs, adam, state, b, [t.data_ptr() for t in staging], s)
    res = zg.zero_step_end(cfg, plan, bufs, adam, state, s)
    torch.cuda.synchronize()
    assert res.overflow == 0 and res.t == 1
    P = plan.shard_elems
    idx = _samples(n, [0, n - 1, P - 1, P, 63 * P, B - 1, B])
    grads = [synth.host_normal16_at(idx, synth.FP16, 1e-3 * S, seed=0, stream=synth.STREAM_GRAD, step=1, rank=r)
             for r in range(N)]
    w = synth.host_normal32_at(idx, 0.02, seed=0, stream=synth.STREAM_WEIGHT)
    m, v = np.zeros_like(w), np.zeros_like(w)
    ref = oracle.step(grads, w, m, v, dtype=oracle.FP16, t=0, loss_scale=S, **ADAM)
    gw, gm, gv = bufs.state()
    assert np.array_equal(as_u32(_at(gw, idx)), as_u32(w))
    assert np.array_equal(as_u32(_at(gm, idx)), as_u32(m))
    assert np.array_equal(as_u32(_at(gv, idx)), as_u32(v))
    # each sampled element's 16-bit value sits in its owner's shard
    owners = idx // P
    for o in np.unique(owners):
        sel = owners == o
        got = as_u16(_at(bufs.params16[int(o)], idx[sel] - o * P))
        assert np.array_equal(got, ref["p16"][sel]), int(o)
    # gather the embedding and the last block into 3 destinations; compare the sampled part
    dst = [torch.zeros(plan.max_layer_elems, dtype=torch.int16, device="cuda") for _ in range(3)]
    starts = np.cumsum([0] + layers)
    for l in (0, len(layers) - 1):
        zg.zero_gather_layer(cfg, plan, l, [t.data_ptr() for t in bufs.params16], [d.data_ptr() for d in dst], s)
        torch.cuda.synchronize()
        sel = (idx >= starts[l]) & (idx < starts[l + 1])
        assert sel.any()
        for d in dst:
            assert np.array_equal(as_u16(_at(d, idx[sel] - starts[l])), ref["p16"][sel])


def test_cfg4_as_the_benchmark_runs_it():
    """The default benchmark's stage-3 step exactly as bench.py times it
    (bench_workloads.Stage3Job: the device-state protocol, two gathers per
    layer into 64 constant-size buffers, each bucket's 64 gradient copies
    from the ring of pre-generated sets), two steps.  Sampled elements
    against the oracle, which regenerates each sampled element's gradients
    from the ring set its bucket reads; the 64 gather buffers hold layer 0
    as gathered by the second step's backward pass, i.e. after step 1."""
    import bench_workloads as bw
    job = bw.Stage3Job(torch.device("cuda", 0), ring=4)
    n, N, B, S = job.n, job.N, job.B, job.S
    assert n == 6_648_827_904 and N == 64 and B == 1 << 24
    for _ in range(2):
        job.step()
    st, last = zg.zero_dev_state_read(job.dev_state, job.stream)
    assert st.t == 2 and last.overflow == 0 and last.skipped == 0
    P = job.plan.shard_elems
    idx = _samples(n, [0, n - 1, P - 1, P, 63 * P, B - 1, B, 3 * B, 4 * B - 1, job.starts[1], job.starts[1] - 1])
    sets = (idx // B) % len(job.ring)
    grads = []
    for r in range(N):
        g = np.empty(idx.size, np.uint16)
        for k in range(len(job.ring)):
            sel = sets == k
            g[sel] = synth.host_normal16_at(idx[sel] % B, synth.FP16, 1e-3 * S, seed=0, stream=synth.STREAM_GRAD,
                                            step=k + 1, rank=r)
        grads.append(g)
    w = synth.host_normal32_at(idx, 0.02, seed=0, stream=synth.STREAM_WEIGHT)
    m, v = np.zeros_like(w), np.zeros_like(w)
    ref1 = oracle.step(grads, w, m, v, dtype=oracle.FP16, t=0, loss_scale=S, **ADAM)
    ref2 = oracle.step(grads, w, m, v, dtype=oracle.FP16, t=1, loss_scale=S, **ADAM)
    assert ref1["overflow"] == 0 and ref2["overflow"] == 0 and ref2["t"] == 2
    gw, gm, gv = job.bufs.state()
    assert np.array_equal(as_u32(_at(gw, idx)), as_u32(w))
    assert np.array_equal(as_u32(_at(gm, idx)), as_u32(m))
    assert np.array_equal(as_u32(_at(gv, idx)), as_u32(v))
    owners = idx // P
    for o in np.unique(owners):
        sel = owners == o
        got = as_u16(_at(job.bufs.params16[int(o)], idx[sel] - o * P))
        assert np.array_equal(got, ref2["p16"][sel]), int(o)
    sel = idx < job.starts[1]
    assert sel.sum() > 1000
    for d in (0, 31, 63):
        assert np.array_equal(as_u16(_at(job.dst[d], idx[sel])), ref1["p16"][sel]), d


def test_sweep_2p31_n32_bf16_clip_path():
    """Clipping on (max norm 1.0 against a norm near 8: c < 1), two steps.
    The exact norm is checked over all 2^31 reduced values (the oracle's
    integer exponent bins of the GPU's reduced gradient, bit for bit); the
    clip coefficient must be the oracle's from that norm; sampled elements
    follow the oracle's clipped Adam from gradients the oracle regenerates
    and reduces itself."""
    n, N, B = 1 << 31, 32, 1 << 24
    s = torch.cuda.current_stream()
    cfg = zg.Config(n, N, 2, B, 0, None, zg.ZERO_BF16)
    plan = zg.zero_plan(cfg)
    bufs = zg.DeviceBuffers(cfg, plan, device="cuda", grads=False, shadow=False)
    synth.dev_normal32(bufs.w[0].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT, cuda_stream=s.cuda_stream)
    staging = [torch.empty(B, dtype=torch.int16, device="cuda") for _ in range(N)]
    max_norm = 1.0
    adam = zg.zero_adam_t(max_grad_norm=max_norm, **ADAM)
    state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
    idx = _samples(n, [0, n - 1, B - 1, B, n // 2])
    w = synth.host_normal32_at(idx, 0.02, seed=0, stream=synth.STREAM_WEIGHT)
    m, v = np.zeros_like(w), np.zeros_like(w)
    inv = oracle.inv_scale(1.0, N)
    for step in (1, 2):
        zg.zero_step_begin(cfg, plan, bufs, adam, state, s)
        for b in range(plan.n_buckets):
            lo, hi = b * B, min((b + 1) * B, n)
            for r in range(N):
                synth.dev_normal16(staging[r].data_ptr(), hi - lo, synth.BF16, 1e-3, seed=0,
                                   stream=synth.STREAM_GRAD, step=step, rank=r, offset=lo, cuda_stream=s.cuda_stream)
            zg.zero_step_bucket(cfg, plan, bufs, adam, state, b, [t.data_ptr() for t in staging], s)
        res = zg.zero_step_end(cfg, plan, bufs, adam, state, s)
        torch.cuda.synchronize()
        assert res.overflow == 0 and res.path == 1 and res.t == step
        # the exact norm over the whole reduced gradient
        h_all = bufs.reduced[:n].cpu().numpy().view(np.uint16)
        norm = oracle.grad_norm(float(oracle.sumsq_fraction(h_all, oracle.BF16)), inv)
        del h_all
        assert res.grad_norm == norm, (res.grad_norm, norm)
        c = oracle.clip_coef(norm, max_norm)
        assert 0.0 < c < 1.0 and res.clip_coef == c
        # sampled trajectories: the oracle reduces the regenerated gradients itself
        grads = [synth.host_normal16_at(idx, synth.BF16, 1e-3, seed=0, stream=synth.STREAM_GRAD, step=step, rank=r)
                 for r in range(N)]
        h, flag = oracle.reduce(grads, oracle.BF16)
        assert flag == 0
        assert np.array_equal(as_u16(_at(bufs.reduced, idx)), h)
        hyper = oracle.make_hyper(inv=inv, clip=c, t=step, **ADAM)
        p16 = oracle.adam(h, oracle.BF16, hyper, w, m, v)
        gw, gm, gv = bufs.state()
        assert np.array_equal(as_u32(_at(gw, idx)), as_u32(w))
        assert np.array_equal(as_u32(_at(gm, idx)), as_u32(m))
        assert np.array_equal(as_u32(_at(gv, idx)), as_u32(v))
        for r in (0, 13, 31):
            assert np.array_equal(as_u16(_at(bufs.params16[r], idx)), p16)


@pytest.mark.parametrize("dtype", [oracle.FP16, oracle.BF16])
def test_sweep_2p28_n2_clip_staged_pass1(dtype):
    """Two ranks, 2^28 parameters resident in HBM, clipping at 1.0 with the
    gradient spread set so that c < 1: the exact norm over all 2^28 reduced
    values (the oracle's exponent bins of the GPU's reduced gradient), the
    clip coefficient from it, and sampled elements of the reduced gradient,
    state and both ranks' parameters against the oracle, two steps."""
    n, N, B = 1 << 28, 2, 1 << 24
    s = torch.cuda.current_stream()
    dt = zg.ZERO_BF16 if dtype == oracle.BF16 else zg.ZERO_FP16
    cfg = zg.Config(n, N, 2, B, 0, None, dt)
    plan = zg.zero_plan(cfg)
    bufs = zg.DeviceBuffers(cfg, plan, device="cuda", shadow=False)
    synth.dev_normal32(bufs.w[0].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT, cuda_stream=s.cuda_stream)
    max_norm, sigma = 1.0, 2e-4        # norm of the mean gradient about sqrt(2^28 / 2) * 2e-4 = 2.3
    adam = zg.zero_adam_t(max_grad_norm=max_norm, **ADAM)
    state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
    idx = _samples(n, [0, n - 1, B - 1, B, n // 2])
    w = synth.host_normal32_at(idx, 0.02, seed=0, stream=synth.STREAM_WEIGHT)
    m, v = np.zeros_like(w), np.zeros_like(w)
    inv = oracle.inv_scale(1.0, N)
    for step in (1, 2):
        for r in range(N):
            synth.dev_normal16(bufs.grads[r].data_ptr(), n, dt, sigma, seed=0, stream=synth.STREAM_GRAD, step=step,
                               rank=r, cuda_stream=s.cuda_stream)
        res = zg.zero_step_stage2(cfg, plan, bufs, adam, state, s)
        torch.cuda.synchronize()
        assert res.overflow == 0 and res.path == 1 and res.t == step
        h_all = bufs.reduced[:n].cpu().numpy().view(np.uint16)
        norm = oracle.grad_norm(float(oracle.sumsq_fraction(h_all, dtype)), inv)
        del h_all
        assert res.grad_norm == norm, (res.grad_norm, norm)
        c = oracle.clip_coef(norm, max_norm)
        assert 0.0 < c < 1.0 and res.clip_coef == c
        grads = [synth.host_normal16_at(idx, dtype, sigma, seed=0, stream=synth.STREAM_GRAD, step=step, rank=r)
                 for r in range(N)]
        h, flag = oracle.reduce(grads, dtype)
        assert flag == 0
        assert np.array_equal(as_u16(_at(bufs.reduced, idx)), h)
        hyper = oracle.make_hyper(inv=inv, clip=c, t=step, **ADAM)
        p16 = oracle.adam(h, dtype, hyper, w, m, v)
        gw, gm, gv = bufs.state()
        assert np.array_equal(as_u32(_at(gw, idx)), as_u32(w))
        assert np.array_equal(as_u32(_at(gm, idx)), as_u32(m))
        assert np.array_equal(as_u32(_at(gv, idx)), as_u32(v))
        for r in range(N):
            assert np.array_equal(as_u16(_at(bufs.params16[r], idx)), p16)
