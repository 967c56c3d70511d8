"""fp32 training (ZERO_FP32: binary32 gradients and parameters, the pages'
fp32 SGD / SGD-with-momentum examples) on the GPU against the oracle, bit
for bit: every stage, both paths, every optimizer, ragged sizes, overflowed
and clean steps, per-bucket staging, stage-3 gathers and the fetcher, the
device-state step, and the guard regions around every buffer."""
import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_mixed_bucket_gb300 as zg
from tests.gpu_harness import Job, as_bits, as_signed, as_u32

pytestmark = pytest.mark.gpu

FP32 = oracle.FP32
INF = synth.inf_bits(FP32)
OPTS = [zg.ZERO_ADAM, zg.ZERO_SGD_MOMENTUM, zg.ZERO_SGD]


@pytest.mark.parametrize("optimizer", OPTS)
@pytest.mark.parametrize("stage", [0, 1, 2, 3])
@pytest.mark.parametrize("shadow", [True, False])
def test_stages_paths_optimizers(optimizer, stage, shadow):
    n, N, B = 3 * 2048 + 13, 5, 2048
    job = Job(n, N, stage, B, 8, dtype=FP32, shadow=shadow, optimizer=optimizer, loss_scale=128.0, dynamic=True,
              growth=2)
    for t, inject in ((1, ()), (2, ((N - 1, n - 1, INF),)), (3, ()), (4, ((1, 7, 0x7FC00000),)), (5, ())):
        res, ref = job.step(job.make_grads(t, inject))
        job.check(res, ref)
        assert res.overflow == (1 if inject else 0)
    assert job.state.t == 3


def test_edge_sizes_and_many_ranks():
    for n, N, B, stage in ((1, 1, 8, 2), (7, 3, 8, 0), (9, 64, 16, 3), (1000, 64, 64, 2)):
        job = Job(n, N, stage, B, 8, dtype=FP32, optimizer=zg.ZERO_SGD_MOMENTUM)
        res, ref = job.step(job.make_grads(1))
        job.check(res, ref)


def test_params_equal_master_weights():
    """In fp32 training every parameter copy is the master weight itself."""
    n, N = 20_000, 4
    job = Job(n, N, 2, 4096, 8, dtype=FP32, optimizer=zg.ZERO_SGD_MOMENTUM)
    for t in (1, 2):
        res, ref = job.step(job.make_grads(t))
        job.check(res, ref)
    w = as_u32(job.bufs.state()[0][:n])
    for r in range(N):
        assert np.array_equal(as_bits(job.bufs.params16[r][:n]), w)


@pytest.mark.parametrize("stage", [2, 3])
def test_bucket_staging(stage):
    n, N, B = 4 * 1024 + 5, 3, 1024
    job = Job(n, N, stage, B, 8, dtype=FP32, optimizer=zg.ZERO_SGD)
    grads = job.make_grads(1)
    staging = [torch.zeros(B, dtype=torch.int32, device="cuda") for _ in range(N)]
    s = torch.cuda.current_stream()
    zg.zero_step_begin(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
    for b in reversed(range(job.plan.n_buckets)):
        lo, hi = b * B, min((b + 1) * B, n)
        for r in range(N):
            staging[r][:hi - lo].copy_(torch.from_numpy(as_signed(grads[r][lo:hi])))
        zg.zero_step_bucket(job.cfg, job.plan, job.bufs, job.adam, job.state, b, [t.data_ptr() for t in staging], s)
    res = zg.zero_step_end(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
    torch.cuda.synchronize()
    job.check(res, job.oracle_step(grads))


@pytest.mark.parametrize("n_dst", [2, 9])
def test_gathers_and_fetcher(n_dst):
    layers = [1001, 4096, 7, 9000, 3333]
    n, N = sum(layers), 6
    job = Job(n, N, 3, 2048, 8, layers=layers, dtype=FP32, optimizer=zg.ZERO_SGD_MOMENTUM)
    res, ref = job.step(job.make_grads(1))
    job.check(res, ref)
    starts = np.cumsum([0] + layers)
    shards = [t.data_ptr() for t in job.bufs.params16]
    dst = [torch.full((job.plan.max_layer_elems,), -1, dtype=torch.int32, device="cuda") for _ in range(n_dst)]
    for l, ln in enumerate(layers):
        zg.zero_gather_layer(job.cfg, job.plan, l, shards, [d.data_ptr() for d in dst])
        torch.cuda.synchronize()
        for d in dst:
            assert np.array_equal(as_bits(d[:ln]), job.p16[starts[l]:starts[l] + ln]), l
    # the fetcher: reverse order under a budget of the two largest layers
    cap = 9000 + 4096 + 16
    pool = [torch.zeros(cap, dtype=torch.int32, device="cuda") for _ in range(n_dst)]
    side = torch.cuda.Stream()
    order = list(reversed(range(len(layers))))
    f = zg.Fetcher(job.cfg, job.plan, shards, pool, cap, order, 2, side)
    s = torch.cuda.current_stream()
    for pos, l in enumerate(order):
        off = f.fetch(pos, s)
        torch.cuda.synchronize()
        for p in pool:
            assert np.array_equal(as_bits(p[off:off + layers[l]]), job.p16[starts[l]:starts[l + 1]]), l
        f.release(pos, s)
    torch.cuda.synchronize()


def test_async_steps_and_graph():
    from tests.test_async_gpu import AsyncJob
    n, N, B = 3 * 4096 + 9, 4, 4096
    job = AsyncJob(n, N, 2, B, 8, None, FP32, loss_scale=64.0, dynamic=True, growth=2,
                   optimizer=zg.ZERO_SGD_MOMENTUM)
    res, ref = job.step(job.make_grads(1))
    job.check(res, ref)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    graphs = []
    for _ in range(2):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            job.launch(torch.cuda.current_stream())
        graphs.append(g)
    for step in range(2, 8):
        grads = job.make_grads(step, ((2, 11, INF),) if step == 4 else ())
        job.load_grads(grads)
        graphs[(step - 2) % 2].replay()
        torch.cuda.synchronize()
        res, ref = job.read(), job.oracle_step(grads)
        job.bufs.b.cur = 1 - job.bufs.b.cur
        job.check(res, ref)
        assert res.overflow == (1 if step == 4 else 0)


def test_full_size_sampled_stage2_sgdm():
    """The 12-layer d=768 parameter list (123,568,896 params), N_d = 8, in
    fp32 with SGD and momentum: sampled elements against the oracle."""
    layers = [50257 * 768] + [12 * 768 * 768 + 4 * 768] * 12
    n, N, B = sum(layers), 8, 1 << 24
    s = torch.cuda.current_stream()
    cfg = zg.Config(n, N, 2, B, 0, layers, zg.ZERO_FP32, zg.ZERO_SGD_MOMENTUM)
    plan = zg.zero_plan(cfg)
    bufs = zg.DeviceBuffers(cfg, plan, device="cuda")
    for k in range(2):
        bufs.b.v[k] = None
    synth.dev_normal32(bufs.w[0].data_ptr(), n, 0.02, seed=0, stream=synth.STREAM_WEIGHT, cuda_stream=s.cuda_stream)
    adam = zg.zero_adam_t(lr=1e-4, momentum=0.9)
    state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
    rng = np.random.default_rng(3)
    idx = np.unique(np.concatenate([rng.integers(0, n, 1 << 15), [0, n - 1, B - 1, B, plan.shard_elems]]))
    w = synth.host_normal32_at(idx, 0.02, seed=0, stream=synth.STREAM_WEIGHT)
    m, v = np.zeros_like(w), np.zeros_like(w)
    sel = torch.from_numpy(idx).cuda()
    for step in (1, 2):
        for r in range(N):
            synth.dev_grad(bufs.grads[r].data_ptr(), n, FP32, 1e-3, seed=0, stream=synth.STREAM_GRAD, step=step,
                           rank=r, cuda_stream=s.cuda_stream)
        res = zg.zero_step_stage2(cfg, plan, bufs, adam, state, s)
        torch.cuda.synchronize()
        assert res.overflow == 0 and res.t == step and res.path == 0
        grads = [synth.host_grad_at(idx, FP32, 1e-3, seed=0, stream=synth.STREAM_GRAD, step=step, rank=r)
                 for r in range(N)]
        ref = oracle.step(grads, w, m, v, dtype=FP32, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, t=step - 1,
                          loss_scale=1.0, optimizer="sgdm", momentum=0.9)
        gw, gm, _ = bufs.state()
        assert np.array_equal(as_u32(gw.index_select(0, sel)), as_u32(w))
        assert np.array_equal(as_u32(gm.index_select(0, sel)), as_u32(m))
        for r in (0, 3, 7):
            assert np.array_equal(as_bits(bufs.params16[r].index_select(0, sel)), ref["p16"])
    assert res.hbm_bytes == oracle.hbm_bytes_per_param(N, 2, "fused", 8, 4) * n
