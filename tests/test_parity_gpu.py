"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the
same seeded inputs.

Bar: 16-bit parameters, the overflow flag, the reduced gradient and the
partition offsets bit-exact; fp32 master weights, momentum and variance within
1e-6 relative -- in fact required bit-identical here, since both sides
evaluate the same IEEE operations in the same order (and a single differing
fp32 ulp would flip 16-bit roundings).
"""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
import zero_sharded_mixed_bucket_gb300 as zg
from tests.gpu_harness import Job, as_u16, as_u32

pytestmark = pytest.mark.gpu

FP16, BF16 = oracle.FP16, oracle.BF16


def test_first_config_stage2_exact():
    """Stage 2, 2^20 parameters, N_d = 4, grads N(0,1e-3) x 1024 loss scale,
    Adam lr 1e-4, betas (0.9, 0.999), eps 1e-8, t = 1, m = v = 0."""
    job = Job(1 << 20, 4, 2, 1 << 24, loss_scale=1024.0)
    res, ref = job.step(job.make_grads(1))
    assert res.path == 0 and res.kernel_launches == 1
    job.check(res, ref)


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("shadow", [True, False])
def test_stages_ragged_multi_step(stage, dtype, shadow):
    """Three buckets with a ragged tail, N_d = 3 (not a power of two), three
    steps, both paths (fused with shadow state; two-pass in place)."""
    n = 3 * 8192 + 37
    job = Job(n, 3, stage, 8192, 64, dtype=dtype, shadow=shadow, loss_scale=8.0)
    for t in range(1, 4):
        res, ref = job.step(job.make_grads(t))
        assert res.path == (0 if shadow else 1)
        job.check(res, ref)


@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("sigma", [1e-3, 0.3])
def test_clipped_steps(dtype, sigma):
    """Global-norm clipping at 1.0: the exact integer sum of squares must give
    the oracle's fp64 norm bit for bit, hence the same clip coefficient."""
    n = (1 << 18) + 5
    job = Job(n, 8, 2, 1 << 16, dtype=dtype, max_norm=1.0, sigma=sigma)
    clipped = []
    for t in range(1, 4):
        res, ref = job.step(job.make_grads(t))
        job.check(res, ref)
        clipped.append(ref["clip"] < 1.0)
    assert all(clipped) == (sigma > 0.1)


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
def test_clipped_all_stages(stage):
    job = Job(20_000 + 3, 4, stage, 4096, 16, max_norm=0.05, sigma=1e-2, loss_scale=4.0)
    for t in range(1, 3):
        res, ref = job.step(job.make_grads(t))
        job.check(res, ref)


@pytest.mark.parametrize("shadow", [True, False])
@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_overflow_skips_and_halves(shadow, dtype):
    """An inf in one rank's gradient: flag set, state bit-identical, 16-bit
    parameters unchanged, loss scale halved, t unchanged; the next clean step
    proceeds from the unchanged state."""
    n = 5 * 4096 + 11
    job = Job(n, 4, 2, 4096, dtype=dtype, shadow=shadow, loss_scale=1024.0, dynamic=True)
    res, ref = job.step(job.make_grads(1))
    job.check(res, ref)
    w_before = as_u32(job.bufs.state()[0][:n]).copy()
    p_before = as_u16(job.bufs.params16[2][:n]).copy()
    inf = synth.inf_bits(dtype)
    res, ref = job.step(job.make_grads(2, inject=[(3, n - 2, inf)]))
    assert res.overflow == 1 and res.skipped == 1 and res.new_loss_scale == 512.0 and res.t == 1
    job.check(res, ref)
    if shadow:     # the skipped fused step also ran the parameter restore
        assert res.hbm_bytes == job.plan.hbm_bytes_fused + n * oracle.hbm_bytes_per_param(4, 2, "restore")
    else:
        assert res.hbm_bytes == job.plan.hbm_bytes_two_pass
    assert np.array_equal(as_u32(job.bufs.state()[0][:n]), w_before)
    assert np.array_equal(as_u16(job.bufs.params16[2][:n]), p_before)
    res, ref = job.step(job.make_grads(3))
    assert res.overflow == 0 and res.t == 2
    job.check(res, ref)


@pytest.mark.parametrize("stage", [0, 1, 3])
def test_overflow_other_stages(stage):
    n = 3 * 2048 + 5
    job = Job(n, 2, stage, 2048, 8, loss_scale=64.0, dynamic=True)
    res, ref = job.step(job.make_grads(1, inject=[(0, 17, 0x7E00)]))   # NaN
    assert res.overflow == 1
    job.check(res, ref)
    full = job.plan.hbm_bytes_fused + n * oracle.hbm_bytes_per_param(2, stage, "restore")
    if stage <= 1:     # every bucket writes the all-reduced gradient back: nothing is skipped
        assert res.hbm_bytes == full
    else:              # later bucket kernels may skip once the flag is up
        assert 0 < res.hbm_bytes <= full
    res, ref = job.step(job.make_grads(2))
    job.check(res, ref)


@pytest.mark.parametrize("stage,optimizer", [(2, zg.ZERO_ADAM), (2, zg.ZERO_SGD), (3, zg.ZERO_ADAM)])
@pytest.mark.parametrize("where", ["first", "middle", "last"])
@pytest.mark.parametrize("order", ["forward", "backward"])
def test_overflow_skips_later_buckets(stage, optimizer, where, order):
    """Buckets launched one at a time (plain stream order) after the flag is
    raised do nothing; the restore covers only the window the kernels that
    ran wrote.  State and parameters equal the oracle's (state unchanged,
    loss scale halved, t unchanged), and hbm_bytes counts exactly the buckets
    that ran (fused bytes) and their window (restore bytes).  Stage 2 with
    SGD takes the tile kernel."""
    n, B, N = 8 * 4096 + 101, 4096, 4
    nb = 9
    job = Job(n, N, stage, B, 8, loss_scale=1024.0, dynamic=True, optimizer=optimizer)
    res, ref = job.step(job.make_grads(1))
    job.check(res, ref)
    kb = {"first": 0, "middle": 4, "last": nb - 1}[where]
    i = min(kb * B + 1000, n - 1)
    grads = job.make_grads(2, inject=[(1, i, synth.inf_bits(job.dtype))])
    job.load_grads(grads)
    s = torch.cuda.current_stream()
    buckets = list(range(nb)) if order == "forward" else list(reversed(range(nb)))
    zg.zero_step_begin(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
    for b in buckets:
        zg.zero_step_bucket(job.cfg, job.plan, job.bufs, job.adam, job.state, b, None, s)
    res = zg.zero_step_end(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
    torch.cuda.synchronize()
    ref = job.oracle_step(grads)
    assert res.overflow == 1 and res.skipped == 1 and res.new_loss_scale == 512.0
    job.check(res, ref)
    ran = buckets[:buckets.index(kb) + 1]
    updated = sum(min((b + 1) * B, n) - b * B for b in ran)
    window = min((max(ran) + 1) * B, n) - min(ran) * B
    sb = {zg.ZERO_ADAM: 12, zg.ZERO_SGD: 4}[optimizer]
    assert res.hbm_bytes == (updated * oracle.hbm_bytes_per_param(N, stage, "fused", sb)
                             + window * oracle.hbm_bytes_per_param(N, stage, "restore", sb))
    res, ref = job.step(job.make_grads(3))
    assert res.overflow == 0
    job.check(res, ref)


@pytest.mark.parametrize("stage", [2, 3])
@pytest.mark.parametrize("where", ["first", "middle", "last"])
def test_overflow_anywhere_whole_step(stage, where):
    """The whole-step entry point (bucket kernels chained by programmatic
    dependent launch, so how many skip depends on timing) with the inf in the
    first, a middle or the last of 17 buckets: bit-exact against the oracle,
    and the bytes reported are positive and at most the full step plus a
    full restore."""
    n, B, N = 16 * 8192 + 77, 8192, 8
    job = Job(n, N, stage, B, 8, loss_scale=256.0, dynamic=True)
    kb = {"first": 0, "middle": 8, "last": 16}[where]
    for t, inject in ((1, []), (2, [(N - 1, min(kb * B + 5, n - 1), 0x7C00)]), (3, [])):
        res, ref = job.step(job.make_grads(t, inject))
        job.check(res, ref)
        if inject:
            fb = oracle.hbm_bytes_per_param(N, stage, "fused")
            rb = oracle.hbm_bytes_per_param(N, stage, "restore")
            assert 0 < res.hbm_bytes <= n * (fb + rb)


@pytest.mark.parametrize("stage", [1, 2])
@pytest.mark.parametrize("N,dtype", [(2, FP16), (8, BF16), (33, oracle.FP32), (64, FP16)])
def test_overflow_restore_tiles(stage, N, dtype):
    """An overflowed fused step in stages 1-2 with several ranks puts every
    rank's parameters back through shared-memory tiles and bulk copies
    (tiles of 4096 16-bit or 2048 binary32 values; a ragged tail of fewer
    than 16 bytes); then a clean step."""
    n = 3 * 4096 + 13
    job = Job(n, N, stage, 5000, 8, dtype=dtype, loss_scale=32.0, dynamic=True)
    inf = synth.inf_bits(dtype)
    for t, inject in ((1, ()), (2, ((N // 2, n - 1, inf),)), (3, ())):
        res, ref = job.step(job.make_grads(t, inject))
        job.check(res, ref)
        assert res.path == 0 and res.overflow == (1 if inject else 0)


def test_overflow_by_sum():
    """Finite gradients whose rank sum overflows binary16."""
    n = 1000
    job = Job(n, 2, 2, 512, 8, loss_scale=1.0, dynamic=True)
    g = job.make_grads(1)
    g[0][5] = g[1][5] = 0x7BFF   # 65504 + 65504
    res, ref = job.step(g)
    assert res.overflow == 1 == ref["overflow"]
    job.check(res, ref)


def test_dynamic_scale_sequence():
    """Overflow on steps 2 and 3, growth after 2 clean steps."""
    n = 4096 + 8
    job = Job(n, 2, 2, 1024, 8, loss_scale=256.0, dynamic=True, growth=2, min_scale=1.0)
    scales = []
    for t in range(1, 8):
        inj = [(1, t * 13, 0x7C00)] if t in (2, 3) else []
        res, ref = job.step(job.make_grads(t, inject=inj))
        job.check(res, ref)
        scales.append(res.new_loss_scale)
    assert scales == [256.0, 128.0, 64.0, 64.0, 128.0, 128.0, 256.0]


@pytest.mark.parametrize("n,N,B", [(1, 1, 8), (7, 1, 8), (8, 2, 8), (9, 3, 8), (1, 64, 8), (100, 64, 16),
                                   (5000, 64, 1024)])
@pytest.mark.parametrize("stage", [0, 2, 3])
def test_edge_sizes(n, N, B, stage):
    job = Job(n, N, stage, B, 8)
    for t in (1, 2):
        res, ref = job.step(job.make_grads(t))
        job.check(res, ref)


def test_empty_model():
    job = Job(0, 4, 2, 64)
    res, ref = job.step(job.make_grads(1))
    assert res.kernel_launches == 0 and res.overflow == 0 and res.t == 1


@pytest.mark.parametrize("api", ["sync", "async"])
def test_empty_model_clipped(api):
    """Zero parameters with clipping: the norm finalize runs with no pass-1
    kernel before it (after the workspace clear, or the prepare kernel of a
    device-state step); the norm is 0 and the coefficient 1."""
    job = Job(0, 4, 2, 64, shadow=False, max_norm=1.0)
    placeholder = torch.zeros(8, dtype=torch.int16, device="cuda")
    job.bufs.b.reduced = placeholder.data_ptr()
    s = torch.cuda.current_stream()
    if api == "sync":
        for t in (1, 2):
            res = zg.zero_step_stage2(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
            assert res.kernel_launches == 1 and res.overflow == 0 and res.t == t
            assert res.grad_norm == 0.0 and res.clip_coef == 1.0
    else:
        dev = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device="cuda")
        zg.zero_dev_state_init(dev, job.adam, job.state, s)
        for t in (1, 2):
            assert zg.zero_step_async(job.cfg, job.plan, job.bufs, job.adam, dev, s) == 3
            st, last = zg.zero_dev_state_read(dev, s)
            assert st.t == t and last.overflow == 0 and last.grad_norm == 0.0 and last.clip_coef == 1.0


@pytest.mark.parametrize("stage", [2, 3])
@pytest.mark.parametrize("shadow", [True, False])
def test_per_bucket_protocol(stage, shadow):
    """begin / bucket / end gives the same result as the one-call step."""
    n = 4 * 4096 + 100
    job = Job(n, 4, stage, 4096, 16, shadow=shadow)
    for t in (1, 2):
        res, ref = job.step(job.make_grads(t), per_bucket=True)
        job.check(res, ref)


@pytest.mark.parametrize("stage", [2, 3])
def test_bucket_staging_buffers(stage):
    """Gradients arriving one bucket at a time in a constant-size staging
    buffer per rank (reused for every bucket)."""
    n, N, B = 5 * 2048 + 77, 4, 2048
    job = Job(n, N, stage, B, 8, max_norm=1.0 if stage == 3 else 0.0)
    grads = job.make_grads(1)
    staging = [torch.zeros(B, dtype=torch.int16, device="cuda") for _ in range(N)]
    s = torch.cuda.current_stream()
    zg.zero_step_begin(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
    for b in range(job.plan.n_buckets):
        lo, hi = b * B, min((b + 1) * B, n)
        for r in range(N):
            staging[r][:hi - lo].copy_(torch.from_numpy(grads[r][lo:hi].view(np.int16)))
        zg.zero_step_bucket(job.cfg, job.plan, job.bufs, job.adam, job.state, b,
                            [t.data_ptr() for t in staging], s)
    res = zg.zero_step_end(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
    torch.cuda.synchronize()
    ref = oracle.step(grads, job.w, job.m, job.v, dtype=FP16, t=0, loss_scale=1.0, max_grad_norm=job.max_norm,
                      **job.hp)
    job.p16, job.h, job.o["t"] = ref["p16"], ref["h"], ref["t"]
    job.check(res, ref)


def test_partition_invariance():
    """Stage, bucket size and alignment do not change the step's numbers."""
    n = 50_000 + 3
    outs = []
    for stage, B, A in [(0, 4096, 0), (1, 8192, 64), (2, 1 << 20, 8), (3, 2048, 2048), (2, 8, 8)]:
        job = Job(n, 4, stage, B, A)
        job.step(job.make_grads(1))
        res, ref = job.step(job.make_grads(2))
        job.check(res, ref)
        w = as_u32(job.bufs.state()[0][:n])
        if stage == 3:
            P = job.plan.shard_elems
            p = np.concatenate([as_u16(job.bufs.params16[r][:P]) for r in range(4)])[:n]
        else:
            p = as_u16(job.bufs.params16[1][:n])
        outs.append((w, p))
    for w, p in outs[1:]:
        assert np.array_equal(w, outs[0][0]) and np.array_equal(p, outs[0][1])


def test_replicas_identical_stage0():
    n = 10_000
    job = Job(n, 5, 0, 2048, 8)
    res, ref = job.step(job.make_grads(1))
    job.check(res, ref)
    w = job.bufs.state()[0]
    pad = job.plan.padded_elems
    for r in range(1, 5):
        assert torch.equal(w[r * pad:r * pad + n], w[:n])
        assert torch.equal(job.bufs.params16[r], job.bufs.params16[0])


def test_max_ranks_and_rejects_65():
    job = Job(3000, 64, 2, 1024, 8)
    res, ref = job.step(job.make_grads(1))
    job.check(res, ref)
    with pytest.raises(zg.ZeroError) as e:
        zg.zero_plan(zg.Config(3000, 65, 2, 1024))
    assert e.value.status == zg.ZERO_EUNSUPPORTED


def test_deterministic_repeat():
    n = 70_000
    outs = []
    for _ in range(2):
        job = Job(n, 8, 2, 16384, max_norm=1.0)
        res, _ = job.step(job.make_grads(1))
        outs.append((res.grad_norm, as_u32(job.bufs.state()[0][:n])))
    assert outs[0][0] == outs[1][0] and np.array_equal(outs[0][1], outs[1][1])


# --- stage-3 layer gather ------------------------------------------------------
@pytest.mark.parametrize("A,n_dst", [(8, 3), (2048, 3), (8, 8), (2048, 17)])
def test_gather_layers(A, n_dst):
    """Layers with unaligned starts, ragged ends and several 8192-unit
    segments, shards smaller than a segment, 3 to 17 destinations (the
    chunked kernel, destination by destination)."""
    layers = [1001, 4096, 7, 20_000, 3333]
    n = sum(layers)
    N = 6
    job = Job(n, N, 3, 2048, A, layers=layers)
    plan = job.plan
    assert plan.max_layer_elems == 20_000
    dst = [torch.full((plan.max_layer_elems,), -1, dtype=torch.int16, device="cuda") for _ in range(n_dst)]
    shards = [t.data_ptr() for t in job.bufs.params16]
    for step in range(2):
        if step:
            res, ref = job.step(job.make_grads(1))
            job.check(res, ref)
        start = 0
        for l, ln in enumerate(layers):
            zg.zero_gather_layer(job.cfg, plan, l, shards, [d.data_ptr() for d in dst])
            torch.cuda.synchronize()
            for d in dst:
                got = as_u16(d[:ln])
                assert np.array_equal(got, job.p16[start:start + ln]), (step, l)
            start += ln


@pytest.mark.parametrize("n_dst", [8, 64])
def test_gather_layers_of_several_chunks(n_dst):
    """The chunked gather on layers longer than its 2 MB chunks: 64 shards,
    a layer ending mid-group, one of exactly two chunks and a group, a tiny
    one; every destination equals the oracle's parameters."""
    layers = [2_500_003, 2 * (1 << 20) + 8, 9]
    n = sum(layers)
    job = Job(n, 64, 3, 1 << 20, 8, layers=layers)
    plan = job.plan
    dst = [torch.full((plan.max_layer_elems,), -1, dtype=torch.int16, device="cuda") for _ in range(n_dst)]
    shards = [t.data_ptr() for t in job.bufs.params16]
    for step in range(2):
        if step:
            res, ref = job.step(job.make_grads(1))
            job.check(res, ref)
        start = 0
        for l, ln in enumerate(layers):
            for d in dst:
                d.fill_(-1)
            zg.zero_gather_layer(job.cfg, plan, l, shards, [d.data_ptr() for d in dst])
            torch.cuda.synchronize()
            want = job.p16[start:start + ln]
            for d in dst:
                assert np.array_equal(as_u16(d[:ln]), want), (step, l)
                assert (d[ln:] == -1).all()
            start += ln


def _gather_cases(k=40, seed=77):
    rng = np.random.default_rng(seed)
    out = []
    for _ in range(k):
        N = int(rng.choice([1, 2, 3, 8, 17, 64]))
        n = int(rng.integers(1, 3_000_000))
        cuts = sorted(set(int(c) for c in rng.integers(1, n, int(rng.integers(0, 5))))) if n > 1 else []
        layers = [b - a for a, b in zip([0] + cuts, cuts + [n])]
        A = int(rng.choice([8, 64, 2048]))
        n_dst = int(rng.choice([1, 5, 8, 9, 17, 33, 64]))
        out.append((N, n, layers, A, n_dst))
    return out


@pytest.mark.parametrize("case", _gather_cases(int(os.environ.get("ZG_GATHER_CASES", "40")),
                                         int(os.environ.get("ZG_GATHER_SEED", "77"))),
                         ids=lambda c: "N%d-n%d-L%d-A%d-d%d" % (c[0], c[1], len(c[2]), c[3], c[4]))
def test_gather_random_layouts(case):
    """Seeded random layer splits (unaligned starts, layers from one element
    to several 2 MB chunks), shard sizes from below a 16 KB segment to
    millions of elements, 1-64 destinations: every destination holds the
    layer's slice of the flat parameter vector (the shards laid end to end),
    bit for bit, and nothing past it.  ZG_GATHER_SEED and ZG_GATHER_CASES
    draw another set (a longer soak)."""
    N, n, layers, A, n_dst = case
    cfg = zg.Config(n, N, 3, 1 << 20, A, layers)
    plan = zg.zero_plan(cfg)
    P = plan.shard_elems
    gen = torch.Generator(device="cuda").manual_seed(n * 31 + N)
    shards = [torch.randint(-32768, 32767, (P,), dtype=torch.int16, device="cuda", generator=gen) for _ in range(N)]
    flat = torch.cat(shards)[:n]
    dst = [torch.empty(plan.max_layer_elems, dtype=torch.int16, device="cuda") for _ in range(n_dst)]
    start = 0
    for l, ln in enumerate(layers):
        for d in dst:
            d.fill_(-1)
        zg.zero_gather_layer(cfg, plan, l, [t.data_ptr() for t in shards], [d.data_ptr() for d in dst])
        torch.cuda.synchronize()
        for d in dst:
            assert torch.equal(d[:ln], flat[start:start + ln]), l
            assert (d[ln:] == -1).all(), l
        start += ln


def test_gather_destinations_change_kind():
    """The library asks the driver what each destination is on every call:
    the same job gathers into device buffers (the chunked kernel),
    then, after those are freed, into pinned host buffers (per-thread
    stores), then into device buffers again; every result equals the
    oracle's parameters."""
    layers = [3001, 20_000, 17]
    n = sum(layers)
    job = Job(n, 4, 3, 4096, layers=layers)
    plan = job.plan
    shards = [t.data_ptr() for t in job.bufs.params16]
    for kind in ("device", "host", "device"):
        if kind == "device":
            dst = [torch.full((plan.max_layer_elems,), -1, dtype=torch.int16, device="cuda") for _ in range(8)]
        else:
            dst = [torch.full((plan.max_layer_elems,), -1, dtype=torch.int16).pin_memory() for _ in range(8)]
        start = 0
        for l, ln in enumerate(layers):
            zg.zero_gather_layer(job.cfg, plan, l, shards, [d.data_ptr() for d in dst])
            torch.cuda.synchronize()
            for d in dst:
                assert np.array_equal(d[:ln].cpu().numpy().view(np.uint16), job.p16[start:start + ln]), (kind, l)
            start += ln
        del dst
        torch.cuda.empty_cache()


def test_gather_max_destinations():
    layers = [5000, 5000]
    job = Job(10_000, 4, 3, 1024, 8, layers=layers)
    dst = [torch.zeros(5000, dtype=torch.int16, device="cuda") for _ in range(64)]
    zg.zero_gather_layer(job.cfg, job.plan, 1, [t.data_ptr() for t in job.bufs.params16],
                         [d.data_ptr() for d in dst])
    torch.cuda.synchronize()
    for d in dst:
        assert np.array_equal(as_u16(d), job.p16[5000:])


# --- input generator: device == host ---------------------------------------------
@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("offset,n", [(0, 100_000), (1, 99_999), (12_345, 7)])
def test_synth_device_matches_host(dtype, offset, n):
    t = torch.zeros(n, dtype=torch.int16, device="cuda")
    synth.dev_normal16(t.data_ptr(), n, dtype, 1e-3, seed=3, stream=1, step=5, rank=7, offset=offset)
    f = torch.zeros(n, dtype=torch.float32, device="cuda")
    synth.dev_normal32(f.data_ptr(), n, 0.02, seed=3, stream=2, step=0, rank=1, offset=offset)
    torch.cuda.synchronize()
    h = synth.host_normal16(n, dtype, 1e-3, seed=3, stream=1, step=5, rank=7, offset=offset)
    assert np.array_equal(as_u16(t), h)
    hf = synth.host_normal32(n, 0.02, seed=3, stream=2, step=0, rank=1, offset=offset)
    assert np.array_equal(as_u32(f), as_u32(hf))


# --- the benchmark's workload at full size, sampled -------------------------------
def _transformer_params(vocab, d, layers):
    return vocab * d + layers * (12 * d * d + 4 * d)


@pytest.mark.parametrize("stage,api", [(2, "sync"), (0, "sync"), (2, "async")])
def test_full_size_sampled(stage, api):
    """The 12-layer d=768 parameter list (123,568,896 params), N_d = 8, bucket
    2^24, inputs generated on the device; 2^16 sampled elements recomputed by
    the oracle from the host generator, every rank checked at those indices.
    api "async": through zero_step_async, the entry point the benchmark times."""
    n = _transformer_params(50257, 768, 12)
    assert n == 123_568_896
    N, B = 8, 1 << 24
    cfg = zg.Config(n, N, stage, B)
    plan = zg.zero_plan(cfg)
    bufs = zg.DeviceBuffers(cfg, plan, device="cuda")
    s = torch.cuda.current_stream()
    reps = N if stage == 0 else 1
    for r in range(reps):
        off = r * plan.padded_elems
        synth.dev_normal32(bufs.w[0].data_ptr() + 4 * off, n, 0.02, seed=0, stream=synth.STREAM_WEIGHT,
                           cuda_stream=s.cuda_stream)
    w0_dev = bufs.w[0][:n]
    # 16-bit copy = cast of the master weights, made on the host for a sample only;
    # the device copy is produced by one clean step from zero learning rate
    for r in range(N):
        synth.dev_normal16(bufs.grads[r].data_ptr(), n, FP16, 1e-3, seed=0, stream=synth.STREAM_GRAD, step=1,
                           rank=r, cuda_stream=s.cuda_stream)
    adam = zg.zero_adam_t(**{**dict(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8), "max_grad_norm": 0.0})
    state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
    if api == "async":
        dev = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device="cuda")
        zg.zero_dev_state_init(dev, adam, state, s)
        launches = zg.zero_step_async(cfg, plan, bufs, adam, dev, s)
        st, res = zg.zero_dev_state_read(dev, s)
        assert res.overflow == 0 and st.t == 1 and launches == plan.n_buckets + 2
    else:
        fn = zg.zero_step_stage2 if stage == 2 else zg.zero_step_stage0
        res = fn(cfg, plan, bufs, adam, state, s)
        torch.cuda.synchronize()
        assert res.overflow == 0 and res.t == 1 and res.kernel_launches == plan.n_buckets

    rng = np.random.default_rng(99)
    idx = np.unique(np.concatenate([rng.integers(0, n, 1 << 16), [0, 1, n - 1, n - 2, B - 1, B, 7 * B - 1]]))
    grads = [synth.host_normal16_at(idx, FP16, 1e-3, seed=0, stream=synth.STREAM_GRAD, step=1, rank=r)
             for r in range(N)]
    w = synth.host_normal32_at(idx, 0.02, seed=0, stream=synth.STREAM_WEIGHT)
    m = np.zeros_like(w)
    v = np.zeros_like(w)
    ref = oracle.step(grads, w, m, v, dtype=FP16, lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8, t=0, loss_scale=1.0)
    assert ref["overflow"] == 0
    ti = torch.from_numpy(idx).cuda()
    gw, gm, gv = (t.index_select(0, ti) for t in bufs.state())
    assert np.array_equal(as_u32(gw), as_u32(w)) and np.array_equal(as_u32(gm), as_u32(m))
    assert np.array_equal(as_u32(gv), as_u32(v))
    for r in range(N):
        assert np.array_equal(as_u16(bufs.params16[r].index_select(0, ti)), ref["p16"])
    if stage == 0:
        pad = plan.padded_elems
        for r in range(1, N):
            assert torch.equal(bufs.state()[0][r * pad:r * pad + n], bufs.state()[0][:n])
    del w0_dev


def test_gradients_in_pinned_host_memory():
    """The fused kernel may read the ranks' gradients straight from pinned
    host memory (NVLink-C2C on GB300): same results as the oracle."""
    import ctypes
    n, N = 3 * 4096 + 19, 4
    job = Job(n, N, 2, 4096, 8, loss_scale=16.0)
    grads = job.make_grads(1)
    host = [torch.from_numpy(g.view(np.int16).copy()).pin_memory() for g in grads]
    ptrs = (ctypes.c_void_p * N)(*[t.data_ptr() for t in host])
    job.bufs.b.grads = ctypes.cast(ptrs, ctypes.POINTER(ctypes.c_void_p))
    res = zg.zero_step_stage2(job.cfg, job.plan, job.bufs, job.adam, job.state, torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref = oracle.step(grads, job.w, job.m, job.v, dtype=FP16, t=0, loss_scale=16.0, **job.hp)
    job.p16, job.h, job.o["t"] = ref["p16"], ref["h"], ref["t"]
    job.check(res, ref)


@pytest.mark.parametrize("shadow", [True, False])
def test_optimizer_state_in_pinned_host_memory(shadow):
    """fp32 master weights, momentum and variance (and the shadow copy) kept
    in pinned host memory and updated by the kernels over NVLink-C2C -- the
    optimizer-state offload axis: three steps against the oracle."""
    n, N = 5 * 2048 + 3, 4
    job = Job(n, N, 2, 2048, 8, shadow=shadow, loss_scale=4.0, max_norm=0.0 if shadow else 1.0, sigma=0.05)
    ncopy = 2 if shadow else 1
    host = {}
    for name in ("w", "m", "v"):
        dev_t = getattr(job.bufs, name)
        host[name] = [torch.empty(dev_t[0].numel(), dtype=torch.float32).pin_memory() for _ in range(ncopy)]
        for k in range(ncopy):
            host[name][k].copy_(dev_t[k].cpu())
            getattr(job.bufs.b, name)[k] = host[name][k].data_ptr()
    job.bufs.w, job.bufs.m, job.bufs.v = host["w"], host["m"], host["v"]     # state() now reads host tensors
    for t in (1, 2, 3):
        res, ref = job.step(job.make_grads(t))
        job.check(res, ref)


@pytest.mark.parametrize("optimizer", [zg.ZERO_SGD_MOMENTUM, zg.ZERO_SGD])
@pytest.mark.parametrize("stage", [0, 1, 2, 3])
@pytest.mark.parametrize("shadow,max_norm", [(True, 0.0), (False, 0.0), (False, 1.0)])
def test_sgd_variants(optimizer, stage, shadow, max_norm):
    """SGD with momentum and plain SGD in the same kernels: fused and
    two-pass paths, with and without clipping, three steps (the unused state
    arrays are not handed to the library)."""
    n = 3 * 4096 + 29
    job = Job(n, 3, stage, 4096, 16, shadow=shadow, max_norm=max_norm, sigma=0.05, loss_scale=8.0,
              optimizer=optimizer, momentum=0.9, adam=dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8))
    for t in (1, 2, 3):
        res, ref = job.step(job.make_grads(t))
        job.check(res, ref)


def test_sgd_overflow_skips():
    n = 2 * 2048 + 5
    job = Job(n, 2, 2, 2048, 8, optimizer=zg.ZERO_SGD_MOMENTUM, loss_scale=64.0, dynamic=True,
              adam=dict(lr=1e-2, beta1=0.9, beta2=0.999, eps=1e-8))
    res, ref = job.step(job.make_grads(1))
    job.check(res, ref)
    res, ref = job.step(job.make_grads(2, inject=[(1, 100, 0x7C00)]))
    assert res.skipped == 1
    job.check(res, ref)


@pytest.mark.parametrize("depth", [0, 2])
def test_fetcher_prefetch_under_budget_with_step(depth):
    """Forward and backward passes of layer fetches (side-stream prefetch,
    live budget below the sum of the layers) around a stage-3 step whose
    bucket kernels update shards while later layers are being prefetched.
    Every layer, copied on the main stream when used, must hold the
    parameters from before the step; the step must match the oracle."""
    layers = [1001, 4096, 7, 20_000, 3333, 900, 12_000]
    n, N, B = sum(layers), 4, 2048
    job = Job(n, N, 3, B, 8, layers=layers, loss_scale=4.0)
    starts = np.cumsum([0] + layers)
    p_before = job.p16.copy()
    cap = 20_008 + 1008                     # the largest layer plus a little: prefetch is budget-limited
    n_dst = 3
    pool = [torch.full((cap,), -1, dtype=torch.int16, device="cuda") for _ in range(n_dst)]
    shards = [t.data_ptr() for t in job.bufs.params16]
    main = torch.cuda.current_stream()
    side = torch.cuda.Stream()
    grads = job.make_grads(1)
    job.load_grads(grads)

    def run_pass(order, between=None):
        f = zg.Fetcher(job.cfg, job.plan, shards, pool, cap, order, depth, side)
        snaps = []
        for pos, layer in enumerate(order):
            off = f.fetch(pos, main)
            snaps.append((layer, [d[off:off + layers[layer]].clone() for d in pool]))
            if between:
                between(layer)
            f.release(pos, main)
        ml, g = f.stats()
        assert ml <= cap and g == len(order)
        return snaps

    fwd = run_pass(list(range(len(layers))))
    zg.zero_step_begin(job.cfg, job.plan, job.bufs, job.adam, job.state, main)
    done = [job.plan.n_buckets]

    def buckets_of(layer):                   # buckets whose first element lies in this layer or above
        while done[0] > 0 and (done[0] - 1) * B >= starts[layer]:
            zg.zero_step_bucket(job.cfg, job.plan, job.bufs, job.adam, job.state, done[0] - 1, None, main)
            done[0] -= 1

    bwd = run_pass(list(reversed(range(len(layers)))), between=buckets_of)
    assert done[0] == 0
    res = zg.zero_step_end(job.cfg, job.plan, job.bufs, job.adam, job.state, main)
    torch.cuda.synchronize()
    for layer, copies in fwd + bwd:
        for c in copies:
            assert np.array_equal(as_u16(c), p_before[starts[layer]:starts[layer + 1]]), layer
    ref = oracle.step(grads, job.w, job.m, job.v, dtype=FP16, t=0, loss_scale=4.0, **job.hp)
    job.p16, job.h, job.o["t"] = ref["p16"], ref["h"], ref["t"]
    job.check(res, ref)


@pytest.mark.parametrize("dtype", [FP16, BF16])
def test_clip_norm_over_full_exponent_range(dtype):
    """Gradients with random exponents over the whole 16-bit range
    (subnormals to near overflow): for bfloat16 many squares fall outside the
    fixed-point window and go through the exponent bins; the norm and the
    clip coefficient must still equal the oracle's bit for bit."""
    n, N = 3 * 4096 + 77, 2
    job = Job(n, N, 2, 4096, 8, dtype=dtype, shadow=False, max_norm=1.0)
    rng = np.random.default_rng(123)
    grads = []
    for r in range(N):
        if dtype == BF16:
            e = rng.integers(-130, 60, n).astype(np.float64)     # stays finite after the 2-rank sum
        else:
            e = rng.integers(-24, 14, n).astype(np.float64)
        x = (rng.choice([-1.0, 1.0], n) * rng.uniform(1.0, 2.0, n) * 2.0 ** e).astype(np.float32)
        grads.append(oracle.from_f32(x, dtype))
    res, ref = job.step(grads)
    assert res.overflow == 0 and ref["overflow"] == 0
    job.check(res, ref)
    # the bins were exercised: some squares lie outside the window
    if dtype == BF16:
        h = oracle.to_f32(ref["h"], dtype)
        assert (np.abs(h[h != 0]) < 2.0 ** -40).any() and (np.abs(h) > 2.0 ** 10).any()


@pytest.mark.parametrize("S", [1.0, 1024.0])
def test_clip_norm_bf16_window_edges(S):
    """bfloat16 squares at both edges of the fixed-point window.  The window
    starts at E = win_lo = e - 40 (S*N in [2^(e-1), 2^e)); a square enters it
    at shift 2(E - win_lo) in 0..62 and goes to its exponent bin below 0 and
    from 64 on.  Rank 1 sends zeros, so the reduced gradient is rank 0's
    values; the norm and clip coefficient equal the oracle's bit for bit."""
    import math
    n, N = 4096 + 45, 2
    job = Job(n, N, 2, 4096, 8, dtype=BF16, shadow=False, max_norm=1.0, loss_scale=S)
    win_lo = min(max(math.frexp(S * N)[1] - 40, -133), 88)
    rng = np.random.default_rng(7)
    Es = np.array([win_lo + d for d in (-2, -1, 0, 1, 2, 29, 30, 31, 32, 33, 34)], np.float64)
    E = Es[np.arange(n) % len(Es)]
    M = rng.integers(128, 256, n).astype(np.float64)
    x = (rng.choice([-1.0, 1.0], n) * M * 2.0 ** E).astype(np.float32)
    x[::97] = 0.0
    g0 = oracle.from_f32(x, BF16)
    assert np.array_equal(oracle.to_f32(g0, BF16), x)      # every value is exact in bfloat16
    res, ref = job.step([g0, np.zeros(n, g0.dtype)])
    assert res.overflow == 0 and ref["overflow"] == 0
    job.check(res, ref)


def test_clip_norm_bf16_group_edges():
    """bfloat16 squares are summed 8 at a time (one aligned group of 8
    elements): first against a fixed window, the top 23 binades of the
    accumulator's (exponent fields 105..127 here); a group with a nonzero
    value outside it is summed relative to its largest exponent field e_max,
    down to e_max - 22 or the window's first binade, whichever is higher; a
    group with a nonzero value below that, or with e_max above the window, is
    summed value by value.  Groups built on each side of those edges (S*N = 2,
    so the window's first exponent field is 96 and its last 127), a ragged
    tail; the norm and clip coefficient equal the oracle's bit for bit."""
    Z = None   # a zero
    patterns = [
        [105, 127, 105, 126, Z, 110, 105, 127],  # the fixed window's both ends
        [104, 127, 105, 126, Z, 110, 105, 120],  # one value just below it
        [105, 106, 107, 108, 109, 110, 111, 105],
        [Z, Z, Z, Z, Z, Z, Z, Z],                # all zero
        [120, 98, 99, Z, 110, 120, 105, 98],     # down to e_max - 22 exactly
        [120, 97, 110, 120, Z, 101, 99, 98],     # one value 23 below: per-value path
        [120, Z, Z, Z, Z, Z, Z, Z],              # zeros below never count
        [60, 70, 90, 95, 61, 62, 63, 64],        # all below the window: exponent bins
        [128, 120, 110, 100, 99, 98, 127, 126],  # e_max past the window: per-value path
        [110, 96, 97, 100, 110, Z, 96, 105],     # base clamped to the window's first exponent
        [110, 95, 97, 100, 110, Z, 96, 105],     # one value below the window
        [127, 127, 106, 105, 120, Z, 110, 127],  # e_max at the window's last exponent
        [120, 0, 110, Z, 100, 0, 99, 98],        # subnormals (field 0, nonzero fraction)
    ]
    reps = 40
    n = 8 * len(patterns) * reps + 5
    rng = np.random.default_rng(11)
    bits = np.zeros(n, np.uint16)
    for g in range(len(patterns) * reps):
        for j, e in enumerate(patterns[g % len(patterns)]):
            if e is None:
                continue
            f = int(rng.integers(1 if e == 0 else 0, 128))
            bits[8 * g + j] = (int(rng.integers(0, 2)) << 15) | (e << 7) | f
    bits[-5:] = np.array([(115 << 7) | 3, 0, (97 << 7) | 1, 1 << 15, (126 << 7)], np.uint16)
    x = oracle.to_f32(bits, BF16)
    assert np.isfinite(x).all()
    job = Job(n, 2, 2, 4096, 8, dtype=BF16, shadow=False, max_norm=1.0, loss_scale=1.0)
    res, ref = job.step([bits, np.zeros(n, np.uint16)])
    assert res.overflow == 0 and ref["overflow"] == 0
    job.check(res, ref)


def test_tiny_partitions_brute_force():
    """Every combination of tiny sizes, rank counts, bucket sizes, alignments
    and stages (448 jobs, one step each) against the oracle: partition
    offsets, owner shards and ragged tails all exercised."""
    count = 0
    for n in (1, 7, 8, 9, 17, 63, 64):
        for N in (1, 2, 3, 4):
            for B in (8, 24):
                for A in (8, 32):
                    for stage in (0, 1, 2, 3):
                        job = Job(n, N, stage, B, A, seed=n * 131 + N, loss_scale=2.0)
                        res, ref = job.step(job.make_grads(1))
                        job.check(res, ref)
                        count += 1
    assert count == 448


# --- pass 2 with the parameters copied out through shared-memory tiles ------
@pytest.mark.parametrize("stage", [1, 2])
@pytest.mark.parametrize("N", [1, 2, 4, 8, 16, 33, 64])
@pytest.mark.parametrize("dtype,optimizer", [(FP16, zg.ZERO_ADAM), (BF16, zg.ZERO_SGD_MOMENTUM),
                                             (oracle.FP32, zg.ZERO_SGD)])
def test_two_pass_many_ranks(stage, N, dtype, optimizer):
    """Stages 1-2 on the two-pass path: from 2 ranks the update pass writes
    every rank's parameters with bulk copies from shared-memory tiles (tiles
    of 4096 or 2048 elements, so a 5000-element bucket is one full tile and
    a ragged one, a skipped step in between); 1 rank keeps per-thread
    stores."""
    n, B = 3 * 5000 + 3, 5000
    job = Job(n, N, stage, B, 8, dtype=dtype, shadow=False, optimizer=optimizer,
              max_norm=1.0 if dtype != oracle.FP32 else 0.0, loss_scale=16.0, dynamic=True)
    inf = synth.inf_bits(dtype)
    for t, inject in ((1, ()), (2, ((N - 1, 4999, inf),)), (3, ())):
        res, ref = job.step(job.make_grads(t, inject))
        job.check(res, ref)
        assert res.path == 1 and res.overflow == (1 if inject else 0)


@pytest.mark.parametrize("N", [1, 2])
@pytest.mark.parametrize("stage", [2, 3])
@pytest.mark.parametrize("dtype", [FP16, BF16])
@pytest.mark.parametrize("max_norm", [0.0, 1.0])
def test_staged_pass1_one_or_two_ranks(N, stage, dtype, max_norm):
    """Pass 1 with one or two ranks in stages 2 and 3 streams the gradient
    tiles into shared memory (bulk copies on mbarriers, 4096-element tiles,
    each block striding over several): buckets of several tiles with a
    ragged last tile and a last group shorter than 8, a bucket smaller than
    one tile, an overflowed step and clean steps after it, against the
    oracle bit for bit (reduced gradient, norm, clip coefficient, state)."""
    n, B = 5 * 40960 + 4096 + 5, 40960           # 6 buckets; the last of 4101 elements
    job = Job(n, N, stage, B, 8, dtype=dtype, shadow=False, loss_scale=64.0, dynamic=True, max_norm=max_norm,
              sigma=0.02)
    inf = synth.inf_bits(dtype)
    for t, inject in ((1, ()), (2, ((N - 1, n - 3, inf),)), (3, ()), (4, ())):
        res, ref = job.step(job.make_grads(t, inject))
        assert res.path == 1 and res.overflow == (1 if inject else 0)
        job.check(res, ref)
        if max_norm > 0 and not inject:
            assert 0.0 < res.clip_coef < 1.0


@pytest.mark.parametrize("N", [1, 2])
def test_staged_pass1_many_tiles_per_block_and_staging(N):
    """One bucket of 2^24 + 8 * 1000 + 3 elements -- more tiles than blocks
    resident at once, so every block cycles its stage ring several times --
    through the per-bucket protocol with gradient windows in separate staging
    buffers, clipped; then the same through the device-state step."""
    n, B = (1 << 24) + 8 * 1000 + 3, 1 << 24
    job = Job(n, N, 2, B, 8, dtype=FP16, shadow=False, loss_scale=1.0, max_norm=1.0)
    s = torch.cuda.current_stream()
    grads = job.make_grads(1)
    staging = [torch.empty(B, dtype=torch.int16, device="cuda") for _ in range(N)]
    zg.zero_step_begin(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
    for b in range(job.plan.n_buckets):
        lo, hi = b * B, min((b + 1) * B, n)
        for r in range(N):
            staging[r][:hi - lo].copy_(torch.from_numpy(grads[r][lo:hi].view(np.int16)))
        zg.zero_step_bucket(job.cfg, job.plan, job.bufs, job.adam, job.state, b, [t.data_ptr() for t in staging], s)
    res = zg.zero_step_end(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
    torch.cuda.synchronize()
    job.check(res, job.oracle_step(grads))
    assert 0.0 < res.clip_coef < 1.0
    dev = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device="cuda")
    zg.zero_dev_state_init(dev, job.adam, job.state, s)
    grads = job.make_grads(2)
    job.load_grads(grads)
    zg.zero_step_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
    st, last = zg.zero_dev_state_read(dev, s)
    job.state = st
    ref = job.oracle_step(grads)
    last.path = 1
    job.check(last, ref)


@pytest.mark.parametrize("stage,shadow,max_norm,api", [(2, True, 0.0, "sync"), (3, True, 0.0, "async"),
                                                       (2, False, 1.0, "async"), (1, True, 0.0, "sync"),
                                                       (3, False, 0.0, "sync")])
def test_bucket_runs(stage, shadow, max_norm, api):
    """Buckets given to the library in runs (zero_step_buckets and its
    device-state twin): runs of 1-3 buckets in an arbitrary order, whose
    consecutive kernels overlap their edges; stages 2/3 from separate
    windows per bucket (the flat pointer table), stage 1 from the full
    gradient buffers.  Two steps, each against the oracle bit for bit."""
    n, N, B = 7 * 3000 + 13, 4, 3000
    job = Job(n, N, stage, B, 8, shadow=shadow, max_norm=max_norm, loss_scale=16.0)
    s = torch.cuda.current_stream()
    runs = [[6, 5], [0], [3, 1, 2], [4, 7]]
    dev = None
    if api == "async":
        dev = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device="cuda")
        zg.zero_dev_state_init(dev, job.adam, job.state, s)
    for t in (1, 2):
        grads = job.make_grads(t)
        if stage >= 2:
            win = [[torch.from_numpy(grads[r][b * B:min((b + 1) * B, n)].view(np.int16).copy()).cuda()
                    for r in range(N)] for b in range(job.plan.n_buckets)]
        else:
            job.load_grads(grads)
        if api == "sync":
            zg.zero_step_begin(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
        else:
            zg.zero_step_begin_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
        for run in runs:
            table = [[w.data_ptr() for w in win[b]] for b in run] if stage >= 2 else None
            if api == "sync":
                zg.zero_step_buckets(job.cfg, job.plan, job.bufs, job.adam, job.state, run, table, s)
            else:
                zg.zero_step_buckets_async(job.cfg, job.plan, job.bufs, job.adam, run, table, s)
        if api == "sync":
            res = zg.zero_step_end(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
        else:
            zg.zero_step_end_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
            st, res = zg.zero_dev_state_read(dev, s)
            job.state = st
            res.path = 0 if (shadow and max_norm == 0) else 1
        torch.cuda.synchronize()
        ref = job.oracle_step(grads)
        job.check(res, ref)


def test_staged_wait_that_runs_out_reports_etimeout(monkeypatch):
    """The staged pass 1's waits are bounded.  With the test hook
    ZERO_TEST_WITHHOLD_TILE set, block 0 announces its first tile's bytes to
    the stage's mbarrier but issues no copy, so its consumers' wait for that
    tile, and its producer's wait for the stage's release, run out after 2 s
    of global time.  The step is not applied and returns ZERO_ETIMEOUT (the
    device-state step: zero_dev_state_read does), t and the loss scale
    unchanged.  With the hook cleared the next steps run on the same context
    and match the oracle."""
    n, B, N = 3 * 40960 + 5, 40960, 2
    job = Job(n, N, 2, B, 8, shadow=False, max_norm=1.0, loss_scale=64.0, dynamic=True)
    s = torch.cuda.current_stream()
    res, ref = job.step(job.make_grads(1))
    job.check(res, ref)
    before = [as_u32(t[:n]).copy() for t in job.bufs.state()]
    p_before = as_u16(job.bufs.params16[1][:n]).copy()
    grads = job.make_grads(2)
    job.load_grads(grads)
    monkeypatch.setenv("ZERO_TEST_WITHHOLD_TILE", "1")
    with pytest.raises(zg.ZeroError) as e:
        zg.zero_step_stage2(job.cfg, job.plan, job.bufs, job.adam, job.state, s)
    assert e.value.status == zg.ZERO_ETIMEOUT and "bounded wait" in str(e.value)
    monkeypatch.delenv("ZERO_TEST_WITHHOLD_TILE")
    assert job.state.t == 1 and job.state.loss_scale == 64.0
    for a, b in zip(before, job.bufs.state()):
        assert np.array_equal(a, as_u32(b[:n]))
    assert np.array_equal(p_before, as_u16(job.bufs.params16[1][:n]))
    res, ref = job.step(grads)                       # the same step again, now normally
    job.check(res, ref)
    # the device-state step
    dev = torch.zeros(zg.DEV_STATE_BYTES // 8, dtype=torch.int64, device="cuda")
    zg.zero_dev_state_init(dev, job.adam, job.state, s)
    grads = job.make_grads(3)
    job.load_grads(grads)
    monkeypatch.setenv("ZERO_TEST_WITHHOLD_TILE", "1")
    zg.zero_step_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
    monkeypatch.delenv("ZERO_TEST_WITHHOLD_TILE")
    with pytest.raises(zg.ZeroError) as e:
        zg.zero_dev_state_read(dev, s)
    assert e.value.status == zg.ZERO_ETIMEOUT
    zg.zero_step_async(job.cfg, job.plan, job.bufs, job.adam, dev, s)
    st, last = zg.zero_dev_state_read(dev, s)
    assert st.t == 3 and st.loss_scale == 64.0
    job.state = st
    last.path = 1
    job.check(last, job.oracle_step(grads))


@pytest.mark.parametrize("N,stage", [(1, 2), (2, 2), (2, 0), (4, 3)])
def test_clip_norm_f16_fast_path_edges(N, stage):
    """The binary16 sum of squares adds a group's eight squares with integer
    multiply-adds when no exponent field reaches 20 (|h| < 32).  Groups at
    that edge: eight times the largest such value (31.98: the largest 64-bit
    group sum), one value at 32 among small ones (the per-value path),
    subnormals, zeros, mixed signs; one or two ranks (the staged pass 1), and
    the per-thread pass 1 (stage 0, four ranks).  Norm, clip coefficient and
    state equal the oracle's bit for bit."""
    kinds = [0x4FFF, 0xCFFF, 0x5000, 0x0001, 0x8003, 0x0000, 0x3C00, 0x4BFF]
    rng = np.random.default_rng(N * 10 + stage)
    groups = []
    for g in range(4096):
        c = g % 5
        if c == 0:
            grp = [kinds[int(rng.integers(0, 2))]] * 8             # all at the largest fast-path magnitude
        elif c == 1:
            grp = [int(rng.integers(0, 0x4FFF + 1)) | (0x8000 if rng.integers(0, 2) else 0) for _ in range(8)]
        elif c == 2:                                               # one value at 32: the per-value path
            grp = [int(rng.integers(0, 0x3000)) for _ in range(8)]
            grp[int(rng.integers(0, 8))] = 0x5000
        elif c == 3:
            grp = [int(rng.choice(kinds)) for _ in range(8)]
        else:
            grp = [int(rng.integers(0, 0x0400)) for _ in range(8)]  # subnormals and zero
        groups.extend(grp)
    n = len(groups) + 5
    h = np.array(groups + [0x4FFF] * 5, np.uint16)
    job = Job(n, N, stage, 8192, 8, dtype=FP16, shadow=False, max_norm=1.0, loss_scale=1.0)
    # rank 0 carries h, the others +0, so the reduced gradient is h itself
    grads = [h.copy()] + [np.zeros(n, np.uint16) for _ in range(N - 1)]
    res, ref = job.step(grads)
    assert res.overflow == 0 and res.path == 1
    job.check(res, ref)
    assert 0.0 < res.clip_coef < 1.0
