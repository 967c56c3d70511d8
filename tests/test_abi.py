"""The C-ABI library on the CPU: it loads, exports every function the header
declares, its structs have the header's sizes, and its host-side logic --
planning, accounting, argument checks -- agrees with the oracle and the
pages.  No call here reaches a CUDA API: every step call is rejected by the
host checks before any launch."""
import ctypes
import os
import re
from fractions import Fraction

import pytest

import oracle
import zero_sharded_mixed_bucket_gb300 as zg
from tests.conftest import ROOT, read_golden

HEADER = os.path.join(ROOT, "include", "zero_gb300.h")


def _declared_functions():
    text = open(HEADER, encoding="utf-8").read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zero_[a-z0-9_]+)\s*\(", text)))


def test_library_exports_every_declared_function():
    names = _declared_functions()
    assert len(names) >= 15
    L = ctypes.CDLL(zg.lib_path())
    for n in names:
        assert hasattr(L, n), n
    assert zg.zero_version() == 1


def test_struct_sizes_match_header():
    text = open(HEADER, encoding="utf-8").read()
    for name, cls in [("zero_config", zg.zero_config_t), ("zero_plan", zg.zero_plan_t), ("zero_adam", zg.zero_adam_t),
                      ("zero_state", zg.zero_state_t), ("zero_buffers", zg.zero_buffers_t),
                      ("zero_step_result", zg.zero_step_result_t), ("zero_pa_plan", zg.zero_pa_plan_t)]:
        m = re.search(r"(\d+) bytes\. \*/\s*typedef struct %s \{" % name, text)
        assert m, name
        assert ctypes.sizeof(cls) == int(m.group(1)), name


CONFIGS = [
    (1 << 20, 4, 2, 1 << 24, 0, None),
    (123_568_896, 8, 2, 1 << 24, 0, None),
    (1_555_278_400, 8, 2, 500_000_000, 0, None),
    (6_648_827_904, 64, 3, 1 << 24, 0, [50257 * 4096] + [12 * 4096 * 4096 + 4 * 4096] * 32),
    (1, 1, 0, 8, 8, None),
    (7, 3, 1, 8, 16, None),
    (0, 5, 2, 64, 0, None),
    (100_003, 7, 3, 4096, 64, [3, 100_000]),
]


@pytest.mark.parametrize("n,N,stage,B,A,layers", CONFIGS)
def test_plan_matches_oracle(n, N, stage, B, A, layers):
    p = zg.zero_plan(zg.Config(n, N, stage, B, A, layers))
    o = oracle.plan(n, N, B, A, layers)
    assert p.shard_elems == o["shard"] and p.padded_elems == o["padded"]
    assert p.n_buckets == o["n_buckets"] and p.max_layer_elems == o["max_layer"]
    assert p.n_layers == len(o["layer_sizes"])
    assert p.state_elems == (N * o["padded"] if stage == 0 else o["padded"])
    assert p.param16_elems == (o["shard"] if stage == 3 else o["padded"])
    assert p.hbm_bytes_fused == oracle.hbm_bytes_per_param(N, stage, "fused") * n
    assert p.hbm_bytes_two_pass == oracle.hbm_bytes_per_param(N, stage, "two_pass") * n
    for opt, name in ((zg.ZERO_SGD_MOMENTUM, "sgdm"), (zg.ZERO_SGD, "sgd")):
        q = zg.zero_plan(zg.Config(n, N, stage, B, A, layers, zg.ZERO_FP16, opt))
        K = oracle.OPTIM_K[name]
        assert q.hbm_bytes_fused == oracle.hbm_bytes_per_param(N, stage, "fused", K) * n
        assert q.hbm_bytes_two_pass == oracle.hbm_bytes_per_param(N, stage, "two_pass", K) * n
        exact = oracle.model_state_bytes(n, N, stage, K=K)["total"]
        assert abs(Fraction(q.mem_total_bytes) - exact) <= exact * Fraction(1, 10 ** 15)
    for opt, name in ((zg.ZERO_ADAM, "adam"), (zg.ZERO_SGD_MOMENTUM, "sgdm"), (zg.ZERO_SGD, "sgd")):
        # fp32 training: 4-byte gradients and parameters, the same fp32 state
        q = zg.zero_plan(zg.Config(n, N, stage, B, A, layers, zg.ZERO_FP32, opt))
        K = oracle.OPTIM_K[name]
        assert (q.shard_elems, q.padded_elems, q.grad16_elems) == (p.shard_elems, p.padded_elems, p.grad16_elems)
        assert q.hbm_bytes_fused == oracle.hbm_bytes_per_param(N, stage, "fused", K, 4) * n
        assert q.hbm_bytes_two_pass == oracle.hbm_bytes_per_param(N, stage, "two_pass", K, 4) * n
        c4 = oracle.comm_bytes(n, N, stage, b=4)
        assert q.comm_counted_bytes == c4["counted"] and Fraction(q.comm_paper_bytes) == c4["paper"]
        exact = oracle.model_state_bytes(n, N, stage, b=4, K=K)["total"]
        assert abs(Fraction(q.mem_total_bytes) - exact) <= exact * Fraction(1, 10 ** 15)
    c = oracle.comm_bytes(n, N, stage)
    assert p.comm_counted_bytes == c["counted"] and Fraction(p.comm_paper_bytes) == c["paper"]
    # a double: exact when N is a power of two, else within a few ulps
    exact = oracle.model_state_bytes(n, N, stage)["total"]
    assert abs(Fraction(p.mem_total_bytes) - exact) <= exact * Fraction(1, 10 ** 15)
    for b in sorted({0, o["n_buckets"] // 2, o["n_buckets"] - 1}):
        if not 0 <= b < o["n_buckets"]:
            continue
        assert zg.zero_plan_bucket(zg.Config(n, N, stage, B, A, layers), b) == oracle.bucket_segments(o, b)
    if layers:
        for l in range(len(layers)):
            assert zg.zero_plan_layer(zg.Config(n, N, stage, B, A, layers), l) == (o["layer_starts"][l], layers[l])


@pytest.mark.parametrize("N", [1, 2, 3, 4, 7])
@pytest.mark.parametrize("n", [1, 9, 63, 65, 200])
def test_bucket_segments_brute_force(N, n):
    cfg = zg.Config(n, N, 2, 16, 8)
    p = zg.zero_plan(cfg)
    o = oracle.plan(n, N, 16, 8)
    for b in range(p.n_buckets):
        assert zg.zero_plan_bucket(cfg, b) == oracle.bucket_segments(o, b)


def test_table1_through_the_library():
    sizes = {"7.5B": 7_500_000_000, "128B": 128_000_000_000, "1T": 1_000_000_000_000}
    for row in read_golden("table1_model_state_gb.txt"):
        n = int(row[0])
        for si, size in enumerate(sizes):
            for stage in (1, 2, 3):
                total = zg.zero_model_state_bytes(sizes[size], n, stage)[3]
                assert oracle.display_gb(Fraction(total) / 10 ** 9) == row[1 + 3 * si + stage - 1]


def test_examples_and_comm_through_the_library():
    for name, psi, n, b, K, stage, total in read_golden("worked_examples.txt"):
        psi_i = int(float(psi))
        got = zg.zero_model_state_bytes(psi_i, int(n), int(stage), int(b), int(K))[3]
        assert Fraction(got) / 10 ** 9 == Fraction(total), (name, stage)
    assert zg.zero_comm_bytes(7_500_000_000, 64, 2)[0] == 30e9
    assert zg.zero_comm_bytes(7_500_000_000, 64, 3)[0] == 45e9
    assert zg.zero_comm_bytes(128_000_000_000, 64, 0)[0] == 512e9
    assert zg.zero_comm_bytes(128_000_000_000, 64, 3)[0] == 768e9
    for stage in range(4):
        assert zg.zero_comm_bytes(10 ** 9, 8, stage)[1] == oracle.comm_bytes(10 ** 9, 8, stage)["counted"]


@pytest.mark.parametrize("kw,status", [
    (dict(n_ranks=0), zg.ZERO_EUNSUPPORTED),
    (dict(n_ranks=65), zg.ZERO_EUNSUPPORTED),
    (dict(stage=4), zg.ZERO_EINVAL),
    (dict(bucket_elems=12), zg.ZERO_EINVAL),
    (dict(bucket_elems=0), zg.ZERO_EINVAL),
    (dict(align_elems=6), zg.ZERO_EINVAL),
    (dict(n_params=-1), zg.ZERO_EINVAL),
    (dict(dtype=3), zg.ZERO_EINVAL),
    (dict(optimizer=3), zg.ZERO_EINVAL),
])
def test_config_rejected(kw, status):
    base = dict(n_params=1000, n_ranks=4, stage=2, bucket_elems=64, align_elems=0, dtype=0, optimizer=0)
    base.update(kw)
    cfg = zg.zero_config_t(**base)
    with pytest.raises(zg.ZeroError) as e:
        zg.zero_plan(cfg)
    assert e.value.status == status
    assert zg.zero_last_error()


def test_layer_sizes_checked():
    with pytest.raises(zg.ZeroError) as e:
        zg.zero_plan(zg.Config(100, 2, 3, 16, 0, [50, 49]))
    assert e.value.status == zg.ZERO_EINVAL
    with pytest.raises(zg.ZeroError):
        zg.zero_plan(zg.Config(100, 2, 3, 16, 0, [50, 0, 50]))


class _FakeBuffers:
    """zero_buffers_t with made-up device addresses; only the host checks
    ever see them."""

    def __init__(self, N, good=0x10000000, bad=None):
        self.gp = (ctypes.c_void_p * N)(*[good + 0x100000 * r for r in range(N)])
        self.pp = (ctypes.c_void_p * N)(*[good + 0x8000000 + 0x100000 * r for r in range(N)])
        b = zg.zero_buffers_t()
        b.grads = ctypes.cast(self.gp, ctypes.POINTER(ctypes.c_void_p))
        b.params16 = ctypes.cast(self.pp, ctypes.POINTER(ctypes.c_void_p))
        for k in range(2):
            b.w[k] = good + 0x20000000 + k * 0x1000000
            b.m[k] = good + 0x30000000 + k * 0x1000000
            b.v[k] = good + 0x40000000 + k * 0x1000000
        b.reduced = good + 0x50000000
        b.workspace = good + 0x60000000
        self.b = b


def _step_status(cfg, plan, fb, adam=None, state=None):
    adam = adam or zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8)
    state = state or zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
    res = zg.zero_step_result_t()
    return zg.lib().zero_step(ctypes.byref(cfg.c), ctypes.byref(plan), ctypes.byref(fb.b), ctypes.byref(adam),
                              ctypes.byref(state), None, ctypes.byref(res))


def test_step_argument_checks_reject_before_any_launch():
    cfg = zg.Config(1000, 4, 2, 64)
    plan = zg.zero_plan(cfg)
    fb = _FakeBuffers(4)
    fb.pp[2] = 0x10000008                      # misaligned parameter buffer
    assert _step_status(cfg, plan, fb) == zg.ZERO_EALIGN
    assert "params16[2]" in zg.zero_last_error()
    fb = _FakeBuffers(4)
    fb.b.workspace = 0x10000004
    assert _step_status(cfg, plan, fb) == zg.ZERO_EALIGN
    fb = _FakeBuffers(4)
    fb.b.workspace = None
    assert _step_status(cfg, plan, fb) == zg.ZERO_ENOMEM
    fb = _FakeBuffers(4)
    fb.gp[3] = None
    assert _step_status(cfg, plan, fb) == zg.ZERO_ENOMEM
    fb = _FakeBuffers(4)
    fb.b.cur = 2
    assert _step_status(cfg, plan, fb) == zg.ZERO_EINVAL
    # a plan for another config
    other = zg.zero_plan(zg.Config(1001, 4, 2, 64))
    assert _step_status(cfg, other, _FakeBuffers(4)) == zg.ZERO_EINVAL
    # hyper-parameters and loss scale
    assert _step_status(cfg, plan, _FakeBuffers(4), adam=zg.zero_adam_t(lr=1e-4, beta1=1.0, beta2=0.999)) == \
        zg.ZERO_EINVAL
    assert _step_status(cfg, plan, _FakeBuffers(4), state=zg.zero_state_t(loss_scale=0.0)) == zg.ZERO_EINVAL
    assert _step_status(cfg, plan, _FakeBuffers(4), state=zg.zero_state_t(loss_scale=float("inf"))) == \
        zg.ZERO_EINVAL
    # the two-pass path of stage 2 needs the reduced buffer
    fb = _FakeBuffers(4)
    fb.b.reduced = None
    assert _step_status(cfg, plan, fb, adam=zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999,
                                                           max_grad_norm=1.0)) == zg.ZERO_ENOMEM
    # fp32 training has no clipping path
    cfg32 = zg.Config(1000, 4, 2, 64, 0, None, zg.ZERO_FP32)
    plan32 = zg.zero_plan(cfg32)
    assert _step_status(cfg32, plan32, _FakeBuffers(4), adam=zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999,
                                                                           max_grad_norm=1.0)) == zg.ZERO_EUNSUPPORTED
    assert "ZERO_FP32" in zg.zero_last_error()
    res32 = zg.zero_step_result_t()
    st = zg.lib().zero_step_stage2_noalloc(ctypes.byref(cfg32.c), ctypes.byref(plan32),
                                           ctypes.byref(_FakeBuffers(4).b),
                                           ctypes.byref(zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999)),
                                           ctypes.byref(zg.zero_state_t(loss_scale=1.0)), None, ctypes.byref(res32))
    assert st == zg.ZERO_EUNSUPPORTED
    assert zg.lib().zero_plan(ctypes.byref(zg.Config(1000, 4, 2, 64, 0, None, 3).c),
                              ctypes.byref(zg.zero_plan_t())) == zg.ZERO_EINVAL
    # wrong stage entry point
    res = zg.zero_step_result_t()
    st = zg.lib().zero_step_stage3(ctypes.byref(cfg.c), ctypes.byref(plan), ctypes.byref(_FakeBuffers(4).b),
                                   ctypes.byref(zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999)),
                                   ctypes.byref(zg.zero_state_t(loss_scale=1.0)), None, ctypes.byref(res))
    assert st == zg.ZERO_EINVAL


def test_bucket_and_gather_checks():
    cfg = zg.Config(1000, 4, 1, 64)
    plan = zg.zero_plan(cfg)
    fb = _FakeBuffers(4)
    adam = zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999)
    state = zg.zero_state_t(loss_scale=1.0)
    bg = (ctypes.c_void_p * 4)(*[0x70000000] * 4)
    # stages 0/1 keep full gradients: per-bucket gradient windows are refused
    st = zg.lib().zero_step_bucket(ctypes.byref(cfg.c), ctypes.byref(plan), ctypes.byref(fb.b), ctypes.byref(adam),
                                   ctypes.byref(state), 0, bg, None)
    assert st == zg.ZERO_EINVAL
    st = zg.lib().zero_step_bucket(ctypes.byref(cfg.c), ctypes.byref(plan), ctypes.byref(fb.b), ctypes.byref(adam),
                                   ctypes.byref(state), plan.n_buckets, None, None)
    assert st == zg.ZERO_EINVAL
    # gathers belong to stage 3
    dst = (ctypes.c_void_p * 2)(0x70000000, 0x71000000)
    st = zg.lib().zero_gather_layer(ctypes.byref(cfg.c), ctypes.byref(plan), 0, fb.pp, dst, 2, None)
    assert st == zg.ZERO_EINVAL
    cfg3 = zg.Config(1000, 4, 3, 64, 0, [400, 600])
    plan3 = zg.zero_plan(cfg3)
    st = zg.lib().zero_gather_layer(ctypes.byref(cfg3.c), ctypes.byref(plan3), 2, fb.pp, dst, 2, None)
    assert st == zg.ZERO_EINVAL
    st = zg.lib().zero_gather_layer(ctypes.byref(cfg3.c), ctypes.byref(plan3), 0, fb.pp, dst, 0, None)
    assert st == zg.ZERO_EUNSUPPORTED
    dst_bad = (ctypes.c_void_p * 2)(0x70000000, 0x71000002)
    st = zg.lib().zero_gather_layer(ctypes.byref(cfg3.c), ctypes.byref(plan3), 0, fb.pp, dst_bad, 2, None)
    assert st == zg.ZERO_EALIGN


def test_bias_correction_early_exit_is_exact():
    """The library stops forming beta^t once it is below 2^-60; (float)(1 -
    beta^t) is then 1 either way.  Checked against the oracle's full loop
    through the plan-independent scalar: for large t both give 1.0."""
    for beta in (0.9, 0.99, 0.999):
        bc = oracle.bias_corrections(beta, beta, 5000)[0]
        assert bc == (1.0 if beta < 0.999 else bc)


def test_device_state_checks_reject_before_any_copy():
    cfg = zg.Config(1000, 4, 2, 64)
    plan = zg.zero_plan(cfg)
    adam = zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8)
    L = zg.lib()
    state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
    assert L.zero_dev_state_init(None, ctypes.byref(adam), ctypes.byref(state), None) == zg.ZERO_EINVAL
    assert L.zero_dev_state_init(0x10000008, ctypes.byref(adam), ctypes.byref(state), None) == zg.ZERO_EALIGN
    bad = zg.zero_state_t(t=0, loss_scale=0.0)
    assert L.zero_dev_state_init(0x10000000, ctypes.byref(adam), ctypes.byref(bad), None) == zg.ZERO_EINVAL
    bad = zg.zero_state_t(t=-1, loss_scale=1.0)
    assert L.zero_dev_state_init(0x10000000, ctypes.byref(adam), ctypes.byref(bad), None) == zg.ZERO_EINVAL
    bad = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=0.0, dynamic=1)
    assert L.zero_dev_state_init(0x10000000, ctypes.byref(adam), ctypes.byref(bad), None) == zg.ZERO_EINVAL
    one = zg.zero_adam_t(lr=1e-4, beta1=1.0, beta2=0.999)
    assert L.zero_dev_state_init(0x10000000, ctypes.byref(one), ctypes.byref(state), None) == zg.ZERO_EINVAL
    assert L.zero_dev_state_read(None, None, None, None) == zg.ZERO_EINVAL
    n = ctypes.c_int32(-1)

    def step(fb, dev=0x10000000, a=adam):
        return L.zero_step_async(ctypes.byref(cfg.c), ctypes.byref(plan), ctypes.byref(fb.b), ctypes.byref(a),
                                 dev, None, ctypes.byref(n))

    assert step(_FakeBuffers(4), dev=None) == zg.ZERO_EALIGN
    assert step(_FakeBuffers(4), dev=0x10000004) == zg.ZERO_EALIGN
    fb = _FakeBuffers(4)
    fb.pp[1] = 0x10000002
    assert step(fb) == zg.ZERO_EALIGN
    fb = _FakeBuffers(4)
    fb.gp[0] = None
    assert step(fb) == zg.ZERO_ENOMEM
    assert step(_FakeBuffers(4), a=one) == zg.ZERO_EINVAL
    assert n.value == -1                       # nothing was launched


def test_buffer_allocation_failure_propagates(monkeypatch):
    """A failing device allocation in the binding surfaces as the allocator's
    own error; nothing falls back to another memory or another path."""
    import torch
    cfg = zg.Config(1000, 2, 2, 64)
    plan = zg.zero_plan(cfg)
    calls = []
    real = torch.zeros

    def failing_zeros(*a, **kw):
        calls.append(1)
        if len(calls) == 3:
            raise torch.OutOfMemoryError("simulated: out of device memory")
        return real(*a, **{k: v for k, v in kw.items() if k != "device"})

    monkeypatch.setattr(torch, "zeros", failing_zeros)
    with pytest.raises(torch.OutOfMemoryError):
        zg.DeviceBuffers(cfg, plan, device="cuda")
    assert len(calls) == 3


@pytest.mark.parametrize("A,N,dtype,align", [(0, 1, 0, 0), (1, 1, 0, 0), (7, 3, 1, 8), (32 * 1024 * 1600, 16, 0, 0),
                                             (100_003, 64, 2, 64), (10, 64, 0, 0)])
def test_pa_plan_matches_oracle(A, N, dtype, align):
    p = zg.zero_pa_plan(A, N, dtype, align)
    b = 4 if dtype == zg.ZERO_FP32 else 2
    o = oracle.pa_plan(A, N, value_bytes=b, align_elems=align)
    assert p.shard_elems == o["shard"] and p.n_mp == N and p.act_elems == A
    assert p.mem_per_rank_bytes == o["mem_per_rank"] and p.mem_per_rank_pa_bytes == o["mem_per_rank_pa"]
    assert p.gather_bytes == sum(o["gather_recv_per_rank"])


def test_pa_argument_checks():
    for args, status in [((100, 0, 0, 0), zg.ZERO_EUNSUPPORTED), ((100, 65, 0, 0), zg.ZERO_EUNSUPPORTED),
                         ((100, 4, 3, 0), zg.ZERO_EINVAL), ((100, 4, 0, 12), zg.ZERO_EINVAL),
                         ((-1, 4, 0, 0), zg.ZERO_EINVAL)]:
        with pytest.raises(zg.ZeroError) as e:
            zg.zero_pa_plan(*args)
        assert e.value.status == status
    p = zg.zero_pa_plan(10_000, 4)
    good = [0x10000000 + 0x100000 * r for r in range(4)]
    L = zg.lib()
    arr = lambda xs: (ctypes.c_void_p * len(xs))(*xs)
    assert L.zero_pa_partition(ctypes.byref(p), arr(good), arr(good[:3] + [0x10000008]), None) == zg.ZERO_EALIGN
    assert L.zero_pa_partition(ctypes.byref(p), arr(good[:3] + [None]), arr(good), None) == zg.ZERO_ENOMEM
    assert L.zero_pa_gather(ctypes.byref(p), arr(good), arr(good[:1]), 0, None) == zg.ZERO_EUNSUPPORTED
    assert L.zero_pa_gather(ctypes.byref(p), arr(good), arr([0x10000002]), 1, None) == zg.ZERO_EALIGN
    forged = zg.zero_pa_plan_t.from_buffer_copy(p)
    forged.shard_elems += 8
    assert L.zero_pa_gather(ctypes.byref(forged), arr(good), arr(good[:1]), 1, None) == zg.ZERO_EINVAL


def test_bucket_runs_checked_before_any_launch():
    """zero_step_buckets / zero_step_buckets_async refuse a bad run on the host
    (made-up device addresses: nothing is launched)."""
    L = zg.lib()
    cfg = zg.Config(1000, 4, 2, 64)
    plan = zg.zero_plan(cfg)
    fb = _FakeBuffers(4)
    adam = zg.zero_adam_t(lr=1e-4, beta1=0.9, beta2=0.999, eps=1e-8)
    state = zg.zero_state_t(t=0, loss_scale=1.0, min_loss_scale=1.0)
    idx = lambda xs: (ctypes.c_int64 * max(1, len(xs)))(*xs)
    good = [0x70000000 + 0x100000 * r for r in range(8)]
    grads = (ctypes.c_void_p * 8)(*good)

    def both(buckets, count, g, stage_cfg=cfg, stage_plan=plan):
        a = L.zero_step_buckets(ctypes.byref(stage_cfg.c), ctypes.byref(stage_plan), ctypes.byref(fb.b),
                                ctypes.byref(adam), ctypes.byref(state), buckets, count, g, None)
        b = L.zero_step_buckets_async(ctypes.byref(stage_cfg.c), ctypes.byref(stage_plan), ctypes.byref(fb.b),
                                      ctypes.byref(adam), buckets, count, g, None)
        return a, b

    assert both(idx([0, 16]), 2, None) == (zg.ZERO_EINVAL, zg.ZERO_EINVAL)      # 16 buckets: 0..15
    assert "outside 0..15" in zg.zero_last_error()
    assert both(idx([-1]), 1, None) == (zg.ZERO_EINVAL, zg.ZERO_EINVAL)
    assert both(None, 3, None) == (zg.ZERO_EINVAL, zg.ZERO_EINVAL)
    assert both(idx([0]), -1, None) == (zg.ZERO_EINVAL, zg.ZERO_EINVAL)
    assert both(idx([]), 0, None) == (zg.ZERO_OK, zg.ZERO_OK)                    # an empty run launches nothing
    bad = (ctypes.c_void_p * 8)(*(good[:5] + [0x70000008] + good[6:]))        # bucket 1, rank 1 misaligned
    assert both(idx([2, 3]), 2, bad) == (zg.ZERO_EALIGN, zg.ZERO_EALIGN)
    assert "bucket_grads[1]" in zg.zero_last_error()
    cfg1 = zg.Config(1000, 4, 1, 64)
    plan1 = zg.zero_plan(cfg1)
    assert both(idx([0, 1]), 2, grads, cfg1, plan1) == (zg.ZERO_EINVAL, zg.ZERO_EINVAL)
    assert "stage 2 or 3" in zg.zero_last_error()
