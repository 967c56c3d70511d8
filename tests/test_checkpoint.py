"""Checkpoint / resume of the sharded state: a CPU round trip of the files,
and on the GPU a bit-identical continuation after resuming into fresh
buffers."""
import numpy as np
import pytest
import torch

import zero_sharded_mixed_bucket_gb300 as zg
from zero_sharded_mixed_bucket_gb300.checkpoint import load_checkpoint, save_checkpoint


@pytest.mark.parametrize("stage", [0, 1, 2, 3])
@pytest.mark.parametrize("optimizer", [zg.ZERO_ADAM, zg.ZERO_SGD_MOMENTUM])
def test_round_trip_files_cpu(tmp_path, stage, optimizer):
    cfg = zg.Config(10_003, 3, stage, 1024, 8, None, zg.ZERO_FP16, optimizer)
    plan = zg.zero_plan(cfg)
    a = zg.DeviceBuffers(cfg, plan, device="cpu")
    g = torch.Generator().manual_seed(stage)
    for name in ("w", "m", "v"):
        for t in getattr(a, name):
            t.copy_(torch.randn(t.shape, generator=g))
    for t in a.params16:
        t.copy_(torch.randint(-30000, 30000, t.shape, dtype=torch.int16, generator=g))
    st = zg.zero_state_t(t=7, loss_scale=256.0, min_loss_scale=1.0, dynamic=1, growth_interval=5, good_steps=3)
    save_checkpoint(str(tmp_path), cfg, plan, a, st)
    b = zg.DeviceBuffers(cfg, plan, device="cpu")
    st2 = zg.zero_state_t()
    load_checkpoint(str(tmp_path), cfg, plan, b, st2)
    n = 10_003
    used = ("w", "m", "v") if optimizer == zg.ZERO_ADAM else ("w", "m")
    reps = 3 if stage == 0 else 1
    for name in used:
        for r in range(reps):
            off = r * plan.padded_elems
            assert torch.equal(getattr(a, name)[0][off:off + n], getattr(b, name)[0][off:off + n])
    for r in range(3):
        m = plan.param16_elems if stage == 3 else n
        m = min(m, max(0, n - r * plan.shard_elems)) if stage == 3 else n
        assert torch.equal(a.params16[r][:m], b.params16[r][:m])
    assert (st2.t, st2.loss_scale, st2.good_steps, st2.dynamic) == (7, 256.0, 3, 1)
    with pytest.raises(ValueError):
        load_checkpoint(str(tmp_path), zg.Config(10_003, 3, stage, 2048, 8, None, zg.ZERO_FP16, optimizer),
                        zg.zero_plan(zg.Config(10_003, 3, stage, 2048, 8, None, zg.ZERO_FP16, optimizer)), b, st2)


def test_resume_rejects_another_layer_split(tmp_path):
    """Same size, stage, ranks and partition, but another split into layers:
    the stage-3 gather units and the fetch offsets would no longer match the
    saved job, so resuming is refused."""
    layers = [4000, 3000, 3003]
    cfg = zg.Config(10_003, 3, 3, 1024, 8, layers)
    plan = zg.zero_plan(cfg)
    a = zg.DeviceBuffers(cfg, plan, device="cpu")
    st = zg.zero_state_t(t=1, loss_scale=1.0, min_loss_scale=1.0)
    save_checkpoint(str(tmp_path), cfg, plan, a, st)
    load_checkpoint(str(tmp_path), cfg, plan, zg.DeviceBuffers(cfg, plan, device="cpu"), zg.zero_state_t())
    for other in ([4000, 3003, 3000], None):
        cfg2 = zg.Config(10_003, 3, 3, 1024, 8, other)
        plan2 = zg.zero_plan(cfg2)
        assert plan2.shard_elems == plan.shard_elems
        with pytest.raises(ValueError, match="layer sizes"):
            load_checkpoint(str(tmp_path), cfg2, plan2, zg.DeviceBuffers(cfg2, plan2, device="cpu"),
                            zg.zero_state_t())


@pytest.mark.gpu
@pytest.mark.parametrize("stage", [1, 3])
def test_resume_continues_bit_for_bit(tmp_path, stage):
    from tests.gpu_harness import Job, as_u16, as_u32
    n = 3 * 4096 + 11
    a = Job(n, 4, stage, 4096, 8, loss_scale=64.0, dynamic=True, growth=2)
    for t in (1, 2):
        a.step(a.make_grads(t))
    save_checkpoint(str(tmp_path), a.cfg, a.plan, a.bufs, a.state)
    later = {}
    for t in (3, 4):
        later[t] = a.make_grads(t)       # generated at the loss scale of that step
        a.step(later[t])
    b = Job(n, 4, stage, 4096, 8, loss_scale=1.0, dynamic=True, growth=2)
    load_checkpoint(str(tmp_path), b.cfg, b.plan, b.bufs, b.state)
    assert b.state.t == 2
    for t in (3, 4):
        b.load_grads(later[t])           # the uninterrupted run's gradients
        fn = zg.zero_step_stage1 if stage == 1 else zg.zero_step_stage3
        fn(b.cfg, b.plan, b.bufs, b.adam, b.state, torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert (b.state.t, b.state.loss_scale, b.state.good_steps) == (a.state.t, a.state.loss_scale, a.state.good_steps)
    for x, y in zip(a.bufs.state(), b.bufs.state()):
        assert np.array_equal(as_u32(x[:n]), as_u32(y[:n]))
    for r in range(4):
        assert torch.equal(a.bufs.params16[r], b.bufs.params16[r])
