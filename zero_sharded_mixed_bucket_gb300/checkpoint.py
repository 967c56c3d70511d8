"""Checkpoint and resume of a ZeRO job's sharded state.

Each simulated rank writes its own partition, as a data-parallel rank of a
ZeRO job would: rank r's slice [r*P, (r+1)*P) of the fp32 master weights and
of the optimizer state the optimizer keeps (stages 1-3; in stage 0 every rank
holds the full state and rank r writes its replica), and its 16-bit
parameters (the full vector in stages 0-2, its shard in stage 3).  A JSON
manifest records the config and the host-side step state (t, loss scale,
clean-step count).  Resuming restores everything into the current state copy
and continues bit for bit.  Host I/O only: no kernel runs here.
"""
from __future__ import annotations

import json
import os

import numpy as np

from . import ZERO_ADAM, ZERO_SGD, ZERO_SGD_MOMENTUM, Config, zero_config_t, zero_state_t

_ARRAYS = {ZERO_ADAM: ("w", "m", "v"), ZERO_SGD_MOMENTUM: ("w", "m"), ZERO_SGD: ("w",)}


def _c(cfg):
    return cfg.c if isinstance(cfg, Config) else cfg


def _slices(c, plan, r):
    """(state slice, parameter slice) of rank r."""
    P, pad = plan.shard_elems, plan.padded_elems
    n = c.n_params
    if c.stage == 0:
        st = slice(r * pad, r * pad + n)
    else:
        st = slice(min(r * P, n), min((r + 1) * P, n))
    pr = slice(0, max(0, min(P, n - r * P))) if c.stage == 3 else slice(0, n)
    return st, pr


def save_checkpoint(path: str, cfg, plan, bufs, state: zero_state_t) -> None:
    c = _c(cfg)
    os.makedirs(path, exist_ok=True)
    arrays = _ARRAYS[c.optimizer]
    k = bufs.cur
    for r in range(c.n_ranks):
        st, pr = _slices(c, plan, r)
        data = {name: getattr(bufs, name)[k][st].detach().cpu().numpy() for name in arrays}
        data["params16"] = bufs.params16[r][pr].detach().cpu().numpy()
        np.savez(os.path.join(path, "rank%05d.npz" % r), **data)
    manifest = {
        "format": "zero-gb300 sharded checkpoint 1",
        "config": {f: getattr(c, f) for f in ("n_params", "bucket_elems", "align_elems", "stage", "n_ranks",
                                              "dtype", "optimizer")},
        "layer_sizes": [int(c.layer_sizes[i]) for i in range(c.n_layers)] if c.n_layers else None,
        "shard_elems": plan.shard_elems,
        "state": {f: getattr(state, f) for f in ("t", "loss_scale", "min_loss_scale", "dynamic", "growth_interval",
                                                 "good_steps")},
    }
    with open(os.path.join(path, "manifest.json"), "w") as f:
        json.dump(manifest, f, indent=1)


def load_checkpoint(path: str, cfg, plan, bufs, state: zero_state_t) -> None:
    """Restore into bufs' current state copy and into `state`.  The config
    must describe the same job (sizes, layer split, stage, ranks, dtype,
    optimizer); ValueError otherwise."""
    import torch
    c = _c(cfg)
    with open(os.path.join(path, "manifest.json")) as f:
        man = json.load(f)
    for key, val in man["config"].items():
        if getattr(c, key) != val:
            raise ValueError("checkpoint was written for %s=%r, the config has %r" % (key, val, getattr(c, key)))
    if man["shard_elems"] != plan.shard_elems:
        raise ValueError("checkpoint partition differs from the plan")
    # the layer split fixes the stage-3 gather units and the fetch offsets
    layers = [int(c.layer_sizes[i]) for i in range(c.n_layers)] if c.n_layers else None
    if man.get("layer_sizes") != layers:
        raise ValueError("checkpoint was written for layer sizes %r, the config has %r"
                         % (man.get("layer_sizes"), layers))
    arrays = _ARRAYS[c.optimizer]
    k = bufs.cur
    for r in range(c.n_ranks):
        st, pr = _slices(c, plan, r)
        with np.load(os.path.join(path, "rank%05d.npz" % r)) as z:
            for name in arrays:
                getattr(bufs, name)[k][st].copy_(torch.from_numpy(z[name]))
            bufs.params16[r][pr].copy_(torch.from_numpy(z["params16"]))
    for f, val in man["state"].items():
        setattr(state, f, val)
