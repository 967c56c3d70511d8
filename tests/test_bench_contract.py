"""bench.py's output contract: one JSON line with the keys and types the
benchmark's readers rely on.  The reference arm (the CPU oracle) runs here
on the CPU; the GPU arm runs on the GPU (marked)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, timeout):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args], cwd=ROOT, capture_output=True,
                       text=True, timeout=timeout)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout[-2000:]
    return json.loads(lines[0])


BASE_KEYS = {"metric": str, "value": float, "unit": str, "n_gpus": int, "steps": int, "warmup": int,
             "ms_per_step": float, "higher_is_better": bool, "scaling": str, "dtype": str, "data": str,
             "config": dict}


def _check_base(d, steps, warmup):
    for k, t in BASE_KEYS.items():
        assert k in d, k
        assert isinstance(d[k], t) or (t is float and isinstance(d[k], int)), (k, d[k])
    assert "vs_baseline" in d and d["vs_baseline"] is None
    assert d["steps"] == steps and d["warmup"] == warmup and d["n_gpus"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert "workload" in d["config"]


def test_reference_arm_line():
    d = _run(["--impl", "reference", "--steps", "1", "--warmup", "3"], timeout=600)
    _check_base(d, 1, 3)
    assert d["impl"] == "reference"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == d["value"] and cb["sample"]
    e = d["e2e"]
    assert e["value"] == d["value"] and e["unit"] == d["unit"]
    assert e["h2d_bytes_per_step"] == 0 and e["d2h_bytes_per_step"] == 0


def test_warmup_below_three_is_refused():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--warmup", "2"], cwd=ROOT,
                       capture_output=True, text=True, timeout=120)
    assert r.returncode != 0 and "warm-up" in r.stderr


@pytest.mark.gpu
def test_gpu_arm_line():
    """The default line: the stage-3 step at 6.65B parameters (about 210 GB
    of device memory, in a child process), its legs, end to end and the CPU
    baseline."""
    import torch
    torch.cuda.empty_cache()
    d = _run(["--steps", "4", "--warmup", "3", "--e2e-steps", "1"], timeout=1200)
    _check_base(d, 4, 3)
    assert d["config"]["n_params"] == 6_648_827_904 and d["config"]["stage"] == 3
    assert d["config"]["n_ranks"] == 64
    r = d["roofline"]
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["peak"] > 0
    assert r["frac"] == pytest.approx(r["achieved"] / r["peak"])
    assert r["traffic"] is None or (r["traffic"] > 0 and r["traffic_source"]["summary"])
    assert 0.5 < r["share_of_step_bytes"] < 0.7
    # the gather mostly writes: beside the copy bandwidth, the write-only
    # ceiling measured on the same GPU, which the gather cannot pass by much
    w = r["write_only_ceiling"]
    assert w["gbs"] > 0 and w["frac"] == pytest.approx(r["achieved"] / w["gbs"]) and w["frac"] < 1.1
    assert d["step_roofline"]["bytes_per_param"] == 414
    e = d["e2e"]
    assert e["value"] > 0 and e["h2d_bytes_per_step"] > 0 and e["d2h_bytes_per_step"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["host_cores"] >= 1 and cb["value"] > 0
    c = d["clocks"]
    assert {"sm_mhz", "sm_max_mhz", "reasons"} <= set(c)
    # per step: prepare, 2 x 33 gathers, 397 bucket kernels, restore/commit
    assert d["gpu_launches"] == 4 * (1 + 66 + 397 + 1)
    assert r["launches"] == 1 * 66
    legs = d["legs"]
    for name in ("workload2_stage2", "clip_2p31_n2_bf16", "clip_2p31_n32_bf16"):
        assert "error" not in legs[name], legs[name]
        assert legs[name]["roofline"]["frac"] > 0
