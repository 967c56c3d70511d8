"""The library used from plain C (tests/c_client/zero_c_client.c): cudaMalloc'd
buffers, zero_plan and zero_step_stage2 called directly -- or the step state
in device memory and two CUDA graphs captured from zero_step_async, replayed
alternately -- no Python or PyTorch in the client.  Its results must equal
the oracle's."""
import os
import subprocess

import numpy as np
import pytest

import oracle
import synth
import zero_sharded_mixed_bucket_gb300 as zg
from tests.conftest import ROOT

CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
SRC = os.path.join(ROOT, "tests", "c_client", "zero_c_client.c")


def build_client(out_dir):
    exe = os.path.join(out_dir, "zero_c_client")
    lib_dir = os.path.dirname(zg.lib_path())
    subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-o", exe, SRC, "-I" + os.path.join(ROOT, "include"),
                    "-I" + os.path.join(CUDA, "include"), "-L" + lib_dir, "-lzero_gb300",
                    "-Wl,-rpath," + lib_dir, "-L" + os.path.join(CUDA, "lib64"), "-lcudart",
                    "-Wl,-rpath," + os.path.join(CUDA, "lib64")], check=True)
    return exe


def test_client_compiles_against_the_header(tmp_path):
    zg.lib()
    build_client(str(tmp_path))


@pytest.mark.gpu
@pytest.mark.parametrize("mode", ["sync", "graph"])
def test_c_client_matches_oracle(tmp_path, mode):
    n, N, steps, lr, S = 3 * 4096 + 21, 3, 3, 1e-4, 256.0
    w0 = synth.host_normal32(n, 0.02, seed=5, stream=synth.STREAM_WEIGHT)
    grads = [[synth.host_normal16(n, synth.FP16, 1e-3 * S, seed=5, stream=synth.STREAM_GRAD, step=k, rank=r)
              for r in range(N)] for k in range(steps)]
    grads[1][2][10] = 0x7C00                     # step 2 overflows: skipped, scale halved
    with open(tmp_path / "in.bin", "wb") as f:
        f.write(np.array([n], np.int64).tobytes() + np.array([N, steps], np.int32).tobytes()
                + np.array([lr, S], np.float32).tobytes() + w0.tobytes())
        for k in range(steps):
            for r in range(N):
                f.write(grads[k][r].tobytes())
    exe = build_client(str(tmp_path))
    subprocess.run([exe, str(tmp_path)] + (["graph"] if mode == "graph" else []), check=True)
    raw = open(tmp_path / "out.bin", "rb").read()
    w = np.frombuffer(raw, np.float32, n, 0)
    m = np.frombuffer(raw, np.float32, n, 4 * n)
    v = np.frombuffer(raw, np.float32, n, 8 * n)
    p = [np.frombuffer(raw, np.uint16, n, 12 * n + 2 * n * r) for r in range(N)]
    t, = np.frombuffer(raw, np.int64, 1, 12 * n + 2 * n * N)
    ow, om, ov = w0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    ot, scale = 0, S
    for k in range(steps):
        # the client's gradients for step k+1 were generated at the initial scale;
        # the oracle sees exactly those bits and the loss scale in force
        ref = oracle.step(grads[k], ow, om, ov, dtype=oracle.FP16, lr=lr, beta1=0.9, beta2=0.999, eps=1e-8, t=ot,
                          loss_scale=scale, dynamic=True)
        ot, scale = ref["t"], ref["loss_scale"]
    assert t == ot == 2
    assert np.array_equal(w.view(np.uint32), ow.view(np.uint32))
    assert np.array_equal(m.view(np.uint32), om.view(np.uint32))
    assert np.array_equal(v.view(np.uint32), ov.view(np.uint32))
    for r in range(N):
        assert np.array_equal(p[r], ref["p16"])
