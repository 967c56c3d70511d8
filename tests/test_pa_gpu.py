"""P_a (partitioned activation checkpoints) on the GPU against the oracle, bit
for bit: partition of every rank's replica into its slice, all-gather into
one or many destinations (chunk by chunk, destination by destination; with
the slices in host memory, each value read once and stored to every
destination), slices in device memory or in pinned host memory
(P_a+cpu), ragged sizes, 16-bit and binary32 activations, guard regions."""
import numpy as np
import pytest
import torch

import oracle
import zero_sharded_mixed_bucket_gb300 as zg
from tests.gpu_harness import as_bits

pytestmark = pytest.mark.gpu


def _run(A, N, dtype, n_dst, host_slices=False, align=0, seed=0):
    p = zg.zero_pa_plan(A, N, dtype, align)
    vt = torch.int32 if dtype == zg.ZERO_FP32 else torch.int16
    npt = np.uint32 if dtype == zg.ZERO_FP32 else np.uint16
    rng = np.random.default_rng(seed)
    x = rng.integers(0, 2 ** (32 if dtype == zg.ZERO_FP32 else 16), A, dtype=np.uint64).astype(npt)
    # each model-parallel rank holds the checkpoint as it computed it
    replicas = [torch.from_numpy(x.view(np.int32 if vt == torch.int32 else np.int16)).to("cuda") for _ in range(N)]
    if host_slices:
        shards = [torch.full((max(p.shard_elems, 1),), -1, dtype=vt).pin_memory() for _ in range(N)]
    else:
        shards = [torch.full((max(p.shard_elems, 1),), -1, dtype=vt, device="cuda") for _ in range(N)]
    zg.zero_pa_partition(p, replicas, shards)
    torch.cuda.synchronize()
    ref = oracle.pa_partition([x] * N, N, p.shard_elems)
    for r in range(N):
        own = ref[r].size
        assert np.array_equal(as_bits(shards[r][:own]), ref[r]), "slice of rank %d" % r
        if own < p.shard_elems:
            assert (shards[r][own:] == -1).all().item(), "rank %d wrote past its slice" % r
    del replicas
    dst = [torch.full((max(A, 1) + 8,), -1, dtype=vt, device="cuda") for _ in range(n_dst)]
    zg.zero_pa_gather(p, shards, dst)
    torch.cuda.synchronize()
    full = oracle.pa_gather(ref, A)
    for d in dst:
        assert np.array_equal(as_bits(d[:A]), full)
        assert (d[A:] == -1).all().item(), "the gather wrote past the checkpoint"
    return p


@pytest.mark.parametrize("A,N", [(1, 1), (7, 3), (2048 * 5 + 3, 4), (100_003, 16), (50_000, 64), (3 * 8192 + 1, 2)])
@pytest.mark.parametrize("n_dst", [1, 3, 8, 16])
def test_partition_and_gather_fp16(A, N, n_dst):
    _run(A, N, zg.ZERO_FP16, n_dst, seed=A + N)


@pytest.mark.parametrize("n_dst", [2, 9])
def test_partition_and_gather_fp32_small_align(n_dst):
    _run(33_333, 5, zg.ZERO_FP32, n_dst, align=8)


@pytest.mark.parametrize("n_dst", [1, 16])
def test_slices_in_pinned_host_memory(n_dst):
    """P_a+cpu: the slices live in host memory; the partition writes them and
    the all-gather reads them over the host link."""
    _run(200_003, 16, zg.ZERO_BF16, n_dst, host_slices=True)


def test_empty_checkpoint():
    p = zg.zero_pa_plan(0, 4)
    assert p.shard_elems == 0 and p.mem_per_rank_bytes == 0
    x = [torch.zeros(8, dtype=torch.int16, device="cuda") for _ in range(4)]
    zg.zero_pa_partition(p, x, x)
    zg.zero_pa_gather(p, x, x[:2])
    torch.cuda.synchronize()


def test_full_size_checkpoint():
    """The checkpoint the benchmark uses: batch 32 x sequence 1024 x hidden
    1600 fp16 (105 MB), N_m = 16, all-gathered into 16 buffers."""
    p = _run(32 * 1024 * 1600, 16, zg.ZERO_FP16, 16, seed=1)
    assert p.mem_per_rank_bytes // p.mem_per_rank_pa_bytes == 16
