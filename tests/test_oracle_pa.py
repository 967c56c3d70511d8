"""Pins for the oracle's P_a (partitioned activation checkpoint) functions:
the pages state that the activation memory of a rank drops by the
model-parallel degree N_m and to (nearly) nothing with the CPU variant, and
that the checkpoint is rebuilt by an all-gather -- so the partition followed
by the gather must give back the original bit for bit, the slices must be
disjoint and cover it, and the per-rank memory must be 1/N_m of the
replicated one whenever N_m divides the size on the alignment grid."""
import numpy as np
import pytest

import oracle


@pytest.mark.parametrize("A,N", [(1, 1), (7, 3), (4096, 16), (32 * 1024 * 1600, 16), (100_003, 64), (10, 64)])
def test_partition_then_gather_is_identity(A, N):
    p = oracle.pa_plan(A, N)
    rng = np.random.default_rng(A % 1000 + N)
    x = rng.integers(0, 2 ** 16, min(A, 1 << 20), dtype=np.uint64).astype(np.uint16)
    if x.size < A:   # the large case: only the sizes, not the values
        assert sum(p["own"]) == A
        return
    replicas = [x.copy() for _ in range(N)]
    shards = oracle.pa_partition(replicas, N, p["shard"])
    assert [s.size for s in shards] == p["own"]
    assert np.array_equal(oracle.pa_gather(shards, A), x)


def test_slices_are_disjoint_and_cover():
    for A in (1, 2, 2047, 2048, 2049, 10 ** 6 + 7):
        for N in (1, 2, 3, 16, 64):
            p = oracle.pa_plan(A, N)
            P = p["shard"]
            covered = np.zeros(A, np.int8)
            for r in range(N):
                lo, hi = r * P, min((r + 1) * P, A)
                if hi > lo:
                    covered[lo:hi] += 1
            assert covered.min() == 1 and covered.max() == 1
            assert P % 2048 == 0 and P * N >= A and (P - 2048) * N < A


def test_memory_per_rank_drops_by_the_model_parallel_degree():
    # GPT-2 1.5B layer checkpoint at batch 32, sequence 1024, hidden 1600 (the
    # pages' activation example), fp16, N_m = 16: 1/16 of the replica
    A = 32 * 1024 * 1600
    p = oracle.pa_plan(A, 16, value_bytes=2)
    assert p["mem_per_rank"] == A * 2 == 104_857_600
    assert p["mem_per_rank"] / p["mem_per_rank_pa"] == 16
    assert p["mem_per_rank_pa_cpu"] == 0
    # each rank receives the other 15 slices in one all-gather
    assert p["gather_recv_per_rank"] == [A * 2 * 15 // 16] * 16
    # binary32 activations: 4 bytes per value
    assert oracle.pa_plan(A, 16, value_bytes=4)["mem_per_rank_pa"] == A * 4 // 16


def test_planted_mistakes_are_caught():
    x = np.arange(10_000, dtype=np.uint16)
    p = oracle.pa_plan(x.size, 4, align_elems=8)
    shards = oracle.pa_partition([x] * 4, 4, p["shard"])
    # gathering in the wrong rank order, or dropping a rank, changes the result
    assert not np.array_equal(oracle.pa_gather(shards[::-1], x.size), x)
    assert oracle.pa_gather(shards[:3], x.size).size < x.size
