"""The stage-3 fetch schedule on the CPU (zero_fetch_schedule: the decisions
the GPU fetcher takes), replayed and checked by brute force: every layer is
gathered before its use and at most `depth` positions ahead, the resident
layers' pool ranges never overlap and never exceed the capacity, and with
room to spare the schedule prefetches the full depth."""
import random

import pytest

import zero_sharded_mixed_bucket_gb300 as zg


def r8(x):
    return (x + 7) // 8 * 8


def replay(sizes, order, cap, depth):
    issue, offs, max_live = zg.zero_fetch_schedule(sizes, order, cap, depth)
    n = len(order)
    seen_live = 0
    for p in range(n):
        resident = [q for q in range(n) if issue[q] <= p <= q]   # issued, not yet used/released
        assert p in resident
        spans = sorted((offs[q], offs[q] + r8(sizes[order[q]])) for q in resident)
        for a, b in spans:
            assert 0 <= a and b <= cap and a % 8 == 0
        for (a0, b0), (a1, b1) in zip(spans, spans[1:]):
            assert b0 <= a1, "resident layers overlap"
        live = sum(b - a for a, b in spans)
        assert live <= cap
        seen_live = max(seen_live, live)
    for q in range(n):
        assert max(0, q - depth) <= issue[q] <= q
        assert issue[q] == 0 or issue[q] >= q - depth
    assert max_live == seen_live
    return issue, offs


@pytest.mark.parametrize("seed", range(30))
def test_schedule_invariants_random(seed):
    rng = random.Random(seed)
    L = rng.randint(1, 40)
    sizes = [rng.choice([rng.randint(1, 50), rng.randint(100, 5000)]) for _ in range(L)]
    order = list(range(L)) if seed % 2 else list(reversed(range(L)))
    biggest = max(r8(s) for s in sizes)
    cap = biggest + rng.randint(0, 3 * biggest)
    depth = rng.randint(0, 6)
    replay(sizes, order, cap, depth)


def test_full_prefetch_when_everything_fits():
    sizes = [300, 5, 1000, 64, 7]
    order = [0, 1, 2, 3, 4, 4, 3, 2, 1, 0]          # forward then backward
    cap = 2 * sum(r8(s) for s in sizes)
    for depth in range(0, 5):
        issue, _ = replay(sizes, order, cap, depth)
        assert issue == [max(0, q - depth) for q in range(len(order))]


def test_depth_zero_gathers_on_demand():
    sizes = [16, 16, 16]
    issue, offs = replay(sizes, [0, 1, 2], 16, 0)
    assert issue == [0, 1, 2] and offs == [0, 0, 0]


def test_budget_of_one_largest_layer_serialises():
    sizes = [100, 200, 150]
    issue, _ = replay(sizes, [0, 1, 2], 200, 4)
    assert issue == [0, 1, 2]


def test_capacity_below_largest_layer_refused():
    with pytest.raises(zg.ZeroError) as e:
        zg.zero_fetch_schedule([100, 300], [0, 1], 200, 1)
    assert e.value.status == zg.ZERO_EINVAL
