"""Pins for the oracle's partition, memory and communication accounting.

Everything here is checked against values the pages print (tests/golden/,
each file headed by its citation), closed forms stated on the pages, or brute
force over tiny partitions.  CPU only.
"""
from fractions import Fraction

import pytest

import oracle
from tests.conftest import read_golden

GB = Fraction(10 ** 9)
SIZES = {"7.5B": Fraction(75, 10) * 10 ** 9, "128B": Fraction(128 * 10 ** 9), "1T": Fraction(10 ** 12)}


def _psi(tok):
    return Fraction(tok.replace("e9", "")) * 10 ** 9 if tok.endswith("e9") else Fraction(tok)


# --- Table 1: all 54 cells ---------------------------------------------------
def test_table1_every_cell():
    rows = read_golden("table1_model_state_gb.txt")
    assert len(rows) == 6
    checked = 0
    for row in rows:
        n = int(row[0])
        cells = row[1:]
        for si, size in enumerate(["7.5B", "128B", "1T"]):
            for stage in (1, 2, 3):
                printed = cells[3 * si + stage - 1]
                total = oracle.model_state_bytes(SIZES[size], n, stage)["total"] / GB
                assert oracle.display_gb(total) == printed, (n, size, stage, float(total))
                checked += 1
    assert checked == 54


# --- Worked examples A, B, C (exact totals) ---------------------------------
def test_worked_example_totals_exact():
    for name, psi, n, b, K, stage, total in read_golden("worked_examples.txt"):
        got = oracle.model_state_bytes(_psi(psi), int(n), int(stage), b=int(b), K=int(K))["total"] / GB
        assert got == Fraction(total), (name, stage, got)


def test_worked_example_component_tables():
    for name, stage, params, grads, optim, total, comm, comm_s1 in read_golden("worked_example_tables.txt"):
        psi = SIZES["7.5B"] if name == "A" else SIZES["128B"]
        stage = int(stage)
        mem = oracle.model_state_bytes(psi, 64, stage)
        assert oracle.display_gb(mem["params"] / GB) == params
        assert oracle.display_gb(mem["grads"] / GB) == grads
        assert oracle.display_gb(mem["optim"] / GB) == optim
        assert oracle.display_gb(mem["total"] / GB) == total
        c = oracle.comm_bytes(int(psi), 64, stage)
        assert oracle.display_gb(c["paper"] / GB) == comm
        if comm_s1 != "-":
            # stage 1 with its end-of-step all-gather counted: 3 passes of psi
            assert c["counted_passes"] == 3
            assert oracle.display_gb(c["counted_passes"] * psi * 2 / GB) == comm_s1


def test_compression_ratios_of_examples_c():
    # C1: 90 / 1.40625 = 64x; C2: 12 / 1.5 = 8x (ZeRO visual reading, example C)
    c1 = [oracle.model_state_bytes(Fraction(75, 10) * 10 ** 9, 64, s, b=4, K=4)["total"] for s in (0, 3)]
    c2 = [oracle.model_state_bytes(Fraction(15, 10) * 10 ** 9, 8, s, b=4, K=0)["total"] for s in (0, 3)]
    assert c1[0] / c1[1] == 64
    assert c2[0] / c2[1] == 8


# --- Statements of the pages -------------------------------------------------
def test_sixteen_bytes_per_parameter():
    # 16 Psi: GPT-2 1.5B needs 24 GB, its fp16 weights alone 3 GB; 1T needs 16 TB
    # ("AI论文陪读·ZeRO" section 01)
    m = oracle.model_state_bytes(Fraction(15, 10) * 10 ** 9, 1, 0)
    assert m["total"] / GB == 24
    assert m["params"] / GB == 3
    assert oracle.model_state_bytes(10 ** 12, 1, 0)["total"] == 16 * 10 ** 12
    # 1T over 1024 GPUs at stage 3: 15.625 GB each (printed as about 16 GB)
    assert oracle.model_state_bytes(10 ** 12, 1024, 3)["total"] / GB == Fraction(15625, 1000)


def test_reduction_limits_and_floors():
    # P_os -> 4x, P_os+g -> 8x as N_d grows; stage 3 scales as N_d
    # ("ZeRO：大模型训练的内存优化革命" 3.1.1-3.1.3); floors 4 Psi and 2 Psi
    psi = 10 ** 9
    base = oracle.model_state_bytes(psi, 1, 0)["total"]
    big = 10 ** 12
    r1 = base / oracle.model_state_bytes(psi, big, 1)["total"]
    r2 = base / oracle.model_state_bytes(psi, big, 2)["total"]
    assert abs(r1 - 4) < Fraction(1, 10 ** 9) and r1 < 4
    assert abs(r2 - 8) < Fraction(1, 10 ** 9) and r2 < 8
    for n in (1, 2, 64, 1024):
        assert oracle.model_state_bytes(psi, n, 3)["total"] * n == base
        assert oracle.model_state_bytes(psi, n, 1)["total"] >= 4 * psi
        assert oracle.model_state_bytes(psi, n, 2)["total"] >= 2 * psi


# --- Communication -----------------------------------------------------------
@pytest.mark.parametrize("psi,gb02,gb3", [(Fraction(75, 10) * 10 ** 9, 30, 45), (128 * 10 ** 9, 512, 768)])
def test_comm_volume_printed(psi, gb02, gb3):
    # 30/45 GB at 7.5B and 512/768 GB at 128B (ZeRO visual reading, examples A, B)
    for stage in (0, 1, 2):
        assert oracle.comm_bytes(int(psi), 64, stage)["paper"] / GB == gb02
    assert oracle.comm_bytes(int(psi), 64, 3)["paper"] / GB == gb3


def test_comm_ratio_and_counted_limit():
    # stage 3 moves 1.5x the baseline ("ZeRO：大模型训练的内存优化革命" 1.2 table);
    # the counted bytes of a ring over N ranks approach the paper's volume per rank
    psi, n = 10 ** 9, 10 ** 6
    assert oracle.comm_bytes(psi, 8, 3)["paper"] / oracle.comm_bytes(psi, 8, 0)["paper"] == Fraction(3, 2)
    for stage in range(4):
        c = oracle.comm_bytes(psi, n, stage)
        per_rank = Fraction(c["counted"], n)
        limit = c["counted_passes"] * psi * 2
        assert per_rank < limit and limit - per_rank == Fraction(limit, n)
    assert oracle.comm_bytes(psi, 1, 2)["counted"] == 0


# --- Table 2 (theoretical columns) -----------------------------------------
def _tok_to_b(tok):
    if tok.endswith("T"):
        return Fraction(tok[:-1]) * 1000
    return Fraction(tok[:-1])


def _one_decimal(x):
    # Table 2 prints sizes in billions with one decimal, no trailing zero
    q = Fraction(int(x * 10 + Fraction(1, 2)), 10)
    return f"{float(q):.1f}".rstrip("0").rstrip(".")


def test_table2_first_row_exact_and_scaling():
    rows = read_golden("table2_max_model_size.txt")
    mp1 = rows[0]
    assert mp1[0] == "1" and mp1[1] == "64"
    for col, stage in zip(mp1[2:], (0, 1, 2, 3)):
        size_b = oracle.max_model_size(32 * GB, 64, stage) / GB
        assert _one_decimal(size_b) == col[:-1], (stage, float(size_b))
    # every other row is MP times the first row (GPUs = MP * 64)
    for row in rows[1:]:
        mp = int(row[0])
        assert int(row[1]) == 64 * mp
        for col, base in zip(row[2:], mp1[2:]):
            scaled = mp * _tok_to_b(base)
            printed = _tok_to_b(col)
            if col.endswith("T"):
                assert abs(printed - scaled) / scaled < Fraction(25, 1000)
            else:
                assert printed == scaled


# --- Partition: brute force on tiny sizes ------------------------------------
@pytest.mark.parametrize("n_ranks", [1, 2, 3, 4, 7])
@pytest.mark.parametrize("psi", [0, 1, 7, 8, 9, 63, 64, 65, 200])
@pytest.mark.parametrize("bucket,align", [(8, 8), (16, 8), (24, 16), (64, 8), (8, 32)])
def test_partition_brute_force(n_ranks, psi, bucket, align):
    p = oracle.plan(psi, n_ranks, bucket, align)
    P = p["shard"]
    assert P % align == 0 and P * n_ranks >= psi
    # smallest aligned shard that covers psi
    assert P == 0 or (P - align) * n_ranks < psi
    seen = {}
    for b in range(p["n_buckets"]):
        lo, hi = p["buckets"][b]
        assert lo == b * bucket and hi - lo <= bucket and hi > lo
        total = 0
        for rank, off, ln in oracle.bucket_segments(p, b):
            for j in range(ln):
                i = rank * P + off + j
                assert lo <= i < hi
                assert i not in seen
                seen[i] = rank
                assert oracle.owner(p, i) == rank
            total += ln
        assert total == hi - lo
    assert sorted(seen) == list(range(psi))
    # segments come in rank order and are contiguous
    for b in range(p["n_buckets"]):
        segs = oracle.bucket_segments(p, b)
        flat = [r * P + off for r, off, _ in segs]
        assert flat == sorted(flat)


def test_layer_table():
    p = oracle.plan(100, 3, 16, 8, layer_sizes=[10, 50, 40])
    assert p["layer_starts"] == [0, 10, 60] and p["max_layer"] == 50
    with pytest.raises(ValueError):
        oracle.plan(100, 3, 16, 8, layer_sizes=[10, 50])


def test_display_rule_examples():
    # the page's own examples: 31.0 shows as 31, 1.50 as 1.5
    assert oracle.display_gb(Fraction(31)) == "31"
    assert oracle.display_gb(Fraction(15, 10)) == "1.5"
    assert oracle.display_gb(Fraction(41125, 1000)) == "41.1"
    assert oracle.display_gb(Fraction(4187.5)) == "4187"


def test_hbm_bytes_per_param_count():
    # bytes per parameter from counting each array access once: 16-bit = 2,
    # fp32 state = 3 arrays x 4 bytes, read and written
    N = 8
    # stage 2 fused: read N grads, read w,m,v, write w,m,v, write N params
    assert oracle.hbm_bytes_per_param(N, 2, "fused") == 2 * N + 12 + 12 + 2 * N
    # stage 2 two-pass adds the reduced gradient written then read
    assert oracle.hbm_bytes_per_param(N, 2, "two_pass") == oracle.hbm_bytes_per_param(N, 2, "fused") + 4
    # stage 0: all-reduce write-back to N grad buffers, N replicas updated
    assert oracle.hbm_bytes_per_param(N, 0, "fused") == 2 * N + 2 * N + N * (24 + 2)


def test_mixed_precision_optimizer_multipliers():
    # the page's calculator: K = optimizer multiplier + 4 B fp32 master in mixed
    # precision (Adam 8 + 4 = 12, SGD+m 4 + 4 = 8, SGD 0 + 4 = 4); stage 0 = (2b+K) Psi
    import oracle as o
    assert o.OPTIM_K == {"adam": 12, "sgdm": 8, "sgd": 4}
    for name, K in o.OPTIM_K.items():
        assert o.model_state_bytes(10 ** 9, 1, 0, b=2, K=K)["total"] == (4 + K) * 10 ** 9
    # byte counts per parameter reduce to the Adam table for 12-byte state
    for stage in range(4):
        for N in (1, 8, 64):
            assert oracle.hbm_bytes_per_param(N, stage, "fused", 12) == {0: 30 * N, 1: 24 + 6 * N, 2: 24 + 4 * N,
                                                                        3: 26 + 2 * N}[stage]
            assert oracle.hbm_bytes_per_param(N, stage, "two_pass", 12) == {0: 32 * N, 1: 26 + 6 * N,
                                                                           2: 28 + 4 * N, 3: 30 + 2 * N}[stage]
