"""The seeded input generator on the CPU: its Philox4x32-10 against a plain
Python restatement of the published round function, and its normal draws'
moments.  (The device generator is checked against this one on the GPU.)"""
import numpy as np

import synth

M0, M1 = 0xD2511F53, 0xCD9E8D57
W0, W1 = 0x9E3779B9, 0xBB67AE85
MASK = 0xFFFFFFFF


def philox_py(ctr, key, rounds=10):
    c = list(ctr)
    k0, k1 = key
    for r in range(rounds):
        if r:
            k0, k1 = (k0 + W0) & MASK, (k1 + W1) & MASK
        p0, p1 = M0 * c[0], M1 * c[2]
        c = [((p1 >> 32) ^ c[1] ^ k0) & MASK, p1 & MASK, ((p0 >> 32) ^ c[3] ^ k1) & MASK, p0 & MASK]
    return c


def test_philox_against_python():
    rng = np.random.default_rng(0)
    for _ in range(200):
        ctr = [int(x) for x in rng.integers(0, 2 ** 32, 4)]
        key = [int(x) for x in rng.integers(0, 2 ** 32, 2)]
        assert synth.philox(ctr, key) == philox_py(ctr, key)
    assert synth.philox([0, 0, 0, 0], [0, 0]) == philox_py([0, 0, 0, 0], [0, 0])


def test_normal_moments_and_gather_form():
    x = synth.host_normal32(1 << 20, 0.02, seed=1, stream=synth.STREAM_WEIGHT)
    assert abs(x.mean()) < 1e-4 and abs(x.std() - 0.02) < 2e-4
    idx = np.array([0, 1, 2, 12345, (1 << 20) - 1])
    assert np.array_equal(synth.host_normal32_at(idx, 0.02, seed=1, stream=synth.STREAM_WEIGHT), x[idx])
    h = synth.host_normal16(1000, synth.FP16, 1e-3, seed=2, stream=1, step=3, rank=4, offset=77)
    h2 = synth.host_normal16_at(np.arange(77, 1077), synth.FP16, 1e-3, seed=2, stream=1, step=3, rank=4)
    assert np.array_equal(h, h2)
    # ranks and steps draw different numbers
    a = synth.host_normal16(100, synth.FP16, 1e-3, seed=2, stream=1, step=3, rank=5)
    b = synth.host_normal16(100, synth.FP16, 1e-3, seed=2, stream=1, step=4, rank=4)
    assert not np.array_equal(a, h[:100]) and not np.array_equal(b, h[:100])


def test_inf_positions_one_per_period():
    pos = synth.inf_positions(1_555_278_400, 8, seed=0, step=1)
    assert len(pos) in (12, 13)          # 8 * 1.555e9 / 1e9 positions
    flat = [r * 1_555_278_400 + e for r, e in pos]
    assert all(b - a == 10 ** 9 for a, b in zip(flat, flat[1:]))
    assert synth.inf_positions(1_555_278_400, 8, seed=0, step=2) != pos
