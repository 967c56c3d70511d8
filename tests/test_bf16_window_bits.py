"""The bfloat16 sum-of-squares fast path tests two values per 32-bit word
with carry-free 16-bit additions and forms each value's X = M << (e - fbase)
with a shift whose counts of 32 or more give 0.  Here that arithmetic,
modelled in numpy, is compared with the value-by-value definition (e, f,
hidden bit, the window [fbase, fbase + 22], a zero adding nothing) for every
16-bit pattern and window positions from the lowest to the highest."""
import numpy as np
import pytest


def _per_value(v, fbase):
    e = (v >> 7) & 0xFF
    f = v & 0x7F
    hid = np.minimum(e, 1)
    M = f + hid * 0x80
    d = (e + 1 - hid - fbase) & 0xFFFFFFFF
    outside = (d > 22) & (M != 0)
    X = (M << (d & 31)) & 0xFFFFFFFF
    return outside, np.where(outside, 0, X)


def _packed(v, fbase):
    mag = v & 0x7FFF
    k_hi = 0x8000 - ((fbase + 23) << 7)
    k_lo = 0x8000 - (fbase << 7)
    assert 0 < k_hi < 0x8000 and 0 < k_lo < 0x8000
    s_hi, s_lo, s_nz = mag + k_hi, mag + k_lo, mag + 0x7FFF
    assert (s_hi < 0x10000).all() and (s_lo < 0x10000).all() and (s_nz < 0x10000).all()   # no carry into the other half
    outside = (((s_hi | (s_nz & ~s_lo)) >> 15) & 1) == 1
    M = (v & 0x7F) | 0x80
    count = (((v >> 7) & 0xFF) - fbase) & 0xFFFFFFFF
    X = np.where(count >= 32, 0, (M << np.minimum(count, 31)) & 0xFFFFFFFF)
    return outside, np.where(outside, 0, X)


@pytest.mark.parametrize("fbase", [10, 11, 64, 105, 127, 200, 230, 231])
def test_packed_window_equals_value_by_value(fbase):
    v = np.arange(1 << 16, dtype=np.int64)
    out_ref, x_ref = _per_value(v, fbase)
    out_new, x_new = _packed(v, fbase)
    assert np.array_equal(out_ref, out_new)
    assert np.array_equal(x_ref, x_new)
    # inside the window X < 2^30, so eight squares add up in 64 bits
    assert (x_ref < (1 << 30)).all()
