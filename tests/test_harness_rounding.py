"""The rounding helpers the GPU parity tests use to compare kernel outputs
with the oracle rounded once to the output dtype: correct rounding (nearest,
ties to even, no double rounding through binary32), value-ordered ulp
distance and spacing."""
import numpy as np

import workloads as W
from harness import _ordered, bits_to_f64, round_bits, ulp_spacing


def _neighbours(b, dt):
    b = b.astype(np.int64)
    up = bits_to_f64(((b & 0x8000) | ((b & 0x7FFF) + 1)).astype(np.uint16), dt)
    dn = bits_to_f64(((b & 0x8000) | np.maximum((b & 0x7FFF) - 1, 0)).astype(np.uint16), dt)
    return up, dn


def test_round_bits_is_nearest():
    rng = np.random.default_rng(0)
    x = rng.standard_normal(200000) * np.exp(rng.uniform(-30, 12, 200000))
    for dt, lim in ((W.BF16, 3e38), (W.F16, 65000.0)):
        xx = x[np.abs(x) < lim]
        b = round_bits(xx, dt)
        v = bits_to_f64(b, dt)
        up, dn = _neighbours(b, dt)
        e = np.abs(v - xx)
        assert np.all(e <= np.abs(up - xx)) and np.all(e <= np.abs(dn - xx))
        assert np.all(np.sign(v) * np.sign(xx) >= 0)


def test_round_bits_ties_to_even_and_no_double_rounding():
    rng = np.random.default_rng(1)
    for dt, top in ((W.BF16, 0x7F00), (W.F16, 0x7BFF)):
        b = rng.integers(1, top, 5000).astype(np.int64)
        lo = bits_to_f64(b.astype(np.uint16), dt)
        hi = bits_to_f64((b + 1).astype(np.uint16), dt)
        mid = (lo + hi) / 2
        assert np.array_equal(round_bits(mid, dt), np.where(b % 2 == 0, b, b + 1).astype(np.uint16))
        # just past the midpoint either way: a rounding through binary32 first
        # would land on the midpoint and then on the even neighbour
        assert np.array_equal(round_bits(np.nextafter(mid, np.inf), dt), (b + 1).astype(np.uint16))
        assert np.array_equal(round_bits(np.nextafter(mid, -np.inf), dt), b.astype(np.uint16))


def test_ordered_distance_and_spacing():
    # +0 and -0 coincide; crossing zero counts the patterns in between
    assert _ordered(np.array([0x0000, 0x8000, 0x0001, 0x8001]), ).tolist() == [0, 0, 1, -1]
    one_bf16, one_f16 = np.array([0x3F80], np.uint16), np.array([0x3C00], np.uint16)
    assert ulp_spacing(one_bf16, W.BF16)[0] == 2.0 ** -7
    assert ulp_spacing(one_f16, W.F16)[0] == 2.0 ** -10
    assert ulp_spacing(np.array([0xBF80], np.uint16), W.BF16)[0] == 2.0 ** -7
