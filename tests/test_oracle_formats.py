"""Pins for the oracle's binary16 conversions (CPU only).

The quantizer stores its scale and zero-point as binary16 with directed
rounding (zero toward -inf, scale toward +inf): a reading taken where the
pages (youngju.dev "Why Naive INT4 Breaks"; gist.science s.2) only say
"one scale per token".  These tests pin the hand-written converter against
numpy's own binary16 type and against the IEEE definition of directed
rounding (bracketing and adjacency), not against the converter itself.
"""
import numpy as np
import pytest

import oracle

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _random_f32(rng, n):
    # log-uniform magnitudes across the binary16 subnormal and normal range,
    # plus exact binary16 values and their neighbours
    mag = np.exp2(rng.uniform(-26, 16, n)).astype(np.float32)
    sign = np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    x = mag * sign
    exact = rng.integers(0, 0x7BFF, 64).astype(np.uint16).view(np.float16).astype(np.float32)
    nb = np.nextafter(exact, np.float32(np.inf))
    return np.concatenate([x, exact, -exact, nb, -nb]).astype(np.float32)


def test_f16_to_f64_all_patterns():
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = oracle.f16_bits_to_f64(bits)
    finite = np.isfinite(ref)
    np.testing.assert_array_equal(got[finite], ref[finite])
    assert np.all(np.isinf(got[np.isinf(ref)]))
    assert np.all(np.isnan(got[np.isnan(ref)]))


def test_nearest_even_matches_numpy():
    rng = np.random.default_rng(1)
    x = _random_f32(rng, 4000)
    x = x[np.abs(x) <= 65504]
    got = oracle.f32_to_f16_bits(x, oracle.RN)
    ref = x.astype(np.float16)
    ref_bits = ref.view(np.uint16).copy()
    ref_bits[ref == 0] = 0  # the oracle writes every zero as +0
    np.testing.assert_array_equal(got, ref_bits)


@pytest.mark.parametrize("mode", [oracle.RD, oracle.RU])
def test_directed_rounding_brackets(mode):
    rng = np.random.default_rng(2 + mode)
    x = _random_f32(rng, 4000)
    x = x[np.abs(x) <= 65504]
    got = oracle.f32_to_f16_bits(x, mode).view(np.float16).astype(np.float64)
    xd = x.astype(np.float64)
    rn = x.astype(np.float16).astype(np.float64)
    if mode == oracle.RD:
        assert np.all(got <= xd)
        # no binary16 value strictly between the result and x
        nxt = np.nextafter(got.astype(np.float16), np.float16(np.inf)).astype(np.float64)
        assert np.all((got == xd) | (nxt > xd))
    else:
        assert np.all(got >= xd)
        prv = np.nextafter(got.astype(np.float16), np.float16(-np.inf)).astype(np.float64)
        assert np.all((got == xd) | (prv < xd))
    # the nearest value is one of the two directed ones
    lo = oracle.f32_to_f16_bits(x, oracle.RD).view(np.float16).astype(np.float64)
    hi = oracle.f32_to_f16_bits(x, oracle.RU).view(np.float16).astype(np.float64)
    assert np.all((rn == lo) | (rn == hi))
    exact = lo == hi
    np.testing.assert_array_equal(lo[exact], xd[exact])


def test_saturation_and_zero_sign():
    B = lambda v, m: int(oracle.f32_to_f16_bits(np.float32(v), m))
    for m in (oracle.RN, oracle.RD, oracle.RU):
        assert B(1e6, m) == 0x7BFF
        assert B(-1e6, m) == 0xFBFF
        assert B(np.inf, m) == 0x7BFF
        assert B(-0.0, m) == 0x0000
        assert B(0.0, m) == 0x0000
    assert B(65519.0, oracle.RN) == 0x7BFF
    assert B(65505.0, oracle.RD) == 0x7BFF
    # smallest subnormal is 2^-24
    assert B(1e-10, oracle.RU) == 0x0001
    assert B(1e-10, oracle.RD) == 0x0000
    assert B(-1e-10, oracle.RD) == 0x8001
    assert B(-1e-10, oracle.RU) == 0x0000  # -0 written as +0
    assert B(np.nan, oracle.RN) == 0x7E00
