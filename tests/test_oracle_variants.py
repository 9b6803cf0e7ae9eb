"""Pins for the oracle at the variant shapes: head_dim 64 and 256, rotation
blocks h = 32 and 256 (CPU only).

The oracle's functions take head_dim and h as arguments; these tests pin them
at the other shapes the same ways the head_dim-128 pins do: scipy's Hadamard,
exact one-hot and small-integer butterflies, the s/2 error bound, the cache
layout, and a dense original-domain attention.
"""
import math

import numpy as np
import pytest
import scipy.linalg

import oracle
from test_oracle_attention import _build, _dense_reference
from test_oracle_quantizer import _cache_rows, _rows, bits_to_f32, unpack


@pytest.mark.parametrize("h,D", [(256, 256), (128, 256), (64, 64), (32, 64)])
def test_canon_one_hot_is_exact(h, D):
    c = np.float32(1.0 / math.sqrt(h))
    H = scipy.linalg.hadamard(h).astype(np.float32)
    for j in (0, 1, h // 2, h - 1, D - 1):
        x = np.zeros(D, np.float32)
        x[j] = 1.0
        y = oracle.rotate_canon(x, h)
        b0 = (j // h) * h
        exp = np.zeros(D, np.float32)
        exp[b0:b0 + h] = H[:, j - b0] * c
        np.testing.assert_array_equal(y, exp)


@pytest.mark.parametrize("h,D", [(256, 256), (64, 64)])
def test_canon_on_small_integers_is_exact(h, D):
    rng = np.random.default_rng(h + D)
    x = rng.integers(-100, 101, (6, D)).astype(np.float32)
    y = oracle.rotate_canon(x, h)
    H = scipy.linalg.hadamard(h).astype(np.int64)
    c = np.float32(1.0 / math.sqrt(h))
    for b0 in range(0, D, h):
        ints = x[:, b0:b0 + h].astype(np.int64) @ H.T
        np.testing.assert_array_equal(y[:, b0:b0 + h], ints.astype(np.float32) * c)
    # and R-exact is orthogonal at this size
    e = oracle.rotate_exact(oracle.rotate_exact(x.astype(np.float64)[0], h), h)
    np.testing.assert_allclose(e, x[0], atol=1e-10)


@pytest.mark.parametrize("kind", ["normal", "outlier", "heavy", "huge"])
@pytest.mark.parametrize("rotate,h,D", [(True, 64, 64), (False, 64, 64), (True, 256, 256),
                                        (True, 32, 256)])
def test_error_bound_and_coverage(kind, rotate, h, D):
    rng = np.random.default_rng(D * 7 + h + int(rotate))
    xb = _rows(rng, 48, D, kind)
    codes, s, z = oracle.quantize_rows(xb, rotate, h)
    assert codes.shape == (48, D // 2)
    y = bits_to_f32(xb)
    if rotate:
        y = oracle.rotate_canon(y, h)
    y = y.astype(np.float64)
    sv = oracle.f16_bits_to_f64(s)[:, None]
    zv = oracle.f16_bits_to_f64(z)[:, None]
    assert np.all(zv <= y.min(1, keepdims=True))
    deq = oracle.dequant_rows(codes, s, z)
    slack = 2.0 ** -20 * (np.abs(y) + np.abs(zv) + 15 * sv)
    assert np.all(np.abs(y - deq) <= sv / 2 + slack)
    q = unpack(codes)
    assert q.max() <= 15


@pytest.mark.parametrize("D,P", [(64, 16), (256, 32)])
def test_append_layout(D, P):
    rng = np.random.default_rng(D + P)
    T, Hkv, num_pages = 20, 2, 5
    k = _rows(rng, T * Hkv, D, "outlier").reshape(T, Hkv, D)
    v = _rows(rng, T * Hkv, D, "heavy").reshape(T, Hkv, D)
    slots = rng.permutation(num_pages * P)[:T].astype(np.int32)
    nbytes = oracle.cache_bytes(num_pages, P, Hkv, D)
    assert nbytes == num_pages * Hkv * (P * D // 2 + 4 * P)
    kc = np.full(nbytes, 0xAB, np.uint8)
    vc = np.full(nbytes, 0xAB, np.uint8)
    h = min(D, 256)
    assert oracle.quantize_append(k, v, slots, Hkv, D, kc, vc, num_pages, P, True, True, h) == 0
    for hd in range(Hkv):
        c, s, z = _cache_rows(kc, slots, hd, Hkv, P, D)
        c2, s2, z2 = oracle.quantize_rows(k[:, hd], True, h)
        np.testing.assert_array_equal(c, c2)
        np.testing.assert_array_equal(s, s2)
        np.testing.assert_array_equal(z, z2)


@pytest.mark.parametrize("D,h,rk,rv", [(64, 64, True, True), (64, 32, True, False),
                                       (256, 256, True, True), (256, 128, True, False),
                                       (256, 256, False, False)])
def test_attention_equals_dense_original_domain(D, h, rk, rv):
    rng = np.random.default_rng(D + h + int(rv))
    seq_lens = [1, 21, 40]
    Hq, Hkv, P = 4, 2, 16
    d = _build(rng, seq_lens, Hq, Hkv, D, P, rk, rv, h)
    got = oracle.decode(d["q"], d["kc"], d["vc"], d["bt"], seq_lens, Hq, Hkv, D, d["num_pages"],
                        P, rk, rv, h).reshape(len(seq_lens), Hq, D)
    ref = _dense_reference(d, seq_lens, Hq, Hkv, D, P, rk, rv, h, 1 / math.sqrt(D))
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=1e-12)
