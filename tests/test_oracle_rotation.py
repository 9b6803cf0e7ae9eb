"""Pins for the oracle's block-diagonal Hadamard rotation (CPU only).

What the pages fix (youngju.dev "The Rotation Trick -- Block-Diagonal
Hadamard"; gist.science s.2 "Rotazione Block-Diagonale"): the rotation is an
orthogonal Hadamard transform, lossless and undoable, applied within
independent blocks of size h, and it spreads one outlier channel evenly over
all the others.  These tests check the oracle against scipy's Sylvester
Hadamard, the closed form (-1)^popcount(i & j), a hand-written H_4, and the
properties above -- never against a retyped copy of the oracle.
"""
import math

import numpy as np
import pytest
import scipy.linalg

import oracle
from conftest import read_golden

POW2 = [1, 2, 4, 8, 16, 32, 64, 128, 256]


@pytest.mark.parametrize("h", POW2)
def test_sylvester_matches_scipy_and_closed_form(h):
    H = oracle.sylvester(h).astype(np.int64)
    np.testing.assert_array_equal(H, scipy.linalg.hadamard(h))
    i = np.arange(h)[:, None]
    j = np.arange(h)[None, :]
    popc = np.vectorize(lambda v: bin(int(v)).count("1"))(i & j)
    np.testing.assert_array_equal(H, (-1) ** popc)
    np.testing.assert_array_equal(H @ H.T, h * np.eye(h, dtype=np.int64))
    np.testing.assert_array_equal(H, H.T)


def test_sylvester_h4_golden():
    _, rows = read_golden("sylvester_h4.txt")
    ref = np.array([[int(v) for v in r] for r in rows])
    np.testing.assert_array_equal(oracle.sylvester(4), ref)


def test_block_scale_constant():
    assert oracle.block_scale_f32(128).view(np.uint32) == 0x3DB504F3
    assert oracle.block_scale_f32(64) == np.float32(0.125)
    for h in POW2:
        assert oracle.block_scale_f32(h) == np.float32(1.0 / math.sqrt(h))


@pytest.mark.parametrize("h,D", [(128, 128), (64, 128), (16, 64), (2, 8)])
def test_exact_is_orthogonal_and_self_inverse(h, D):
    rng = np.random.default_rng(h + D)
    x = rng.standard_normal((5, D))
    y = oracle.rotate_exact(x, h)
    np.testing.assert_allclose(np.linalg.norm(y, axis=1), np.linalg.norm(x, axis=1), rtol=1e-13)
    # (1/sqrt h) H is symmetric orthogonal: applying it twice gives x back
    np.testing.assert_allclose(oracle.rotate_exact(y, h), x, atol=1e-12)
    # block-diagonal: each block only sees its own inputs
    x2 = x.copy()
    x2[:, :h] += 3.0
    y2 = oracle.rotate_exact(x2, h)
    np.testing.assert_allclose(y2[:, h:], y[:, h:], atol=1e-13)


@pytest.mark.parametrize("h,D", [(128, 128), (64, 128)])
def test_one_hot_spreads_evenly(h, D):
    a = 20.0
    for j in (0, 5, h - 1, D - 1):
        x = np.zeros(D)
        x[j] = a
        y = oracle.rotate_exact(x, h)
        b0 = (j // h) * h
        blk = y[b0:b0 + h]
        np.testing.assert_allclose(np.abs(blk), a / math.sqrt(h), rtol=1e-14)
        # the signs are column j of H
        H = scipy.linalg.hadamard(h)
        np.testing.assert_array_equal(np.sign(blk), H[:, j - b0])
        rest = np.delete(y, np.arange(b0, b0 + h))
        assert np.all(rest == 0.0)


def test_constant_block_collapses():
    h = 128
    a = 0.75
    y = oracle.rotate_exact(np.full(h, a), h)
    assert y[0] == pytest.approx(a * math.sqrt(h), rel=1e-14)
    assert np.max(np.abs(y[1:])) < 1e-13


@pytest.mark.parametrize("h", [2, 4, 8, 16, 32, 64, 128])
def test_canon_one_hot_is_exact(h):
    """The binary32 butterfly of e_j adds only +-1 and 0, so it must equal
    c * H[:, j] bit for bit: this pins its index order and signs."""
    D = 128
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


@pytest.mark.parametrize("h", [8, 64, 128])
def test_canon_on_small_integers_is_exact(h):
    """Small-integer inputs keep every butterfly sum exact, so the butterfly
    must equal the integer matrix product, then one binary32 multiply by c."""
    D = 128
    rng = np.random.default_rng(h)
    x = rng.integers(-100, 101, (6, D)).astype(np.float32)
    y = oracle.rotate_canon(x, h)
    H = scipy.linalg.hadamard(h).astype(np.int64)
    u = np.concatenate([x[:, b:b + h].astype(np.int64) @ H.T for b in range(0, D, h)], axis=1)
    exp = u.astype(np.float32) * np.float32(1.0 / math.sqrt(h))
    np.testing.assert_array_equal(y, exp)


def _inputs(rng, D):
    base = rng.standard_normal((8, D)).astype(np.float32)
    heavy = (rng.standard_t(3, (8, D)) * 2).astype(np.float32)
    out = base.copy()
    out[:, rng.choice(D, 4, replace=False)] *= 20
    return np.concatenate([base, heavy, out, base + 7.0])


@pytest.mark.parametrize("h,D", [(128, 128), (64, 128), (32, 256), (4, 16)])
def test_canon_within_bound_of_exact(h, D):
    """|R_canon - R_exact| <= log2(h) * 2^-23 * ||x_block||_1 * c per element
    (one rounding per butterfly stage, each bounded by the block's l1 norm)."""
    rng = np.random.default_rng(7 * h + D)
    x = _inputs(rng, D)
    yc = oracle.rotate_canon(x, h).astype(np.float64)
    ye = oracle.rotate_exact(x.astype(np.float64), h)
    n = int(math.log2(h))
    c = 1.0 / math.sqrt(h)
    l1 = np.repeat(np.abs(x.astype(np.float64)).reshape(x.shape[0], D // h, h).sum(-1), h, axis=1)
    bound = max(n, 2) * 2.0 ** -23 * l1 * c
    assert np.all(np.abs(yc - ye) <= bound)


@pytest.mark.parametrize("h", [64, 128])
def test_canon_twice_returns_input(h):
    D = 128
    rng = np.random.default_rng(h)
    x = _inputs(rng, D)
    y = oracle.rotate_canon(x, h)
    x2 = oracle.rotate_canon(y, h).astype(np.float64)
    n = int(math.log2(h))
    c = 1.0 / math.sqrt(h)
    l1x = np.repeat(np.abs(x.astype(np.float64)).reshape(-1, D // h, h).sum(-1), h, axis=1)
    l1y = np.repeat(np.abs(y.astype(np.float64)).reshape(-1, D // h, h).sum(-1), h, axis=1)
    e1 = n * 2.0 ** -23 * l1x * c
    bound = n * 2.0 ** -23 * l1y * c + math.sqrt(h) * np.max(e1, axis=1, keepdims=True)
    assert np.all(np.abs(x2 - x) <= bound)
