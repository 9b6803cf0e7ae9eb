"""Pins for the oracle's two format variants (CPU only).

* binary16 K/V/q input.  The fused-kernel diagram of youngju.dev ("The System
  Is the Design -- A Fused Kernel") feeds the kernel "K,V (fp16)".  Both
  bfloat16 and binary16 widen exactly to binary32, so after widening the
  quantizer is the same function: the pins check the widening (values that
  exist in both formats give identical bytes; binary16-only values give the
  closed-form codes).
* bfloat16 (scale, zero) metadata.  The pages fix one scale per token but
  not its storage format; the variant keeps the binary16 reading's rules (zero
  rounded down, scale rounded up, a zero stored as +0) in bfloat16 and
  saturates at the largest finite bfloat16.  The converter is pinned against
  brute force over every finite bfloat16 value, the quantizer against the
  directed-rounding error bound and closed forms, and attention against a
  dense scipy softmax over the dequantized rows.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import scipy.special

import oracle
from test_oracle_quantizer import _rows, bf16_bits, bits_to_f32, to_bf16, unpack

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")

BF16_MAX = float(np.float32(2.0 ** 128 - 2.0 ** 120))


def _bf16_values():
    """(sorted finite bfloat16 values as float64, their bit patterns)."""
    bits = np.arange(0, 1 << 16, dtype=np.uint32)
    vals = (bits << 16).view(np.float32).astype(np.float64)
    ok = np.isfinite(vals)
    vals, bits = vals[ok], bits[ok]
    # one entry per value: +0 (not -0)
    keep = ~((vals == 0) & (bits != 0))
    vals, bits = vals[keep], bits[keep]
    order = np.argsort(vals, kind="stable")
    return vals[order], bits[order].astype(np.uint16)


def _brute_bf16(x, mode):
    """bfloat16 rounding of float32 x by search over every finite value."""
    vals, bits = _bf16_values()
    out = np.empty(len(x), np.uint16)
    for i, v in enumerate(np.asarray(x, np.float64)):
        v = min(max(v, -BF16_MAX), BF16_MAX)
        j = np.searchsorted(vals, v)  # vals[j-1] < v <= vals[j]
        if j < len(vals) and vals[j] == v:
            out[i] = bits[j]
            continue
        lo, hi = j - 1, j
        if mode == oracle.RD:
            k = lo
        elif mode == oracle.RU:
            k = hi
        else:
            dl, dh = v - vals[lo], vals[hi] - v
            k = lo if dl < dh else hi if dh < dl else (lo if (bits[lo] & 1) == 0 else hi)
        out[i] = bits[k]
    return out


def _bf16_scale(step):
    """The bfloat16 metadata scale: round up, and at least 2^-126 if nonzero."""
    sb = _brute_bf16(step, oracle.RU)
    return np.where((np.asarray(step) > 0) & (sb < 0x0080), 0x0080, sb).astype(np.uint16)


def _random_f32(rng, n):
    mag = np.exp2(rng.uniform(-140, 127.9, n)).astype(np.float32)
    sign = np.where(rng.random(n) < 0.5, -1, 1).astype(np.float32)
    x = mag * sign
    exact = bits_to_f32(rng.integers(0, 0x7F7F, 64).astype(np.uint16))
    nb = np.nextafter(exact, np.float32(np.inf))
    return np.concatenate([x, exact, -exact, nb, -nb]).astype(np.float32)


@pytest.mark.parametrize("mode", [oracle.RN, oracle.RD, oracle.RU])
def test_bf16_rounding_is_brute_force(mode):
    rng = np.random.default_rng(40 + mode)
    x = _random_f32(rng, 1500)
    got = oracle.f32_to_bf16_bits(x, mode)
    np.testing.assert_array_equal(got, _brute_bf16(x, mode))


def test_bf16_nearest_matches_bit_rounding():
    """Round-to-nearest-even on the binary32 bits (add 0x7FFF plus the lowest
    kept bit) is the textbook bfloat16 conversion for finite values."""
    rng = np.random.default_rng(7)
    x = _random_f32(rng, 3000)
    ref = to_bf16(x)
    finite = np.isfinite(bits_to_f32(ref))
    ref = np.where(bits_to_f32(ref) == 0, 0, ref).astype(np.uint16)
    got = oracle.f32_to_bf16_bits(x, oracle.RN)
    np.testing.assert_array_equal(got[finite], ref[finite])


def test_bf16_saturation_zero_and_subnormals():
    B = lambda v, m: int(oracle.f32_to_bf16_bits(np.float32(v), m))
    for m in (oracle.RN, oracle.RD, oracle.RU):
        assert B(np.finfo(np.float32).max, m) == 0x7F7F
        assert B(-np.finfo(np.float32).max, m) == 0xFF7F
        assert B(np.inf, m) == 0x7F7F
        assert B(-0.0, m) == 0x0000
        assert B(1.0, m) == 0x3F80
    tiny = np.float32(1e-45)  # the smallest binary32 subnormal, 2^-149
    assert B(tiny, oracle.RU) == 0x0001  # 2^-133
    assert B(tiny, oracle.RD) == 0x0000
    assert B(-tiny, oracle.RD) == 0x8001
    assert B(-tiny, oracle.RU) == 0x0000
    assert B(1.0 + 2.0 ** -8, oracle.RN) == 0x3F80  # tie -> even
    assert B(1.0 + 3 * 2.0 ** -8, oracle.RN) == 0x3F82
    assert B(1.0 + 2.0 ** -20, oracle.RU) == 0x3F81
    assert B(np.nan, oracle.RN) == 0x7FC0


# ---------------------------------------------------------------- binary16 input

def _both_formats(rng, n, D):
    """Rows whose values exist in bfloat16 and in binary16 (8 significant bits,
    binary16 normal range): (bf16 bits, f16 bits, float32 values)."""
    m = rng.integers(-255, 256, (n, D)).astype(np.float32)
    e = rng.integers(-6, 5, (n, 1)).astype(np.float32)
    x = (m * np.exp2(e)).astype(np.float32)
    return bf16_bits(x), x.astype(np.float16).view(np.uint16), x


@pytest.mark.parametrize("rotate,h", [(False, 128), (True, 128), (True, 16)])
@pytest.mark.parametrize("meta_bf16", [False, True])
def test_f16_input_equals_bf16_input_on_shared_values(rotate, h, meta_bf16):
    rng = np.random.default_rng(int(rotate) * 100 + h + int(meta_bf16))
    xb, xh, _ = _both_formats(rng, 40, 128)
    a = oracle.quantize_rows(xb, rotate, h, meta_bf16=meta_bf16)
    b = oracle.quantize_rows(xh, rotate, h, in_f16=True, meta_bf16=meta_bf16)
    for u, v in zip(a, b):
        np.testing.assert_array_equal(u, v)


def test_f16_only_values_give_closed_form_codes():
    """1 + k 2^-10 (k = 0..15) exists in binary16, not in bfloat16: the row's
    zero is 1, its scale 2^-10 exactly, so the codes are k."""
    k = np.tile(np.arange(16), 8)
    x = (1.0 + k * 2.0 ** -10).astype(np.float16)
    codes, s, z = oracle.quantize_rows(x.view(np.uint16)[None], False, 128, in_f16=True)
    assert int(z[0]) == 0x3C00 and int(s[0]) == 0x1400
    np.testing.assert_array_equal(unpack(codes[0]), k)


def test_f16_subnormal_inputs_widen_exactly():
    """Binary16 subnormals m 2^-24 (m = 0..15): with a bfloat16 zero of 0 and
    scale 2^-24 every code is m."""
    m = np.tile(np.arange(16, dtype=np.uint16), 8)
    codes, s, z = oracle.quantize_rows(m[None], False, 128, in_f16=True, meta_bf16=True)
    assert int(z[0]) == 0 and int(s[0]) == 0x3380  # 2^-24 in bfloat16
    np.testing.assert_array_equal(unpack(codes[0]), m)


# ---------------------------------------------------------------- bfloat16 metadata

KINDS = ["normal", "outlier", "heavy", "bias", "tiny", "huge"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("rotate,h", [(False, 128), (True, 128), (True, 32)])
def test_bf16_meta_rounding_and_error_bound(kind, rotate, h):
    D = 128
    rng = np.random.default_rng(KINDS.index(kind) * 97 + int(rotate) * 7 + h)
    xb = _rows(rng, 48, D, kind)
    codes, s, z = oracle.quantize_rows(xb, rotate, h, meta_bf16=True)
    y = bits_to_f32(xb)
    if rotate:
        y = oracle.rotate_canon(y, h)
    mn, mx = y.min(1), y.max(1)
    # zero: the largest bfloat16 <= min; scale: the smallest >= RN((max - z)/15)
    np.testing.assert_array_equal(z, _brute_bf16(mn, oracle.RD))
    zf = bits_to_f32(z)
    step = ((mx - zf).astype(np.float32) / np.float32(15)).astype(np.float32)
    np.testing.assert_array_equal(s, _bf16_scale(step))
    sv = bits_to_f32(s).astype(np.float64)[:, None]
    zv = zf.astype(np.float64)[:, None]
    yd = y.astype(np.float64)
    deq = oracle.dequant_rows(codes, s, z, meta_bf16=True)
    slack = 2.0 ** -20 * (np.abs(yd) + np.abs(zv) + 15 * sv)
    assert np.all(np.abs(yd - deq) <= sv / 2 + slack)
    # the codes are round-half-even of (y - z) / s in binary32, clamped
    r = np.where(sv[:, 0] == 0, 0, (np.float32(1) / sv[:, 0].astype(np.float32))).astype(np.float32)
    v = ((y - zf[:, None]).astype(np.float32) * r[:, None]).astype(np.float32)
    np.testing.assert_array_equal(unpack(codes), np.clip(np.rint(v), 0, 15).astype(np.uint8))


def test_bf16_meta_subnormal_rows_floor_the_scale():
    """Rows of bfloat16 subnormals: the scale rounded up would be subnormal
    too, and its reciprocal would overflow binary32; it is raised to 2^-126,
    and every value still lies within s/2 of its dequantized value."""
    m = np.tile(np.arange(16, dtype=np.uint16), 8)  # m 2^-133
    codes, s, z = oracle.quantize_rows(m[None], False, 128, meta_bf16=True)
    assert int(z[0]) == 0 and int(s[0]) == 0x0080
    assert np.all(unpack(codes[0]) == 0)  # every value is below 2^-127 = s/2
    y = bits_to_f32(m).astype(np.float64)
    deq = oracle.dequant_rows(codes, s, z, meta_bf16=True)[0]
    assert np.all(np.abs(y - deq) <= 2.0 ** -127)
    big = np.concatenate([m[:64], np.full(64, 0x0100, np.uint16)])  # 2^-125 at the top
    codes, s, z = oracle.quantize_rows(big[None], False, 128, meta_bf16=True)
    assert int(s[0]) == 0x0080
    np.testing.assert_array_equal(unpack(codes[0])[64:], 2)


def test_bf16_meta_closed_form():
    """z0 + k s0 with z0, s0 exact in bfloat16 and every step exact: codes k."""
    k = np.tile(np.arange(16), 8)
    z0, s0 = -3.0, 0.375
    x = (z0 + k * s0).astype(np.float32)
    codes, s, z = oracle.quantize_rows(bf16_bits(x)[None], False, 128, meta_bf16=True)
    assert int(z[0]) == int(bf16_bits(np.float32(z0))) and int(s[0]) == int(bf16_bits(np.float32(s0)))
    np.testing.assert_array_equal(unpack(codes[0]), k)


def test_bf16_meta_covers_what_binary16_saturates():
    """Rows beyond the binary16 range (|x| up to 10^6): binary16 metadata
    saturates and its codes clamp; bfloat16 metadata keeps the s/2 bound."""
    rng = np.random.default_rng(11)
    xb = to_bf16((rng.standard_normal((16, 128)) * 3e5).astype(np.float32))
    y = bits_to_f32(xb).astype(np.float64)
    c16, s16, z16 = oracle.quantize_rows(xb, False, 128)
    cb, sb, zb = oracle.quantize_rows(xb, False, 128, meta_bf16=True)
    err16 = np.abs(y - oracle.dequant_rows(c16, s16, z16)).max()
    errb = np.abs(y - oracle.dequant_rows(cb, sb, zb, meta_bf16=True))
    sv = bits_to_f32(sb).astype(np.float64)[:, None]
    assert np.all(errb <= sv / 2 * (1 + 2.0 ** -18))
    assert err16 > 10 * errb.max()


def test_bf16_meta_degenerate_rows():
    D = 128
    const = bf16_bits(np.full(D, 2.5, np.float32))[None]
    codes, s, z = oracle.quantize_rows(const, False, 128, meta_bf16=True)
    assert int(s[0]) == 0 and int(z[0]) == int(bf16_bits(np.float32(2.5)))
    assert np.all(codes == 0)
    zero = np.zeros((1, D), np.uint16)
    codes, s, z = oracle.quantize_rows(zero, True, 128, meta_bf16=True)
    assert int(s[0]) == 0 and int(z[0]) == 0 and np.all(codes == 0)
    negz = np.full((1, D), 0x8000, np.uint16)  # -0.0 everywhere: the zero is stored as +0
    codes, s, z = oracle.quantize_rows(negz, False, 128, meta_bf16=True)
    assert int(z[0]) == 0 and int(s[0]) == 0


# ---------------------------------------------------------------- attention

def _paged(rng, L, Hkv, D, P, rotate_k, rotate_v, h, in_f16, meta_bf16):
    npages = -(-L // P) + 2
    ids = rng.permutation(npages)
    bt = ids[: -(-L // P)].astype(np.int32)[None]
    slots = np.array([bt[0, j // P] * P + j % P for j in range(L)], np.int32)
    if in_f16:
        k = (rng.standard_normal((L, Hkv, D)) * 2).astype(np.float16).view(np.uint16)
        v = rng.standard_t(3, (L, Hkv, D)).astype(np.float16).view(np.uint16)
    else:
        k = _rows(rng, L * Hkv, D, "outlier").reshape(L, Hkv, D)
        v = _rows(rng, L * Hkv, D, "heavy").reshape(L, Hkv, D)
    nb = oracle.cache_bytes(npages, P, Hkv, D)
    kc, vc = np.zeros(nb, np.uint8), np.zeros(nb, np.uint8)
    assert oracle.quantize_append(k, v, slots, Hkv, D, kc, vc, npages, P, rotate_k, rotate_v, h,
                                  in_f16=in_f16, meta_bf16=meta_bf16) == 0
    return bt, slots, kc, vc, npages


@pytest.mark.parametrize("in_f16,meta_bf16", [(True, False), (False, True), (True, True)])
def test_decode_variants_equal_dense_softmax(in_f16, meta_bf16):
    """Attention over the variant caches equals scipy's softmax over the rows
    that the oracle's own dequantizer reads back, in the rotated domain."""
    rng = np.random.default_rng(int(in_f16) * 2 + int(meta_bf16))
    L, Hq, Hkv, D, P, h = 45, 4, 2, 128, 16, 64
    bt, slots, kc, vc, npages = _paged(rng, L, Hkv, D, P, True, True, h, in_f16, meta_bf16)
    if in_f16:
        q = rng.standard_normal((1, Hq, D)).astype(np.float16).view(np.uint16)
        qf = q.view(np.float16).astype(np.float64)[0]
    else:
        q = _rows(rng, Hq, D, "normal").reshape(1, Hq, D)
        qf = bits_to_f32(q[0]).astype(np.float64)
    got = oracle.decode(q, kc, vc, bt, [L], Hq, Hkv, D, npages, P, True, True, h,
                        in_f16=in_f16, meta_bf16=meta_bf16)
    Hm = np.kron(np.eye(D // h), scipy.linalg.hadamard(h)) / math.sqrt(h)
    chunk = P * D // 2 + 4 * P
    for hq in range(Hq):
        kvh = hq // (Hq // Hkv)
        rows_k, rows_v = [], []
        for j in range(L):
            base = (int(bt[0, j // P]) * Hkv + kvh) * chunk
            off = j % P
            for cache, dst in ((kc, rows_k), (vc, rows_v)):
                codes = cache[base + off * D // 2: base + (off + 1) * D // 2]
                meta = cache[base + P * D // 2 + 4 * off: base + P * D // 2 + 4 * off + 4]
                sb = int(meta[0]) | int(meta[1]) << 8
                zb = int(meta[2]) | int(meta[3]) << 8
                dst.append(oracle.dequant_rows(codes, sb, zb, meta_bf16=meta_bf16)[0])
        kh, vh = np.array(rows_k), np.array(rows_v)
        p = scipy.special.softmax((kh @ (Hm @ qf[hq])) / math.sqrt(D))
        ref = Hm @ (p @ vh)
        np.testing.assert_allclose(got[hq], ref, rtol=1e-11, atol=1e-12)


def test_decode_f16_q_equals_bf16_q_on_shared_values():
    rng = np.random.default_rng(5)
    L, Hq, Hkv, D, P, h = 30, 2, 1, 128, 16, 128
    bt, slots, kc, vc, npages = _paged(rng, L, Hkv, D, P, True, False, h, False, False)
    xb, xh, _ = _both_formats(rng, Hq, D)
    a = oracle.decode(xb.reshape(1, Hq, D), kc, vc, bt, [L], Hq, Hkv, D, npages, P, True, False, h)
    b = oracle.decode(xh.reshape(1, Hq, D), kc, vc, bt, [L], Hq, Hkv, D, npages, P, True, False, h,
                      in_f16=True)
    np.testing.assert_array_equal(a, b)


def test_prefill_variants_equal_decode_prefixes():
    rng = np.random.default_rng(9)
    L, Hq, Hkv, D, P, h = 24, 2, 1, 128, 16, 128
    bt, slots, kc, vc, npages = _paged(rng, L, Hkv, D, P, True, True, h, True, True)
    qlen = 5
    q = rng.standard_normal((qlen, Hq, D)).astype(np.float16).view(np.uint16)
    out = oracle.prefill(q, [0, qlen], kc, vc, bt, [L], Hq, Hkv, D, npages, P, True, True, h,
                         in_f16=True, meta_bf16=True)
    for i in range(qlen):
        ref = oracle.decode(q[i:i + 1], kc, vc, bt, [L - qlen + i + 1], Hq, Hkv, D, npages, P,
                            True, True, h, in_f16=True, meta_bf16=True)
        np.testing.assert_array_equal(out[i * Hq:(i + 1) * Hq], ref)
