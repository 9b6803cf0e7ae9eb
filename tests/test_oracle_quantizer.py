"""Pins for the oracle's token-wise INT4 quantizer and paged append (CPU only).

What the pages fix: one scale per token, computed when the token arrives,
appended into a paged block without revisiting past tokens (youngju.dev
"Why Naive INT4 Breaks", "The System Is the Design -- A Fused Kernel";
gist.science s.2 "Quantizzazione Token-wise").  Readings where they are
silent: an asymmetric binary16 (scale, zero) from the row's min/max, zero
rounded down and scale rounded up, round-half-even codes, even index in the
low nibble.  Pins: hand-worked fixtures, the error bound that the directed
rounding guarantees, closed forms, and token-wise independence.
"""
import numpy as np
import pytest
import scipy.linalg

import oracle
from conftest import read_golden


def bf16_bits(x):
    """float32 values that are exactly bfloat16 -> their bit patterns."""
    x = np.asarray(x, dtype=np.float32)
    b = x.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value is not exactly representable in bfloat16"
    return (b >> 16).astype(np.uint16)


def to_bf16(x, rng=None):
    """Round float32 values to bfloat16 (nearest-even) -> bit patterns."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16).astype(np.uint16)
    return r


def bits_to_f32(b):
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def unpack(codes):
    codes = np.asarray(codes, dtype=np.uint8)
    out = np.empty(codes.shape[:-1] + (codes.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = codes & 15
    out[..., 1::2] = codes >> 4
    return out


@pytest.mark.parametrize("block", [0, 1])
def test_hand_worked_examples(block):
    blocks, _ = read_golden("asym_int4_8elem.txt")
    ex = blocks[block]
    x = np.array([float(v) for v in ex["x"].split()], np.float32)
    codes, s, z = oracle.quantize_rows(bf16_bits(x)[None], rotate=False, h=8)
    assert int(z[0]) == int(ex["z_bits"], 16)
    assert int(s[0]) == int(ex["s_bits"], 16)
    np.testing.assert_array_equal(unpack(codes[0]), [int(v) for v in ex["codes"].split()])
    np.testing.assert_array_equal(codes[0], [int(v, 16) for v in ex["packed"].split()])
    deq = oracle.dequant_rows(codes, s, z)[0]
    sv = oracle.f16_bits_to_f64(s)[0]
    assert np.all(np.abs(deq - x) <= sv / 2)


def test_one_hot_closed_form():
    blocks, _ = read_golden("onehot_h128.txt")
    ex = blocks[0]
    j, h = int(ex["j"]), int(ex["h"])
    x = np.zeros(h, np.float32)
    x[j] = 1.0
    codes, s, z = oracle.quantize_rows(bf16_bits(x)[None], rotate=True, h=h)
    assert int(z[0]) == int(ex["z_bits"], 16)
    assert int(s[0]) == int(ex["s_bits"], 16)
    H = scipy.linalg.hadamard(h)
    np.testing.assert_array_equal(unpack(codes[0]), np.where(H[:, j] > 0, 15, 0))


def _rows(rng, n, D, kind):
    if kind == "normal":
        x = rng.standard_normal((n, D))
    elif kind == "outlier":
        x = rng.standard_normal((n, D))
        x[:, rng.choice(D, 4, replace=False)] *= 20
    elif kind == "heavy":
        x = rng.standard_t(3, (n, D))
    elif kind == "bias":
        x = rng.standard_normal((n, D)) + 2 * rng.standard_normal(D)
    elif kind == "tiny":
        x = rng.standard_normal((n, D)) * 1e-6
    elif kind == "huge":
        x = rng.standard_normal((n, D)) * 3000
    return to_bf16(x.astype(np.float32))


KINDS = ["normal", "outlier", "heavy", "bias", "tiny", "huge"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("rotate,h", [(False, 128), (True, 128), (True, 64)])
def test_error_bound_and_coverage(kind, rotate, h):
    """Directed rounding of (s, z) puts every value inside [z, z + 15 s], so
    |y - y_hat| <= s/2 up to binary32 slack."""
    D = 128
    rng = np.random.default_rng(KINDS.index(kind) * 1000 + int(rotate) * 300 + h)
    xb = _rows(rng, 64, D, kind)
    codes, s, z = oracle.quantize_rows(xb, rotate, h)
    y = bits_to_f32(xb)
    if rotate:
        y = oracle.rotate_canon(y, h)
    y = y.astype(np.float64)
    sv = oracle.f16_bits_to_f64(s)[:, None]
    zv = oracle.f16_bits_to_f64(z)[:, None]
    mn, mx = y.min(1, keepdims=True), y.max(1, keepdims=True)
    assert np.all(zv <= mn)
    assert np.all(zv + 15 * sv >= mx * (1 - 2.0 ** -20) - 2.0 ** -20 * np.abs(zv))
    deq = oracle.dequant_rows(codes, s, z)
    slack = 2.0 ** -20 * (np.abs(y) + np.abs(zv) + 15 * sv)
    assert np.all(np.abs(y - deq) <= sv / 2 + slack)
    q = unpack(codes)
    rows = np.arange(len(y))
    # the maximum lands on code 15 whenever s is a normal binary16 value (its
    # upward rounding is then below 2^-10 relative); the minimum on 0 unless
    # binary16 rounding of z is coarser than half a step
    normal = sv[:, 0] >= 2.0 ** -14
    assert np.all(q[rows, y.argmax(1)][normal] == 15)
    assert np.all(q[rows, y.argmax(1)] >= np.floor(15 * (mx[:, 0] - zv[:, 0]) / (15 * sv[:, 0]) - 1e-6))
    spacing = np.maximum(np.abs(mn[:, 0]) * 2.0 ** -10, 2.0 ** -24)
    ok = spacing < sv[:, 0] / 2
    assert np.all(q[rows, y.argmin(1)][ok] == 0)


def test_degenerate_rows():
    D = 128
    # constant binary16-exact row: zero = value, scale 0, all codes 0, exact
    x = np.full((1, D), 1.5, np.float32)
    codes, s, z = oracle.quantize_rows(bf16_bits(x), False, 128)
    assert int(s[0]) == 0 and oracle.f16_bits_to_f64(z)[0] == 1.5
    assert np.all(codes == 0)
    np.testing.assert_array_equal(oracle.dequant_rows(codes, s, z), x)
    # all-zero row with rotation, including negative zeros: z = s = +0
    xb = np.zeros((1, D), np.uint16)
    xb[0, ::3] = 0x8000
    codes, s, z = oracle.quantize_rows(xb, True, 128)
    assert int(s[0]) == 0 and int(z[0]) == 0 and np.all(codes == 0)
    # constant row below binary16's normal range: z rounds down, s > 0
    xb = np.full((1, D), to_bf16(np.float32(1e-6)), np.uint16)
    codes, s, z = oracle.quantize_rows(xb, False, 128)
    assert oracle.f16_bits_to_f64(z)[0] < 1e-6 and int(s[0]) != 0


def test_unrotated_is_textbook_minmax():
    """Rotation off, values where binary16 rounding is exact: the codes are
    the textbook round((x - min) / ((max - min)/15))."""
    rng = np.random.default_rng(3)
    # integers in [0, 15*k] scaled by powers of two keep s and z exact
    for k in (1, 2, 4):
        q = rng.integers(0, 16, (32, 128))
        q[:, 0], q[:, 1] = 0, 15
        x = (q * k - 8.0).astype(np.float32)
        codes, s, z = oracle.quantize_rows(bf16_bits(x), False, 128)
        np.testing.assert_array_equal(unpack(codes), q)
        assert np.all(oracle.f16_bits_to_f64(s) == k)
        assert np.all(oracle.f16_bits_to_f64(z) == -8.0)


def _cache_rows(cache, slots, head, Hkv, P, D):
    """Read (codes, s, z) of given slots back from a cache byte array, by the
    layout reading: chunk = P*D/2 code bytes then P*(s,z) binary16 words."""
    chunk = P * D // 2 + P * 4
    out_c, out_s, out_z = [], [], []
    for sl in slots:
        page, off = divmod(int(sl), P)
        base = (page * Hkv + head) * chunk
        out_c.append(cache[base + off * D // 2: base + (off + 1) * D // 2])
        m = cache[base + P * D // 2 + 4 * off: base + P * D // 2 + 4 * off + 4]
        out_s.append(int(m[0]) | int(m[1]) << 8)
        out_z.append(int(m[2]) | int(m[3]) << 8)
    return np.array(out_c), np.array(out_s, np.uint16), np.array(out_z, np.uint16)


def test_append_layout_and_independence():
    """Token-wise independence: any subset, order or batch split of appends
    gives the same bytes at those slots and leaves every other byte alone."""
    rng = np.random.default_rng(11)
    T, Hkv, D, P, num_pages = 40, 2, 128, 16, 6
    k = _rows(rng, T * Hkv, D, "outlier").reshape(T, Hkv, D)
    v = _rows(rng, T * Hkv, D, "heavy").reshape(T, Hkv, D)
    slots = rng.permutation(num_pages * P)[:T].astype(np.int32)
    nbytes = oracle.cache_bytes(num_pages, P, Hkv, D)
    assert nbytes == num_pages * Hkv * (P * D // 2 + 4 * P)

    def fresh():
        return np.full(nbytes, 0xAB, np.uint8), np.full(nbytes, 0xAB, np.uint8)

    kc, vc = fresh()
    assert oracle.quantize_append(k, v, slots, Hkv, D, kc, vc, num_pages, P, True, False, 128) == 0
    # rows land where the layout says, with the row quantizer's bytes
    for hd in range(Hkv):
        c, s, z = _cache_rows(kc, slots, hd, Hkv, P, D)
        c2, s2, z2 = oracle.quantize_rows(k[:, hd], True, 128)
        np.testing.assert_array_equal(c, c2)
        np.testing.assert_array_equal(s, s2)
        np.testing.assert_array_equal(z, z2)
        c, s, z = _cache_rows(vc, slots, hd, Hkv, P, D)
        c2, s2, z2 = oracle.quantize_rows(v[:, hd], False, 128)
        np.testing.assert_array_equal(c, c2)
        np.testing.assert_array_equal(s, s2)
    # reversed order, in three batches, with a padded (-1) entry mixed in
    kc2, vc2 = fresh()
    order = np.arange(T)[::-1]
    for part in np.array_split(order, 3):
        sl = slots[part].copy()
        kk, vv = k[part], v[part]
        sl = np.concatenate([sl, [-1]]).astype(np.int32)
        kk = np.concatenate([kk, k[:1]])
        vv = np.concatenate([vv, v[:1]])
        oracle.quantize_append(kk, vv, sl, Hkv, D, kc2, vc2, num_pages, P, True, False, 128)
    np.testing.assert_array_equal(kc, kc2)
    np.testing.assert_array_equal(vc, vc2)
    # untouched slots keep the sentinel
    touched = np.zeros(nbytes, bool)
    chunk = P * D // 2 + 4 * P
    for sl in slots:
        page, off = divmod(int(sl), P)
        for hd in range(Hkv):
            base = (page * Hkv + hd) * chunk
            touched[base + off * D // 2: base + (off + 1) * D // 2] = True
            touched[base + P * D // 2 + 4 * off: base + P * D // 2 + 4 * off + 4] = True
    assert np.all(kc[~touched] == 0xAB)
    # threads split the token range without changing a byte
    kc3, vc3 = fresh()
    oracle.quantize_append(k, v, slots, Hkv, D, kc3, vc3, num_pages, P, True, False, 128, threads=4)
    np.testing.assert_array_equal(kc, kc3)


def test_bad_slots_are_counted_and_skipped():
    rng = np.random.default_rng(5)
    Hkv, D, P, num_pages = 1, 128, 16, 2
    k = _rows(rng, 4, D, "normal").reshape(4, 1, D)
    slots = np.array([0, -1, num_pages * P, -7], np.int32)
    nbytes = oracle.cache_bytes(num_pages, P, Hkv, D)
    kc = np.full(nbytes, 0xAB, np.uint8)
    bad = oracle.quantize_append(k, None, slots, Hkv, D, kc, None, num_pages, P, True, True, 128)
    assert bad == 2
    c, _, _ = _cache_rows(kc, [0], 0, Hkv, P, D)
    c2, _, _ = oracle.quantize_rows(k[:1, 0], True, 128)
    np.testing.assert_array_equal(c, c2)
