"""Pins of the BF16-cache baseline in the oracle (the unquantized KV cache that
gist.science s.4 compares SAW-INT4's throughput against).

The append is a placement (checked element by element against the layout);
the decode is checked against a dense attention over the un-paged rows, a
hand-worked softmax, and invariances that hold for any attention.
"""
import math

import numpy as np
import pytest

import oracle


def _bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bfloat16 bit patterns (round to nearest even)."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def _f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint32) << 16).view(np.float32)


def _caches(num_pages, P, Hkv, D, fill=0xABCD):
    n = oracle.bf16_cache_bytes(num_pages, P, Hkv, D) // 2
    return np.full(n, fill, np.uint16), np.full(n, fill, np.uint16)


def test_layout_padding_and_bad_slots():
    rng = np.random.default_rng(0)
    T, Hkv, D, P, pages = 12, 3, 128, 16, 2
    k = _bits(rng.standard_normal((T, Hkv, D)))
    v = _bits(rng.standard_normal((T, Hkv, D)))
    slots = rng.permutation(pages * P)[:T].astype(np.int32)
    slots[2] = -1            # padding: skipped silently
    slots[5] = pages * P     # one past the end: skipped and counted
    slots[7] = -3            # negative: skipped and counted
    kc, vc = _caches(pages, P, Hkv, D)
    bad = oracle.bf16_append(k, v, slots, Hkv, D, kc, vc, pages, P)
    assert bad == 2
    written = np.zeros(kc.size, bool)
    for t in range(T):
        s = int(slots[t])
        if s < 0 or s >= pages * P:
            continue
        for hd in range(Hkv):
            base = ((s // P * Hkv + hd) * P + s % P) * D
            assert np.array_equal(kc[base:base + D], k[t, hd])
            assert np.array_equal(vc[base:base + D], v[t, hd])
            written[base:base + D] = True
    assert np.all(kc[~written] == 0xABCD) and np.all(vc[~written] == 0xABCD)


def _fill(lens, Hkv, D, P, rng, shuffle=True):
    """Caches with every token of every sequence, and the rows in order."""
    pages_per = [-(-L // P) for L in lens]
    num_pages = sum(pages_per) + 2
    ids = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    bt = np.full((len(lens), max(max(pages_per), 1)), -7, np.int32)
    rows_k, rows_v, c = [], [], 0
    kc, vc = _caches(num_pages, P, Hkv, D)
    for b, L in enumerate(lens):
        bt[b, :pages_per[b]] = ids[c:c + pages_per[b]]
        c += pages_per[b]
        k = _bits(rng.standard_normal((L, Hkv, D)) * 2)
        v = _bits(rng.standard_normal((L, Hkv, D)))
        slots = np.array([bt[b, j // P] * P + j % P for j in range(L)], np.int32)
        assert oracle.bf16_append(k, v, slots, Hkv, D, kc, vc, num_pages, P) == 0
        rows_k.append(k)
        rows_v.append(v)
    return kc, vc, bt, num_pages, rows_k, rows_v


@pytest.mark.parametrize("Hq,Hkv,P", [(4, 2, 16), (8, 1, 64), (6, 3, 32)])
def test_decode_equals_dense_attention_over_unpaged_rows(Hq, Hkv, P):
    rng = np.random.default_rng(Hq * 10 + P)
    D, lens = 128, [1, 37, 100, 0, 16]
    kc, vc, bt, num_pages, rk, rv = _fill(lens, Hkv, D, P, rng)
    q = _bits(rng.standard_normal((len(lens), Hq, D)))
    out = oracle.decode_bf16(q, kc, vc, bt, lens, Hq, Hkv, D, num_pages, P)
    G = Hq // Hkv
    i = 0
    for b, L in enumerate(lens):
        for hq in range(Hq):
            if L == 0:
                ref = np.zeros(D)
            else:
                K = _f32(rk[b][:, hq // G]).astype(np.float64)
                V = _f32(rv[b][:, hq // G]).astype(np.float64)
                t = K @ _f32(q[b, hq]).astype(np.float64) / math.sqrt(D)
                p = np.exp(t - t.max())
                ref = p @ V / p.sum()
            np.testing.assert_allclose(out[i], ref, rtol=1e-12, atol=1e-12)
            i += 1


def test_hand_worked_two_tokens():
    """q = e0, k0 = 0, k1 = e0, sm_scale = ln 2: t = (0, ln 2), p = (1/3, 2/3);
    v0 = 3 e1, v1 = 6 e1, so o = 5 e1 exactly."""
    D, P = 128, 16
    k = np.zeros((2, 1, D), np.float32)
    k[1, 0, 0] = 1.0
    v = np.zeros((2, 1, D), np.float32)
    v[0, 0, 1], v[1, 0, 1] = 3.0, 6.0
    kc, vc = _caches(1, P, 1, D)
    oracle.bf16_append(_bits(k), _bits(v), np.array([0, 1], np.int32), 1, D, kc, vc, 1, P)
    q = np.zeros((1, 1, D), np.float32)
    q[0, 0, 0] = 1.0
    out = oracle.decode_bf16(_bits(q), kc, vc, np.zeros((1, 1), np.int32), [2], 1, 1, D, 1, P,
                             sm_scale=math.log(2.0))
    ref = np.zeros(D)
    ref[1] = 5.0
    np.testing.assert_allclose(out[0], ref, rtol=0, atol=1e-14)


def test_single_token_identical_keys_and_page_permutation():
    rng = np.random.default_rng(3)
    D, P, Hkv, Hq = 128, 16, 1, 2
    # one token: the output is its value row
    kc, vc, bt, npg, rk, rv = _fill([1], Hkv, D, P, rng)
    q = _bits(rng.standard_normal((1, Hq, D)))
    out = oracle.decode_bf16(q, kc, vc, bt, [1], Hq, Hkv, D, npg, P)
    assert np.array_equal(out[0], _f32(rv[0][0, 0]).astype(np.float64))
    # identical keys: the output is the mean of the values
    L = 40
    k = np.tile(_bits(rng.standard_normal((1, 1, D))), (L, 1, 1))
    v = _bits(rng.standard_normal((L, 1, D)))
    kc, vc = _caches(3, P, 1, D)
    bt = np.array([[2, 0, 1]], np.int32)
    slots = np.array([bt[0, j // P] * P + j % P for j in range(L)], np.int32)
    oracle.bf16_append(k, v, slots, 1, D, kc, vc, 3, P)
    out = oracle.decode_bf16(q[:, :1], kc, vc, bt, [L], 1, 1, D, 3, P)
    np.testing.assert_allclose(out[0], _f32(v[:, 0]).astype(np.float64).mean(0), rtol=1e-12,
                               atol=1e-12)
    # the same tokens through another page permutation give the same output
    kc2, vc2 = _caches(3, P, 1, D)
    bt2 = np.array([[1, 2, 0]], np.int32)
    slots2 = np.array([bt2[0, j // P] * P + j % P for j in range(L)], np.int32)
    oracle.bf16_append(k, v, slots2, 1, D, kc2, vc2, 3, P)
    out2 = oracle.decode_bf16(q[:, :1], kc2, vc2, bt2, [L], 1, 1, D, 3, P)
    assert np.array_equal(out, out2)
