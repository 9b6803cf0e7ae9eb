"""Pins for the oracle's decode attention over INT4 pages (CPU only).

The oracle attends in the rotated domain: it rotates q once and un-rotates
the output when V was rotated.  That rests on the rotation being orthogonal
and undoable (youngju.dev "The Rotation Trick -- Block-Diagonal Hadamard";
gist.science s.2 "Rotazione Block-Diagonale").  These tests compute the
same attention a different way -- dense, un-paged, in the ORIGINAL domain,
with keys and values explicitly rotated back by scipy's Hadamard matrix and
scipy's softmax -- and check special cases with closed forms.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import scipy.special

import oracle
from test_oracle_quantizer import _cache_rows, _rows, bits_to_f32


def _build(rng, seq_lens, Hq, Hkv, D, P, rotate_k, rotate_v, h, shuffle=True, kv=None):
    B = len(seq_lens)
    pages_per = [-(-L // P) for L in seq_lens]
    num_pages = sum(pages_per) + 3
    ids = rng.permutation(num_pages) if shuffle else np.arange(num_pages)
    max_blocks = max(pages_per)
    bt = np.full((B, max_blocks), -1, np.int32)
    nxt = 0
    for b in range(B):
        for i in range(pages_per[b]):
            bt[b, i] = ids[nxt]
            nxt += 1
    T = sum(seq_lens)
    if kv is None:
        k = _rows(rng, T * Hkv, D, "outlier").reshape(T, Hkv, D)
        v = _rows(rng, T * Hkv, D, "heavy").reshape(T, Hkv, D)
    else:
        k, v = kv
    slots = []
    for b in range(B):
        for j in range(seq_lens[b]):
            slots.append(bt[b, j // P] * P + j % P)
    slots = np.array(slots, np.int32)
    nbytes = oracle.cache_bytes(num_pages, P, Hkv, D)
    kc = np.zeros(nbytes, np.uint8)
    vc = np.zeros(nbytes, np.uint8)
    assert oracle.quantize_append(k, v, slots, Hkv, D, kc, vc, num_pages, P, rotate_k, rotate_v, h) == 0
    q = _rows(rng, B * Hq, D, "normal").reshape(B, Hq, D)
    return dict(bt=bt, slots=slots, kc=kc, vc=vc, q=q, num_pages=num_pages, k=k, v=v)


def _dense_reference(d, seq_lens, Hq, Hkv, D, P, rotate_k, rotate_v, h, scale):
    """Original-domain attention: dequantize each appended row, rotate it back
    with scipy's Hadamard (1/sqrt h) H, and attend with the un-rotated q."""
    R = np.zeros((D, D))
    Hh = scipy.linalg.hadamard(h) / math.sqrt(h)
    for b0 in range(0, D, h):
        R[b0:b0 + h, b0:b0 + h] = Hh
    G = Hq // Hkv
    out = np.zeros((len(seq_lens), Hq, D))
    start = 0
    for b, L in enumerate(seq_lens):
        sl = d["slots"][start:start + L]
        start += L
        for hq in range(Hq):
            kvh = hq // G
            c, s, z = _cache_rows(d["kc"], sl, kvh, Hkv, P, D)
            kh = oracle.dequant_rows(c, s, z)
            c, s, z = _cache_rows(d["vc"], sl, kvh, Hkv, P, D)
            vh = oracle.dequant_rows(c, s, z)
            if rotate_k:
                kh = kh @ R  # R symmetric: row-wise R^-1 k = R k
            if rotate_v:
                vh = vh @ R
            q = bits_to_f32(d["q"][b, hq]).astype(np.float64)
            p = scipy.special.softmax(scale * (kh @ q))
            out[b, hq] = p @ vh
    return out


@pytest.mark.parametrize("rotate_k,rotate_v,h", [(True, True, 128), (True, False, 128),
                                                  (False, False, 128), (True, True, 64)])
def test_rotated_q_equals_dense_original_domain(rotate_k, rotate_v, h):
    rng = np.random.default_rng(int(rotate_k) * 2 + int(rotate_v) + h)
    seq_lens = [1, 17, 40, 16]
    Hq, Hkv, D, P = 4, 2, 128, 16
    d = _build(rng, seq_lens, Hq, Hkv, D, P, rotate_k, rotate_v, h)
    got = oracle.decode(d["q"], d["kc"], d["vc"], d["bt"], seq_lens, Hq, Hkv, D, d["num_pages"],
                        P, rotate_k, rotate_v, h).reshape(len(seq_lens), Hq, D)
    ref = _dense_reference(d, seq_lens, Hq, Hkv, D, P, rotate_k, rotate_v, h, 1 / math.sqrt(D))
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=1e-12)


def test_single_token_returns_its_value():
    rng = np.random.default_rng(1)
    Hq, Hkv, D, P, h = 2, 1, 128, 16, 128
    d = _build(rng, [1], Hq, Hkv, D, P, True, True, h)
    got = oracle.decode(d["q"], d["kc"], d["vc"], d["bt"], [1], Hq, Hkv, D, d["num_pages"], P,
                        True, True, h)
    c, s, z = _cache_rows(d["vc"], d["slots"][:1], 0, Hkv, P, D)
    v0 = oracle.dequant_rows(c, s, z)[0] @ (scipy.linalg.hadamard(h) / math.sqrt(h))
    np.testing.assert_allclose(got[0], v0, atol=1e-13)
    np.testing.assert_allclose(got[1], v0, atol=1e-13)


def test_identical_keys_give_plain_mean():
    rng = np.random.default_rng(2)
    L, Hkv, D, P = 37, 1, 128, 16
    k = np.repeat(_rows(rng, 1, D, "outlier").reshape(1, 1, D), L, axis=0)
    v = _rows(rng, L, D, "heavy").reshape(L, 1, D)
    d = _build(rng, [L], 2, Hkv, D, P, True, False, 128, kv=(k, v))
    got = oracle.decode(d["q"], d["kc"], d["vc"], d["bt"], [L], 2, Hkv, D, d["num_pages"], P,
                        True, False, 128)
    c, s, z = _cache_rows(d["vc"], d["slots"], 0, Hkv, P, D)
    np.testing.assert_allclose(got[0], oracle.dequant_rows(c, s, z).mean(0), atol=1e-13)


def test_page_permutation_is_invisible():
    rng = np.random.default_rng(3)
    seq_lens = [33, 5]
    Hq, Hkv, D, P = 4, 2, 128, 16
    d = _build(rng, seq_lens, Hq, Hkv, D, P, True, True, 128, shuffle=False)
    base = oracle.decode(d["q"], d["kc"], d["vc"], d["bt"], seq_lens, Hq, Hkv, D, d["num_pages"],
                         P, True, True, 128)
    # move every page to a new physical id, copying its bytes, and remap
    perm = rng.permutation(d["num_pages"])
    chunk = P * D // 2 + 4 * P
    kc2, vc2 = np.zeros_like(d["kc"]), np.zeros_like(d["vc"])
    for old in range(d["num_pages"]):
        new = perm[old]
        src = slice(old * Hkv * chunk, (old + 1) * Hkv * chunk)
        dst = slice(new * Hkv * chunk, (new + 1) * Hkv * chunk)
        kc2[dst], vc2[dst] = d["kc"][src], d["vc"][src]
    bt2 = np.where(d["bt"] >= 0, perm[np.maximum(d["bt"], 0)], -1).astype(np.int32)
    moved = oracle.decode(d["q"], kc2, vc2, bt2, seq_lens, Hq, Hkv, D, d["num_pages"], P, True,
                          True, 128)
    np.testing.assert_array_equal(base, moved)


def test_empty_sequence_and_bad_page():
    rng = np.random.default_rng(4)
    Hq, Hkv, D, P = 2, 1, 128, 16
    d = _build(rng, [20], Hq, Hkv, D, P, True, True, 128)
    out = oracle.decode(d["q"], d["kc"], d["vc"], d["bt"], [0], Hq, Hkv, D, d["num_pages"], P,
                        True, True, 128)
    assert np.all(out == 0.0)
    bt = d["bt"].copy()
    bt[0, 1] = d["num_pages"] + 5
    with pytest.raises(RuntimeError):
        oracle.decode(d["q"], d["kc"], d["vc"], bt, [20], Hq, Hkv, D, d["num_pages"], P, True,
                      True, 128)


def test_gqa_heads_share_their_kv_head():
    """q-heads hq and hq' of the same group see the same keys: giving them
    the same query must give the same output; another group must differ."""
    rng = np.random.default_rng(5)
    Hq, Hkv, D, P = 4, 2, 128, 16
    d = _build(rng, [24], Hq, Hkv, D, P, True, False, 128)
    q = d["q"].copy()
    q[0, 1] = q[0, 0]
    q[0, 2] = q[0, 0]
    out = oracle.decode(q, d["kc"], d["vc"], d["bt"], [24], Hq, Hkv, D, d["num_pages"], P, True,
                        False, 128)
    np.testing.assert_array_equal(out[0], out[1])
    assert np.max(np.abs(out[0] - out[2])) > 1e-3
