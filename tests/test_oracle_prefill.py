"""Pins for the oracle's chunked-prefill attention over INT4 pages (CPU only).

Reading (the pages define attention only through decode): the query of the
token at position p of its sequence attends causally to cached tokens
0..p.  The oracle computes each row as a decode over the first p + 1
tokens; these tests compute the same thing a different way -- one dense,
un-paged, ORIGINAL-domain causal attention per sequence with scipy's
Hadamard and an explicit lower-triangular mask -- and check causality and
special cases.
"""
import math

import numpy as np
import pytest
import scipy.linalg
import scipy.special

import oracle
from test_oracle_attention import _build
from test_oracle_quantizer import _cache_rows, _rows, bits_to_f32


def _chunk_queries(rng, q_lens, Hq, D):
    T = sum(q_lens)
    q = _rows(rng, T * Hq, D, "normal").reshape(T, Hq, D)
    cu = np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)
    return q, cu


def _dense_causal(d, seq_lens, q, cu, Hq, Hkv, D, P, rotate_k, rotate_v, h, scale):
    """Original domain: dequantize every cached row, rotate it back with
    scipy's (1/sqrt h) H, and run masked softmax attention for the chunk."""
    R = np.zeros((D, D))
    Hh = scipy.linalg.hadamard(h) / math.sqrt(h)
    for b0 in range(0, D, h):
        R[b0:b0 + h, b0:b0 + h] = Hh
    G = Hq // Hkv
    out = np.zeros((q.shape[0], Hq, D))
    start = 0
    for b, L in enumerate(seq_lens):
        sl = d["slots"][start:start + L]
        start += L
        n = cu[b + 1] - cu[b]
        pos = np.arange(L - n, L)                      # positions of the chunk's queries
        mask = np.arange(L)[None, :] <= pos[:, None]   # [n, L] causal
        for hq in range(Hq):
            kvh = hq // G
            kh = oracle.dequant_rows(*_cache_rows(d["kc"], sl, kvh, Hkv, P, D))
            vh = oracle.dequant_rows(*_cache_rows(d["vc"], sl, kvh, Hkv, P, D))
            if rotate_k:
                kh = kh @ R
            if rotate_v:
                vh = vh @ R
            qq = bits_to_f32(q[cu[b]:cu[b + 1], hq]).astype(np.float64)   # [n, D]
            t = np.where(mask, scale * (qq @ kh.T), -np.inf)
            out[cu[b]:cu[b + 1], hq] = scipy.special.softmax(t, axis=1) @ vh
    return out


@pytest.mark.parametrize("rotate_k,rotate_v,h,P", [(True, True, 128, 16), (True, False, 128, 32),
                                                    (False, False, 128, 16), (True, True, 64, 64)])
def test_equals_dense_causal_attention(rotate_k, rotate_v, h, P):
    rng = np.random.default_rng(10 * h + P + int(rotate_v))
    seq_lens = [1, 40, 23, 70]
    q_lens = [1, 40, 7, 17]     # a whole prompt, a chunk after a prefix, a single token
    Hq, Hkv, D = 4, 2, 128
    d = _build(rng, seq_lens, Hq, Hkv, D, P, rotate_k, rotate_v, h)
    q, cu = _chunk_queries(rng, q_lens, Hq, D)
    got = oracle.prefill(q, cu, d["kc"], d["vc"], d["bt"], seq_lens, Hq, Hkv, D, d["num_pages"],
                         P, rotate_k, rotate_v, h).reshape(q.shape[0], Hq, D)
    ref = _dense_causal(d, seq_lens, q, cu, Hq, Hkv, D, P, rotate_k, rotate_v, h,
                        1 / math.sqrt(D))
    np.testing.assert_allclose(got, ref, atol=1e-12, rtol=1e-12)


def test_later_tokens_do_not_reach_earlier_queries():
    """Overwrite the cached K and V of the chunk's last 10 tokens: the outputs
    of the queries before them do not change by a single bit; the last
    query's does."""
    rng = np.random.default_rng(4)
    L, n, Hq, Hkv, D, P = 50, 30, 2, 1, 128, 16
    d = _build(rng, [L], Hq, Hkv, D, P, True, True, 128)
    q, cu = _chunk_queries(rng, [n], Hq, D)
    base = oracle.prefill(q, cu, d["kc"], d["vc"], d["bt"], [L], Hq, Hkv, D, d["num_pages"], P,
                          True, True, 128)
    k2 = _rows(rng, 10 * Hkv, D, "outlier").reshape(10, Hkv, D)
    v2 = _rows(rng, 10 * Hkv, D, "heavy").reshape(10, Hkv, D)
    assert oracle.quantize_append(k2, v2, d["slots"][L - 10:], Hkv, D, d["kc"], d["vc"],
                                  d["num_pages"], P, True, True, 128) == 0
    after = oracle.prefill(q, cu, d["kc"], d["vc"], d["bt"], [L], Hq, Hkv, D, d["num_pages"], P,
                           True, True, 128)
    first_changed = (n - 10) * Hq   # rows are (token, head), token-major
    np.testing.assert_array_equal(after[:first_changed], base[:first_changed])
    assert not np.array_equal(after[-Hq:], base[-Hq:])


def test_single_query_chunk_is_the_decode_and_position_zero_returns_v0():
    rng = np.random.default_rng(5)
    seq_lens = [33, 1]
    Hq, Hkv, D, P = 4, 2, 128, 16
    d = _build(rng, seq_lens, Hq, Hkv, D, P, True, True, 128)
    q, cu = _chunk_queries(rng, [1, 1], Hq, D)
    got = oracle.prefill(q, cu, d["kc"], d["vc"], d["bt"], seq_lens, Hq, Hkv, D, d["num_pages"],
                         P, True, True, 128)
    dec = oracle.decode(q, d["kc"], d["vc"], d["bt"], seq_lens, Hq, Hkv, D, d["num_pages"], P,
                        True, True, 128)
    np.testing.assert_array_equal(got, dec)
    # the second sequence's only query sits at position 0: softmax over one key
    Hh = scipy.linalg.hadamard(128) / math.sqrt(128)
    for hq in range(Hq):
        c, s, z = _cache_rows(d["vc"], d["slots"][33:34], hq // 2, Hkv, P, D)
        np.testing.assert_allclose(got[Hq + hq], oracle.dequant_rows(c, s, z)[0] @ Hh,
                                   atol=1e-13)


def test_row_selection_and_threads():
    rng = np.random.default_rng(6)
    seq_lens = [20, 45]
    Hq, Hkv, D, P = 8, 2, 128, 16
    d = _build(rng, seq_lens, Hq, Hkv, D, P, True, False, 128)
    q, cu = _chunk_queries(rng, [20, 12], Hq, D)
    full = oracle.prefill(q, cu, d["kc"], d["vc"], d["bt"], seq_lens, Hq, Hkv, D, d["num_pages"],
                          P, True, False, 128, threads=4)
    rows = [(0, 0), (19, 7), (20, 3), (31, 5)]
    some = oracle.prefill(q, cu, d["kc"], d["vc"], d["bt"], seq_lens, Hq, Hkv, D,
                          d["num_pages"], P, True, False, 128, rows=rows)
    for n, (i, hq) in enumerate(rows):
        np.testing.assert_array_equal(some[n], full[i * Hq + hq])
