"""CPU oracle for the SAW-INT4 hot path -- TEST INFRASTRUCTURE.

Plain, slow and independent of the CUDA library: it is the statement the GPU
path is checked against.  Only `tests/`, `__graft_entry__.smoke()` and the
benchmark's CPU-baseline leg may import it; the product path never does.

Every arithmetic step lives in `saw_oracle.c` (see its header for the pages
and sections each function follows); this module only marshals numpy arrays
through ctypes.  ctypes releases the GIL during a foreign call, so the
`threads=` arguments below run disjoint token / query ranges in parallel.

Parity pins: each function here is checked by `tests/test_oracle_*.py`
against closed forms, library routines, hand-worked fixtures and brute force.
End-to-end model accuracy (the pages' 73.78 vs 75.64 on Qwen3-4B) is parity
unpinned: it needs trained weights and evaluation datasets.
"""
from __future__ import annotations

import ctypes as C
import os
from concurrent.futures import ThreadPoolExecutor

import numpy as np

from . import build as _build

RN, RD, RU = 0, 1, 2

_lib = None


def load() -> C.CDLL:
    """Build (if needed) and load the oracle library."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.build()
    lib = C.CDLL(path)
    P = C.c_void_p
    i32, i64, f64 = C.c_int32, C.c_int64, C.c_double
    sig = {
        "oracle_f16_to_f64": (f64, [C.c_uint16]),
        "oracle_f32_to_f16": (C.c_uint16, [C.c_float, i32]),
        "oracle_f32_to_bf16": (C.c_uint16, [C.c_float, i32]),
        "oracle_sylvester": (i32, [i32, P]),
        "oracle_rotate_exact": (i32, [P, i32, i32, P]),
        "oracle_block_scale_f32": (C.c_float, [i32]),
        "oracle_rotate_canon": (i32, [P, i32, i32]),
        "oracle_quantize_row": (i32, [P, i32, i32, i32, i32, i32, P, P, P]),
        "oracle_dequant_row": (i32, [P, C.c_uint16, C.c_uint16, i32, i32, P]),
        "oracle_chunk_bytes": (i64, [i32, i32]),
        "oracle_cache_bytes": (i64, [i32, i32, i32, i32]),
        "oracle_quantize_append": (i64, [P, P, i64, i64, P, i32, i32, i32, i32, P, P, i32, i32,
                                         i32, i32, i32, i32, i32]),
        "oracle_decode_one": (i32, [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32, f64,
                                    P, i32, i32]),
        "oracle_prefill_one": (i32, [P, P, P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32,
                                     f64, P, i32, i32]),
        "oracle_bf16_cache_bytes": (i64, [i32, i32, i32, i32]),
        "oracle_bf16_append": (i64, [P, P, i64, i64, P, i32, i32, i32, i32, P, P, i32, i32]),
        "oracle_decode_bf16_one": (i32, [P, P, P, P, i32, i32, i32, i32, i32, i32, f64, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def _check(rc: int, what: str) -> None:
    if rc < 0:
        raise RuntimeError(f"oracle {what} failed with code {rc}")


# ---------------------------------------------------------------- formats

def f16_bits_to_f64(bits) -> np.ndarray:
    lib = load()
    b = np.asarray(bits, dtype=np.uint16)
    return np.array([lib.oracle_f16_to_f64(int(x)) for x in b.ravel()]).reshape(b.shape)


def f32_to_f16_bits(x, mode: int) -> np.ndarray:
    lib = load()
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_f32_to_f16(float(v), mode) for v in a.ravel()],
                    dtype=np.uint16).reshape(a.shape)


def f32_to_bf16_bits(x, mode: int) -> np.ndarray:
    lib = load()
    a = np.asarray(x, dtype=np.float32)
    return np.array([lib.oracle_f32_to_bf16(float(v), mode) for v in a.ravel()],
                    dtype=np.uint16).reshape(a.shape)


# ---------------------------------------------------------------- rotation

def sylvester(h: int) -> np.ndarray:
    H = np.zeros((h, h), dtype=np.int8)
    _check(load().oracle_sylvester(h, _ptr(H)), "sylvester")
    return H


def block_scale_f32(h: int) -> np.float32:
    return np.float32(load().oracle_block_scale_f32(h))


def rotate_exact(x, h: int) -> np.ndarray:
    """(R-exact) per-row block-diagonal (1/sqrt h) H x in float64; x is [..., D]."""
    a = np.ascontiguousarray(np.asarray(x, dtype=np.float64))
    D = a.shape[-1]
    flat = a.reshape(-1, D)
    out = np.empty_like(flat)
    lib = load()
    for r in range(flat.shape[0]):
        _check(lib.oracle_rotate_exact(_ptr(flat[r]), D, h, _ptr(out[r])), "rotate_exact")
    return out.reshape(a.shape)


def rotate_canon(x, h: int) -> np.ndarray:
    """(R-canon) the binary32 butterfly rotation; x is [..., D] float32."""
    a = np.array(x, dtype=np.float32, copy=True, order="C")
    D = a.shape[-1]
    flat = a.reshape(-1, D)
    lib = load()
    for r in range(flat.shape[0]):
        _check(lib.oracle_rotate_canon(_ptr(flat[r]), D, h), "rotate_canon")
    return flat.reshape(a.shape)


# ---------------------------------------------------------------- quantizer

def quantize_rows(x_bits, rotate: bool, h: int, in_f16: bool = False, meta_bf16: bool = False):
    """Quantize rows of bfloat16 (binary16 if in_f16) bit patterns [N, D] ->
    (codes [N, D/2] u8, s [N] u16, z [N] u16); s and z are binary16 bits, or
    bfloat16 bits if meta_bf16."""
    x = np.ascontiguousarray(np.asarray(x_bits, dtype=np.uint16))
    if x.ndim == 1:
        x = x[None]
    N, D = x.shape
    codes = np.zeros((N, D // 2), dtype=np.uint8)
    s = np.zeros(N, dtype=np.uint16)
    z = np.zeros(N, dtype=np.uint16)
    lib = load()
    for r in range(N):
        _check(lib.oracle_quantize_row(_ptr(x[r]), int(in_f16), D, int(rotate), h, int(meta_bf16),
                                       _ptr(codes[r]), s[r:].ctypes.data, z[r:].ctypes.data),
               "quantize_row")
    return codes, s, z


def dequant_rows(codes, s_bits, z_bits, meta_bf16: bool = False) -> np.ndarray:
    c = np.ascontiguousarray(np.asarray(codes, dtype=np.uint8))
    if c.ndim == 1:
        c = c[None]
    s_bits = np.atleast_1d(np.asarray(s_bits, dtype=np.uint16))
    z_bits = np.atleast_1d(np.asarray(z_bits, dtype=np.uint16))
    N, half = c.shape
    out = np.zeros((N, 2 * half), dtype=np.float64)
    lib = load()
    for r in range(N):
        _check(lib.oracle_dequant_row(_ptr(c[r]), int(s_bits[r]), int(z_bits[r]), int(meta_bf16),
                                      2 * half, _ptr(out[r])), "dequant_row")
    return out


# ---------------------------------------------------------------- paged cache

def chunk_bytes(page_size: int, head_dim: int) -> int:
    return int(load().oracle_chunk_bytes(page_size, head_dim))


def cache_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load().oracle_cache_bytes(num_pages, page_size, num_kv_heads, head_dim))


def _ranges(n: int, parts: int):
    parts = max(1, min(parts, n)) if n > 0 else 1
    step = -(-n // parts) if n > 0 else 0
    return [(b, min(n, b + step)) for b in range(0, n, step)] if n > 0 else []


def quantize_append(k_bits, v_bits, slot_mapping, num_kv_heads: int, head_dim: int,
                    k_cache: np.ndarray, v_cache, num_pages: int, page_size: int,
                    rotate_k: bool, rotate_v: bool, block_h: int, threads: int = 1,
                    in_f16: bool = False, meta_bf16: bool = False) -> int:
    """Quantize-append every token of k (and v) into the caches in place.

    k_bits / v_bits: uint16 [T, stride] (or [T, Hkv, D]) bfloat16 bit
    patterns (binary16 if in_f16); meta_bf16 stores the (scale, zero) pairs
    as bfloat16.
    Returns the number of out-of-range slots that were skipped.
    """
    k = np.ascontiguousarray(np.asarray(k_bits, dtype=np.uint16))
    T = k.shape[0]
    k2 = k.reshape(T, -1)
    v2 = None
    if v_bits is not None:
        v2 = np.ascontiguousarray(np.asarray(v_bits, dtype=np.uint16)).reshape(T, -1)
    slots = np.ascontiguousarray(np.asarray(slot_mapping, dtype=np.int32))
    assert slots.shape == (T,)
    assert k_cache.dtype == np.uint8 and k_cache.flags["C_CONTIGUOUS"]
    if v2 is not None:
        assert v_cache.dtype == np.uint8 and v_cache.flags["C_CONTIGUOUS"]
    lib = load()

    def run(rng):
        b, e = rng
        return lib.oracle_quantize_append(
            _ptr(k2), _ptr(v2) if v2 is not None else None, k2.shape[1],
            v2.shape[1] if v2 is not None else 0, _ptr(slots), b, e, num_kv_heads, head_dim,
            _ptr(k_cache), _ptr(v_cache) if v2 is not None else None, num_pages, page_size,
            int(rotate_k), int(rotate_v), block_h, int(in_f16), int(meta_bf16))

    rngs = _ranges(T, threads)
    if threads <= 1 or len(rngs) <= 1:
        res = [run(r) for r in rngs]
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            res = list(ex.map(run, rngs))
    for r in res:
        _check(r, "quantize_append")
    return int(sum(res))


def decode(q_bits, k_cache, v_cache, block_tables, seq_lens, num_q_heads: int,
           num_kv_heads: int, head_dim: int, num_pages: int, page_size: int, rotate_k: bool,
           rotate_v: bool, block_h: int, sm_scale: float | None = None, pairs=None,
           threads: int = 1, in_f16: bool = False, meta_bf16: bool = False) -> np.ndarray:
    """fp64 decode attention for the (seq, q_head) pairs given (default: all).

    q_bits: uint16 [B, Hq, D] bfloat16 bit patterns (binary16 if in_f16);
    meta_bf16: the caches hold bfloat16 (scale, zero) pairs.  The q-head -> kv-head map
    is contiguous groups: kv = q_head // (Hq / Hkv) (a reading; the pages do
    not say).  Returns float64 [len(pairs), D].
    """
    q = np.ascontiguousarray(np.asarray(q_bits, dtype=np.uint16))
    B = q.shape[0]
    q = q.reshape(B, num_q_heads, head_dim)
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    sl = np.asarray(seq_lens, dtype=np.int64)
    G = num_q_heads // num_kv_heads
    if sm_scale is None or sm_scale == 0.0:
        sm_scale = 1.0 / np.sqrt(head_dim)
    if pairs is None:
        pairs = [(b, hq) for b in range(B) for hq in range(num_q_heads)]
    pairs = list(pairs)
    out = np.zeros((len(pairs), head_dim), dtype=np.float64)
    lib = load()

    def run(i):
        b, hq = pairs[i]
        qrow = np.ascontiguousarray(q[b, hq])
        row = np.ascontiguousarray(bt[b]) if bt.ndim == 2 and bt.shape[1] > 0 else np.zeros(1, np.int32)
        o = np.zeros(head_dim, dtype=np.float64)
        rc = lib.oracle_decode_one(_ptr(qrow), _ptr(k_cache), _ptr(v_cache), _ptr(row),
                                   int(sl[b]), hq // G, num_kv_heads, head_dim, num_pages,
                                   page_size, int(rotate_k), int(rotate_v), block_h,
                                   float(sm_scale), _ptr(o), int(in_f16), int(meta_bf16))
        _check(rc, "decode_one")
        out[i] = o

    if threads <= 1 or len(pairs) <= 1:
        for i in range(len(pairs)):
            run(i)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(run, range(len(pairs))))
    return out


def prefill(q_bits, cu_q_lens, k_cache, v_cache, block_tables, seq_lens, num_q_heads: int,
            num_kv_heads: int, head_dim: int, num_pages: int, page_size: int, rotate_k: bool,
            rotate_v: bool, block_h: int, sm_scale: float | None = None, rows=None,
            threads: int = 1, in_f16: bool = False, meta_bf16: bool = False) -> np.ndarray:
    """fp64 chunked-prefill attention (causal) for the (query row, q_head)
    pairs given (default: all).

    q_bits: uint16 [T, Hq, D] bfloat16 (binary16 if in_f16; meta_bf16 as for
    decode), the query rows of every sequence's
    chunk, sequence after sequence; rows cu_q_lens[b] .. cu_q_lens[b+1] - 1
    belong to sequence b and are its last q_len = cu_q_lens[b+1] - cu_q_lens[b]
    tokens, so row i sits at position seq_lens[b] - q_len + (i - cu_q_lens[b]).
    Returns float64 [len(rows), D].
    """
    q = np.ascontiguousarray(np.asarray(q_bits, dtype=np.uint16))
    T = q.shape[0]
    q = q.reshape(T, num_q_heads, head_dim)
    cu = np.asarray(cu_q_lens, dtype=np.int64)
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    sl = np.asarray(seq_lens, dtype=np.int64)
    G = num_q_heads // num_kv_heads
    if sm_scale is None or sm_scale == 0.0:
        sm_scale = 1.0 / np.sqrt(head_dim)
    seq_of = np.zeros(T, dtype=np.int64)
    for b in range(len(cu) - 1):
        seq_of[cu[b]:cu[b + 1]] = b
    if rows is None:
        rows = [(i, hq) for i in range(T) for hq in range(num_q_heads)]
    rows = list(rows)
    out = np.zeros((len(rows), head_dim), dtype=np.float64)
    lib = load()

    def run(n):
        i, hq = rows[n]
        b = int(seq_of[i])
        pos = int(sl[b] - (cu[b + 1] - cu[b]) + (i - cu[b]))
        qrow = np.ascontiguousarray(q[i, hq])
        row = np.ascontiguousarray(bt[b])
        o = np.zeros(head_dim, dtype=np.float64)
        rc = lib.oracle_prefill_one(_ptr(qrow), _ptr(k_cache), _ptr(v_cache), _ptr(row), pos,
                                    hq // G, num_kv_heads, head_dim, num_pages, page_size,
                                    int(rotate_k), int(rotate_v), block_h, float(sm_scale),
                                    _ptr(o), int(in_f16), int(meta_bf16))
        _check(rc, "prefill_one")
        out[n] = o

    if threads <= 1 or len(rows) <= 1:
        for n in range(len(rows)):
            run(n)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(run, range(len(rows))))
    return out


# ---------------------------------------------------------------- BF16 baseline

def bf16_cache_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(load().oracle_bf16_cache_bytes(num_pages, page_size, num_kv_heads, head_dim))


def bf16_append(k_bits, v_bits, slot_mapping, num_kv_heads: int, head_dim: int,
                k_cache: np.ndarray, v_cache, num_pages: int, page_size: int) -> int:
    """Copy every token's bf16 rows into its slot of the BF16 caches (uint16
    arrays) in place; returns the number of out-of-range slots skipped."""
    k = np.ascontiguousarray(np.asarray(k_bits, dtype=np.uint16))
    T = k.shape[0]
    if T == 0:
        return 0
    k2 = k.reshape(T, -1)
    v2 = None
    if v_bits is not None:
        v2 = np.ascontiguousarray(np.asarray(v_bits, dtype=np.uint16)).reshape(T, -1)
    slots = np.ascontiguousarray(np.asarray(slot_mapping, dtype=np.int32))
    assert slots.shape == (T,)
    assert k_cache.dtype == np.uint16 and k_cache.flags["C_CONTIGUOUS"]
    rc = load().oracle_bf16_append(_ptr(k2), _ptr(v2) if v2 is not None else None, k2.shape[1],
                                   v2.shape[1] if v2 is not None else 0, _ptr(slots), 0, T,
                                   num_kv_heads, head_dim, _ptr(k_cache),
                                   _ptr(v_cache) if v2 is not None else None, num_pages,
                                   page_size)
    _check(rc, "bf16_append")
    return int(rc)


def decode_bf16(q_bits, k_cache, v_cache, block_tables, seq_lens, num_q_heads: int,
                num_kv_heads: int, head_dim: int, num_pages: int, page_size: int,
                sm_scale: float | None = None, pairs=None, threads: int = 1) -> np.ndarray:
    """fp64 decode attention over BF16 pages for the (seq, q_head) pairs given
    (default: all); same q-head -> kv-head map as `decode`."""
    q = np.ascontiguousarray(np.asarray(q_bits, dtype=np.uint16))
    B = q.shape[0]
    q = q.reshape(B, num_q_heads, head_dim)
    bt = np.ascontiguousarray(np.asarray(block_tables, dtype=np.int32))
    sl = np.asarray(seq_lens, dtype=np.int64)
    G = num_q_heads // num_kv_heads
    if sm_scale is None or sm_scale == 0.0:
        sm_scale = 1.0 / np.sqrt(head_dim)
    if pairs is None:
        pairs = [(b, hq) for b in range(B) for hq in range(num_q_heads)]
    pairs = list(pairs)
    out = np.zeros((len(pairs), head_dim), dtype=np.float64)
    lib = load()

    def run(i):
        b, hq = pairs[i]
        qrow = np.ascontiguousarray(q[b, hq])
        row = np.ascontiguousarray(bt[b]) if bt.ndim == 2 and bt.shape[1] > 0 else np.zeros(1, np.int32)
        o = np.zeros(head_dim, dtype=np.float64)
        rc = lib.oracle_decode_bf16_one(_ptr(qrow), _ptr(k_cache), _ptr(v_cache), _ptr(row),
                                        int(sl[b]), hq // G, num_kv_heads, head_dim, num_pages,
                                        page_size, float(sm_scale), _ptr(o))
        _check(rc, "decode_bf16_one")
        out[i] = o

    if threads <= 1 or len(pairs) <= 1:
        for i in range(len(pairs)):
            run(i)
    else:
        with ThreadPoolExecutor(max_workers=threads) as ex:
            list(ex.map(run, range(len(pairs))))
    return out


def host_threads() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)
