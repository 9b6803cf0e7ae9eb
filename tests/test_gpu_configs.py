"""Parity at the full sizes of the five workloads, in the launch
configuration the benchmark times (automatic split plan).

Append: every byte of the sampled layers' caches against the oracle.
Decode: max |o_gpu - o_ref| / max |o_ref| <= 2e-3 per layer on sampled
(sequence, q-head) rows that the oracle computes one by one.
Workload shapes: gist.science s.3 point 4 (Qwen3-4B/8B/32B) and s.4
(h = 128, K-only rotation); the distributions stand in for the outlier
channels youngju.dev "Why Naive INT4 Breaks" describes.
"""
import numpy as np
import pytest
import torch

from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import (ATTN_TOL, assert_bytes_equal, bits, fill_layer, gpu_append, gpu_decode,
                         oracle_append, oracle_decode, rel_err)

import oracle

pytestmark = pytest.mark.gpu


def _append_parity(wl, layer, lens, bt, npages, kc, vc, k, v, slots, extra=None):
    kr, vr, bad = oracle_append(k, v, slots, npages, wl.page_size, wl.rotate_k, wl.rotate_v,
                                wl.block_h)
    assert bad == 0
    if extra is not None:
        k1, v1, s1 = extra
        oracle_append(k1, v1, s1, npages, wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                      kc=kr, vc=vr)
    assert_bytes_equal(kc, kr, f"{wl.name} layer {layer} K")
    assert_bytes_equal(vc, vr, f"{wl.name} layer {layer} V")
    return kr, vr


def _decode_parity(wl, layer, lens, bt, npages, kc, vc, kr, vr, pairs):
    q = W.q_rows(wl, layer, "cuda")
    out, st = gpu_decode(q, kc, vc, bt.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                         wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h)
    assert st == 0
    ref = oracle_decode(q, kr, vr, bt, lens, wl.num_kv_heads, npages, wl.page_size, wl.rotate_k,
                        wl.rotate_v, wl.block_h, pairs=pairs)
    got = out.cpu().numpy()[[b for b, _ in pairs], [h for _, h in pairs]]
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"{wl.name}-L{layer}-rk{int(wl.rotate_k)}rv{int(wl.rotate_v)}-h{wl.block_h}")
    row_err = max(rel_err(got[i], ref[i], "row") for i in range(len(pairs)))
    print(f"{wl.name} layer {layer}: rel err {err:.3e} (worst row {row_err:.3e})")
    assert err <= ATTN_TOL, f"{wl.name} layer {layer}: relative error {err:.3e}"


def _sample_seqs(wl, n):
    g = torch.Generator().manual_seed(wl.seed * 7 + 1)
    return sorted(torch.randperm(wl.num_seqs, generator=g)[:n].tolist())


def test_qwen3_4b_latency_all_layers():
    """Config 2: 36 layers, batch 1, context 32768, K-only rotation; prefill
    32767 tokens, append the step's token, decode.  Append bytes on every
    layer; attention on the first and last."""
    wl = W.QWEN3_4B_LATENCY
    lens = W.seq_lens(wl)
    bt, npages = W.page_tables(wl, lens)
    L = int(lens[0])
    for layer in range(wl.num_layers):
        kc, vc, k, v, slots = fill_layer(wl, layer, lens, bt, npages, upto=lambda n: n - 1)
        k1 = W.kv_rows(wl, layer, W.K, 1, "cuda", token_offset=L - 1)
        v1 = W.kv_rows(wl, layer, W.V, 1, "cuda", token_offset=L - 1)
        s1 = W.slots_for(bt.cuda(), wl.page_size, 0, L - 1, L)
        gpu_append(k1, v1, s1, npages, wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                   kc=kc, vc=vc)
        kr, vr = _append_parity(wl, layer, lens, bt, npages, kc, vc, k, v, slots,
                                extra=(k1, v1, s1))
        if layer in (0, wl.num_layers - 1):
            pairs = [(0, h) for h in range(wl.num_q_heads)]
            _decode_parity(wl, layer, lens, bt, npages, kc, vc, kr, vr, pairs)


@pytest.mark.parametrize("wl", [W.QWEN3_8B_CONCURRENT, W.QWEN3_32B_HIGH_CONCURRENCY],
                         ids=lambda w: w.name)
def test_concurrent_first_and_last_layer(wl):
    """Configs 3 and 4: full-layer append bytes and attention on 16 seeded
    sequences (all their q-heads) for the first and last layer."""
    lens = W.seq_lens(wl)
    bt, npages = W.page_tables(wl, lens)
    seqs = _sample_seqs(wl, 16)
    pairs = [(b, h) for b in seqs for h in range(wl.num_q_heads)]
    for layer in (0, wl.num_layers - 1):
        kc, vc, k, v, slots = fill_layer(wl, layer, lens, bt, npages)
        kr, vr = _append_parity(wl, layer, lens, bt, npages, kc, vc, k, v, slots)
        del k, v
        _decode_parity(wl, layer, lens, bt, npages, kc, vc, kr, vr, pairs)


@pytest.mark.parametrize("rot", [(True, False), (False, False)], ids=["k-only", "unrotated"])
def test_qwen3_32b_rotation_variants(rot):
    """Config 4's K-only and unrotated INT4 variants (K+V is covered above),
    first layer."""
    wl = W.QWEN3_32B_HIGH_CONCURRENCY.variant(rotate_k=rot[0], rotate_v=rot[1])
    lens = W.seq_lens(wl)
    bt, npages = W.page_tables(wl, lens)
    seqs = _sample_seqs(wl, 8)
    pairs = [(b, h) for b in seqs for h in range(wl.num_q_heads)]
    kc, vc, k, v, slots = fill_layer(wl, 0, lens, bt, npages)
    kr, vr = _append_parity(wl, 0, lens, bt, npages, kc, vc, k, v, slots)
    del k, v
    _decode_parity(wl, 0, lens, bt, npages, kc, vc, kr, vr, pairs)


@pytest.mark.parametrize("h", [128, 64])
def test_long_prefill_and_decode(h):
    """Config 5: bulk append of 131072-token chunks for 8 sequences (page 64),
    then decode at context 131072, all sequences and q-heads."""
    wl = W.LONG_PREFILL.variant(block_h=h)
    lens = W.seq_lens(wl)
    bt, npages = W.page_tables(wl, lens)
    kc, vc, k, v, slots = fill_layer(wl, 0, lens, bt, npages)
    kr, vr = _append_parity(wl, 0, lens, bt, npages, kc, vc, k, v, slots)
    del k, v
    pairs = [(b, hq) for b in range(wl.num_seqs) for hq in range(wl.num_q_heads)]
    _decode_parity(wl, 0, lens, bt, npages, kc, vc, kr, vr, pairs)
