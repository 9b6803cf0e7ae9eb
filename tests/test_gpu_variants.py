"""GPU parity at head_dim 64 and 256 (rotation blocks up to h = 256): the
variant append writes the oracle's bytes, and the variant decode matches the
oracle's float64 attention within the decode's bar.

Pages: youngju.dev "The Rotation Trick -- Block-Diagonal Hadamard" (blocks
of h), "Why Naive INT4 Breaks" (one scale per token); gist.science s.2."""
import numpy as np
import pytest
import torch

import bit_paged_kv_gb300 as saw
from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import (ATTN_TOL, assert_bytes_equal, fill_layer, gpu_append, gpu_decode,
                         oracle_append, oracle_decode, rel_err)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("D,h", [(64, 64), (64, 32), (64, 16), (256, 256), (256, 128),
                                 (256, 32)])
@pytest.mark.parametrize("rot", [(True, True), (True, False), (False, False)])
def test_append_bytes(D, h, rot):
    wl = W.TINY.variant(head_dim=D, block_h=h, num_kv_heads=4, dist="student_t", nu=3)
    T, P, pages = 300, 16, 24
    k = W.kv_rows(wl, 0, W.K, T, "cuda")
    v = W.kv_rows(wl, 0, W.V, T, "cuda")
    perm = torch.randperm(pages * P, generator=torch.Generator().manual_seed(D + h))[:T]
    slots = perm.to(torch.int32)
    slots[3] = -1
    kc, vc, st = gpu_append(k, v, slots.cuda(), pages, P, rot[0], rot[1], h)
    assert st == 0
    kr, vr, bad = oracle_append(k, v, slots, pages, P, rot[0], rot[1], h)
    assert bad == 0
    assert_bytes_equal(kc, kr, f"K D{D} h{h}")
    assert_bytes_equal(vc, vr, f"V D{D} h{h}")


@pytest.mark.parametrize("D,h", [(64, 64), (64, 32), (64, 16), (256, 256), (256, 128),
                                 (256, 64), (256, 32), (256, 16)])
@pytest.mark.parametrize("rot", [(True, True), (True, False), (False, True), (False, False)])
@pytest.mark.parametrize("fmt", ["bf16", "f16", "bf16-meta"])
def test_append_bytes_bulk(D, h, rot, fmt):
    """Bulk appends at head_dim 64 and 256 (above 4096 rows: the tiled
    kernels, one thread per row at 64 and four per row at 256, where the
    stride-64 and stride-128 steps cross threads): 2501 tokens x 4 kv-heads,
    a ragged last tile, one skipped slot, every byte against the oracle, for
    each tensor rotated or not, both input formats and both metadata
    formats."""
    wl = W.TINY.variant(head_dim=D, block_h=h, num_kv_heads=4, dist="student_t", nu=3)
    T, P, pages = 2501, 16, 170
    dt = torch.float16 if fmt == "f16" else torch.bfloat16
    meta_bf16 = fmt == "bf16-meta"
    k = W.kv_rows(wl, 0, W.K, T, "cuda", dtype=dt)
    v = W.kv_rows(wl, 0, W.V, T, "cuda", dtype=dt)
    perm = torch.randperm(pages * P, generator=torch.Generator().manual_seed(h + T))[:T]
    slots = perm.to(torch.int32)
    slots[5] = -1
    kc, vc, st = gpu_append(k, v, slots.cuda(), pages, P, rot[0], rot[1], h, meta_bf16=meta_bf16)
    assert st == 0
    kr, vr, bad = oracle_append(k, v, slots, pages, P, rot[0], rot[1], h, meta_bf16=meta_bf16)
    assert bad == 0
    assert_bytes_equal(kc, kr, f"K D{D} bulk h{h} {fmt}")
    assert_bytes_equal(vc, vr, f"V D{D} bulk h{h} {fmt}")


@pytest.mark.parametrize("D", [64, 256])
def test_append_bulk_strided_k_only_and_bad_slot(D):
    h, P, pages, Hkv = D, 64, 60, 2
    wl = W.TINY.variant(head_dim=D, block_h=h, num_kv_heads=Hkv)
    T = 3000  # 6000 rows: the tiled kernel
    raw = W.kv_rows(wl.variant(num_kv_heads=2 * Hkv), 0, W.K, T, "cuda")  # [T, 2 Hkv, D]
    k = raw[:, :Hkv]                                                      # token stride 2 Hkv D
    slots = torch.randperm(pages * P, generator=torch.Generator().manual_seed(3))[:T].to(torch.int32)
    slots[7] = pages * P
    kc, _, st = gpu_append(k, None, slots.cuda(), pages, P, True, False, h)
    assert st == saw.SAW_ERR_DEVICE_INDEX
    kr, _, bad = oracle_append(k.contiguous(), None, slots, pages, P, True, False, h)
    assert bad == 1
    assert_bytes_equal(kc, kr, f"K strided D{D} bulk")


def test_append_strided_k_only_and_bad_slot():
    D, h, P, pages, Hkv = 256, 256, 32, 8, 2
    wl = W.TINY.variant(head_dim=D, block_h=h, num_kv_heads=Hkv)
    T = 100
    raw = W.kv_rows(wl.variant(num_kv_heads=2 * Hkv), 0, W.K, T, "cuda")  # [T, 2 Hkv, D]
    k = raw[:, :Hkv]                                                      # token stride 2 Hkv D
    slots = torch.randperm(pages * P, generator=torch.Generator().manual_seed(1))[:T].to(torch.int32)
    slots[7] = pages * P
    kc, _, st = gpu_append(k, None, slots.cuda(), pages, P, True, False, h)
    assert st == saw.SAW_ERR_DEVICE_INDEX
    kr, _, bad = oracle_append(k.contiguous(), None, slots, pages, P, True, False, h)
    assert bad == 1
    assert_bytes_equal(kc, kr, "K strided D256")


def _setup(wl, lens_l, spare=3):
    lens = torch.tensor(lens_l, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=spare)
    kc, vc, _, _, _ = fill_layer(wl, 0, lens, bt, npages)
    q = W.q_rows(wl, 0, "cuda", num_seqs=len(lens_l))
    return lens, bt, npages, kc, vc, q


def _check(wl, lens, bt, npages, kc, vc, q, label, pps=0, pairs=None, sm_scale=0.0):
    out, st = gpu_decode(q, kc, vc, bt.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                         wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                         pages_per_split=pps, sm_scale=sm_scale)
    assert st == 0
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads, npages,
                        wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h, pairs=pairs,
                        sm_scale=sm_scale or None)
    if pairs is None:
        got = out.cpu().numpy().reshape(-1, wl.head_dim)
    else:
        got = np.stack([out[b, h].cpu().numpy() for b, h in pairs])
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"var-{label}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"


EDGE = [0, 1, 31, 32, 33, 100, 700, 2500]


@pytest.mark.parametrize("D,h", [(64, 64), (64, 16), (256, 256), (256, 64)])
@pytest.mark.parametrize("group", [1, 4, 8])
@pytest.mark.parametrize("P", [16, 64])
def test_decode_edges(D, h, group, P):
    wl = W.TINY.variant(head_dim=D, block_h=h, num_kv_heads=2, num_q_heads=2 * group,
                        page_size=P, shuffle_pages=True, dist="student_t", nu=4)
    lens, bt, npages, kc, vc, q = _setup(wl, EDGE)
    _check(wl, lens, bt, npages, kc, vc, q, f"D{D}-h{h}-G{group}-P{P}")
    _check(wl, lens, bt, npages, kc, vc, q, f"D{D}-h{h}-G{group}-P{P}-pps3", pps=3)


PAIR_LENS = [0, 1, 15, 16, 17, 33, 100, 511, 700, 1024, 2047, 2500]


@pytest.mark.parametrize("D", [64])
@pytest.mark.parametrize("case", ["one-split", "splits"])
@pytest.mark.parametrize("rot,h", [((1, 1), 64), ((1, 0), 32), ((0, 0), 64), ((0, 1), 16)])
@pytest.mark.parametrize("fmt", ["bf16", "f16", "bf16-meta"])
def test_decode_kv_head_pairs(D, case, rot, h, fmt):
    """head_dim 64 at GQA 4 with many CTAs: each CTA serves two
    neighbouring kv-heads as one head of twice the head_dim (8 q-head
    columns, each q zero in the other kv-head's half).  80 sequences (one
    split each) or 40 sequences up to ~12000 tokens (several splits, the
    merge, partial rows twice as wide); lengths 0, 1, page edges and ragged
    tails; every output against the oracle."""
    dt = torch.float16 if fmt == "f16" else torch.bfloat16
    meta_bf16 = fmt == "bf16-meta"
    wl = W.QWEN3_8B_CONCURRENT.variant(head_dim=D, block_h=h, rotate_k=bool(rot[0]),
                                       rotate_v=bool(rot[1]), dist="student_t", nu=4)
    if case == "one-split":
        lens_l = (PAIR_LENS * 7)[:80]
    else:
        g = torch.Generator().manual_seed(h + rot[0])
        lens_l = PAIR_LENS + torch.randint(3000, 12000, (28,), generator=g).tolist()
    B, Hq, Hkv, P = len(lens_l), wl.num_q_heads, wl.num_kv_heads, wl.page_size
    assert Hq == 4 * Hkv and P == 16
    lens = torch.tensor(lens_l, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=3)
    kc, vc, _, _, _ = fill_layer(wl, 0, lens, bt, npages, dtype=dt, meta_bf16=meta_bf16)
    q = W.q_rows(wl, 0, "cuda", num_seqs=B, dtype=dt)
    Lmax = max(lens_l)
    splits, _ = saw.saw_decode_plan(B, Hkv, P, Lmax, 0)
    if case == "splits":
        # the pair form is on: its partial rows are 2 D floats wide
        rows = B * Hq * splits
        assert splits > 1
        assert saw.saw_decode_workspace_bytes(B, Hq, Hkv, D, P, Lmax, 0) == \
            (B * Hkv * 8 + 15) // 16 * 16 + rows * 2 * D * 4 + rows * 2 * 4
    out, st = gpu_decode(q, kc, vc, bt.cuda(), lens.cuda(), Hkv, npages, P, wl.rotate_k,
                         wl.rotate_v, h, meta_bf16=meta_bf16)
    assert st == 0
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, Hkv, npages, P,
                        wl.rotate_k, wl.rotate_v, h, meta_bf16=meta_bf16)
    got = out.cpu().numpy().reshape(-1, D)
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"var-D{D}-pairs-{case}-rot{rot[0]}{rot[1]}-h{h}-{fmt}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"


@pytest.mark.parametrize("D", [64, 256])
@pytest.mark.parametrize("rot", [(1, 0), (0, 0), (0, 1)])
def test_decode_rotation_variants(D, rot):
    wl = W.TINY.variant(head_dim=D, block_h=D, num_kv_heads=2, num_q_heads=8, page_size=32,
                        rotate_k=bool(rot[0]), rotate_v=bool(rot[1]), shuffle_pages=True)
    lens, bt, npages, kc, vc, q = _setup(wl, [1, 77, 300, 1500])
    _check(wl, lens, bt, npages, kc, vc, q, f"D{D}-rot{rot[0]}{rot[1]}", sm_scale=0.2)


@pytest.mark.parametrize("D", [64, 256])
def test_decode_long_context_all_heads(D):
    """1 sequence x 32768 tokens, Hq 32, Hkv 8, page 16, K-only rotation: the
    latency shape at the other head sizes (many splits, one merge)."""
    wl = W.QWEN3_4B_LATENCY.variant(head_dim=D, block_h=min(D, 128))
    lens, bt, npages, kc, vc, q = _setup(wl, [32768], spare=0)
    pairs = [(0, h) for h in range(0, 32, 3)]
    _check(wl, lens, bt, npages, kc, vc, q, f"D{D}-32k", pairs=pairs)


def test_noalloc_and_workspace_reuse_at_head_dim_64():
    wl = W.TINY.variant(head_dim=64, block_h=64, num_q_heads=8, shuffle_pages=True)
    lens, bt, npages, kc, vc, q = _setup(wl, [900, 40, 2000])
    B, Hq, D = q.shape
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads, npages,
                        16, True, True, 64)
    for _ in range(2):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        saw.saw_paged_decode_int4_noalloc(q, kc, vc, bt.cuda(), lens.cuda(), 2000,
                                          wl.num_kv_heads, npages, 16, True, True, 64, out,
                                          pages_per_split=8, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert rel_err(out.cpu().numpy().reshape(-1, D), ref, "var-noalloc-D64") <= ATTN_TOL


def test_fused_step_and_prefill_stay_head_dim_128():
    wl = W.TINY.variant(head_dim=64, block_h=64)
    lens, bt, npages, kc, vc, q = _setup(wl, [40, 40, 40, 40])
    B, Hq, D = q.shape
    knew = torch.zeros(B, wl.num_kv_heads, D, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(B, Hq, D, dtype=torch.float32, device="cuda")
    with pytest.raises(saw.SawError) as e:
        saw.saw_decode_step(q, knew, knew, kc, vc, bt.cuda(), lens.cuda(), 40, wl.num_kv_heads,
                            npages, 16, True, True, 64, out)
    assert e.value.status == saw.SAW_ERR_UNSUPPORTED
