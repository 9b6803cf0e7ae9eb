"""GPU parity of the fused rotate + INT4 quantize-append kernel (through the
C-ABI) against the oracle: every byte of both caches must match, including
the untouched sentinel bytes.  Pages: youngju.dev "The System Is the Design
-- A Fused Kernel"; gist.science s.2 (token-wise INT4, block-diagonal
rotation, fused kernel)."""
import numpy as np
import pytest
import torch

import bit_paged_kv_gb300 as saw
from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import assert_bytes_equal, gpu_append, oracle_append

pytestmark = pytest.mark.gpu


def _inputs(wl, T, device="cuda", layer=0):
    k = W.kv_rows(wl, layer, W.K, T, device)
    v = W.kv_rows(wl, layer, W.V, T, device)
    return k, v


@pytest.mark.parametrize("rotate_k,rotate_v,h", [(1, 1, 128), (1, 0, 128), (0, 0, 128),
                                                  (0, 1, 128), (1, 1, 64), (1, 1, 32),
                                                  (1, 1, 16)])
def test_tiny_all_tokens(rotate_k, rotate_v, h):
    """Config 'tiny': 4 sequences x 256 tokens, 2 kv-heads, every token."""
    wl = W.TINY
    lens = W.seq_lens(wl)
    bt, npages = W.page_tables(wl, lens, spare_pages=3)
    slots = W.prefill_slots(bt.cuda(), lens.tolist(), wl.page_size)
    k, v = _inputs(wl, int(lens.sum()))
    kc, vc, st = gpu_append(k, v, slots, npages, wl.page_size, rotate_k, rotate_v, h)
    kr, vr, bad = oracle_append(k, v, slots, npages, wl.page_size, rotate_k, rotate_v, h)
    assert st == 0 and bad == 0
    assert_bytes_equal(kc, kr, "K cache")
    assert_bytes_equal(vc, vr, "V cache")


@pytest.mark.parametrize("size", ["warp", "tiled"])
@pytest.mark.parametrize("P", [16, 32, 64])
@pytest.mark.parametrize("hkv", [1, 3, 8])
def test_ragged_strided_shuffled(P, hkv, size):
    """Row counts that are not a multiple of the CTA tile, a strided token
    dimension, scattered slots and padding entries -- on the warp-per-row
    kernel (77 tokens) and on the tiled kernel (above 4096 rows, with a
    ragged last tile)."""
    wl = W.TINY.variant(num_kv_heads=hkv, page_size=P, dist="student_t", nu=3)
    T = 77 if size == "warp" else 4096 // hkv + 333
    num_pages = -(-T // P) + 5
    g = torch.Generator().manual_seed(P * 10 + hkv)
    slots = torch.randperm(num_pages * P, generator=g)[:T].to(torch.int32)
    slots[[3, 40, 76]] = -1
    big_k = W.kv_rows(wl, 0, W.K, T, "cuda")
    big_v = W.kv_rows(wl, 0, W.V, T, "cuda")
    # strided views: token stride of (hkv + 2) * 128 elements
    kpad = torch.zeros(T, hkv + 2, 128, dtype=torch.bfloat16, device="cuda")
    vpad = torch.zeros(T, hkv + 2, 128, dtype=torch.bfloat16, device="cuda")
    kpad[:, 1:hkv + 1] = big_k
    vpad[:, 1:hkv + 1] = big_v
    k, v = kpad[:, 1:hkv + 1], vpad[:, 1:hkv + 1]
    assert k.stride(0) == (hkv + 2) * 128
    kc, vc, st = gpu_append(k, v, slots.cuda(), num_pages, P, True, False, 128)
    kr, vr, bad = oracle_append(big_k, big_v, slots, num_pages, P, True, False, 128)
    assert st == 0 and bad == 0
    assert_bytes_equal(kc, kr, "K cache")
    assert_bytes_equal(vc, vr, "V cache")


@pytest.mark.parametrize("T", [40, 5000, 160000], ids=["warp", "tiled", "tiled-many-per-warp"])
def test_k_only_and_bad_slots(T):
    """K only; a slot one past the end and a negative slot are reported and
    skipped, padding (-1) is skipped silently, every other row is stored.
    At 160000 tokens every warp of the tiled kernel takes several row tiles,
    so its K-only ring wraps."""
    wl = W.TINY
    P = 16
    num_pages = -(-T // P)
    k, _ = _inputs(wl, T)
    slots = torch.arange(T, dtype=torch.int32)
    slots[5] = num_pages * P       # one past the end
    slots[9] = -2                  # negative, not padding
    slots[11] = -1                 # padding
    kc, vc, st = gpu_append(k, None, slots.cuda(), num_pages, P, True, True, 128)
    kr, _, bad = oracle_append(k, None, slots, num_pages, P, True, True, 128)
    assert vc is None
    assert st == saw.SAW_ERR_DEVICE_INDEX and bad == 2
    assert_bytes_equal(kc, kr, "K cache")


@pytest.mark.parametrize("repeat", [1, 1024], ids=["warp-per-row", "row-per-thread"])
def test_special_rows(repeat):
    """Constant rows, all-zero rows with negative zeros, one-hot rows, and
    magnitudes at the edges of binary16 (subnormal zero-points, saturating
    scales).  Few rows take the warp-per-row kernel; tiled to 9216 rows they
    take the row-per-thread kernel."""
    D, hkv = 128, 1
    rows = []
    rows.append(torch.full((D,), 1.5))
    z = torch.zeros(D)
    z[::3] = -0.0
    rows.append(z)
    oh = torch.zeros(D)
    oh[5] = 1.0
    rows.append(oh)
    rows.append(torch.full((D,), 1e-6))
    rows.append(torch.linspace(-3e-7, 5e-7, D))
    rows.append(torch.linspace(-1e5, 2e5, D))          # range / 15 above binary16 max
    rows.append(torch.linspace(-7e4, -6.9e4, D))       # min below -65504
    rows.append(torch.linspace(-0.5, 0.5, D) + 300.0)  # large bias, tiny spread
    g = torch.Generator().manual_seed(0)
    rows.append(torch.randn(D, generator=g) * 1e-3)
    x = torch.stack(rows).to(torch.bfloat16).view(-1, hkv, D).repeat(repeat, 1, 1)
    T = x.shape[0]
    slots = torch.arange(T, dtype=torch.int32)
    pages = -(-T // 16)
    for rot in (0, 1):
        k = x.cuda()
        kc, vc, st = gpu_append(k, k, slots.cuda(), pages, 16, rot, rot, 128)
        kr, vr, bad = oracle_append(x, x, slots, pages, 16, rot, rot, 128)
        assert st == 0
        assert_bytes_equal(kc, kr, f"K cache rot={rot}")
        assert_bytes_equal(vc, vr, f"V cache rot={rot}")


def test_append_order_and_batching_do_not_matter():
    """Token-wise independence on the GPU: one call vs token-by-token calls
    in reverse order give identical caches."""
    wl = W.TINY
    T, num_pages, P = 48, 4, 16
    k, v = _inputs(wl, T)
    slots = torch.randperm(num_pages * P, generator=torch.Generator().manual_seed(1))[:T]
    slots = slots.to(torch.int32).cuda()
    kc, vc, _ = gpu_append(k, v, slots, num_pages, P, True, True, 128)
    from gpu_helpers import new_caches
    kc2, vc2 = new_caches(num_pages, P, wl.num_kv_heads, 128)
    for t in reversed(range(T)):
        gpu_append(k[t:t + 1], v[t:t + 1], slots[t:t + 1], num_pages, P, True, True, 128,
                   kc=kc2, vc=vc2)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2)


def test_empty_append_is_a_no_op():
    kc = torch.full((1088,), 7, dtype=torch.uint8, device="cuda")
    k = torch.zeros(0, 1, 128, dtype=torch.bfloat16, device="cuda")
    s = torch.zeros(0, dtype=torch.int32, device="cuda")
    saw.saw_quantize_append(k, None, s, kc, None, 1, 16, True, False, 128)
    torch.cuda.synchronize()
    assert torch.all(kc == 7)


@pytest.mark.parametrize("h", [16, 32, 64, 128])
@pytest.mark.parametrize("rotate_k,rotate_v", [(1, 1), (1, 0), (0, 1)])
def test_tiled_block_sizes(h, rotate_k, rotate_v):
    """Every block size on the tiled kernel (3000 tokens x 2 kv-heads, a
    ragged last tile), with each tensor rotated or not."""
    wl = W.TINY.variant(dist="student_t", nu=4)
    T = 3000
    k, v = _inputs(wl, T)
    num_pages = -(-T // 16) + 1
    slots = torch.randperm(num_pages * 16, generator=torch.Generator().manual_seed(h))[:T]
    slots = slots.to(torch.int32)
    kc, vc, st = gpu_append(k, v, slots.cuda(), num_pages, 16, rotate_k, rotate_v, h)
    kr, vr, bad = oracle_append(k, v, slots, num_pages, 16, rotate_k, rotate_v, h)
    assert st == 0 and bad == 0
    assert_bytes_equal(kc, kr, "K cache")
    assert_bytes_equal(vc, vr, "V cache")


@pytest.mark.parametrize("T", [1, 3, 511, 512, 513, 3000])
def test_both_kernels_across_the_size_switch(T):
    """Appends just below, at and above the warp-per-row size limit (4096 rows)
    with 8 kv-heads: every size must give the oracle's bytes."""
    wl = W.TINY.variant(num_kv_heads=8, dist="student_t", nu=3)
    k, v = _inputs(wl, T)
    num_pages = -(-T // 16) + 2
    slots = torch.randperm(num_pages * 16, generator=torch.Generator().manual_seed(T))[:T]
    slots = slots.to(torch.int32)
    kc, vc, st = gpu_append(k, v, slots.cuda(), num_pages, 16, True, False, 128)
    kr, vr, bad = oracle_append(k, v, slots, num_pages, 16, True, False, 128)
    assert st == 0 and bad == 0
    assert_bytes_equal(kc, kr, "K cache")
    assert_bytes_equal(vc, vr, "V cache")
