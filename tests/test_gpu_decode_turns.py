"""GPU parity of the decode's check-free path against the oracle's float64
attention: the whole-tile turns of a warp's ring (two steps of two tiles
with four stages, three single-tile steps with the three stages of
head_dim 256), the tiles left to the checked step after them, a warp whose
tile list is longer than the shared-memory list it keeps (checked refills
for the whole split), a skipped page (a warp that is not clean), and the
4-warp CTA shape (decode and fused step).

Bar: max |o_gpu - o_ref| / max |o_ref| <= 2e-3.  Pages: gist.science s.2
point 3 (dequantization fused into decoding); youngju.dev "The Rotation
Trick" (q.k = Hq.Hk, output rotated back)."""
import numpy as np
import pytest
import torch

import bit_paged_kv_gb300 as saw
from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import ATTN_TOL, fill_layer, gpu_decode, oracle_decode, rel_err

pytestmark = pytest.mark.gpu

# Tokens per warp turn: 16-token tiles, 16 or 8 warps per CTA.  Lengths that
# give a warp 4, 5-6, 8, 9-10 and 12-13 tiles (16-warp CTAs; twice as many
# with 8 warps), with and without a ragged last tile.
TURN_LENS = [16 * 16 * 4, 16 * 16 * 4 + 1, 16 * (16 * 5 + 3) + 7, 16 * 16 * 8 - 1,
             16 * (16 * 9 + 15), 16 * (16 * 12 + 8) + 9]


def _setup(wl, lens, spare=5):
    lens = torch.tensor(lens, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=spare)
    kc, vc, _, _, _ = fill_layer(wl, 0, lens, bt, npages)
    q = W.q_rows(wl, 0, "cuda", num_seqs=len(lens))
    return lens, bt, npages, kc, vc, q


def _check(wl, lens, bt, npages, kc, vc, q, pps, label):
    out, st = gpu_decode(q, kc, vc, bt.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                         wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                         pages_per_split=pps)
    assert st == 0
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads, npages,
                        wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h)
    got = out.cpu().numpy().reshape(-1, wl.head_dim)
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, label)
    assert err <= ATTN_TOL, f"relative error {err:.3e}"


@pytest.mark.parametrize("D,group", [(128, 4), (128, 8), (256, 4), (256, 8), (64, 2)])
@pytest.mark.parametrize("rot", [(True, True), (True, False)])
def test_turn_boundaries(D, group, rot):
    """Every sequence in one split (each warp runs its whole tiles in turns
    of the ring, then the checked tail), and the automatic plan (short
    splits of a few tiles per warp)."""
    wl = W.TINY.variant(head_dim=D, block_h=min(D, 128), num_kv_heads=2, num_q_heads=2 * group,
                        rotate_k=rot[0], rotate_v=rot[1], shuffle_pages=True,
                        dist="student_t", nu=4)
    lens, bt, npages, kc, vc, q = _setup(wl, TURN_LENS)
    one_split = int(bt.shape[1])
    for pps in (one_split, 0):
        _check(wl, lens, bt, npages, kc, vc, q, pps, f"turns-D{D}-G{group}-rot{rot}-pps{pps}")


@pytest.mark.parametrize("D,tiles", [(128, 260), (256, 70)])
def test_tile_list_longer_than_kept(D, tiles):
    """One split whose warps own more tiles than the chunk indices a warp
    keeps in shared memory (256 at head_dim <= 128, 64 at 256): every refill
    takes the checked path and reads the block table for the tiles beyond
    the list."""
    wl = W.TINY.variant(head_dim=D, block_h=128, num_kv_heads=2, num_q_heads=8,
                        shuffle_pages=True)
    L = 16 * 16 * tiles + 5  # more than `tiles` tiles per warp even with 16-warp CTAs
    lens, bt, npages, kc, vc, q = _setup(wl, [L, 1000])
    _check(wl, lens, bt, npages, kc, vc, q, int(bt.shape[1]), f"long-list-D{D}")


@pytest.mark.parametrize("group", [4, 8])
def test_skipped_page_leaves_the_rest_exact(group):
    """A bad page id in the middle of a long sequence is reported and its 16
    tokens are left out; the output equals the oracle's attention over the
    sequence without that page (attention does not depend on where a token
    sits), and the other sequence is untouched."""
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=2 * group, shuffle_pages=True)
    lens, bt, npages, kc, vc, q = _setup(wl, [3000, 4000])
    bad_lp = 40
    bt_bad = bt.clone()
    bt_bad[1, bad_lp] = npages + 7
    for pps in (int(bt.shape[1]), 0):
        out, st = gpu_decode(q, kc, vc, bt_bad.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                             wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                             pages_per_split=pps)
        assert st == saw.SAW_ERR_DEVICE_INDEX
        # sequence 1 without its page bad_lp: the later pages move up one entry
        bt_ref = bt.clone()
        row = bt[1].tolist()
        kept = row[:bad_lp] + row[bad_lp + 1:] + [-1]
        bt_ref[1] = torch.tensor(kept, dtype=torch.int32)
        lens_ref = lens.clone()
        lens_ref[1] -= wl.page_size
        ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt_ref, lens_ref,
                            wl.num_kv_heads, npages, wl.page_size, wl.rotate_k, wl.rotate_v,
                            wl.block_h)
        got = out.cpu().numpy().reshape(-1, wl.head_dim)
        assert np.all(np.isfinite(got))
        err = rel_err(got, ref, f"skipped-page-G{group}-pps{pps}")
        assert err <= ATTN_TOL, f"relative error {err:.3e}"


def _four_warp_lens(seed, n=320, hi=4096):
    """Lengths for a grid of 4-warp CTAs: 320 sequences x 2 kv-heads = 640
    (sequence, kv-head) units, more than four per SM, none longer than one
    4096-token split."""
    g = torch.Generator().manual_seed(seed)
    return [0, 1, 16, 17, hi] + torch.randint(1, hi + 1, (n - 5,), generator=g).tolist()


@pytest.mark.parametrize("group", [4, 8])
def test_many_units_one_split_four_warp_ctas(group):
    """Hundreds of unsplit (sequence, kv-head) units: the plan serves them
    with 4-warp CTAs, four per SM."""
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=2 * group, shuffle_pages=True,
                        dist="student_t", nu=4)
    lens, bt, npages, kc, vc, q = _setup(wl, _four_warp_lens(group))
    splits, _ = saw.saw_decode_plan(len(lens), wl.num_kv_heads, wl.page_size, int(lens.max()), 0)
    assert splits == 1
    _check(wl, lens, bt, npages, kc, vc, q, 0, f"four-warp-G{group}")


@pytest.mark.parametrize("group,flags", [(8, 1), (4, 0)])
def test_fused_step_four_warp_ctas(group, flags):
    """The fused decode step on the same grid: cache bytes equal the
    oracle's append of each sequence's new token, attention the oracle's."""
    from gpu_helpers import assert_bytes_equal, oracle_append
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=2 * group, shuffle_pages=True,
                        rotate_v=bool(flags), dist="student_t", nu=4)
    lens_l = _four_warp_lens(10 + group)
    lens = torch.tensor(lens_l, dtype=torch.int32)
    P = wl.page_size
    bt, npages = W.page_tables(wl, lens, spare_pages=3)
    kc, vc, k_pre, v_pre, slots_pre = fill_layer(wl, 0, lens, bt, npages,
                                                 upto=lambda n: max(n - 1, 0))
    B, D = len(lens_l), wl.head_dim
    knew = (torch.randn(B, wl.num_kv_heads, D, device="cuda") * 2).to(torch.bfloat16)
    vnew = (torch.randn(B, wl.num_kv_heads, D, device="cuda") * 2).to(torch.bfloat16)
    q = W.q_rows(wl, 0, "cuda", num_seqs=B)
    Lmax = int(lens.max())
    out = torch.full((B, wl.num_q_heads, D), float("nan"), dtype=torch.float32, device="cuda")
    wsb = saw.saw_decode_workspace_bytes(B, wl.num_q_heads, wl.num_kv_heads, D, P, Lmax, 0)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_decode_step(q, knew, vnew, kc, vc, bt.cuda(), lens.cuda(), Lmax, wl.num_kv_heads,
                        npages, P, wl.rotate_k, wl.rotate_v, wl.block_h, out, ws, flags=flags,
                        dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kr, vr, _ = oracle_append(k_pre, v_pre, slots_pre.cpu(), npages, P, wl.rotate_k, wl.rotate_v,
                              wl.block_h)
    keep = [b for b in range(B) if lens_l[b] > 0]
    slots_new = torch.tensor([int(bt[b, (lens_l[b] - 1) // P]) * P + (lens_l[b] - 1) % P
                              for b in keep], dtype=torch.int32)
    oracle_append(knew[keep], vnew[keep], slots_new, npages, P, wl.rotate_k, wl.rotate_v,
                  wl.block_h, kc=kr, vc=vr)
    assert_bytes_equal(kc, kr, "K cache after the step")
    assert_bytes_equal(vc, vr, "V cache after the step")
    ref = oracle_decode(q, kr, vr, bt, lens, wl.num_kv_heads, npages, P, wl.rotate_k, wl.rotate_v,
                        wl.block_h)
    got = out.cpu().numpy().reshape(-1, D)
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"four-warp-step-G{group}-flags{flags}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"
