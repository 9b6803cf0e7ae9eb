"""GPU parity of the paged INT4 decode attention (through the C-ABI) against
the oracle's float64 attention on the same cache bytes.

Bar: max |o_gpu - o_ref| / max |o_ref| <= 2e-3.  Pages: gist.science s.2
point 3 (dequantization fused into decoding); youngju.dev "The Rotation
Trick" (q.k = Hq.Hk, output rotated back)."""
import numpy as np
import pytest
import torch

import bit_paged_kv_gb300 as saw
from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import (ATTN_TOL, fill_layer, gpu_append, gpu_decode, new_caches,
                         oracle_decode, rel_err)

pytestmark = pytest.mark.gpu


def _setup(wl, lens, spare=5):
    lens = torch.tensor(lens, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=spare)
    kc, vc, _, _, _ = fill_layer(wl, 0, lens, bt, npages)
    q = W.q_rows(wl, 0, "cuda", num_seqs=len(lens))
    return lens, bt, npages, kc, vc, q


def _check(wl, lens, bt, npages, kc, vc, q, pps=0, pairs=None, max_seq_len=None):
    out, st = gpu_decode(q, kc, vc, bt.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                         wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                         max_seq_len=max_seq_len, pages_per_split=pps)
    assert st == 0
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads, npages,
                        wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h, pairs=pairs)
    got = out.cpu().numpy().reshape(-1, wl.head_dim)
    if pairs is not None:
        got = np.stack([out[b, h].cpu().numpy() for b, h in pairs])
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"{wl.name}-G{wl.group}-P{wl.page_size}-h{wl.block_h}-pps{pps}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"
    return err


@pytest.mark.parametrize("pps", [0, 1, 3, 100])
def test_tiny_full(pps):
    """Config 'tiny' in full: 4 seqs x 256 tokens, GQA 2, K and V rotated."""
    wl = W.TINY
    lens, bt, npages, kc, vc, q = _setup(wl, W.seq_lens(wl).tolist())
    _check(wl, lens, bt, npages, kc, vc, q, pps=pps)


EDGE_LENS = [0, 1, 15, 16, 17, 33, 255, 700]


@pytest.mark.parametrize("group", [1, 4, 8])
@pytest.mark.parametrize("P", [16, 32, 64])
def test_many_sequences_eight_warp_ctas(group, P):
    """100 sequences x 2 kv-heads of short, mixed lengths: a grid of several
    waves of short splits, which the plan serves with 8-warp CTAs, two per SM
    (automatic plan and a forced split size)."""
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=2 * group, page_size=P, shuffle_pages=True,
                        dist="student_t", nu=4)
    g = torch.Generator().manual_seed(7 * P + group)
    lens_l = EDGE_LENS + torch.randint(1, 700, (92,), generator=g).tolist()
    lens, bt, npages, kc, vc, q = _setup(wl, lens_l)
    for pps in (0, 2):
        _check(wl, lens, bt, npages, kc, vc, q, pps=pps)


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("rot", [(1, 1), (1, 0), (0, 0), (0, 1)])
def test_edge_lengths_groups_rotations(group, rot):
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=2 * group, rotate_k=bool(rot[0]),
                        rotate_v=bool(rot[1]), shuffle_pages=True, dist="student_t", nu=4)
    lens, bt, npages, kc, vc, q = _setup(wl, EDGE_LENS)
    _check(wl, lens, bt, npages, kc, vc, q, pps=0)
    _check(wl, lens, bt, npages, kc, vc, q, pps=2)


@pytest.mark.parametrize("P", [32, 64])
@pytest.mark.parametrize("h", [128, 64, 16])
def test_page_sizes_and_blocks(P, h):
    wl = W.TINY.variant(page_size=P, block_h=h, num_q_heads=8, num_kv_heads=2,
                        shuffle_pages=True)
    lens, bt, npages, kc, vc, q = _setup(wl, [1, P - 1, P, P + 1, 5 * P + 3, 1000])
    _check(wl, lens, bt, npages, kc, vc, q, pps=0)
    _check(wl, lens, bt, npages, kc, vc, q, pps=1)


def test_max_seq_len_bound_and_lengths_below_it():
    """A plan made for a larger max_seq_len than any sequence uses."""
    wl = W.TINY.variant(shuffle_pages=True)
    lens, bt, npages, kc, vc, q = _setup(wl, [40, 300, 7, 256])
    bt_wide = torch.full((bt.shape[0], 200), -1, dtype=torch.int32)
    bt_wide[:, :bt.shape[1]] = bt
    _check(wl, lens, bt_wide, npages, kc, vc, q, pps=0, max_seq_len=200 * 16)


def test_bad_page_and_bad_length_are_reported():
    wl = W.TINY
    lens, bt, npages, kc, vc, q = _setup(wl, [64, 64])
    bt_bad = bt.clone()
    bt_bad[0, 1] = npages + 10
    out, st = gpu_decode(q, kc, vc, bt_bad.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                         wl.page_size, True, True, 128)
    assert st == saw.SAW_ERR_DEVICE_INDEX
    assert torch.all(torch.isfinite(out[1]))
    lens_bad = torch.tensor([64, 5000], dtype=torch.int32)
    out, st = gpu_decode(q, kc, vc, bt.cuda(), lens_bad.cuda(), wl.num_kv_heads, npages,
                         wl.page_size, True, True, 128, max_seq_len=64)
    assert st == saw.SAW_ERR_DEVICE_INDEX
    assert torch.all(out[1] == 0)


def test_explicit_sm_scale():
    wl = W.TINY
    lens, bt, npages, kc, vc, q = _setup(wl, [100, 31])
    out, st = gpu_decode(q, kc, vc, bt.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                         wl.page_size, True, True, 128, sm_scale=0.3)
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads,
                        npages, wl.page_size, True, True, 128, sm_scale=0.3)
    assert st == 0
    assert rel_err(out.cpu().numpy().reshape(-1, 128), ref, "tiny-sm_scale-0.3") <= ATTN_TOL


def test_rotation_mismatch_is_detectable():
    """Decoding with rotation flags that differ from the append's gives a
    clearly wrong answer (the caller's contract)."""
    wl = W.TINY
    lens, bt, npages, kc, vc, q = _setup(wl, [256])
    good = _check(wl, lens, bt, npages, kc, vc, q)
    out, _ = gpu_decode(q, kc, vc, bt.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                        wl.page_size, True, False, 128)
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads, npages,
                        wl.page_size, True, True, 128)
    assert rel_err(out.cpu().numpy().reshape(-1, 128), ref, "mismatch") > 50 * max(good, 1e-5)


def test_decode_after_single_token_append():
    """The decode step: append one token per sequence, then attend including it."""
    wl = W.TINY.variant(num_seqs=3)
    lens0 = [31, 64, 100]
    lens, bt, npages, kc, vc, q = _setup(wl, [L + 1 for L in lens0], spare=2)
    # overwrite the last token of every sequence through a one-token append
    knew = torch.randn(3, wl.num_kv_heads, 128, device="cuda").to(torch.bfloat16) * 3
    vnew = torch.randn(3, wl.num_kv_heads, 128, device="cuda").to(torch.bfloat16) * 3
    slots = torch.stack([W.slots_for(bt, wl.page_size, b, L, L + 1)[0]
                         for b, L in enumerate(lens0)]).to(torch.int32).cuda()
    gpu_append(knew, vnew, slots, npages, wl.page_size, True, True, 128, kc=kc, vc=vc)
    _check(wl, lens, bt, npages, kc, vc, q)


def test_workspace_reuse_across_calls_and_plans():
    """One zero-filled workspace serves many calls with different split plans:
    the merge's counters are back at zero after every call."""
    wl = W.TINY.variant(shuffle_pages=True)
    lens, bt, npages, kc, vc, q = _setup(wl, [300, 47, 128, 256])
    B, Hq, D = q.shape
    Lmax = int(lens.max())
    wsb = max(saw.saw_decode_workspace_bytes(B, Hq, wl.num_kv_heads, D, wl.page_size, Lmax, p)
              for p in (1, 2, 3))
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads, npages,
                        wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h)
    for pps in (1, 2, 3, 1, 3):
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        saw.saw_paged_decode_int4(q, kc, vc, bt.cuda(), lens.cuda(), Lmax, wl.num_kv_heads,
                                  npages, wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                                  out, ws, pages_per_split=pps, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        assert rel_err(out.cpu().numpy().reshape(-1, 128), ref, f"tiny-ws-reuse-pps{pps}") <= ATTN_TOL
    n_counters = 2 * B * wl.num_kv_heads
    assert torch.all(ws[:4 * n_counters].view(torch.int32) == 0)


@pytest.mark.parametrize("P,group,pps,flags,many", [
    (16, 4, 0, 0, False), (16, 4, 2, 1, False), (16, 1, 3, 0, False), (16, 8, 1, 1, False),
    (32, 4, 1, 0, False), (64, 2, 1, 1, False), (64, 8, 0, 0, False),
    (16, 4, 0, 1, True), (16, 8, 2, 0, True), (64, 1, 0, 1, True)])
def test_fused_decode_step(P, group, pps, flags, many):
    """saw_decode_step = append the new token at seq_len - 1, then attend, in
    one launch: cache bytes equal the oracle's append, attention the oracle's.
    many = 100 sequences: several waves of short splits, 8-warp CTAs."""
    from gpu_helpers import new_caches, oracle_append
    wl = W.TINY.variant(page_size=P, num_q_heads=2 * group, num_kv_heads=2, shuffle_pages=True,
                        rotate_v=False, dist="student_t", nu=4)
    lens_l = [1, 17, 16, P + 1, 300, 31, 0]
    if many:
        g = torch.Generator().manual_seed(P + group)
        lens_l = lens_l + torch.randint(1, 400, (93,), generator=g).tolist()
    lens = torch.tensor(lens_l, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=3)
    # prefill all but the last token, with the append kernel
    kc, vc, k_pre, v_pre, slots_pre = fill_layer(wl, 0, lens, bt, npages,
                                                 upto=lambda n: max(n - 1, 0))
    B, D = len(lens_l), 128
    knew = (torch.randn(B, wl.num_kv_heads, D, device="cuda") * 2).to(torch.bfloat16)
    vnew = (torch.randn(B, wl.num_kv_heads, D, device="cuda") * 2).to(torch.bfloat16)
    q = W.q_rows(wl, 0, "cuda", num_seqs=B)
    Lmax = int(lens.max())
    out = torch.full((B, wl.num_q_heads, D), float("nan"), dtype=torch.float32, device="cuda")
    wsb = saw.saw_decode_workspace_bytes(B, wl.num_q_heads, wl.num_kv_heads, D, P, Lmax, pps)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_decode_step(q, knew, vnew, kc, vc, bt.cuda(), lens.cuda(), Lmax, wl.num_kv_heads,
                        npages, P, wl.rotate_k, wl.rotate_v, wl.block_h, out, ws,
                        pages_per_split=pps, flags=flags, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    # oracle: same prefill, then append the new token of each non-empty sequence
    kr, vr, _ = oracle_append(k_pre, v_pre, slots_pre.cpu(), npages, P, wl.rotate_k, wl.rotate_v,
                              wl.block_h)
    keep = [b for b in range(B) if lens_l[b] > 0]
    slots_new = torch.tensor([int(bt[b, (lens_l[b] - 1) // P]) * P + (lens_l[b] - 1) % P
                              for b in keep], dtype=torch.int32)
    oracle_append(knew[keep], vnew[keep], slots_new, npages, P, wl.rotate_k, wl.rotate_v,
                  wl.block_h, kc=kr, vc=vr)
    from gpu_helpers import assert_bytes_equal
    assert_bytes_equal(kc, kr, "K cache after the step")
    assert_bytes_equal(vc, vr, "V cache after the step")
    ref = oracle_decode(q, kr, vr, bt, lens, wl.num_kv_heads, npages, P, wl.rotate_k, wl.rotate_v,
                        wl.block_h)
    got = out.cpu().numpy().reshape(-1, D)
    assert np.all(np.isfinite(got))
    assert rel_err(got, ref, f"step-P{P}-G{group}-pps{pps}{'-many' if many else ''}") <= ATTN_TOL


def test_merge_wait_times_out_and_reports():
    """Failure detection without a fault: the 'published' counter words of a
    workspace are set to a value no call reaches, so the merging split's
    bounded wait runs out (about a second).  The call returns, reports
    SAW_ERR_DEVICE_TIMEOUT, writes finite numbers, and a clean workspace
    works again afterwards on the same context."""
    import time
    wl = W.TINY
    lens, bt, npages, kc, vc, q = _setup(wl, [256, 200])
    B, Hq, D = q.shape
    Lmax = int(lens.max())
    pps = 2
    splits, _ = saw.saw_decode_plan(B, wl.num_kv_heads, wl.page_size, Lmax, pps)
    assert splits > 1
    wsb = saw.saw_decode_workspace_bytes(B, Hq, wl.num_kv_heads, D, wl.page_size, Lmax, pps)
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    counters = ws[:8 * B * wl.num_kv_heads].view(torch.int32).view(-1, 2)
    counters[:, 1] = 0x40000000  # 'published': never equals a split count
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.time()
    saw.saw_paged_decode_int4(q, kc, vc, bt.cuda(), lens.cuda(), Lmax, wl.num_kv_heads, npages,
                              wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h, out, ws,
                              pages_per_split=pps, dev_status=st)
    torch.cuda.synchronize()
    assert time.time() - t0 < 30.0
    assert int(st.item()) == saw.SAW_ERR_DEVICE_TIMEOUT
    assert torch.all(torch.isfinite(out))
    # the context is still usable: a clean workspace gives the right answer
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads, npages,
                        wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h)
    ws.zero_()
    st.zero_()
    saw.saw_paged_decode_int4(q, kc, vc, bt.cuda(), lens.cuda(), Lmax, wl.num_kv_heads, npages,
                              wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h, out, ws,
                              pages_per_split=pps, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert rel_err(out.cpu().numpy().reshape(-1, 128), ref, "tiny-after-timeout") <= ATTN_TOL
