"""Parity of the fused decode step (saw_decode_step: append the step's token,
then attend, one launch per layer) in the launch configuration the benchmark
times, and where the new token's tile meets a reused ring slot.

1. The Qwen3-4B-shaped latency case at full size: batch 1, context 32768,
   K-only rotation, the automatic split plan, SAW_STEP_EARLY_PAGES, three
   layers (first, second, last) back to back in one CUDA graph, replayed
   twice.  Before each replay the caches are put back to their pre-step
   bytes, so every replay's append is checked: every byte of each layer's K
   and V cache against the oracle's append, and all 32 q-heads against the
   oracle's float64 attention (max |o_gpu - o_ref| / max |o_ref| <= 2e-3).
2. Small pages and forced split sizes chosen so that the tile holding the
   new token is consumed from a ring slot that has already been reused, both
   as the second tile of a two-tile step and as a tile of its own; the
   helper below recomputes the kernel's tile-to-warp mapping and the test
   asserts both situations occur.

Pages: youngju.dev "INT4 KV-cache quantization", "The System Is the Design --
A Fused Kernel" (the new token is rotated, quantized and appended to the
paged cache on the decode path); gist.science "SAW-INT4", s.2 point 3
(quantization fused into decoding).
"""
import numpy as np
import pytest
import torch

import bit_paged_kv_gb300 as saw
from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import (ATTN_TOL, assert_bytes_equal, fill_layer, oracle_append, oracle_decode,
                         rel_err)

pytestmark = pytest.mark.gpu

STEP_TOKENS = 16     # tokens per tile of the decode kernel
RING_STAGES = 4      # tiles in flight per warp
LONG_SPLIT = 8192    # splits longer than this many tokens use 16-warp CTAs


def _capture(fn, stream):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        fn()  # outside the capture first: kernel attributes are set here
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        fn()
    torch.cuda.synchronize()
    return g


def test_latency_step_full_size_graph():
    wl = W.QWEN3_4B_LATENCY
    layers = [0, 1, wl.num_layers - 1]
    lens = W.seq_lens(wl)
    L = int(lens[0])
    bt, npages = W.page_tables(wl, lens)
    btd, lensd = bt.cuda(), lens.cuda()
    B, Hq, Hkv, D, P = wl.num_seqs, wl.num_q_heads, wl.num_kv_heads, wl.head_dim, wl.page_size
    splits, pps = saw.saw_decode_plan(B, Hkv, P, L, 0)
    assert splits > 1 and pps * P < L  # several splits: the merge runs
    per = {}
    for layer in layers:
        kc, vc, kpre, vpre, spre = fill_layer(wl, layer, lens, bt, npages, upto=lambda n: n - 1)
        knew = W.kv_rows(wl, layer, W.K, 1, "cuda", token_offset=L - 1)
        vnew = W.kv_rows(wl, layer, W.V, 1, "cuda", token_offset=L - 1)
        snew = W.slots_for(btd, P, 0, L - 1, L)
        kr, vr, bad = oracle_append(kpre, vpre, spre.cpu(), npages, P, wl.rotate_k, wl.rotate_v,
                                    wl.block_h)
        assert bad == 0
        oracle_append(knew, vnew, snew.cpu(), npages, P, wl.rotate_k, wl.rotate_v, wl.block_h,
                      kc=kr, vc=vr)
        q = W.q_rows(wl, layer, "cuda")
        ref = oracle_decode(q, kr, vr, bt, lens, Hkv, npages, P, wl.rotate_k, wl.rotate_v,
                            wl.block_h)
        per[layer] = dict(kc=kc, vc=vc, kc0=kc.clone(), vc0=vc.clone(), knew=knew, vnew=vnew,
                          q=q, kr=kr, vr=vr, ref=ref,
                          out=torch.empty(B, Hq, D, dtype=torch.float32, device="cuda"))
        del kpre, vpre
    wsb = saw.saw_decode_workspace_bytes(B, Hq, Hkv, D, P, L, 0)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")

    def step():
        for layer in layers:
            x = per[layer]
            saw.saw_decode_step(x["q"], x["knew"], x["vnew"], x["kc"], x["vc"], btd, lensd, L,
                                Hkv, npages, P, wl.rotate_k, wl.rotate_v, wl.block_h, x["out"],
                                ws, flags=saw.SAW_STEP_EARLY_PAGES, dev_status=status)

    stream = torch.cuda.Stream()
    graph = _capture(step, stream)
    for replay in range(2):
        for layer in layers:
            x = per[layer]
            x["kc"].copy_(x["kc0"])
            x["vc"].copy_(x["vc0"])
            x["out"].fill_(float("nan"))
        status.zero_()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for layer in layers:
            x = per[layer]
            assert_bytes_equal(x["kc"], x["kr"], f"replay {replay} layer {layer} K")
            assert_bytes_equal(x["vc"], x["vr"], f"replay {replay} layer {layer} V")
            got = x["out"].cpu().numpy().reshape(-1, D)
            assert np.all(np.isfinite(got))
            err = rel_err(got, x["ref"], f"latency-step-graph-L{layer}")
            print(f"replay {replay} layer {layer}: {splits} splits x {pps} pages, rel err {err:.3e}")
            assert err <= ATTN_TOL, f"replay {replay} layer {layer}: relative error {err:.3e}"
    # the merge left its counters at zero for the next call
    n_counters = 2 * B * Hkv
    assert torch.all(ws[:4 * n_counters].view(torch.int32) == 0)


def _new_token_roles(lens, P, pps, num_kv_heads, sms):
    """For each sequence, where the kernel consumes the tile that holds the
    new token (position seq_len - 1): (i, role) with i the warp's own tile
    index and role 'second' (second tile of a two-tile step), 'first' or
    'single'.  Mirrors the decode kernel: split s covers pages
    [s*pps, (s+1)*pps); its 16-token tiles go to warps round-robin (warp w
    takes tiles w, w+W, ...) and a warp consumes its tiles two at a time,
    the last one alone when it has an odd count."""
    max_pages = max((int(L) + P - 1) // P for L in lens)
    splits = -(-max_pages // pps)
    units = len(lens) * num_kv_heads
    warps = 16 if (units * splits <= sms or pps * P > LONG_SPLIT) else 8
    out = []
    for L in lens:
        L = int(L)
        if L == 0:
            continue
        n_pages = (L + P - 1) // P
        page = (L - 1) // P
        s = page // pps
        p_begin, p_end = s * pps, min(n_pages, (s + 1) * pps)
        n_steps = (p_end - p_begin) * (P // STEP_TOKENS)
        t = ((L - 1) - p_begin * P) // STEP_TOKENS
        w, i = t % warps, t // warps
        n_my = -(-(n_steps - w) // warps)
        if i == n_my - 1 and n_my % 2 == 1:
            role = "single"
        else:
            role = "second" if i % 2 == 1 else "first"
        out.append((i, role))
    return out, warps


@pytest.mark.parametrize("P,pps,group,flags,many", [
    (16, 128, 4, 0, False), (16, 128, 8, 1, False), (64, 32, 4, 1, False),
    (64, 32, 2, 0, False), (16, 64, 4, 1, True), (32, 48, 8, 0, True)])
def test_step_new_token_in_reused_ring_slot(P, pps, group, flags, many):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    Hkv = 2
    wl = W.TINY.variant(page_size=P, num_q_heads=Hkv * group, num_kv_heads=Hkv,
                        shuffle_pages=True, rotate_v=False, dist="student_t", nu=4)
    split_tokens = pps * P
    # the new token's tile t in its split: the warp's tile index is t // W
    lens_l = [1, 17, 16 * (16 * 5 + 3) + 9, 16 * (16 * 4 + 7) + 5, 16 * (16 * 7) + 1,
              16 * (16 * 6 + 9) + 16, split_tokens + 16 * (16 * 5 + 2) + 8,
              2 * split_tokens + 16 * (8 * 5 + 1) + 3, 16 * (8 * 4 + 3) + 2, 16 * (8 * 7) + 7]
    if many:
        g = torch.Generator().manual_seed(P * 31 + group)
        lens_l = lens_l + torch.randint(1, 3 * split_tokens, (80,), generator=g).tolist()
    roles, warps = _new_token_roles(lens_l, P, pps, Hkv, sms)
    reused = [(i, r) for i, r in roles if i >= RING_STAGES]
    assert any(r == "second" for _, r in reused), (warps, roles)
    assert any(r != "second" for _, r in reused), (warps, roles)

    lens = torch.tensor(lens_l, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=3)
    kc, vc, k_pre, v_pre, slots_pre = fill_layer(wl, 0, lens, bt, npages,
                                                 upto=lambda n: max(n - 1, 0))
    B, D = len(lens_l), wl.head_dim
    knew = (torch.randn(B, Hkv, D, device="cuda") * 2).to(torch.bfloat16)
    vnew = (torch.randn(B, Hkv, D, device="cuda") * 2).to(torch.bfloat16)
    q = W.q_rows(wl, 0, "cuda", num_seqs=B)
    Lmax = int(lens.max())
    out = torch.full((B, wl.num_q_heads, D), float("nan"), dtype=torch.float32, device="cuda")
    wsb = saw.saw_decode_workspace_bytes(B, wl.num_q_heads, Hkv, D, P, Lmax, pps)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_decode_step(q, knew, vnew, kc, vc, bt.cuda(), lens.cuda(), Lmax, Hkv, npages, P,
                        wl.rotate_k, wl.rotate_v, wl.block_h, out, ws, pages_per_split=pps,
                        flags=flags, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kr, vr, _ = oracle_append(k_pre, v_pre, slots_pre.cpu(), npages, P, wl.rotate_k, wl.rotate_v,
                              wl.block_h)
    slots_new = torch.tensor([int(bt[b, (L - 1) // P]) * P + (L - 1) % P
                              for b, L in enumerate(lens_l)], dtype=torch.int32)
    oracle_append(knew, vnew, slots_new, npages, P, wl.rotate_k, wl.rotate_v, wl.block_h,
                  kc=kr, vc=vr)
    assert_bytes_equal(kc, kr, "K cache after the step")
    assert_bytes_equal(vc, vr, "V cache after the step")
    ref = oracle_decode(q, kr, vr, bt, lens, Hkv, npages, P, wl.rotate_k, wl.rotate_v,
                        wl.block_h)
    got = out.cpu().numpy().reshape(-1, D)
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"step-ring-P{P}-pps{pps}-G{group}-W{warps}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"
