"""GPU parity of the BF16 paged-KV baseline (through the C-ABI) against the
oracle: the append is a placement and must match byte for byte; the decode
is compared with the oracle's float64 attention over the same cache.

Pages: gist.science s.4 (SAW-INT4's throughput is measured against a BF16 KV
cache).  Bar: max |o_gpu - o_ref| / max |o_ref| <= 2e-3, the bar of the INT4
decode; the BF16 path is far inside it (products of bfloat16 values are exact
in binary32, the softmax weights enter the P.V product as a bfloat16 pair)."""
import numpy as np
import pytest
import torch

import bit_paged_kv_gb300 as saw
import oracle
from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import ATTN_TOL, bits, rel_err

pytestmark = pytest.mark.gpu

FILL = 0xABCD


def _caches(num_pages, P, Hkv, D=128):
    n = saw.saw_bf16_cache_bytes(num_pages, P, Hkv, D) // 2
    kc = torch.full((n,), FILL - 0x10000, dtype=torch.int16, device="cuda")
    return kc, kc.clone()


def _host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy().view(np.uint16)


def _rows(wl, lens_l, device="cuda"):
    total = sum(lens_l)
    return W.kv_rows(wl, 0, W.K, total, device), W.kv_rows(wl, 0, W.V, total, device)


def _setup(wl, lens_l, spare=5):
    """BF16 caches holding every token of every sequence, filled on the GPU;
    the same placement done by the oracle must give the same bytes."""
    lens = torch.tensor(lens_l, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=spare)
    k, v = _rows(wl, lens_l)
    slots = W.prefill_slots(bt.cuda(), lens_l, wl.page_size)
    kc, vc = _caches(npages, wl.page_size, wl.num_kv_heads)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_bf16_append(k, v, slots, kc, vc, npages, wl.page_size, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kr = np.full(kc.numel(), FILL, np.uint16)
    vr = np.full(vc.numel(), FILL, np.uint16)
    T = k.shape[0]
    assert oracle.bf16_append(bits(k).reshape(T, -1), bits(v).reshape(T, -1),
                              slots.cpu().numpy(), wl.num_kv_heads, 128, kr, vr, npages,
                              wl.page_size) == 0
    assert np.array_equal(_host(kc), kr) and np.array_equal(_host(vc), vr)
    q = W.q_rows(wl, 0, "cuda", num_seqs=len(lens_l))
    return lens, bt, npages, kc, vc, kr, vr, q


def _decode(q, kc, vc, bt, lens, hkv, npages, P, max_seq_len=None, sm_scale=0.0, ws=None):
    B, Hq, D = q.shape
    if max_seq_len is None:
        max_seq_len = max(int(x) for x in lens.tolist()) if B else 0
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    if ws is None:
        wsb = saw.saw_decode_bf16_workspace_bytes(B, Hq, hkv, D, P, max_seq_len)
        ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda") if wsb else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_paged_decode_bf16(q, kc, vc, bt.cuda(), lens.cuda(), max_seq_len, hkv, npages, P, out,
                              ws, sm_scale=sm_scale, dev_status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def _check(wl, lens, bt, npages, kc, vc, kr, vr, q, label, pairs=None, max_seq_len=None,
           sm_scale=0.0):
    out, st = _decode(q, kc, vc, bt, lens, wl.num_kv_heads, npages, wl.page_size,
                      max_seq_len=max_seq_len, sm_scale=sm_scale)
    assert st == 0
    ref = oracle.decode_bf16(bits(q), kr, vr, bt.numpy(), lens.numpy(), wl.num_q_heads,
                             wl.num_kv_heads, 128, npages, wl.page_size,
                             sm_scale=sm_scale or None, pairs=pairs,
                             threads=oracle.host_threads())
    if pairs is None:
        got = out.cpu().numpy().reshape(-1, 128)
    else:
        got = np.stack([out[b, h].cpu().numpy() for b, h in pairs])
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"bf16-{label}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"
    return out, err


def test_append_any_bits_strided_padding_and_bad_slots():
    """Every bit pattern is copied unchanged (NaNs and infinities included),
    from a token-strided source; slot -1 is padding, slots out of range are
    skipped and reported."""
    g = torch.Generator(device="cuda").manual_seed(11)
    T, Hkv, P, pages = 300, 8, 16, 40
    raw = torch.randint(-32768, 32767, (T, 3 * Hkv * 128), generator=g, device="cuda",
                        dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    k = raw[:, :Hkv * 128].view(T, Hkv, 128)          # token stride 3 * Hkv * D
    v = raw[:, Hkv * 128:2 * Hkv * 128].view(T, Hkv, 128)
    perm = torch.randperm(pages * P, generator=torch.Generator().manual_seed(3))[:T]
    slots = perm.to(torch.int32)
    slots[5] = -1
    slots[17] = pages * P
    slots[40] = -9
    kc, vc = _caches(pages, P, Hkv)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_bf16_append(k, v, slots.cuda(), kc, vc, pages, P, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == saw.SAW_ERR_DEVICE_INDEX
    kr = np.full(kc.numel(), FILL, np.uint16)
    vr = np.full(vc.numel(), FILL, np.uint16)
    kb = bits(k.contiguous()).reshape(T, -1)
    vb = bits(v.contiguous()).reshape(T, -1)
    assert oracle.bf16_append(kb, vb, slots.numpy(), Hkv, 128, kr, vr, pages, P) == 2
    assert np.array_equal(_host(kc), kr)
    assert np.array_equal(_host(vc), vr)
    # K only (v = None) leaves the V cache alone
    kc2, vc2 = _caches(pages, P, Hkv)
    good = slots.clone()
    good[17] = -1
    good[40] = -1
    saw.saw_bf16_append(k, None, good.cuda(), kc2, None, pages, P)
    torch.cuda.synchronize()
    assert np.array_equal(_host(kc2), kr)
    assert torch.all(vc2 == FILL - 0x10000)
    # no tokens: nothing launched, nothing changed
    saw.saw_bf16_append(k[:0], v[:0], slots[:0].cuda(), kc2, vc2, pages, P)
    torch.cuda.synchronize()
    assert np.array_equal(_host(kc2), kr)


EDGE_LENS = [0, 1, 15, 16, 17, 33, 255, 700, 1025, 4097]


@pytest.mark.parametrize("group", [1, 2, 4, 8])
@pytest.mark.parametrize("P", [16, 32, 64])
def test_edge_lengths_groups_pages(group, P):
    """Lengths at tile and page edges, the empty sequence, and sequences long
    enough for several splits (merged in the last split to finish)."""
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=2 * group, page_size=P, shuffle_pages=True,
                        dist="student_t", nu=4)
    lens, bt, npages, kc, vc, kr, vr, q = _setup(wl, EDGE_LENS)
    B, Hq, D = q.shape
    assert saw.saw_decode_bf16_workspace_bytes(B, Hq, 2, D, P, 4097) > 0  # several splits
    out, _ = _check(wl, lens, bt, npages, kc, vc, kr, vr, q, f"edge-G{group}-P{P}")
    assert torch.all(out[0] == 0)  # length 0


@pytest.mark.parametrize("group", [1, 4, 8])
def test_many_sequences_several_waves(group):
    """150 sequences x 2 kv-heads of mixed lengths up to 3000: a grid of
    several waves."""
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=2 * group, shuffle_pages=True)
    g = torch.Generator().manual_seed(group)
    lens_l = EDGE_LENS + torch.randint(1, 3000, (140,), generator=g).tolist()
    lens, bt, npages, kc, vc, kr, vr, q = _setup(wl, lens_l)
    _check(wl, lens, bt, npages, kc, vc, kr, vr, q, f"many-G{group}")


def test_full_size_latency_shape_sampled():
    """The 1 x 32768-token, 32 q-head / 8 kv-head shape, page 16: 24 sampled
    (sequence, head) rows against the oracle."""
    wl = W.QWEN3_4B_LATENCY
    lens_l = W.seq_lens(wl).tolist()
    lens, bt, npages, kc, vc, kr, vr, q = _setup(wl, lens_l, spare=0)
    rng = np.random.default_rng(5)
    pairs = [(0, int(h)) for h in rng.choice(wl.num_q_heads, 24, replace=False)]
    _check(wl, lens, bt, npages, kc, vc, kr, vr, q, "qwen3-4b-latency-32k", pairs=pairs)


def test_plan_for_larger_max_len_explicit_scale_and_workspace_reuse():
    wl = W.TINY.variant(num_q_heads=8, shuffle_pages=True)
    lens, bt, npages, kc, vc, kr, vr, q = _setup(wl, [40, 3000, 7, 2048])
    bt_wide = torch.full((bt.shape[0], 600), -1, dtype=torch.int32)
    bt_wide[:, :bt.shape[1]] = bt
    _check(wl, lens, bt_wide, npages, kc, vc, kr, vr, q, "maxlen-9600", max_seq_len=600 * 16)
    _check(wl, lens, bt, npages, kc, vc, kr, vr, q, "scale-0.3", sm_scale=0.3)
    # one zero-filled workspace, many calls: the counters come back to zero
    B, Hq, D = q.shape
    wsb = saw.saw_decode_bf16_workspace_bytes(B, Hq, wl.num_kv_heads, D, 16, 3000)
    assert wsb > 0
    ws = torch.zeros(wsb, dtype=torch.uint8, device="cuda")
    ref = oracle.decode_bf16(bits(q), kr, vr, bt.numpy(), lens.numpy(), Hq, wl.num_kv_heads, D,
                             npages, 16, threads=oracle.host_threads())
    for _ in range(3):
        out, st = _decode(q, kc, vc, bt, lens, wl.num_kv_heads, npages, 16, ws=ws)
        assert st == 0
        assert rel_err(out.cpu().numpy().reshape(-1, D), ref, "bf16-ws-reuse") <= ATTN_TOL
    assert torch.all(ws[:8 * B * wl.num_kv_heads] == 0)


def test_bad_page_and_bad_length_are_reported():
    wl = W.TINY
    lens, bt, npages, kc, vc, kr, vr, q = _setup(wl, [64, 64])
    bt_bad = bt.clone()
    bt_bad[0, 1] = npages + 10
    out, st = _decode(q, kc, vc, bt_bad, lens, wl.num_kv_heads, npages, 16)
    assert st == saw.SAW_ERR_DEVICE_INDEX
    assert torch.all(torch.isfinite(out))
    lens_bad = torch.tensor([64, 5000], dtype=torch.int32)
    out, st = _decode(q, kc, vc, bt, lens_bad, wl.num_kv_heads, npages, 16, max_seq_len=64)
    assert st == saw.SAW_ERR_DEVICE_INDEX
    assert torch.all(out[1] == 0)
