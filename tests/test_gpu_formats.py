"""GPU parity of the two format variants against the oracle.

* binary16 input (q, K, V as float16): the youngju.dev fused-kernel diagram
  ("The System Is the Design -- A Fused Kernel") feeds the kernel fp16 K/V.
* bfloat16 (scale, zero) metadata: the same directed-rounding rules stored
  as bfloat16 (the pages fix one scale per token, not its format).

Bars as for the plain path: every cache byte equal to the oracle's, attention
within 2e-3 of the oracle's float64 result (relative to its largest
magnitude).  Every kernel is covered: the tiled and warp-per-row appends,
the head_dim 64/256 append, the head_dim-128 decode (both CTA shapes via the
split plan), the variant decode, the fused decode step and the prefill."""
import numpy as np
import pytest
import torch

import bit_paged_kv_gb300 as saw
import oracle
from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import (ATTN_TOL, assert_bytes_equal, bits, fill_layer, gpu_append, gpu_decode,
                         new_caches, oracle_append, oracle_decode, rel_err)

pytestmark = pytest.mark.gpu

# (input dtype, bfloat16 metadata)
FORMATS = [(torch.float16, False), (torch.bfloat16, True), (torch.float16, True)]
FMT_IDS = ["f16in", "bf16meta", "f16in-bf16meta"]


def _label(dt, bfm):
    return ("f16" if dt == torch.float16 else "bf16") + ("-bfm" if bfm else "")


@pytest.mark.parametrize("fmt", FORMATS, ids=FMT_IDS)
@pytest.mark.parametrize("D,h,T", [(128, 128, 300), (128, 32, 300), (128, 128, 1100),
                                   (128, 16, 1100), (128, 64, 1100), (64, 64, 300),
                                   (256, 256, 300), (256, 128, 300)])
@pytest.mark.parametrize("rot", [(True, True), (True, False), (False, False)])
def test_append_bytes(fmt, D, h, T, rot):
    """T x 4 rows: 1200 rows run the warp-per-row kernel at head_dim 128,
    4400 rows the tiled kernel."""
    dt, bfm = fmt
    wl = W.TINY.variant(head_dim=D, block_h=h, num_kv_heads=4, dist="student_t", nu=3)
    P, pages = 16, (T + 15) // 16 + 8
    k = W.kv_rows(wl, 0, W.K, T, "cuda", dtype=dt)
    v = W.kv_rows(wl, 0, W.V, T, "cuda", dtype=dt)
    perm = torch.randperm(pages * P, generator=torch.Generator().manual_seed(D + h + T))[:T]
    slots = perm.to(torch.int32)
    slots[5] = -1
    kc, vc, st = gpu_append(k, v, slots.cuda(), pages, P, rot[0], rot[1], h, meta_bf16=bfm)
    assert st == 0
    kr, vr, bad = oracle_append(k, v, slots, pages, P, rot[0], rot[1], h, meta_bf16=bfm)
    assert bad == 0
    assert_bytes_equal(kc, kr, f"K {_label(dt, bfm)} D{D} h{h} T{T}")
    assert_bytes_equal(vc, vr, f"V {_label(dt, bfm)} D{D} h{h} T{T}")


def _extreme_rows(T, Hkv, D, dt, seed):
    """Rows at the edges of the formats: huge (beyond binary16 for bfloat16
    input, and near 10^32), bfloat16 subnormals, tiny, constant, signed zeros,
    one-hot, and binary16 subnormals."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, Hkv, D, generator=g)
    kind = torch.arange(T) % 8
    big = 3e5 if dt == torch.bfloat16 else 4e3
    x[kind == 0] *= big
    x[kind == 1] *= 1e-39 if dt == torch.bfloat16 else 1e-7
    x[kind == 2] *= 1e-5
    x[kind == 3] = 2.5
    x[kind == 4] = -0.0
    x[kind == 5] = 0.0
    x[kind == 5, :, 7] = 1.0
    x[kind == 6] = torch.randint(0, 16, (int((kind == 6).sum()), Hkv, D), generator=g) * 2.0 ** -24
    if dt == torch.bfloat16:
        x[kind == 7] *= 1e32  # scales beyond 2^101: the tiled kernel's clamping path
    return x.to(dt).cuda()


@pytest.mark.parametrize("fmt", FORMATS + [(torch.bfloat16, False)],
                         ids=FMT_IDS + ["bf16in-f16meta"])
@pytest.mark.parametrize("D,T", [(128, 1100), (128, 200), (64, 200), (256, 200)])
def test_append_extreme_rows(fmt, D, T):
    dt, bfm = fmt
    Hkv, P = 4, 16
    pages = (T + 15) // 16 + 2
    k = _extreme_rows(T, Hkv, D, dt, 1 + D)
    v = _extreme_rows(T, Hkv, D, dt, 2 + D)
    slots = torch.arange(T, dtype=torch.int32)
    for rot in ((True, False), (False, False)):
        kc, vc, st = gpu_append(k, v, slots.cuda(), pages, P, rot[0], rot[1], min(D, 128),
                                meta_bf16=bfm)
        assert st == 0
        kr, vr, _ = oracle_append(k, v, slots, pages, P, rot[0], rot[1], min(D, 128),
                                  meta_bf16=bfm)
        assert_bytes_equal(kc, kr, f"K extreme {_label(dt, bfm)} D{D} rot{rot}")
        assert_bytes_equal(vc, vr, f"V extreme {_label(dt, bfm)} D{D} rot{rot}")


def _setup(wl, lens_l, dt, bfm, spare=3):
    lens = torch.tensor(lens_l, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=spare)
    kc, vc, _, _, _ = fill_layer(wl, 0, lens, bt, npages, dtype=dt, meta_bf16=bfm)
    q = W.q_rows(wl, 0, "cuda", num_seqs=len(lens_l), dtype=dt)
    return lens, bt, npages, kc, vc, q


@pytest.mark.parametrize("fmt", FORMATS, ids=FMT_IDS)
@pytest.mark.parametrize("D,h", [(128, 128), (128, 32), (64, 64), (256, 128)])
@pytest.mark.parametrize("group", [1, 4, 8])
def test_decode(fmt, D, h, group):
    dt, bfm = fmt
    wl = W.TINY.variant(head_dim=D, block_h=h, num_kv_heads=2, num_q_heads=2 * group,
                        shuffle_pages=True, dist="student_t", nu=4)
    lens, bt, npages, kc, vc, q = _setup(wl, [0, 1, 33, 100, 700, 2500], dt, bfm)
    for pps in (0, 3):
        out, st = gpu_decode(q, kc, vc, bt.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                             wl.page_size, wl.rotate_k, wl.rotate_v, h, pages_per_split=pps,
                             meta_bf16=bfm)
        assert st == 0
        ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads,
                            npages, wl.page_size, wl.rotate_k, wl.rotate_v, h, meta_bf16=bfm)
        got = out.cpu().numpy().reshape(-1, D)
        assert np.all(np.isfinite(got))
        err = rel_err(got, ref, f"fmt-decode-{_label(dt, bfm)}-D{D}-h{h}-G{group}-pps{pps}")
        assert err <= ATTN_TOL, f"relative error {err:.3e}"


@pytest.mark.parametrize("fmt", FORMATS, ids=FMT_IDS)
def test_decode_many_sequences_long_context(fmt):
    """The latency and concurrency shapes: one 32k-token sequence (many
    splits) and 64 short ones (8-warp CTAs), Hq 32, Hkv 8, K-only rotation."""
    dt, bfm = fmt
    wl = W.QWEN3_4B_LATENCY
    g = torch.Generator().manual_seed(3)
    for lens_l in ([32768], torch.randint(1, 900, (64,), generator=g).tolist()):
        lens, bt, npages, kc, vc, q = _setup(wl, lens_l, dt, bfm, spare=0)
        out, st = gpu_decode(q, kc, vc, bt.cuda(), lens.cuda(), wl.num_kv_heads, npages,
                             wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h, meta_bf16=bfm)
        assert st == 0
        pairs = [(b, hq) for b in range(0, len(lens_l), 7) for hq in range(0, 32, 5)]
        ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads,
                            npages, wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                            pairs=pairs, meta_bf16=bfm)
        got = np.stack([out[b, hq].cpu().numpy() for b, hq in pairs])
        err = rel_err(got, ref, f"fmt-decode-{_label(dt, bfm)}-B{len(lens_l)}")
        assert err <= ATTN_TOL, f"relative error {err:.3e}"


@pytest.mark.parametrize("fmt", FORMATS, ids=FMT_IDS)
@pytest.mark.parametrize("P,group,pps,flags", [(16, 4, 0, 0), (16, 8, 2, 1), (64, 1, 1, 0)])
def test_fused_decode_step(fmt, P, group, pps, flags):
    dt, bfm = fmt
    wl = W.TINY.variant(page_size=P, num_q_heads=2 * group, num_kv_heads=2, shuffle_pages=True,
                        rotate_v=False, dist="student_t", nu=4)
    lens_l = [1, 17, 16, P + 1, 300, 31, 0]
    lens = torch.tensor(lens_l, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=3)
    kc, vc, k_pre, v_pre, slots_pre = fill_layer(wl, 0, lens, bt, npages,
                                                 upto=lambda n: max(n - 1, 0), dtype=dt,
                                                 meta_bf16=bfm)
    B, D = len(lens_l), 128
    knew = (torch.randn(B, wl.num_kv_heads, D, device="cuda") * 2).to(dt)
    vnew = (torch.randn(B, wl.num_kv_heads, D, device="cuda") * 2).to(dt)
    q = W.q_rows(wl, 0, "cuda", num_seqs=B, dtype=dt)
    Lmax = int(lens.max())
    out = torch.full((B, wl.num_q_heads, D), float("nan"), dtype=torch.float32, device="cuda")
    wsb = saw.saw_decode_workspace_bytes(B, wl.num_q_heads, wl.num_kv_heads, D, P, Lmax, pps)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_decode_step(q, knew, vnew, kc, vc, bt.cuda(), lens.cuda(), Lmax, wl.num_kv_heads,
                        npages, P, wl.rotate_k, wl.rotate_v, wl.block_h, out, ws,
                        pages_per_split=pps, flags=flags, dev_status=st, meta_bf16=bfm)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    kr, vr, _ = oracle_append(k_pre, v_pre, slots_pre.cpu(), npages, P, wl.rotate_k, wl.rotate_v,
                              wl.block_h, meta_bf16=bfm)
    keep = [b for b in range(B) if lens_l[b] > 0]
    slots_new = torch.tensor([int(bt[b, (lens_l[b] - 1) // P]) * P + (lens_l[b] - 1) % P
                              for b in keep], dtype=torch.int32)
    oracle_append(knew[keep], vnew[keep], slots_new, npages, P, wl.rotate_k, wl.rotate_v,
                  wl.block_h, kc=kr, vc=vr, meta_bf16=bfm)
    assert_bytes_equal(kc, kr, f"K after step {_label(dt, bfm)}")
    assert_bytes_equal(vc, vr, f"V after step {_label(dt, bfm)}")
    ref = oracle_decode(q, kr, vr, bt, lens, wl.num_kv_heads, npages, P, wl.rotate_k, wl.rotate_v,
                        wl.block_h, meta_bf16=bfm)
    got = out.cpu().numpy().reshape(-1, D)
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"fmt-step-{_label(dt, bfm)}-P{P}-G{group}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"


@pytest.mark.parametrize("fmt", FORMATS, ids=FMT_IDS)
@pytest.mark.parametrize("group,P", [(1, 16), (4, 64), (8, 16)])
def test_prefill(fmt, group, P):
    dt, bfm = fmt
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=2 * group, page_size=P, shuffle_pages=True,
                        dist="student_t", nu=4)
    cases = [(300, 300), (700, 97), (33, 1), (64, 0), (17, 16), (1025, 200)]
    lens_l = [L for L, _ in cases]
    q_lens = [n for _, n in cases]
    lens = torch.tensor(lens_l, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=3)
    kc, vc, _, _, _ = fill_layer(wl, 0, lens, bt, npages, dtype=dt, meta_bf16=bfm)
    gq = torch.Generator(device="cuda").manual_seed(group + P)
    T = sum(q_lens)
    q = torch.randn(T, wl.num_q_heads, 128, generator=gq, device="cuda").to(dt)
    cu = torch.tensor([0] + np.cumsum(q_lens).tolist(), dtype=torch.int32)
    out = torch.full((T, wl.num_q_heads, 128), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_prefill_attn_int4(q, cu.cuda(), kc, vc, bt.cuda(), lens.cuda(), max(q_lens),
                              int(lens.max()), wl.num_kv_heads, npages, P, wl.rotate_k,
                              wl.rotate_v, wl.block_h, out, dev_status=st, meta_bf16=bfm)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref = oracle.prefill(bits(q), cu.numpy(), kc.cpu().numpy(), vc.cpu().numpy(), bt.numpy(),
                         lens.numpy(), wl.num_q_heads, wl.num_kv_heads, 128, npages, P,
                         wl.rotate_k, wl.rotate_v, wl.block_h, threads=oracle.host_threads(),
                         in_f16=dt == torch.float16, meta_bf16=bfm)
    got = out.cpu().numpy().reshape(-1, 128)
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"fmt-prefill-{_label(dt, bfm)}-G{group}-P{P}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"


def test_ex_twins_agree_with_dtype_dispatch():
    """The *_ex bindings with explicit flags write the same bytes as the plain
    names with the dtype / meta_bf16 dispatch, and a flag that disagrees with
    the dtype is refused on the host."""
    wl = W.TINY.variant(num_kv_heads=2)
    T, P, pages = 64, 16, 8
    k = W.kv_rows(wl, 0, W.K, T, "cuda", dtype=torch.float16)
    v = W.kv_rows(wl, 0, W.V, T, "cuda", dtype=torch.float16)
    slots = torch.arange(T, dtype=torch.int32, device="cuda")
    kc1, vc1 = new_caches(pages, P, 2, 128)
    kc2, vc2 = new_caches(pages, P, 2, 128)
    fmt = saw.SAW_FMT_F16_INPUT | saw.SAW_FMT_BF16_META
    saw.saw_quantize_append_ex(k, v, slots, kc1, vc1, pages, P, True, True, 128, fmt)
    saw.saw_quantize_append(k, v, slots, kc2, vc2, pages, P, True, True, 128, meta_bf16=True)
    torch.cuda.synchronize()
    assert torch.equal(kc1, kc2) and torch.equal(vc1, vc2)
    with pytest.raises(AssertionError):
        saw.saw_quantize_append_ex(k, v, slots, kc1, vc1, pages, P, True, True, 128,
                                   saw.SAW_FMT_BF16_META)


@pytest.mark.parametrize("fmt", FORMATS, ids=FMT_IDS)
def test_noalloc_decode(fmt):
    """The no-alloc decode under each format equals the oracle."""
    dt, bfm = fmt
    wl = W.TINY.variant(num_q_heads=8, shuffle_pages=True, dist="student_t", nu=4)
    lens, bt, npages, kc, vc, q = _setup(wl, [900, 40, 2000], dt, bfm)
    B, Hq, D = q.shape
    ref = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt, lens, wl.num_kv_heads, npages,
                        wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h, meta_bf16=bfm)
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_paged_decode_int4_noalloc(q, kc, vc, bt.cuda(), lens.cuda(), 2000, wl.num_kv_heads,
                                      npages, wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                                      out, pages_per_split=8, dev_status=st, meta_bf16=bfm)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    err = rel_err(out.cpu().numpy().reshape(-1, D), ref, f"fmt-noalloc-{_label(dt, bfm)}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"
