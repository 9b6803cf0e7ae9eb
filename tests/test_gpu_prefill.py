"""GPU parity of the chunked-prefill attention over the INT4 cache (through
the C-ABI) against the oracle's float64 causal attention on the same cache
bytes.  The chunk's K/V are appended by the CUDA quantize-append first (its
bytes are checked against the oracle's by the append tests).

Bar: max |o_gpu - o_ref| / max |o_ref| <= 2e-3, the decode's.  Pages:
youngju.dev "Why the KV Cache Is the Real Bottleneck" and gist.science s.1
(fused attention over paged KV); causal reading as in the oracle."""
import numpy as np
import pytest
import torch

import bit_paged_kv_gb300 as saw
import oracle
from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import ATTN_TOL, bits, fill_layer, rel_err

pytestmark = pytest.mark.gpu


def _setup(wl, lens_l, q_lens, spare=3, seed=0):
    lens = torch.tensor(lens_l, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=spare)
    kc, vc, _, _, _ = fill_layer(wl, 0, lens, bt, npages)
    g = torch.Generator(device="cuda").manual_seed(seed)
    T = sum(q_lens)
    q = torch.randn(T, wl.num_q_heads, wl.head_dim, generator=g, device="cuda").to(torch.bfloat16)
    cu = torch.tensor([0] + np.cumsum(q_lens).tolist(), dtype=torch.int32)
    return lens, bt, npages, kc, vc, q, cu


def _run(wl, lens, bt, npages, kc, vc, q, cu, max_q_len=None, max_seq_len=None, sm_scale=0.0):
    T = q.shape[0]
    out = torch.full((T, wl.num_q_heads, wl.head_dim), float("nan"), dtype=torch.float32,
                     device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q_lens = (cu[1:] - cu[:-1]).tolist()
    mq = max(q_lens) if max_q_len is None else max_q_len
    ms = int(lens.max()) if max_seq_len is None else max_seq_len
    saw.saw_prefill_attn_int4(q, cu.cuda(), kc, vc, bt.cuda(), lens.cuda(), mq, ms,
                              wl.num_kv_heads, npages, wl.page_size, wl.rotate_k, wl.rotate_v,
                              wl.block_h, out, sm_scale=sm_scale, dev_status=st)
    torch.cuda.synchronize()
    return out, int(st.item())


def _check(wl, lens, bt, npages, kc, vc, q, cu, label, rows=None, sm_scale=0.0, **kw):
    out, st = _run(wl, lens, bt, npages, kc, vc, q, cu, sm_scale=sm_scale, **kw)
    assert st == 0
    ref = oracle.prefill(bits(q), cu.numpy(), kc.cpu().numpy(), vc.cpu().numpy(), bt.numpy(),
                         lens.numpy(), wl.num_q_heads, wl.num_kv_heads, wl.head_dim, npages,
                         wl.page_size, wl.rotate_k, wl.rotate_v, wl.block_h,
                         sm_scale=sm_scale or None, rows=rows, threads=oracle.host_threads())
    if rows is None:
        got = out.cpu().numpy().reshape(-1, wl.head_dim)
    else:
        got = np.stack([out[i, h].cpu().numpy() for i, h in rows])
    assert np.all(np.isfinite(got))
    err = rel_err(got, ref, f"prefill-{label}")
    assert err <= ATTN_TOL, f"relative error {err:.3e}"
    return out


# (seq_len, q_len): a whole prompt, chunks after a prefix, a single token,
# an empty chunk, a one-token sequence, lengths at tile and page edges
CASES = [(300, 300), (700, 97), (33, 1), (64, 0), (1, 1), (17, 16), (129, 64), (1025, 200)]


@pytest.mark.parametrize("group", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("P", [16, 64])
def test_groups_pages_ragged_chunks(group, P):
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=2 * group, page_size=P, shuffle_pages=True,
                        dist="student_t", nu=4)
    lens_l = [L for L, _ in CASES]
    q_lens = [n for _, n in CASES]
    lens, bt, npages, kc, vc, q, cu = _setup(wl, lens_l, q_lens, seed=group * 100 + P)
    _check(wl, lens, bt, npages, kc, vc, q, cu, f"G{group}-P{P}")


@pytest.mark.parametrize("rot", [(1, 1), (1, 0), (0, 0), (0, 1)])
@pytest.mark.parametrize("h", [128, 64, 16])
def test_rotations_and_blocks(rot, h):
    wl = W.TINY.variant(num_kv_heads=2, num_q_heads=8, page_size=32, block_h=h,
                        rotate_k=bool(rot[0]), rotate_v=bool(rot[1]), shuffle_pages=True)
    lens, bt, npages, kc, vc, q, cu = _setup(wl, [260, 45, 90], [260, 45, 30], seed=h)
    _check(wl, lens, bt, npages, kc, vc, q, cu, f"rot{rot[0]}{rot[1]}-h{h}")


def test_explicit_scale_and_loose_bounds():
    """sm_scale given; a grid sized for larger max_q_len / max_seq_len than
    any sequence uses."""
    wl = W.TINY.variant(num_q_heads=8, shuffle_pages=True)
    lens, bt, npages, kc, vc, q, cu = _setup(wl, [200, 31], [50, 31], seed=7)
    bt_wide = torch.full((bt.shape[0], 100), -1, dtype=torch.int32)
    bt_wide[:, :bt.shape[1]] = bt
    _check(wl, lens, bt_wide, npages, kc, vc, q, cu, "scale-0.3", sm_scale=0.3, max_q_len=400,
           max_seq_len=1600)


def test_long_context_chunk_sampled():
    """A 4096-token chunk at the end of a 131072-token sequence (Hq 32, Hkv 8,
    page 64, h 128, heavy-tailed rows): 24 sampled (row, head) outputs."""
    wl = W.LONG_PREFILL.variant(num_seqs=1)
    L, n = 131072, 4096
    lens, bt, npages, kc, vc, q, cu = _setup(wl, [L], [n], spare=0, seed=9)
    rng = np.random.default_rng(3)
    rows = [(int(i), int(h)) for i, h in zip(rng.integers(0, n, 24),
                                             rng.integers(0, wl.num_q_heads, 24))]
    rows[0], rows[1] = (0, 0), (n - 1, wl.num_q_heads - 1)
    _check(wl, lens, bt, npages, kc, vc, q, cu, "long-131072-chunk4096", rows=rows)


def test_bad_page_and_inconsistent_chunk_are_reported():
    wl = W.TINY
    lens, bt, npages, kc, vc, q, cu = _setup(wl, [64, 64], [64, 10], seed=1)
    bt_bad = bt.clone()
    bt_bad[0, 1] = npages + 7
    out, st = _run(wl, lens, bt_bad, npages, kc, vc, q, cu)
    assert st == saw.SAW_ERR_DEVICE_INDEX
    assert torch.all(torch.isfinite(out))
    # a chunk longer than its sequence: skipped and reported, the other
    # sequence is still right
    lens2 = torch.tensor([64, 5], dtype=torch.int32)
    out, st = _run(wl, lens2, bt, npages, kc, vc, q, cu, max_q_len=64, max_seq_len=64)
    assert st == saw.SAW_ERR_DEVICE_INDEX
    ref = oracle.prefill(bits(q[:64]), np.array([0, 64], np.int32), kc.cpu().numpy(),
                         vc.cpu().numpy(), bt[:1].numpy(), [64], wl.num_q_heads,
                         wl.num_kv_heads, 128, npages, 16, True, True, 128)
    assert rel_err(out[:64].cpu().numpy().reshape(-1, 128), ref, "prefill-skip-bad") <= ATTN_TOL
    assert torch.all(torch.isnan(out[64:]))  # untouched
