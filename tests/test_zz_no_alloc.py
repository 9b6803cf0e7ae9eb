"""The allocation-free decode entry point, saw_paged_decode_int4_noalloc.

It serves callers that cannot allocate device memory -- a plugin whose host
framework owns all allocations, or a loop that cannot afford cudaMalloc's
synchronisation.  Its split-K scratch is
the library's fixed 4 MiB device array instead of a caller workspace.  These
tests call it through the C-ABI three times in a row on the same inputs (the
array keeps the previous call's contents, so each call must clear what has
to start at zero) and then on a second shape, and check every result against
saw_paged_decode_int4 with a workspace, within the attention tolerance the
other tests use, and against the oracle.  The file is named to be collected
last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

import bit_paged_kv_gb300 as saw
from bit_paged_kv_gb300 import build as saw_build
from bit_paged_kv_gb300 import workloads as W
from gpu_helpers import ATTN_TOL, fill_layer, gpu_decode, oracle_decode, rel_err

pytestmark = pytest.mark.gpu


def _noalloc(wl, q, kc, vc, bt, lens, npages, pps):
    B, Hq, D = q.shape
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    L = saw.lib()
    rc = L.saw_paged_decode_int4_noalloc(
        C.c_void_p(q.data_ptr()), C.c_void_p(kc.data_ptr()), C.c_void_p(vc.data_ptr()),
        C.c_void_p(bt.data_ptr()), bt.shape[1], C.c_void_p(lens.data_ptr()), B,
        int(lens.max()), Hq, wl.num_kv_heads, D, npages, wl.page_size, int(wl.rotate_k),
        int(wl.rotate_v), wl.block_h, 0.0, C.c_void_p(out.data_ptr()), pps,
        C.c_void_p(status.data_ptr()), C.c_void_p(stream))
    torch.cuda.synchronize()
    return rc, out, int(status.item())


def _case(wl, lens_list):
    lens = torch.tensor(lens_list, dtype=torch.int32)
    bt, npages = W.page_tables(wl, lens, spare_pages=3)
    kc, vc, _, _, _ = fill_layer(wl, 0, lens, bt, npages)
    q = W.q_rows(wl, 0, "cuda", num_seqs=len(lens_list))
    return q, kc, vc, bt.cuda(), lens.cuda(), npages


def test_noalloc_matches_workspace_entry_on_repeated_calls():
    saw_build.build()
    cases = [
        (W.TINY, W.seq_lens(W.TINY).tolist(), 2),
        (W.TINY.variant(num_q_heads=16, num_kv_heads=2, page_size=32, rotate_v=False,
                        shuffle_pages=True, dist="student_t"), [1, 31, 33, 500, 1000], 1),
    ]
    for wl, lens_list, pps in cases:
        q, kc, vc, bt, lens, npages = _case(wl, lens_list)
        splits, _ = saw.saw_decode_plan(len(lens_list), wl.num_kv_heads, wl.page_size,
                                        int(lens.max()), pps)
        assert splits > 1  # the scratch is really used
        ref, st = gpu_decode(q, kc, vc, bt, lens, wl.num_kv_heads, npages, wl.page_size,
                             wl.rotate_k, wl.rotate_v, wl.block_h, pages_per_split=pps)
        assert st == 0
        r = ref.cpu().numpy().reshape(-1, 128)
        exact = oracle_decode(q, kc.cpu().numpy(), vc.cpu().numpy(), bt.cpu(), lens.cpu(),
                              wl.num_kv_heads, npages, wl.page_size, wl.rotate_k, wl.rotate_v,
                              wl.block_h)
        for call in range(3):
            rc, got, st2 = _noalloc(wl, q, kc, vc, bt, lens, npages, pps)
            assert rc == saw.SAW_OK and st2 == 0, f"call {call}"
            g = got.cpu().numpy().reshape(-1, 128)
            assert np.all(np.isfinite(g))
            assert rel_err(g, r, "noalloc-vs-decode") <= ATTN_TOL, f"call {call}"
            assert rel_err(g, exact, "noalloc-vs-oracle") <= ATTN_TOL, f"call {call}"


def test_noalloc_rejects_plans_beyond_its_scratch():
    saw_build.build()
    # 256 seqs x 64 q-heads x 16 splits of numerators is far above 4 MiB;
    # rejected before any launch, so the made-up pointers are never used
    L = saw.lib()
    rc = L.saw_paged_decode_int4_noalloc(
        C.c_void_p(0x10000), C.c_void_p(0x10000), C.c_void_p(0x20000), C.c_void_p(0x10000),
        1024, C.c_void_p(0x20000), 256, 16384, 64, 8, 128, 4096, 16, 1, 1, 128, 0.0,
        C.c_void_p(0x30000), 64, None, None)
    assert rc == saw.SAW_ERR_UNSUPPORTED
