"""Helpers for the GPU parity tests: run the CUDA path through the C-ABI
binding and the oracle on the very same inputs, and compare.

Tolerance for attention: max |o_gpu - o_ref| / max |o_ref| <= 2e-3 per layer
over the compared rows (the oracle is float64; the GPU path uses binary16
operands on the tensor cores with binary32 accumulation).  Codes, scales and
zero-points must match byte for byte.
"""
import numpy as np
import torch

import bit_paged_kv_gb300 as saw
import oracle
from bit_paged_kv_gb300 import workloads as W

ATTN_TOL = 2e-3
SENTINEL = 0xAB


def bits(t: torch.Tensor) -> np.ndarray:
    """bfloat16 or float16 tensor (any device) -> numpy uint16 bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def new_caches(num_pages, P, Hkv, D, device="cuda", with_v=True):
    n = saw.saw_cache_bytes(num_pages, P, Hkv, D)
    kc = torch.full((n,), SENTINEL, dtype=torch.uint8, device=device)
    vc = torch.full((n,), SENTINEL, dtype=torch.uint8, device=device) if with_v else None
    return kc, vc


def gpu_append(k, v, slots, num_pages, P, rotate_k, rotate_v, h, kc=None, vc=None,
               meta_bf16=False):
    T, Hkv, D = k.shape
    if kc is None:
        kc, vc = new_caches(num_pages, P, Hkv, D, with_v=v is not None)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_quantize_append(k, v, slots, kc, vc, num_pages, P, rotate_k, rotate_v, h,
                            dev_status=status, meta_bf16=meta_bf16)
    torch.cuda.synchronize()
    return kc, vc, int(status.item())


def oracle_append(k, v, slots, num_pages, P, rotate_k, rotate_v, h, kc=None, vc=None,
                  meta_bf16=False):
    T, Hkv, D = k.shape
    n = oracle.cache_bytes(num_pages, P, Hkv, D)
    if kc is None:
        kc = np.full(n, SENTINEL, np.uint8)
        vc = np.full(n, SENTINEL, np.uint8) if v is not None else None
    kb = bits(k).reshape(T, -1)
    vb = bits(v).reshape(T, -1) if v is not None else None
    bad = oracle.quantize_append(kb, vb, slots.cpu().numpy(), Hkv, D, kc, vc, num_pages, P,
                                 rotate_k, rotate_v, h, threads=oracle.host_threads(),
                                 in_f16=k.dtype == torch.float16, meta_bf16=meta_bf16)
    return kc, vc, bad


def assert_bytes_equal(gpu: torch.Tensor, ref: np.ndarray, what: str):
    g = gpu.cpu().numpy()
    if not np.array_equal(g, ref):
        diff = np.nonzero(g != ref)[0]
        raise AssertionError(f"{what}: {diff.size} bytes differ, first at {diff[:8].tolist()} "
                             f"(gpu {g[diff[:8]].tolist()} vs oracle {ref[diff[:8]].tolist()})")


def gpu_decode(q, kc, vc, bt, lens, num_kv_heads, num_pages, P, rotate_k, rotate_v, h,
               max_seq_len=None, pages_per_split=0, sm_scale=0.0, meta_bf16=False):
    B, Hq, D = q.shape
    if max_seq_len is None:
        max_seq_len = max(int(x) for x in lens.tolist()) if B else 0
    out = torch.full((B, Hq, D), float("nan"), dtype=torch.float32, device="cuda")
    wsb = saw.saw_decode_workspace_bytes(B, Hq, num_kv_heads, D, P, max_seq_len, pages_per_split)
    ws = torch.zeros(max(wsb, 16), dtype=torch.uint8, device="cuda") if wsb else None
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    saw.saw_paged_decode_int4(q, kc, vc, bt, lens, max_seq_len, num_kv_heads, num_pages, P,
                              rotate_k, rotate_v, h, out, ws, sm_scale=sm_scale,
                              pages_per_split=pages_per_split, dev_status=status,
                              meta_bf16=meta_bf16)
    torch.cuda.synchronize()
    return out, int(status.item())


def oracle_decode(q, kc_host, vc_host, bt, lens, num_kv_heads, num_pages, P, rotate_k, rotate_v,
                  h, pairs=None, sm_scale=None, meta_bf16=False):
    B, Hq, D = q.shape
    return oracle.decode(bits(q), kc_host, vc_host, bt.cpu().numpy(), lens.cpu().numpy(), Hq,
                         num_kv_heads, D, num_pages, P, rotate_k, rotate_v, h,
                         sm_scale=sm_scale, pairs=pairs, threads=oracle.host_threads(),
                         in_f16=q.dtype == torch.float16, meta_bf16=meta_bf16)


ERRORS = []  # (label, relative error) of every attention comparison, for the log


def rel_err(got: np.ndarray, ref: np.ndarray, label: str = "") -> float:
    scale = np.max(np.abs(ref))
    if scale == 0.0:
        e = float(np.max(np.abs(got)))
    else:
        e = float(np.max(np.abs(got - ref)) / scale)
    ERRORS.append((label, e))
    return e


def fill_layer(wl: W.Workload, layer: int, lens, bt, num_pages, device="cuda", upto=None,
               kc=None, vc=None, chunk_tokens=1 << 18, dtype=torch.bfloat16, meta_bf16=False):
    """Quantize-append every token of every sequence (or the first `upto`
    tokens of each) of one layer into fresh caches with the CUDA path.
    Returns (kc, vc, k_rows, v_rows, slots) with the rows appended (`dtype`:
    bfloat16, or float16 for the binary16-input variant)."""
    P = wl.page_size
    lens_l = [int(x) for x in lens.tolist()]
    if upto is not None:
        lens_l = [min(L, upto(L)) for L in lens_l]
    total = sum(lens_l)
    k = W.kv_rows(wl, layer, W.K, total, device, dtype=dtype)
    v = W.kv_rows(wl, layer, W.V, total, device, dtype=dtype)
    slots = W.prefill_slots(bt.to(device), lens_l, P)
    if kc is None:
        kc, vc = new_caches(num_pages, P, wl.num_kv_heads, wl.head_dim, device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    for a in range(0, total, chunk_tokens):
        b = min(total, a + chunk_tokens)
        saw.saw_quantize_append(k[a:b], v[a:b], slots[a:b], kc, vc, num_pages, P, wl.rotate_k,
                                wl.rotate_v, wl.block_h, dev_status=status, meta_bf16=meta_bf16)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    return kc, vc, k, v, slots
