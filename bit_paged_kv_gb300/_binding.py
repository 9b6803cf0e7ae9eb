"""Thin ctypes binding over the C ABI in include/saw_int4.h.

Argument marshalling only: tensors become device pointers, the current torch
stream becomes the cudaStream_t, and a nonzero status raises.  Every step of
the hot path runs in the library's CUDA kernels; there is no fallback.  If
the library has not been built this module raises on first use.
"""
from __future__ import annotations

import ctypes as C
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libsaw_int4.so")

SAW_OK = 0
SAW_ERR_INVALID_ARG = 1
SAW_ERR_UNSUPPORTED = 2
SAW_ERR_CUDA = 3
SAW_ERR_DEVICE_INDEX = 4
SAW_ERR_DEVICE_TIMEOUT = 5
SAW_STEP_EARLY_PAGES = 1
SAW_FMT_F16_INPUT = 1
SAW_FMT_BF16_META = 2

EXPORTS = ("saw_status_string", "saw_cache_bytes", "saw_quantize_append", "saw_decode_plan",
           "saw_decode_workspace_bytes", "saw_paged_decode_int4", "saw_decode_step",
           "saw_paged_decode_int4_noalloc", "saw_bf16_cache_bytes", "saw_bf16_append",
           "saw_decode_bf16_workspace_bytes", "saw_paged_decode_bf16", "saw_prefill_attn_int4",
           "saw_quantize_append_ex", "saw_paged_decode_int4_ex", "saw_decode_step_ex",
           "saw_prefill_attn_int4_ex", "saw_paged_decode_int4_noalloc_ex")

_lib = None


class SawError(RuntimeError):
    def __init__(self, status: int, where: str):
        super().__init__(f"{where}: {saw_status_string(status)} ({status})")
        self.status = status


def lib() -> C.CDLL:
    """Load the in-tree CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"SAW-INT4 CUDA library not found at {LIB_PATH}; build it with "
            "`python -c 'import __graft_entry__ as g; g.build()'` "
            "(or `python bit_paged_kv_gb300/build.py`). There is no CPU fallback.")
    L = C.CDLL(LIB_PATH)
    P, i32, i64, sz, f32 = C.c_void_p, C.c_int32, C.c_int64, C.c_size_t, C.c_float
    L.saw_status_string.restype = C.c_char_p
    L.saw_status_string.argtypes = [i32]
    L.saw_cache_bytes.restype = sz
    L.saw_cache_bytes.argtypes = [i32, i32, i32, i32]
    L.saw_quantize_append.restype = i32
    L.saw_quantize_append.argtypes = [P, P, i64, i64, P, i32, i32, i32, P, P, i32, i32, i32, i32,
                                      i32, P, P]
    L.saw_decode_plan.restype = i32
    L.saw_decode_plan.argtypes = [i32, i32, i32, i32, i32, P, P]
    L.saw_decode_workspace_bytes.restype = sz
    L.saw_decode_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32, i32]
    L.saw_paged_decode_int4.restype = i32
    L.saw_paged_decode_int4.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32,
                                        i32, i32, i32, f32, P, P, sz, i32, P, P]
    L.saw_decode_step.restype = i32
    L.saw_decode_step.argtypes = [P, P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, i32,
                                  i32, i32, f32, P, P, sz, i32, i32, P, P]
    L.saw_paged_decode_int4_noalloc.restype = i32
    L.saw_paged_decode_int4_noalloc.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32,
                                                i32, i32, i32, i32, f32, P, i32, P, P]
    L.saw_bf16_cache_bytes.restype = sz
    L.saw_bf16_cache_bytes.argtypes = [i32, i32, i32, i32]
    L.saw_bf16_append.restype = i32
    L.saw_bf16_append.argtypes = [P, P, i64, i64, P, i32, i32, i32, P, P, i32, i32, P, P]
    L.saw_decode_bf16_workspace_bytes.restype = sz
    L.saw_decode_bf16_workspace_bytes.argtypes = [i32, i32, i32, i32, i32, i32]
    L.saw_paged_decode_bf16.restype = i32
    L.saw_paged_decode_bf16.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, f32,
                                        P, P, sz, P, P]
    L.saw_prefill_attn_int4.restype = i32
    L.saw_prefill_attn_int4.argtypes = [P, P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32,
                                        i32, i32, i32, i32, i32, f32, P, P, P]
    # the *_ex calls: the same arguments plus `formats` before dev_status
    for name in ("saw_quantize_append", "saw_paged_decode_int4", "saw_decode_step",
                 "saw_prefill_attn_int4", "saw_paged_decode_int4_noalloc"):
        base = getattr(L, name).argtypes
        ex = getattr(L, name + "_ex")
        ex.restype = i32
        ex.argtypes = base[:-2] + [i32] + base[-2:]
    _lib = L
    return L


def _ptr(t):
    if t is None:
        return None
    return C.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor, stream):
    if stream is not None:
        return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))
    return C.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _raise(rc: int, where: str) -> None:
    if rc != SAW_OK:
        raise SawError(rc, where)


_IN_DTYPES = (torch.bfloat16, torch.float16)


def _formats(t: torch.Tensor, meta_bf16: bool) -> int:
    """Format flags from the input dtype (bfloat16 or float16) and the cache's
    metadata format."""
    assert t.dtype in _IN_DTYPES, f"inputs must be bfloat16 or float16, not {t.dtype}"
    return (SAW_FMT_F16_INPUT if t.dtype == torch.float16 else 0) | (
        SAW_FMT_BF16_META if meta_bf16 else 0)


def _call(name: str, formats: int, args: list) -> int:
    """The plain entry point for formats 0, else its *_ex twin with `formats`
    inserted before (dev_status, stream)."""
    if formats == 0:
        return getattr(lib(), name)(*args)
    return getattr(lib(), name + "_ex")(*args[:-2], formats, *args[-2:])


def saw_status_string(status: int) -> str:
    return lib().saw_status_string(int(status)).decode()


def saw_cache_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().saw_cache_bytes(num_pages, page_size, num_kv_heads, head_dim))


def saw_quantize_append(k: torch.Tensor, v, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                        v_cache, num_pages: int, page_size: int, rotate_k: bool, rotate_v: bool,
                        block_h: int, dev_status=None, stream=None, meta_bf16: bool = False) -> None:
    """k, v: bfloat16 or float16 [T, Hkv, D] (token dim may be strided); v may
    be None.  meta_bf16: store the (scale, zero) words as bfloat16."""
    T, hkv, d = k.shape
    fmt = _formats(k, meta_bf16)
    assert k.stride(2) == 1 and k.stride(1) == d
    if v is not None:
        assert v.dtype == k.dtype and v.shape == k.shape and v.stride(2) == 1 and v.stride(1) == d
    assert slot_mapping.dtype == torch.int32 and slot_mapping.is_contiguous()
    rc = _call("saw_quantize_append", fmt, [
        _ptr(k), _ptr(v), k.stride(0), v.stride(0) if v is not None else 0, _ptr(slot_mapping),
        T, hkv, d, _ptr(k_cache), _ptr(v_cache) if v is not None else None, num_pages, page_size,
        int(rotate_k), int(rotate_v), block_h, _ptr(dev_status), _stream(k, stream)])
    _raise(rc, "saw_quantize_append")


def saw_decode_plan(num_seqs: int, num_kv_heads: int, page_size: int, max_seq_len: int,
                    pages_per_split: int = 0):
    s, p = C.c_int32(0), C.c_int32(0)
    rc = lib().saw_decode_plan(num_seqs, num_kv_heads, page_size, max_seq_len, pages_per_split,
                               C.byref(s), C.byref(p))
    _raise(rc, "saw_decode_plan")
    return s.value, p.value


def saw_decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                               head_dim: int, page_size: int, max_seq_len: int,
                               pages_per_split: int = 0) -> int:
    return int(lib().saw_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                page_size, max_seq_len, pages_per_split))


def saw_paged_decode_int4(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                          num_kv_heads: int, num_pages: int, page_size: int, rotate_k: bool,
                          rotate_v: bool, block_h: int, out: torch.Tensor, workspace=None,
                          sm_scale: float = 0.0, pages_per_split: int = 0, dev_status=None,
                          stream=None, meta_bf16: bool = False) -> None:
    """q: bfloat16 or float16 [B, Hq, D] contiguous; out: float32 [B, Hq, D].
    workspace: saw_decode_workspace_bytes() bytes, zero-filled before its
    first use (torch.zeros); each call leaves it ready for the next.
    meta_bf16: the caches hold bfloat16 (scale, zero) words."""
    B, hq, d = q.shape
    fmt = _formats(q, meta_bf16)
    assert q.is_contiguous()
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (B, hq, d)
    assert block_tables.dtype == torch.int32 and block_tables.is_contiguous()
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _call("saw_paged_decode_int4", fmt, [
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), B, max_seq_len, hq, num_kv_heads, d, num_pages, page_size,
        int(rotate_k), int(rotate_v), block_h, float(sm_scale), _ptr(out), _ptr(workspace),
        ws_bytes, pages_per_split, _ptr(dev_status), _stream(q, stream)])
    _raise(rc, "saw_paged_decode_int4")


def saw_decode_step(q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                    k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                    seq_lens: torch.Tensor, max_seq_len: int, num_kv_heads: int, num_pages: int,
                    page_size: int, rotate_k: bool, rotate_v: bool, block_h: int,
                    out: torch.Tensor, workspace=None, sm_scale: float = 0.0,
                    pages_per_split: int = 0, flags: int = 0, dev_status=None,
                    stream=None, meta_bf16: bool = False) -> None:
    """One fused decode step: append k_new/v_new (bfloat16 or float16, like q,
    [B, Hkv, D]) at position seq_lens[b] - 1 of each sequence, then attend
    (one launch).  flags=SAW_STEP_EARLY_PAGES: see include/saw_int4.h."""
    B, hq, d = q.shape
    fmt = _formats(q, meta_bf16)
    assert q.is_contiguous()
    for t in (k_new, v_new):
        assert t.dtype == q.dtype and t.is_contiguous() and tuple(t.shape) == (B, num_kv_heads, d)
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (B, hq, d)
    assert block_tables.dtype == torch.int32 and block_tables.is_contiguous()
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = _call("saw_decode_step", fmt, [
        _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), B, max_seq_len, hq, num_kv_heads, d, num_pages,
        page_size, int(rotate_k), int(rotate_v), block_h, float(sm_scale), _ptr(out),
        _ptr(workspace), ws_bytes, pages_per_split, int(flags), _ptr(dev_status),
        _stream(q, stream)])
    _raise(rc, "saw_decode_step")


def saw_paged_decode_int4_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                                  block_tables: torch.Tensor, seq_lens: torch.Tensor,
                                  max_seq_len: int, num_kv_heads: int, num_pages: int,
                                  page_size: int, rotate_k: bool, rotate_v: bool, block_h: int,
                                  out: torch.Tensor, sm_scale: float = 0.0,
                                  pages_per_split: int = 0, dev_status=None, stream=None,
                                  meta_bf16: bool = False) -> None:
    """saw_paged_decode_int4 without a workspace argument: the split-K
    scratch is the library's own fixed 4 MiB device array (for callers that
    cannot allocate).  Raises SawError(SAW_ERR_UNSUPPORTED) if the plan needs
    more than that.  q: bfloat16 or float16."""
    B, hq, d = q.shape
    fmt = _formats(q, meta_bf16)
    assert q.is_contiguous()
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (B, hq, d)
    assert block_tables.dtype == torch.int32 and block_tables.is_contiguous()
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    rc = _call("saw_paged_decode_int4_noalloc", fmt, [
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), B, max_seq_len, hq, num_kv_heads, d, num_pages, page_size,
        int(rotate_k), int(rotate_v), block_h, float(sm_scale), _ptr(out), pages_per_split,
        _ptr(dev_status), _stream(q, stream)])
    _raise(rc, "saw_paged_decode_int4_noalloc")


def saw_bf16_cache_bytes(num_pages: int, page_size: int, num_kv_heads: int, head_dim: int) -> int:
    return int(lib().saw_bf16_cache_bytes(num_pages, page_size, num_kv_heads, head_dim))


def saw_bf16_append(k: torch.Tensor, v, slot_mapping: torch.Tensor, k_cache: torch.Tensor,
                    v_cache, num_pages: int, page_size: int, dev_status=None,
                    stream=None) -> None:
    """k, v: bfloat16 [T, Hkv, D] (token dim may be strided); v may be None."""
    T, hkv, d = k.shape
    assert k.dtype == torch.bfloat16 and k.stride(2) == 1 and k.stride(1) == d
    if v is not None:
        assert v.dtype == torch.bfloat16 and v.shape == k.shape and v.stride(2) == 1 and v.stride(1) == d
    assert slot_mapping.dtype == torch.int32 and slot_mapping.is_contiguous()
    rc = lib().saw_bf16_append(
        _ptr(k), _ptr(v), k.stride(0), v.stride(0) if v is not None else 0, _ptr(slot_mapping),
        T, hkv, d, _ptr(k_cache), _ptr(v_cache) if v is not None else None, num_pages,
        page_size, _ptr(dev_status), _stream(k, stream))
    _raise(rc, "saw_bf16_append")


def saw_decode_bf16_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int,
                                    head_dim: int, page_size: int, max_seq_len: int) -> int:
    return int(lib().saw_decode_bf16_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                     head_dim, page_size, max_seq_len))


def saw_paged_decode_bf16(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                          block_tables: torch.Tensor, seq_lens: torch.Tensor, max_seq_len: int,
                          num_kv_heads: int, num_pages: int, page_size: int, out: torch.Tensor,
                          workspace=None, sm_scale: float = 0.0, dev_status=None,
                          stream=None) -> None:
    """Decode over the BF16 cache.  q: bfloat16 [B, Hq, D]; out: float32
    [B, Hq, D]; workspace: saw_decode_bf16_workspace_bytes() bytes, zero-filled
    before its first use."""
    B, hq, d = q.shape
    assert q.dtype == torch.bfloat16 and q.is_contiguous()
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (B, hq, d)
    assert block_tables.dtype == torch.int32 and block_tables.is_contiguous()
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    rc = lib().saw_paged_decode_bf16(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
        _ptr(seq_lens), B, max_seq_len, hq, num_kv_heads, d, num_pages, page_size,
        float(sm_scale), _ptr(out), _ptr(workspace), ws_bytes, _ptr(dev_status),
        _stream(q, stream))
    _raise(rc, "saw_paged_decode_bf16")


def saw_prefill_attn_int4(q: torch.Tensor, cu_q_lens: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, block_tables: torch.Tensor,
                          seq_lens: torch.Tensor, max_q_len: int, max_seq_len: int,
                          num_kv_heads: int, num_pages: int, page_size: int, rotate_k: bool,
                          rotate_v: bool, block_h: int, out: torch.Tensor, sm_scale: float = 0.0,
                          dev_status=None, stream=None, meta_bf16: bool = False) -> None:
    """Chunked-prefill attention.  q: bfloat16 or float16 [T, Hq, D] (the
    chunks of all sequences, sequence after sequence); cu_q_lens: int32
    [B + 1]; out: float32 [T, Hq, D]."""
    T, hq, d = q.shape
    fmt = _formats(q, meta_bf16)
    assert q.is_contiguous()
    assert out.dtype == torch.float32 and out.is_contiguous() and tuple(out.shape) == (T, hq, d)
    assert cu_q_lens.dtype == torch.int32 and cu_q_lens.is_contiguous()
    assert block_tables.dtype == torch.int32 and block_tables.is_contiguous()
    assert seq_lens.dtype == torch.int32 and seq_lens.is_contiguous()
    B = seq_lens.shape[0]
    assert cu_q_lens.shape[0] == B + 1
    rc = _call("saw_prefill_attn_int4", fmt, [
        _ptr(q), _ptr(cu_q_lens), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(seq_lens), B, T, max_q_len, max_seq_len, hq, num_kv_heads,
        d, num_pages, page_size, int(rotate_k), int(rotate_v), block_h, float(sm_scale),
        _ptr(out), _ptr(dev_status), _stream(q, stream)])
    _raise(rc, "saw_prefill_attn_int4")


# ---------------------------------------------------------------- *_ex twins
# The C ABI's *_ex calls take the format flags explicitly; here the input
# format is the tensors' dtype, so `formats` must agree with it, and its
# SAW_FMT_BF16_META bit selects the metadata format.  Unknown bits are
# passed through for the library to reject.

def _ex_meta(t: torch.Tensor, formats: int) -> bool:
    f16 = bool(formats & SAW_FMT_F16_INPUT)
    assert f16 == (t.dtype == torch.float16), "formats disagrees with the input dtype"
    if formats & ~(SAW_FMT_F16_INPUT | SAW_FMT_BF16_META):
        _raise(SAW_ERR_INVALID_ARG, "formats")
    return bool(formats & SAW_FMT_BF16_META)


def saw_quantize_append_ex(k, v, slot_mapping, k_cache, v_cache, num_pages, page_size, rotate_k,
                           rotate_v, block_h, formats: int, dev_status=None, stream=None) -> None:
    saw_quantize_append(k, v, slot_mapping, k_cache, v_cache, num_pages, page_size, rotate_k,
                        rotate_v, block_h, dev_status, stream, meta_bf16=_ex_meta(k, formats))


def saw_paged_decode_int4_ex(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len,
                             num_kv_heads, num_pages, page_size, rotate_k, rotate_v, block_h, out,
                             formats: int, workspace=None, sm_scale: float = 0.0,
                             pages_per_split: int = 0, dev_status=None, stream=None) -> None:
    saw_paged_decode_int4(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len, num_kv_heads,
                          num_pages, page_size, rotate_k, rotate_v, block_h, out, workspace,
                          sm_scale, pages_per_split, dev_status, stream,
                          meta_bf16=_ex_meta(q, formats))


def saw_decode_step_ex(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len,
                       num_kv_heads, num_pages, page_size, rotate_k, rotate_v, block_h, out,
                       formats: int, workspace=None, sm_scale: float = 0.0,
                       pages_per_split: int = 0, flags: int = 0, dev_status=None,
                       stream=None) -> None:
    saw_decode_step(q, k_new, v_new, k_cache, v_cache, block_tables, seq_lens, max_seq_len,
                    num_kv_heads, num_pages, page_size, rotate_k, rotate_v, block_h, out,
                    workspace, sm_scale, pages_per_split, flags, dev_status, stream,
                    meta_bf16=_ex_meta(q, formats))


def saw_prefill_attn_int4_ex(q, cu_q_lens, k_cache, v_cache, block_tables, seq_lens, max_q_len,
                             max_seq_len, num_kv_heads, num_pages, page_size, rotate_k, rotate_v,
                             block_h, out, formats: int, sm_scale: float = 0.0, dev_status=None,
                             stream=None) -> None:
    saw_prefill_attn_int4(q, cu_q_lens, k_cache, v_cache, block_tables, seq_lens, max_q_len,
                          max_seq_len, num_kv_heads, num_pages, page_size, rotate_k, rotate_v,
                          block_h, out, sm_scale, dev_status, stream,
                          meta_bf16=_ex_meta(q, formats))


def saw_paged_decode_int4_noalloc_ex(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len,
                                     num_kv_heads, num_pages, page_size, rotate_k, rotate_v,
                                     block_h, out, formats: int, sm_scale: float = 0.0,
                                     pages_per_split: int = 0, dev_status=None,
                                     stream=None) -> None:
    saw_paged_decode_int4_noalloc(q, k_cache, v_cache, block_tables, seq_lens, max_seq_len,
                                  num_kv_heads, num_pages, page_size, rotate_k, rotate_v,
                                  block_h, out, sm_scale, pages_per_split, dev_status, stream,
                                  meta_bf16=_ex_meta(q, formats))
