"""SAW-INT4 hot path on GB300: rotate + token-wise INT4 quantize-append into a
paged KV cache, and paged decode attention over that cache.

The compute lives in the CUDA library built from `csrc/` (C ABI in
`include/saw_int4.h`); this package is its thin Python binding, with the
same names as the C entry points.
"""
from ._binding import (  # noqa: F401
    EXPORTS,
    LIB_PATH,
    SAW_ERR_CUDA,
    SAW_ERR_DEVICE_INDEX,
    SAW_ERR_DEVICE_TIMEOUT,
    SAW_ERR_INVALID_ARG,
    SAW_ERR_UNSUPPORTED,
    SAW_FMT_BF16_META,
    SAW_FMT_F16_INPUT,
    SAW_OK,
    SAW_STEP_EARLY_PAGES,
    SawError,
    lib,
    saw_bf16_append,
    saw_bf16_cache_bytes,
    saw_cache_bytes,
    saw_decode_bf16_workspace_bytes,
    saw_decode_plan,
    saw_decode_step,
    saw_decode_step_ex,
    saw_decode_workspace_bytes,
    saw_paged_decode_bf16,
    saw_paged_decode_int4,
    saw_paged_decode_int4_ex,
    saw_paged_decode_int4_noalloc,
    saw_paged_decode_int4_noalloc_ex,
    saw_prefill_attn_int4,
    saw_prefill_attn_int4_ex,
    saw_quantize_append,
    saw_quantize_append_ex,
    saw_status_string,
)
