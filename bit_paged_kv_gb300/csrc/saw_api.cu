// saw_api.cu -- the extern "C" entry points declared in include/saw_int4.h:
// argument checks, the decode split plan, and kernel launches.  No state is
// kept between calls and nothing is allocated.
#include <algorithm>
#include <cmath>
#include <cstdint>

#include "saw_int4.h"
#include "saw_internal.h"

namespace {

using saw::kHeadDim;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }
bool page_size_ok(int p) { return p == 16 || p == 32 || p == 64; }
bool block_h_ok(int h) { return h == 16 || h == 32 || h == 64 || h == 128 || h == 256; }
// head_dim 128 runs the specialised kernels; 64 and 256 the variant kernels
bool head_dim_ok(int d) { return d == 64 || d == kHeadDim || d == 256; }
bool formats_ok(int32_t f) { return (f & ~int32_t(SAW_FMT_F16_INPUT | SAW_FMT_BF16_META)) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

// Split plan.  A split should give every warp several 16-token tiles (at
// least 1024 tokens per split, 4096 when the units fill the GPU without
// splitting).  Among the split counts allowed, take the one
// whose CTA count (sequences x kv-heads x splits) wastes the least of its
// last wave, preferring fewer splits (a smaller merge) unless more splits
// fill the waves clearly better.
// Split search for a grid with `slots` resident CTAs: the split count with
// the least wave quantisation, then, in a one-wave grid, two slots per
// (sequence, kv-head) left free.  Back-to-back launches overlap
// (programmatic dependent launch), and the previous launch's merging splits
// still hold one slot per unit while the next starts; its splits should not
// queue behind them.
int64_t best_splits(int64_t units, int64_t slots, int64_t max_splits) {
  int64_t best = 1;
  double best_q = 1e30;
  for (int64_t s = 1; s <= max_splits; ++s) {
    const int64_t n = units * s;
    const double q = double(ceil_div(n, slots) * slots) / double(n);  // >= 1; 1 = full waves
    if (q < best_q - 0.02) {
      best = s;
      best_q = q;
    }
  }
  if (units * best <= slots && best > 1) {
    const int64_t fit = (slots - 2 * units) / units;
    if (fit >= 1 && fit < best) best = fit;
  }
  return best;
}

// The split plan and the CTA shape.  16-warp CTAs (one per SM) serve grids of
// one wave and long splits; grids of several waves of short splits use 8-warp
// CTAs, two per SM, so that one CTA's prologue and merge overlap the other's
// streaming, or, unsplit with units for four CTAs per SM, 4-warp CTAs.
int32_t make_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t page_size, int32_t max_seq_len,
                  int32_t pages_per_split, int32_t* splits_out,
                  int32_t* pps_out, int32_t* warps_out = nullptr) {
  if (num_seqs < 0 || num_kv_heads <= 0 || !page_size_ok(page_size) || max_seq_len < 0 ||
      pages_per_split < 0)
    return SAW_ERR_INVALID_ARG;
  const int64_t max_pages = ceil_div(max_seq_len, page_size);
  const int64_t units = int64_t(num_seqs > 0 ? num_seqs : 1) * num_kv_heads;
  const int sms_raw = sm_count();
  const int64_t sms = sms_raw > 0 ? sms_raw : 148;
  auto shape_for = [&](int64_t splits, int64_t pps) -> int32_t {
    const bool one_wave = units * splits <= sms;
    const bool long_splits = pps * page_size > saw::kLongSplitTokens;
    return (one_wave || long_splits) ? 16 : 8;
  };
  int64_t pps, splits;
  int32_t warps;
  if (max_pages == 0) {
    pps = 1;
    splits = 1;
    warps = 16;
  } else if (pages_per_split > 0) {
    pps = pages_per_split;
    splits = ceil_div(max_pages, pps);
    warps = shape_for(splits, pps);
  } else {
    // When the (sequence, kv-head) units alone fill every CTA slot of the
    // 8-warp shape, splitting only adds CTA prologues and merges (several
    // waves balance the load anyway): splits of at least 4096 tokens then,
    // at every head dimension.  Smaller grids split down to 1024 tokens to
    // reach every SM.
    const int64_t min_tokens = units >= 2 * sms ? 4096 : 1024;
    const int64_t min_pps = ceil_div(min_tokens, page_size);
    const int64_t max_splits = std::min<int64_t>(64, ceil_div(max_pages, min_pps));
    int64_t s16 = best_splits(units, sms, max_splits);
    int64_t p16 = ceil_div(max_pages, s16);
    s16 = ceil_div(max_pages, p16);
    if (shape_for(s16, p16) == 16) {
      pps = p16;
      splits = s16;
      warps = 16;
    } else {
      const int64_t s8 = best_splits(units, 2 * sms, max_splits);
      pps = ceil_div(max_pages, s8);
      splits = ceil_div(max_pages, pps);
      // one split and units for four CTAs per SM: 4-warp CTAs, so that more
      // CTAs share an SM and one's prologue and epilogue (and, in the fused
      // step, the next launch's early page copies) overlap the others'
      // streaming; with splits the 8-warp shape measured faster
      warps = (splits == 1 && units >= 4 * sms) ? 4 : 8;
    }
    // Whole turns for every warp: a split of a multiple of `warps` 16-token
    // tiles gives no warp a tile more than the others (the slowest warp sets
    // the split's time).  8192 tokens, the long-split bound, is such a
    // multiple, so the rounding never changes the CTA shape.
    const int64_t unit = std::max<int64_t>(1, warps / (page_size / 16));
    pps = ceil_div(pps, unit) * unit;
    splits = ceil_div(max_pages, pps);
  }
  if (splits > 65535) return SAW_ERR_UNSUPPORTED;
  *splits_out = int32_t(splits);
  *pps_out = int32_t(pps);
  if (warps_out) *warps_out = warps;
  return SAW_OK;
}

// Split plan of the BF16 baseline: one 8-warp CTA per SM, at least 1024
// tokens per split, the split count with the least wave quantisation.
int32_t make_plan_bf16(int32_t num_seqs, int32_t num_kv_heads, int32_t page_size,
                       int32_t max_seq_len, int32_t* splits_out, int32_t* pps_out) {
  if (num_seqs < 0 || num_kv_heads <= 0 || !page_size_ok(page_size) || max_seq_len < 0)
    return SAW_ERR_INVALID_ARG;
  const int64_t max_pages = ceil_div(max_seq_len, page_size);
  int64_t pps = 1, splits = 1;
  if (max_pages > 0) {
    const int64_t units = int64_t(num_seqs > 0 ? num_seqs : 1) * num_kv_heads;
    const int sms_raw = sm_count();
    const int64_t sms = sms_raw > 0 ? sms_raw : 148;
    const int64_t max_splits = std::min<int64_t>(64, ceil_div(max_pages, ceil_div(1024, page_size)));
    const int64_t best = best_splits(units, sms, max_splits);
    pps = ceil_div(max_pages, best);
    splits = ceil_div(max_pages, pps);
  }
  *splits_out = int32_t(splits);
  *pps_out = int32_t(pps);
  return SAW_OK;
}

// Whether the decode runs two head_dim-64 kv-heads per CTA as one
// head_dim-128 head (paged_decode.cu, PAIR): GQA 4, an even number of
// kv-heads, 16-token pages, and a grid that keeps at least two CTAs per SM
// with half as many CTAs (the plan's split count does not change).
bool decode_pairs(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                  int32_t page_size, int32_t splits) {
  if (head_dim != 64 || page_size != 16 || num_kv_heads % 2 || num_q_heads != 4 * num_kv_heads)
    return false;
  const int sms = sm_count();
  return int64_t(num_seqs) * (num_kv_heads / 2) * splits >= 2 * int64_t(sms > 0 ? sms : 148);
}

}  // namespace

extern "C" {

const char* saw_status_string(int32_t status) {
  switch (status) {
    case SAW_OK: return "SAW_OK";
    case SAW_ERR_INVALID_ARG: return "SAW_ERR_INVALID_ARG";
    case SAW_ERR_UNSUPPORTED: return "SAW_ERR_UNSUPPORTED";
    case SAW_ERR_CUDA: return "SAW_ERR_CUDA";
    case SAW_ERR_DEVICE_INDEX: return "SAW_ERR_DEVICE_INDEX";
    case SAW_ERR_DEVICE_TIMEOUT: return "SAW_ERR_DEVICE_TIMEOUT";
    default: return "SAW_ERR_UNKNOWN";
  }
}

size_t saw_cache_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads,
                       int32_t head_dim) {
  if (num_pages <= 0 || page_size <= 0 || num_kv_heads <= 0 || head_dim <= 0 || (head_dim & 1))
    return 0;
  const size_t chunk = size_t(page_size) * size_t(head_dim / 2) + 4 * size_t(page_size);
  return size_t(num_pages) * size_t(num_kv_heads) * chunk;
}

int32_t saw_quantize_append_ex(const void* k, const void* v, int64_t k_token_stride,
                               int64_t v_token_stride, const int32_t* slot_mapping,
                               int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                               void* k_cache, void* v_cache, int32_t num_pages,
                               int32_t page_size, int32_t rotate_k, int32_t rotate_v,
                               int32_t block_h, int32_t formats, int32_t* dev_status,
                               void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_pages < 0) return SAW_ERR_INVALID_ARG;
  if (!formats_ok(formats)) return SAW_ERR_INVALID_ARG;
  if (!head_dim_ok(head_dim) || !page_size_ok(page_size)) return SAW_ERR_UNSUPPORTED;
  if ((rotate_k != 0 && rotate_k != 1) || (rotate_v != 0 && rotate_v != 1))
    return SAW_ERR_INVALID_ARG;
  const bool has_v = v != nullptr;
  if (rotate_k || (has_v && rotate_v)) {
    if (!pow2(block_h) || block_h > head_dim || head_dim % block_h) return SAW_ERR_INVALID_ARG;
    if (!block_h_ok(block_h)) return SAW_ERR_UNSUPPORTED;
  }
  if (int64_t(num_tokens) * num_kv_heads > INT32_MAX / 2) return SAW_ERR_UNSUPPORTED;
  if (num_tokens == 0) return SAW_OK;
  if (!k || !slot_mapping || !k_cache || (has_v && !v_cache)) return SAW_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(k_cache) || (has_v && (!aligned16(v) || !aligned16(v_cache))))
    return SAW_ERR_INVALID_ARG;
  if (k_token_stride < int64_t(num_kv_heads) * head_dim || (k_token_stride & 7))
    return SAW_ERR_INVALID_ARG;
  if (has_v && (v_token_stride < int64_t(num_kv_heads) * head_dim || (v_token_stride & 7)))
    return SAW_ERR_INVALID_ARG;

  saw::AppendParams p{};
  p.src[0] = static_cast<const uint16_t*>(k);
  p.src[1] = static_cast<const uint16_t*>(v);
  p.stride[0] = k_token_stride;
  p.stride[1] = has_v ? v_token_stride : 0;
  p.cache[0] = static_cast<uint8_t*>(k_cache);
  p.cache[1] = static_cast<uint8_t*>(v_cache);
  p.rotate[0] = rotate_k;
  p.rotate[1] = has_v ? rotate_v : 0;
  p.slot_mapping = slot_mapping;
  p.dev_status = dev_status;
  p.num_tokens = num_tokens;
  p.num_kv_heads = num_kv_heads;
  p.num_tensors = has_v ? 2 : 1;
  p.page_size = page_size;
  p.block_h = block_h;
  p.num_slots = int64_t(num_pages) * page_size;
  p.c_h = (rotate_k || rotate_v) ? float(1.0 / std::sqrt(double(block_h))) : 1.0f;
  p.in_f16 = (formats & SAW_FMT_F16_INPUT) ? 1 : 0;
  p.meta_bf16 = (formats & SAW_FMT_BF16_META) ? 1 : 0;
  cudaError_t err =
      head_dim == kHeadDim
          ? saw::launch_quantize_append(p, has_v ? 2 : 1, static_cast<cudaStream_t>(stream))
          : saw::launch_quantize_append_var(p, head_dim, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SAW_OK : SAW_ERR_CUDA;
}

int32_t saw_quantize_append(const void* k, const void* v, int64_t k_token_stride,
                            int64_t v_token_stride, const int32_t* slot_mapping,
                            int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                            void* k_cache, void* v_cache, int32_t num_pages, int32_t page_size,
                            int32_t rotate_k, int32_t rotate_v, int32_t block_h,
                            int32_t* dev_status, void* stream) {
  return saw_quantize_append_ex(k, v, k_token_stride, v_token_stride, slot_mapping, num_tokens,
                                num_kv_heads, head_dim, k_cache, v_cache, num_pages, page_size,
                                rotate_k, rotate_v, block_h, 0, dev_status, stream);
}

int32_t saw_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t page_size,
                        int32_t max_seq_len, int32_t pages_per_split, int32_t* num_splits,
                        int32_t* pages_per_split_out) {
  if (!num_splits || !pages_per_split_out) return SAW_ERR_INVALID_ARG;
  return make_plan(num_seqs, num_kv_heads, page_size, max_seq_len, pages_per_split, num_splits,
                   pages_per_split_out);
}

size_t saw_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t page_size, int32_t max_seq_len,
                                  int32_t pages_per_split) {
  if (!head_dim_ok(head_dim) || num_q_heads <= 0) return 0;
  int32_t splits = 0, pps = 0;
  if (make_plan(num_seqs, num_kv_heads, page_size, max_seq_len, pages_per_split, &splits, &pps) !=
      SAW_OK)
    return 0;
  if (splits <= 1) return 0;
  const size_t rows = size_t(num_seqs) * size_t(num_q_heads) * size_t(splits);
  // kv-head pairs keep 128-float partial rows
  const int row_dim = decode_pairs(num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, splits)
                          ? 2 * head_dim
                          : head_dim;
  return saw::decode_ticket_bytes(num_seqs, num_kv_heads) + rows * size_t(row_dim) * 4 +
         rows * 2 * 4;
}

}  // extern "C"

namespace saw {

// Checks shared by the decode entry points; fills the kernel parameters.
// Makes no CUDA call that enqueues work.
int32_t prepare_decode(saw::DecodeParams& p, const void* q, const void* k_cache,
                       const void* v_cache, const int32_t* block_tables,
                       int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs,
                       int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                       int32_t head_dim, int32_t num_pages, int32_t page_size, int32_t rotate_k,
                       int32_t rotate_v, int32_t block_h, float sm_scale, float* out,
                       void* workspace, size_t workspace_bytes, int32_t pages_per_split,
                       int32_t formats, int32_t* dev_status) {
  if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_pages < 0 || max_seq_len < 0)
    return SAW_ERR_INVALID_ARG;
  if (!formats_ok(formats)) return SAW_ERR_INVALID_ARG;
  if (!head_dim_ok(head_dim) || !page_size_ok(page_size)) return SAW_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads) return SAW_ERR_INVALID_ARG;
  if (num_q_heads / num_kv_heads > saw::kMaxGroup) return SAW_ERR_UNSUPPORTED;
  if ((rotate_k != 0 && rotate_k != 1) || (rotate_v != 0 && rotate_v != 1))
    return SAW_ERR_INVALID_ARG;
  if (rotate_k || rotate_v) {
    if (!pow2(block_h) || block_h > head_dim || head_dim % block_h) return SAW_ERR_INVALID_ARG;
    if (!block_h_ok(block_h)) return SAW_ERR_UNSUPPORTED;
  }
  if (!(sm_scale >= 0.0f) || std::isinf(sm_scale)) return SAW_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_kv_heads > 65535) return SAW_ERR_UNSUPPORTED;
  if (num_seqs == 0) return SAW_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
    return SAW_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q) || !aligned16(out))
    return SAW_ERR_INVALID_ARG;
  if (int64_t(max_blocks_per_seq) * page_size < int64_t(max_seq_len)) return SAW_ERR_INVALID_ARG;

  int32_t splits = 0, pps = 0, warps = 16;
  int32_t rc = make_plan(num_seqs, num_kv_heads, page_size, max_seq_len, pages_per_split, &splits,
                         &pps, &warps);
  if (rc != SAW_OK) return rc;
  const size_t need = saw_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 page_size, max_seq_len, pages_per_split);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return SAW_ERR_INVALID_ARG;

  p.q = static_cast<const uint16_t*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = out;
  p.dev_status = dev_status;
  p.max_blocks = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.max_seq_len = max_seq_len;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.num_pages = num_pages;
  p.page_size = page_size;
  p.rotate_k = rotate_k;
  p.rotate_v = rotate_v;
  p.block_h = block_h;
  p.pages_per_split = pps;
  p.num_splits = splits;
  p.warps = warps;
  p.head_dim = head_dim;
  p.c_h = (rotate_k || rotate_v) ? float(1.0 / std::sqrt(double(block_h))) : 1.0f;
  const double scale = sm_scale > 0.0f ? double(sm_scale) : 1.0 / std::sqrt(double(head_dim));
  p.q_scale = float(scale * 1.4426950408889634);  // log2(e)
  p.in_f16 = (formats & SAW_FMT_F16_INPUT) ? 1 : 0;
  p.meta_bf16 = (formats & SAW_FMT_BF16_META) ? 1 : 0;
  p.pair = decode_pairs(num_seqs, num_q_heads, num_kv_heads, head_dim, page_size, splits) ? 1 : 0;
  if (need > 0) bind_decode_workspace(p, workspace);
  return SAW_OK;
}

void bind_decode_workspace(DecodeParams& p, void* workspace) {
  const size_t rows = size_t(p.num_seqs) * size_t(p.num_q_heads) * size_t(p.num_splits);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  p.tickets = reinterpret_cast<uint32_t*>(ws);
  p.part_o = reinterpret_cast<float*>(ws + decode_ticket_bytes(p.num_seqs, p.num_kv_heads));
  p.part_ml = p.part_o + rows * (p.pair ? 2 * p.head_dim : p.head_dim);
}

cudaError_t launch_decode_any(const DecodeParams& p, cudaStream_t stream) {
  return launch_paged_decode(p, stream);
}

}  // namespace saw

using saw::prepare_decode;

extern "C" {

int32_t saw_paged_decode_int4_ex(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t num_pages, int32_t page_size, int32_t rotate_k,
                                 int32_t rotate_v, int32_t block_h, float sm_scale, float* out,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t pages_per_split, int32_t formats, int32_t* dev_status,
                                 void* stream) {
  saw::DecodeParams p{};
  const int32_t rc = prepare_decode(p, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads,
                                    head_dim, num_pages, page_size, rotate_k, rotate_v, block_h,
                                    sm_scale, out, workspace, workspace_bytes, pages_per_split,
                                    formats, dev_status);
  if (rc != SAW_OK || num_seqs == 0) return rc;
  const cudaError_t err = saw::launch_decode_any(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SAW_OK : SAW_ERR_CUDA;
}

int32_t saw_paged_decode_int4(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t num_pages, int32_t page_size, int32_t rotate_k,
                              int32_t rotate_v, int32_t block_h, float sm_scale, float* out,
                              void* workspace, size_t workspace_bytes, int32_t pages_per_split,
                              int32_t* dev_status, void* stream) {
  return saw_paged_decode_int4_ex(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads,
                                  head_dim, num_pages, page_size, rotate_k, rotate_v, block_h,
                                  sm_scale, out, workspace, workspace_bytes, pages_per_split, 0,
                                  dev_status, stream);
}

int32_t saw_decode_step_ex(const void* q, const void* k_new, const void* v_new, void* k_cache,
                           void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t num_pages, int32_t page_size, int32_t rotate_k,
                           int32_t rotate_v, int32_t block_h, float sm_scale, float* out,
                           void* workspace, size_t workspace_bytes, int32_t pages_per_split,
                           int32_t flags, int32_t formats, int32_t* dev_status, void* stream) {
  saw::DecodeParams p{};
  if (flags & ~int32_t(SAW_STEP_EARLY_PAGES)) return SAW_ERR_INVALID_ARG;
  if (head_dim != kHeadDim) return SAW_ERR_UNSUPPORTED;  // the fused step is built for 128
  const int32_t rc = prepare_decode(p, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads,
                                    head_dim, num_pages, page_size, rotate_k, rotate_v, block_h,
                                    sm_scale, out, workspace, workspace_bytes, pages_per_split,
                                    formats, dev_status);
  if (rc != SAW_OK) return rc;
  if (num_seqs == 0) return SAW_OK;
  if (!k_new || !v_new || !aligned16(k_new) || !aligned16(v_new)) return SAW_ERR_INVALID_ARG;
  p.k_new = static_cast<const uint16_t*>(k_new);
  p.v_new = static_cast<const uint16_t*>(v_new);
  p.k_new_stride = int64_t(num_kv_heads) * head_dim;
  p.v_new_stride = int64_t(num_kv_heads) * head_dim;
  p.k_cache_w = static_cast<uint8_t*>(k_cache);
  p.v_cache_w = static_cast<uint8_t*>(v_cache);
  p.append = 1;
  p.early_pages = (flags & SAW_STEP_EARLY_PAGES) ? 1 : 0;
  cudaError_t err = saw::launch_paged_decode(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SAW_OK : SAW_ERR_CUDA;
}

int32_t saw_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t num_pages, int32_t page_size, int32_t rotate_k, int32_t rotate_v,
                        int32_t block_h, float sm_scale, float* out, void* workspace,
                        size_t workspace_bytes, int32_t pages_per_split, int32_t flags,
                        int32_t* dev_status, void* stream) {
  return saw_decode_step_ex(q, k_new, v_new, k_cache, v_cache, block_tables, max_blocks_per_seq,
                            seq_lens, num_seqs, max_seq_len, num_q_heads, num_kv_heads, head_dim,
                            num_pages, page_size, rotate_k, rotate_v, block_h, sm_scale, out,
                            workspace, workspace_bytes, pages_per_split, flags, 0, dev_status,
                            stream);
}


// ---------------------------------------------------------------- prefill

int32_t saw_prefill_attn_int4_ex(const void* q, const int32_t* cu_q_lens, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                                 int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t num_pages, int32_t page_size,
                                 int32_t rotate_k, int32_t rotate_v, int32_t block_h,
                                 float sm_scale, float* out, int32_t formats,
                                 int32_t* dev_status, void* stream) {
  if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_pages < 0 || total_q < 0 ||
      max_q_len < 0 || max_seq_len < 0 || max_q_len > max_seq_len)
    return SAW_ERR_INVALID_ARG;
  if (!formats_ok(formats)) return SAW_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || !page_size_ok(page_size)) return SAW_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads) return SAW_ERR_INVALID_ARG;
  if ((rotate_k != 0 && rotate_k != 1) || (rotate_v != 0 && rotate_v != 1))
    return SAW_ERR_INVALID_ARG;
  if (rotate_k || rotate_v) {
    if (!pow2(block_h) || block_h > head_dim || head_dim % block_h) return SAW_ERR_INVALID_ARG;
    if (!block_h_ok(block_h)) return SAW_ERR_UNSUPPORTED;
  }
  if (!(sm_scale >= 0.0f) || std::isinf(sm_scale)) return SAW_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_kv_heads > 65535) return SAW_ERR_UNSUPPORTED;
  const int64_t rows = int64_t(max_q_len) * (num_q_heads / num_kv_heads);
  const int64_t row_blocks = ceil_div(rows, saw::prefill_rows_per_cta());
  if (row_blocks > INT32_MAX || int64_t(total_q) * num_q_heads * head_dim > INT64_MAX / 8)
    return SAW_ERR_UNSUPPORTED;
  if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return SAW_OK;
  if (!q || !cu_q_lens || !k_cache || !v_cache || !block_tables || !seq_lens || !out)
    return SAW_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q) || !aligned16(out))
    return SAW_ERR_INVALID_ARG;
  if (int64_t(max_blocks_per_seq) * page_size < int64_t(max_seq_len)) return SAW_ERR_INVALID_ARG;
  saw::PrefillParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.cu_q = cu_q_lens;
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = out;
  p.dev_status = dev_status;
  p.max_blocks = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.total_q = total_q;
  p.max_q_len = max_q_len;
  p.max_seq_len = max_seq_len;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.num_pages = num_pages;
  p.page_size = page_size;
  p.rotate_k = rotate_k;
  p.rotate_v = rotate_v;
  p.block_h = block_h;
  p.row_blocks = int32_t(row_blocks);
  p.c_h = (rotate_k || rotate_v) ? float(1.0 / std::sqrt(double(block_h))) : 1.0f;
  const double scale = sm_scale > 0.0f ? double(sm_scale) : 1.0 / std::sqrt(double(head_dim));
  p.q_scale = float(scale * 1.4426950408889634);  // log2(e)
  p.in_f16 = (formats & SAW_FMT_F16_INPUT) ? 1 : 0;
  p.meta_bf16 = (formats & SAW_FMT_BF16_META) ? 1 : 0;
  const cudaError_t err = saw::launch_prefill_attn(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SAW_OK : SAW_ERR_CUDA;
}

int32_t saw_prefill_attn_int4(const void* q, const int32_t* cu_q_lens, const void* k_cache,
                              const void* v_cache, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                              int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t num_pages, int32_t page_size,
                              int32_t rotate_k, int32_t rotate_v, int32_t block_h, float sm_scale,
                              float* out, int32_t* dev_status, void* stream) {
  return saw_prefill_attn_int4_ex(q, cu_q_lens, k_cache, v_cache, block_tables,
                                  max_blocks_per_seq, seq_lens, num_seqs, total_q, max_q_len,
                                  max_seq_len, num_q_heads, num_kv_heads, head_dim, num_pages,
                                  page_size, rotate_k, rotate_v, block_h, sm_scale, out, 0,
                                  dev_status, stream);
}

// ---------------------------------------------------------------- BF16 baseline

size_t saw_bf16_cache_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads,
                            int32_t head_dim) {
  if (num_pages < 0 || page_size <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  return size_t(num_pages) * size_t(num_kv_heads) * size_t(page_size) * size_t(head_dim) * 2;
}

int32_t saw_bf16_append(const void* k, const void* v, int64_t k_token_stride,
                        int64_t v_token_stride, const int32_t* slot_mapping, int32_t num_tokens,
                        int32_t num_kv_heads, int32_t head_dim, void* k_cache, void* v_cache,
                        int32_t num_pages, int32_t page_size, int32_t* dev_status, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || num_pages < 0) return SAW_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || !page_size_ok(page_size)) return SAW_ERR_UNSUPPORTED;
  if (int64_t(num_tokens) * num_kv_heads > INT32_MAX / 2) return SAW_ERR_UNSUPPORTED;
  if (num_tokens == 0) return SAW_OK;
  const bool has_v = v != nullptr;
  if (!k || !slot_mapping || !k_cache || (has_v && !v_cache)) return SAW_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(k_cache) || (has_v && (!aligned16(v) || !aligned16(v_cache))))
    return SAW_ERR_INVALID_ARG;
  if (k_token_stride < int64_t(num_kv_heads) * head_dim || (k_token_stride & 7))
    return SAW_ERR_INVALID_ARG;
  if (has_v && (v_token_stride < int64_t(num_kv_heads) * head_dim || (v_token_stride & 7)))
    return SAW_ERR_INVALID_ARG;
  const cudaError_t err = saw::launch_bf16_append(
      static_cast<const uint16_t*>(k), static_cast<const uint16_t*>(v), k_token_stride,
      has_v ? v_token_stride : 0, slot_mapping, num_tokens, num_kv_heads,
      static_cast<uint16_t*>(k_cache), static_cast<uint16_t*>(v_cache),
      int64_t(num_pages) * page_size, page_size, dev_status, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SAW_OK : SAW_ERR_CUDA;
}

size_t saw_decode_bf16_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                       int32_t max_seq_len) {
  if (head_dim != kHeadDim || num_q_heads <= 0) return 0;
  int32_t splits = 0, pps = 0;
  if (make_plan_bf16(num_seqs, num_kv_heads, page_size, max_seq_len, &splits, &pps) != SAW_OK)
    return 0;
  if (splits <= 1) return 0;
  const size_t rows = size_t(num_seqs) * size_t(num_q_heads) * size_t(splits);
  return saw::decode_ticket_bytes(num_seqs, num_kv_heads) + rows * size_t(head_dim) * 4 +
         rows * 2 * 4;
}

int32_t saw_paged_decode_bf16(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t num_pages, int32_t page_size, float sm_scale, float* out,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream) {
  if (num_seqs < 0 || num_kv_heads <= 0 || num_q_heads <= 0 || num_pages < 0 || max_seq_len < 0)
    return SAW_ERR_INVALID_ARG;
  if (head_dim != kHeadDim || !page_size_ok(page_size)) return SAW_ERR_UNSUPPORTED;
  if (num_q_heads % num_kv_heads) return SAW_ERR_INVALID_ARG;
  if (num_q_heads / num_kv_heads > saw::kMaxGroup) return SAW_ERR_UNSUPPORTED;
  if (!(sm_scale >= 0.0f) || std::isinf(sm_scale)) return SAW_ERR_INVALID_ARG;
  if (num_seqs > 65535 || num_kv_heads > 65535) return SAW_ERR_UNSUPPORTED;
  if (int64_t(num_pages) * num_kv_heads * page_size > INT32_MAX) return SAW_ERR_UNSUPPORTED;
  if (num_seqs == 0) return SAW_OK;
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !out) return SAW_ERR_INVALID_ARG;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(q) || !aligned16(out))
    return SAW_ERR_INVALID_ARG;
  if (int64_t(max_blocks_per_seq) * page_size < int64_t(max_seq_len)) return SAW_ERR_INVALID_ARG;
  int32_t splits = 0, pps = 0;
  int32_t rc = make_plan_bf16(num_seqs, num_kv_heads, page_size, max_seq_len, &splits, &pps);
  if (rc != SAW_OK) return rc;
  const size_t need = saw_decode_bf16_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                      head_dim, page_size, max_seq_len);
  if (need > 0 && (!workspace || workspace_bytes < need || !aligned16(workspace)))
    return SAW_ERR_INVALID_ARG;
  saw::DecodeParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.k_cache = static_cast<const uint8_t*>(k_cache);
  p.v_cache = static_cast<const uint8_t*>(v_cache);
  p.block_tables = block_tables;
  p.seq_lens = seq_lens;
  p.out = out;
  if (need > 0) {
    const size_t rows = size_t(num_seqs) * size_t(num_q_heads) * size_t(splits);
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    p.tickets = reinterpret_cast<uint32_t*>(ws);
    p.part_o = reinterpret_cast<float*>(ws + saw::decode_ticket_bytes(num_seqs, num_kv_heads));
    p.part_ml = p.part_o + rows * head_dim;
  }
  p.dev_status = dev_status;
  p.max_blocks = max_blocks_per_seq;
  p.num_seqs = num_seqs;
  p.max_seq_len = max_seq_len;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = num_q_heads / num_kv_heads;
  p.num_pages = num_pages;
  p.page_size = page_size;
  p.pages_per_split = pps;
  p.num_splits = splits;
  const double scale = sm_scale > 0.0f ? double(sm_scale) : 1.0 / std::sqrt(double(head_dim));
  p.q_scale = float(scale * 1.4426950408889634);  // log2(e)
  const cudaError_t err = saw::launch_paged_decode_bf16(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SAW_OK : SAW_ERR_CUDA;
}

}  // extern "C"
