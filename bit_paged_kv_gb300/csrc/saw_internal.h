// saw_internal.h -- kernel parameter blocks and launchers (library-internal).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace saw {

constexpr int kHeadDim = 128;       // the one head size this build supports
constexpr int kMaxGroup = 8;        // q-heads per kv-head served by one CTA (MMA N = 8)
// Decode CTA shapes: 16 warps, one CTA per SM (one-wave grids and long
// splits), or 8 warps, two CTAs per SM (many short splits: one CTA's prologue
// and merge overlap the other's streaming).  Splits of more than this many
// tokens count as long.
constexpr int kLongSplitTokens = 8192;

__host__ __device__ constexpr int chunk_bytes(int page_size) {
  return page_size * (kHeadDim / 2) + 4 * page_size;
}

// ---------------------------------------------------------------- append

struct AppendParams {
  const uint16_t* src[2];       // K, V bfloat16 (binary16 if in_f16) bits [T][Hkv][D] with token stride
  int64_t stride[2];            // token stride in elements
  uint8_t* cache[2];            // K, V caches
  int32_t rotate[2];
  const int32_t* slot_mapping;  // [T]
  int32_t* dev_status;
  int32_t num_tokens;
  int32_t num_kv_heads;
  int32_t num_tensors;          // 2 = K and V, 1 = K only
  int32_t page_size;
  int32_t block_h;
  int64_t num_slots;            // num_pages * page_size
  float c_h;                    // binary32(1/sqrt(block_h))
  int32_t in_f16;               // 1: the rows are binary16
  int32_t meta_bf16;            // 1: (scale, zero) stored as bfloat16
  // set by the launcher: row / num_kv_heads = (row * hkv_mul) >> hkv_shift
  // for rows below 2^31, and page_size = 1 << page_shift
  uint32_t hkv_mul;
  uint32_t hkv_shift;
  int32_t page_shift;
};

cudaError_t launch_quantize_append(const AppendParams& p, int num_tensors, cudaStream_t stream);

// ---------------------------------------------------------------- decode

struct DecodeParams {
  const uint16_t* q;            // [B][Hq][D] bfloat16 (binary16 if in_f16) bits
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;  // [B][max_blocks]
  const int32_t* seq_lens;      // [B]
  float* out;                   // [B][Hq][D]
  float* part_o;                // [B][Hq][num_splits][D]
  float* part_ml;               // [B][Hq][num_splits][2]
  uint32_t* tickets;            // [B][Hkv][2] split counters (arrived, published), zero between calls
  // decode step only: the new token's K and V rows, bfloat16 (binary16 if
  // in_f16) [B][Hkv][D]
  // with a per-sequence stride, quantized and appended at position
  // seq_len - 1 before attending
  const uint16_t* k_new;
  const uint16_t* v_new;
  int64_t k_new_stride;
  int64_t v_new_stride;
  uint8_t* k_cache_w;           // writable views of the caches (decode step)
  uint8_t* v_cache_w;
  int32_t append;               // 1: decode step (append, then attend)
  int32_t early_pages;          // 1: tables and pages may be read before the previous kernel ends
  int32_t* dev_status;
  int32_t max_blocks;
  int32_t num_seqs;
  int32_t max_seq_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;                // num_q_heads / num_kv_heads
  int32_t num_pages;
  int32_t page_size;
  int32_t rotate_k;
  int32_t rotate_v;
  int32_t block_h;
  int32_t pages_per_split;
  int32_t num_splits;
  float c_h;                    // 1/sqrt(block_h)
  float q_scale;                // sm_scale * log2(e)
  int32_t warps;                // CTA shape: 16 (one per SM) or 8 (two per SM)
  int32_t head_dim;             // 128, or 64 / 256
  int32_t in_f16;               // 1: q, k_new and v_new are binary16
  int32_t meta_bf16;            // 1: the caches' (scale, zero) words are bfloat16
  // 1: head_dim 64, GQA 4: each CTA serves two neighbouring kv-heads as one
  // head_dim-128 "pair" head with 8 q-head columns (part_o rows are 128
  // floats wide, the grid has num_kv_heads / 2 rows)
  int32_t pair;
};

// One launcher per CTA shape (paged_decode.cu compiled once per shape), and
// per shape for head_dim 64 and 256 (the same source built for those sizes).
cudaError_t launch_paged_decode_w16(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_paged_decode_w8(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_paged_decode_w4(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_paged_decode_dims_w16(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_paged_decode_dims_w8(const DecodeParams& p, cudaStream_t stream);
// head_dim 64 and 256 append (variants.cu); bulk appends run the tiled
// kernels of quantize_append.cu
cudaError_t launch_quantize_append_var(const AppendParams& p, int head_dim, cudaStream_t stream);
cudaError_t launch_quantize_append_tiled64(const AppendParams& p, int num_tensors,
                                           cudaStream_t stream);
cudaError_t launch_quantize_append_tiled256(const AppendParams& p, int num_tensors,
                                            cudaStream_t stream);
// BF16 baseline (paged_decode_bf16.cu)
cudaError_t launch_paged_decode_bf16(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_bf16_append(const uint16_t* k, const uint16_t* v, int64_t k_stride,
                               int64_t v_stride, const int32_t* slots, int num_tokens, int hkv,
                               uint16_t* kc, uint16_t* vc, int64_t num_slots, int P,
                               int32_t* dev_status, cudaStream_t stream);
// (head_dim 64 and 256 have no 4-warp build: they take the 8-warp shape)
inline cudaError_t launch_paged_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.head_dim != kHeadDim)
    return p.warps <= 8 ? launch_paged_decode_dims_w8(p, stream)
                        : launch_paged_decode_dims_w16(p, stream);
  if (p.warps == 4) return launch_paged_decode_w4(p, stream);
  return p.warps == 8 ? launch_paged_decode_w8(p, stream) : launch_paged_decode_w16(p, stream);
}

// Host side of the INT4 decode entry points (saw_api.cu).  prepare_decode
// checks every argument and fills p (split plan, CTA shape, scales) without
// enqueueing anything; when the plan needs a workspace, `workspace` must be
// non-null, 16-byte aligned and at least workspace_bytes long, and p's
// workspace fields point into it.  bind_decode_workspace points them at
// another buffer of the same layout.  launch_decode_any picks the head_dim
// 128 kernel or the 64/256 variant.
int32_t prepare_decode(DecodeParams& p, const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                       int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                       int32_t num_pages, int32_t page_size, int32_t rotate_k, int32_t rotate_v,
                       int32_t block_h, float sm_scale, float* out, void* workspace,
                       size_t workspace_bytes, int32_t pages_per_split, int32_t formats,
                       int32_t* dev_status);
void bind_decode_workspace(DecodeParams& p, void* workspace);
cudaError_t launch_decode_any(const DecodeParams& p, cudaStream_t stream);

// ---------------------------------------------------------------- prefill

struct PrefillParams {
  const uint16_t* q;            // [total_q][Hq][D] bfloat16 (binary16 if in_f16) bits, sequence after sequence
  const int32_t* cu_q;          // [B + 1] first query row of each sequence
  const uint8_t* k_cache;
  const uint8_t* v_cache;
  const int32_t* block_tables;  // [B][max_blocks]
  const int32_t* seq_lens;      // [B] cached tokens, the chunk included
  float* out;                   // [total_q][Hq][D]
  int32_t* dev_status;
  int32_t max_blocks;
  int32_t num_seqs;
  int32_t total_q;
  int32_t max_q_len;
  int32_t max_seq_len;
  int32_t num_q_heads;
  int32_t num_kv_heads;
  int32_t group;
  int32_t num_pages;
  int32_t page_size;
  int32_t rotate_k;
  int32_t rotate_v;
  int32_t block_h;
  int32_t row_blocks;           // grid x: ceil(max_q_len * group / rows per CTA)
  float c_h;
  float q_scale;                // sm_scale * log2(e)
  int32_t in_f16;               // 1: q is binary16
  int32_t meta_bf16;            // 1: the caches' (scale, zero) words are bfloat16
};

int prefill_rows_per_cta();
cudaError_t launch_prefill_attn(const PrefillParams& p, cudaStream_t stream);

// Split-K workspace layout: the merge's counter words first, two per
// (sequence, kv-head), rounded to 16 bytes; then the numerators
// [B][Hq][splits][D], then (m, l) pairs [B][Hq][splits][2].
inline size_t decode_ticket_bytes(int num_seqs, int num_kv_heads) {
  return (size_t(num_seqs) * size_t(num_kv_heads) * 8 + 15) / 16 * 16;
}

}  // namespace saw
