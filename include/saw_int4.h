/*
 * saw_int4.h -- C ABI of the SAW-INT4 hot path on GB300 (sm_103a).
 *
 * Two operations, from the pages on SAW-INT4 (Jia et al., 2026):
 *
 *  1. saw_quantize_append: each new token's K/V vector of head_dim values
 *     per kv-head is rotated by a block-diagonal Hadamard transform (blocks
 *     of h), quantized token-wise to INT4 with its own scale, and appended
 *     into a paged KV cache without touching any other token.
 *     youngju.dev, "INT4 KV-cache quantization" (English transcription),
 *     "Why Naive INT4 Breaks", "The Rotation Trick -- Block-Diagonal
 *     Hadamard" and the fused-kernel diagram in "The System Is the Design --
 *     A Fused Kernel"; gist.science, "SAW-INT4: System-Aware 4-Bit KV-Cache
 *     Quantization for Real-World LLM Serving", s.2 "Metodologia" (token-wise
 *     quantization, Block-Diagonal Rotation, fused kernel) and s.4 (h = 128,
 *     rotation of K only).
 *
 *  2. saw_paged_decode_int4: decode attention of one query token per
 *     sequence over that INT4 cache, with dequantization fused into the
 *     attention kernel (gist.science s.2 point 3, fusion into decoding).
 *     q is rotated once (q.k = Hq.Hk because H is orthogonal), and the output
 *     is rotated back when V was rotated.
 *
 * Further calls build on these two: saw_decode_step (both in one launch),
 * saw_prefill_attn_int4 (causal attention of a chunk of queries over the
 * same cache), the *_ex forms with binary16 inputs or bfloat16 scale/zero
 * metadata, and a BF16 paged cache with the same decode (saw_bf16_*), the
 * baseline the pages compare INT4 against.
 *
 * Readings taken where the pages are silent: Sylvester ordering of H, the
 * 1/sqrt(h) scale applied after an ascending-stride butterfly, one binary16
 * (scale, zero) pair per (token, kv-head) from the rotated row's min/max
 * (zero rounded toward -inf, scale toward +inf), round-half-even codes 0..15,
 * two codes per byte (even index in the low nibble), and the page layout
 * below.  Each is stated with the function it governs.
 *
 * Common rules for every entry point:
 *  - All buffers are owned by the caller.  The library allocates nothing and
 *    keeps no state between calls (saw_paged_decode_int4_noalloc's fixed
 *    scratch array aside); every call is thread-safe.
 *  - Pointers marked "device" must be device memory of the current device.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *    enqueued asynchronously on it.  The return value reports argument
 *    checks and launch errors only.
 *  - `dev_status` is an optional device int32 (may be NULL).  A kernel that
 *    meets a bad index or a wait that runs out writes a nonzero
 *    saw_status code into it (the first one wins); it never traps.  The
 *    caller zeroes it and reads it after the stream has finished.
 */
#ifndef SAW_INT4_H
#define SAW_INT4_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum saw_status {
  SAW_OK = 0,
  SAW_ERR_INVALID_ARG = 1,    /* a null pointer, a bad size, a misaligned buffer */
  SAW_ERR_UNSUPPORTED = 2,    /* a shape this build has no kernel for */
  SAW_ERR_CUDA = 3,           /* a CUDA runtime error at launch */
  SAW_ERR_DEVICE_INDEX = 4,   /* device-side: a slot, page id or length out of range (skipped) */
  SAW_ERR_DEVICE_TIMEOUT = 5  /* device-side: a bounded wait on a copy ran out */
} saw_status;

/* Human-readable name of a status code.  Never NULL. */
const char* saw_status_string(int32_t status);

/*
 * Bytes of one cache tensor (K or V of one layer):
 *   [num_pages][num_kv_heads][chunk],  chunk = page_size*head_dim/2 + 4*page_size.
 * Inside a chunk: token offset o's packed codes at o*head_dim/2 (byte j holds
 * code 2j in the low nibble and 2j+1 in the high nibble), then, from
 * page_size*head_dim/2, one 4-byte word per offset: binary16 scale, binary16
 * zero, little-endian.  A row dequantizes as code*scale + zero.  The layout
 * is a reading: the pages require only a paged, token-wise layout.
 * Returns 0 for a negative or zero argument.
 */
size_t saw_cache_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads,
                       int32_t head_dim);

/*
 * Rotate, quantize and append num_tokens tokens of K (and V) into the paged
 * caches (youngju.dev "The System Is the Design -- A Fused Kernel";
 * gist.science s.2 and s.3 point 3).
 *
 * k, v          device bfloat16 [num_tokens][num_kv_heads][head_dim], rows of
 *               a token contiguous; token stride k_token_stride /
 *               v_token_stride elements (>= num_kv_heads*head_dim, multiple
 *               of 8).  v may be NULL: K only (v_cache is then ignored).
 * slot_mapping  device int32 [num_tokens]: slot = page*page_size + offset.
 *               -1 marks padding and is skipped; any other value outside
 *               [0, num_pages*page_size) is skipped and reported through
 *               dev_status as SAW_ERR_DEVICE_INDEX.
 * k_cache, v_cache  device, saw_cache_bytes() each, 16-byte aligned.
 * rotate_k, rotate_v  0 or 1: apply the block-diagonal Hadamard rotation
 *               before quantizing.  The gist.science page (s.4) reports that
 *               rotating K only matches rotating both.
 * block_h       rotation block size h: 16, 32, 64, 128 or 256, at most
 *               head_dim (ignored when neither tensor is rotated).
 *
 * Per row, exactly: widen to binary32; if rotated, an in-place butterfly per
 * h-block with strides 1, 2, ..., h/2 (each a+b, a-b rounded to nearest),
 * then multiply by binary32(1/sqrt(h)); mn/mx over the row; zero =
 * binary16 round-down(mn), scale = binary16 round-up((mx - zero)/15), both
 * saturating at +-65504 and writing zero as +0; r = 1/scale (0 if scale is
 * 0); code = clamp(round-half-even((y - zero)*r), 0, 15).  Each operation is
 * one binary32 round-to-nearest step, so the bytes are fully determined.
 * Inputs are expected finite; non-finite inputs give unspecified codes.
 *
 * Supported: head_dim 64, 128 or 256 (128 runs the tiled bulk kernel, 64
 * and 256 a warp-per-row kernel; the bytes follow the same rule); page_size
 * 16, 32 or 64; num_kv_heads >= 1.  Other sizes: SAW_ERR_UNSUPPORTED.
 * Rows whose slot is written by two tokens of the same call race.
 */
int32_t saw_quantize_append(const void* k, const void* v, int64_t k_token_stride,
                            int64_t v_token_stride, const int32_t* slot_mapping,
                            int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                            void* k_cache, void* v_cache, int32_t num_pages, int32_t page_size,
                            int32_t rotate_k, int32_t rotate_v, int32_t block_h,
                            int32_t* dev_status, void* stream);

/*
 * How many splits of the context the decode will use, and how many pages
 * each split covers, for these sizes on the current device
 * (pages_per_split = 0 picks them from the SM count; > 0 forces it).  The
 * plan is the same at every head dimension.
 * Writes *num_splits and *pages_per_split_out; returns a saw_status.
 */
int32_t saw_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t page_size,
                        int32_t max_seq_len, int32_t pages_per_split, int32_t* num_splits,
                        int32_t* pages_per_split_out);

/*
 * Workspace bytes saw_paged_decode_int4 needs for these sizes with the same
 * pages_per_split argument, on the current device (0 when the plan has one
 * split, which writes the output directly).  Returns 0 on bad arguments.
 * The workspace holds the split partials and, first, two counter words per
 * (sequence, kv-head) that the merge uses: zero-fill a new workspace once
 * (e.g. cudaMemset) before its first use; every call leaves those words at
 * zero again.
 */
size_t saw_decode_workspace_bytes(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t page_size, int32_t max_seq_len,
                                  int32_t pages_per_split);

/*
 * Decode attention for one query token per sequence over the INT4 pages
 * (gist.science s.2 point 3: the rotation and dequantization live inside
 * the decode kernel; youngju.dev "The Rotation Trick": H is orthogonal, so
 * attention can run in the rotated domain).
 *
 * q             device bfloat16 [num_seqs][num_q_heads][head_dim].
 * k_cache, v_cache  device caches written by saw_quantize_append with the
 *               same num_kv_heads, head_dim, page_size, rotate_* and block_h
 *               (the caller's contract; a mismatch gives wrong numbers).
 * block_tables  device int32 [num_seqs][max_blocks_per_seq]: logical page i
 *               of a sequence -> physical page id.  Ids outside
 *               [0, num_pages) are skipped and reported as
 *               SAW_ERR_DEVICE_INDEX.
 * seq_lens      device int32 [num_seqs]: tokens to attend over (including a
 *               token just appended).  0 gives a zero output row.  A value
 *               below 0 or above max_seq_len is reported as
 *               SAW_ERR_DEVICE_INDEX and treated as 0.
 * max_seq_len   host upper bound on seq_lens; fixes the split plan.
 *               max_blocks_per_seq must be >= ceil(max_seq_len / page_size).
 * num_q_heads   a multiple of num_kv_heads with at most 8 q-heads per
 *               kv-head; q-head j reads kv-head j / (num_q_heads/num_kv_heads).
 * sm_scale      softmax scale on q.k; 0 means 1/sqrt(head_dim).
 * out           device float32 [num_seqs][num_q_heads][head_dim].
 * workspace     device, >= saw_decode_workspace_bytes(...) bytes, 16-byte
 *               aligned (may be NULL when that is 0), zero-filled before its
 *               first use (calls leave it reusable).  The last split to
 *               finish for a (sequence, kv-head) merges the partials, so one
 *               launch covers the whole decode.  Calls sharing a workspace
 *               must be ordered (one stream).
 * pages_per_split  0 = automatic; > 0 forces the split size (tests).
 *
 * Computes, per (sequence, q-head): q' = (1/sqrt(h)) H q if K was rotated;
 * t_j = sm_scale * q'.(code_j*s_j + z_j); p = softmax(t); o' = sum_j p_j
 * (code_j*s_j + z_j) over V; o = (1/sqrt(h)) H o' if V was rotated.  The
 * GQA group of a kv-head is served by one pass over its pages.  Arithmetic
 * (head_dim 64, 128 and 256 alike): q' and p*s in binary16 on the tensor
 * cores with binary32 accumulation, softmax in binary32; results match a
 * float64 evaluation to about 1e-3 of the output's largest magnitude.
 * Up to 8 q-heads per kv-head; head_dim 64, 128 or 256 (else
 * SAW_ERR_UNSUPPORTED).
 */
int32_t saw_paged_decode_int4(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t num_pages, int32_t page_size, int32_t rotate_k,
                              int32_t rotate_v, int32_t block_h, float sm_scale, float* out,
                              void* workspace, size_t workspace_bytes, int32_t pages_per_split,
                              int32_t* dev_status, void* stream);

/*
 * One decode step of a layer, fused into one launch: for every sequence b,
 * quantize-append the new token's K and V rows at position seq_lens[b] - 1
 * (slot = block_tables[b][(L-1)/page_size]*page_size + (L-1)%page_size),
 * then attend over all seq_lens[b] tokens -- the per-token path of the
 * fused-kernel diagram in youngju.dev "The System Is the Design -- A Fused
 * Kernel" (rotate, quantize, append to the paged block) followed by the
 * decode of gist.science s.2 point 3.
 *
 * k_new, v_new  device bfloat16 [num_seqs][num_kv_heads][head_dim],
 *               contiguous, 16-byte aligned: the new token of each sequence.
 * k_cache, v_cache  written (the new rows) and read.
 * seq_lens      lengths INCLUDING the new token (>= 1).  A length of 0
 *               appends nothing and gives a zero output row.
 * flags         0, or SAW_STEP_EARLY_PAGES: the caller guarantees that the
 *               kernel issued just before this call on `stream` writes none
 *               of block_tables, seq_lens, k_cache and v_cache.  The kernel
 *               may then read them and start its page copies while that
 *               kernel finishes (programmatic dependent launch); it still
 *               waits for it before reading q, k_new, v_new or writing.
 * Other arguments as saw_paged_decode_int4.  The appended bytes equal those
 * of saw_quantize_append on the same row, and the output equals
 * saw_quantize_append followed by saw_paged_decode_int4.  head_dim 128 only
 * (SAW_ERR_UNSUPPORTED otherwise).
 */
#define SAW_STEP_EARLY_PAGES 1
int32_t saw_decode_step(const void* q, const void* k_new, const void* v_new, void* k_cache,
                        void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                        int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                        int32_t num_pages, int32_t page_size, int32_t rotate_k, int32_t rotate_v,
                        int32_t block_h, float sm_scale, float* out, void* workspace,
                        size_t workspace_bytes, int32_t pages_per_split, int32_t flags,
                        int32_t* dev_status, void* stream);

/*
 * saw_paged_decode_int4_noalloc -- the same decode as saw_paged_decode_int4
 * for callers that cannot allocate device memory.  The pages have no
 * counterpart: this is a deployment convenience of this library.
 *
 * Who needs it: a plugin or custom op whose host framework owns every device
 * allocation (it may not call cudaMalloc itself), or a latency-critical loop
 * that cannot afford cudaMalloc/cudaFree's device synchronisation.  The split-K scratch comes
 * from a fixed 4 MiB array in device memory declared by the library itself;
 * the caller passes only inputs and outputs (arguments as in
 * saw_paged_decode_int4, without the workspace).
 *
 *  - Limit: the plan's scratch (saw_decode_workspace_bytes) must be at most
 *    4 MiB; a larger plan returns SAW_ERR_UNSUPPORTED before any launch
 *    (use saw_paged_decode_int4, or a larger pages_per_split).
 *  - Memory: every GPU that loads the library holds the 4 MiB until the
 *    process exits.  No cudaMalloc/cudaFree is ever called.
 *  - Set-up: the first call on a device looks up the array's device address
 *    (cudaGetSymbolAddress, with that device current) and keeps it.
 *  - Sharing: all calls on a device share the array, so calls whose kernels
 *    may overlap on the GPU (different streams without ordering) race.
 *    Each call first clears the merge's counter words in it
 *    (cudaMemsetAsync on `stream`); the rest needs no clearing.
 */
int32_t saw_paged_decode_int4_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* seq_lens, int32_t num_seqs,
                                      int32_t max_seq_len, int32_t num_q_heads,
                                      int32_t num_kv_heads, int32_t head_dim, int32_t num_pages,
                                      int32_t page_size, int32_t rotate_k, int32_t rotate_v,
                                      int32_t block_h, float sm_scale, float* out,
                                      int32_t pages_per_split, int32_t* dev_status, void* stream);

/*
 * saw_prefill_attn_int4 -- chunked-prefill attention over the INT4 cache.
 *
 * Pages: youngju.dev "INT4 KV-cache quantization", "Why the KV Cache Is the
 * Real Bottleneck", and gist.science "SAW-INT4", s.1: the method has to work
 * inside engines that run fused attention over paged KV.  Reading: the
 * query of the token at position p of its sequence attends causally to that
 * sequence's cached tokens 0..p; dequantization, q rotation and the inverse
 * V rotation are those of saw_paged_decode_int4.  Append the chunk's K/V
 * with saw_quantize_append first (same stream).
 *
 *  q             device bfloat16 [total_q][num_q_heads][head_dim]: the query
 *                rows of every sequence's chunk, sequence after sequence.
 *  cu_q_lens     device int32 [num_seqs + 1]: rows cu_q_lens[b] ..
 *                cu_q_lens[b+1] - 1 belong to sequence b and are its last
 *                q_len_b = cu_q_lens[b+1] - cu_q_lens[b] tokens, so row i sits
 *                at position seq_lens[b] - q_len_b + (i - cu_q_lens[b]).
 *  seq_lens      device int32 [num_seqs]: cached tokens, the chunk included.
 *  max_q_len     a bound on every q_len_b (sizes the grid; <= max_seq_len).
 *  k/v caches, block tables, rotation and block_h, sm_scale (0 = 1/sqrt(D)):
 *                as in saw_paged_decode_int4.
 *  out           device float32 [total_q][num_q_heads][head_dim].
 *
 * No workspace.  head_dim 128 and page_size 16/32/64 (else
 * SAW_ERR_UNSUPPORTED); any number of q-heads per kv-head.  A sequence
 * whose q_len, seq_len or cu_q_lens entries are inconsistent (q_len < 0,
 * q_len > seq_len, q_len > max_q_len, seq_len > max_seq_len, rows beyond
 * total_q) is skipped and
 * SAW_ERR_DEVICE_INDEX is stored in *dev_status; a bad page id is skipped
 * and reported the same way; a copy that never lands ends the wait after
 * about a second with SAW_ERR_DEVICE_TIMEOUT.  Asynchronous on `stream`.
 */
int32_t saw_prefill_attn_int4(const void* q, const int32_t* cu_q_lens, const void* k_cache,
                              const void* v_cache, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                              int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                              int32_t head_dim, int32_t num_pages, int32_t page_size,
                              int32_t rotate_k, int32_t rotate_v, int32_t block_h, float sm_scale,
                              float* out, int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * Format variants.  The fused-kernel diagram of youngju.dev ("The System Is
 * the Design -- A Fused Kernel") feeds the kernel binary16 ("fp16") K and V;
 * engines also run in bfloat16.  The pages fix one scale per token but not
 * the storage format of the (scale, zero) pair.  The *_ex calls below are
 * the calls above with one extra argument, `formats`, an OR of:
 *
 *   SAW_FMT_F16_INPUT  q, K and V (and k_new, v_new) are binary16 instead of
 *                      bfloat16.  Both widen to binary32 exactly, so every
 *                      rule after that step is unchanged.
 *   SAW_FMT_BF16_META  the caches' per-row words hold {scale, zero} as
 *                      bfloat16 instead of binary16 (same place, same
 *                      order).  zero = bfloat16 round-down(min), scale =
 *                      bfloat16 round-up((max - zero)/15), both saturating
 *                      at +-(2^128 - 2^120), a zero stored as +0, and a
 *                      nonzero scale raised to at least 2^-126 (so that
 *                      1/scale is finite); codes as before.  A cache must be
 *                      written and read with the same metadata format.
 *
 * formats 0 is the plain call.  Any other bit: SAW_ERR_INVALID_ARG, before
 * anything is enqueued.
 * Supported shapes are those of the plain calls (all head dims for append
 * and decode; head_dim 128 for the decode step and the prefill).
 * Precision note: the head_dim-128 decode and the prefill carry p * scale_V
 * as a binary16 MMA operand, as they do for binary16 metadata, so their
 * error bound assumes V scales below 65504 (rows spanning less than about
 * 9.8e5); the head_dim 64/256 decode computes in binary32 throughout.
 * ------------------------------------------------------------------------ */
#define SAW_FMT_F16_INPUT 1
#define SAW_FMT_BF16_META 2

int32_t saw_quantize_append_ex(const void* k, const void* v, int64_t k_token_stride,
                               int64_t v_token_stride, const int32_t* slot_mapping,
                               int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                               void* k_cache, void* v_cache, int32_t num_pages,
                               int32_t page_size, int32_t rotate_k, int32_t rotate_v,
                               int32_t block_h, int32_t formats, int32_t* dev_status,
                               void* stream);

int32_t saw_paged_decode_int4_ex(const void* q, const void* k_cache, const void* v_cache,
                                 const int32_t* block_tables, int32_t max_blocks_per_seq,
                                 const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                                 int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                 int32_t num_pages, int32_t page_size, int32_t rotate_k,
                                 int32_t rotate_v, int32_t block_h, float sm_scale, float* out,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t pages_per_split, int32_t formats, int32_t* dev_status,
                                 void* stream);

int32_t saw_decode_step_ex(const void* q, const void* k_new, const void* v_new, void* k_cache,
                           void* v_cache, const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                           int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                           int32_t num_pages, int32_t page_size, int32_t rotate_k,
                           int32_t rotate_v, int32_t block_h, float sm_scale, float* out,
                           void* workspace, size_t workspace_bytes, int32_t pages_per_split,
                           int32_t flags, int32_t formats, int32_t* dev_status, void* stream);

int32_t saw_paged_decode_int4_noalloc_ex(const void* q, const void* k_cache,
                                         const void* v_cache, const int32_t* block_tables,
                                         int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                         int32_t num_seqs, int32_t max_seq_len,
                                         int32_t num_q_heads, int32_t num_kv_heads,
                                         int32_t head_dim, int32_t num_pages, int32_t page_size,
                                         int32_t rotate_k, int32_t rotate_v, int32_t block_h,
                                         float sm_scale, float* out, int32_t pages_per_split,
                                         int32_t formats, int32_t* dev_status, void* stream);

int32_t saw_prefill_attn_int4_ex(const void* q, const int32_t* cu_q_lens, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 int32_t max_blocks_per_seq, const int32_t* seq_lens,
                                 int32_t num_seqs, int32_t total_q, int32_t max_q_len,
                                 int32_t max_seq_len, int32_t num_q_heads, int32_t num_kv_heads,
                                 int32_t head_dim, int32_t num_pages, int32_t page_size,
                                 int32_t rotate_k, int32_t rotate_v, int32_t block_h,
                                 float sm_scale, float* out, int32_t formats,
                                 int32_t* dev_status, void* stream);

/* ------------------------------------------------------------------------
 * BF16 baseline.  gist.science "SAW-INT4: System-Aware 4-Bit KV-Cache
 * Quantization for Real-World LLM Serving", s.4 measures SAW-INT4's serving
 * throughput against an unquantized BF16 KV cache.  These two calls are that
 * baseline at the kernel level: the same paging and split-K decode, over a
 * cache of bfloat16 rows, so that INT4 and BF16 can be timed side by side.
 *
 * Cache layout, per layer and tensor (K and V separately):
 *   [num_pages][num_kv_heads][page_size][head_dim] bfloat16, rows of 256 B
 *   (head_dim 128).  Token t of a sequence lives in page block_tables[b][t /
 *   page_size], row t % page_size.  Owned by the caller; 16-byte aligned.
 * ------------------------------------------------------------------------ */

/* Bytes of one BF16 cache tensor; 0 for a nonpositive size. */
size_t saw_bf16_cache_bytes(int32_t num_pages, int32_t page_size, int32_t num_kv_heads,
                            int32_t head_dim);

/*
 * saw_bf16_append -- copy the bfloat16 rows k[t][h][:] (and v, if not NULL)
 * to slot slot_mapping[t] of the BF16 cache, unchanged.  Argument meaning,
 * strides (in elements, multiples of 8), the -1 padding slot and the
 * out-of-range rule (skipped, SAW_ERR_DEVICE_INDEX in *dev_status) are those
 * of saw_quantize_append.  head_dim must be 128 and page_size 16, 32 or 64
 * (else SAW_ERR_UNSUPPORTED).  Asynchronous on `stream`.
 */
int32_t saw_bf16_append(const void* k, const void* v, int64_t k_token_stride,
                        int64_t v_token_stride, const int32_t* slot_mapping, int32_t num_tokens,
                        int32_t num_kv_heads, int32_t head_dim, void* k_cache, void* v_cache,
                        int32_t num_pages, int32_t page_size, int32_t* dev_status, void* stream);

/*
 * Bytes of device workspace saw_paged_decode_bf16 needs for this shape (its
 * own split plan: one CTA per SM, at least 1024 tokens per split); 0 if it
 * needs none or the shape is invalid.  Zero-fill it before its first use;
 * each call leaves it ready for the next.
 */
size_t saw_decode_bf16_workspace_bytes(int32_t num_seqs, int32_t num_q_heads,
                                       int32_t num_kv_heads, int32_t head_dim, int32_t page_size,
                                       int32_t max_seq_len);

/*
 * saw_paged_decode_bf16 -- out[b][h][:] = softmax(sm_scale * K_b q_bh) V_b
 * over the seq_lens[b] cached tokens of kv-head h / (num_q_heads /
 * num_kv_heads), K and V read from the BF16 cache (no rotation, no
 * quantization).  q: bfloat16 [num_seqs][num_q_heads][128]; out: float32,
 * same shape.  Other arguments, sequences of length 0 (output zero), the
 * device-side index and timeout reports, and the return codes are those of
 * saw_paged_decode_int4.  Asynchronous on `stream`.
 */
int32_t saw_paged_decode_bf16(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t num_pages, int32_t page_size, float sm_scale, float* out,
                              void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream);

#ifdef __cplusplus
}
#endif

#endif /* SAW_INT4_H */
