// decode_static_scratch.cu -- saw_paged_decode_int4_noalloc: the decode entry
// point for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc: a plugin or custom op inside an
// inference server whose framework owns every device allocation (the
// plugin may not allocate on its own), or a latency-critical loop that must
// not pay cudaMalloc/cudaFree's implicit device synchronisation.  This entry point takes the split-K
// scratch from a fixed array in device memory that the library itself
// declares, so the caller passes only inputs and outputs.
//
// The array is kStaticScratchBytes (4 MiB).  Every GPU that loads the
// library holds it until the process exits.  All calls on a device share
// it, so two calls whose kernels overlap on the GPU (different streams, no
// ordering between them) race on it.
#include <mutex>

#include "saw_int4.h"
#include "saw_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(4) << 20;

// One copy per device, for the life of the process.
__device__ __align__(256) unsigned char g_decode_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::once_flag g_once[kMaxDevices];
void* g_scratch_ptr[kMaxDevices];
cudaError_t g_scratch_err[kMaxDevices];

// The host-side name of a __device__ array is only a stand-in, not a device
// address: a kernel handed it would fault or read host memory.  The real
// address is looked up once per device, with that device current.
int32_t scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SAW_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SAW_ERR_UNSUPPORTED;
  std::call_once(g_once[dev], [dev] {
    void* p = nullptr;
    g_scratch_err[dev] = cudaGetSymbolAddress(&p, g_decode_scratch);
    g_scratch_ptr[dev] = p;
  });
  if (g_scratch_err[dev] != cudaSuccess || g_scratch_ptr[dev] == nullptr) return SAW_ERR_CUDA;
  *out = g_scratch_ptr[dev];
  return SAW_OK;
}

}  // namespace

extern "C" int32_t saw_paged_decode_int4_noalloc_ex(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_pages,
    int32_t page_size, int32_t rotate_k, int32_t rotate_v, int32_t block_h, float sm_scale,
    float* out, int32_t pages_per_split, int32_t formats, int32_t* dev_status, void* stream) {
  if (formats & ~int32_t(SAW_FMT_F16_INPUT | SAW_FMT_BF16_META)) return SAW_ERR_INVALID_ARG;
  const size_t need = saw_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 page_size, max_seq_len, pages_per_split);
  if (need > kStaticScratchBytes) return SAW_ERR_UNSUPPORTED;
  // Every argument check runs before anything is enqueued, so a call that
  // fails leaves the stream (and the shared array) untouched.  The checks
  // only need to know that a large enough workspace exists: a stand-in
  // address is passed, never dereferenced, and replaced below.
  saw::DecodeParams p{};
  void* const stand_in = reinterpret_cast<void*>(uintptr_t(256));
  const int32_t rc = saw::prepare_decode(
      p, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs, max_seq_len,
      num_q_heads, num_kv_heads, head_dim, num_pages, page_size, rotate_k, rotate_v, block_h,
      sm_scale, out, need > 0 ? stand_in : nullptr, need > 0 ? kStaticScratchBytes : 0,
      pages_per_split, formats, dev_status);
  if (rc != SAW_OK || num_seqs == 0) return rc;
  if (need > 0) {
    void* scratch = nullptr;
    const int32_t rs = scratch_for_current_device(&scratch);
    if (rs != SAW_OK) return rs;
    saw::bind_decode_workspace(p, scratch);
    // The merge counts finished splits in the first words of the array;
    // they must start at zero, so clear them (the split partials need no
    // clearing: every partial the merge reads is written earlier in the call).
    const size_t tb = saw::decode_ticket_bytes(num_seqs, num_kv_heads);
    if (cudaMemsetAsync(scratch, 0, tb, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return SAW_ERR_CUDA;
  }
  const cudaError_t err = saw::launch_decode_any(p, static_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? SAW_OK : SAW_ERR_CUDA;
}

extern "C" int32_t saw_paged_decode_int4_noalloc(
    const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
    int32_t max_blocks_per_seq, const int32_t* seq_lens, int32_t num_seqs, int32_t max_seq_len,
    int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim, int32_t num_pages,
    int32_t page_size, int32_t rotate_k, int32_t rotate_v, int32_t block_h, float sm_scale,
    float* out, int32_t pages_per_split, int32_t* dev_status, void* stream) {
  return saw_paged_decode_int4_noalloc_ex(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                          seq_lens, num_seqs, max_seq_len, num_q_heads,
                                          num_kv_heads, head_dim, num_pages, page_size, rotate_k,
                                          rotate_v, block_h, sm_scale, out, pages_per_split, 0,
                                          dev_status, stream);
}
