// quantize_append.cu -- K1: fused block-diagonal Hadamard rotation, token-wise
// INT4 quantization and paged append (SAW-INT4).
//
// Pages: youngju.dev "INT4 KV-cache quantization" (English), "The Rotation
// Trick -- Block-Diagonal Hadamard" and the fused-kernel diagram in "The
// System Is the Design -- A Fused Kernel"; gist.science "SAW-INT4: System-
// Aware 4-Bit KV-Cache Quantization for Real-World LLM Serving", s.2
// "Metodologia".  The rounding rules are the readings stated in
// include/saw_int4.h; each binary32 step below is one explicit
// round-to-nearest intrinsic so that no contraction changes a bit.
//
// Mapping (bulk appends): one CTA quantizes 128 consecutive (token, kv-head)
// rows of one tensor (K or V, blockIdx.y).  Warps first stream the 32 KB tile from HBM
// with coalesced 16-byte loads into XOR-swizzled shared memory; then each
// thread owns one row: 128 binary32 values in registers, the butterfly runs
// without any shuffle, min/max reduce as a tree, and the 64 code bytes plus
// the 4-byte (scale, zero) word are stored into the page slot.
#include "saw_device.cuh"
#include "saw_int4.h"
#include "saw_quant_row.cuh"

namespace saw {
namespace {

constexpr int kRows = 128;       // rows per CTA, one per thread
constexpr int kRowBytes = kHeadDim * 2;

// In-register butterfly over each H-block of the row, strides 1, 2, ..., H/2,
// then one multiply by c = binary32(1/sqrt(H)).
template <int H>
__device__ __forceinline__ void rotate_row(float (&u)[kHeadDim], float c) {
#pragma unroll
  for (int len = 1; len < H; len *= 2) {
#pragma unroll
    for (int i = 0; i < kHeadDim; ++i) {
      if ((i & len) == 0) {
        const float a = u[i];
        const float b = u[i + len];
        u[i] = __fadd_rn(a, b);
        u[i + len] = __fsub_rn(a, b);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kHeadDim; ++i) u[i] = __fmul_rn(u[i], c);
}

// Row min and max as a balanced tree (exact: no rounding involved).
__device__ __forceinline__ void row_min_max(const float (&u)[kHeadDim], float& mn, float& mx) {
  float lo[kHeadDim / 2], hi[kHeadDim / 2];
#pragma unroll
  for (int i = 0; i < kHeadDim / 2; ++i) {
    lo[i] = fminf(u[2 * i], u[2 * i + 1]);
    hi[i] = fmaxf(u[2 * i], u[2 * i + 1]);
  }
#pragma unroll
  for (int n = kHeadDim / 4; n >= 1; n /= 2) {
#pragma unroll
    for (int i = 0; i < n; ++i) {
      lo[i] = fminf(lo[i], lo[i + n]);
      hi[i] = fmaxf(hi[i], hi[i + n]);
    }
  }
  mn = lo[0];
  mx = hi[0];
}

// Scale/zero from min/max, then codes, packed two per byte (even index low).
__device__ __forceinline__ uint32_t quantize_pack(const float (&u)[kHeadDim],
                                                  uint32_t (&packed)[kHeadDim / 8]) {
  float mn, mx;
  row_min_max(u, mn, mx);
  const uint16_t zb = f16_round_down_sat(mn);
  const float z = f16_bits_to_f32(zb);
  const float range = __fsub_rn(mx, z);
  const float step = __fdiv_rn(range, 15.0f);
  const uint16_t sb = f16_round_up_sat(step);
  const float s = f16_bits_to_f32(sb);
  const float r = (s == 0.0f) ? 0.0f : __frcp_rn(s);
#pragma unroll
  for (int w = 0; w < kHeadDim / 8; ++w) {
    uint32_t word = 0;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float v = __fmul_rn(__fsub_rn(u[8 * w + k], z), r);
      int q = __float2int_rn(v);  // round half to even
      q = min(max(q, 0), 15);
      word |= uint32_t(q) << (4 * k);
    }
    packed[w] = word;
  }
  return uint32_t(sb) | (uint32_t(zb) << 16);
}

template <int H>
__global__ void __launch_bounds__(kRows) quantize_append_kernel(const AppendParams p) {
  __shared__ __align__(16) uint8_t tile[kRows * kRowBytes];

  pdl_wait_then_release();
  const int tensor = blockIdx.y;
  const uint16_t* __restrict__ src = p.src[tensor];
  const int64_t stride = p.stride[tensor];
  const int hkv = p.num_kv_heads;
  const int num_rows = p.num_tokens * hkv;
  const int row0 = blockIdx.x * kRows;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Coalesced tile load: each instruction moves two 256-byte rows per warp.
#pragma unroll 4
  for (int it = 0; it < 16; ++it) {
    const int r = warp * 32 + it * 2 + (lane >> 4);
    const int ch = lane & 15;
    const int row = row0 + r;
    uint4 val = make_uint4(0u, 0u, 0u, 0u);
    if (row < num_rows) {
      const int t = row / hkv;
      const int hd = row - t * hkv;
      const uint4* g =
          reinterpret_cast<const uint4*>(src + int64_t(t) * stride + int64_t(hd) * kHeadDim) + ch;
      val = __ldg(g);
    }
    *reinterpret_cast<uint4*>(tile + r * kRowBytes + ((ch ^ (r & 15)) << 4)) = val;
  }
  __syncthreads();

  const int r = threadIdx.x;
  const int row = row0 + r;
  if (row >= num_rows) return;
  const int t = row / hkv;
  const int hd = row - t * hkv;
  const int32_t slot = p.slot_mapping[t];
  if (slot == -1) return;
  if (slot < 0 || int64_t(slot) >= p.num_slots) {
    report(p.dev_status, SAW_ERR_DEVICE_INDEX);
    return;
  }

  float u[kHeadDim];
#pragma unroll
  for (int ch = 0; ch < 16; ++ch) {
    const uint4 w = *reinterpret_cast<const uint4*>(tile + r * kRowBytes + ((ch ^ (r & 15)) << 4));
    u[8 * ch + 0] = bf16_lo(w.x);
    u[8 * ch + 1] = bf16_hi(w.x);
    u[8 * ch + 2] = bf16_lo(w.y);
    u[8 * ch + 3] = bf16_hi(w.y);
    u[8 * ch + 4] = bf16_lo(w.z);
    u[8 * ch + 5] = bf16_hi(w.z);
    u[8 * ch + 6] = bf16_lo(w.w);
    u[8 * ch + 7] = bf16_hi(w.w);
  }

  if (p.rotate[tensor]) rotate_row<H>(u, p.c_h);

  uint32_t packed[kHeadDim / 8];
  const uint32_t meta = quantize_pack(u, packed);

  const int P = p.page_size;
  const int page = slot / P;
  const int off = slot - page * P;
  uint8_t* chunk = p.cache[tensor] + (int64_t(page) * hkv + hd) * int64_t(P * (kHeadDim / 2 + 4));
  uint4* dst = reinterpret_cast<uint4*>(chunk + off * (kHeadDim / 2));
#pragma unroll
  for (int j = 0; j < 4; ++j)
    dst[j] = make_uint4(packed[4 * j], packed[4 * j + 1], packed[4 * j + 2], packed[4 * j + 3]);
  *reinterpret_cast<uint32_t*>(chunk + P * (kHeadDim / 2) + 4 * off) = meta;
}

// Small appends (a decode step appends one token: Hkv rows per tensor): one
// warp per row, lane l holding elements 4l..4l+3.  The butterfly is the same
// ascending-stride sequence of (a+b, a-b) steps as the row kernel -- strides
// 1 and 2 inside a lane, the rest across lanes with shuffles -- so every value,
// and therefore every stored byte, is identical.
constexpr int kWarpRowsPerCta = 4;

template <int H>
__global__ void __launch_bounds__(32 * kWarpRowsPerCta) quantize_append_warp_kernel(
    const AppendParams p) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int hkv = p.num_kv_heads;
  const int rows_per_tensor = p.num_tokens * hkv;
  const int gw = blockIdx.x * kWarpRowsPerCta + (threadIdx.x >> 5);
  const int tensor = gw / rows_per_tensor;
  const int row = gw - tensor * rows_per_tensor;
  if (tensor >= p.num_tensors) return;
  const int t = row / hkv;
  const int hd = row - t * hkv;
  const int32_t slot = p.slot_mapping[t];
  if (slot == -1) return;
  if (slot < 0 || int64_t(slot) >= p.num_slots) {
    if (lane == 0) report(p.dev_status, SAW_ERR_DEVICE_INDEX);
    return;
  }
  uint32_t meta;
  const uint16_t codes = warp_quantize_row(
      p.src[tensor] + int64_t(t) * p.stride[tensor] + int64_t(hd) * kHeadDim, p.rotate[tensor] != 0,
      H, p.c_h, lane, &meta);
  const int P = p.page_size;
  const int page = slot / P;
  const int off = slot - page * P;
  uint8_t* chunk = p.cache[tensor] + (int64_t(page) * hkv + hd) * int64_t(P * (kHeadDim / 2 + 4));
  reinterpret_cast<uint16_t*>(chunk + off * (kHeadDim / 2))[lane] = codes;
  if (lane == 0) *reinterpret_cast<uint32_t*>(chunk + P * (kHeadDim / 2) + 4 * off) = meta;
}

}  // namespace

// Rows up to which the warp-per-row kernel is used (small appends).
constexpr int kWarpPathMaxRows = 4096;

template <typename K>
cudaError_t launch_pdl(K kernel, dim3 grid, int threads, cudaStream_t stream, const AppendParams& p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

cudaError_t launch_quantize_append(const AppendParams& p, int num_tensors, cudaStream_t stream) {
  const int num_rows = p.num_tokens * p.num_kv_heads;
  if (num_rows == 0) return cudaSuccess;
  const bool any_rot = p.rotate[0] || (num_tensors > 1 && p.rotate[1]);
  const int h = any_rot ? p.block_h : kHeadDim;
  if (num_rows <= kWarpPathMaxRows) {
    // one warp per (tensor, row): K rows first, then V rows
    AppendParams q = p;
    q.num_tensors = num_tensors;
    const dim3 grid((num_rows * num_tensors + kWarpRowsPerCta - 1) / kWarpRowsPerCta);
    const int nt = 32 * kWarpRowsPerCta;
    switch (h) {
      case 16: return launch_pdl(quantize_append_warp_kernel<16>, grid, nt, stream, q);
      case 32: return launch_pdl(quantize_append_warp_kernel<32>, grid, nt, stream, q);
      case 64: return launch_pdl(quantize_append_warp_kernel<64>, grid, nt, stream, q);
      case 128: return launch_pdl(quantize_append_warp_kernel<128>, grid, nt, stream, q);
      default: return cudaErrorInvalidValue;
    }
  }
  dim3 grid((num_rows + kRows - 1) / kRows, num_tensors);
  switch (h) {
    case 16: return launch_pdl(quantize_append_kernel<16>, grid, kRows, stream, p);
    case 32: return launch_pdl(quantize_append_kernel<32>, grid, kRows, stream, p);
    case 64: return launch_pdl(quantize_append_kernel<64>, grid, kRows, stream, p);
    case 128: return launch_pdl(quantize_append_kernel<128>, grid, kRows, stream, p);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace saw
