// variants.cu -- the SAW-INT4 quantize-append at head_dim 64 and 256
// (rotation blocks up to h = 256).
//
// Pages: youngju.dev "INT4 KV-cache quantization", "Why Naive INT4 Breaks"
// (one scale per token), "The Rotation Trick -- Block-Diagonal Hadamard"
// (blocks of h); gist.science "SAW-INT4", s.2.  The method is stated for any
// head size; the head_dim-128 append (quantize_append.cu) is specialised for
// 128, and this serves the other sizes with the same cache layout (chunk =
// P*D/2 code bytes, then P words {s, z}, binary16 or bfloat16) and the same
// bits, for bfloat16 or binary16 input rows.  (The decode at these sizes is
// paged_decode.cu built for head_dim 64 and 256.)
//
//  * Small appends (up to 4096 rows, e.g. a decode step): one warp per
//    (token, kv-head) row, lane l holding elements E l .. E l + E - 1
//    (E = D/32).  Bulk appends run the tiled kernels of quantize_append.cu
//    (one thread per row at head_dim 64, four per row at 256).  The butterfly is the ascending-stride
//    sequence of RN(a + b), RN(a - b) steps -- strides below E inside a lane,
//    the rest across lanes -- then one RN multiply by binary32(1/sqrt h), so
//    the codes and (s, z) are the oracle's to the bit, as in the 128 path.
#include "saw_device.cuh"
#include "saw_int4.h"
#include "saw_quant_row.cuh"

namespace saw {
namespace {

constexpr uint32_t kAll = 0xFFFFFFFFu;
constexpr int kVarRowsPerCta = 4;

template <int D, int H>
__global__ void __launch_bounds__(32 * kVarRowsPerCta) quantize_append_var_kernel(
    const AppendParams p) {
  pdl_wait_then_release();
  constexpr int E = D / 32;
  const int lane = threadIdx.x & 31;
  const int hkv = p.num_kv_heads;
  const int64_t rows = int64_t(p.num_tokens) * hkv;
  const int64_t gw = int64_t(blockIdx.x) * kVarRowsPerCta + (threadIdx.x >> 5);
  if (gw >= rows * p.num_tensors) return;
  const int tensor = gw >= rows ? 1 : 0;
  const int64_t row = gw - tensor * rows;
  const int t = int(row / hkv), hd = int(row - int64_t(t) * hkv);
  const int32_t slot = p.slot_mapping[t];
  if (slot == -1) return;
  if (slot < 0 || int64_t(slot) >= p.num_slots) {
    if (lane == 0) report(p.dev_status, SAW_ERR_DEVICE_INDEX);
    return;
  }
  // (selects, not p.x[tensor]: indexing the parameter arrays would copy them to the stack)
  const uint16_t* src = (tensor ? p.src[1] : p.src[0]) +
                        int64_t(t) * (tensor ? p.stride[1] : p.stride[0]) + int64_t(hd) * D + E * lane;
  const bool f16 = p.in_f16 != 0;
  float x[E];
  if (E == 2) {
    const uint32_t w = *reinterpret_cast<const uint32_t*>(src);
    x[0] = in_lo(w, f16);
    x[1] = in_hi(w, f16);
  } else {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < E / 2; ++j) {
      x[2 * j] = in_lo(ws[j], f16);
      x[2 * j + 1] = in_hi(ws[j], f16);
    }
  }
  if ((tensor ? p.rotate[1] : p.rotate[0]) != 0) {
#pragma unroll
    for (int s = 1; s < E && s < H; s <<= 1) {
#pragma unroll
      for (int i = 0; i < E; ++i)
        if (!(i & s)) {
          const float a = x[i], b = x[i + s];
          x[i] = __fadd_rn(a, b);
          x[i + s] = __fsub_rn(a, b);
        }
    }
#pragma unroll
    for (int s = E; s < H; s <<= 1) {
      const int m = s / E;
      const bool upper = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < E; ++i) {
        const float o = __shfl_xor_sync(kAll, x[i], m);
        x[i] = upper ? __fsub_rn(o, x[i]) : __fadd_rn(x[i], o);
      }
    }
#pragma unroll
    for (int i = 0; i < E; ++i) x[i] = __fmul_rn(x[i], p.c_h);
  }
  float mn = x[0], mx = x[0];
#pragma unroll
  for (int i = 1; i < E; ++i) {
    mn = fminf(mn, x[i]);
    mx = fmaxf(mx, x[i]);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(kAll, mn, m));
    mx = fmaxf(mx, __shfl_xor_sync(kAll, mx, m));
  }
  const RowMeta m = row_meta(mn, mx, p.meta_bf16 != 0);
  const uint16_t zb = m.zb, sb = m.sb;
  uint32_t codes = 0;
#pragma unroll
  for (int i = 0; i < E; ++i) {
    int q = __float2int_rn(__fmul_rn(__fsub_rn(x[i], m.z), m.rcp));
    q = min(max(q, 0), 15);
    codes |= uint32_t(q) << (4 * i);
  }
  const int P = p.page_size;
  const int page = slot / P, off = slot - page * P;
  uint8_t* chunk = (tensor ? p.cache[1] : p.cache[0]) + (int64_t(page) * hkv + hd) * int64_t(P * (D / 2 + 4));
  if (E == 2)
    chunk[off * (D / 2) + lane] = uint8_t(codes);
  else
    reinterpret_cast<uint32_t*>(chunk + off * (D / 2))[lane] = codes;
  if (lane == 0)
    *reinterpret_cast<uint32_t*>(chunk + P * (D / 2) + 4 * off) = uint32_t(sb) | (uint32_t(zb) << 16);
}

template <int D, int H>
cudaError_t launch_append_var_h(const AppendParams& p, cudaStream_t stream) {
  const int64_t warps = int64_t(p.num_tokens) * p.num_kv_heads * p.num_tensors;
  const dim3 grid(unsigned((warps + kVarRowsPerCta - 1) / kVarRowsPerCta));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(32 * kVarRowsPerCta);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, quantize_append_var_kernel<D, H>, p);
}

template <int D>
cudaError_t launch_append_var_d(const AppendParams& p, int h, cudaStream_t stream) {
  switch (h) {
    case 16: return launch_append_var_h<D, 16>(p, stream);
    case 32: return launch_append_var_h<D, 32>(p, stream);
    case 64: return launch_append_var_h<D, 64>(p, stream);
    case 128: return D >= 128 ? launch_append_var_h<D, (D >= 128 ? 128 : 64)>(p, stream) : cudaErrorInvalidValue;
    case 256: return D >= 256 ? launch_append_var_h<D, (D >= 256 ? 256 : 64)>(p, stream) : cudaErrorInvalidValue;
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Rows from which a head_dim-64 or -256 append runs the tiled kernel.
constexpr int64_t kTiledMinRows = 4096;

cudaError_t launch_quantize_append_var(const AppendParams& p, int head_dim, cudaStream_t stream) {
  if (int64_t(p.num_tokens) * p.num_kv_heads == 0) return cudaSuccess;
  if (int64_t(p.num_tokens) * p.num_kv_heads > kTiledMinRows) {
    if (head_dim == 64) return launch_quantize_append_tiled64(p, p.num_tensors, stream);
    if (head_dim == 256) return launch_quantize_append_tiled256(p, p.num_tensors, stream);
  }
  const bool any_rot = p.rotate[0] || (p.num_tensors > 1 && p.rotate[1]);
  const int h = any_rot ? p.block_h : 16;  // unrotated: h is not used
  switch (head_dim) {
    case 64: return launch_append_var_d<64>(p, h, stream);
    case 256: return launch_append_var_d<256>(p, h, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace saw
