// saw_quant_row.cuh -- the token-wise INT4 quantizer of one (token, kv-head)
// row, shared by the append kernels and the fused decode-step kernel so that
// every path writes the same bytes.
//
// Pages: youngju.dev "INT4 KV-cache quantization" (English), "Why Naive INT4
// Breaks" (one scale per token) and "The Rotation Trick -- Block-Diagonal
// Hadamard"; gist.science "SAW-INT4 ...", s.2.  Readings where the pages are
// silent (stated in include/saw_int4.h): Sylvester butterfly with ascending
// strides, then binary32(1/sqrt h); zero = fp16 round-down(min), scale =
// fp16 round-up((max - zero)/15), saturating, a zero stored as +0; codes
// round-half-even of (y - zero) * (1/scale), clamped to 0..15.  Every binary32
// step is an explicit round-to-nearest intrinsic, so no contraction can
// change a bit whatever the translation unit's FMA setting.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>

#include "saw_device.cuh"

namespace saw {

__device__ __forceinline__ uint16_t f16_round_down_sat(float x) {
  x = fminf(fmaxf(x, -65504.0f), 65504.0f);
  const uint16_t b = __half_as_ushort(__float2half_rd(x));
  return (b & 0x7FFFu) ? b : uint16_t(0);  // any zero is stored as +0
}

__device__ __forceinline__ uint16_t f16_round_up_sat(float x) {
  x = fminf(fmaxf(x, -65504.0f), 65504.0f);
  const uint16_t b = __half_as_ushort(__float2half_ru(x));
  return (b & 0x7FFFu) ? b : uint16_t(0);
}

__device__ __forceinline__ float f16_bits_to_f32(uint16_t b) {
  return __half2float(__ushort_as_half(b));
}

// The bfloat16 metadata variant: the same directed rounding, saturating at
// the largest finite bfloat16 (2^128 - 2^120), a zero stored as +0.
constexpr float kBf16Max = 3.38953139e38f;
constexpr uint16_t kBf16MinNormal = 0x0080;  // 2^-126

__device__ __forceinline__ uint16_t bf16_round_down_sat(float x) {
  x = fminf(fmaxf(x, -kBf16Max), kBf16Max);
  const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_rd(x));
  return (b & 0x7FFFu) ? b : uint16_t(0);
}

__device__ __forceinline__ uint16_t bf16_round_up_sat(float x) {
  x = fminf(fmaxf(x, -kBf16Max), kBf16Max);
  const uint16_t b = __bfloat16_as_ushort(__float2bfloat16_ru(x));
  return (b & 0x7FFFu) ? b : uint16_t(0);
}

// (zero, scale) of a row from its binary32 min and max: zero rounded down,
// scale = (max - zero)/15 rounded up.  A nonzero bfloat16 scale is at least
// 2^-126, so that its reciprocal stays finite.  `fast` is set when no code
// can need the clamp -- the zero is not below every element only when min
// saturated, and the scale only overflows when it saturated -- and, for
// bfloat16 metadata, the scale is at most 2^101, so that 1/s times 2^-24 is
// still a normal binary32 number (the tiled kernel's fast path scales the
// reciprocal by 2^-24 and relies on that product being exact).
struct RowMeta {
  uint16_t zb, sb;
  float z, rcp;
  bool fast;
};

__device__ __forceinline__ RowMeta row_meta(float mn, float mx, bool bfm) {
  RowMeta m;
  const float lim = bfm ? 0x1p100f : 65504.0f;
  m.zb = bfm ? bf16_round_down_sat(mn) : f16_round_down_sat(mn);
  m.z = bfm ? __uint_as_float(uint32_t(m.zb) << 16) : f16_bits_to_f32(m.zb);
  const float step = __fdiv_rn(__fsub_rn(mx, m.z), 15.0f);
  uint16_t sb = bfm ? bf16_round_up_sat(step) : f16_round_up_sat(step);
  if (bfm && step > 0.0f && sb < kBf16MinNormal) sb = kBf16MinNormal;
  m.sb = sb;
  const float sv = bfm ? __uint_as_float(uint32_t(sb) << 16) : f16_bits_to_f32(sb);
  m.rcp = (sv == 0.0f) ? 0.0f : __frcp_rn(sv);
  // With z <= every element and an unsaturated scale: 0 <= y - z <= max - z
  // and r <= (1 + 2^-24) / s with s >= (max - z) / 15 (1 - 2^-24), so
  // (y - z) * r stays below 15.5 and no clamp can bite.  (For bfloat16 the
  // bound 2^100 on min and step is tighter than saturation needs: it also
  // keeps s <= 2^101.)
  m.fast = (mn >= -lim) && (step <= lim);
  return m;
}

// One warp quantizes one row of kHeadDim bfloat16 (binary16 with f16in)
// values, with binary16 (bfloat16 with bfm) metadata: lane l holds
// elements 4l..4l+3 and returns their four codes (bits 4e..4e+3 = element
// 4l+e, i.e. bytes 2l and 2l+1 of the packed row).  *meta receives
// (scale | zero << 16) as binary16 bits, identical in every lane.  The
// butterfly is the same ascending-stride sequence of (a+b, a-b) steps as a
// scalar loop -- strides 1 and 2 inside a lane, 4..h/2 across lanes.
__device__ __forceinline__ uint16_t warp_quantize_row(const uint16_t* __restrict__ row,
                                                      bool rotate, int h, float c_h, int lane,
                                                      uint32_t* meta, bool f16in, bool bfm) {
  const uint2 raw = *reinterpret_cast<const uint2*>(row + 4 * lane);
  float x[4] = {in_lo(raw.x, f16in), in_hi(raw.x, f16in), in_lo(raw.y, f16in),
                in_hi(raw.y, f16in)};
  if (rotate) {
    const float a0 = __fadd_rn(x[0], x[1]), a1 = __fsub_rn(x[0], x[1]);
    const float a2 = __fadd_rn(x[2], x[3]), a3 = __fsub_rn(x[2], x[3]);
    x[0] = __fadd_rn(a0, a2);
    x[2] = __fsub_rn(a0, a2);
    x[1] = __fadd_rn(a1, a3);
    x[3] = __fsub_rn(a1, a3);
    // the lower element of a pair gets a + b, the upper a - b
    for (int len = 4; len < h; len *= 2) {
      const int mask = len >> 2;
      const bool upper = (lane & mask) != 0;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float o = __shfl_xor_sync(0xFFFFFFFFu, x[e], mask);
        x[e] = upper ? __fsub_rn(o, x[e]) : __fadd_rn(x[e], o);
      }
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) x[e] = __fmul_rn(x[e], c_h);
  }
  float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
  float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, m));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, m));
  }
  const RowMeta m = row_meta(mn, mx, bfm);
  uint32_t codes = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    int q = __float2int_rn(__fmul_rn(__fsub_rn(x[e], m.z), m.rcp));
    q = min(max(q, 0), 15);
    codes |= uint32_t(q) << (4 * e);
  }
  *meta = uint32_t(m.sb) | (uint32_t(m.zb) << 16);
  return uint16_t(codes);
}

// Programmatic dependent launch: wait until the previous kernel in the stream
// has completed (its writes visible), then let the next kernel start
// launching.  Both are no-ops for a launch without the PDL attribute.
__device__ __forceinline__ void pdl_wait_then_release() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

}  // namespace saw
