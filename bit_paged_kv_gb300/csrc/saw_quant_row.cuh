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

// One warp quantizes one row of kHeadDim bfloat16 values: lane l holds
// elements 4l..4l+3 and returns their four codes (bits 4e..4e+3 = element
// 4l+e, i.e. bytes 2l and 2l+1 of the packed row).  *meta receives
// (scale | zero << 16) as binary16 bits, identical in every lane.  The
// butterfly is the same ascending-stride sequence of (a+b, a-b) steps as a
// scalar loop -- strides 1 and 2 inside a lane, 4..h/2 across lanes.
__device__ __forceinline__ uint16_t warp_quantize_row(const uint16_t* __restrict__ row,
                                                      bool rotate, int h, float c_h, int lane,
                                                      uint32_t* meta) {
  const uint2 raw = *reinterpret_cast<const uint2*>(row + 4 * lane);
  float x[4] = {bf16_lo(raw.x), bf16_hi(raw.x), bf16_lo(raw.y), bf16_hi(raw.y)};
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
  const uint16_t zb = f16_round_down_sat(mn);
  const float z = f16_bits_to_f32(zb);
  const float step = __fdiv_rn(__fsub_rn(mx, z), 15.0f);
  const uint16_t sb = f16_round_up_sat(step);
  const float sv = f16_bits_to_f32(sb);
  const float r = (sv == 0.0f) ? 0.0f : __frcp_rn(sv);
  uint32_t codes = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    int q = __float2int_rn(__fmul_rn(__fsub_rn(x[e], z), r));
    q = min(max(q, 0), 15);
    codes |= uint32_t(q) << (4 * e);
  }
  *meta = uint32_t(sb) | (uint32_t(zb) << 16);
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
