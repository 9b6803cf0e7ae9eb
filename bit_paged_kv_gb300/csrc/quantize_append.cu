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
// Mapping (bulk appends): a persistent kernel, a few 128-thread CTAs per SM.
// A tile is 128 consecutive (token, kv-head) rows of one tensor (K or V),
// 32 KB of bfloat16.  Each CTA walks its tiles with two shared-memory
// buffers: every thread issues 16-byte asynchronous copies of the next tile
// into an XOR-swizzled layout while the current tile is being quantized, so
// HBM reads overlap the arithmetic.  Then each thread owns one row: 128
// binary32 values in registers, the butterfly runs two lanes at a time with
// packed f32x2 adds, min/max reduce three at a time, and the 64 code bytes
// plus the 4-byte (scale, zero) word are stored into the page slot.
#include <algorithm>

#include "saw_device.cuh"
#include "saw_int4.h"
#include "saw_quant_row.cuh"

namespace saw {
namespace {

constexpr int kTileRows = 128;  // rows per tile, one per thread
constexpr int kRowBytes = kHeadDim * 2;
constexpr int kTileBytes = kTileRows * kRowBytes;  // 32 KB
constexpr int kTileCtasPerSm = 3;

// ------------------------------------------------------------ PTX pieces

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// (a0, a1) <- (a0 + b0, a1 + b1) and (b0, b1) <- (a0 - b0, a1 - b1): two
// butterfly pairs per instruction, each lane an ordinary binary32 RN op.
__device__ __forceinline__ void bfly2(float& a0, float& a1, float& b0, float& b1) {
  asm("{\n\t.reg .b64 x, y, s, d;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "add.rn.f32x2 s, x, y;\n\tsub.rn.f32x2 d, x, y;\n\t"
      "mov.b64 {%0, %1}, s;\n\tmov.b64 {%2, %3}, d;\n\t}"
      : "+f"(a0), "+f"(a1), "+f"(b0), "+f"(b1));
}

__device__ __forceinline__ void mul2(float& a0, float& a1, float c) {
  asm("{\n\t.reg .b64 x, k;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 k, {%2, %2};\n\t"
      "mul.rn.f32x2 x, x, k;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(c));
}

__device__ __forceinline__ float min3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Codes of two elements when no clamp is needed (0 <= (y - z) * r <= 15 +
// a few ulp): v = RN(RN(y - z) * r) as in the scalar rule (two lanes per
// instruction), then v + 1.5 * 2^23 rounds to the nearest integer with ties
// to even in the low mantissa bits, so byte 0 of each result is the code
// (high bits 0x4B40....).  The magic add is a scalar RN add: it must round
// the already-rounded product, never be fused with the multiply.
__device__ __forceinline__ void codes2(float y0, float y1, float z, float r, uint32_t& t0,
                                       uint32_t& t1) {
  float v0, v1;
  asm("{\n\t.reg .b64 y, zz, rr;\n\t"
      "mov.b64 y, {%2, %3};\n\tmov.b64 zz, {%4, %4};\n\tmov.b64 rr, {%5, %5};\n\t"
      "sub.rn.f32x2 y, y, zz;\n\tmul.rn.f32x2 y, y, rr;\n\t"
      "mov.b64 {%0, %1}, y;\n\t}"
      : "=f"(v0), "=f"(v1)
      : "f"(y0), "f"(y1), "f"(z), "f"(r));
  t0 = __float_as_uint(__fadd_rn(v0, 12582912.0f));
  t1 = __float_as_uint(__fadd_rn(v1, 12582912.0f));
}

// q = n / d for 0 <= n < 2^31 with a host-computed multiplier (m, sh):
// m = ceil(2^sh / d), sh = 31 + ceil(log2 d), exact on that range.
__device__ __forceinline__ uint32_t div_rows(uint32_t n, uint32_t m, uint32_t sh) {
  return uint32_t((uint64_t(n) * m) >> sh);
}

// ------------------------------------------------------------ one row

// In-register butterfly over each H-block of the row, strides 1, 2, ..., H/2
// (stride 1 scalar, the rest two pairs per instruction), then one multiply
// by c = binary32(1/sqrt(H)).
template <int H>
__device__ __forceinline__ void rotate_row(float (&u)[kHeadDim], float c) {
#pragma unroll
  for (int i = 0; i < kHeadDim; i += 2) {
    const float a = u[i], b = u[i + 1];
    u[i] = __fadd_rn(a, b);
    u[i + 1] = __fsub_rn(a, b);
  }
#pragma unroll
  for (int len = 2; len < H; len *= 2) {
#pragma unroll
    for (int i = 0; i < kHeadDim; i += 2) {
      if ((i & len) == 0) bfly2(u[i], u[i + 1], u[i + len], u[i + len + 1]);
    }
  }
#pragma unroll
  for (int i = 0; i < kHeadDim; i += 2) mul2(u[i], u[i + 1], c);
}

// Row min and max, three at a time (exact: no rounding involved).
__device__ __forceinline__ void row_min_max(const float (&u)[kHeadDim], float& mn, float& mx) {
  float lo[43], hi[43];
#pragma unroll
  for (int i = 0; i < 42; ++i) {
    lo[i] = min3(u[3 * i], u[3 * i + 1], u[3 * i + 2]);
    hi[i] = max3(u[3 * i], u[3 * i + 1], u[3 * i + 2]);
  }
  lo[42] = fminf(u[126], u[127]);
  hi[42] = fmaxf(u[126], u[127]);
#pragma unroll
  for (int i = 0; i < 14; ++i) {
    lo[i] = min3(lo[3 * i], lo[3 * i + 1], lo[3 * i + 2]);
    hi[i] = max3(hi[3 * i], hi[3 * i + 1], hi[3 * i + 2]);
  }
  lo[14] = lo[42];
  hi[14] = hi[42];
#pragma unroll
  for (int i = 0; i < 5; ++i) {
    lo[i] = min3(lo[3 * i], lo[3 * i + 1], lo[3 * i + 2]);
    hi[i] = max3(hi[3 * i], hi[3 * i + 1], hi[3 * i + 2]);
  }
  mn = fminf(min3(lo[0], lo[1], lo[2]), fminf(lo[3], lo[4]));
  mx = fmaxf(max3(hi[0], hi[1], hi[2]), fmaxf(hi[3], hi[4]));
}

// Quantize the row and store its 64 code bytes (two codes per byte, even
// index in the low nibble) at dst; returns (scale | zero << 16).
__device__ __forceinline__ uint32_t quantize_store(const float (&u)[kHeadDim], uint4* dst) {
  float mn, mx;
  row_min_max(u, mn, mx);
  const uint16_t zb = f16_round_down_sat(mn);
  const float z = f16_bits_to_f32(zb);
  const float step = __fdiv_rn(__fsub_rn(mx, z), 15.0f);
  const uint16_t sb = f16_round_up_sat(step);
  const float s = f16_bits_to_f32(sb);
  const float r = (s == 0.0f) ? 0.0f : __frcp_rn(s);
  // No clamp can bite when z <= every element (min not below -65504) and
  // the scale did not saturate: then 0 <= y - z <= max - z and
  // r <= (1 + 2^-24) / s with s >= (max - z) / 15 (1 - 2^-24), so
  // (y - z) * r stays below 15.5.
  const bool fast = (mn >= -65504.0f) && (step <= 65504.0f);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    uint32_t word[4];
#pragma unroll
    for (int w4 = 0; w4 < 4; ++w4) {
      const int w = 4 * j + w4;
      if (fast) {
        uint32_t t[8];
#pragma unroll
        for (int e = 0; e < 4; ++e)
          codes2(u[8 * w + 2 * e], u[8 * w + 2 * e + 1], z, r, t[2 * e], t[2 * e + 1]);
        const uint32_t even = prmt(prmt(t[0], t[2], 0x0040u), prmt(t[4], t[6], 0x0040u), 0x5410u);
        const uint32_t odd = prmt(prmt(t[1], t[3], 0x0040u), prmt(t[5], t[7], 0x0040u), 0x5410u);
        word[w4] = even | (odd << 4);
      } else {
        uint32_t acc = 0;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const float v = __fmul_rn(__fsub_rn(u[8 * w + k], z), r);
          int q = __float2int_rn(v);  // round half to even
          q = min(max(q, 0), 15);
          acc |= uint32_t(q) << (4 * k);
        }
        word[w4] = acc;
      }
    }
    dst[j] = make_uint4(word[0], word[1], word[2], word[3]);
  }
  return uint32_t(sb) | (uint32_t(zb) << 16);
}

// ------------------------------------------------------------ tiled kernel

// Tiles 0 .. tiles_per_tensor-1 are K rows, the rest V rows.
template <int H>
__global__ void __launch_bounds__(kTileRows, kTileCtasPerSm)
    quantize_append_tiled_kernel(const AppendParams p, int tiles_per_tensor, int num_tiles) {
  extern __shared__ __align__(128) uint8_t tiles[];  // two tiles

  pdl_wait_then_release();
  const int tid = threadIdx.x;
  const int hkv = p.num_kv_heads;
  const int num_rows = p.num_tokens * hkv;

  // Copies of one tile: 16 per thread, 16 threads per 256-byte row; chunk c
  // of row r lands at 16 * (c ^ (r & 15)) so that the row-per-thread reads
  // below hit distinct banks.
  auto issue = [&](int tile, uint8_t* buf) {
    const int tensor = tile >= tiles_per_tensor ? 1 : 0;
    const int row0 = (tile - tensor * tiles_per_tensor) * kTileRows;
    const uint16_t* __restrict__ src = tensor ? p.src[1] : p.src[0];
    const int64_t stride = tensor ? p.stride[1] : p.stride[0];
    const int ch = tid & 15;
#pragma unroll
    for (int it = 0; it < kTileRows / 8; ++it) {
      const int r = it * 8 + (tid >> 4);
      const int row = row0 + r;
      if (row < num_rows) {
        const uint32_t t = div_rows(uint32_t(row), p.hkv_mul, p.hkv_shift);
        const uint32_t hd = uint32_t(row) - t * uint32_t(hkv);
        cp_async16(buf + r * kRowBytes + ((ch ^ (r & 15)) << 4),
                   src + int64_t(t) * stride + hd * kHeadDim + ch * 8);
      }
    }
  };

  int tile = blockIdx.x;
  if (tile < num_tiles) issue(tile, tiles);
  cp_async_commit();
  for (int k = 0; tile < num_tiles; ++k, tile += gridDim.x) {
    uint8_t* buf = tiles + (k & 1) * kTileBytes;
    const int nxt = tile + gridDim.x;
    if (nxt < num_tiles) issue(nxt, tiles + ((k + 1) & 1) * kTileBytes);
    cp_async_commit();

    const int tensor = tile >= tiles_per_tensor ? 1 : 0;
    const int row = (tile - tensor * tiles_per_tensor) * kTileRows + tid;
    const bool live = row < num_rows;
    uint32_t t = 0, hd = 0;
    int32_t slot = -1;
    if (live) {
      t = div_rows(uint32_t(row), p.hkv_mul, p.hkv_shift);
      hd = uint32_t(row) - t * uint32_t(hkv);
      slot = __ldg(p.slot_mapping + t);
    }
    cp_async_wait<1>();  // this thread's copies of the current tile landed
    __syncthreads();     // ... and everyone's

    if (live && slot != -1) {
      if (slot < 0 || int64_t(slot) >= p.num_slots) {
        report(p.dev_status, SAW_ERR_DEVICE_INDEX);
      } else {
        float u[kHeadDim];
        const int r = tid;
#pragma unroll
        for (int ch = 0; ch < 16; ++ch) {
          const uint4 w =
              *reinterpret_cast<const uint4*>(buf + r * kRowBytes + ((ch ^ (r & 15)) << 4));
          u[8 * ch + 0] = bf16_lo(w.x);
          u[8 * ch + 1] = bf16_hi(w.x);
          u[8 * ch + 2] = bf16_lo(w.y);
          u[8 * ch + 3] = bf16_hi(w.y);
          u[8 * ch + 4] = bf16_lo(w.z);
          u[8 * ch + 5] = bf16_hi(w.z);
          u[8 * ch + 6] = bf16_lo(w.w);
          u[8 * ch + 7] = bf16_hi(w.w);
        }
        if (tensor ? p.rotate[1] : p.rotate[0]) rotate_row<H>(u, p.c_h);
        const int P = p.page_size;
        const int page = slot >> p.page_shift;
        const int off = slot & (P - 1);
        uint8_t* chunk = (tensor ? p.cache[1] : p.cache[0]) +
                         (int64_t(page) * hkv + hd) * int64_t(chunk_bytes(P));
        const uint32_t meta =
            quantize_store(u, reinterpret_cast<uint4*>(chunk + off * (kHeadDim / 2)));
        *reinterpret_cast<uint32_t*>(chunk + P * (kHeadDim / 2) + 4 * off) = meta;
      }
    }
    __syncthreads();  // the buffer is refilled by the next-but-one issue
  }
  cp_async_wait<0>();
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
      (tensor ? p.src[1] : p.src[0]) + int64_t(t) * (tensor ? p.stride[1] : p.stride[0]) +
          int64_t(hd) * kHeadDim,
      (tensor ? p.rotate[1] : p.rotate[0]) != 0,
      H, p.c_h, lane, &meta);
  const int P = p.page_size;
  const int page = slot / P;
  const int off = slot - page * P;
  uint8_t* chunk = (tensor ? p.cache[1] : p.cache[0]) +
                   (int64_t(page) * hkv + hd) * int64_t(chunk_bytes(P));
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

template <typename K>
cudaError_t launch_tiled(K kernel, dim3 grid, cudaStream_t stream, const AppendParams& p,
                         int tiles_per_tensor, int num_tiles) {
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 2 * kTileBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kTileRows);
  cfg.dynamicSmemBytes = 2 * kTileBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p, tiles_per_tensor, num_tiles);
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
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const int tiles_per_tensor = (num_rows + kTileRows - 1) / kTileRows;
  const int num_tiles = tiles_per_tensor * num_tensors;
  const dim3 grid(std::min(num_tiles, sms * kTileCtasPerSm));
  AppendParams q = p;
  q.num_tensors = num_tensors;
  int lg = 0;
  while ((1 << lg) < q.num_kv_heads) ++lg;
  q.hkv_shift = uint32_t(31 + lg);
  q.hkv_mul = uint32_t(((uint64_t(1) << q.hkv_shift) + q.num_kv_heads - 1) / q.num_kv_heads);
  q.page_shift = 0;
  while ((1 << q.page_shift) < q.page_size) ++q.page_shift;
  switch (h) {
    case 16: return launch_tiled(quantize_append_tiled_kernel<16>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 32: return launch_tiled(quantize_append_tiled_kernel<32>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 64: return launch_tiled(quantize_append_tiled_kernel<64>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 128: return launch_tiled(quantize_append_tiled_kernel<128>, grid, stream, q, tiles_per_tensor, num_tiles);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace saw
