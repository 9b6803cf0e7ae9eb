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
// Mapping (bulk appends): a persistent kernel, two 256-thread CTAs per SM,
// each warp an independent worker.  A tile is 16 consecutive (token,
// kv-head) rows of one tensor (K or V), 4 KB of bfloat16.  Each warp walks
// its tiles through a private ring of three shared-memory buffers: its
// lanes issue 16-byte asynchronous copies of the tile two ahead into a
// swizzled layout while the current tile is being quantized, so HBM reads
// overlap the arithmetic, and no CTA-wide barrier is needed.  Two
// neighbouring threads own one row, 64 binary32 values each: butterfly
// strides up to 32 stay inside a thread (two lanes per packed f32x2
// instruction), stride 64 is one shuffle with the partner, min/max reduce
// in four chains three at a time, and each thread stores its 32 code
// bytes; the (scale, zero) word goes to the page's metadata run.  The same
// scheme serves head_dim 64 (one thread per row) and 256 (four per row)
// below.
#include <algorithm>

#include "saw_device.cuh"
#include "saw_int4.h"
#include "saw_quant_row.cuh"

namespace saw {
namespace {

constexpr int kTileRows = 16;                      // rows per warp tile (two threads per row)
constexpr int kHalfRow = kHeadDim / 2;             // elements per thread
constexpr int kRowBytes = kHeadDim * 2;
constexpr int kTileBytes = kTileRows * kRowBytes;  // 4 KB
constexpr int kTileStages = 3;                     // tiles in flight per warp
constexpr int kTileWarps = 8;                      // warps per CTA
constexpr int kTileThreads = 32 * kTileWarps;
constexpr int kTileCtasPerSm = 2;

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

// {a, b} as one 64-bit register pair, for the packed instructions' operands
// that are the same for a whole row (built once, not per instruction).
__device__ __forceinline__ uint64_t pair(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}

// (a0, a1) <- RN((a0, a1) * k)
__device__ __forceinline__ void mul2(float& a0, float& a1, uint64_t k) {
  asm("{\n\t.reg .b64 x;\n\t"
      "mov.b64 x, {%0, %1};\n\tmul.rn.f32x2 x, x, %2;\n\tmov.b64 {%0, %1}, x;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "l"(k));
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

// q = n / d for 0 <= n < 2^31 with a host-computed multiplier (m, sh):
// m = ceil(2^sh / d), sh = 31 + ceil(log2 d), exact on that range.
__device__ __forceinline__ uint32_t div_rows(uint32_t n, uint32_t m, uint32_t sh) {
  return uint32_t((uint64_t(n) * m) >> sh);
}

// ------------------------------------------------------------ half row
//
// Two neighbouring threads share a row.  Writing G0..G3 for its four
// 32-element quarters, the lower thread (h = 0) holds G0 in local elements
// 0..31 and G1 in 32..63; the upper thread (h = 1) holds G3 in 0..31 and G2
// in 32..63.  Strides up to 16 stay inside a quarter.  Stride 32 pairs local
// j with local 32 + j in both threads, and stride 64 pairs the lower
// thread's local j (G0) with the upper thread's local 32 + j (G2), and the
// upper thread's local j (G3) with the lower thread's 32 + j (G1): one
// shuffle of local 32 + j covers both.  In both steps the thread whose pair
// members sit in swapped roles computes the same two RN sums through
// x' = RN(sg * x + y), y' = RN(-sg * y + x) with sg = +-1 (exact products).
// After a stride-64 step the lower thread's local 32..63 hold G2 and the
// upper thread's hold G1.

// (x0, x1) and (y0, y1) <- RN(sg * x + y) and RN(-sg * y + x), with
// p = {sg, sg} and m = {-sg, -sg}.
__device__ __forceinline__ void bfly2_signed(float& x0, float& x1, float& y0, float& y1,
                                             uint64_t p, uint64_t m) {
  asm("{\n\t.reg .b64 x, y, a, b;\n\t"
      "mov.b64 x, {%0, %1};\n\tmov.b64 y, {%2, %3};\n\t"
      "fma.rn.f32x2 a, x, %4, y;\n\tfma.rn.f32x2 b, y, %5, x;\n\t"
      "mov.b64 {%0, %1}, a;\n\tmov.b64 {%2, %3}, b;\n\t}"
      : "+f"(x0), "+f"(x1), "+f"(y0), "+f"(y1)
      : "l"(p), "l"(m));
}

// Butterfly of the row's H-blocks (strides 1, 2, ..., H/2 in ascending
// order, every step an RN add or subtract), then one multiply by
// c = binary32(1/sqrt(H)).  The stride-1 step reads the input pairs
// straight from the loaded words: a mixed-precision add takes the even
// element as bfloat16 (binary16 with F16IN; exact widening either way) and
// the odd one as binary32.
template <int H, bool F16IN>
__device__ __forceinline__ void rotate_half(const uint32_t (&wd)[kHalfRow / 2],
                                            float (&u)[kHalfRow], float c, int h) {
#pragma unroll
  for (int i = 0; i < kHalfRow / 2; ++i) {
    if (F16IN) {
      const float odd = f16_hi(wd[i]);
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
          "add.rn.f32.f16 %0, lo, %3;\n\tsub.rn.f32.f16 %1, lo, %3;\n\t}"
          : "=f"(u[2 * i]), "=f"(u[2 * i + 1])
          : "r"(wd[i]), "f"(odd));
    } else {
      const float odd = bf16_hi(wd[i]);
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
          "add.rn.f32.bf16 %0, lo, %3;\n\tsub.rn.f32.bf16 %1, lo, %3;\n\t}"
          : "=f"(u[2 * i]), "=f"(u[2 * i + 1])
          : "r"(wd[i]), "f"(odd));
    }
  }
#pragma unroll
  for (int len = 2; len < (H < 32 ? H : 32); len *= 2) {
#pragma unroll
    for (int i = 0; i < kHalfRow; i += 2) {
      if ((i & len) == 0) bfly2(u[i], u[i + 1], u[i + len], u[i + len + 1]);
    }
  }
  const float sg = h ? -1.0f : 1.0f;
  const uint64_t sp = pair(sg, sg), sm = pair(-sg, -sg);
  if (H >= 64) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) bfly2_signed(u[j], u[j + 1], u[32 + j], u[33 + j], sp, sm);
  }
  if (H == 128) {
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float o0 = __shfl_xor_sync(0xFFFFFFFFu, u[32 + j], 1);
      const float o1 = __shfl_xor_sync(0xFFFFFFFFu, u[33 + j], 1);
      u[32 + j] = o0;
      u[33 + j] = o1;
      bfly2_signed(u[j], u[j + 1], u[32 + j], u[33 + j], sp, sm);
    }
  }
  const uint64_t cc = pair(c, c);
#pragma unroll
  for (int i = 0; i < kHalfRow; i += 2) mul2(u[i], u[i + 1], cc);
}

// Min and max of the whole row: 64 values here in four chains of 16, three
// values per instruction (exact, so the order is free), then (PAIR) the
// partner's.  The chains keep only eight partial results live beside u.
template <bool PAIR = true>
__device__ __forceinline__ void half_min_max(const float (&u)[kHalfRow], float& mn, float& mx) {
  float lo[4], hi[4];
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    lo[c] = min3(u[16 * c], u[16 * c + 1], u[16 * c + 2]);
    hi[c] = max3(u[16 * c], u[16 * c + 1], u[16 * c + 2]);
  }
#pragma unroll
  for (int k = 3; k < 15; k += 2) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      lo[c] = min3(lo[c], u[16 * c + k], u[16 * c + k + 1]);
      hi[c] = max3(hi[c], u[16 * c + k], u[16 * c + k + 1]);
    }
  }
  // element 15 of each chain joins the final combination
  mn = fminf(min3(min3(lo[0], lo[1], u[15]), min3(lo[2], lo[3], u[31]), u[47]), u[63]);
  mx = fmaxf(max3(max3(hi[0], hi[1], u[15]), max3(hi[2], hi[3], u[31]), u[47]), u[63]);
  if (PAIR) {
    mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
  }
}

// Codes of this thread's 64 elements, packed two per byte (even local index
// in the low nibble): words 0..3 hold local 0..31, words 4..7 local 32..63.
//
// Fast path (no clamp can bite, see the caller): with r24 = r * 2^-24 (exact),
// RN((y - z) * r24) = RN((y - z) * r) * 2^-24 whenever the result is normal,
// and below that the code is 0 either way.  Binary16 spaces its subnormals
// 2^-24 apart, so the RN conversion to binary16 of that value rounds
// (y - z) * r to the nearest integer with ties to even, and the code is the
// binary16 bit pattern itself.
__device__ __forceinline__ void quantize_half(const float (&u)[kHalfRow], float z, float r,
                                              bool fast, uint32_t (&word)[8]) {
  if (fast) {
    const float r24 = __fmul_rn(r, 5.9604644775390625e-08f);  // 2^-24
    const uint64_t zz = pair(z, z), rr = pair(r24, r24);
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      float v[8];
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        v[e] = u[8 * w + e];
        v[e + 1] = u[8 * w + e + 1];
        asm("{\n\t.reg .b64 y;\n\t"
            "mov.b64 y, {%0, %1};\n\t"
            "sub.rn.f32x2 y, y, %2;\n\tmul.rn.f32x2 y, y, %3;\n\t"
            "mov.b64 {%0, %1}, y;\n\t}"
            : "+f"(v[e]), "+f"(v[e + 1])
            : "l"(zz), "l"(rr));
      }
      // binary16 pairs (low half first): d[k] = c(a) | c(b) << 16 for
      // (a, b) = (0, 2), (1, 3), (4, 6), (5, 7)
      uint32_t d[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int a = (k & 1) + 4 * (k >> 1);
        const __half2 hv = __floats2half2_rn(v[a], v[a + 2]);
        d[k] = *reinterpret_cast<const uint32_t*>(&hv);
      }
      // bytes 0 and 2 of x: (c0 c1), (c2 c3); of y: (c4 c5), (c6 c7).  A code
      // of -0 (y = -0, z = +0) converts to 0x8000: its sign bit stays in the
      // discarded bytes 1 and 3 of d[0], d[2], and is masked off after the
      // shift for d[1], d[3].
      const uint32_t x = d[0] | ((d[1] << 4) & 0x00F000F0u);
      const uint32_t y = d[2] | ((d[3] << 4) & 0x00F000F0u);
      word[w] = prmt(x, y, 0x6420u);
    }
  } else {
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      uint32_t acc = 0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float v = __fmul_rn(__fsub_rn(u[8 * w + k], z), r);
        int q = __float2int_rn(v);  // round half to even
        q = min(max(q, 0), 15);
        acc |= uint32_t(q) << (4 * k);
      }
      word[w] = acc;
    }
  }
}

// ------------------------------------------------------------ tiled kernel

// Chunk c (16 bytes: elements 8c .. 8c+7) of tile row r sits in 16-byte slot
// c ^ (r & 3) of the row's 256 bytes: the copy (16 consecutive chunks of a
// row per half-warp) and the reads (rows r..r+3, both halves, chunks
// j and 8 + (j ^ 4) per phase) both hit 8 distinct bank groups.
__device__ __forceinline__ int chunk_slot(int r, int c) { return c ^ (r & 3); }

// Tiles 0 .. tiles_per_tensor-1 are K rows, the rest V rows.  Each warp is
// an independent worker with its own ring of kTileStages tiles: no CTA-wide
// barrier, so a warp waiting for its data never holds up the others.
// F16IN: the rows are binary16 instead of bfloat16; BFM: the (scale, zero)
// words are bfloat16 instead of binary16.
template <int H, bool F16IN, bool BFM>
__global__ void __launch_bounds__(kTileThreads, kTileCtasPerSm)
    quantize_append_tiled_kernel(const AppendParams p, int tiles_per_tensor, int num_tiles) {
  extern __shared__ __align__(128) uint8_t ring_all[];

  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t* ring = ring_all + warp * (kTileStages * kTileBytes);
  const int hkv = p.num_kv_heads;
  const int num_rows = p.num_tokens * hkv;

  // Copies of one tile: 8 per lane, 16 lanes per 256-byte row.  Copy `it`
  // of a lane lands in row r = 2 it + rl at slot ch ^ (r & 3), and r & 3 is
  // rl for even it and 2 + rl for odd it: two offsets per lane, fixed.
  const int ch = lane & 15;
  const int rl = lane >> 4;
  const int so_even = rl * kRowBytes + ((ch ^ rl) << 4);
  const int so_odd = rl * kRowBytes + ((ch ^ (2 | rl)) << 4);
  auto issue = [&](int tile, uint8_t* buf) {
    const int tensor = tile >= tiles_per_tensor ? 1 : 0;
    const int row0 = (tile - tensor * tiles_per_tensor) * kTileRows;
    const uint16_t* __restrict__ src = tensor ? p.src[1] : p.src[0];
    const int64_t stride = tensor ? p.stride[1] : p.stride[0];
    const bool full = row0 + kTileRows <= num_rows;
    if (full && stride == int64_t(hkv) * kHeadDim) {
      // contiguous rows: row i of the tile starts 128 elements after row i-1
      const uint16_t* g = src + (int64_t(row0) + rl) * kHeadDim + ch * 8;
#pragma unroll
      for (int it = 0; it < kTileRows / 2; ++it)
        cp_async16(buf + it * 2 * kRowBytes + ((it & 1) ? so_odd : so_even),
                   g + it * 2 * kHeadDim);
    } else {
#pragma unroll
      for (int it = 0; it < kTileRows / 2; ++it) {
        const int r = it * 2 + (lane >> 4);
        const int row = row0 + r;
        if (row < num_rows) {
          const uint32_t t = div_rows(uint32_t(row), p.hkv_mul, p.hkv_shift);
          const uint32_t hd = uint32_t(row) - t * uint32_t(hkv);
          cp_async16(buf + r * kRowBytes + (chunk_slot(r, ch) << 4),
                     src + int64_t(t) * stride + hd * kHeadDim + ch * 8);
        }
      }
    }
  };

  const int r = lane >> 1;  // this thread's row in the tile
  const int h = lane & 1;   // and its half
  const int step = int(gridDim.x) * kTileWarps;
  int tile = int(blockIdx.x) * kTileWarps + warp;
#pragma unroll
  for (int s = 0; s < kTileStages - 1; ++s) {
    const int pre = tile + s * step;
    if (pre < num_tiles) issue(pre, ring + s * kTileBytes);
    cp_async_commit();
  }
  int cur = 0;                  // ring slot of the current tile
  int ahead = kTileStages - 1;  // ring slot of the tile issued next
  for (; tile < num_tiles; tile += step) {
    uint8_t* buf = ring + cur * kTileBytes;
    const int nxt = tile + (kTileStages - 1) * step;
    if (nxt < num_tiles) issue(nxt, ring + ahead * kTileBytes);
    cp_async_commit();
    cur = (cur + 1 == kTileStages) ? 0 : cur + 1;
    ahead = (ahead + 1 == kTileStages) ? 0 : ahead + 1;

    const int tensor = tile >= tiles_per_tensor ? 1 : 0;
    const int row = (tile - tensor * tiles_per_tensor) * kTileRows + r;
    const bool live = row < num_rows;
    uint32_t t = 0, hd = 0;
    int32_t slot = -1;
    if (live) {
      t = div_rows(uint32_t(row), p.hkv_mul, p.hkv_shift);
      hd = uint32_t(row) - t * uint32_t(hkv);
      slot = __ldg(p.slot_mapping + t);
    }
    cp_async_wait<kTileStages - 1>();  // this lane's copies of the current tile landed
    __syncwarp();                      // ... and the whole warp's

    // Every thread computes (rows past the end or without a slot on stale
    // data) so that the pair shuffles run converged; only stores are guarded.
    uint32_t wd[kHalfRow / 2];  // this thread's 64 input values, in pairs
    {
      // local chunk j of thread h: chunk j (h = 0), chunk 8 + (j ^ 4) (h = 1)
      const uint8_t* rowp = buf + r * kRowBytes + h * (kRowBytes / 2);
      const int x = (r & 3) ^ (h << 2);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 w = *reinterpret_cast<const uint4*>(rowp + ((j ^ x) << 4));
        wd[4 * j + 0] = w.x;
        wd[4 * j + 1] = w.y;
        wd[4 * j + 2] = w.z;
        wd[4 * j + 3] = w.w;
      }
    }
    float u[kHalfRow];
    const bool rot = tensor ? p.rotate[1] != 0 : p.rotate[0] != 0;
    if (rot) {
      rotate_half<H, F16IN>(wd, u, p.c_h, h);
    } else {
#pragma unroll
      for (int i = 0; i < kHalfRow / 2; ++i) {
        u[2 * i] = F16IN ? f16_lo(wd[i]) : bf16_lo(wd[i]);
        u[2 * i + 1] = F16IN ? f16_hi(wd[i]) : bf16_hi(wd[i]);
      }
    }
    float mn, mx;
    half_min_max(u, mn, mx);
    const RowMeta m = row_meta(mn, mx, BFM);
    const uint16_t zb = m.zb, sb = m.sb;
    uint32_t word[8];
    quantize_half(u, m.z, m.rcp, m.fast, word);

    if (live && slot != -1) {
      if (slot < 0 || int64_t(slot) >= p.num_slots) {
        if (h == 0) report(p.dev_status, SAW_ERR_DEVICE_INDEX);
      } else {
        const int P = p.page_size;
        const int page = slot >> p.page_shift;
        const int off = slot & (P - 1);
        uint8_t* chunk = (tensor ? p.cache[1] : p.cache[0]) +
                         (int64_t(page) * hkv + hd) * int64_t(chunk_bytes(P));
        // local quarter 0 is G0 (h = 0) or G3 (h = 1); local quarter 1 is G1 /
        // G2, or G2 / G1 after a stride-64 step; quarter g = code bytes 16g..
        uint8_t* codes = chunk + off * (kHeadDim / 2);
        const bool swapped = rot && H == kHeadDim;
        const int q1 = h ? (swapped ? 1 : 2) : (swapped ? 2 : 1);
        *reinterpret_cast<uint4*>(codes + (h ? 48 : 0)) =
            make_uint4(word[0], word[1], word[2], word[3]);
        *reinterpret_cast<uint4*>(codes + 16 * q1) = make_uint4(word[4], word[5], word[6], word[7]);
        if (h == 0)
          *reinterpret_cast<uint32_t*>(chunk + P * (kHeadDim / 2) + 4 * off) =
              uint32_t(sb) | (uint32_t(zb) << 16);
      }
    }
    __syncwarp();  // the buffer is refilled by a later issue
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------ head_dim 64
//
// The same persistent tiled scheme at head_dim 64: one thread per row (its
// 64 values), 32 rows per warp tile (4 KB).  Every butterfly stride stays
// inside the thread, and the row's min/max needs no partner.  Chunk c
// (16 bytes) of tile row r sits in slot c ^ (r & 7) of the row's 128 bytes,
// so a thread reading its own row chunk by chunk and the copies (eight
// chunks of four rows per instruction) both spread over all bank groups.
constexpr int kD64 = 64;
constexpr int kRowBytes64 = kD64 * 2;
constexpr int kTileRows64 = kTileBytes / kRowBytes64;  // 32

template <int H, bool F16IN>
__global__ void __launch_bounds__(kTileThreads, kTileCtasPerSm)
    quantize_append_tiled64_kernel(const AppendParams p, int tiles_per_tensor, int num_tiles) {
  extern __shared__ __align__(128) uint8_t ring_all[];

  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t* ring = ring_all + warp * (kTileStages * kTileBytes);
  const int hkv = p.num_kv_heads;
  const int num_rows = p.num_tokens * hkv;

  // Copies of one tile: 8 per lane, 8 lanes per 128-byte row.
  auto issue = [&](int tile, uint8_t* buf) {
    const int tensor = tile >= tiles_per_tensor ? 1 : 0;
    const int row0 = (tile - tensor * tiles_per_tensor) * kTileRows64;
    const uint16_t* __restrict__ src = tensor ? p.src[1] : p.src[0];
    const int64_t stride = tensor ? p.stride[1] : p.stride[0];
    const int ch = lane & 7;
    const bool full = row0 + kTileRows64 <= num_rows;
    if (full && stride == int64_t(hkv) * kD64) {
      const uint16_t* g = src + int64_t(row0) * kD64 + ch * 8;
#pragma unroll
      for (int it = 0; it < kTileRows64 / 4; ++it) {
        const int r = it * 4 + (lane >> 3);
        cp_async16(buf + r * kRowBytes64 + ((ch ^ (r & 7)) << 4), g + r * kD64);
      }
    } else {
#pragma unroll
      for (int it = 0; it < kTileRows64 / 4; ++it) {
        const int r = it * 4 + (lane >> 3);
        const int row = row0 + r;
        if (row < num_rows) {
          const uint32_t t = div_rows(uint32_t(row), p.hkv_mul, p.hkv_shift);
          const uint32_t hd = uint32_t(row) - t * uint32_t(hkv);
          cp_async16(buf + r * kRowBytes64 + ((ch ^ (r & 7)) << 4),
                     src + int64_t(t) * stride + hd * kD64 + ch * 8);
        }
      }
    }
  };

  const int step = int(gridDim.x) * kTileWarps;
  int tile = int(blockIdx.x) * kTileWarps + warp;
#pragma unroll
  for (int s = 0; s < kTileStages - 1; ++s) {
    const int pre = tile + s * step;
    if (pre < num_tiles) issue(pre, ring + s * kTileBytes);
    cp_async_commit();
  }
  int cur = 0;
  int ahead = kTileStages - 1;
  for (; tile < num_tiles; tile += step) {
    uint8_t* buf = ring + cur * kTileBytes;
    const int nxt = tile + (kTileStages - 1) * step;
    if (nxt < num_tiles) issue(nxt, ring + ahead * kTileBytes);
    cp_async_commit();
    cur = (cur + 1 == kTileStages) ? 0 : cur + 1;
    ahead = (ahead + 1 == kTileStages) ? 0 : ahead + 1;

    const int tensor = tile >= tiles_per_tensor ? 1 : 0;
    const int row = (tile - tensor * tiles_per_tensor) * kTileRows64 + lane;
    const bool live = row < num_rows;
    uint32_t t = 0, hd = 0;
    int32_t slot = -1;
    if (live) {
      t = div_rows(uint32_t(row), p.hkv_mul, p.hkv_shift);
      hd = uint32_t(row) - t * uint32_t(hkv);
      slot = __ldg(p.slot_mapping + t);
    }
    cp_async_wait<kTileStages - 1>();  // this lane's copies of the current tile landed
    __syncwarp();                      // ... and the whole warp's

    // rows past the end compute on stale data; only stores are guarded
    uint32_t wd[kHalfRow / 2];
    {
      const uint8_t* rowp = buf + lane * kRowBytes64;
      const int x = lane & 7;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint4 w = *reinterpret_cast<const uint4*>(rowp + ((j ^ x) << 4));
        wd[4 * j + 0] = w.x;
        wd[4 * j + 1] = w.y;
        wd[4 * j + 2] = w.z;
        wd[4 * j + 3] = w.w;
      }
    }
    float u[kHalfRow];
    const bool rot = tensor ? p.rotate[1] != 0 : p.rotate[0] != 0;
    if (rot) {
      // the whole row in one thread: the lower-thread form of every step
      rotate_half<H, F16IN>(wd, u, p.c_h, 0);
    } else {
#pragma unroll
      for (int i = 0; i < kHalfRow / 2; ++i) {
        u[2 * i] = F16IN ? f16_lo(wd[i]) : bf16_lo(wd[i]);
        u[2 * i + 1] = F16IN ? f16_hi(wd[i]) : bf16_hi(wd[i]);
      }
    }
    float mn, mx;
    half_min_max<false>(u, mn, mx);
    const RowMeta m = row_meta(mn, mx, p.meta_bf16 != 0);
    uint32_t word[8];
    quantize_half(u, m.z, m.rcp, m.fast, word);

    if (live && slot != -1) {
      if (slot < 0 || int64_t(slot) >= p.num_slots) {
        report(p.dev_status, SAW_ERR_DEVICE_INDEX);
      } else {
        const int P = p.page_size;
        const int page = slot >> p.page_shift;
        const int off = slot & (P - 1);
        uint8_t* chunk = (tensor ? p.cache[1] : p.cache[0]) +
                         (int64_t(page) * hkv + hd) * int64_t(P * (kD64 / 2 + 4));
        uint8_t* codes = chunk + off * (kD64 / 2);
        *reinterpret_cast<uint4*>(codes) = make_uint4(word[0], word[1], word[2], word[3]);
        *reinterpret_cast<uint4*>(codes + 16) = make_uint4(word[4], word[5], word[6], word[7]);
        *reinterpret_cast<uint32_t*>(chunk + P * (kD64 / 2) + 4 * off) =
            uint32_t(m.sb) | (uint32_t(m.zb) << 16);
      }
    }
    __syncwarp();  // the buffer is refilled by a later issue
  }
  cp_async_wait<0>();
}

// ------------------------------------------------------------ head_dim 256
//
// The persistent tiled scheme at head_dim 256: four threads per row (64
// values each, as two 32-value blocks X and Y), 8 rows per 4 KB warp tile.
// Writing B0..B7 for the row's 32-value blocks, thread T = 0..3 of a row
// holds X = B0, B3, B5, B6 and Y = B1, B2, B4, B7.  Stride 32 pairs X with
// Y inside the thread; stride 64 pairs threads T and T ^ 1, stride 128
// threads T and T ^ 3, and in both each thread keeps X and trades Y with its
// partner.  Every step is x' = RN(sg x + y), y' = RN(-sg y + x) (exact +-1
// products) with sg = -1 where X is the upper member of the pair, so X keeps
// its block and Y takes the block it received: after the steps Y holds B1,
// B2, B4, B7 (h <= 64), B2, B1, B7, B4 (h = 128) or B4, B7, B1, B2 (h = 256).
constexpr int kD256 = 256;
constexpr int kRowBytes256 = kD256 * 2;
constexpr int kTileRows256 = kTileBytes / kRowBytes256;  // 8

__device__ __forceinline__ int xblock256(int t) { return (0x6530 >> (4 * t)) & 15; }
// Y's block after the butterfly steps of block size h (rot) or none.
__device__ __forceinline__ int yblock256(int t, int h, bool rot) {
  const int table = !rot || h <= 64 ? 0x7421 : (h == 128 ? 0x4712 : 0x2174);
  return (table >> (4 * t)) & 15;
}

// Chunk c (16 bytes, elements 8c .. 8c+7) of tile row r sits in slot
// c ^ (2 ((c >> 4) & 1) + (r & 1)) of the row's 512 bytes: the 8 lanes of a
// quarter warp (rows 2k and 2k+1, threads 0-3) reading chunk j of their X
// (or of their Y) blocks then hit 8 distinct 16-byte bank groups.
__device__ __forceinline__ int slot256(int r, int c) { return c ^ ((((c >> 4) & 1) << 1) | (r & 1)); }

// The butterfly of this thread's 64 values (X in local 0..31, Y in 32..63)
// for blocks of h, then the multiply by c = binary32(1/sqrt(h)).  Strides
// 1..16 inside each block as in rotate_half; the signs of the stride-32, 64
// and 128 steps follow from X's block (bits 0, 1, 2 set: X is the upper
// member).
template <int H, bool F16IN>
__device__ __forceinline__ void rotate_quarter(const uint32_t (&wd)[kHalfRow / 2],
                                               float (&u)[kHalfRow], float c, int xb) {
#pragma unroll
  for (int i = 0; i < kHalfRow / 2; ++i) {
    if (F16IN) {
      const float odd = f16_hi(wd[i]);
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
          "add.rn.f32.f16 %0, lo, %3;\n\tsub.rn.f32.f16 %1, lo, %3;\n\t}"
          : "=f"(u[2 * i]), "=f"(u[2 * i + 1])
          : "r"(wd[i]), "f"(odd));
    } else {
      const float odd = bf16_hi(wd[i]);
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
          "add.rn.f32.bf16 %0, lo, %3;\n\tsub.rn.f32.bf16 %1, lo, %3;\n\t}"
          : "=f"(u[2 * i]), "=f"(u[2 * i + 1])
          : "r"(wd[i]), "f"(odd));
    }
  }
#pragma unroll
  for (int len = 2; len < (H < 32 ? H : 32); len *= 2) {
#pragma unroll
    for (int i = 0; i < kHalfRow; i += 2) {
      if ((i & len) == 0) bfly2(u[i], u[i + 1], u[i + len], u[i + len + 1]);
    }
  }
  if (H >= 64) {
    const float sg = (xb & 1) ? -1.0f : 1.0f;
    const uint64_t sp = pair(sg, sg), sm = pair(-sg, -sg);
#pragma unroll
    for (int j = 0; j < 32; j += 2) bfly2_signed(u[j], u[j + 1], u[32 + j], u[33 + j], sp, sm);
  }
  if (H >= 128) {
    const float sg = (xb & 2) ? -1.0f : 1.0f;
    const uint64_t sp = pair(sg, sg), sm = pair(-sg, -sg);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float o0 = __shfl_xor_sync(0xFFFFFFFFu, u[32 + j], 1);
      const float o1 = __shfl_xor_sync(0xFFFFFFFFu, u[33 + j], 1);
      u[32 + j] = o0;
      u[33 + j] = o1;
      bfly2_signed(u[j], u[j + 1], u[32 + j], u[33 + j], sp, sm);
    }
  }
  if (H >= 256) {
    const float sg = (xb & 4) ? -1.0f : 1.0f;
    const uint64_t sp = pair(sg, sg), sm = pair(-sg, -sg);
#pragma unroll
    for (int j = 0; j < 32; j += 2) {
      const float o0 = __shfl_xor_sync(0xFFFFFFFFu, u[32 + j], 3);
      const float o1 = __shfl_xor_sync(0xFFFFFFFFu, u[33 + j], 3);
      u[32 + j] = o0;
      u[33 + j] = o1;
      bfly2_signed(u[j], u[j + 1], u[32 + j], u[33 + j], sp, sm);
    }
  }
  const uint64_t cc = pair(c, c);
#pragma unroll
  for (int i = 0; i < kHalfRow; i += 2) mul2(u[i], u[i + 1], cc);
}

template <int H, bool F16IN>
__global__ void __launch_bounds__(kTileThreads, kTileCtasPerSm)
    quantize_append_tiled256_kernel(const AppendParams p, int tiles_per_tensor, int num_tiles) {
  extern __shared__ __align__(128) uint8_t ring_all[];

  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  uint8_t* ring = ring_all + warp * (kTileStages * kTileBytes);
  const int hkv = p.num_kv_heads;
  const int num_rows = p.num_tokens * hkv;

  // Copies of one tile: 8 per lane, one 512-byte row per instruction (lane
  // l moves chunk l); the slot depends on the row only through its parity.
  const int so_even = slot256(0, lane) << 4, so_odd = slot256(1, lane) << 4;
  auto issue = [&](int tile, uint8_t* buf) {
    const int tensor = tile >= tiles_per_tensor ? 1 : 0;
    const int row0 = (tile - tensor * tiles_per_tensor) * kTileRows256;
    const uint16_t* __restrict__ src = tensor ? p.src[1] : p.src[0];
    const int64_t stride = tensor ? p.stride[1] : p.stride[0];
    if (row0 + kTileRows256 <= num_rows && stride == int64_t(hkv) * kD256) {
      const uint16_t* g = src + int64_t(row0) * kD256 + lane * 8;
#pragma unroll
      for (int it = 0; it < kTileRows256; ++it)
        cp_async16(buf + it * kRowBytes256 + ((it & 1) ? so_odd : so_even), g + it * kD256);
    } else {
#pragma unroll
      for (int it = 0; it < kTileRows256; ++it) {
        const int row = row0 + it;
        if (row < num_rows) {
          const uint32_t t = div_rows(uint32_t(row), p.hkv_mul, p.hkv_shift);
          const uint32_t hd = uint32_t(row) - t * uint32_t(hkv);
          cp_async16(buf + it * kRowBytes256 + ((it & 1) ? so_odd : so_even),
                     src + int64_t(t) * stride + hd * kD256 + lane * 8);
        }
      }
    }
  };

  const int r = lane >> 2;   // this thread's row in the tile
  const int th = lane & 3;   // and its place in the row
  const int xb = xblock256(th);
  const int yb0 = yblock256(th, 0, false);
  const int step = int(gridDim.x) * kTileWarps;
  int tile = int(blockIdx.x) * kTileWarps + warp;
#pragma unroll
  for (int s = 0; s < kTileStages - 1; ++s) {
    const int pre = tile + s * step;
    if (pre < num_tiles) issue(pre, ring + s * kTileBytes);
    cp_async_commit();
  }
  int cur = 0;
  int ahead = kTileStages - 1;
  for (; tile < num_tiles; tile += step) {
    uint8_t* buf = ring + cur * kTileBytes;
    const int nxt = tile + (kTileStages - 1) * step;
    if (nxt < num_tiles) issue(nxt, ring + ahead * kTileBytes);
    cp_async_commit();
    cur = (cur + 1 == kTileStages) ? 0 : cur + 1;
    ahead = (ahead + 1 == kTileStages) ? 0 : ahead + 1;

    const int tensor = tile >= tiles_per_tensor ? 1 : 0;
    const int row = (tile - tensor * tiles_per_tensor) * kTileRows256 + r;
    const bool live = row < num_rows;
    uint32_t t = 0, hd = 0;
    int32_t slot = -1;
    if (live) {
      t = div_rows(uint32_t(row), p.hkv_mul, p.hkv_shift);
      hd = uint32_t(row) - t * uint32_t(hkv);
      slot = __ldg(p.slot_mapping + t);
    }
    cp_async_wait<kTileStages - 1>();  // this lane's copies of the current tile landed
    __syncwarp();                      // ... and the whole warp's

    // rows past the end compute on stale data (the shuffles run converged);
    // only stores are guarded
    uint32_t wd[kHalfRow / 2];  // X's 32 values, then Y's, in pairs
    {
      const uint8_t* rowp = buf + r * kRowBytes256;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint4 a = *reinterpret_cast<const uint4*>(rowp + (slot256(r, 4 * xb + j) << 4));
        const uint4 b = *reinterpret_cast<const uint4*>(rowp + (slot256(r, 4 * yb0 + j) << 4));
        wd[4 * j + 0] = a.x;
        wd[4 * j + 1] = a.y;
        wd[4 * j + 2] = a.z;
        wd[4 * j + 3] = a.w;
        wd[16 + 4 * j + 0] = b.x;
        wd[16 + 4 * j + 1] = b.y;
        wd[16 + 4 * j + 2] = b.z;
        wd[16 + 4 * j + 3] = b.w;
      }
    }
    float u[kHalfRow];
    const bool rot = tensor ? p.rotate[1] != 0 : p.rotate[0] != 0;
    if (rot) {
      rotate_quarter<H, F16IN>(wd, u, p.c_h, xb);
    } else {
#pragma unroll
      for (int i = 0; i < kHalfRow / 2; ++i) {
        u[2 * i] = F16IN ? f16_lo(wd[i]) : bf16_lo(wd[i]);
        u[2 * i + 1] = F16IN ? f16_hi(wd[i]) : bf16_hi(wd[i]);
      }
    }
    float mn, mx;
    half_min_max<false>(u, mn, mx);
#pragma unroll
    for (int x = 1; x <= 2; x <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xFFFFFFFFu, mn, x));
      mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, x));
    }
    const RowMeta m = row_meta(mn, mx, p.meta_bf16 != 0);
    uint32_t word[8];
    quantize_half(u, m.z, m.rcp, m.fast, word);

    if (live && slot != -1) {
      if (slot < 0 || int64_t(slot) >= p.num_slots) {
        if (th == 0) report(p.dev_status, SAW_ERR_DEVICE_INDEX);
      } else {
        const int P = p.page_size;
        const int page = slot >> p.page_shift;
        const int off = slot & (P - 1);
        uint8_t* chunk = (tensor ? p.cache[1] : p.cache[0]) +
                         (int64_t(page) * hkv + hd) * int64_t(P * (kD256 / 2 + 4));
        // block b's 32 codes are bytes 16b .. 16b+15 of the token's code row
        uint8_t* codes = chunk + off * (kD256 / 2);
        const int yb = yblock256(th, H, rot);
        *reinterpret_cast<uint4*>(codes + 16 * xb) = make_uint4(word[0], word[1], word[2], word[3]);
        *reinterpret_cast<uint4*>(codes + 16 * yb) = make_uint4(word[4], word[5], word[6], word[7]);
        if (th == 0)
          *reinterpret_cast<uint32_t*>(chunk + P * (kD256 / 2) + 4 * off) =
              uint32_t(m.sb) | (uint32_t(m.zb) << 16);
      }
    }
    __syncwarp();  // the buffer is refilled by a later issue
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
      H, p.c_h, lane, &meta, p.in_f16 != 0, p.meta_bf16 != 0);
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
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           kTileWarps * kTileStages * kTileBytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kTileThreads);
  cfg.dynamicSmemBytes = kTileWarps * kTileStages * kTileBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p, tiles_per_tensor, num_tiles);
}

template <bool F16IN, bool BFM>
cudaError_t launch_tiled_h(int h, dim3 grid, cudaStream_t stream, const AppendParams& q,
                           int tiles_per_tensor, int num_tiles) {
  switch (h) {
    case 16: return launch_tiled(quantize_append_tiled_kernel<16, F16IN, BFM>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 32: return launch_tiled(quantize_append_tiled_kernel<32, F16IN, BFM>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 64: return launch_tiled(quantize_append_tiled_kernel<64, F16IN, BFM>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 128: return launch_tiled(quantize_append_tiled_kernel<128, F16IN, BFM>, grid, stream, q, tiles_per_tensor, num_tiles);
    default: return cudaErrorInvalidValue;
  }
}

template <bool F16IN>
cudaError_t launch_tiled64_h(int h, dim3 grid, cudaStream_t stream, const AppendParams& q,
                             int tiles_per_tensor, int num_tiles) {
  switch (h) {
    case 16: return launch_tiled(quantize_append_tiled64_kernel<16, F16IN>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 32: return launch_tiled(quantize_append_tiled64_kernel<32, F16IN>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 64: return launch_tiled(quantize_append_tiled64_kernel<64, F16IN>, grid, stream, q, tiles_per_tensor, num_tiles);
    default: return cudaErrorInvalidValue;
  }
}

template <bool F16IN>
cudaError_t launch_tiled256_h(int h, dim3 grid, cudaStream_t stream, const AppendParams& q,
                              int tiles_per_tensor, int num_tiles) {
  switch (h) {
    case 16: return launch_tiled(quantize_append_tiled256_kernel<16, F16IN>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 32: return launch_tiled(quantize_append_tiled256_kernel<32, F16IN>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 64: return launch_tiled(quantize_append_tiled256_kernel<64, F16IN>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 128: return launch_tiled(quantize_append_tiled256_kernel<128, F16IN>, grid, stream, q, tiles_per_tensor, num_tiles);
    case 256: return launch_tiled(quantize_append_tiled256_kernel<256, F16IN>, grid, stream, q, tiles_per_tensor, num_tiles);
    default: return cudaErrorInvalidValue;
  }
}

// The tiled kernels' launch: the grid (at most kTileCtasPerSm CTAs per SM)
// and the divisions the kernels replace by multiplies.
struct TiledLaunch {
  AppendParams q;
  dim3 grid;
  int tiles_per_tensor = 0, num_tiles = 0;
};
cudaError_t tiled_launch(const AppendParams& p, int num_tensors, int rows_per_tile, TiledLaunch& l) {
  const int num_rows = p.num_tokens * p.num_kv_heads;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  l.tiles_per_tensor = (num_rows + rows_per_tile - 1) / rows_per_tile;
  l.num_tiles = l.tiles_per_tensor * num_tensors;
  l.grid = dim3(std::min((l.num_tiles + kTileWarps - 1) / kTileWarps, sms * kTileCtasPerSm));
  l.q = p;
  l.q.num_tensors = num_tensors;
  int lg = 0;
  while ((1 << lg) < l.q.num_kv_heads) ++lg;
  l.q.hkv_shift = uint32_t(31 + lg);
  l.q.hkv_mul = uint32_t(((uint64_t(1) << l.q.hkv_shift) + l.q.num_kv_heads - 1) / l.q.num_kv_heads);
  l.q.page_shift = 0;
  while ((1 << l.q.page_shift) < l.q.page_size) ++l.q.page_shift;
  return cudaSuccess;
}

// Bulk appends at head_dim 64 and 256 (the warp-per-row kernel in
// variants.cu serves small ones).
cudaError_t launch_quantize_append_tiled64(const AppendParams& p, int num_tensors,
                                           cudaStream_t stream) {
  if (p.num_tokens * p.num_kv_heads == 0) return cudaSuccess;
  const bool any_rot = p.rotate[0] || (num_tensors > 1 && p.rotate[1]);
  const int h = any_rot ? p.block_h : kD64;
  TiledLaunch l;
  cudaError_t e = tiled_launch(p, num_tensors, kTileRows64, l);
  if (e != cudaSuccess) return e;
  return l.q.in_f16 ? launch_tiled64_h<true>(h, l.grid, stream, l.q, l.tiles_per_tensor, l.num_tiles)
                    : launch_tiled64_h<false>(h, l.grid, stream, l.q, l.tiles_per_tensor, l.num_tiles);
}

cudaError_t launch_quantize_append_tiled256(const AppendParams& p, int num_tensors,
                                            cudaStream_t stream) {
  if (p.num_tokens * p.num_kv_heads == 0) return cudaSuccess;
  const bool any_rot = p.rotate[0] || (num_tensors > 1 && p.rotate[1]);
  const int h = any_rot ? p.block_h : kD256;
  TiledLaunch l;
  cudaError_t e = tiled_launch(p, num_tensors, kTileRows256, l);
  if (e != cudaSuccess) return e;
  return l.q.in_f16
             ? launch_tiled256_h<true>(h, l.grid, stream, l.q, l.tiles_per_tensor, l.num_tiles)
             : launch_tiled256_h<false>(h, l.grid, stream, l.q, l.tiles_per_tensor, l.num_tiles);
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
  const dim3 grid(std::min((num_tiles + kTileWarps - 1) / kTileWarps, sms * kTileCtasPerSm));
  AppendParams q = p;
  q.num_tensors = num_tensors;
  int lg = 0;
  while ((1 << lg) < q.num_kv_heads) ++lg;
  q.hkv_shift = uint32_t(31 + lg);
  q.hkv_mul = uint32_t(((uint64_t(1) << q.hkv_shift) + q.num_kv_heads - 1) / q.num_kv_heads);
  q.page_shift = 0;
  while ((1 << q.page_shift) < q.page_size) ++q.page_shift;
  if (q.meta_bf16)
    return q.in_f16 ? launch_tiled_h<true, true>(h, grid, stream, q, tiles_per_tensor, num_tiles)
                    : launch_tiled_h<false, true>(h, grid, stream, q, tiles_per_tensor, num_tiles);
  return q.in_f16 ? launch_tiled_h<true, false>(h, grid, stream, q, tiles_per_tensor, num_tiles)
                  : launch_tiled_h<false, false>(h, grid, stream, q, tiles_per_tensor, num_tiles);
}

}  // namespace saw
