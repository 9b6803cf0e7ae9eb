// prefill_attn.cu -- chunked-prefill attention over the paged INT4 cache.
//
// Pages: youngju.dev "INT4 KV-cache quantization", "Why the KV Cache Is the
// Real Bottleneck" and gist.science "SAW-INT4", s.1 (the method has to live
// inside engines that run fused, FlashAttention-style attention over paged
// KV); the attention itself is the decode's, with the reading that a query
// at position p of its sequence attends causally to cached tokens 0..p.
// The chunk's K/V are appended (saw_quantize_append) before this runs.
//
// Design (sm_103a), FlashAttention-2 shape on the legacy warp MMA:
//  * CTA = (block of 112 query rows, kv-head, sequence); a row is one
//    (query token, q-head of the kv-head's group) pair, token-major, so the
//    whole GQA group shares every K/V tile.  Seven consumer warps own 16 rows
//    each (about 200 registers a thread: eight warps of it fit an SM's four
//    register files, two per file); an eighth warp streams 16-key tiles
//    (K codes + metadata, V codes + metadata: 2176 B) through an 8-stage
//    ring with the bulk-copy engine, full/empty mbarriers (every wait
//    bounded).
//  * S = Q K^T on mma.m16n8k16: rows on M, keys on N, dims on K.  The K
//    operand is the raw codes masked into binary16 subnormals (n * 2^-24 for
//    a low nibble, n * 2^-20 for a high one), so no dequantization pass; q'
//    is rotated in registers, scaled per row by 2^S (odd dims 2^(S-4)) and
//    split into binary16 hi + lo, held in registers as A fragments.
//  * t = sm' (s_k 2^(24-S) acc + z_k sum(q')), online softmax in base 2.
//  * O += (p s_v) V on the MMA: P straight from the score accumulators (the
//    C layout of two key n-tiles is the A layout of one k16 step), V codes
//    paired across keys with byte permutes and masked the same way; sum(p z_v)
//    is added per row at the end, then the inverse V rotation in registers.
#include "saw_device.cuh"
#include "saw_int4.h"
#include "saw_quant_row.cuh"

namespace saw {
namespace {

constexpr int kPW = 7;                       // consumer warps
constexpr int kPThreads = 32 * (kPW + 1);    // + one producer warp
constexpr int kPRows = 16 * kPW;             // query rows per CTA
constexpr int kPStages = 8;
constexpr int kTileTok = 16;
constexpr int kCodes = kTileTok * kHeadDim / 2;    // 1024 B of codes per tile and tensor
constexpr int kMeta = kTileTok * 4;                // 64 B of (s, z) per tile and tensor
constexpr int kHalfStage = kCodes + kMeta;         // 1088
constexpr int kPStage = 2 * kHalfStage;            // 2176
constexpr int kOffFull = kPStages * kPStage;
constexpr int kOffEmpty = kOffFull + kPStages * 8;
constexpr int kOffOk = kOffEmpty + kPStages * 8;
constexpr int kPSmem = kOffOk + kPStages * 4;
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr uint32_t kLo = 0x000F000Fu;        // low nibbles of bytes 0 and 2 -> two halves
constexpr uint32_t kHi = 0x00F000F0u;        // high nibbles

// In-register block-diagonal Sylvester butterfly over one row whose 128
// values are spread over the 4 lanes of an MMA quad, 32 consecutive dims
// each (lane c holds dims 32c..32c+31 in v[0..31]).  Strides below 32 are
// local, 32 and 64 pair lanes c ^ 1 and c ^ 2.  Unscaled: H, not H/sqrt(h).
__device__ __forceinline__ void quad_fwht(float (&v)[32], int h, int c) {
#pragma unroll
  for (int s = 1; s < 32; s <<= 1) {
    if (s < h) {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        if (!(i & s)) {
          const float a = v[i], b = v[i + s];
          v[i] = a + b;
          v[i + s] = a - b;
        }
    }
  }
#pragma unroll
  for (int s = 32; s < 128; s <<= 1) {
    if (s < h) {
      const int m = s >> 5;                 // lane bit
      const bool upper = (c & m) != 0;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float o = __shfl_xor_sync(kFull, v[i], m);
        v[i] = upper ? (o - v[i]) : (v[i] + o);
      }
    }
  }
}

__device__ __forceinline__ float quad_sum(float x) {
  x += __shfl_xor_sync(kFull, x, 1);
  return x + __shfl_xor_sync(kFull, x, 2);
}
__device__ __forceinline__ float quad_max(float x) {
  x = fmaxf(x, __shfl_xor_sync(kFull, x, 1));
  return fmaxf(x, __shfl_xor_sync(kFull, x, 2));
}

// 2^e for -126 <= e <= 127, exactly
__device__ __forceinline__ float pow2f(int e) { return __uint_as_float(uint32_t(127 + e) << 23); }

__device__ __forceinline__ float f16lo(uint32_t w) {
  return __half2float(__ushort_as_half(uint16_t(w & 0xFFFFu)));
}
__device__ __forceinline__ float f16hi(uint32_t w) {
  return __half2float(__ushort_as_half(uint16_t(w >> 16)));
}

template <int P>
__global__ void __launch_bounds__(kPThreads, 1) prefill_attn_kernel(const PrefillParams p) {
  pdl_wait_then_release();
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffFull);
  uint64_t* empty = reinterpret_cast<uint64_t*>(smem + kOffEmpty);
  int32_t* stage_ok = reinterpret_cast<int32_t*>(smem + kOffOk);
  constexpr int kTilesPerPage = P / kTileTok;

  const int kvh = blockIdx.y, seq = blockIdx.z;
  const int rb = p.row_blocks - 1 - blockIdx.x;  // longest blocks first
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group;

  // ---- this CTA's rows and key range
  const int L = p.seq_lens[seq];
  const int q0 = p.cu_q[seq];
  const int ql = p.cu_q[seq + 1] - q0;
  if (L < 0 || L > p.max_seq_len || ql < 0 || ql > L || ql > p.max_q_len || q0 < 0 ||
      q0 + ql > p.total_q) {
    if (rb == 0 && kvh == 0 && tid == 0) report(p.dev_status, SAW_ERR_DEVICE_INDEX);
    return;
  }
  const int R = ql * G;
  const int row0 = rb * kPRows;
  if (row0 >= R) return;
  const int row_end = min(R, row0 + kPRows);
  const int pos_base = L - ql;                      // position of the chunk's first token
  const int pos_max = pos_base + (row_end - 1) / G;
  const int n_tiles = pos_max / kTileTok + 1;

  if (tid == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kPW);
    }
    mbar_fence_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == kPW) {
    const int32_t* btab = p.block_tables + int64_t(seq) * p.max_blocks;
    const int chunk = chunk_bytes(P);
    int issued = 0;
    bool failed = false;
    int ids = -1;  // page id of logical page (lane + base), refreshed every 32 pages
    int ids_base = -32;
    for (int i = 0; i < n_tiles; ++i) {
      const int s = i % kPStages;
      if (i >= kPStages &&
          !__all_sync(kFull, mbar_wait_bounded(&empty[s], ((i / kPStages) - 1) & 1))) {
        failed = true;
        break;
      }
      const int lp = i / kTilesPerPage;
      if (lp >= ids_base + 32) {
        ids_base = lp - (lp & 31);
        const int e = ids_base + lane;
        ids = (e < p.max_blocks && int64_t(e) * P < L) ? btab[e] : -1;
      }
      int pid = __shfl_sync(kFull, ids, lp - ids_base);
      if (pid < 0 || pid >= p.num_pages) {
        if (lane == 0) report(p.dev_status, SAW_ERR_DEVICE_INDEX);
        pid = -1;
      }
      if (lane == 0) {
        uint8_t* st = smem + s * kPStage;
        stage_ok[s] = pid >= 0;
        if (pid < 0) {
          mbar_arrive(&full[s]);
        } else {
          mbar_arrive_expect_tx(&full[s], kPStage);
          const int64_t off = (int64_t(pid) * p.num_kv_heads + kvh) * chunk;
          const int part = i % kTilesPerPage;
          if (P == 16) {
            bulk_g2s(st, p.k_cache + off, kHalfStage, &full[s]);
            bulk_g2s(st + kHalfStage, p.v_cache + off, kHalfStage, &full[s]);
          } else {
            const int64_t codes = off + part * kCodes;
            const int64_t meta = off + P * (kHeadDim / 2) + part * kMeta;
            bulk_g2s(st, p.k_cache + codes, kCodes, &full[s]);
            bulk_g2s(st + kCodes, p.k_cache + meta, kMeta, &full[s]);
            bulk_g2s(st + kHalfStage, p.v_cache + codes, kCodes, &full[s]);
            bulk_g2s(st + kHalfStage + kCodes, p.v_cache + meta, kMeta, &full[s]);
          }
        }
      }
      __syncwarp();
      issued = i + 1;
    }
    if (failed && lane == 0) report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
    // the CTA must not exit while a copy into its shared memory is in flight
    for (int i = max(0, issued - kPStages); i < issued; ++i)
      (void)mbar_wait_bounded(&full[i % kPStages], (i / kPStages) & 1);
    return;
  }

  // ------------------------------------------------------------ consumers
  const int g = lane >> 2, c = lane & 3;
  const int wrow0 = row0 + 16 * warp;
  const int ra = wrow0 + g, rbw = wrow0 + g + 8;
  const bool va = ra < row_end, vb = rbw < row_end;
  const int pos_a = va ? pos_base + ra / G : -1;
  const int pos_b = vb ? pos_base + rbw / G : -1;
  // the warp's rows see keys up to w_max; keys up to w_min are visible to all
  const int w_last = min(row_end, wrow0 + 16) - 1;
  const int w_max = (wrow0 < row_end) ? pos_base + w_last / G : -1;
  const int w_min = (wrow0 < row_end) ? pos_base + wrow0 / G : -1;

  // ---- q: rotate, scale, split into binary16 hi + lo A fragments.
  // Fragment (k-step ks, half e) of lane c pairs local dims
  // (8(ks>>1) + 2(ks&1) + f, +4), f = 0 for b0 / a0,a1 and 1 for b1 / a2,a3,
  // matching the order in which the K codes are unpacked below.
  uint32_t ah[8][4], al[8][4];
  float qsum[2], rowA[2];
  {
    const float qscale = p.q_scale;
#pragma unroll
    for (int rr = 0; rr < 2; ++rr) {
      const bool valid = rr ? vb : va;
      const int r = rr ? rbw : ra;
      float v[32];
      if (valid) {
        const int t = r / G, hh = r - t * G;
        const uint4* src = reinterpret_cast<const uint4*>(
            p.q + (int64_t(q0 + t) * p.num_q_heads + kvh * G + hh) * kHeadDim + 32 * c);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 w = src[k];
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            v[8 * k + 2 * j] = bf16_lo(ws[j]);
            v[8 * k + 2 * j + 1] = bf16_hi(ws[j]);
          }
        }
      } else {
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = 0.0f;
      }
      if (p.rotate_k) {
        quad_fwht(v, p.block_h, c);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= p.c_h;
      }
      float sum = 0.0f, mx = 0.0f;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        sum += v[i];
        mx = fmaxf(mx, fabsf(v[i]));
      }
      sum = quad_sum(sum);
      mx = quad_max(mx);
      // 2^S with max |q'| 2^S < 2^14 (binary16 range, products stay exact):
      // max |q'| < 2^(E - 126) for biased exponent E, so S = 140 - E, kept
      // within [-100, 100] (a row of zeros, or one that small, takes 100)
      const int E = int((__float_as_uint(mx) >> 23) & 0xFFu);
      const int S = min(100, max(-100, 140 - E));
      const float sc = pow2f(S), sco = pow2f(S - 4);
      qsum[rr] = sum * qscale;
      rowA[rr] = qscale * pow2f(24 - S);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
#pragma unroll
        for (int f = 0; f < 2; ++f) {
          const int d0 = 8 * (ks >> 1) + 2 * (ks & 1) + f;
          const float m = f ? sco : sc;
          const float x0 = v[d0] * m, x1 = v[d0 + 4] * m;
          const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
          const float l0 = x0 - __half2float(h0), l1 = x1 - __half2float(h1);
          const uint32_t hw = uint32_t(__half_as_ushort(h0)) | (uint32_t(__half_as_ushort(h1)) << 16);
          const uint32_t lw = pack_half2(l0, l1);
          ah[ks][2 * f + rr] = hw;  // a0/a1: f = 0, rows g / g+8; a2/a3: f = 1
          al[ks][2 * f + rr] = lw;
        }
      }
    }
  }

  float o[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f}, pz[2] = {0.0f, 0.0f};
  bool failed = false;

  for (int i = 0; i < n_tiles; ++i) {
    const int s = i % kPStages;
    if (!__all_sync(kFull, mbar_wait_bounded(&full[s], (i / kPStages) & 1))) {
      failed = true;
      break;
    }
    const int k0 = i * kTileTok;
    if (k0 <= w_max) {
      const uint8_t* st = smem + s * kPStage;
      const bool ok = stage_ok[s] != 0;
      // ---- S = Q K^T: n-tile 0 = keys k0..k0+7 (B column g <- key g),
      // n-tile 1 = keys k0+8..k0+15
      // four independent accumulators (q' hi / lo x two n-tiles): chains of
      // 8 dependent MMAs instead of 16
      float s0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, s1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      {
        float u0[4] = {0.0f, 0.0f, 0.0f, 0.0f}, u1[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        const uint4 wk0 = *reinterpret_cast<const uint4*>(st + g * 64 + 16 * c);
        const uint4 wk1 = *reinterpret_cast<const uint4*>(st + (g + 8) * 64 + 16 * c);
        const uint32_t w0[4] = {wk0.x, wk0.y, wk0.z, wk0.w};
        const uint32_t w1[4] = {wk1.x, wk1.y, wk1.z, wk1.w};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t x0 = (ks & 1) ? (w0[ks >> 1] >> 8) : w0[ks >> 1];
          const uint32_t x1 = (ks & 1) ? (w1[ks >> 1] >> 8) : w1[ks >> 1];
          mma_16816(s0, ah[ks], x0 & kLo, x0 & kHi);
          mma_16816(s1, ah[ks], x1 & kLo, x1 & kHi);
          mma_16816(u0, al[ks], x0 & kLo, x0 & kHi);
          mma_16816(u1, al[ks], x1 & kLo, x1 & kHi);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          s0[j] += u0[j];
          s1[j] += u1[j];
        }
      }
      // ---- logits: this lane holds keys 2c, 2c+1 (n-tile 0) and 8+2c, 9+2c
      const uint2 km0 = *reinterpret_cast<const uint2*>(st + kCodes + 8 * c);
      const uint2 km1 = *reinterpret_cast<const uint2*>(st + kCodes + 32 + 8 * c);
      const float ks_[4] = {f16lo(km0.x), f16lo(km0.y), f16lo(km1.x), f16lo(km1.y)};
      const float kz_[4] = {f16hi(km0.x), f16hi(km0.y), f16hi(km1.x), f16hi(km1.y)};
      const int key[4] = {k0 + 2 * c, k0 + 2 * c + 1, k0 + 8 + 2 * c, k0 + 9 + 2 * c};
      // t[row][j]: row 0 = g, row 1 = g+8; j indexes key[]
      float t[2][4];
      t[0][0] = fmaf(rowA[0] * ks_[0], s0[0], qsum[0] * kz_[0]);
      t[0][1] = fmaf(rowA[0] * ks_[1], s0[1], qsum[0] * kz_[1]);
      t[1][0] = fmaf(rowA[1] * ks_[0], s0[2], qsum[1] * kz_[0]);
      t[1][1] = fmaf(rowA[1] * ks_[1], s0[3], qsum[1] * kz_[1]);
      t[0][2] = fmaf(rowA[0] * ks_[2], s1[0], qsum[0] * kz_[2]);
      t[0][3] = fmaf(rowA[0] * ks_[3], s1[1], qsum[0] * kz_[3]);
      t[1][2] = fmaf(rowA[1] * ks_[2], s1[2], qsum[1] * kz_[2]);
      t[1][3] = fmaf(rowA[1] * ks_[3], s1[3], qsum[1] * kz_[3]);
      const bool partial = !ok || (k0 + kTileTok - 1 > w_min);
      if (partial) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          t[0][j] = (ok && key[j] <= pos_a) ? t[0][j] : -INFINITY;
          t[1][j] = (ok && key[j] <= pos_b) ? t[1][j] : -INFINITY;
        }
      }
      // ---- online softmax (base 2)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const float mt = quad_max(fmaxf(fmaxf(t[rr][0], t[rr][1]), fmaxf(t[rr][2], t[rr][3])));
        if (mt > m_run[rr]) {
          const float al_ = ex2(m_run[rr] - mt);  // 0 when m_run is -inf
          m_run[rr] = mt;
          l_run[rr] *= al_;
          pz[rr] *= al_;
#pragma unroll
          for (int n = 0; n < 16; ++n) {
            o[n][2 * rr] *= al_;
            o[n][2 * rr + 1] *= al_;
          }
        }
      }
      const float mu0 = (m_run[0] == -INFINITY) ? 0.0f : m_run[0];
      const float mu1 = (m_run[1] == -INFINITY) ? 0.0f : m_run[1];
      float pr[2][4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        pr[0][j] = ex2(t[0][j] - mu0);
        pr[1][j] = ex2(t[1][j] - mu1);
      }
      // ---- V scale / zero of the same keys; keys past the sequence end (or
      // on a bad page) may hold anything, so their terms are selected away
      const uint2 vm0 = *reinterpret_cast<const uint2*>(st + kHalfStage + kCodes + 8 * c);
      const uint2 vm1 = *reinterpret_cast<const uint2*>(st + kHalfStage + kCodes + 32 + 8 * c);
      float vs[4] = {f16lo(vm0.x), f16lo(vm0.y), f16lo(vm1.x), f16lo(vm1.y)};
      float vz[4] = {f16hi(vm0.x), f16hi(vm0.y), f16hi(vm1.x), f16hi(vm1.y)};
      if (partial) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const bool live = ok && key[j] < L;
          vs[j] = live ? vs[j] : 0.0f;
          vz[j] = live ? vz[j] : 0.0f;
        }
      }
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        l_run[rr] += (pr[rr][0] + pr[rr][1]) + (pr[rr][2] + pr[rr][3]);
        pz[rr] = fmaf(pr[rr][0], vz[0], fmaf(pr[rr][1], vz[1],
                 fmaf(pr[rr][2], vz[2], fmaf(pr[rr][3], vz[3], pz[rr]))));
      }
      // A fragment of p*s: a0 (row g, keys 2c, 2c+1), a1 (row g+8, same),
      // a2 (row g, keys 8+2c, 9+2c), a3 (row g+8, same)
      uint32_t pa[4];
      pa[0] = pack_half2(pr[0][0] * vs[0], pr[0][1] * vs[1]);
      pa[1] = pack_half2(pr[1][0] * vs[0], pr[1][1] * vs[1]);
      pa[2] = pack_half2(pr[0][2] * vs[2], pr[0][3] * vs[3]);
      pa[3] = pack_half2(pr[1][2] * vs[2], pr[1][3] * vs[3]);

      // ---- O += (p s) V: B column g of n-tile nt is dim 16g + nt; its k
      // pairs are keys (2c, 2c+1) for b0 and (8+2c, 9+2c) for b1, the same
      // bytes of the two keys' rows side by side (one byte permute)
      const uint8_t* vc = st + kHalfStage;
      const uint2 xa = *reinterpret_cast<const uint2*>(vc + (2 * c) * 64 + 8 * g);
      const uint2 ya = *reinterpret_cast<const uint2*>(vc + (2 * c + 1) * 64 + 8 * g);
      const uint2 xb = *reinterpret_cast<const uint2*>(vc + (2 * c + 8) * 64 + 8 * g);
      const uint2 yb = *reinterpret_cast<const uint2*>(vc + (2 * c + 9) * 64 + 8 * g);
#pragma unroll
      for (int w = 0; w < 2; ++w) {
        const uint32_t xw0 = w ? xa.y : xa.x, yw0 = w ? ya.y : ya.x;
        const uint32_t xw1 = w ? xb.y : xb.x, yw1 = w ? yb.y : yb.x;
#pragma unroll
        for (int pp = 0; pp < 2; ++pp) {
          const uint32_t sel = pp ? 0x7632u : 0x5410u;
          const uint32_t r0 = prmt(xw0, yw0, sel), r1 = prmt(xw1, yw1, sel);
          const uint32_t q0_ = r0 >> 8, q1_ = r1 >> 8;
          const int nt = 8 * w + 4 * pp;
          mma_16816(o[nt + 0], pa, r0 & kLo, r1 & kLo);
          mma_16816(o[nt + 1], pa, r0 & kHi, r1 & kHi);
          mma_16816(o[nt + 2], pa, q0_ & kLo, q1_ & kLo);
          mma_16816(o[nt + 3], pa, q0_ & kHi, q1_ & kHi);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (failed && lane == 0) report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);

  // ---- epilogue: code scales, sum(p z), normalise, inverse V rotation
#pragma unroll
  for (int rr = 0; rr < 2; ++rr) {
    const float l = quad_sum(l_run[rr]);
    const float z = quad_sum(pz[rr]);
    const float inv = (l > 0.0f) ? 1.0f / l : 0.0f;
    float v[32];
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
      const float cs = (nt & 1) ? 1048576.0f : 16777216.0f;  // 2^20 : 2^24
      v[nt] = fmaf(o[nt][2 * rr], cs, z) * inv;              // dim 32c + nt
      v[16 + nt] = fmaf(o[nt][2 * rr + 1], cs, z) * inv;     // dim 32c + 16 + nt
    }
    if (p.rotate_v) {
      quad_fwht(v, p.block_h, c);
#pragma unroll
      for (int i = 0; i < 32; ++i) v[i] *= p.c_h;
    }
    const bool valid = rr ? vb : va;
    if (valid) {
      const int r = rr ? rbw : ra;
      const int t = r / G, hh = r - t * G;
      float4* dst = reinterpret_cast<float4*>(
          p.out + (int64_t(q0 + t) * p.num_q_heads + kvh * G + hh) * kHeadDim + 32 * c);
#pragma unroll
      for (int k = 0; k < 8; ++k) dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    }
  }
}

template <int P>
cudaError_t launch_prefill_p(const PrefillParams& p, cudaStream_t stream) {
  auto kernel = prefill_attn_kernel<P>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.row_blocks, p.num_kv_heads, p.num_seqs);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

}  // namespace

int prefill_rows_per_cta() { return kPRows; }

cudaError_t launch_prefill_attn(const PrefillParams& p, cudaStream_t stream) {
  if (p.num_seqs == 0 || p.row_blocks == 0) return cudaSuccess;
  switch (p.page_size) {
    case 16: return launch_prefill_p<16>(p, stream);
    case 32: return launch_prefill_p<32>(p, stream);
    case 64: return launch_prefill_p<64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace saw
