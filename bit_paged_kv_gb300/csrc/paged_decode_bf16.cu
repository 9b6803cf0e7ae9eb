// paged_decode_bf16.cu -- the BF16 paged-KV baseline: decode attention over
// an unquantized bfloat16 cache, and the append that fills it.
//
// Pages: gist.science "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization for
// Real-World LLM Serving", s.4 "Risultati" (INT4 + rotation is compared with a
// BF16 KV cache for throughput at up to 256 concurrent requests).  This is
// that baseline at the kernel level, built like the INT4 decode so that the
// two differ in the bytes they read and the work per byte, not in structure.
//
// Design (sm_103a):
//  * Cache: per layer and tensor [num_pages][Hkv][P][D] bfloat16.
//  * One 8-warp CTA per (split, kv-head, sequence), one CTA per SM.  Warp w
//    takes 16-token tiles w, w+8, ... through a private three-stage ring.  A
//    stage is four tensor-copy boxes (K and V, dims 0-63 and 64-127), each
//    16 rows x 128 bytes landing 128-byte swizzled (16-byte chunk c of row r
//    at chunk c ^ (r & 7)), completing on one mbarrier (bounded waits).
//  * Scores: mma.m16n8k16 bf16 -> f32, 16 tokens on M (ldmatrix from the
//    swizzled K box), q-heads on N (q exact in bf16), dims on K.
//  * Output: O^T += V^T P, dims on M (ldmatrix.trans from the V box), tokens
//    on K, heads on N; P as bfloat16 hi + lo parts (two MMAs, ~16 bits).
//  * Online softmax in base 2; splits merge in the last split to arrive, as
//    in the INT4 decode (two counters in the workspace).
#include <cuda.h>

#include "saw_device.cuh"
#include "saw_int4.h"
#include "saw_quant_row.cuh"

namespace saw {
namespace {

constexpr int kBW = 8;                       // warps per CTA
constexpr int kBThreads = kBW * 32;
constexpr int kBStages = 3;
constexpr int kBTile = 16;                   // tokens per tile
constexpr int kBRowBytes = kHeadDim * 2;     // 256
constexpr int kBox = kBTile * 128;           // one copy: 16 rows x 64 dims = 2 KB
constexpr int kBStage = 4 * kBox;            // K lo, K hi, V lo, V hi
constexpr int kBRing = kBW * kBStages * kBStage;  // 192 KB
constexpr int kBIdCap = 64;
constexpr int kBRedStride = kHeadDim + 8;
constexpr uint32_t kFullMask = 0xFFFFFFFFu;

constexpr int kBRed = (kBW * kMaxGroup * kBRedStride + 3 * kBW * kMaxGroup + 3 * kMaxGroup) * 4;
constexpr int kBOffQs = (kBRed + 15) / 16 * 16;  // f32 [8][128], inside the ring
static_assert(kBOffQs + kMaxGroup * kHeadDim * 4 <= kBRing, "epilogue scratch must fit the ring");
constexpr int kBOffBars = kBRing;
constexpr int kBOffOk = kBOffBars + kBW * kBStages * 8;
constexpr int kBOffIds = kBOffOk + kBW * kBStages * 4;
constexpr int kBOffFlag = kBOffIds + kBW * kBIdCap * 4;
constexpr int kBSmem = kBOffFlag + 16;

__device__ __forceinline__ int bred_col(int d) { return d + (d >> 4); }

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                            uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D = A(16x16) * B(16x8) + D, bfloat16 in, binary32 accumulate.
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
      "{%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// (lo, hi) as a bfloat16x2 word, round to nearest even
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}

// byte address in a swizzled box of row r, 16-byte chunk c
__device__ __forceinline__ uint32_t box_addr(uint32_t base, int r, int c) {
  return base + uint32_t(r * 128 + ((c ^ (r & 7)) << 4));
}

template <int P>
__global__ void __launch_bounds__(kBThreads, 1)
    paged_decode_bf16_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                             const __grid_constant__ CUtensorMap vmap) {
  pdl_wait_then_release();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBOffBars);
  int32_t* stage_ok = reinterpret_cast<int32_t*>(smem + kBOffOk);
  float* qs = reinterpret_cast<float*>(smem + kBOffQs);
  int* flag = reinterpret_cast<int*>(smem + kBOffFlag);

  const int split = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, c = lane & 3;
  const int G = p.group;
  const int hq0 = kvh * G;
  constexpr int kTilesPerPage = P / kBTile;

  int L = p.seq_lens[seq];
  if (L < 0 || L > p.max_seq_len) {
    if (split == 0 && kvh == 0 && tid == 0) report(p.dev_status, SAW_ERR_DEVICE_INDEX);
    L = 0;
  }
  const int n_pages = (L + P - 1) / P;
  const int p_begin = split * p.pages_per_split;
  const int p_end = min(n_pages, p_begin + p.pages_per_split);
  const bool direct = (p.num_splits == 1);
  if (p_begin >= p_end) {
    if (split == 0 && n_pages == 0)
      for (int idx = tid; idx < G * kHeadDim; idx += kBThreads)
        p.out[(int64_t(seq) * p.num_q_heads + hq0) * kHeadDim + idx] = 0.0f;
    return;
  }

  const int n_tiles = (p_end - p_begin) * kTilesPerPage;
  const int n_my = (warp < n_tiles) ? (n_tiles - warp + kBW - 1) / kBW : 0;
  uint8_t* ring = smem + warp * kBStages * kBStage;
  uint64_t* wbars = bars + warp * kBStages;
  int32_t* wok = stage_ok + warp * kBStages;
  const int32_t* btab = p.block_tables + int64_t(seq) * p.max_blocks;
  auto page_id = [&](int i) {
    const int lp = p_begin + (warp + i * kBW) / kTilesPerPage;
    int id = btab[lp];
    if (id < 0 || id >= p.num_pages) {
      report(p.dev_status, SAW_ERR_DEVICE_INDEX);
      id = -1;
    }
    return id;
  };
  int32_t* wids = reinterpret_cast<int32_t*>(smem + kBOffIds) + warp * kBIdCap;
  for (int e = lane; e < n_my && e < kBIdCap; e += 32) wids[e] = page_id(e);
  __syncwarp();

  auto issue = [&](int i) {  // lane 0 only
    const int s = i % kBStages;
    uint8_t* st = ring + s * kBStage;
    const int pid = (i < kBIdCap) ? wids[i] : page_id(i);
    wok[s] = (pid >= 0);
    if (pid < 0) {
      mbar_arrive(&wbars[s]);
      return;
    }
    mbar_arrive_expect_tx(&wbars[s], kBStage);
    const int row = (pid * p.num_kv_heads + kvh) * P + ((warp + i * kBW) % kTilesPerPage) * kBTile;
    tma_load_2d(st, &kmap, 0, row, &wbars[s]);
    tma_load_2d(st + kBox, &kmap, 64, row, &wbars[s]);
    tma_load_2d(st + 2 * kBox, &vmap, 0, row, &wbars[s]);
    tma_load_2d(st + 3 * kBox, &vmap, 64, row, &wbars[s]);
  };
  if (lane == 0) {
    for (int i = 0; i < kBStages; ++i) mbar_init(&wbars[i], 1);
    mbar_fence_init();
    for (int i = 0; i < kBStages && i < n_my; ++i) issue(i);
  }
  __syncwarp();

  // B fragments of q for k-step t: rows (dims) 16t + 2c, +1 and 16t + 8 + 2c,
  // +1 of column (head) g; zero beyond the group
  uint32_t bq[8][2];
  {
    const uint16_t* qrow = p.q + (int64_t(seq) * p.num_q_heads + hq0 + g) * kHeadDim;
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      bq[t][0] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * t + 2 * c) : 0u;
      bq[t][1] = g < G ? *reinterpret_cast<const uint32_t*>(qrow + 16 * t + 8 + 2 * c) : 0u;
    }
  }
  const float qscale = p.q_scale;

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.0f, 0.0f};
  bool failed = false;
  int waited = 0;

  // ldmatrix source rows: lane l feeds row (l & 7) of matrix (l >> 3)
  const int mrow = lane & 7, mat = lane >> 3;
  for (int i = 0; i < n_my; ++i) {
    const int s = i % kBStages;
    const bool ok = mbar_wait_bounded(&wbars[s], (i / kBStages) & 1);
    if (!__all_sync(kFullMask, ok)) {
      failed = true;
      break;
    }
    waited = i + 1;
    const uint32_t st = smem_u32(ring + s * kBStage);
    const int tok0 = p_begin * P + (warp + i * kBW) * kBTile;
    const bool pok = wok[s] != 0;
    const bool full = pok && tok0 + kBTile <= L;
    const bool v0 = pok && (tok0 + g) < L, v1 = pok && (tok0 + g + 8) < L;

    // ---- scores: token rows g, g+8 x heads 2c, 2c+1
    float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      // matrices: (tokens 0-7 | 8-15) x (chunk 2(t%4) | 2(t%4)+1) of box t/4
      const int r = (mat & 1) * 8 + mrow;
      const int ch = 2 * (t & 3) + (mat >> 1);
      uint32_t a[4];
      ldsm_x4(a, box_addr(st + (t >> 2) * kBox, r, ch));
      mma_bf16(d, a, bq[t][0], bq[t][1]);
    }
    float sc[4] = {d[0] * qscale, d[1] * qscale, d[2] * qscale, d[3] * qscale};
    if (!full) {
      sc[0] = v0 ? sc[0] : -INFINITY;
      sc[1] = v0 ? sc[1] : -INFINITY;
      sc[2] = v1 ? sc[2] : -INFINITY;
      sc[3] = v1 ? sc[3] : -INFINITY;
    }

    // ---- online softmax
    float mloc0 = fmaxf(sc[0], sc[2]), mloc1 = fmaxf(sc[1], sc[3]);
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      mloc0 = fmaxf(mloc0, __shfl_xor_sync(kFullMask, mloc0, x));
      mloc1 = fmaxf(mloc1, __shfl_xor_sync(kFullMask, mloc1, x));
    }
    if (__any_sync(kFullMask, (mloc0 > m_run[0]) || (mloc1 > m_run[1]))) {
      const float mn0 = fmaxf(m_run[0], mloc0), mn1 = fmaxf(m_run[1], mloc1);
      const float al0 = ex2(m_run[0] - ((mn0 == -INFINITY) ? 0.0f : mn0));
      const float al1 = ex2(m_run[1] - ((mn1 == -INFINITY) ? 0.0f : mn1));
      m_run[0] = mn0;
      m_run[1] = mn1;
      l_run[0] *= al0;
      l_run[1] *= al1;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        acc[k][0] *= al0;
        acc[k][1] *= al1;
        acc[k][2] *= al0;
        acc[k][3] *= al1;
      }
    }
    const float mu0 = (m_run[0] == -INFINITY) ? 0.0f : m_run[0];
    const float mu1 = (m_run[1] == -INFINITY) ? 0.0f : m_run[1];
    const float p0 = ex2(sc[0] - mu0), p1 = ex2(sc[1] - mu1);
    const float p2 = ex2(sc[2] - mu0), p3 = ex2(sc[3] - mu1);
    l_run[0] += p0 + p2;
    l_run[1] += p1 + p3;

    // ---- P as bf16 hi + lo, moved to the B layout (tokens 2c.., head g)
    const uint32_t Xh = pack_bf16x2(p0, p2), Yh = pack_bf16x2(p1, p3);
    const float h0 = __bfloat162float(__ushort_as_bfloat16(uint16_t(Xh)));
    const float h2 = __bfloat162float(__ushort_as_bfloat16(uint16_t(Xh >> 16)));
    const float h1 = __bfloat162float(__ushort_as_bfloat16(uint16_t(Yh)));
    const float h3 = __bfloat162float(__ushort_as_bfloat16(uint16_t(Yh >> 16)));
    const uint32_t Xl = pack_bf16x2(p0 - h0, p2 - h2), Yl = pack_bf16x2(p1 - h1, p3 - h3);
    const int src0 = 8 * c + (g >> 1);
    uint32_t bh0, bh1, bl0, bl1;
    {
      const uint32_t xa = __shfl_sync(kFullMask, Xh, src0), ya = __shfl_sync(kFullMask, Yh, src0);
      const uint32_t xb = __shfl_sync(kFullMask, Xh, src0 + 4);
      const uint32_t yb = __shfl_sync(kFullMask, Yh, src0 + 4);
      const uint32_t va = (g & 1) ? ya : xa, vb = (g & 1) ? yb : xb;
      bh0 = prmt(va, vb, 0x5410u);
      bh1 = prmt(va, vb, 0x7632u);
    }
    {
      const uint32_t xa = __shfl_sync(kFullMask, Xl, src0), ya = __shfl_sync(kFullMask, Yl, src0);
      const uint32_t xb = __shfl_sync(kFullMask, Xl, src0 + 4);
      const uint32_t yb = __shfl_sync(kFullMask, Yl, src0 + 4);
      const uint32_t va = (g & 1) ? ya : xa, vb = (g & 1) ? yb : xb;
      bl0 = prmt(va, vb, 0x5410u);
      bl1 = prmt(va, vb, 0x7632u);
    }
    // rows past the end may hold anything: their V rows must not reach the
    // sum even with p = 0 (0 * inf), so the partial tile zeroes them first
    if (!full) {
      __syncwarp();
      for (int e = lane; e < kBTile * 16; e += 32) {  // 16 rows x 16 chunks of V
        const int row = e >> 4, ch = e & 15;
        const bool live = pok && (tok0 + row) < L;
        if (!live)
          *reinterpret_cast<uint4*>(ring + s * kBStage + 2 * kBox + (ch >> 3) * kBox + row * 128 +
                                    (((ch & 7) ^ (row & 7)) << 4)) = make_uint4(0, 0, 0, 0);
      }
      // order these generic-proxy stores before a later tensor copy into the stage
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
    }

    // ---- O^T += V^T P for dims 16j .. 16j + 15
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      // matrices: (tokens 0-7 | 8-15) x (dims 16j.. | 16j+8..) of V box j/4
      const int r = (mat >> 1) * 8 + mrow;
      const int ch = 2 * (j & 3) + (mat & 1);
      uint32_t a[4];
      ldsm_x4_t(a, box_addr(st + 2 * kBox + (j >> 2) * kBox, r, ch));
      mma_bf16(acc[j], a, bh0, bh1);
      mma_bf16(acc[j], a, bl0, bl1);
    }
    __syncwarp();
    if (lane == 0 && i + kBStages < n_my) issue(i + kBStages);
  }
  if (failed) {
    if (lane == 0) report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
    for (int i = waited; i < n_my && i < waited + kBStages; ++i)
      (void)mbar_wait_bounded(&wbars[i % kBStages], (i / kBStages) & 1);
  }

  // ---- merge protocol, part 1 (as in the INT4 decode): count this split
  const int ns = (n_pages + p.pages_per_split - 1) / p.pages_per_split;
  uint32_t* tk = p.tickets + 2 * (int64_t(seq) * p.num_kv_heads + kvh);  // {arrived, published}
  uint32_t arrived = 0;
  if (!direct && tid == 0)
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], 1;" : "=r"(arrived) : "l"(tk) : "memory");

#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l_run[0] += __shfl_xor_sync(kFullMask, l_run[0], x);
    l_run[1] += __shfl_xor_sync(kFullMask, l_run[1], x);
  }
  __syncthreads();  // every warp is done with its ring: reuse it

  float* red_acc = reinterpret_cast<float*>(smem);           // [8 warps][8 heads][136]
  float* red_m = red_acc + kBW * kMaxGroup * kBRedStride;   // [8][8]
  float* red_l = red_m + kBW * kMaxGroup;
  float* wgt = red_l + kBW * kMaxGroup;
  float* tot = wgt + kBW * kMaxGroup;                       // den, -, M [3][8]
  {
    const int hb = 2 * c;  // this lane's heads hb, hb+1
    if (g == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        red_m[warp * kMaxGroup + hb + hh] = m_run[hh];
        red_l[warp * kMaxGroup + hb + hh] = l_run[hh];
      }
    }
    float* base0 = red_acc + (warp * kMaxGroup + hb) * kBRedStride;
    float* base1 = base0 + kBRedStride;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      base0[bred_col(16 * j + g)] = acc[j][0];
      base1[bred_col(16 * j + g)] = acc[j][1];
      base0[bred_col(16 * j + 8 + g)] = acc[j][2];
      base1[bred_col(16 * j + 8 + g)] = acc[j][3];
    }
  }
  __syncthreads();
  const int nw = min(kBW, n_tiles);
  if (tid < kMaxGroup * kBW) {
    const int h = tid / kBW, w = tid % kBW;
    const bool in = h < G && w < nw;
    const float m = in ? red_m[w * kMaxGroup + h] : -INFINITY;
    float M = m;
#pragma unroll
    for (int x = 1; x < kBW; x <<= 1) M = fmaxf(M, __shfl_xor_sync(kFullMask, M, x));
    const float Mu = (M == -INFINITY) ? 0.0f : M;
    const float f = in ? ex2(m - Mu) : 0.0f;
    float den = in ? red_l[w * kMaxGroup + h] * f : 0.0f;
#pragma unroll
    for (int x = 1; x < kBW; x <<= 1) den += __shfl_xor_sync(kFullMask, den, x);
    wgt[w * kMaxGroup + h] = f;
    if (w == 0) {
      tot[h] = den;
      tot[2 * kMaxGroup + h] = M;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * kHeadDim; idx += kBThreads) {
    const int h = idx / kHeadDim, dd = idx - h * kHeadDim;
    float num = 0.0f;
#pragma unroll
    for (int w = 0; w < kBW; ++w)
      if (w < nw) num += red_acc[(w * kMaxGroup + h) * kBRedStride + bred_col(dd)] * wgt[w * kMaxGroup + h];
    if (direct) {
      const float den = tot[h];
      qs[h * kHeadDim + dd] = (den > 0.0f) ? num / den : 0.0f;
    } else {
      qs[h * kHeadDim + dd] = num;
      const int64_t row = (int64_t(seq) * p.num_q_heads + hq0 + h) * p.num_splits + split;
      p.part_o[row * kHeadDim + dd] = num;
      if (dd == 0) {
        p.part_ml[2 * row] = tot[2 * kMaxGroup + h];
        p.part_ml[2 * row + 1] = tot[h];
      }
    }
  }
  if (!direct) {
    if (tid == 0) {
      const uint32_t done = arrived + 1u;
      if (done > uint32_t(ns)) report(p.dev_status, SAW_ERR_DEVICE_INDEX);  // not zero-filled
      *flag = (done == uint32_t(ns));
    }
    __syncthreads();
    const bool last = *flag != 0;
    if (!last) {
      if (tid == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(tk + 1) : "memory");
      return;
    }
    if (tid == 0) {
      const uint32_t want = uint32_t(ns - 1);
      bool ok = ld_acquire_u32(tk + 1) == want;
      if (!ok) {
        const long long t0 = clock64();
        while (!(ok = (ld_acquire_u32(tk + 1) == want))) {
          if (clock64() - t0 > kWaitLimitCycles) break;
          __nanosleep(32);
        }
      }
      if (ok) {
        tk[0] = 0u;
        tk[1] = 0u;
      } else {
        report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
      }
      flag[1] = ok ? 1 : 0;
    }
    __syncthreads();
    const bool merge_ok = flag[1] != 0;
    // item = (head, dim): each thread merges the splits of its items
    for (int idx = tid; idx < G * kHeadDim; idx += kBThreads) {
      const int h = idx / kHeadDim, dd = idx - h * kHeadDim;
      const int64_t row0 = (int64_t(seq) * p.num_q_heads + hq0 + h) * p.num_splits;
      float M = -INFINITY;
      for (int sp = 0; sp < ns; ++sp) {
        const float m = (sp == split) ? tot[2 * kMaxGroup + h]
                                      : (merge_ok ? __ldcg(&p.part_ml[2 * (row0 + sp)]) : -INFINITY);
        M = fmaxf(M, m);
      }
      const float Mu = (M == -INFINITY) ? 0.0f : M;
      float num = 0.0f, den = 0.0f;
      for (int sp = 0; sp < ns; ++sp) {
        const bool mine = sp == split;
        if (!mine && !merge_ok) continue;
        const float m = mine ? tot[2 * kMaxGroup + h] : __ldcg(&p.part_ml[2 * (row0 + sp)]);
        const float l = mine ? tot[h] : __ldcg(&p.part_ml[2 * (row0 + sp) + 1]);
        const float o = mine ? qs[idx] : __ldcg(&p.part_o[(row0 + sp) * kHeadDim + dd]);
        const float f = ex2(m - Mu);
        den += l * f;
        num += o * f;
      }
      p.out[(int64_t(seq) * p.num_q_heads + hq0) * kHeadDim + idx] = (den > 0.0f) ? num / den : 0.0f;
    }
    return;
  }
  __syncthreads();
  for (int idx = tid; idx < G * kHeadDim; idx += kBThreads)
    p.out[(int64_t(seq) * p.num_q_heads + hq0) * kHeadDim + idx] = qs[idx];
}

// One warp per (token, kv-head) row of one tensor: 256 bytes, 8 per lane.
constexpr int kAppendRowsPerCta = 8;

__global__ void __launch_bounds__(32 * kAppendRowsPerCta) bf16_append_kernel(
    const uint16_t* __restrict__ k, const uint16_t* __restrict__ v, int64_t k_stride,
    int64_t v_stride, const int32_t* __restrict__ slots, int num_tokens, int hkv,
    uint16_t* __restrict__ kc, uint16_t* __restrict__ vc, int64_t num_slots, int P,
    int num_tensors, int32_t* dev_status) {
  pdl_wait_then_release();
  const int lane = threadIdx.x & 31;
  const int64_t gw = int64_t(blockIdx.x) * kAppendRowsPerCta + (threadIdx.x >> 5);
  const int64_t rows = int64_t(num_tokens) * hkv;
  if (gw >= rows * num_tensors) return;
  const int tensor = gw >= rows ? 1 : 0;
  const int64_t row = gw - tensor * rows;
  const int t = int(row / hkv), hd = int(row - int64_t(t) * hkv);
  const int32_t slot = slots[t];
  if (slot == -1) return;
  if (slot < 0 || int64_t(slot) >= num_slots) {
    if (lane == 0 && tensor == 0) report(dev_status, SAW_ERR_DEVICE_INDEX);
    return;
  }
  const uint16_t* src = (tensor ? v + int64_t(t) * v_stride : k + int64_t(t) * k_stride) +
                        int64_t(hd) * kHeadDim;
  uint16_t* dst = (tensor ? vc : kc) +
                  ((int64_t(slot / P) * hkv + hd) * P + slot % P) * int64_t(kHeadDim);
  reinterpret_cast<uint2*>(dst)[lane] = reinterpret_cast<const uint2*>(src)[lane];
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no
// link-time dependency on the driver library).
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

cudaError_t encode_cache_map(CUtensorMap* map, const void* cache, int64_t rows) {
  static EncodeFn fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e =
        cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !f) return cudaErrorNotSupported;
    fn = reinterpret_cast<EncodeFn>(f);
  }
  const cuuint64_t dims[2] = {cuuint64_t(kHeadDim), cuuint64_t(rows > 0 ? rows : 1)};
  const cuuint64_t strides[1] = {cuuint64_t(kBRowBytes)};
  const cuuint32_t box[2] = {64, kBTile};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(cache), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

template <int P>
cudaError_t launch_bf16_p(const DecodeParams& p, const CUtensorMap& km, const CUtensorMap& vm,
                          cudaStream_t stream) {
  auto kernel = paged_decode_bf16_kernel<P>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBSmem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits, p.num_kv_heads, p.num_seqs);
  cfg.blockDim = dim3(kBThreads);
  cfg.dynamicSmemBytes = kBSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p, km, vm);
}

}  // namespace

cudaError_t launch_paged_decode_bf16(const DecodeParams& p, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  const int64_t rows = int64_t(p.num_pages) * p.num_kv_heads * p.page_size;
  CUtensorMap km, vm;
  cudaError_t e = encode_cache_map(&km, p.k_cache, rows);
  if (e == cudaSuccess) e = encode_cache_map(&vm, p.v_cache, rows);
  if (e != cudaSuccess) return e;
  switch (p.page_size) {
    case 16: return launch_bf16_p<16>(p, km, vm, stream);
    case 32: return launch_bf16_p<32>(p, km, vm, stream);
    case 64: return launch_bf16_p<64>(p, km, vm, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_bf16_append(const uint16_t* k, const uint16_t* v, int64_t k_stride,
                               int64_t v_stride, const int32_t* slots, int num_tokens, int hkv,
                               uint16_t* kc, uint16_t* vc, int64_t num_slots, int P,
                               int32_t* dev_status, cudaStream_t stream) {
  const int num_tensors = v ? 2 : 1;
  const int64_t warps = int64_t(num_tokens) * hkv * num_tensors;
  if (warps == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned((warps + kAppendRowsPerCta - 1) / kAppendRowsPerCta));
  cfg.blockDim = dim3(32 * kAppendRowsPerCta);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, bf16_append_kernel, k, v, k_stride, v_stride, slots, num_tokens,
                            hkv, kc, vc, num_slots, P, num_tensors, dev_status);
}

}  // namespace saw
