// paged_decode.cu -- K2/K3: split-K decode attention over the INT4 paged
// cache (SAW-INT4), with dequantization fused into the attention loop.
//
// Pages: gist.science "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization
// for Real-World LLM Serving", s.2 point 3 (rotation and quantization fused
// into the decoding path, hidden inside a memory-bound data flow); youngju.dev
// "INT4 KV-cache quantization" (English), "The Rotation Trick": H is an
// orthogonal, undoable rotation, so q.k = (Hq).(Hk) and o = H^-1 o'.
//
// Design (sm_103a):
//  * One CTA per (split of the context, kv-head, sequence); 4 warps.  The
//    whole GQA group of the kv-head is served by the CTA, so each page chunk
//    is read from HBM once.
//  * Each warp streams its own pages (pages w, w+4, ... of the split) through
//    a private ring of shared-memory stages filled by the bulk-copy engine
//    (cp.async.bulk + mbarrier complete_tx).  One K chunk and one V chunk per
//    page; the chunk carries the page's codes and (scale, zero) words.
//  * Scores: S = K~ q' on the tensor cores (mma.m16n8k16, binary16 in,
//    binary32 accumulate), 16 tokens on M, the <= 8 q-heads on N, the head
//    dimension on K.  K~ are the raw codes 0..15, exact in binary16,
//    converted in registers with the 0x6400 exponent trick; the per-token
//    scale and zero are applied afterwards: t = s*(K~.q') + z*sum(q').
//  * Output: O'^T += V~^T (p*s) on the tensor cores, dims on M, tokens on K,
//    heads on N, plus sum_j p_j z_j on the CUDA cores.  p*s is moved from the
//    score fragment to the B-operand layout with four warp shuffles.
//  * Online softmax in base 2 per head; sm_scale*log2(e) scales the binary32
//    score after the MMA, so an unrotated q enters the MMA exactly.
//  * Splits write (m, l, numerator) partials; K3 merges them, normalizes and
//    applies the inverse rotation to V's output.  With one split the CTA
//    finishes the row itself.
#include "saw_device.cuh"
#include "saw_int4.h"

namespace saw {
namespace {

constexpr int kWarps = kDecodeWarps;
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kFull = 0xFFFFFFFFu;
constexpr int kRedStride = kHeadDim + 4;  // padded row of the cross-warp reduction

template <int P>
struct Cfg {
  static constexpr int kChunk = chunk_bytes(P);
  static constexpr int kStage = 2 * kChunk;  // K chunk, then V chunk
  static constexpr int kStages = (P == 16) ? 4 : (P == 32) ? 3 : 2;
  static constexpr int kTiles = P / 16;
  static constexpr int kRing = kWarps * kStages * kStage;
  static constexpr int kRed = kWarps * kMaxGroup * kRedStride * 4 + 3 * kWarps * kMaxGroup * 4;
  static_assert(kRed <= kRing, "reduction scratch must fit in the ring");
  // dynamic shared memory layout
  static constexpr int kOffBars = kRing;
  static constexpr int kOffOk = kOffBars + kWarps * kStages * 8;
  static constexpr int kOffQ = (kOffOk + kWarps * kStages * 4 + 15) / 16 * 16;  // float [8][128]
  static constexpr int kOffQh = kOffQ + kMaxGroup * kHeadDim * 4;   // half [2][8][128]: hi, lo
  static constexpr int kOffQsum = kOffQh + 2 * kMaxGroup * kHeadDim * 2;         // float [8]
  static constexpr int kSmem = kOffQsum + kMaxGroup * 4;
};

// In-place butterfly over each h-block of nvec vectors of 128 floats in shared
// memory (all threads of the CTA take part).  Mathematically (H x) per block;
// the 1/sqrt(h) factor is left to the caller.
__device__ void smem_fwht(float* buf, int nvec, int h) {
  const int lanes = nvec * (kHeadDim / 2);
  for (int len = 1; len < h; len *= 2) {
    for (int idx = threadIdx.x; idx < lanes; idx += blockDim.x) {
      const int v = idx / (kHeadDim / 2);
      const int k = idx - v * (kHeadDim / 2);
      // k-th index with bit `len` clear
      const int i = ((k & ~(len - 1)) << 1) | (k & (len - 1));
      float* row = buf + v * kHeadDim;
      const float a = row[i], b = row[i + len];
      row[i] = a + b;
      row[i + len] = a - b;
    }
    __syncthreads();
  }
}

__device__ __forceinline__ uint32_t hsub_1024(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2*>(&x);
  h = __hsub2(h, __half2half2(__ushort_as_half(0x6400)));
  return *reinterpret_cast<uint32_t*>(&h);
}

// (1024 + 16 n) / 16 - 64 = n, exact in binary16
__device__ __forceinline__ uint32_t hfma_hi(uint32_t x) {
  __half2 h = *reinterpret_cast<__half2*>(&x);
  h = __hfma2(h, __half2half2(__ushort_as_half(0x2C00)), __half2half2(__ushort_as_half(0xD400)));
  return *reinterpret_cast<uint32_t*>(&h);
}

constexpr uint32_t kMagic = 0x64006400u;  // binary16 1024.0 in both halves

template <int P>
__global__ void __launch_bounds__(kThreads, (P == 64) ? 3 : 4) paged_decode_kernel(const DecodeParams p) {
  using C = Cfg<P>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  int32_t* stage_ok = reinterpret_cast<int32_t*>(smem + C::kOffOk);
  float* qs = reinterpret_cast<float*>(smem + C::kOffQ);
  __half* qh = reinterpret_cast<__half*>(smem + C::kOffQh);
  float* qsum = reinterpret_cast<float*>(smem + C::kOffQsum);

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int seq = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;  // MMA group id
  const int c = lane & 3;   // thread in group
  const int G = p.group;
  const int hq0 = kvh * G;

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
    // nothing to attend over: a direct launch still owes the output row
    if (direct) {
      for (int idx = tid; idx < G * kHeadDim; idx += kThreads)
        p.out[(int64_t(seq) * p.num_q_heads + hq0) * kHeadDim + idx] = 0.0f;
    }
    return;
  }

  // ---- per-warp page stream: barriers and the first copies go out first,
  // so HBM latency overlaps the q prologue below
  const int my_first = p_begin + warp;
  const int n_my = (my_first < p_end) ? (p_end - my_first + kWarps - 1) / kWarps : 0;
  uint8_t* ring = smem + warp * C::kStages * C::kStage;
  uint64_t* wbars = bars + warp * C::kStages;
  int32_t* wok = stage_ok + warp * C::kStages;
  const int32_t* btab = p.block_tables + int64_t(seq) * p.max_blocks;

  auto issue = [&](int i) {  // lane 0 only
    const int lp = my_first + i * kWarps;
    const int s = i % C::kStages;
    const int pid = btab[lp];
    if (pid >= 0 && pid < p.num_pages) {
      wok[s] = 1;
      mbar_arrive_expect_tx(&wbars[s], 2 * C::kChunk);
      const int64_t off = (int64_t(pid) * p.num_kv_heads + kvh) * C::kChunk;
      bulk_g2s(ring + s * C::kStage, p.k_cache + off, C::kChunk, &wbars[s]);
      bulk_g2s(ring + s * C::kStage + C::kChunk, p.v_cache + off, C::kChunk, &wbars[s]);
    } else {
      wok[s] = 0;
      report(p.dev_status, SAW_ERR_DEVICE_INDEX);
      mbar_arrive(&wbars[s]);
    }
  };

  if (lane == 0) {
    for (int i = 0; i < C::kStages; ++i) mbar_init(&wbars[i], 1);
    mbar_fence_init();
    for (int i = 0; i < C::kStages && i < n_my; ++i) issue(i);
  }
  __syncwarp();

  // ---- q' = (1/sqrt h) H q for the group's heads, as binary16 hi + lo parts
  // (q' = hi + lo to ~22 bits; zeros beyond G).  Warp w rotates heads w and
  // w + 4, lane l holding elements 4l..4l+3; sm_scale*log2(e) is applied to
  // the binary32 score, so an unrotated q enters the MMA exactly.
  __half* qh_hi = qh;
  __half* qh_lo = qh + kMaxGroup * kHeadDim;
  for (int h = warp; h < kMaxGroup; h += kWarps) {
    float x[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    if (h < G) {
      const uint2 raw = *reinterpret_cast<const uint2*>(
          p.q + (int64_t(seq) * p.num_q_heads + hq0 + h) * kHeadDim + 4 * lane);
      x[0] = bf16_lo(raw.x);
      x[1] = bf16_hi(raw.x);
      x[2] = bf16_lo(raw.y);
      x[3] = bf16_hi(raw.y);
      if (p.rotate_k) {
        const int hb = p.block_h;
        float a0 = x[0] + x[1], a1 = x[0] - x[1], a2 = x[2] + x[3], a3 = x[2] - x[3];
        if (hb > 2) {
          x[0] = a0 + a2; x[1] = a1 + a3; x[2] = a0 - a2; x[3] = a1 - a3;
        } else {
          x[0] = a0; x[1] = a1; x[2] = a2; x[3] = a3;
        }
        for (int len = 4; len < hb; len *= 2) {
          const int mask = len >> 2;
          const bool upper = (lane & mask) != 0;
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float o = __shfl_xor_sync(kFull, x[e], mask);
            x[e] = upper ? (o - x[e]) : (x[e] + o);
          }
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) x[e] *= p.c_h;
      }
    }
    float part = 0.0f;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const __half hi = __float2half_rn(x[e]);
      const __half lo = __float2half_rn(x[e] - __half2float(hi));
      qh_hi[h * kHeadDim + 4 * lane + e] = hi;
      qh_lo[h * kHeadDim + 4 * lane + e] = lo;
      part += __half2float(hi) + __half2float(lo);
    }
#pragma unroll
    for (int x2 = 16; x2 >= 1; x2 >>= 1) part += __shfl_xor_sync(kFull, part, x2);
    if (lane == 0) qsum[h] = part;
  }
  __syncthreads();

  // B fragments of q' for the score MMA (k-step t uses word 4c + t/2 of a
  // token's codes: bytes (0,2) for even t, (1,3) for odd t).
  uint32_t bq[8][2], bl[8][2];
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    const int base = 8 * (4 * c + t / 2) + ((t & 1) ? 2 : 0);
    const __half* rh = qh_hi + g * kHeadDim;
    const __half* rl = qh_lo + g * kHeadDim;
    __half2 v0 = __halves2half2(rh[base], rh[base + 4]);
    __half2 v1 = __halves2half2(rh[base + 1], rh[base + 5]);
    __half2 w0 = __halves2half2(rl[base], rl[base + 4]);
    __half2 w1 = __halves2half2(rl[base + 1], rl[base + 5]);
    bq[t][0] = *reinterpret_cast<uint32_t*>(&v0);
    bq[t][1] = *reinterpret_cast<uint32_t*>(&v1);
    bl[t][0] = *reinterpret_cast<uint32_t*>(&w0);
    bl[t][1] = *reinterpret_cast<uint32_t*>(&w1);
  }
  const float qsum0 = qsum[2 * c] * p.q_scale, qsum1 = qsum[2 * c + 1] * p.q_scale;

  float acc[8][4];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.0f, 0.0f};
  float z_run[2] = {0.0f, 0.0f};
  bool failed = false;
  int waited = 0;

  for (int i = 0; i < n_my; ++i) {
    const int s = i % C::kStages;
    const bool ok = mbar_wait_bounded(&wbars[s], (i / C::kStages) & 1);
    if (!__all_sync(kFull, ok)) {
      failed = true;
      break;
    }
    waited = i + 1;
    const uint8_t* kst = ring + s * C::kStage;
    const uint8_t* vst = kst + C::kChunk;
    const bool page_ok = wok[s] != 0;
    const int tok_base = (my_first + i * kWarps) * P;

    // ---- scores for every 16-token tile of the page
    float sc[C::kTiles][4];
#pragma unroll
    for (int tt = 0; tt < C::kTiles; ++tt) {
      const uint8_t* krow = kst + (16 * tt + g) * (kHeadDim / 2) + 16 * c;
      const uint4 ka = *reinterpret_cast<const uint4*>(krow);
      const uint4 kb = *reinterpret_cast<const uint4*>(krow + 8 * (kHeadDim / 2));
      const uint32_t kaw[4] = {ka.x, ka.y, ka.z, ka.w};
      const uint32_t kbw[4] = {kb.x, kb.y, kb.z, kb.w};
      float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int w = 0; w < 4; ++w) {
#pragma unroll
        for (int hb = 0; hb < 2; ++hb) {
          const uint32_t ya = hb ? (kaw[w] >> 8) : kaw[w];
          const uint32_t yb = hb ? (kbw[w] >> 8) : kbw[w];
          uint32_t a[4];
          a[0] = hsub_1024(and_or(ya, 0x000F000Fu, kMagic));
          a[1] = hsub_1024(and_or(yb, 0x000F000Fu, kMagic));
          a[2] = hfma_hi(and_or(ya, 0x00F000F0u, kMagic));
          a[3] = hfma_hi(and_or(yb, 0x00F000F0u, kMagic));
          mma_16816(d, a, bq[2 * w + hb][0], bq[2 * w + hb][1]);
          mma_16816(d, a, bl[2 * w + hb][0], bl[2 * w + hb][1]);
        }
      }
      const uint32_t mk0 =
          *reinterpret_cast<const uint32_t*>(kst + P * (kHeadDim / 2) + (16 * tt + g) * 4);
      const uint32_t mk1 =
          *reinterpret_cast<const uint32_t*>(kst + P * (kHeadDim / 2) + (16 * tt + g + 8) * 4);
      const float sk0 = __half2float(__ushort_as_half(uint16_t(mk0 & 0xFFFF))) * p.q_scale;
      const float zk0 = __half2float(__ushort_as_half(uint16_t(mk0 >> 16)));
      const float sk1 = __half2float(__ushort_as_half(uint16_t(mk1 & 0xFFFF))) * p.q_scale;
      const float zk1 = __half2float(__ushort_as_half(uint16_t(mk1 >> 16)));
      const bool v0 = page_ok && (tok_base + 16 * tt + g) < L;
      const bool v1 = page_ok && (tok_base + 16 * tt + g + 8) < L;
      sc[tt][0] = v0 ? fmaf(sk0, d[0], zk0 * qsum0) : -INFINITY;
      sc[tt][1] = v0 ? fmaf(sk0, d[1], zk0 * qsum1) : -INFINITY;
      sc[tt][2] = v1 ? fmaf(sk1, d[2], zk1 * qsum0) : -INFINITY;
      sc[tt][3] = v1 ? fmaf(sk1, d[3], zk1 * qsum1) : -INFINITY;
    }

    // ---- online softmax update (per head 2c, 2c+1)
    float mloc0 = -INFINITY, mloc1 = -INFINITY;
#pragma unroll
    for (int tt = 0; tt < C::kTiles; ++tt) {
      mloc0 = fmaxf(mloc0, fmaxf(sc[tt][0], sc[tt][2]));
      mloc1 = fmaxf(mloc1, fmaxf(sc[tt][1], sc[tt][3]));
    }
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      mloc0 = fmaxf(mloc0, __shfl_xor_sync(kFull, mloc0, x));
      mloc1 = fmaxf(mloc1, __shfl_xor_sync(kFull, mloc1, x));
    }
    const float mn0 = fmaxf(m_run[0], mloc0), mn1 = fmaxf(m_run[1], mloc1);
    const float mu0 = (mn0 == -INFINITY) ? 0.0f : mn0;
    const float mu1 = (mn1 == -INFINITY) ? 0.0f : mn1;
    const float al0 = ex2(m_run[0] - mu0), al1 = ex2(m_run[1] - mu1);
    m_run[0] = mn0;
    m_run[1] = mn1;
    l_run[0] *= al0;
    l_run[1] *= al1;
    z_run[0] *= al0;
    z_run[1] *= al1;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      acc[k][0] *= al0;
      acc[k][1] *= al1;
      acc[k][2] *= al0;
      acc[k][3] *= al1;
    }

    // ---- probabilities, V terms, and the PV product per tile
#pragma unroll
    for (int tt = 0; tt < C::kTiles; ++tt) {
      const float p0 = ex2(sc[tt][0] - mu0), p1 = ex2(sc[tt][1] - mu1);
      const float p2 = ex2(sc[tt][2] - mu0), p3 = ex2(sc[tt][3] - mu1);
      const uint32_t mv0 =
          *reinterpret_cast<const uint32_t*>(vst + P * (kHeadDim / 2) + (16 * tt + g) * 4);
      const uint32_t mv1 =
          *reinterpret_cast<const uint32_t*>(vst + P * (kHeadDim / 2) + (16 * tt + g + 8) * 4);
      const bool v0 = page_ok && (tok_base + 16 * tt + g) < L;
      const bool v1 = page_ok && (tok_base + 16 * tt + g + 8) < L;
      const float sv0 = v0 ? __half2float(__ushort_as_half(uint16_t(mv0 & 0xFFFF))) : 0.0f;
      const float zv0 = v0 ? __half2float(__ushort_as_half(uint16_t(mv0 >> 16))) : 0.0f;
      const float sv1 = v1 ? __half2float(__ushort_as_half(uint16_t(mv1 & 0xFFFF))) : 0.0f;
      const float zv1 = v1 ? __half2float(__ushort_as_half(uint16_t(mv1 >> 16))) : 0.0f;
      l_run[0] += p0 + p2;
      l_run[1] += p1 + p3;
      z_run[0] += p0 * zv0 + p2 * zv1;
      z_run[1] += p1 * zv0 + p3 * zv1;
      // (p*s) for head 2c / 2c+1 over tokens (g, g+8) -> B layout for head g
      const uint32_t X = pack_half2(p0 * sv0, p2 * sv1);
      const uint32_t Y = pack_half2(p1 * sv0, p3 * sv1);
      const int src0 = 8 * c + (g >> 1);
      const uint32_t xa = __shfl_sync(kFull, X, src0);
      const uint32_t ya = __shfl_sync(kFull, Y, src0);
      const uint32_t xb = __shfl_sync(kFull, X, src0 + 4);
      const uint32_t yb = __shfl_sync(kFull, Y, src0 + 4);
      const uint32_t va = (g & 1) ? ya : xa;  // tokens (2c, 2c+8)
      const uint32_t vb = (g & 1) ? yb : xb;  // tokens (2c+1, 2c+9)
      const uint32_t b0 = prmt(va, vb, 0x5410u);
      const uint32_t b1 = prmt(va, vb, 0x7632u);

      const uint8_t* vrow = vst + (16 * tt) * (kHeadDim / 2) + 8 * g;
      const uint2 r0 = *reinterpret_cast<const uint2*>(vrow + (2 * c) * (kHeadDim / 2));
      const uint2 r1 = *reinterpret_cast<const uint2*>(vrow + (2 * c + 1) * (kHeadDim / 2));
      const uint2 r2 = *reinterpret_cast<const uint2*>(vrow + (2 * c + 8) * (kHeadDim / 2));
      const uint2 r3 = *reinterpret_cast<const uint2*>(vrow + (2 * c + 9) * (kHeadDim / 2));
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint32_t w0 = (k < 4) ? r0.x : r0.y;
        const uint32_t w1 = (k < 4) ? r1.x : r1.y;
        const uint32_t w2 = (k < 4) ? r2.x : r2.y;
        const uint32_t w3 = (k < 4) ? r3.x : r3.y;
        const uint32_t sel = uint32_t(k & 3) | (uint32_t((k & 3) + 4) << 8);
        const uint32_t x01 = prmt(w0, w1, sel);
        const uint32_t x23 = prmt(w2, w3, sel);
        uint32_t a[4];
        a[0] = hsub_1024(and_or(x01, 0x000F000Fu, kMagic));
        a[1] = hfma_hi(and_or(x01, 0x00F000F0u, kMagic));
        a[2] = hsub_1024(and_or(x23, 0x000F000Fu, kMagic));
        a[3] = hfma_hi(and_or(x23, 0x00F000F0u, kMagic));
        mma_16816(acc[k], a, b0, b1);
      }
    }

    __syncwarp();
    if (lane == 0 && i + C::kStages < n_my) issue(i + C::kStages);
  }

  if (failed) {
    if (lane == 0) report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
    // let this warp's copies in flight land before the CTA's memory is reused
    for (int i = waited; i < n_my && i < waited + C::kStages; ++i)
      (void)mbar_wait_bounded(&wbars[i % C::kStages], (i / C::kStages) & 1);
  }

  // ---- cross-thread reductions of l and the z term (lanes sharing c)
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l_run[0] += __shfl_xor_sync(kFull, l_run[0], x);
    l_run[1] += __shfl_xor_sync(kFull, l_run[1], x);
    z_run[0] += __shfl_xor_sync(kFull, z_run[0], x);
    z_run[1] += __shfl_xor_sync(kFull, z_run[1], x);
  }
  __syncthreads();  // every warp is done with its ring: reuse it

  float* red_acc = reinterpret_cast<float*>(smem);                     // [4][8][132]
  float* red_m = red_acc + kWarps * kMaxGroup * kRedStride;           // [4][8]
  float* red_l = red_m + kWarps * kMaxGroup;
  float* red_z = red_l + kWarps * kMaxGroup;
  if (g == 0) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      red_m[warp * kMaxGroup + 2 * c + hh] = m_run[hh];
      red_l[warp * kMaxGroup + 2 * c + hh] = l_run[hh];
      red_z[warp * kMaxGroup + 2 * c + hh] = z_run[hh];
    }
  }
  {
    float* base0 = red_acc + (warp * kMaxGroup + 2 * c) * kRedStride;
    float* base1 = base0 + kRedStride;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      base0[16 * g + 2 * k] = acc[k][0];
      base1[16 * g + 2 * k] = acc[k][1];
      base0[16 * g + 2 * k + 1] = acc[k][2];
      base1[16 * g + 2 * k + 1] = acc[k][3];
    }
  }
  __syncthreads();

  // ---- merge the warps: thread = output dimension
  const int dd = tid;  // kThreads == kHeadDim
  for (int h = 0; h < G; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, red_m[w * kMaxGroup + h]);
    const float Mu = (M == -INFINITY) ? 0.0f : M;
    float num = 0.0f, den = 0.0f, zz = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float f = ex2(red_m[w * kMaxGroup + h] - Mu);
      num += red_acc[(w * kMaxGroup + h) * kRedStride + dd] * f;
      den += red_l[w * kMaxGroup + h] * f;
      zz += red_z[w * kMaxGroup + h] * f;
    }
    num += zz;
    if (direct) {
      qs[h * kHeadDim + dd] = (den > 0.0f) ? num / den : 0.0f;
    } else {
      const int64_t row = (int64_t(seq) * p.num_q_heads + hq0 + h) * p.num_splits + split;
      p.part_o[row * kHeadDim + dd] = num;
      if (dd == 0) {
        p.part_ml[2 * row] = M;
        p.part_ml[2 * row + 1] = den;
      }
    }
  }
  if (direct) {
    __syncthreads();
    if (p.rotate_v) smem_fwht(qs, G, p.block_h);
    const float post = p.rotate_v ? p.c_h : 1.0f;
    for (int idx = tid; idx < G * kHeadDim; idx += kThreads)
      p.out[(int64_t(seq) * p.num_q_heads + hq0) * kHeadDim + idx] = qs[idx] * post;
  }
}

// K3: merge the split partials of one (sequence, q-head), normalise, and
// rotate V's output back.  Warp w folds splits w, w+4, ... with lane l owning
// dims 4l..4l+3 (coalesced float4 reads), then the four warps are summed.
__global__ void __launch_bounds__(kHeadDim) combine_kernel(const DecodeParams p) {
  __shared__ float red[kWarps][kHeadDim];
  __shared__ float wmax[kWarps], wden[kWarps];
  __shared__ float buf[kHeadDim];
  const int hq = blockIdx.x;
  const int seq = blockIdx.y;
  const int tid = threadIdx.x;
  const int warp = tid >> 5, lane = tid & 31;
  int L = p.seq_lens[seq];
  if (L < 0 || L > p.max_seq_len) L = 0;
  const int n_pages = (L + p.page_size - 1) / p.page_size;
  const int ns = (n_pages + p.pages_per_split - 1) / p.pages_per_split;
  const int64_t row0 = (int64_t(seq) * p.num_q_heads + hq) * p.num_splits;
  const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + row0;

  float m = -INFINITY;
  for (int s = tid; s < ns; s += kHeadDim) m = fmaxf(m, ml[s].x);
#pragma unroll
  for (int x = 16; x >= 1; x >>= 1) m = fmaxf(m, __shfl_xor_sync(kFull, m, x));
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  const float M = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
  const float Mu = (M == -INFINITY) ? 0.0f : M;

  float4 acc = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  float den = 0.0f;
  const float4* po = reinterpret_cast<const float4*>(p.part_o + row0 * kHeadDim) + lane;
#pragma unroll 4
  for (int s = warp; s < ns; s += kWarps) {
    const float2 v = ml[s];
    const float4 o = po[int64_t(s) * (kHeadDim / 4)];
    const float f = ex2(v.x - Mu);
    den += v.y * f;
    acc.x += o.x * f;
    acc.y += o.y * f;
    acc.z += o.z * f;
    acc.w += o.w * f;
  }
  red[warp][4 * lane + 0] = acc.x;
  red[warp][4 * lane + 1] = acc.y;
  red[warp][4 * lane + 2] = acc.z;
  red[warp][4 * lane + 3] = acc.w;
  if (lane == 0) wden[warp] = den;
  __syncthreads();
  const float num = red[0][tid] + red[1][tid] + red[2][tid] + red[3][tid];
  const float dsum = wden[0] + wden[1] + wden[2] + wden[3];
  float val = (ns > 0 && dsum > 0.0f) ? num / dsum : 0.0f;
  if (p.rotate_v) {
    buf[tid] = val;
    __syncthreads();
    smem_fwht(buf, 1, p.block_h);
    val = buf[tid] * p.c_h;
  }
  p.out[(int64_t(seq) * p.num_q_heads + hq) * kHeadDim + tid] = val;
}

template <int P>
cudaError_t launch_p(const DecodeParams& p, cudaStream_t stream) {
  using C = Cfg<P>;
  cudaError_t err = cudaFuncSetAttribute(paged_decode_kernel<P>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  dim3 grid(p.num_splits, p.num_kv_heads, p.num_seqs);
  paged_decode_kernel<P><<<grid, kThreads, C::kSmem, stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess || p.num_splits == 1) return err;
  combine_kernel<<<dim3(p.num_q_heads, p.num_seqs), kHeadDim, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_paged_decode(const DecodeParams& p, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  switch (p.page_size) {
    case 16: return launch_p<16>(p, stream);
    case 32: return launch_p<32>(p, stream);
    case 64: return launch_p<64>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace saw
