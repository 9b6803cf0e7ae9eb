// prefill_attn.cu -- chunked-prefill attention over the paged INT4 cache on
// the 5th-generation tensor cores (tcgen05; accumulators in tensor memory).
//
// Pages: youngju.dev "INT4 KV-cache quantization", "Why the KV Cache Is the
// Real Bottleneck" and gist.science "SAW-INT4", s.1 (the method has to live
// inside engines that run fused, FlashAttention-style attention over paged
// KV); the attention itself is the decode's, with the reading that a query
// at position p of its sequence attends causally to cached tokens 0..p.
// The chunk's K/V are appended (saw_quantize_append) before this runs.
//
// Design (sm_103a):
//  * CTA = (block of 128 query rows, kv-head, sequence); a row is one
//    (query token, q-head of the group) pair, token-major, so the whole GQA
//    group shares every K/V tile.  Keys go by tiles of 64.
//  * Fourteen warps, specialised:
//      0-7   softmax: two threads per row r (tensor-memory lane r), one per
//            half: keys 32h .. 32h+31 of a tile, and dims 64h .. 64h+63 of
//            q' and of the output.  They rotate q' (the stride-64 butterfly
//            step through shared memory), scale it by 2^S and write it as
//            binary16 hi + lo operands; per tile they read their half of the
//            scores from tensor memory, mask, exchange the row max with the
//            other half (named barrier), rescale their half of the output
//            accumulator in tensor memory when the max grows, and write p*s_V
//            as the binary16 A operand of the P.V product; at the end they
//            normalise, inverse-rotate V and store.
//      8-11  expanders: widen a raw INT4 tile into the K and V operands
//            (both keys x dims, the same layout), each code n as the
//            binary16 subnormal n * 2^-24 (exact), and unpack the tile's
//            (s, z) metadata (binary16 or bfloat16) to binary32.
//      12    producer: 16-key slices (codes and metadata of K and V) through
//            a 4-stage ring with the bulk-copy engine.
//      13    MMA: S = Q' K^T (M 128, N 64, K 128; q' hi and lo accumulate
//            into the same scores) and O += P V (M 128, N 128, K 64) with
//            tcgen05.mma, completion signalled by tcgen05.commit; the warp
//            also allocates the 256 tensor-memory columns (S double-buffered
//            at columns 0 and 64, O at 128).
//    The producer and MMA warps run converged on warp-uniform values, and one
//    lane chosen by elect.sync inside the inline PTX issues each copy, MMA,
//    commit and barrier arrival (instead of a lane-0 branch: the copy and MMA
//    instructions take uniform registers, and a divergent lane-0 region
//    converts every operand to them per instruction).
//  * Operands are unswizzled 8-row x 16-byte core matrices: K-major, except
//    V, which the P.V product reads MN-major (dims contiguous per key).
//    Every mbarrier wait is bounded to about a second; the softmax warps,
//    which also meet at a named barrier, never leave their loop early (a
//    failed wait only marks the result), so that barrier always completes.
#include <type_traits>

#include "saw_device.cuh"
#include "saw_int4.h"
#include "saw_quant_row.cuh"
#include "saw_tcgen05.cuh"

namespace saw {
namespace {

constexpr int kBM = 128;               // query rows per CTA (MMA M)
constexpr int kBN = 64;                // keys per tile
constexpr int kRawStages = 4;
constexpr int kSoftWarps = 8;
constexpr int kTThreads = 32 * (kSoftWarps + 4 + 2);  // softmax, expanders, producer, MMA
constexpr int kWarpExp0 = kSoftWarps;
constexpr int kWarpProd = kSoftWarps + 4;
constexpr int kWarpMma = kSoftWarps + 5;
constexpr uint32_t kAllLanes = 0xFFFFFFFFu;

constexpr int kKxBytes = kBN * kHeadDim * 2;       // K operand of one tile
constexpr int kVxBytes = kBN * kHeadDim * 2;       // V operand of one tile
constexpr int kRawCodes = kBN * (kHeadDim / 2);    // 4096 code bytes per tensor
// raw stage: K codes | V codes | K meta | V meta | slice-ok word
constexpr int kRawV = kRawCodes;
constexpr int kRawKM = 2 * kRawCodes;
constexpr int kRawVM = kRawKM + kBN * 4;
constexpr int kRawOk = kRawVM + kBN * 4;
constexpr int kRawBytes = kRawOk + 16;
constexpr int kMetaBytes = kBN * 16 + 16;          // s_k[64], z_k[64], s_v[64], z_v[64] + ok word

constexpr int kOffKx = 0;
constexpr int kOffVx = kOffKx + 2 * kKxBytes;
constexpr int kOffRaw = kOffVx + 2 * kVxBytes;
constexpr int kOffMeta = kOffRaw + kRawStages * kRawBytes;
constexpr int kOffXm = kOffMeta + 2 * kMetaBytes;          // f32 [2 tiles][2 halves][128] row maxima
constexpr int kOffXl = kOffXm + 2 * 2 * kBM * 4;           // f32x2 [2 halves][128]
constexpr int kOffBar = kOffXl + 2 * kBM * 8;
enum {
  kRawFull = 0, kRawEmpty = 4, kMetaFull = 8, kMetaEmpty = 10, kKxFull = 12, kKxEmpty = 14,
  kVxFull = 16, kPvDone = 18, kSFull = 20, kSEmpty = 22, kPFull = 24, kMmaDone = 26, kNumBars = 27
};
constexpr int kOffTmem = kOffBar + kNumBars * 8;
constexpr int kTSmem = kOffTmem + 16;
static_assert(kTSmem <= 227 * 1024, "shared memory");
static_assert(kRawBytes % 16 == 0 && kMetaBytes % 16 == 0 && kOffBar % 8 == 0, "alignment");
// the 128 x 128 binary32 exchange of the q' and output rotations reuses the
// K/V operand buffers (free before the first tile and after the last)
static_assert(2 * kKxBytes + 2 * kVxBytes >= kBM * kHeadDim * 4, "exchange space");
// tensor memory: S (2 x 64 columns), O (128), P (2 x 32 columns of binary16
// pairs), and the A operands q' hi and lo (64 columns of binary16 pairs
// each): the score products read only K from shared memory
constexpr uint32_t kTmemCols = 512;  // 448 used
constexpr uint32_t kColO = 128;
constexpr uint32_t kColP = 256;
constexpr uint32_t kColQh = 320;
constexpr uint32_t kColQl = 384;
// named barriers 1 .. 4: softmax warps w and w + 4, which share rows 32w .. 32w+31
constexpr int kSoftBar = 1;

// 2^e for -126 <= e <= 127, exactly
__device__ __forceinline__ float pow2i(int e) { return __uint_as_float(uint32_t(127 + e) << 23); }

// tcgen05 MMA / commit issued by one elected lane of a converged warp whose
// operands are warp-uniform (the same lane is elected every time: the MMAs
// and the commits that track them come from one thread).
__device__ __forceinline__ void umma_f16_ta_elect(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                  uint32_t idesc, bool accumulate) {
  asm volatile(
      "{\n\t.reg .pred p, e;\n\tsetp.ne.u32 p, %4, 0;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
      : "memory");
}
__device__ __forceinline__ void umma_commit_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
          smem_u32(bar))
      : "memory");
}
// Executed by a whole warp with warp-uniform operands: one elected lane
// arms the mbarrier / issues the bulk copy.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t"
      "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
      : "memory");
}
__device__ __forceinline__ void mbar_arrive_elect(uint64_t* bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t"
      "@p mbarrier.arrive.shared::cta.b64 _, [%0];\n\t}" ::"r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ void bulk_g2s_elect(uint32_t dst, const void* src, uint32_t bytes,
                                               uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t"
      "@p cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n\t}" ::
          "r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}
// Byte-permute selectors that build a binary16 pair (x byte m, y byte m) with
// zero upper bytes from two nibble planes x, y: the zeros replicate the sign
// bit of a byte below 128 (selector nibble with bit 3 set).
__device__ __constant__ const uint32_t kPairSel[4] = {0x8480u, 0x9591u, 0xA6A2u, 0xB7B3u};

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// The barrier of the two softmax warps that share this thread's rows;
// returns the AND of `ok` over their threads.
__device__ __forceinline__ bool soft_sync_and(bool ok) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
      "barrier.cta.red.and.pred q, %2, %3, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(uint32_t(ok)), "r"(kSoftBar + int((threadIdx.x >> 5) & 3)), "r"(64)
      : "memory");
  return r != 0;
}

// Half of a row's block-diagonal Sylvester butterfly: the 64 values this
// thread holds (dims 64h .. 64h+63), strides 1 .. 32 (unscaled).
__device__ __forceinline__ void half_fwht(float (&v)[64], int hblk) {
#pragma unroll
  for (int s = 1; s < 64; s <<= 1) {
    if (s < hblk) {
#pragma unroll
      for (int i = 0; i < 64; ++i)
        if (!(i & s)) {
          const float a = v[i], b = v[i + s];
          v[i] = a + b;
          v[i + s] = a - b;
        }
    }
  }
}

// The stride-64 step (h = 128): lower half gets a + b, upper half a - b,
// through a [128][128] binary32 scratch row in shared memory.
__device__ __forceinline__ void stride64_step(float (&v)[64], float* scratch_row, int half) {
#pragma unroll
  for (int k = 0; k < 16; ++k)
    reinterpret_cast<float4*>(scratch_row + 64 * half)[k] =
        make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
  (void)soft_sync_and(true);
  const float* other = scratch_row + 64 * (1 - half);
#pragma unroll
  for (int k = 0; k < 16; ++k) {
    const float4 o = reinterpret_cast<const float4*>(other)[k];
    const float w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int i = 4 * k + e;
      v[i] = half ? (w[e] - v[i]) : (v[i] + w[e]);
    }
  }
}

// try_wait with a suspend-time hint: a thread whose phase has not completed
// may be parked for up to `ns` nanoseconds (woken earlier when the phase
// completes) instead of returning at once to poll again.
__device__ __forceinline__ bool mbar_try_wait_for(uint64_t* bar, uint32_t parity, uint32_t ns) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(ns)
      : "memory");
  return ok != 0;
}

// mbar_wait_bounded with the suspend hint on every try.
__device__ __forceinline__ bool mbar_wait_bounded_for(uint64_t* bar, uint32_t parity, uint32_t ns) {
  if (mbar_try_wait_for(bar, parity, ns)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait_for(bar, parity, ns)) {
    if (clock64() - t0 > kWaitLimitCycles) return false;
  }
  return true;
}

// The other roles' waiting threads are parked on the mbarrier (woken when
// its phase completes, or after kSuspendNs to re-check the time limit)
// rather than polling, leaving their scheduler's issue slots to the softmax
// warps, which spin (they are on the critical path).
constexpr uint32_t kSuspendNs = 20000;

// The softmax warps' wait; a wait after a failure returns at once.
__device__ __forceinline__ bool wait_soft(uint64_t* bar, uint32_t parity, bool& failed) {
  if (failed) return false;
  const bool ok = __all_sync(kAllLanes, mbar_wait_bounded(bar, parity));
  failed = !ok;
  return ok;
}

// The other roles' wait.
__device__ __forceinline__ bool wait_sleep(uint64_t* bar, uint32_t parity) {
  return mbar_wait_bounded_for(bar, parity, kSuspendNs);
}
__device__ __forceinline__ bool wait_sleep_all(uint64_t* bar, uint32_t parity) {
  return __all_sync(kAllLanes, wait_sleep(bar, parity));
}

// One expander thread's share of widening a tile's 64 x 128 codes into a
// binary16 operand: element (key n, dim k) at (k/8)*1024 + n*16 + (k%8)*2,
// each code n as the subnormal n * 2^-24 (exact).  Thread te takes key
// te % 64 and dims 64 (te / 64) .. + 63 in two 16-byte pieces of codes.
__device__ __forceinline__ void widen_codes(const uint8_t* codes, uint8_t* dst, int te) {
  const int n = te & 63, hk = te >> 6;
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    const int q = (2 * hk + s + (n >> 1)) & 3;  // 16-byte piece: dims 32q .. 32q+31
    const uint4 w = *reinterpret_cast<const uint4*>(codes + n * 64 + 16 * q);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      // byte m of the word holds dims 2m (low nibble) and 2m+1: one
      // permute per pair from the low- and high-nibble planes
      const uint32_t lo = ws[u] & 0x0F0F0F0Fu, hi = (ws[u] >> 4) & 0x0F0F0F0Fu;
      *reinterpret_cast<uint4*>(dst + (4 * q + u) * 1024 + n * 16) =
          make_uint4(prmt(lo, hi, kPairSel[0]), prmt(lo, hi, kPairSel[1]),
                     prmt(lo, hi, kPairSel[2]), prmt(lo, hi, kPairSel[3]));
    }
  }
}

// F16IN: q is binary16 (else bfloat16); BFM: the caches' (scale, zero)
// words are bfloat16 (else binary16).
template <int P, bool F16IN, bool BFM>
__global__ void __launch_bounds__(kTThreads, 1) prefill_tc_kernel(const PrefillParams p) {
  pdl_wait_then_release();
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kOffBar);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  constexpr int kChunk = P * (kHeadDim / 2 + 4);

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
  const int row0 = rb * kBM;
  if (row0 >= R) return;
  const int row_end = min(R, row0 + kBM);
  const int pos_base = L - ql;
  const int pos_max = pos_base + (row_end - 1) / G;
  const int n_tiles = pos_max / kBN + 1;
  const int n_pages = (L + P - 1) / P;

  if (tid == 0) {
    for (int s = 0; s < kRawStages; ++s) {
      mbar_init(&bars[kRawFull + s], 1);
      mbar_init(&bars[kRawEmpty + s], 4);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&bars[kMetaFull + b], 4);
      mbar_init(&bars[kMetaEmpty + b], kSoftWarps);
      mbar_init(&bars[kKxFull + b], 4);
      mbar_init(&bars[kKxEmpty + b], 1);
      mbar_init(&bars[kVxFull + b], 4);
      mbar_init(&bars[kPvDone + b], 1);
      mbar_init(&bars[kSFull + b], 1);
      mbar_init(&bars[kSEmpty + b], kSoftWarps);
      mbar_init(&bars[kPFull + b], kSoftWarps);
    }
    mbar_init(&bars[kMmaDone], 1);
    mbar_fence_init();
  }
  if (warp == kWarpMma) tmem_alloc(tslot, kTmemCols);

  // ---- softmax warps: q' rows into the A operands
  const int half = warp >> 2;                // softmax threads: keys / dims half
  const int r = 32 * (warp & 3) + lane;      // and row (tensor-memory lane)
  bool row_valid = false;
  int pos_r = -1, out_t = 0, out_h = 0;
  float rowA = 0.0f, qc = 0.0f, qsc = 0.0f;
  float2* xl = reinterpret_cast<float2*>(smem + kOffXl);
  float qv[64];
  if (warp < kSoftWarps) {
    const int row = row0 + r;
    row_valid = row < row_end;
    float (&v)[64] = qv;
    if (row_valid) {
      out_t = row / G;
      out_h = row - out_t * G;
      pos_r = pos_base + out_t;
      const uint4* src = reinterpret_cast<const uint4*>(
          p.q + (int64_t(q0 + out_t) * p.num_q_heads + kvh * G + out_h) * kHeadDim + 64 * half);
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 w = src[k];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          v[8 * k + 2 * j] = in_lo(ws[j], F16IN);
          v[8 * k + 2 * j + 1] = in_hi(ws[j], F16IN);
        }
      }
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] = 0.0f;
    }
    if (p.rotate_k) {
      // the butterfly steps commute: stride 64 first (through shared memory),
      // then 1 .. 32 in registers
      if (p.block_h == kHeadDim)
        stride64_step(v, reinterpret_cast<float*>(smem + kOffKx) + r * kHeadDim, half);
      half_fwht(v, p.block_h);
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] *= p.c_h;
    }
    float sum = 0.0f, mx = 0.0f;
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      sum += v[i];
      mx = fmaxf(mx, fabsf(v[i]));
    }
    xl[half * kBM + r] = make_float2(sum, mx);
    (void)soft_sync_and(true);
    const float2 o = xl[(1 - half) * kBM + r];
    sum += o.x;
    mx = fmaxf(mx, o.y);
    // 2^S with max |q'| 2^S < 2^14: S = 140 - (biased exponent of the max),
    // kept within [-100, 100]
    const int E = int((__float_as_uint(mx) >> 23) & 0xFFu);
    const int S = min(100, max(-100, 140 - E));
    qsc = pow2i(S);
    // K operand codes are n * 2^-24, so acc = 2^(S-24) q'.n; the logit is
    // rowA * (s_k acc + qc z_k) with qc = sum(q') / rowA
    rowA = p.q_scale * pow2i(24 - S);
    qc = (sum * p.q_scale) / rowA;
  }
  tc_fence_before();
  __syncthreads();  // tensor memory allocated
  tc_fence_after();
  const uint32_t tmem = *tslot;
  if (warp < kSoftWarps) {
    // q' as the A operand in tensor memory: row r in lane r, dims (2j, 2j+1)
    // in column j; this thread's dims 64h .. 64h+63 fill columns 32h .. 32h+31
    const uint32_t trow = tmem + (uint32_t(32 * (warp & 3)) << 16) + 32 * half;
#pragma unroll
    for (int kk = 0; kk < 8; ++kk) {
      uint32_t hw[4], lw[4];
#pragma unroll
      for (int m = 0; m < 4; ++m) {
        const float x0 = qv[8 * kk + 2 * m] * qsc, x1 = qv[8 * kk + 2 * m + 1] * qsc;
        const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
        hw[m] = uint32_t(__half_as_ushort(h0)) | (uint32_t(__half_as_ushort(h1)) << 16);
        lw[m] = pack_half2(x0 - __half2float(h0), x1 - __half2float(h1));
      }
      tmem_st4u(trow + kColQh + 4 * kk, hw);
      tmem_st4u(trow + kColQl + 4 * kk, lw);
    }
    tmem_wait_st();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();

  if (warp == kWarpProd) {
    // ---------------------------------------------------------- producer
    const int32_t* btab = p.block_tables + int64_t(seq) * p.max_blocks;
    int ids = -1, ids_base = -32, issued = 0;
    bool failed = false;
    for (int i = 0; i < n_tiles; ++i) {
      const int rs = i % kRawStages;
      if (i >= kRawStages && !wait_sleep_all(&bars[kRawEmpty + rs], ((i / kRawStages) - 1) & 1)) {
        failed = true;
        break;
      }
      int pid[4];
      int okm = 0;
#pragma unroll
      for (int sl = 0; sl < 4; ++sl) {
        const int lp = (i * kBN + 16 * sl) / P;
        if (lp >= ids_base + 32) {
          ids_base = lp - (lp & 31);
          const int e = ids_base + lane;
          ids = (e < p.max_blocks && e < n_pages) ? btab[e] : -1;
        }
        int id = __shfl_sync(kAllLanes, ids, lp - ids_base);
        if (lp >= n_pages) {
          id = -1;  // past the sequence: nothing to copy, keys masked
        } else if (id < 0 || id >= p.num_pages) {
          if (lane == 0) report(p.dev_status, SAW_ERR_DEVICE_INDEX);
          id = -1;
        }
        pid[sl] = id;
        okm |= (id >= 0) << sl;
      }
      {
        // the whole warp on warp-uniform values; one elected lane arms the
        // barrier and issues the copies
        uint8_t* st = smem + kOffRaw + rs * kRawBytes;
        if (lane == 0) *reinterpret_cast<int*>(st + kRawOk) = okm;
        __syncwarp();
        const uint32_t nbytes = __popc(okm) * (2 * 1024 + 2 * 64);
        const uint32_t bar = smem_u32(&bars[kRawFull + rs]);
        if (nbytes == 0) {
          if (lane == 0) mbar_arrive(&bars[kRawFull + rs]);
        } else {
          mbar_arrive_expect_tx_elect(bar, nbytes);
          const uint32_t st32 = smem_u32(st);
#pragma unroll
          for (int sl = 0; sl < 4; ++sl) {
            if (pid[sl] < 0) continue;
            const int part = ((i * kBN + 16 * sl) % P) / 16;
            const int64_t off = (int64_t(pid[sl]) * p.num_kv_heads + kvh) * kChunk;
            const int64_t codes = off + part * 1024;
            const int64_t meta = off + P * (kHeadDim / 2) + part * 64;
            bulk_g2s_elect(st32 + sl * 1024, p.k_cache + codes, 1024, bar);
            bulk_g2s_elect(st32 + kRawV + sl * 1024, p.v_cache + codes, 1024, bar);
            bulk_g2s_elect(st32 + kRawKM + sl * 64, p.k_cache + meta, 64, bar);
            bulk_g2s_elect(st32 + kRawVM + sl * 64, p.v_cache + meta, 64, bar);
          }
        }
      }
      __syncwarp();
      issued = i + 1;
    }
    if (failed && lane == 0) report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
    // the CTA must not exit while a copy into its shared memory is in flight
    for (int i = max(0, issued - kRawStages); i < issued; ++i)
      (void)wait_sleep(&bars[kRawFull + i % kRawStages], (i / kRawStages) & 1);
  } else if (warp == kWarpMma) {
    // ---------------------------------------------------------- MMA issue
    // The whole warp runs the loop on warp-uniform values (every lane polls
    // the same barriers; lane 0's view decides); one elected lane issues each
    // MMA and commit, so descriptors and addresses stay uniform.
    {
      const uint32_t kx0 = smem_u32(smem + kOffKx), vx0 = smem_u32(smem + kOffVx);
      constexpr uint32_t idS = umma_idesc_f16(kBM, kBN);
      constexpr uint32_t idO = umma_idesc_f16(kBM, kHeadDim) | kUmmaBMnMajor;
      const uint64_t kxd[2] = {umma_desc(kx0, 1024, 128), umma_desc(kx0 + kKxBytes, 1024, 128)};
      const uint64_t vxd[2] = {umma_desc(vx0, 128, 1024), umma_desc(vx0 + kVxBytes, 128, 1024)};
      constexpr uint64_t kKxStep = (2 * 1024) >> 4, kVxStep = (2 * 128) >> 4;
      int nS = 0, nP = 0;
      bool ok = true;
      long long t_last = clock64();
      while (nP < n_tiles) {
        bool prog = false;
        bool sready = nS < n_tiles && mbar_test(&bars[kKxFull + (nS & 1)], (nS >> 1) & 1) &&
                      (nS < 2 || mbar_test(&bars[kSEmpty + (nS & 1)], ((nS >> 1) - 1) & 1));
        sready = __shfl_sync(0xFFFFFFFFu, sready, 0);
        if (sready) {
          const int b = nS & 1;
          tc_fence_after();
          const uint32_t sd = tmem + uint32_t(kBN * b);
          const uint64_t bd = kxd[b];
#pragma unroll
          for (int ks = 0; ks < kHeadDim / 16; ++ks)
            umma_f16_ta_elect(sd, tmem + kColQh + 8 * ks, bd + ks * kKxStep, idS, ks > 0);
#pragma unroll
          for (int ks = 0; ks < kHeadDim / 16; ++ks)
            umma_f16_ta_elect(sd, tmem + kColQl + 8 * ks, bd + ks * kKxStep, idS, true);
          umma_commit_elect(&bars[kSFull + b]);
          umma_commit_elect(&bars[kKxEmpty + b]);
          ++nS;
          prog = true;
        }
        bool pready = nP < nS && mbar_test(&bars[kPFull + (nP & 1)], (nP >> 1) & 1) &&
                      mbar_test(&bars[kVxFull + (nP & 1)], (nP >> 1) & 1);
        pready = __shfl_sync(0xFFFFFFFFu, pready, 0);
        if (pready) {
          const int bj = nP & 1;
          tc_fence_after();
          const uint64_t bd = vxd[bj];
#pragma unroll
          for (int ks = 0; ks < kBN / 16; ++ks)
            umma_f16_ta_elect(tmem + kColO, tmem + kColP + 32 * bj + 8 * ks, bd + ks * kVxStep, idO,
                              nP > 0 || ks > 0);
          umma_commit_elect(&bars[kPvDone + bj]);
          ++nP;
          prog = true;
        }
        if (prog) {
          t_last = clock64();
        } else {
          const bool late = __shfl_sync(0xFFFFFFFFu, clock64() - t_last > kWaitLimitCycles, 0);
          if (late) {
            ok = false;
            break;
          }
          __nanosleep(20);  // leave the scheduler's issue slots to the other roles
        }
      }
      if (!ok && lane == 0) report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
      // every MMA has completed before tensor memory is released
      umma_commit_elect(&bars[kMmaDone]);
      (void)wait_sleep(&bars[kMmaDone], 0);
    }
    __syncwarp();
  } else if (warp >= kWarpExp0) {
    // ---------------------------------------------------------- expanders
    const int te = tid - 32 * kWarpExp0;
    bool failed = false;
    for (int i = 0; i < n_tiles; ++i) {
      const int rs = i % kRawStages, b = i & 1;
      if (!wait_sleep_all(&bars[kRawFull + rs], (i / kRawStages) & 1)) { failed = true; break; }
      const uint8_t* st = smem + kOffRaw + rs * kRawBytes;
      // metadata, unpacked to binary32 for the softmax warps
      if (i >= 2 && !wait_sleep_all(&bars[kMetaEmpty + b], ((i >> 1) - 1) & 1)) { failed = true; break; }
      uint8_t* mb = smem + kOffMeta + b * kMetaBytes;
      if (te < kBN) {
        const uint32_t km = *reinterpret_cast<const uint32_t*>(st + kRawKM + 4 * te);
        const uint32_t vm = *reinterpret_cast<const uint32_t*>(st + kRawVM + 4 * te);
        float* mf = reinterpret_cast<float*>(mb);
        mf[te] = meta_lo(km, BFM);
        mf[kBN + te] = meta_hi(km, BFM);
        mf[2 * kBN + te] = meta_lo(vm, BFM);
        mf[3 * kBN + te] = meta_hi(vm, BFM);
      }
      if (te == 0) *reinterpret_cast<int*>(mb + kBN * 16) = *reinterpret_cast<const int*>(st + kRawOk);
      __syncwarp();
      mbar_arrive_elect(&bars[kMetaFull + b]);
      // K operand: element (key n, dim k) at (k/8)*1024 + n*16 + (k%8)*2
      if (i >= 2 && !wait_sleep_all(&bars[kKxEmpty + b], ((i >> 1) - 1) & 1)) { failed = true; break; }
      widen_codes(st, smem + kOffKx + b * kKxBytes, te);
      fence_async_smem();
      __syncwarp();
      mbar_arrive_elect(&bars[kKxFull + b]);
      // V operand: element (key n, dim k) at (k/8)*1024 + n*16 + (k%8)*2, the
      // K operand's layout (read by the P.V product as MN-major)
      if (i >= 2 && !wait_sleep_all(&bars[kPvDone + b], ((i >> 1) - 1) & 1)) { failed = true; break; }
      widen_codes(st + kRawV, smem + kOffVx + b * kVxBytes, te);
      fence_async_smem();
      __syncwarp();
      mbar_arrive_elect(&bars[kVxFull + b]);
      mbar_arrive_elect(&bars[kRawEmpty + rs]);
    }
    if (failed && lane == 0) report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
  } else {
    // ---------------------------------------------------------- softmax
    const uint32_t trow = tmem + (uint32_t(32 * (warp & 3)) << 16);
    float* xm = reinterpret_cast<float*>(smem + kOffXm);
    const int kq = 32 * half;  // this thread's keys within a tile
    float m_run = -INFINITY, l_run = 0.0f, pz = 0.0f;
    bool failed = false;
    for (int i = 0; i < n_tiles; ++i) {
      const int b = i & 1;
      // every wait before the named barrier, so that the barrier always meets
      wait_soft(&bars[kSFull + b], (i >> 1) & 1, failed);
      wait_soft(&bars[kMetaFull + b], (i >> 1) & 1, failed);
      if (i >= 2) wait_soft(&bars[kPvDone + b], ((i >> 1) - 1) & 1, failed);  // P buffer b free
      tc_fence_after();
      float t[32];
      tmem_ld32(trow + uint32_t(kBN * b + kq), t);
      tc_fence_before();
      __syncwarp();
      mbar_arrive_elect(&bars[kSEmpty + b]);
      const float4* msk = reinterpret_cast<const float4*>(smem + kOffMeta + b * kMetaBytes);
      const float4* mzk = msk + kBN / 4;
      const float4* msv = msk + 2 * (kBN / 4);
      const float4* mzv = msk + 3 * (kBN / 4);
      const int okm = *reinterpret_cast<const int*>(smem + kOffMeta + b * kMetaBytes + kBN * 16);
      const int k0 = i * kBN + kq;
      const bool all_vis = ((okm >> (2 * half)) & 3) == 3 && pos_r >= k0 + 31;
      float tm[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
      // Visible keys of this thread as bits of vm (bit j: key kq + j is at or
      // before the row's position and on a page that was copied).  Each loop
      // below has two unrolled copies: without the mask for the tiles a row
      // sees whole (nearly all), with it for the others.
      uint32_t vm = 0xFFFFFFFFu;
      if (!all_vis) {
        const int lim = pos_r - k0;  // keys j <= lim are at or before the row
        vm = lim >= 31 ? 0xFFFFFFFFu : (lim < 0 ? 0u : (2u << lim) - 1u);
        const int sl = (okm >> (2 * half)) & 3;  // 16-key slices 2h, 2h+1 copied
        vm &= ((sl & 1) ? 0x0000FFFFu : 0u) | ((sl & 2) ? 0xFFFF0000u : 0u);
      }
      // t = s_k acc + (qc z_k), two keys per instruction; masked keys -inf
      auto logits = [&](auto maskc) {
        constexpr bool kMask = decltype(maskc)::value;
        const float2 qc2 = make_float2(qc, qc);
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4) {
          const float4 sk = msk[kq / 4 + g4], zk = mzk[kq / 4 + g4];
          const int j = 4 * g4;
          float2 a = fma2(make_float2(sk.x, sk.y), make_float2(t[j], t[j + 1]),
                          mul2(qc2, make_float2(zk.x, zk.y)));
          float2 b = fma2(make_float2(sk.z, sk.w), make_float2(t[j + 2], t[j + 3]),
                          mul2(qc2, make_float2(zk.z, zk.w)));
          if (kMask) {
            a.x = ((vm >> j) & 1u) ? a.x : -INFINITY;
            a.y = ((vm >> (j + 1)) & 1u) ? a.y : -INFINITY;
            b.x = ((vm >> (j + 2)) & 1u) ? b.x : -INFINITY;
            b.y = ((vm >> (j + 3)) & 1u) ? b.y : -INFINITY;
          }
          t[j] = a.x;
          t[j + 1] = a.y;
          t[j + 2] = b.x;
          t[j + 3] = b.y;
          tm[g4 & 3] = fmaxf(tm[g4 & 3], fmaxf(fmaxf(a.x, a.y), fmaxf(b.x, b.y)));
        }
      };
      if (all_vis)
        logits(std::false_type{});
      else
        logits(std::true_type{});
      // row max over both halves
      const float th = rowA * fmaxf(fmaxf(tm[0], tm[1]), fmaxf(tm[2], tm[3]));
      xm[(b * 2 + half) * kBM + r] = th;
      const bool ok_all = soft_sync_and(!failed);
      failed = !ok_all;
      const float tmax = fmaxf(th, xm[(b * 2 + 1 - half) * kBM + r]);
      const bool grow = tmax > m_run;
      if (i > 0 && __any_sync(kAllLanes, grow) &&
          wait_soft(&bars[kPvDone + ((i - 1) & 1)], ((i - 1) >> 1) & 1, failed)) {
        // rescale this half of the output rows, after the previous P.V
        tc_fence_after();
        const float a = grow ? ex2(m_run - tmax) : 1.0f;
        const float2 a2 = make_float2(a, a);
        // eight columns at a time: few registers live beside the scores
#pragma unroll
        for (int cblk = 0; cblk < 8; ++cblk) {
          float o[8];
          tmem_ld8(trow + kColO + 64 * half + 8 * cblk, o);
#pragma unroll
          for (int j = 0; j < 8; j += 2) {
            const float2 v = mul2(make_float2(o[j], o[j + 1]), a2);
            o[j] = v.x;
            o[j + 1] = v.y;
          }
          tmem_st8(trow + kColO + 64 * half + 8 * cblk, o);
        }
        tmem_wait_st();
      }
      if (grow) {
        const float a = ex2(m_run - tmax);  // 0 while m_run is -inf
        l_run *= a;
        pz *= a;
        m_run = tmax;
      }
      const float nmu = (m_run == -INFINITY) ? 0.0f : -m_run;
      // p*s_V, binary16 pairs, into this lane's P columns: keys kq .. kq+31
      uint32_t pw[16];
      float la[4] = {0.0f, 0.0f, 0.0f, 0.0f}, za[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      // p = 2^(rowA t - m), two keys per instruction (each lane the same RN
      // steps as one key).  Masked keys have p = 0, and their (s_V, z_V) are
      // taken as 0: rows past the end may hold anything, even inf.
      auto probs = [&](auto maskc) {
        constexpr bool kMask = decltype(maskc)::value;
        const float2 rowA2 = make_float2(rowA, rowA), nmu2 = make_float2(nmu, nmu);
        float2 la01 = make_float2(0.0f, 0.0f), la23 = la01, za01 = la01, za23 = la01;
#pragma unroll
        for (int g4 = 0; g4 < 8; ++g4) {
          float4 sv = msv[kq / 4 + g4], zv = mzv[kq / 4 + g4];
          const int j = 4 * g4;
          if (kMask) {
            const bool l0 = (vm >> j) & 1u, l1 = (vm >> (j + 1)) & 1u;
            const bool l2 = (vm >> (j + 2)) & 1u, l3 = (vm >> (j + 3)) & 1u;
            sv = make_float4(l0 ? sv.x : 0.0f, l1 ? sv.y : 0.0f, l2 ? sv.z : 0.0f, l3 ? sv.w : 0.0f);
            zv = make_float4(l0 ? zv.x : 0.0f, l1 ? zv.y : 0.0f, l2 ? zv.z : 0.0f, l3 ? zv.w : 0.0f);
          }
          const float2 xa = fma2(rowA2, make_float2(t[j], t[j + 1]), nmu2);
          const float2 xb = fma2(rowA2, make_float2(t[j + 2], t[j + 3]), nmu2);
          const float2 pa = make_float2(ex2(xa.x), ex2(xa.y));
          const float2 pb = make_float2(ex2(xb.x), ex2(xb.y));
          la01 = add2(la01, pa);
          la23 = add2(la23, pb);
          za01 = fma2(pa, make_float2(zv.x, zv.y), za01);
          za23 = fma2(pb, make_float2(zv.z, zv.w), za23);
          const float2 sa = mul2(pa, make_float2(sv.x, sv.y));
          const float2 sb = mul2(pb, make_float2(sv.z, sv.w));
          pw[2 * g4] = pack_half2(sa.x, sa.y);
          pw[2 * g4 + 1] = pack_half2(sb.x, sb.y);
        }
        la[0] = la01.x;
        la[1] = la01.y;
        la[2] = la23.x;
        la[3] = la23.y;
        za[0] = za01.x;
        za[1] = za01.y;
        za[2] = za23.x;
        za[3] = za23.y;
      };
      if (all_vis)
        probs(std::false_type{});
      else
        probs(std::true_type{});
      tmem_st16u(trow + kColP + 32 * b + 16 * half, pw);
      tmem_wait_st();
      l_run += (la[0] + la[1]) + (la[2] + la[3]);
      pz += (za[0] + za[1]) + (za[2] + za[3]);
      tc_fence_before();
      __syncwarp();
      mbar_arrive_elect(&bars[kPFull + b]);
      mbar_arrive_elect(&bars[kMetaEmpty + b]);
    }
    if (failed && lane == 0) report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
    // ---- epilogue: this half of the output row from tensor memory, code
    // scale, sum(p z) and l over both halves, normalise, inverse V rotation
    const int last = n_tiles - 1;
    wait_soft(&bars[kPvDone + (last & 1)], (last >> 1) & 1, failed);
    tc_fence_after();
    float v[64];
#pragma unroll
    for (int cblk = 0; cblk < 8; ++cblk)
      tmem_ld8(trow + kColO + 64 * half + 8 * cblk, *reinterpret_cast<float(*)[8]>(v + 8 * cblk));
    xl[half * kBM + r] = make_float2(l_run, pz);
    (void)soft_sync_and(true);
    const float2 ot = xl[(1 - half) * kBM + r];
    const float l = l_run + ot.x, zz = pz + ot.y;
    const float inv = (!failed && l > 0.0f) ? 1.0f / l : 0.0f;
#pragma unroll
    for (int i = 0; i < 64; ++i) v[i] = fmaf(v[i], 16777216.0f, zz) * inv;  // codes were n 2^-24
    if (p.rotate_v) {
      // every product has completed (the last P.V came after all of them):
      // the K/V operand buffers are free for the exchange
      if (p.block_h == kHeadDim)
        stride64_step(v, reinterpret_cast<float*>(smem + kOffKx) + r * kHeadDim, half);
      half_fwht(v, p.block_h);
#pragma unroll
      for (int i = 0; i < 64; ++i) v[i] *= p.c_h;
    }
    if (row_valid) {
      float4* dst = reinterpret_cast<float4*>(
          p.out + (int64_t(q0 + out_t) * p.num_q_heads + kvh * G + out_h) * kHeadDim + 64 * half);
#pragma unroll
      for (int k = 0; k < 16; ++k)
        dst[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int P, bool F16IN, bool BFM>
cudaError_t launch_prefill_f(const PrefillParams& p, cudaStream_t stream) {
  auto kernel = prefill_tc_kernel<P, F16IN, BFM>;
  cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kTSmem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.row_blocks, p.num_kv_heads, p.num_seqs);
  cfg.blockDim = dim3(kTThreads);
  cfg.dynamicSmemBytes = kTSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int P>
cudaError_t launch_prefill_p(const PrefillParams& p, cudaStream_t stream) {
  if (p.in_f16)
    return p.meta_bf16 ? launch_prefill_f<P, true, true>(p, stream)
                       : launch_prefill_f<P, true, false>(p, stream);
  return p.meta_bf16 ? launch_prefill_f<P, false, true>(p, stream)
                     : launch_prefill_f<P, false, false>(p, stream);
}

}  // namespace

int prefill_rows_per_cta() { return kBM; }

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
