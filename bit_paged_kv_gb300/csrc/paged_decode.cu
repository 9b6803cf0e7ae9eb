// paged_decode.cu -- K2: split-K decode attention over the INT4 paged cache
// (SAW-INT4), with dequantization fused into the attention loop and the
// split merge done by the last split to finish.
//
// Pages: gist.science "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization
// for Real-World LLM Serving", s.2 point 3 (rotation and quantization fused
// into the decoding path, hidden inside a memory-bound data flow); youngju.dev
// "INT4 KV-cache quantization" (English), "The Rotation Trick": H is an
// orthogonal, undoable rotation, so q.k = (Hq).(Hk) and o = H^-1 o'.
//
// Design (sm_103a):
//  * One CTA per (split of the context, kv-head, sequence): 16 warps, one
//    CTA per SM, 8 warps, two CTAs per SM, or 4 warps, four per SM (this file
//    is compiled once per shape, and once more for head_dim 64 and 256 with
//    16 and 8 warps; the host plan picks the shape).  The whole GQA group
//    of the kv-head is served by the CTA, so each page is read from HBM
//    once, and q is rotated once per CTA.
//  * The split is cut into 16-token tiles; warp w of W takes tiles w, w+W, ...
//    through a private four-stage shared-memory ring filled by the bulk-copy
//    engine (cp.async.bulk + mbarrier complete_tx).  A stage holds one tile's
//    K and V codes and their (scale, zero) words: a whole 16-token page, or
//    16 rows of a larger page (codes and metadata copied separately).  A warp
//    consumes its tiles two at a time; the two share one softmax update, and
//    (four-stage rings) one mbarrier: one wait, one refill arrival.  With a
//    clean chunk list the whole warp runs the refill on warp-uniform values
//    and one elected lane arms the barrier and issues the copies; otherwise
//    lane 0 does it with the checks.
//  * The loop is bound by instruction issue, so the common case carries no
//    per-tile bookkeeping: a warp whose (page, kv-head) chunk indices are all
//    valid and held in shared memory runs its whole tiles in turns of the
//    ring with constant stage offsets and no checks; the last tiles, the one
//    holding the new token and any warp with a bad page take a checked step.
//  * Scores: S = K~ q' on the tensor cores (mma.m16n8k16, binary16 in,
//    binary32 accumulate), 16 tokens on M, q-heads on N, the head dimension
//    on K.  K~ are the raw codes, masked in place into binary16 subnormals
//    (n * 2^-24 or n * 2^-20, exact); q' carries the matching power of two.
//    The per-token scale and zero are applied afterwards:
//    t = s*(K~.q') + z*sum(q').  MMA row j of a tile is token tok_of_row(j),
//    a permutation that keeps the K-row and V-row reads conflict-free.
//  * Output: O'^T += V~^T (p*s) on the tensor cores, dims on M, tokens on K,
//    heads on N, plus sum_j p_j z_j on the CUDA cores.  p*s goes from the
//    score fragment to the B-operand layout by two movmatrix transposes, and
//    V~^T from the V rows (read like the K rows) by movmatrix transposes of
//    their 8 x 8 blocks of code-byte pairs, masked like K.
//  * Online softmax in base 2 per head; sm_scale*log2(e) scales the binary32
//    score after the MMA, so an unrotated q enters the MMA exactly; the
//    accumulators are rescaled only when a running max grows (the lanes
//    compare their own scores first; the warp reduces only then).
//  * Splits write (m, l, numerator) partials and take a ticket; the last
//    split of a (sequence, kv-head) to finish merges them, normalizes and
//    applies the inverse rotation to V's output.  With one split the CTA
//    finishes the row itself.  No CTA waits for another.
#include <type_traits>

#include "saw_device.cuh"
#include "saw_int4.h"
#include "saw_quant_row.cuh"

namespace saw {
namespace {

#ifndef SAW_DECODE_WARPS
#define SAW_DECODE_WARPS 16
#endif
constexpr int kWarps = SAW_DECODE_WARPS;              // this object's CTA shape
constexpr int kCtasPerSm = 16 / kWarps;               // 128 registers per thread either way
static_assert(kWarps == 16 || kWarps == 8 || kWarps == 4, "decode CTAs have 16, 8 or 4 warps");
constexpr int kThreads = kWarps * 32;
constexpr uint32_t kFull = 0xFFFFFFFFu;
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// Transpose of an 8 x 8 matrix of 16-bit elements held as MMA fragments
// (lane 4r + q holds row r, columns 2q, 2q + 1).
__device__ __forceinline__ uint32_t movm_t(uint32_t a) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
// Token of MMA row j (and j + 8) of a 16-token tile: a permutation that keeps
// the K-row and V-row reads of a warp at the minimum number of shared-memory
// wavefronts for 32- and 64-byte rows.
__device__ __forceinline__ constexpr int tok_of_row(int j) { return j ^ (((j >> 1) ^ (j >> 2)) & 1); }
// Executed by a whole warp with warp-uniform operands: one elected lane
// arms the mbarrier / issues the bulk copy.
__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
  asm volatile(
      "{\n\t.reg .pred p;\n\telect.sync _|p, 0xffffffff;\n\t"
      "@p mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
      "r"(bytes)
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
// dim d of a reduction row sits at d + d / 16: the stores (lane group g
// writes dims (D/8) g + ..) and the per-dim reads are then free of bank
// conflicts
__device__ __forceinline__ int red_col(int d) { return d + (d >> 4); }
constexpr int kStepTok = 16;              // tokens per step (one MMA tile, one softmax update)

// What depends on the head dimension D (64, 128 or 256).
template <int D>
struct Dims {
  static constexpr int kCodeRow = D / 2;           // code bytes per token
  static constexpr int kStages = D == 256 ? 3 : 4;  // tiles in flight per warp
  static constexpr int kRedStride = D + D / 16;    // padded row of the cross-warp reduction
  static constexpr int kE = D / 32;                // q and output elements per lane
  static constexpr int kKWords = D / 32;           // K-row words per thread-in-group
  static constexpr int kMT = D / 16;               // 16-dim tiles of the output product
  static constexpr int kKSteps = D / 16;           // k-steps of the score product
  static constexpr bool kFragSmem = D > kHeadDim;  // q' fragments read per k-step from shared memory
  static constexpr int kIdCap = D <= kHeadDim ? 256 : 64;  // chunk indices a warp keeps in shared memory
};

// Stage layout for a 16-token step, the same for every page size:
// [K codes 16 rows | K meta 16 words | V codes 16 rows | V meta 16 words].
// A 16-token page is exactly [K chunk | V chunk]; larger pages are copied
// as 16-row slices of their code and meta regions.
//
// PAIR (D = 128 standing for two head_dim-64 kv-heads, 16-token pages; the
// code is written for D = 256 over two head_dim-128 kv-heads too, which on
// GB300 measured slower than one kv-head per CTA): each tensor's part of a
// stage is the two kv-heads' page chunks back to back, [codes 16 x D/4 B |
// meta 16 words] twice, one copy; dims 0 .. D/2-1 of the pair head are the
// first kv-head's, the rest the second's.  The lanes whose K bytes, V dims or
// head columns fall in the second half read there.
template <int D, int P, bool PAIR = false>
struct Cfg {
  using DM = Dims<D>;
  static_assert(!PAIR || ((D == 128 || D == 256) && P == kStepTok),
                "pairs are two head_dim-64 or -128 heads, page 16");
  static constexpr int kCodeRow = PAIR ? D / 4 : DM::kCodeRow;  // code bytes of one row in a chunk
  static constexpr int kStages = DM::kStages;
  static constexpr int kChunk = P * kCodeRow + 4 * P;
  static constexpr int kStepsPerPage = P / kStepTok;
  // one tensor (1088 at D 128; 1152 for a pair)
  static constexpr int kHalf = (PAIR ? 2 : 1) * (kStepTok * kCodeRow + kStepTok * 4);
  static constexpr int kStage = 2 * kHalf;
  // byte offset of K's code row / meta word `row` in a stage (of the pair's
  // kv-head `hb`); V's are at the same offsets from kHalf
  __device__ static constexpr int kcode(int row, int hb = 0) { return hb * kChunk + row * kCodeRow; }
  __device__ static constexpr int kmeta(int row, int hb = 0) {
    return hb * kChunk + kStepTok * kCodeRow + row * 4;
  }
  static constexpr int kRing = kWarps * kStages * kStage;
  // after the main loop the ring is reused: cross-warp reduction, then rows
  // red_acc [W][8][D + D/16], red_m / red_l / red_z / weights [W][8],
  // per-head totals [3][8]
  static constexpr int kRed = (kWarps * kMaxGroup * DM::kRedStride + 4 * kWarps * kMaxGroup + 3 * kMaxGroup) * 4;
  static constexpr int kOffQ = (kRed + 15) / 16 * 16;                          // f32 [8][D]
  static_assert(kOffQ + kMaxGroup * D * 4 <= kRing, "epilogue scratch must fit the ring");
  static constexpr int kOffBars = kRing;
  static constexpr int kOffOk = kOffBars + kWarps * kStages * 8;               // int [W][stages]
  static constexpr int kOffIds = kOffOk + kWarps * kStages * 4;               // int [W][kIdCap]
  static constexpr int kOffQh = kOffIds + kWarps * DM::kIdCap * 4;                // half [2][D/16 t][32 lanes][4]
  static constexpr int kOffQsum = kOffQh + 2 * kMaxGroup * D * 2;             // float [2][8]
  static constexpr int kOffFlag = kOffQsum + 2 * kMaxGroup * 4;               // int
  static constexpr int kOffNew = kOffFlag + 16;  // new token: [K, V] x (code bytes, meta)
  static constexpr int kSmem = kOffNew + 2 * (kCodeRow + 16);
  static_assert(kSmem <= (kCtasPerSm == 1 ? 227 * 1024 : kCtasPerSm == 2 ? 113 * 1024 : 56 * 1024),
                "shared memory per CTA");
};

// In-place butterfly over each h-block of nvec vectors of D floats in shared
// memory (all threads of the CTA take part).  Mathematically (H x) per block;
// the 1/sqrt(h) factor is left to the caller.
template <int D>
__device__ void smem_fwht(float* buf, int nvec, int h) {
  const int lanes = nvec * (D / 2);
  for (int len = 1; len < h; len *= 2) {
    for (int idx = threadIdx.x; idx < lanes; idx += blockDim.x) {
      const int v = idx / (D / 2);
      const int k = idx - v * (D / 2);
      // k-th index with bit `len` clear
      const int i = ((k & ~(len - 1)) << 1) | (k & (len - 1));
      float* row = buf + v * D;
      const float a = row[i], b = row[i + len];
      row[i] = a + b;
      row[i + len] = a - b;
    }
    __syncthreads();
  }
}

// Codes enter the MMAs as binary16 subnormals: a nibble n masked in place at
// bits 0-3 of a half is n * 2^-24, at bits 4-7 it is n * 2^-20 -- exact, with
// no offset to remove.  The other operand carries the matching power of two.
constexpr uint32_t kLoNib = 0x000F000Fu;  // bits 0-3 of both halves
constexpr uint32_t kHiNib = 0x00F000F0u;  // bits 4-7 of both halves

// PACKED (group <= 4): the score MMA's 8 columns carry q' of the (up to) 4
// heads as (hi, lo) pairs, head h in columns 2h, 2h + 1, so thread-in-group c
// holds both parts of head c and adds them in place: one head per lane.  In
// the output product head h is column 2h (columns 2h + 1 are zero).  WIDE
// (group 5..8): all 8 columns are heads, two per lane; the score product
// runs twice (q' hi, then lo).
// BFM: the caches' (scale, zero) words are bfloat16 instead of binary16;
// they are widened to binary32 either way, so only that step differs.
// D: the head dimension.  A thread-in-group c of an MMA quad covers dims
// [c D/4, (c+1) D/4) of a K row (and reads the same bytes of a V row), 32-bit
// word w of it dims 8w .. 8w+7 of that range; output tile k row g holds dim
// vdim(g, k) (below).
// PAIR: D stands for two neighbouring kv-heads of head_dim D/2 and GQA 4
// (Cfg above): q-head column v < 4 is a q-head of the first kv-head, its q
// zero in the second half of the D dims, v >= 4 one of the second, zero in
// the first half; each column's output is its own half.  The tensor cores do the
// zero products; every per-tile cost is shared by the two kv-heads.
template <int D, int P, bool PACKED, bool APPEND, bool BFM, bool PAIR = false>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) paged_decode_kernel(const DecodeParams p) {
  static_assert(!APPEND || D == kHeadDim, "the fused step is built for head_dim 128");
  static_assert(!PAIR || (!PACKED && !APPEND), "pairs use the wide form, without the fused step");
  using C = Cfg<D, P, PAIR>;
  using DM = Dims<D>;
  constexpr int kStages = DM::kStages;
  constexpr int kCodeRow = DM::kCodeRow;
  constexpr int kRedStride = DM::kRedStride;
  // Wait for the previous kernel in the stream before reading anything --
  // unless the caller declared that it writes neither the tables nor the
  // pages: then the page copies start first and the wait comes just before q
  // and the new token are read (and before anything is written).
  const bool early = p.early_pages != 0;
  if (!early) pdl_wait_then_release();
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBars);
  int32_t* stage_ok = reinterpret_cast<int32_t*>(smem + C::kOffOk);
  float* qs = reinterpret_cast<float*>(smem + C::kOffQ);
  __half* qh = reinterpret_cast<__half*>(smem + C::kOffQh);
  float* qsum = reinterpret_cast<float*>(smem + C::kOffQsum);
  int* flag = reinterpret_cast<int*>(smem + C::kOffFlag);

  const int split = blockIdx.x;
  const int kvh = blockIdx.y;
  const int seq = blockIdx.z;
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int g = lane >> 2;  // MMA group id
  const int c = lane & 3;   // thread in group
  const int sg = tok_of_row(g);  // the token (and sg + 8) of this lane's score rows g, g + 8
  const int hkc = PAIR ? c >> 1 : 0;  // a pair's kv-head of this lane's head columns
  const int G = PAIR ? kMaxGroup : p.group;  // q-head columns of this CTA
  const int hq0 = kvh * G;
  constexpr int kOutD = PAIR ? D / 2 : D;     // dims of an output row
  const int kv0 = PAIR ? 2 * kvh : kvh;       // (first) kv-head of this CTA

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
    // nothing to attend over here; an empty sequence still owes a zero row
    if (split == 0 && n_pages == 0) {
      if (early) pdl_wait_then_release();
      for (int idx = tid; idx < G * kOutD; idx += kThreads)
        p.out[(int64_t(seq) * p.num_q_heads + hq0) * kOutD + idx] = 0.0f;
    }
    return;
  }

  // ---- this warp's steps: step j covers tokens [p_begin*P + 16j, +16);
  // warp w takes steps w, w+W, ...
  const int n_steps = (p_end - p_begin) * C::kStepsPerPage;
  const int n_my = (warp < n_steps) ? (n_steps - warp + kWarps - 1) / kWarps : 0;
  // this warp's leading steps whose 16 tokens all lie before L
  const int full_steps = min(n_steps, (L - p_begin * P) / kStepTok);
  const int n_full = (warp < full_steps) ? (full_steps - warp + kWarps - 1) / kWarps : 0;
  uint8_t* ring = smem + warp * kStages * C::kStage;
  uint64_t* wbars = bars + warp * kStages;
  int32_t* wok = stage_ok + warp * kStages;
  const int32_t* btab = p.block_tables + int64_t(seq) * p.max_blocks;

  // the (page, kv-head) chunk index of this warp's step i (-1: invalid page)
  auto chunk_id = [&](int i) {
    const int lp = p_begin + (warp + i * kWarps) / C::kStepsPerPage;
    const int id = btab[lp];
    if (id < 0 || id >= p.num_pages) {
      report(p.dev_status, SAW_ERR_DEVICE_INDEX);
      return -1;
    }
    return id * p.num_kv_heads + kv0;
  };
  // the warp's chunk indices, fetched once instead of one dependent global
  // load in front of every copy
  constexpr int kIdCap = DM::kIdCap;
  int32_t* wids = reinterpret_cast<int32_t*>(smem + C::kOffIds) + warp * kIdCap;
  bool bad = false;
  for (int e = lane; e < n_my && e < kIdCap; e += 32) {
    const int ci = chunk_id(e);
    wids[e] = ci;
    bad = bad || ci < 0;
  }
  // clean: every chunk index of this warp is in the list and valid, so a
  // copy needs no checks and every stage holds its page
  const bool clean = !__any_sync(kFull, bad) && n_my <= kIdCap;
  __syncwarp();

  // With an even ring, stages 2b and 2b + 1 complete on one barrier: a
  // warp's tiles are consumed and refilled two at a time, so one wait and
  // one arrival serve both.
  constexpr bool kPairBars = kStages % 2 == 0;
  auto bar_of = [&](int s) { return kPairBars ? &wbars[s >> 1] : &wbars[s]; };
  // lane 0 only: tiles i .. i + n - 1 (n = 2 only with paired barriers) into
  // stages s = i % kStages, s + 1.  CHECKED: an index may be missing from the
  // list or invalid (a skipped page: the stage is marked and not filled).
  auto issue = [&](auto checked, int i, int s, int n) {
    int ci[2] = {-1, -1};
    int valid = 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u < n) {
        if constexpr (decltype(checked)::value) {
          ci[u] = (i + u < kIdCap) ? wids[i + u] : chunk_id(i + u);
          wok[s + u] = (ci[u] >= 0);
        } else {
          ci[u] = wids[i + u];
        }
        valid += ci[u] >= 0;
      }
    }
    uint64_t* bar = bar_of(s);
    if (valid == 0) {
      mbar_arrive(bar);
      return;
    }
    mbar_arrive_expect_tx(bar, valid * C::kStage);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u < n && ci[u] >= 0) {
        uint8_t* st = ring + (s + u) * C::kStage;
        const int64_t off = int64_t(ci[u]) * C::kChunk;
        if (P == 16) {  // the page's chunk (a pair: both kv-heads' chunks), K then V
          bulk_g2s(st, p.k_cache + off, C::kHalf, bar);
          bulk_g2s(st + C::kHalf, p.v_cache + off, C::kHalf, bar);
        } else {
          const int part = (warp + (i + u) * kWarps) % C::kStepsPerPage;
          const int64_t codes = off + part * (kStepTok * kCodeRow);
          const int64_t meta = off + P * kCodeRow + part * (kStepTok * 4);
          bulk_g2s(st, p.k_cache + codes, kStepTok * kCodeRow, bar);
          bulk_g2s(st + kStepTok * kCodeRow, p.k_cache + meta, kStepTok * 4, bar);
          bulk_g2s(st + C::kHalf, p.v_cache + codes, kStepTok * kCodeRow, bar);
          bulk_g2s(st + C::kHalf + kStepTok * kCodeRow, p.v_cache + meta, kStepTok * 4, bar);
        }
      }
    }
  };

  // the whole warp, clean lists only: tiles i .. i + n - 1 into stages s ..
  // (the values are the same in every lane, so no lane-0 branch is needed;
  // one elected lane arms the barrier and issues the copies)
  auto issue_w = [&](int i, int s, int n) {
    const uint32_t bar = smem_u32(bar_of(s));
    mbar_arrive_expect_tx_elect(bar, n * C::kStage);
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (u < n) {
        const int ci = __shfl_sync(kFull, wids[i + u], 0);
        const uint32_t st = smem_u32(ring + (s + u) * C::kStage);
        const int64_t off = int64_t(ci) * C::kChunk;
        if (P == 16) {
          bulk_g2s_elect(st, p.k_cache + off, C::kHalf, bar);
          bulk_g2s_elect(st + C::kHalf, p.v_cache + off, C::kHalf, bar);
        } else {
          const int part = (warp + (i + u) * kWarps) % C::kStepsPerPage;
          const int64_t codes = off + part * (kStepTok * kCodeRow);
          const int64_t meta = off + P * kCodeRow + part * (kStepTok * 4);
          bulk_g2s_elect(st, p.k_cache + codes, kStepTok * kCodeRow, bar);
          bulk_g2s_elect(st + kStepTok * kCodeRow, p.k_cache + meta, kStepTok * 4, bar);
          bulk_g2s_elect(st + C::kHalf, p.v_cache + codes, kStepTok * kCodeRow, bar);
          bulk_g2s_elect(st + C::kHalf + kStepTok * kCodeRow, p.v_cache + meta, kStepTok * 4, bar);
        }
      }
    }
  };

  if (lane == 0) {
    for (int i = 0; i < (kPairBars ? kStages / 2 : kStages); ++i) mbar_init(&wbars[i], 1);
    mbar_fence_init();
    if constexpr (kPairBars) {
      for (int i = 0; i < kStages && i < n_my; i += 2) issue(std::true_type{}, i, i, min(2, n_my - i));
    } else {
      for (int i = 0; i < kStages && i < n_my; ++i) issue(std::true_type{}, i, i, 1);
    }
  }
  // decode step: the page that receives the new token (position L-1)
  const int new_tok = L - 1;
  const bool owner = APPEND && new_tok >= 0 && new_tok / P >= p_begin && new_tok / P < p_end;
  const int new_pid = owner ? btab[new_tok / P] : -1;
  if (early && lane < D / 64) {
    // warm L2 with the rows read right after the wait (a prefetch only
    // hints the cache, which stays coherent with the previous kernel's
    // writes, so it may run before the wait)
    const uint16_t* row = nullptr;
    if (warp < G) row = p.q + (int64_t(seq) * p.num_q_heads + hq0 + warp) * kOutD;
    if (owner && warp == kWarps - 2) row = p.k_new + int64_t(seq) * p.k_new_stride + int64_t(kvh) * D;
    if (owner && warp == kWarps - 1) row = p.v_new + int64_t(seq) * p.v_new_stride + int64_t(kvh) * D;
    if (row) asm volatile("prefetch.global.L2 [%0];" ::"l"(row + lane * 64));
  }
  __syncwarp();
  if (early) pdl_wait_then_release();

  // ---- decode step: the CTA whose split holds the new token quantizes its
  // K and V rows for this kv-head (the same warp quantizer as the append
  // kernels, so the bytes match), writes them into the cache, and keeps them
  // to patch its own copy of that page below.
  uint8_t* newrow = smem + C::kOffNew;
  if (owner && warp >= kWarps - 2) {
    const int tensor = warp - (kWarps - 2);
    const uint16_t* src = (tensor == 0 ? p.k_new + int64_t(seq) * p.k_new_stride
                                       : p.v_new + int64_t(seq) * p.v_new_stride) +
                          int64_t(kvh) * D;
    const bool rot = (tensor == 0 ? p.rotate_k : p.rotate_v) != 0;
    uint32_t meta;
    const uint16_t codes =
        warp_quantize_row(src, rot, p.block_h, p.c_h, lane, &meta, p.in_f16 != 0, BFM);
    uint8_t* nr = newrow + tensor * (kCodeRow + 16);
    reinterpret_cast<uint16_t*>(nr)[lane] = codes;
    if (lane == 0) *reinterpret_cast<uint32_t*>(nr + kCodeRow) = meta;
    if (new_pid >= 0 && new_pid < p.num_pages) {
      const int off = new_tok % P;
      uint8_t* chunk = (tensor == 0 ? p.k_cache_w : p.v_cache_w) +
                       (int64_t(new_pid) * p.num_kv_heads + kvh) * C::kChunk;
      reinterpret_cast<uint16_t*>(chunk + off * kCodeRow)[lane] = codes;
      if (lane == 0) *reinterpret_cast<uint32_t*>(chunk + P * kCodeRow + 4 * off) = meta;
    }
  }
  // the step (and its row) that holds the new token, for the patch
  const int new_local = new_tok - p_begin * P;
  const int new_step = owner ? new_local / kStepTok : -1;
  // this warp's tile index of that step (-1: another warp's, or none)
  const int new_i = (new_step >= warp && (new_step - warp) % kWarps == 0) ? (new_step - warp) / kWarps : -1;

  // ---- b = 2^S q', q' = (1/sqrt h) H q for the group's heads, as binary16
  // hi + lo parts (b = hi + lo to ~22 bits; zeros beyond G).  Warp h < 8
  // rotates head h, lane l holding elements E l .. E l + E - 1 (E = D/32).
  // S is per head, the largest with |b| < 2^14, and odd elements get
  // 2^(S-4): they meet the high nibbles (n * 2^-20) and even ones the low
  // nibbles (n * 2^-24), so every product is n q' 2^(S-24).
  // sm_scale*log2(e) is applied to the binary32 score, so an unrotated q
  // enters the MMA exactly.
  // q' is stored in the B-fragment order of the score MMA: buffer 0 holds,
  // for k-step t and lane (g, c), the four binary16 values of that lane's
  // two fragment registers (PACKED: column g = hi of head g / 2 for even g,
  // lo for odd g; WIDE: hi of head g); buffer 1 (WIDE) the lo parts.
  // Element d of a head, with c = d / (D/4), o = d mod (D/4) and j = o mod 8,
  // sits at k-step 2 (o / 8) + ((j >> 1) & 1), thread-in-group c, register
  // j & 1, half (j >> 2) & 1: the nibble the K codes put there.
  constexpr int kE = DM::kE;
  for (int h = warp; h < kMaxGroup; h += kWarps) {  // (4-warp CTAs: two heads per warp)
    float x[kE];
#pragma unroll
    for (int e = 0; e < kE; ++e) x[e] = 0.0f;
    if (h < G) {
      // PAIR: column h's q fills its kv-head's half (lanes 16 (h / 4) ..),
      // the other half stays zero
      if (!PAIR || (lane >> 4) == (h >> 2)) {
        const uint16_t* qrow = p.q + (int64_t(seq) * p.num_q_heads + hq0 + h) * kOutD +
                               kE * (PAIR ? (lane & 15) : lane);
        const bool f16 = p.in_f16 != 0;
        uint32_t raw[kE / 2];
        if (kE == 2) {
          raw[0] = *reinterpret_cast<const uint32_t*>(qrow);
        } else {
#pragma unroll
          for (int u = 0; u < kE / 2; u += 2) {
            const uint2 r2 = *reinterpret_cast<const uint2*>(qrow + 2 * u);
            raw[u] = r2.x;
            raw[u + 1] = r2.y;
          }
        }
#pragma unroll
        for (int u = 0; u < kE / 2; ++u) {
          x[2 * u] = in_lo(raw[u], f16);
          x[2 * u + 1] = in_hi(raw[u], f16);
        }
      }
      if (p.rotate_k) {
        const int hb = p.block_h;
        // strides below E inside the lane, ascending, then across lanes
#pragma unroll
        for (int len = 1; len < kE; len *= 2) {
          if (len < hb) {
#pragma unroll
            for (int e = 0; e < kE; ++e) {
              if (!(e & len)) {
                const float a = x[e], b = x[e + len];
                x[e] = a + b;
                x[e + len] = a - b;
              }
            }
          }
        }
        for (int len = kE; len < hb; len *= 2) {
          const int mask = len / kE;
          const bool upper = (lane & mask) != 0;
#pragma unroll
          for (int e = 0; e < kE; ++e) {
            const float o = __shfl_xor_sync(kFull, x[e], mask);
            x[e] = upper ? (o - x[e]) : (x[e] + o);
          }
        }
#pragma unroll
        for (int e = 0; e < kE; ++e) x[e] *= p.c_h;
      }
    }
    float amax = 0.0f;
#pragma unroll
    for (int e = 0; e < kE; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int x2 = 16; x2 >= 1; x2 >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, x2));
    int ex;
    frexpf(amax, &ex);                       // amax < 2^ex (ex = 0 for amax = 0)
    const int S = min(max(14 - ex, -100), 100);
    float part = 0.0f;
#pragma unroll
    for (int e = 0; e < kE; ++e) {
      const int d = kE * lane + e;
      const int se = (d & 1) ? S - 4 : S;
      const float y = ldexpf(x[e], se);
      const __half hi = __float2half_rn(y);
      const __half lo = __float2half_rn(y - __half2float(hi));
      const int c_ = d / (D / 4);
      const int o = d % (D / 4);
      const int jj = o & 7;
      const int t = 2 * (o >> 3) + ((jj >> 1) & 1);
      const int w2 = (jj & 1) * 2 + ((jj >> 2) & 1);
      constexpr int kLo = DM::kKSteps * 32 * 4;  // halves in buffer 0
      if (PACKED) {
        if (h < kMaxGroup / 2) {
          qh[(t * 32 + 2 * h * 4 + c_) * 4 + w2] = hi;
          qh[(t * 32 + (2 * h + 1) * 4 + c_) * 4 + w2] = lo;
        }
      } else {
        qh[(t * 32 + h * 4 + c_) * 4 + w2] = hi;
        qh[kLo + (t * 32 + h * 4 + c_) * 4 + w2] = lo;
      }
      part += ldexpf(__half2float(hi) + __half2float(lo), -se);
    }
#pragma unroll
    for (int x2 = 16; x2 >= 1; x2 >>= 1) part += __shfl_xor_sync(kFull, part, x2);
    if (lane == 0) {
      qsum[h] = part;
      qsum[kMaxGroup + h] = ldexpf(1.0f, 24 - S);
    }
  }
  __syncthreads();

  // B fragments of q' for the score MMA (k-step t uses word t/2 of the
  // thread-in-group's share of a token's codes: bytes (0,2) for even t,
  // (1,3) for odd t).  Column g: PACKED -> hi (even g) or lo (odd g) of
  // head g / 2; WIDE -> head g.  Kept in registers up to D = 128; read from
  // shared memory per k-step beyond (the output accumulators take the room).
  constexpr int kKS = DM::kKSteps;
  constexpr int kRegKS = DM::kFragSmem ? 1 : kKS;
  const uint2* qf = reinterpret_cast<const uint2*>(qh);
  uint32_t bq[kRegKS][2];
  uint32_t bl[(PACKED || DM::kFragSmem) ? 1 : kKS][2];
  if constexpr (!DM::kFragSmem) {
#pragma unroll
    for (int t = 0; t < kRegKS; ++t) {
      const uint2 v = qf[t * 32 + lane];
      bq[t][0] = v.x;
      bq[t][1] = v.y;
      if (!PACKED) {
        const uint2 u = qf[kKS * 32 + t * 32 + lane];
        bl[PACKED ? 0 : t][0] = u.x;
        bl[PACKED ? 0 : t][1] = u.y;
      }
    }
  }
  // this thread's heads (PACKED: head c, as A; WIDE: heads 2c, 2c + 1): the
  // MMA gives acc = 2^(S-24) (n . q'), so the base-2 logit
  // t = sm'*(s (n.q') + z sum(q')) = (sm' 2^(24-S) s) acc + (sm' sum(q')) z.
  const int hb = PACKED ? c : 2 * c;
  const float qsA = qsum[hb] * p.q_scale, qsB = qsum[hb + 1] * p.q_scale;
  const float skA = qsum[kMaxGroup + hb] * p.q_scale, skB = qsum[kMaxGroup + hb + 1] * p.q_scale;
  const float2 skAB = make_float2(skA, skB), qsAB = make_float2(qsA, qsB);

  constexpr int kMT = DM::kMT;
  // output tile k = 2 db + hh: row g is dim vdim(g, k) (low nibbles), row
  // g + 8 the next dim (high nibbles): byte hh of byte pair g of block db
  auto vdim = [](int gg, int k) { return (gg >> 1) * (D / 4) + 8 * (k >> 1) + 4 * (gg & 1) + 2 * (k & 1); };
  float acc[kMT][4];
#pragma unroll
  for (int i = 0; i < kMT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_run[2] = {0.0f, 0.0f};
  float z_run[2] = {0.0f, 0.0f};
  float2 nmu = make_float2(-0.0f, -0.0f);  // minus the running maxes (0 while they are -inf)
  bool failed = false;
  int waited = 0;  // first of this warp's tiles not yet consumed

  // One step consumes NT consecutive tiles of this warp (i, i+1, ...): the
  // tiles' score products and PV products are independent, and they share
  // one max reduction and one rescale of the online softmax.
  // S0 >= 0: i % kStages == S0, known here, so the stage offsets are
  // constants; and the warp is clean and the tiles are whole and do not hold
  // the new token, so no tile needs a check.
  auto step = [&](auto ntc, auto s0c, int i) -> bool {
    constexpr int NT = decltype(ntc)::value;
    constexpr int S0 = decltype(s0c)::value;
    constexpr bool kChecks = S0 < 0;
    auto stage = [&](int t) { return S0 >= 0 ? (S0 + t) % kStages : (i + t) % kStages; };
    waited = i;
    bool ok = true;
    if constexpr (kPairBars) {
      ok = mbar_wait_bounded(bar_of(stage(0)), (i / kStages) & 1);  // i is even
    } else {
#pragma unroll
      for (int t = 0; t < NT; ++t)
        ok = mbar_wait_bounded(bar_of(stage(t)), ((i + t) / kStages) & 1) && ok;
    }
    if (!__all_sync(kFull, ok)) return false;
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      if (APPEND && kChecks && i + t == new_i) {
        // replace the copied row of the new token by its freshly quantized one
        const int row = new_local % kStepTok;
        uint8_t* w = ring + stage(t) * C::kStage;
        if (lane < 16) {
          const int tensor = lane >> 3, part = lane & 7;  // 8 x 8 bytes per tensor
          const uint8_t* nr = newrow + tensor * (kCodeRow + 16);
          uint8_t* dst = w + (tensor ? C::kHalf : 0) + C::kcode(row);
          reinterpret_cast<uint2*>(dst)[part] = reinterpret_cast<const uint2*>(nr)[part];
        } else if (lane < 18) {
          const int tensor = lane - 16;
          const uint8_t* nr = newrow + tensor * (kCodeRow + 16);
          *reinterpret_cast<uint32_t*>(w + (tensor ? C::kHalf : 0) + C::kmeta(row)) =
              *reinterpret_cast<const uint32_t*>(nr + kCodeRow);
        }
        __syncwarp();
      }
    }

    // ---- scores of the NT x 16 tokens
    float sc[NT][4];
    bool full[NT];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const int s_ = stage(t);
      const uint8_t* st = ring + s_ * C::kStage;
      full[t] = !kChecks || ((i + t < n_full) && (clean || wok[s_] != 0));  // warp-uniform
      constexpr int kKW = DM::kKWords;
      // (a pair: thread-in-group c reads half c & 1 of kv-head c / 2's row)
      const uint8_t* krow = PAIR ? st + C::kcode(sg, c >> 1) + (D / 8) * (c & 1)
                                 : st + C::kcode(sg) + (D / 8) * c;
      uint32_t kaw[kKW], kbw[kKW];
      if constexpr (kKW == 2) {
        const uint2 ka = *reinterpret_cast<const uint2*>(krow);
        const uint2 kb = *reinterpret_cast<const uint2*>(krow + 8 * C::kCodeRow);
        kaw[0] = ka.x; kaw[1] = ka.y;
        kbw[0] = kb.x; kbw[1] = kb.y;
      } else {
#pragma unroll
        for (int u = 0; u < kKW; u += 4) {
          const uint4 ka = *reinterpret_cast<const uint4*>(krow + 4 * u);
          const uint4 kb = *reinterpret_cast<const uint4*>(krow + 8 * C::kCodeRow + 4 * u);
          kaw[u] = ka.x; kaw[u + 1] = ka.y; kaw[u + 2] = ka.z; kaw[u + 3] = ka.w;
          kbw[u] = kb.x; kbw[u + 1] = kb.y; kbw[u + 2] = kb.z; kbw[u + 3] = kb.w;
        }
      }
      // two independent accumulator chains (even / odd byte pairs)
      float d[4] = {0.0f, 0.0f, 0.0f, 0.0f};
      float e2[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll
      for (int w = 0; w < kKW; ++w) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          // bytes (0,2) in place, bytes (1,3) moved down by 8: low nibbles
          // for columns 2c, 2c+1, high nibbles for 2c+8, 2c+9
          const uint32_t wa = hh ? (kaw[w] >> 8) : kaw[w];
          const uint32_t wb = hh ? (kbw[w] >> 8) : kbw[w];
          uint32_t a[4];
          a[0] = wa & kLoNib;
          a[1] = wb & kLoNib;
          a[2] = wa & kHiNib;
          a[3] = wb & kHiNib;
          float (&dst)[4] = hh ? e2 : d;
          const int kt = 2 * w + hh;
          if constexpr (DM::kFragSmem) {
            const uint2 v = qf[kt * 32 + lane];
            mma_16816(dst, a, v.x, v.y);
            if (!PACKED) {
              const uint2 u = qf[kKS * 32 + kt * 32 + lane];
              mma_16816(dst, a, u.x, u.y);
            }
          } else {
            mma_16816(dst, a, bq[kt][0], bq[kt][1]);
            if (!PACKED) mma_16816(dst, a, bl[PACKED ? 0 : kt][0], bl[PACKED ? 0 : kt][1]);
          }
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) d[j] += e2[j];
      // the (scale, zero) words of this lane's rows (a pair: of kv-head c / 2)
      const uint32_t mk0 = *reinterpret_cast<const uint32_t*>(st + C::kmeta(sg, hkc));
      const uint32_t mk1 = *reinterpret_cast<const uint32_t*>(st + C::kmeta(sg + 8, hkc));
      const float s0 = meta_lo(mk0, BFM), z0 = meta_hi(mk0, BFM);
      const float s1 = meta_lo(mk1, BFM), z1 = meta_hi(mk1, BFM);
      if constexpr (PACKED) {
        // head c of rows g and g + 8: hi part (column 2c) + lo part (2c+1)
        const float2 hl = add2(make_float2(d[0], d[2]), make_float2(d[1], d[3]));
        const float2 r = fma2(mul2(make_float2(s0, s1), make_float2(skA, skA)), hl,
                              mul2(make_float2(z0, z1), make_float2(qsA, qsA)));
        sc[t][0] = r.x;
        sc[t][2] = r.y;
        sc[t][1] = sc[t][3] = 0.0f;
      } else {
        // heads (A, B) of rows g and g + 8, two per instruction
        const float2 r0 = fma2(mul2(make_float2(s0, s0), skAB), make_float2(d[0], d[1]),
                               mul2(make_float2(z0, z0), qsAB));
        const float2 r1 = fma2(mul2(make_float2(s1, s1), skAB), make_float2(d[2], d[3]),
                               mul2(make_float2(z1, z1), qsAB));
        sc[t][0] = r0.x;
        sc[t][1] = r0.y;
        sc[t][2] = r1.x;
        sc[t][3] = r1.y;
      }
      if (!full[t]) {  // the tile holding the end of the sequence, or a bad page
        const int tok0 = p_begin * P + (warp + (i + t) * kWarps) * kStepTok;
        const bool pok = clean || wok[s_] != 0;
        const bool v0 = pok && (tok0 + sg) < L;
        const bool v1 = pok && (tok0 + sg + 8) < L;
        sc[t][0] = v0 ? sc[t][0] : -INFINITY;
        sc[t][1] = v0 ? sc[t][1] : -INFINITY;
        sc[t][2] = v1 ? sc[t][2] : -INFINITY;
        sc[t][3] = v1 ? sc[t][3] : -INFINITY;
      }
    }

    // ---- online softmax: rescale only when a running max grows.  A head's
    // max over the warp exceeds its running max exactly when one lane's
    // does, so the lanes compare first and reduce only when one grew.
    float mloc0, mloc1;
    if (NT == 2) {
      mloc0 = fmaxf(fmax3(sc[0][0], sc[0][2], sc[1][0]), sc[1][2]);
      mloc1 = PACKED ? -INFINITY : fmaxf(fmax3(sc[0][1], sc[0][3], sc[1][1]), sc[1][3]);
    } else {
      mloc0 = fmaxf(sc[0][0], sc[0][2]);
      mloc1 = PACKED ? -INFINITY : fmaxf(sc[0][1], sc[0][3]);
    }
    if (PACKED ? __any_sync(kFull, mloc0 > m_run[0])
               : __any_sync(kFull, (mloc0 > m_run[0]) || (mloc1 > m_run[1]))) {
      if constexpr (PACKED) {
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) mloc0 = fmaxf(mloc0, __shfl_xor_sync(kFull, mloc0, x));
        const float mn0 = fmaxf(m_run[0], mloc0);
        const float mu0 = (mn0 == -INFINITY) ? 0.0f : mn0;
        const float al0 = ex2(m_run[0] - mu0);
        m_run[0] = mn0;
        l_run[0] *= al0;
        z_run[0] *= al0;
#pragma unroll
        for (int k = 0; k < kMT; ++k) {  // columns 2c + 1 stay zero
          acc[k][0] *= al0;
          acc[k][2] *= al0;
        }
        nmu.x = -mu0;
      } else {
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
          mloc0 = fmaxf(mloc0, __shfl_xor_sync(kFull, mloc0, x));
          mloc1 = fmaxf(mloc1, __shfl_xor_sync(kFull, mloc1, x));
        }
        const float mn0 = fmaxf(m_run[0], mloc0), mn1 = fmaxf(m_run[1], mloc1);
        const float al0 = ex2(m_run[0] - ((mn0 == -INFINITY) ? 0.0f : mn0));
        const float al1 = ex2(m_run[1] - ((mn1 == -INFINITY) ? 0.0f : mn1));
        m_run[0] = mn0;
        m_run[1] = mn1;
        const float2 al = make_float2(al0, al1);  // columns 0, 2 are head A, 1, 3 head B
        const float2 lz = mul2(make_float2(l_run[0], l_run[1]), al);
        const float2 zz = mul2(make_float2(z_run[0], z_run[1]), al);
        l_run[0] = lz.x;
        l_run[1] = lz.y;
        z_run[0] = zz.x;
        z_run[1] = zz.y;
#pragma unroll
        for (int k = 0; k < kMT; ++k) {
          const float2 a01 = mul2(make_float2(acc[k][0], acc[k][1]), al);
          const float2 a23 = mul2(make_float2(acc[k][2], acc[k][3]), al);
          acc[k][0] = a01.x;
          acc[k][1] = a01.y;
          acc[k][2] = a23.x;
          acc[k][3] = a23.y;
        }
        // x - mu = x + (-mu), exactly
        nmu = make_float2(-((mn0 == -INFINITY) ? 0.0f : mn0), -((mn1 == -INFINITY) ? 0.0f : mn1));
      }
    }

    // ---- probabilities, V terms, and the PV products
#pragma unroll
    for (int t = 0; t < NT; ++t) {
      const uint8_t* vst = ring + stage(t) * C::kStage + C::kHalf;
      float2 p01, p23;  // PACKED: p01 = (row g, row g + 8) of head c
      if constexpr (PACKED) {
        const float2 x = add2(make_float2(sc[t][0], sc[t][2]), make_float2(nmu.x, nmu.x));
        p01 = make_float2(ex2(x.x), ex2(x.y));
        p23 = p01;
      } else {
        const float2 x01 = add2(make_float2(sc[t][0], sc[t][1]), nmu);
        const float2 x23 = add2(make_float2(sc[t][2], sc[t][3]), nmu);
        p01 = make_float2(ex2(x01.x), ex2(x01.y));
        p23 = make_float2(ex2(x23.x), ex2(x23.y));
      }
      const uint32_t mv0 = *reinterpret_cast<const uint32_t*>(vst + C::kmeta(sg, hkc));
      const uint32_t mv1 = *reinterpret_cast<const uint32_t*>(vst + C::kmeta(sg + 8, hkc));
      float sv0 = meta_lo(mv0, BFM), zv0 = meta_hi(mv0, BFM);
      float sv1 = meta_lo(mv1, BFM), zv1 = meta_hi(mv1, BFM);
      if (!full[t]) {  // rows past the end may hold anything, even inf
        // (a valid row's score is never -inf: only the masking above sets it)
        const bool v0 = sc[t][0] != -INFINITY, v1 = sc[t][2] != -INFINITY;
        sv0 = v0 ? sv0 : 0.0f;
        zv0 = v0 ? zv0 : 0.0f;
        sv1 = v1 ? sv1 : 0.0f;
        zv1 = v1 ? zv1 : 0.0f;
      }
      uint32_t b0, b1;
      if constexpr (PACKED) {
        l_run[0] = l_run[0] + (p01.x + p01.y);
        z_run[0] = z_run[0] + fmaf(p01.y, zv1, p01.x * zv0);
        const float2 ps = mul2(p01, make_float2(sv0, sv1));
        // the two 8 x 8 blocks (score rows 0-7 and 8-15 by columns 2c: head
        // c; columns 2c + 1 zero), transposed: B column 2h carries head h
        b0 = movm_t(pack_half2(ps.x, 0.0f));
        b1 = movm_t(pack_half2(ps.y, 0.0f));
      } else {
        const float2 l2 = add2(make_float2(l_run[0], l_run[1]), add2(p01, p23));
        const float2 z2 = add2(make_float2(z_run[0], z_run[1]),
                               fma2(p23, make_float2(zv1, zv1), mul2(p01, make_float2(zv0, zv0))));
        l_run[0] = l2.x;
        l_run[1] = l2.y;
        z_run[0] = z2.x;
        z_run[1] = z2.y;
        // (p*s) for this thread's columns over tokens (g, g+8) as binary16
        const float2 ps01 = mul2(p01, make_float2(sv0, sv0));
        const float2 ps23 = mul2(p23, make_float2(sv1, sv1));
        // the two 8 x 8 blocks (score rows 0-7 and 8-15 by head columns),
        // transposed, are the B fragments of the PV product: k-columns
        // 2c, 2c+1 (and 2c+8, 2c+9) carry the tokens of score rows 2c, 2c+1
        b0 = movm_t(pack_half2(ps01.x, ps01.y));
        b1 = movm_t(pack_half2(ps23.x, ps23.y));
      }

      // V^T operands: the 8 x 8 blocks of 16-bit elements (8 token rows of
      // the tile by 8 code-byte pairs) are read like the K rows and
      // transposed by movmatrix; lane (g, c) then holds byte pair g of
      // tokens 2c, 2c + 1 of the block, which is, masked, the A fragment
      // over those tokens for the dims of the pair (see vdim below).
      constexpr int kKW = DM::kKWords;
      const uint8_t* vrow = PAIR ? vst + C::kcode(sg, c >> 1) + (D / 8) * (c & 1)
                                 : vst + C::kcode(sg) + (D / 8) * c;
      uint32_t vaw[kKW], vbw[kKW];
      if constexpr (kKW == 2) {
        const uint2 va = *reinterpret_cast<const uint2*>(vrow);
        const uint2 vb = *reinterpret_cast<const uint2*>(vrow + 8 * C::kCodeRow);
        vaw[0] = va.x; vaw[1] = va.y;
        vbw[0] = vb.x; vbw[1] = vb.y;
      } else {
#pragma unroll
        for (int u = 0; u < kKW; u += 4) {
          const uint4 va = *reinterpret_cast<const uint4*>(vrow + 4 * u);
          const uint4 vb = *reinterpret_cast<const uint4*>(vrow + 8 * C::kCodeRow + 4 * u);
          vaw[u] = va.x; vaw[u + 1] = va.y; vaw[u + 2] = va.z; vaw[u + 3] = va.w;
          vbw[u] = vb.x; vbw[u + 1] = vb.y; vbw[u + 2] = vb.z; vbw[u + 3] = vb.w;
        }
      }
#pragma unroll
      for (int db = 0; db < kKW; ++db) {
        const uint32_t ta = movm_t(vaw[db]);  // tokens of score rows 0-7
        const uint32_t tb = movm_t(vbw[db]);  // rows 8-15
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const uint32_t x = hh ? (ta >> 8) : ta;
          const uint32_t y = hh ? (tb >> 8) : tb;
          uint32_t a[4];
          a[0] = x & kLoNib;  // dims of rows g: n * 2^-24
          a[1] = x & kHiNib;  // dims of rows g + 8: n * 2^-20
          a[2] = y & kLoNib;
          a[3] = y & kHiNib;
          mma_16816(acc[2 * db + hh], a, b0, b1);
        }
      }
    }

    __syncwarp();
    if (kPairBars && (!kChecks || clean)) {
      const int nxt = i + kStages;  // the tiles that refill this step's stages
      const int n = min(NT, n_my - nxt);
      if (n > 0) issue_w(nxt, stage(0), n);
    } else if (lane == 0) {
      if constexpr (kPairBars) {
        const int nxt = i + kStages;  // the tiles that refill this step's stages
        const int n = min(NT, n_my - nxt);
        if (n > 0) issue(std::true_type{}, nxt, stage(0), n);
      } else {
#pragma unroll
        for (int t = 0; t < NT; ++t) {
          if (i + t + kStages < n_my) {
            if (!kChecks || clean) {
              issue(std::false_type{}, i + t + kStages, stage(t), 1);
            } else {
              issue(std::true_type{}, i + t + kStages, stage(t), 1);
            }
          }
        }
      }
    }
    return true;
  };

  {
    using Dyn = std::integral_constant<int, -1>;
    int i = 0;
    using I0 = std::integral_constant<int, 0>;
    using I1 = std::integral_constant<int, 1>;
    using I2 = std::integral_constant<int, 2>;
    // whole turns of the ring with constant stages, up to the first tile that
    // is not whole or holds the new token: two steps of two tiles (four
    // stages), or three of one (a three-stage ring, head_dim 256, steps one
    // tile at a time: its accumulators leave no registers for a second
    // tile's operands)
    const int lim = clean ? min(n_full, new_i >= 0 ? new_i : n_my) : 0;
    if constexpr (kStages == 4) {
      for (; i + 3 < lim; i += 4) {
        if (!step(I2{}, I0{}, i) || !step(I2{}, I2{}, i + 2)) {
          failed = true;
          break;
        }
      }
    } else {
      static_assert(kStages == 3, "rings of three or four stages");
      for (; i + 2 < lim; i += 3) {
        if (!step(I1{}, I0{}, i) || !step(I1{}, I1{}, i + 1) || !step(I1{}, I2{}, i + 2)) {
          failed = true;
          break;
        }
      }
    }
    constexpr int kNT = kStages % 2 == 0 ? 2 : 1;
    for (; !failed && i + kNT - 1 < n_my; i += kNT) {
      if (!step(std::integral_constant<int, kNT>{}, Dyn{}, i)) {
        failed = true;
        break;
      }
    }
    if (kNT == 2 && !failed && i < n_my && !step(I1{}, Dyn{}, i)) failed = true;
  }

  if (failed) {
    if (lane == 0) report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
    // let this warp's copies in flight land before the CTA's memory is reused
    for (int i = waited; i < n_my && i < waited + kStages; ++i)
      (void)mbar_wait_bounded(bar_of(i % kStages), (i / kStages) & 1);
  }

  // ---- merge protocol, part 1: with several splits, count this one as
  // arrived.  From here on it finishes without waiting for anyone, which is
  // what lets the last arrival wait for the others' partials below.  The
  // returned count is needed only after the CTA's own reduction, so the
  // round trip overlaps it.
  const int ns = (n_pages + p.pages_per_split - 1) / p.pages_per_split;  // splits with pages
  uint32_t* tk = p.tickets + 2 * (int64_t(seq) * p.num_kv_heads + kvh);  // {arrived, published}
  uint32_t arrived = 0;
  if (!direct && tid == 0)
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], 1;" : "=r"(arrived) : "l"(tk) : "memory");

  // ---- cross-thread reductions of l and the z term (lanes sharing c)
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l_run[0] += __shfl_xor_sync(kFull, l_run[0], x);
    l_run[1] += __shfl_xor_sync(kFull, l_run[1], x);
    z_run[0] += __shfl_xor_sync(kFull, z_run[0], x);
    z_run[1] += __shfl_xor_sync(kFull, z_run[1], x);
  }
  // output rows g (even dims) carried n * 2^-24, rows g + 8 (odd) n * 2^-20
#pragma unroll
  for (int k = 0; k < kMT; ++k) {
    acc[k][0] *= 16777216.0f;
    acc[k][1] *= 16777216.0f;
    acc[k][2] *= 1048576.0f;
    acc[k][3] *= 1048576.0f;
  }
  __syncthreads();  // every warp is done with its ring: reuse it

  float* red_acc = reinterpret_cast<float*>(smem);                     // [W][8][D + D/16]
  float* red_m = red_acc + kWarps * kMaxGroup * kRedStride;           // [W][8]
  float* red_l = red_m + kWarps * kMaxGroup;
  float* red_z = red_l + kWarps * kMaxGroup;
  float* wgt = red_z + kWarps * kMaxGroup;                            // [16][8]
  float* tot = wgt + kWarps * kMaxGroup;                              // den, zz, M [3][8]
  if constexpr (PACKED) {  // head c: output columns 2c
    if (g == 0) {
      red_m[warp * kMaxGroup + c] = m_run[0];
      red_l[warp * kMaxGroup + c] = l_run[0];
      red_z[warp * kMaxGroup + c] = z_run[0];
    }
    float* base0 = red_acc + (warp * kMaxGroup + c) * kRedStride;
#pragma unroll
    for (int k = 0; k < kMT; ++k) {
      base0[red_col(vdim(g, k))] = acc[k][0];
      base0[red_col(vdim(g, k) + 1)] = acc[k][2];
    }
  } else {
    if (g == 0) {
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        red_m[warp * kMaxGroup + hb + hh] = m_run[hh];
        red_l[warp * kMaxGroup + hb + hh] = l_run[hh];
        red_z[warp * kMaxGroup + hb + hh] = z_run[hh];
      }
    }
    float* base0 = red_acc + (warp * kMaxGroup + hb) * kRedStride;
    float* base1 = base0 + kRedStride;
#pragma unroll
    for (int k = 0; k < kMT; ++k) {
      base0[red_col(vdim(g, k))] = acc[k][0];
      base1[red_col(vdim(g, k))] = acc[k][1];
      base0[red_col(vdim(g, k) + 1)] = acc[k][2];
      base1[red_col(vdim(g, k) + 1)] = acc[k][3];
    }
  }
  __syncthreads();

  // ---- merge the warps.  Weights 2^(m_w - M) per (head, warp): thread
  // 16h + w of warps 0-3, reduced over the 16 warps with shuffles inside
  // each half-warp; then one (head, dim) per thread.
  const int nw = min(kWarps, n_steps);  // warps that saw any step
  static_assert(kMaxGroup * kWarps % 32 == 0, "the weight step's shuffles take whole warps");
  if (tid < kMaxGroup * kWarps) {
    const int h = tid / kWarps, w = tid % kWarps;
    const bool in = h < G && w < nw;
    const float m = in ? red_m[w * kMaxGroup + h] : -INFINITY;
    float M = m;
#pragma unroll
    for (int x = 1; x < kWarps; x <<= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, x));
    const float Mu = (M == -INFINITY) ? 0.0f : M;
    const float f = in ? ex2(m - Mu) : 0.0f;
    float den = in ? red_l[w * kMaxGroup + h] * f : 0.0f;
    float zz = in ? red_z[w * kMaxGroup + h] * f : 0.0f;
#pragma unroll
    for (int x = 1; x < kWarps; x <<= 1) {
      den += __shfl_xor_sync(kFull, den, x);
      zz += __shfl_xor_sync(kFull, zz, x);
    }
    wgt[w * kMaxGroup + h] = f;
    if (w == 0) {
      tot[h] = den;
      tot[kMaxGroup + h] = zz;
      tot[2 * kMaxGroup + h] = M;
    }
  }
  __syncthreads();
  for (int idx = tid; idx < G * D; idx += kThreads) {
    const int h = idx / D, dd = idx - h * D;
    float num = tot[kMaxGroup + h];
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      if (w < nw) num += red_acc[(w * kMaxGroup + h) * kRedStride + red_col(dd)] * wgt[w * kMaxGroup + h];
    if (direct) {
      const float den = tot[h];
      qs[h * D + dd] = (den > 0.0f) ? num / den : 0.0f;
    } else {
      // publish the partial, and keep it here in case this split merges
      // (den and M stay in tot)
      qs[h * D + dd] = num;
      const int64_t row = (int64_t(seq) * p.num_q_heads + hq0 + h) * p.num_splits + split;
      p.part_o[row * D + dd] = num;
      if (dd == 0) {
        p.part_ml[2 * row] = tot[2 * kMaxGroup + h];
        p.part_ml[2 * row + 1] = tot[h];
      }
    }
  }

  if (!direct) {
    if (tid == 0) {
      // merge protocol, part 2: the split whose arrival completed the count
      // merges; every other split publishes its partial.  The count's round
      // trip has been overlapping the reduction above.
      const uint32_t done = arrived + 1u;
      if (done > uint32_t(ns)) report(p.dev_status, SAW_ERR_DEVICE_INDEX);  // not zero-filled
      *flag = (done == uint32_t(ns));
    }
    __syncthreads();
    const bool last = *flag != 0;
    if (!last) {
      // publish: release (cumulative over the barrier above) orders this
      // CTA's partials before the count the merging split waits for
      if (tid == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(tk + 1) : "memory");
      return;
    }
    // ---- the last split to arrive: wait (bounded) until every other split
    // has published, then merge all partials, its own from shared memory
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
        tk[0] = 0u;  // every split has counted and published: ready for the next call
        tk[1] = 0u;
      } else {
        report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
      }
      flag[1] = ok ? 1 : 0;  // a word of its own: flag[0] may still be read
    }
    __syncthreads();
    const bool merge_ok = flag[1] != 0;
    // item = (head, 4 dims); four threads per item share the splits.  Every
    // load is issued before any is used (one round of L2 latency).
    constexpr int kMaxSplitsPerThread = 8;
    constexpr int kItems = D / 4;  // (head, 4 dims) items per head
    for (int base = 0; base < G * kItems * 4; base += kThreads) {
      const int t = base + tid;
      const int item = t >> 2, part = t & 3;
      const bool active = item < G * kItems;
      const int h = active ? item / kItems : 0, ch = item % kItems;
      const int64_t row0 = (int64_t(seq) * p.num_q_heads + hq0 + h) * p.num_splits;
      const float2* ml = reinterpret_cast<const float2*>(p.part_ml) + row0;
      const float4* po = reinterpret_cast<const float4*>(p.part_o + row0 * D) + ch;
      const float4* own = reinterpret_cast<const float4*>(qs + h * D) + ch;
      float M = -INFINITY;
      float4 a = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
      float den = 0.0f;
      for (int sp0 = part; sp0 < ns; sp0 += 4 * kMaxSplitsPerThread) {
        float2 v[kMaxSplitsPerThread];
        float4 o[kMaxSplitsPerThread];
#pragma unroll
        for (int u = 0; u < kMaxSplitsPerThread; ++u) {
          const int sp = sp0 + 4 * u;
          const bool mine = sp == split;
          const bool in = active && sp < ns && (mine || merge_ok);
          v[u] = !in ? make_float2(-INFINITY, 0.0f)
                     : mine ? make_float2(tot[2 * kMaxGroup + h], tot[h]) : __ldcg(&ml[sp]);
          o[u] = !in ? make_float4(0.0f, 0.0f, 0.0f, 0.0f)
                     : mine ? *own : __ldcg(&po[int64_t(sp) * (D / 4)]);
        }
        float Mb = -INFINITY;
#pragma unroll
        for (int u = 0; u < kMaxSplitsPerThread; ++u) Mb = fmaxf(Mb, v[u].x);
        const float Mn = fmaxf(M, Mb);
        const float Mu = (Mn == -INFINITY) ? 0.0f : Mn;
        const float al = ex2(M - Mu);
        a.x *= al; a.y *= al; a.z *= al; a.w *= al; den *= al;
#pragma unroll
        for (int u = 0; u < kMaxSplitsPerThread; ++u) {
          const float f = ex2(v[u].x - Mu);
          den += v[u].y * f;
          a.x += o[u].x * f;
          a.y += o[u].y * f;
          a.z += o[u].z * f;
          a.w += o[u].w * f;
        }
        M = Mn;
      }
      // combine the four parts of the item
#pragma unroll
      for (int x = 1; x <= 2; x <<= 1) {
        const float Mo = __shfl_xor_sync(kFull, M, x);
        const float Mn = fmaxf(M, Mo);
        const float Mu = (Mn == -INFINITY) ? 0.0f : Mn;
        const float fs = ex2(M - Mu), fo = ex2(Mo - Mu);
        const float dn = __shfl_xor_sync(kFull, den, x);
        const float ox = __shfl_xor_sync(kFull, a.x, x), oy = __shfl_xor_sync(kFull, a.y, x);
        const float oz = __shfl_xor_sync(kFull, a.z, x), ow = __shfl_xor_sync(kFull, a.w, x);
        den = den * fs + dn * fo;
        a.x = a.x * fs + ox * fo;
        a.y = a.y * fs + oy * fo;
        a.z = a.z * fs + oz * fo;
        a.w = a.w * fs + ow * fo;
        M = Mn;
      }
      if (active && part == 0) {
        const float inv = (den > 0.0f) ? 1.0f / den : 0.0f;
        float* dst = qs + h * D + 4 * ch;
        dst[0] = a.x * inv;
        dst[1] = a.y * inv;
        dst[2] = a.z * inv;
        dst[3] = a.w * inv;
      }
    }
  }
  __syncthreads();
  if (p.rotate_v) smem_fwht<D>(qs, G, p.block_h);
  const float post = p.rotate_v ? p.c_h : 1.0f;
  // (a pair: column v's output is its own kv-head's half of the 128 dims)
  for (int idx = tid; idx < G * kOutD; idx += kThreads) {
    const int h = idx / kOutD, dd = idx - h * kOutD;
    const float o = PAIR ? qs[h * D + (h >> 2) * kOutD + dd] : qs[idx];
    p.out[(int64_t(seq) * p.num_q_heads + hq0) * kOutD + idx] = o * post;
  }
}

// Launched with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream drains; it waits for it (griddepcontrol)
// before reading anything.
template <int D, int P, bool PACKED, bool APPEND, bool BFM, bool PAIR = false>
cudaError_t launch_p(const DecodeParams& p, cudaStream_t stream) {
  using C = Cfg<D, P, PAIR>;
  auto kernel = paged_decode_kernel<D, P, PACKED, APPEND, BFM, PAIR>;
  cudaError_t err =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.num_splits, PAIR ? p.num_kv_heads / 2 : p.num_kv_heads, p.num_seqs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::kSmem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int D, int P, bool BFM>
cudaError_t launch_page_m(const DecodeParams& p, cudaStream_t stream) {
  const bool packed = p.group <= kMaxGroup / 2;
  if constexpr (D == kHeadDim) {
    if (p.append)
      return packed ? launch_p<D, P, true, true, BFM>(p, stream)
                    : launch_p<D, P, false, true, BFM>(p, stream);
  }
  return packed ? launch_p<D, P, true, false, BFM>(p, stream)
                : launch_p<D, P, false, false, BFM>(p, stream);
}

template <int D>
cudaError_t launch_dim(const DecodeParams& p, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  switch (p.page_size) {
    case 16: return p.meta_bf16 ? launch_page_m<D, 16, true>(p, stream) : launch_page_m<D, 16, false>(p, stream);
    case 32: return p.meta_bf16 ? launch_page_m<D, 32, true>(p, stream) : launch_page_m<D, 32, false>(p, stream);
    case 64: return p.meta_bf16 ? launch_page_m<D, 64, true>(p, stream) : launch_page_m<D, 64, false>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

#define SAW_CAT2(a, b) a##b
#define SAW_CAT(a, b) SAW_CAT2(a, b)
#ifndef SAW_DECODE_OTHER_DIMS
// head_dim 128 (and the fused decode step)
cudaError_t SAW_CAT(launch_paged_decode_w, SAW_DECODE_WARPS)(const DecodeParams& p,
                                                             cudaStream_t stream) {
  return launch_dim<kHeadDim>(p, stream);
}
#else
// head_dim 64 and 256 (this object is the same source built for those sizes)
cudaError_t SAW_CAT(launch_paged_decode_dims_w, SAW_DECODE_WARPS)(const DecodeParams& p,
                                                                  cudaStream_t stream) {
  if (p.append) return cudaErrorInvalidValue;
  switch (p.head_dim) {
    case 64:
      if (p.pair) {  // two kv-heads per CTA, as one head_dim-128 head (16-token pages)
        if (p.num_seqs == 0) return cudaSuccess;
        if (p.page_size != 16 || p.group != 4 || p.num_kv_heads % 2) return cudaErrorInvalidValue;
        return p.meta_bf16 ? launch_p<128, 16, false, false, true, true>(p, stream)
                           : launch_p<128, 16, false, false, false, true>(p, stream);
      }
      return launch_dim<64>(p, stream);
    case 256: return launch_dim<256>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}
#endif

}  // namespace saw
