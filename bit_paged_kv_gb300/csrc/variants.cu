// variants.cu -- the SAW-INT4 path at head_dim 64 and 256 (rotation blocks
// up to h = 256): quantize-append and paged decode attention.
//
// Pages: youngju.dev "INT4 KV-cache quantization", "Why Naive INT4 Breaks"
// (one scale per token), "The Rotation Trick -- Block-Diagonal Hadamard"
// (blocks of h); gist.science "SAW-INT4", s.2.  The method is stated for any
// head size; the head_dim-128 kernels (quantize_append.cu, paged_decode.cu)
// are specialised for 128, and these serve the other sizes with the same
// cache layout (chunk = P*D/2 code bytes, then P words {s, z}, binary16 or
// bfloat16) and the same bits, for bfloat16 or binary16 input rows.
//
//  * Append: one warp per (token, kv-head) row, lane l holding elements
//    E l .. E l + E - 1 (E = D/32).  The butterfly is the ascending-stride
//    sequence of RN(a + b), RN(a - b) steps -- strides below E inside a lane,
//    the rest across lanes -- then one RN multiply by binary32(1/sqrt h), so
//    the codes and (s, z) are the oracle's to the bit, as in the 128 path.
//  * Decode: CUDA-core kernel, one 4-warp CTA per (split, kv-head, sequence),
//    the GQA group fused (a page is read once).  Scores with lane = token
//    (q' broadcast from shared memory), each lane also staging its token's
//    V row in shared memory; P.V with lane = 2D/64 dims (the chunk's p*s
//    broadcast from shared memory, V rows from the staged copy); online
//    softmax per head;
//    split partials merged in the last split to arrive (two counters per
//    (sequence, kv-head), bounded wait), as in the 128 path.
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

// ------------------------------------------------------------------ decode

constexpr int kVW = 4;                 // warps per CTA
constexpr int kVThreads = 32 * kVW;

template <int D>
struct VarCfg {
  static constexpr int kQr = 0;                                   // f32 [8][D] q'
  static constexpr int kQsum = kQr + kMaxGroup * D * 4;           // f32 [8]
  static constexpr int kPs = kQsum + kMaxGroup * 4;               // f32 [warps][8][32]
  static constexpr int kRed = kPs + kVW * kMaxGroup * 32 * 4;     // f32 [warps][8][D]
  static constexpr int kRedM = kRed + kVW * kMaxGroup * D * 4;    // f32 [warps][8] m, l, z
  static constexpr int kTot = kRedM + 3 * kVW * kMaxGroup * 4;    // f32 [3][8]: den, M, Z
  static constexpr int kFlag = kTot + 3 * kMaxGroup * 4;          // int [4]
  // each warp's 32 V rows of the current chunk, rows padded by 16 bytes so
  // that the lanes' 16-byte stores of their own rows hit distinct banks
  static constexpr int kVRow = D / 2 + 16;
  static constexpr int kVbuf = (kFlag + 16 + 15) / 16 * 16;       // u8 [warps][32][kVRow]
  static constexpr int kSmem = kVbuf + kVW * 32 * kVRow;
};

// In-place Sylvester butterfly over the first `rows` rows of a [rows][D]
// shared array, within blocks of h, then scaled by c.
template <int D>
__device__ void smem_fwht(float* a, int rows, int h, float c) {
  for (int len = 1; len < h; len *= 2) {
    for (int idx = threadIdx.x; idx < rows * (D / 2); idx += blockDim.x) {
      const int r = idx / (D / 2), k = idx - r * (D / 2);
      const int i = ((k & ~(len - 1)) << 1) | (k & (len - 1));
      float* row = a + r * D;
      const float x = row[i], y = row[i + len];
      row[i] = x + y;
      row[i + len] = x - y;
    }
    __syncthreads();
  }
  for (int idx = threadIdx.x; idx < rows * D; idx += blockDim.x) a[idx] *= c;
  __syncthreads();
}

template <int D, int P>
__global__ void __launch_bounds__(kVThreads) paged_decode_var_kernel(const DecodeParams p) {
  pdl_wait_then_release();
  using C = VarCfg<D>;
  constexpr int E = D / 32;       // dims per lane in the P.V phase
  constexpr int NB = D / 64;      // their code bytes
  constexpr int kRowB = D / 2;    // code bytes per token row
  constexpr int kChunk = P * (D / 2 + 4);
  extern __shared__ __align__(16) uint8_t smem[];
  float* qr = reinterpret_cast<float*>(smem + C::kQr);
  float* qsum = reinterpret_cast<float*>(smem + C::kQsum);
  float* psb = reinterpret_cast<float*>(smem + C::kPs);
  float* red = reinterpret_cast<float*>(smem + C::kRed);
  float* red_m = reinterpret_cast<float*>(smem + C::kRedM);
  float* red_l = red_m + kVW * kMaxGroup;
  float* red_z = red_l + kVW * kMaxGroup;
  float* tot = reinterpret_cast<float*>(smem + C::kTot);
  int* flag = reinterpret_cast<int*>(smem + C::kFlag);

  const int split = blockIdx.x, kvh = blockIdx.y, seq = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group, hq0 = kvh * G;
  int L = p.seq_lens[seq];
  if (L < 0 || L > p.max_seq_len) {
    if (split == 0 && kvh == 0 && tid == 0) report(p.dev_status, SAW_ERR_DEVICE_INDEX);
    L = 0;
  }
  const int n_pages = (L + P - 1) / P;
  const int p_begin = split * p.pages_per_split;
  const int p_end = min(n_pages, p_begin + p.pages_per_split);
  const bool direct = p.num_splits == 1;
  if (p_begin >= p_end) {
    if (split == 0 && n_pages == 0)
      for (int idx = tid; idx < G * D; idx += kVThreads)
        p.out[(int64_t(seq) * p.num_q_heads + hq0) * D + idx] = 0.0f;
    return;
  }

  // ---- q' = (1/sqrt h) H q per head of the group, and sum(q')
  for (int idx = tid; idx < G * D; idx += kVThreads) {
    const uint16_t b = p.q[(int64_t(seq) * p.num_q_heads + hq0) * D + idx];
    qr[idx] = in_lo(b, p.in_f16 != 0);
  }
  __syncthreads();
  if (p.rotate_k) smem_fwht<D>(qr, G, p.block_h, p.c_h);
  for (int h = warp; h < G; h += kVW) {
    float s = 0.0f;
    for (int d = lane; d < D; d += 32) s += qr[h * D + d];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) s += __shfl_xor_sync(kAll, s, m);
    if (lane == 0) qsum[h] = s;
  }
  __syncthreads();

  const float qscale = p.q_scale;
  const int32_t* btab = p.block_tables + int64_t(seq) * p.max_blocks;
  const int tok_begin = p_begin * P, tok_end = min(L, p_end * P);
  float m_run[kMaxGroup], l_run[kMaxGroup], z_run[kMaxGroup], o[kMaxGroup][E];
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.0f;
    z_run[h] = 0.0f;
#pragma unroll
    for (int e = 0; e < E; ++e) o[h][e] = 0.0f;
  }
  float* ps = psb + warp * kMaxGroup * 32;
  uint8_t* vbuf = smem + C::kVbuf + warp * 32 * C::kVRow;

  for (int t0 = tok_begin + 32 * warp; t0 < tok_end; t0 += 32 * kVW) {
    const int tok = t0 + lane;
    const bool live = tok < tok_end;
    int pid = -1;
    if (live) {
      pid = btab[tok / P];
      if (pid < 0 || pid >= p.num_pages) {
        report(p.dev_status, SAW_ERR_DEVICE_INDEX);
        pid = -1;
      }
    }
    const bool ok = pid >= 0;
    const int off = tok % P;
    // ---- scores, lane = token
    float t[kMaxGroup];
    float vs = 0.0f, vz = 0.0f;
    if (ok) {
      const uint8_t* kc = p.k_cache + (int64_t(pid) * p.num_kv_heads + kvh) * kChunk;
      const uint8_t* vcb = p.v_cache + (int64_t(pid) * p.num_kv_heads + kvh) * kChunk;
      const uint32_t km = *reinterpret_cast<const uint32_t*>(kc + P * kRowB + 4 * off);
      const uint32_t vm = *reinterpret_cast<const uint32_t*>(vcb + P * kRowB + 4 * off);
      const bool bfm = p.meta_bf16 != 0;
      const float ks = meta_lo(km, bfm), kz = meta_hi(km, bfm);
      vs = meta_lo(vm, bfm);
      vz = meta_hi(vm, bfm);
      // this token's V row into the warp's buffer: all 32 rows arrive in one
      // round of memory latency, not one round per token of the P.V loop
      {
        const uint4* vsrc = reinterpret_cast<const uint4*>(vcb + off * kRowB);
        uint4* vdst = reinterpret_cast<uint4*>(vbuf + lane * C::kVRow);
#pragma unroll
        for (int piece = 0; piece < kRowB / 16; ++piece) vdst[piece] = vsrc[piece];
      }
      float dot[kMaxGroup];
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) dot[h] = 0.0f;
      const uint4* krow = reinterpret_cast<const uint4*>(kc + off * kRowB);
#pragma unroll
      for (int piece = 0; piece < kRowB / 16; ++piece) {
        const uint4 w = krow[piece];
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          // 8 dims: 32 piece + 8 j + (0..7), low nibble first
          float n[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) n[e] = float((ws[j] >> (4 * e)) & 15u);
          const int d0 = 32 * piece + 8 * j;
#pragma unroll
          for (int h = 0; h < kMaxGroup; ++h) {
            if (h < G) {
              const float4 qa = *reinterpret_cast<const float4*>(qr + h * D + d0);
              const float4 qb = *reinterpret_cast<const float4*>(qr + h * D + d0 + 4);
              dot[h] = fmaf(qa.x, n[0], fmaf(qa.y, n[1], fmaf(qa.z, n[2], fmaf(qa.w, n[3], dot[h]))));
              dot[h] = fmaf(qb.x, n[4], fmaf(qb.y, n[5], fmaf(qb.z, n[6], fmaf(qb.w, n[7], dot[h]))));
            }
          }
        }
      }
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) t[h] = qscale * fmaf(ks, dot[h], kz * qsum[h < G ? h : 0]);
    } else {
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) t[h] = -INFINITY;
    }
    // ---- online softmax per head over the chunk's 32 tokens
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h < G) {
        float mt = t[h];
#pragma unroll
        for (int m = 16; m >= 1; m >>= 1) mt = fmaxf(mt, __shfl_xor_sync(kAll, mt, m));
        if (mt > m_run[h]) {
          const float a = ex2(m_run[h] - mt);
          m_run[h] = mt;
          l_run[h] *= a;
          z_run[h] *= a;
#pragma unroll
          for (int e = 0; e < E; ++e) o[h][e] *= a;
        }
        const float mu = (m_run[h] == -INFINITY) ? 0.0f : m_run[h];
        const float pr = ok ? ex2(t[h] - mu) : 0.0f;
        l_run[h] += pr;
        z_run[h] = fmaf(pr, vz, z_run[h]);
        ps[h * 32 + lane] = pr * vs;
      }
    }
    __syncwarp();
    // ---- P.V, lane = dims [E lane, E lane + E)
    const int n_tok = min(32, tok_end - t0);
    for (int j = 0; j < n_tok; ++j) {
      const int pj = __shfl_sync(kAll, pid, j);
      if (pj < 0) continue;  // warp-uniform
      const uint8_t* vrow = vbuf + j * C::kVRow + NB * lane;
      uint32_t cw;
      if (NB == 1)
        cw = *vrow;
      else
        cw = *reinterpret_cast<const uint32_t*>(vrow);
      float n[E];
#pragma unroll
      for (int e = 0; e < E; ++e) n[e] = float((cw >> (4 * e)) & 15u);
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) {
        if (h < G) {
          const float w = ps[h * 32 + j];
#pragma unroll
          for (int e = 0; e < E; ++e) o[h][e] = fmaf(w, n[e], o[h][e]);
        }
      }
    }
    __syncwarp();
  }

  // ---- merge the warps
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    float l = l_run[h], z = z_run[h];
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) {
      l += __shfl_xor_sync(kAll, l, m);
      z += __shfl_xor_sync(kAll, z, m);
    }
    if (h < G) {
      if (lane == 0) {
        red_m[warp * kMaxGroup + h] = m_run[h];
        red_l[warp * kMaxGroup + h] = l;
        red_z[warp * kMaxGroup + h] = z;
      }
#pragma unroll
      for (int e = 0; e < E; ++e) red[(warp * kMaxGroup + h) * D + E * lane + e] = o[h][e];
    }
  }
  // the split's arrival, counted early so the round trip overlaps the merge
  const int ns = (n_pages + p.pages_per_split - 1) / p.pages_per_split;
  uint32_t* tk = p.tickets + 2 * (int64_t(seq) * p.num_kv_heads + kvh);
  uint32_t arrived = 0;
  if (!direct && tid == 0)
    asm volatile("atom.relaxed.gpu.global.add.u32 %0, [%1], 1;" : "=r"(arrived) : "l"(tk) : "memory");
  __syncthreads();
  if (tid < kMaxGroup) {
    const int h = tid;
    float M = -INFINITY;
    for (int w = 0; w < kVW; ++w) M = fmaxf(M, red_m[w * kMaxGroup + h]);
    const float Mu = (M == -INFINITY) ? 0.0f : M;
    float den = 0.0f, zz = 0.0f;
    for (int w = 0; w < kVW; ++w) {
      const float f = ex2(red_m[w * kMaxGroup + h] - Mu);
      red_m[w * kMaxGroup + h] = f;  // now the warp's weight
      den += red_l[w * kMaxGroup + h] * f;
      zz += red_z[w * kMaxGroup + h] * f;
    }
    tot[h] = den;
    tot[kMaxGroup + h] = M;
    tot[2 * kMaxGroup + h] = zz;
  }
  __syncthreads();
  // numerator per (head, dim): sum_w f_w O_w + sum(p z); keep it in red[0]
  for (int idx = tid; idx < G * D; idx += kVThreads) {
    const int h = idx / D;
    float num = tot[2 * kMaxGroup + h];
#pragma unroll
    for (int w = 0; w < kVW; ++w) num = fmaf(red_m[w * kMaxGroup + h], red[w * kMaxGroup * D + idx], num);
    red[idx] = num;
  }
  if (!direct) {
    for (int idx = tid; idx < G * D; idx += kVThreads) {
      const int h = idx / D, dd = idx - h * D;
      const int64_t row = (int64_t(seq) * p.num_q_heads + hq0 + h) * p.num_splits + split;
      p.part_o[row * D + dd] = red[idx];
      if (dd == 0) {
        p.part_ml[2 * row] = tot[kMaxGroup + h];
        p.part_ml[2 * row + 1] = tot[h];
      }
    }
    if (tid == 0) {
      const uint32_t done = arrived + 1u;
      if (done > uint32_t(ns)) report(p.dev_status, SAW_ERR_DEVICE_INDEX);  // not zero-filled
      flag[0] = (done == uint32_t(ns));
    }
    __syncthreads();
    if (!flag[0]) {
      if (tid == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(tk + 1) : "memory");
      return;
    }
    if (tid == 0) {
      const uint32_t want = uint32_t(ns - 1);
      bool okw = ld_acquire_u32(tk + 1) == want;
      if (!okw) {
        const long long c0 = clock64();
        while (!(okw = (ld_acquire_u32(tk + 1) == want))) {
          if (clock64() - c0 > kWaitLimitCycles) break;
          __nanosleep(32);
        }
      }
      if (okw) {
        tk[0] = 0u;
        tk[1] = 0u;
      } else {
        report(p.dev_status, SAW_ERR_DEVICE_TIMEOUT);
      }
      flag[1] = okw ? 1 : 0;
    }
    __syncthreads();
    const bool merge_ok = flag[1] != 0;
    for (int idx = tid; idx < G * D; idx += kVThreads) {
      const int h = idx / D, dd = idx - h * D;
      const int64_t row0 = (int64_t(seq) * p.num_q_heads + hq0 + h) * p.num_splits;
      float M = tot[kMaxGroup + h];
      if (merge_ok)
        for (int sp = 0; sp < ns; ++sp)
          if (sp != split) M = fmaxf(M, __ldcg(&p.part_ml[2 * (row0 + sp)]));
      const float Mu = (M == -INFINITY) ? 0.0f : M;
      float num = red[idx] * ex2(tot[kMaxGroup + h] - Mu);
      float den = tot[h] * ex2(tot[kMaxGroup + h] - Mu);
      if (merge_ok)
        for (int sp = 0; sp < ns; ++sp) {
          if (sp == split) continue;
          const float f = ex2(__ldcg(&p.part_ml[2 * (row0 + sp)]) - Mu);
          den = fmaf(__ldcg(&p.part_ml[2 * (row0 + sp) + 1]), f, den);
          num = fmaf(__ldcg(&p.part_o[(row0 + sp) * D + dd]), f, num);
        }
      red[kMaxGroup * D + idx] = den;  // scratch: the merged denominators
      red[idx] = num;
    }
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kVThreads) {
      const float den = red[kMaxGroup * D + idx];
      red[idx] = (den > 0.0f) ? red[idx] / den : 0.0f;
    }
  } else {
    __syncthreads();
    for (int idx = tid; idx < G * D; idx += kVThreads) {
      const float den = tot[idx / D];
      red[idx] = (den > 0.0f) ? red[idx] / den : 0.0f;
    }
  }
  __syncthreads();
  if (p.rotate_v) smem_fwht<D>(red, G, p.block_h, p.c_h);
  for (int idx = tid; idx < G * D; idx += kVThreads)
    p.out[(int64_t(seq) * p.num_q_heads + hq0) * D + idx] = red[idx];
}

template <typename K>
cudaError_t launch_var(K kernel, dim3 grid, int threads, int smem, cudaStream_t stream,
                       const DecodeParams& p) {
  if (smem > 48 * 1024) {
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, p);
}

template <int D>
cudaError_t launch_decode_var_d(const DecodeParams& p, cudaStream_t stream) {
  const dim3 grid(p.num_splits, p.num_kv_heads, p.num_seqs);
  const int smem = VarCfg<D>::kSmem;
  switch (p.page_size) {
    case 16: return launch_var(paged_decode_var_kernel<D, 16>, grid, kVThreads, smem, stream, p);
    case 32: return launch_var(paged_decode_var_kernel<D, 32>, grid, kVThreads, smem, stream, p);
    case 64: return launch_var(paged_decode_var_kernel<D, 64>, grid, kVThreads, smem, stream, p);
    default: return cudaErrorInvalidValue;
  }
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

cudaError_t launch_quantize_append_var(const AppendParams& p, int head_dim, cudaStream_t stream) {
  if (int64_t(p.num_tokens) * p.num_kv_heads == 0) return cudaSuccess;
  const bool any_rot = p.rotate[0] || (p.num_tensors > 1 && p.rotate[1]);
  const int h = any_rot ? p.block_h : 16;  // unrotated: h is not used
  switch (head_dim) {
    case 64: return launch_append_var_d<64>(p, h, stream);
    case 256: return launch_append_var_d<256>(p, h, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_paged_decode_var(const DecodeParams& p, int head_dim, cudaStream_t stream) {
  if (p.num_seqs == 0) return cudaSuccess;
  switch (head_dim) {
    case 64: return launch_decode_var_d<64>(p, stream);
    case 256: return launch_decode_var_d<256>(p, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace saw
