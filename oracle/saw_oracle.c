/*
 * saw_oracle.c -- TEST INFRASTRUCTURE, not product code.
 *
 * A plain, slow CPU statement of what the SAW-INT4 hot path computes: the
 * block-diagonal Hadamard rotation, token-wise asymmetric INT4 quantization
 * appended into a paged KV cache, and decode attention over that cache.
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * load this library.  It shares no source, header, table or constant with
 * the CUDA library, and it includes nothing from it.
 *
 * Build: plain C11, -O2 -ffp-contract=off, no fast-math.  Every `float`
 * expression below is therefore one IEEE-754 binary32 operation rounded to
 * nearest-even, in the order written; `double` is used where the result is
 * the mathematical reference (rotation by the explicit matrix, attention).
 *
 * Sources (web pages on SAW-INT4, Jia et al., 2026):
 *   [EN]  youngju.dev, "INT4 KV-cache quantization" (English transcription):
 *         "Why Naive INT4 Breaks", "The Rotation Trick -- Block-Diagonal
 *         Hadamard", "The System Is the Design -- A Fused Kernel".
 *   [IT]  gist.science, "SAW-INT4: System-Aware 4-Bit KV-Cache Quantization
 *         for Real-World LLM Serving": s.2 "Metodologia" (token-wise
 *         quantization; Block-Diagonal Rotation), s.4 "Risultati".
 * Where the pages are silent (scale/zero form, rounding, packing, Hadamard
 * ordering, stage order) the comments say which reading is taken.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-2)
#define ORACLE_EPAGE (-3)

/* fp16 rounding modes used by the quantizer. */
#define ORACLE_RN 0 /* nearest, ties to even */
#define ORACLE_RD 1 /* toward -infinity      */
#define ORACLE_RU 2 /* toward +infinity      */

/*
 * Number formats.  K, V and q rows arrive as bfloat16 (in_f16 = 0) or as
 * binary16 (in_f16 = 1: the [EN] fused-kernel diagram feeds "K,V (fp16)");
 * the per-row (scale, zero) pair is stored as binary16 (meta_bf16 = 0) or
 * as bfloat16 (meta_bf16 = 1).  Both input formats widen exactly to binary32,
 * so the quantizer's arithmetic after step 1 is the same for either.
 */

static int is_pow2(int32_t h) { return h > 0 && (h & (h - 1)) == 0; }

/* ------------------------------------------------------------------ */
/* Number formats                                                      */
/* ------------------------------------------------------------------ */

/* bfloat16 is the top half of a binary32: widening is exact. */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

double oracle_f16_to_f64(uint16_t h) {
  int neg = (h >> 15) & 1;
  int e = (h >> 10) & 31;
  int m = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  else if (e == 31)
    v = m ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  return neg ? -v : v;
}

/*
 * binary32 -> binary16 with an explicit rounding mode, written from the
 * IEEE-754 definition: find the spacing of binary16 values around |x|,
 * count whole spacings (exact in double), round that count by the mode, and
 * encode.  Magnitudes beyond the largest finite binary16 saturate to 65504
 * (the "satfinite" reading).  A zero result is always encoded as +0, so the
 * sign of a zero input can never change the stored bits.  NaN -> 0x7E00.
 */
uint16_t oracle_f32_to_f16(float x, int32_t mode) {
  if (isnan(x)) return 0x7E00;
  int neg = signbit(x) ? 1 : 0;
  double a = fabs((double)x);
  double v;
  if (a > 65504.0) {
    v = 65504.0;
  } else {
    double ulp;
    if (a < ldexp(1.0, -14)) {
      ulp = ldexp(1.0, -24);
    } else {
      int e;
      frexp(a, &e); /* a in [2^(e-1), 2^e) */
      ulp = ldexp(1.0, (e - 1) - 10);
    }
    double m = a / ulp; /* exact: division by a power of two */
    double lo = floor(m), hi = ceil(m), r;
    if (mode == ORACLE_RN) {
      double frac = m - lo;
      if (frac > 0.5)
        r = hi;
      else if (frac < 0.5)
        r = lo;
      else
        r = (fmod(lo, 2.0) == 0.0) ? lo : hi;
    } else if ((mode == ORACLE_RD) != (neg != 0)) {
      r = lo; /* toward -inf on a positive value, toward +inf on a negative one */
    } else {
      r = hi;
    }
    v = r * ulp;
    if (v > 65504.0) v = 65504.0;
  }
  if (v == 0.0) return 0; /* canonical +0 */
  uint16_t bits;
  if (v < ldexp(1.0, -14)) {
    bits = (uint16_t)(v / ldexp(1.0, -24));
  } else {
    int e;
    frexp(v, &e);
    int E = e - 1; /* v in [2^E, 2^(E+1)) */
    double mant = (v / ldexp(1.0, E) - 1.0) * 1024.0;
    bits = (uint16_t)(((E + 15) << 10) | (int)mant);
  }
  if (neg) bits |= 0x8000;
  return bits;
}

/*
 * binary32 -> bfloat16 with an explicit rounding mode, by the same
 * definition.  bfloat16 has binary32's exponent range and 8 significant
 * bits: for |x| in [2^(e-1), 2^e) the spacing is 2^(e-8), and below 2^-126
 * (the subnormals) it is 2^-133.  Magnitudes beyond the largest finite
 * bfloat16, 2^128 - 2^120, saturate to it; a zero result is +0; NaN ->
 * 0x7FC0.  Every bfloat16 value is a binary32 value, so the bits of the
 * result are the upper half of its binary32 encoding.
 */
uint16_t oracle_f32_to_bf16(float x, int32_t mode) {
  if (isnan(x)) return 0x7FC0;
  const double max_bf16 = ldexp(255.0, 120); /* (2 - 2^-7) * 2^127 */
  int neg = signbit(x) ? 1 : 0;
  double a = fabs((double)x);
  double v;
  if (a > max_bf16) {
    v = max_bf16;
  } else {
    double ulp;
    if (a < ldexp(1.0, -126)) {
      ulp = ldexp(1.0, -133);
    } else {
      int e;
      frexp(a, &e); /* a in [2^(e-1), 2^e) */
      ulp = ldexp(1.0, (e - 1) - 7);
    }
    double m = a / ulp; /* exact */
    double lo = floor(m), hi = ceil(m), r;
    if (mode == ORACLE_RN) {
      double frac = m - lo;
      if (frac > 0.5)
        r = hi;
      else if (frac < 0.5)
        r = lo;
      else
        r = (fmod(lo, 2.0) == 0.0) ? lo : hi;
    } else if ((mode == ORACLE_RD) != (neg != 0)) {
      r = lo;
    } else {
      r = hi;
    }
    v = r * ulp;
    if (v > max_bf16) v = max_bf16;
  }
  if (v == 0.0) return 0;
  float f = (float)v; /* exact */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  uint16_t bits = (uint16_t)(u >> 16);
  if (neg) bits |= 0x8000;
  return bits;
}

/* A stored metadata value in double. */
static double meta_to_f64(uint16_t b, int32_t meta_bf16) {
  return meta_bf16 ? (double)bf16_to_f32(b) : oracle_f16_to_f64(b);
}

/* An input element widened to binary32 (exact for either format). */
static float in_to_f32(uint16_t b, int32_t in_f16) {
  return in_f16 ? (float)oracle_f16_to_f64(b) : bf16_to_f32(b);
}

/* ------------------------------------------------------------------ */
/* Rotation: block-diagonal Sylvester Hadamard, blocks of size h        */
/* [EN] "The Rotation Trick"; [IT] s.2 "Rotazione Block-Diagonale"      */
/* ------------------------------------------------------------------ */

/* Sylvester construction: H_1 = [1], H_2n = [[H_n, H_n], [H_n, -H_n]].
 * Writes the h x h matrix row-major into H (entries +1 / -1). */
int32_t oracle_sylvester(int32_t h, int8_t* H) {
  if (!is_pow2(h) || !H) return ORACLE_EINVAL;
  H[0] = 1;
  for (int32_t n = 1; n < h; n *= 2) {
    for (int32_t i = 0; i < n; ++i) {
      for (int32_t j = 0; j < n; ++j) {
        int8_t a = H[i * h + j];
        H[i * h + (j + n)] = a;
        H[(i + n) * h + j] = a;
        H[(i + n) * h + (j + n)] = (int8_t)-a;
      }
    }
  }
  return ORACLE_OK;
}

/* (R-exact) y_b = (1/sqrt(h)) * H_h * x_b for every block b of the D-vector,
 * in double, by the explicit matrix.  This is the mathematical rotation the
 * attention reference uses.  y may not alias x. */
int32_t oracle_rotate_exact(const double* x, int32_t D, int32_t h, double* y) {
  if (!is_pow2(h) || D <= 0 || D % h != 0 || !x || !y) return ORACLE_EINVAL;
  int8_t* H = (int8_t*)malloc((size_t)h * (size_t)h);
  if (!H) return ORACLE_ENOMEM;
  oracle_sylvester(h, H);
  double c = 1.0 / sqrt((double)h);
  for (int32_t b0 = 0; b0 < D; b0 += h) {
    for (int32_t i = 0; i < h; ++i) {
      double acc = 0.0;
      for (int32_t j = 0; j < h; ++j) acc += (double)H[i * h + j] * x[b0 + j];
      y[b0 + i] = c * acc;
    }
  }
  free(H);
  return ORACLE_OK;
}

/* The binary32 normalisation constant: 1/sqrt(h) computed in double and
 * rounded once to binary32. */
float oracle_block_scale_f32(int32_t h) { return (float)(1.0 / sqrt((double)h)); }

/* (R-canon) the binary32 rotation whose bits the quantized cache is defined
 * by.  Reading taken where the pages are silent: an in-place fast
 * Walsh-Hadamard butterfly per block with strides in ascending order
 * (1, 2, ..., h/2), each butterfly (a, b) -> (a + b, a - b) rounded to
 * nearest, then one multiplication by the binary32 1/sqrt(h) after the last
 * stage.  Mathematically this equals R-exact. */
int32_t oracle_rotate_canon(float* u, int32_t D, int32_t h) {
  if (!is_pow2(h) || D <= 0 || D % h != 0 || !u) return ORACLE_EINVAL;
  const float c = oracle_block_scale_f32(h);
  for (int32_t b0 = 0; b0 < D; b0 += h) {
    float* w = u + b0;
    for (int32_t len = 1; len < h; len *= 2) {
      for (int32_t i = 0; i < h; ++i) {
        if ((i & len) == 0) {
          float a = w[i];
          float b = w[i + len];
          w[i] = a + b;
          w[i + len] = a - b;
        }
      }
    }
    for (int32_t i = 0; i < h; ++i) w[i] = w[i] * c;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Token-wise INT4 quantization of one (token, kv-head) row             */
/* [EN] "Why Naive INT4 Breaks" (one scale per token, never revisiting  */
/* past tokens); [IT] s.2 "Quantizzazione Token-wise".                  */
/* ------------------------------------------------------------------ */

/*
 * Quantize one row of D bfloat16 (or binary16, in_f16) values.  Steps, in
 * this order:
 *  1. widen to binary32 (exact);
 *  2. if rotate: R-canon rotation with blocks of h;
 *  3. mn, mx = min and max over all D values (one scale per row, spanning
 *     every h-block);
 *  4. zero-point z = fp16(mn) rounded toward -inf, scale
 *     s = fp16((mx - z) / 15) rounded toward +inf (bfloat16 for both when
 *     meta_bf16, a nonzero scale then at least 2^-126); so every value lies
 *     in [z, z + 15 s] and the dequantization error is at most s/2;
 *  5. r = 1/s (0 when s == 0), code_i = clamp(rne((y_i - z) * r), 0, 15);
 *  6. pack two codes per byte, the even index in the low nibble.
 * The asymmetric fp16 (scale, zero) pair, directed rounding, round-half-even
 * and nibble order are readings taken where the pages are silent; so are
 * the bfloat16 metadata variant and its saturation at the largest finite
 * bfloat16.
 * codes: D/2 bytes.  *s_bits, *z_bits: binary16 (or bfloat16) bit patterns.
 */
int32_t oracle_quantize_row(const uint16_t* x, int32_t in_f16, int32_t D, int32_t rotate,
                            int32_t h, int32_t meta_bf16, uint8_t* codes, uint16_t* s_bits,
                            uint16_t* z_bits) {
  if (!x || !codes || !s_bits || !z_bits || D <= 0 || (D & 1)) return ORACLE_EINVAL;
  if (rotate && (!is_pow2(h) || D % h != 0)) return ORACLE_EINVAL;
  float* y = (float*)malloc(sizeof(float) * (size_t)D);
  uint8_t* q = (uint8_t*)malloc((size_t)D);
  if (!y || !q) {
    free(y);
    free(q);
    return ORACLE_ENOMEM;
  }
  for (int32_t i = 0; i < D; ++i) y[i] = in_to_f32(x[i], in_f16);
  if (rotate) oracle_rotate_canon(y, D, h);

  float mn = y[0], mx = y[0];
  for (int32_t i = 1; i < D; ++i) {
    if (y[i] < mn) mn = y[i];
    if (y[i] > mx) mx = y[i];
  }
  uint16_t zb = meta_bf16 ? oracle_f32_to_bf16(mn, ORACLE_RD) : oracle_f32_to_f16(mn, ORACLE_RD);
  float z = (float)meta_to_f64(zb, meta_bf16);
  float range = mx - z;
  float step = range / 15.0f;
  uint16_t sb =
      meta_bf16 ? oracle_f32_to_bf16(step, ORACLE_RU) : oracle_f32_to_f16(step, ORACLE_RU);
  /* A bfloat16 scale below 2^-126 would make 1/s overflow binary32; such a
   * scale is raised to 2^-126, the smallest normal bfloat16 (a coarser step
   * still covers [z, z + 15 s]).  Binary16 scales are >= 2^-24: no floor. */
  if (meta_bf16 && step > 0.0f && bf16_to_f32(sb) < ldexpf(1.0f, -126)) sb = 0x0080;
  float s = (float)meta_to_f64(sb, meta_bf16);
  float r = (s == 0.0f) ? 0.0f : 1.0f / s;

  for (int32_t i = 0; i < D; ++i) {
    float diff = y[i] - z;
    float v = diff * r;
    float c = nearbyintf(v); /* default rounding mode: to nearest, ties to even */
    if (c < 0.0f) c = 0.0f;
    if (c > 15.0f) c = 15.0f;
    q[i] = (uint8_t)c;
  }
  for (int32_t j = 0; j < D / 2; ++j) codes[j] = (uint8_t)(q[2 * j] | (q[2 * j + 1] << 4));
  *s_bits = sb;
  *z_bits = zb;
  free(y);
  free(q);
  return ORACLE_OK;
}

/* Dequantize one row: y_hat_i = code_i * s + z, in double. */
int32_t oracle_dequant_row(const uint8_t* codes, uint16_t s_bits, uint16_t z_bits,
                           int32_t meta_bf16, int32_t D, double* out) {
  if (!codes || !out || D <= 0 || (D & 1)) return ORACLE_EINVAL;
  double s = meta_to_f64(s_bits, meta_bf16), z = meta_to_f64(z_bits, meta_bf16);
  for (int32_t j = 0; j < D / 2; ++j) {
    out[2 * j] = (double)(codes[j] & 15) * s + z;
    out[2 * j + 1] = (double)(codes[j] >> 4) * s + z;
  }
  return ORACLE_OK;
}

/* ------------------------------------------------------------------ */
/* Paged cache layout                                                   */
/* ------------------------------------------------------------------ */
/*
 * Reading (the pages fix only "paged layout, token-wise, appended"): one
 * tensor (K or V) of a layer is [num_pages][num_kv_heads][chunk] bytes, a
 * chunk being P*D/2 code bytes (token offset o at o*D/2) followed by P
 * metadata words (token offset o at P*D/2 + 4*o: scale, then zero, each a
 * little-endian binary16 -- or bfloat16 in the meta_bf16 variant).  Slot s of the cache is page s / P,
 * offset s % P.
 */
int64_t oracle_chunk_bytes(int32_t P, int32_t D) { return (int64_t)P * (D / 2) + (int64_t)P * 4; }

int64_t oracle_cache_bytes(int32_t num_pages, int32_t P, int32_t Hkv, int32_t D) {
  return (int64_t)num_pages * Hkv * oracle_chunk_bytes(P, D);
}

static uint8_t* chunk_ptr(uint8_t* cache, int64_t page, int32_t head, int32_t Hkv, int32_t P,
                          int32_t D) {
  return cache + (page * Hkv + head) * oracle_chunk_bytes(P, D);
}

static void store_row(uint8_t* cache, int64_t slot, int32_t head, int32_t Hkv, int32_t P,
                      int32_t D, const uint8_t* codes, uint16_t sb, uint16_t zb) {
  int64_t page = slot / P;
  int32_t off = (int32_t)(slot % P);
  uint8_t* base = chunk_ptr(cache, page, head, Hkv, P, D);
  memcpy(base + (int64_t)off * (D / 2), codes, (size_t)(D / 2));
  uint8_t* meta = base + (int64_t)P * (D / 2) + 4 * off;
  meta[0] = (uint8_t)(sb & 0xFF);
  meta[1] = (uint8_t)(sb >> 8);
  meta[2] = (uint8_t)(zb & 0xFF);
  meta[3] = (uint8_t)(zb >> 8);
}

/*
 * Quantize and append tokens [token_begin, token_end) of k (and v, unless
 * NULL) into the caches at slot_mapping[t].  k/v are bfloat16 (binary16 when
 * in_f16) bits laid out [token][Hkv][D] with a token stride in elements.  A slot of -1 is padding
 * and skipped; any other slot outside [0, num_pages*P) is skipped and
 * counted.  Returns the count of such bad slots, or a negative error.
 * Every row is quantized on its own: no other token's values are read and no
 * other slot is written ([EN] "never revisiting past tokens").
 */
int64_t oracle_quantize_append(const uint16_t* k, const uint16_t* v, int64_t k_stride,
                               int64_t v_stride, const int32_t* slot_mapping,
                               int32_t token_begin, int32_t token_end, int32_t Hkv, int32_t D,
                               uint8_t* k_cache, uint8_t* v_cache, int32_t num_pages, int32_t P,
                               int32_t rotate_k, int32_t rotate_v, int32_t h, int32_t in_f16,
                               int32_t meta_bf16) {
  if (!k || !slot_mapping || !k_cache || (v && !v_cache) || Hkv <= 0 || D <= 0 || P <= 0 ||
      num_pages < 0 || token_begin < 0 || token_end < token_begin)
    return ORACLE_EINVAL;
  uint8_t* codes = (uint8_t*)malloc((size_t)(D / 2));
  if (!codes) return ORACLE_ENOMEM;
  int64_t bad = 0;
  int64_t nslots = (int64_t)num_pages * P;
  for (int32_t t = token_begin; t < token_end; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot == -1) continue;
    if (slot < 0 || slot >= nslots) {
      ++bad;
      continue;
    }
    for (int32_t hd = 0; hd < Hkv; ++hd) {
      uint16_t sb, zb;
      int32_t rc = oracle_quantize_row(k + (int64_t)t * k_stride + (int64_t)hd * D, in_f16, D,
                                       rotate_k, h, meta_bf16, codes, &sb, &zb);
      if (rc) {
        free(codes);
        return rc;
      }
      store_row(k_cache, slot, hd, Hkv, P, D, codes, sb, zb);
      if (v) {
        rc = oracle_quantize_row(v + (int64_t)t * v_stride + (int64_t)hd * D, in_f16, D,
                                 rotate_v, h, meta_bf16, codes, &sb, &zb);
        if (rc) {
          free(codes);
          return rc;
        }
        store_row(v_cache, slot, hd, Hkv, P, D, codes, sb, zb);
      }
    }
  }
  free(codes);
  return bad;
}

/* ------------------------------------------------------------------ */
/* Decode attention over the INT4 pages, in double                     */
/* ------------------------------------------------------------------ */

static void read_row(const uint8_t* cache, int64_t page, int32_t off, int32_t head, int32_t Hkv,
                     int32_t P, int32_t D, int32_t meta_bf16, double* out) {
  const uint8_t* base = chunk_ptr((uint8_t*)cache, page, head, Hkv, P, D);
  const uint8_t* meta = base + (int64_t)P * (D / 2) + 4 * off;
  uint16_t sb = (uint16_t)(meta[0] | (meta[1] << 8));
  uint16_t zb = (uint16_t)(meta[2] | (meta[3] << 8));
  oracle_dequant_row(base + (int64_t)off * (D / 2), sb, zb, meta_bf16, D, out);
}

/*
 * Attention output of one query row (one sequence, one q-head) over the
 * first seq_len tokens of its pages, all in double:
 *   q'    = (1/sqrt(h)) H q   if K was rotated, else q   (R-exact);
 *   k^_j  = code * s + z       (dequantized cache row, rotated domain);
 *   t_j   = sm_scale * (q' . k^_j);  p = softmax(t) (max-subtracted);
 *   o'    = sum_j p_j v^_j;
 *   o     = (1/sqrt(h)) H o'  if V was rotated, else o'.
 * (1/sqrt(h)) H is symmetric and orthogonal, so q'.k^ = q.(H^-1 k^) and
 * H o' is the un-rotated output ([EN] "orthogonal ... undoable later").
 * q is bfloat16 (binary16 when in_f16) bits; the cache's metadata is
 * binary16 (bfloat16 when meta_bf16).
 * The caller passes the kv-head that serves this q-head.  seq_len == 0
 * gives a zero output.  Returns ORACLE_EPAGE for a page id outside
 * [0, num_pages).
 */
int32_t oracle_decode_one(const uint16_t* q_bits, const uint8_t* k_cache, const uint8_t* v_cache,
                          const int32_t* block_table_row, int32_t seq_len, int32_t kv_head,
                          int32_t Hkv, int32_t D, int32_t num_pages, int32_t P, int32_t rotate_k,
                          int32_t rotate_v, int32_t h, double sm_scale, double* out,
                          int32_t in_f16, int32_t meta_bf16) {
  if (!q_bits || !k_cache || !v_cache || !out || (seq_len > 0 && !block_table_row) || D <= 0 ||
      P <= 0 || seq_len < 0 || kv_head < 0 || kv_head >= Hkv)
    return ORACLE_EINVAL;
  if ((rotate_k || rotate_v) && (!is_pow2(h) || D % h != 0)) return ORACLE_EINVAL;
  for (int32_t i = 0; i < D; ++i) out[i] = 0.0;
  if (seq_len == 0) return ORACLE_OK;

  double* q = (double*)malloc(sizeof(double) * (size_t)D);
  double* qr = (double*)malloc(sizeof(double) * (size_t)D);
  double* row = (double*)malloc(sizeof(double) * (size_t)D);
  double* acc = (double*)calloc((size_t)D, sizeof(double));
  double* t = (double*)malloc(sizeof(double) * (size_t)seq_len);
  int32_t rc = ORACLE_OK;
  if (!q || !qr || !row || !acc || !t) {
    rc = ORACLE_ENOMEM;
    goto done;
  }
  for (int32_t i = 0; i < D; ++i) q[i] = (double)in_to_f32(q_bits[i], in_f16);
  if (rotate_k)
    oracle_rotate_exact(q, D, h, qr);
  else
    memcpy(qr, q, sizeof(double) * (size_t)D);

  for (int32_t j = 0; j < seq_len; ++j) {
    int64_t page = block_table_row[j / P];
    if (page < 0 || page >= num_pages) {
      rc = ORACLE_EPAGE;
      goto done;
    }
    read_row(k_cache, page, j % P, kv_head, Hkv, P, D, meta_bf16, row);
    double dot = 0.0;
    for (int32_t i = 0; i < D; ++i) dot += qr[i] * row[i];
    t[j] = sm_scale * dot;
  }
  double m = t[0];
  for (int32_t j = 1; j < seq_len; ++j)
    if (t[j] > m) m = t[j];
  double l = 0.0;
  for (int32_t j = 0; j < seq_len; ++j) {
    double p = exp(t[j] - m);
    l += p;
    int64_t page = block_table_row[j / P];
    read_row(v_cache, page, j % P, kv_head, Hkv, P, D, meta_bf16, row);
    for (int32_t i = 0; i < D; ++i) acc[i] += p * row[i];
  }
  for (int32_t i = 0; i < D; ++i) acc[i] /= l;
  if (rotate_v)
    oracle_rotate_exact(acc, D, h, out);
  else
    memcpy(out, acc, sizeof(double) * (size_t)D);

done:
  free(q);
  free(qr);
  free(row);
  free(acc);
  free(t);
  return rc;
}

/*
 * Chunked-prefill attention of one query row over the INT4 cache.  The pages
 * place SAW-INT4 inside engines that run fused (FlashAttention-style)
 * attention over paged KV ([EN] "Why the KV Cache Is the Real Bottleneck";
 * [IT] s.1), and define attention only through decode; the reading taken
 * here is plain causal self-attention: the query of the token at position
 * `query_pos` (0-based) of its sequence attends to that sequence's cached
 * tokens 0 .. query_pos (its own K/V included, appended before the
 * attention).
 * That is exactly the decode above over the first query_pos + 1 tokens, so
 * the arithmetic is oracle_decode_one's.
 */
int32_t oracle_prefill_one(const uint16_t* q_bits, const uint8_t* k_cache,
                           const uint8_t* v_cache, const int32_t* block_table_row,
                           int32_t query_pos, int32_t kv_head, int32_t Hkv, int32_t D,
                           int32_t num_pages, int32_t P, int32_t rotate_k, int32_t rotate_v,
                           int32_t h, double sm_scale, double* out, int32_t in_f16,
                           int32_t meta_bf16) {
  if (query_pos < 0) return ORACLE_EINVAL;
  return oracle_decode_one(q_bits, k_cache, v_cache, block_table_row, query_pos + 1, kv_head,
                           Hkv, D, num_pages, P, rotate_k, rotate_v, h, sm_scale, out, in_f16,
                           meta_bf16);
}

/* ------------------------------------------------------------------ */
/* BF16 paged cache: the unquantized baseline ([IT] s.4 compares the   */
/* throughput of INT4 + rotation against a BF16 KV cache)              */
/* ------------------------------------------------------------------ */
/*
 * Layout (ours; the pages name only "BF16"): per layer and tensor,
 * [num_pages][Hkv][P][D] bfloat16, token `off` of page `page` for kv-head
 * `head` at element ((page * Hkv + head) * P + off) * D.
 */
int64_t oracle_bf16_cache_bytes(int32_t num_pages, int32_t P, int32_t Hkv, int32_t D) {
  if (num_pages < 0 || P <= 0 || Hkv <= 0 || D <= 0) return 0;
  return (int64_t)num_pages * Hkv * P * D * 2;
}

/* Copy the rows of tokens [t_begin, t_end) into their slots (slot -1 is
 * padding and skipped; other out-of-range slots are skipped and counted).
 * Returns the count of bad slots. */
int64_t oracle_bf16_append(const uint16_t* k, const uint16_t* v, int64_t k_stride,
                           int64_t v_stride, const int32_t* slot_mapping, int32_t t_begin,
                           int32_t t_end, int32_t Hkv, int32_t D, uint16_t* k_cache,
                           uint16_t* v_cache, int32_t num_pages, int32_t P) {
  if (!k || !slot_mapping || !k_cache || (v && !v_cache) || Hkv <= 0 || D <= 0 || P <= 0)
    return ORACLE_EINVAL;
  int64_t bad = 0;
  const int64_t num_slots = (int64_t)num_pages * P;
  for (int32_t t = t_begin; t < t_end; ++t) {
    const int64_t slot = slot_mapping[t];
    if (slot == -1) continue;
    if (slot < 0 || slot >= num_slots) {
      ++bad;
      continue;
    }
    const int64_t page = slot / P, off = slot % P;
    for (int32_t hd = 0; hd < Hkv; ++hd) {
      const int64_t dst = ((page * Hkv + hd) * P + off) * D;
      memcpy(k_cache + dst, k + (int64_t)t * k_stride + (int64_t)hd * D, sizeof(uint16_t) * D);
      if (v)
        memcpy(v_cache + dst, v + (int64_t)t * v_stride + (int64_t)hd * D, sizeof(uint16_t) * D);
    }
  }
  return bad;
}

/* Attention output of one query row over the first seq_len tokens of its
 * BF16 pages, in double: t_j = sm_scale * (q . k_j), p = softmax(t),
 * o = sum_j p_j v_j.  seq_len == 0 gives zeros; ORACLE_EPAGE for a page id
 * outside [0, num_pages). */
int32_t oracle_decode_bf16_one(const uint16_t* q_bf16, const uint16_t* k_cache,
                               const uint16_t* v_cache, const int32_t* block_table_row,
                               int32_t seq_len, int32_t kv_head, int32_t Hkv, int32_t D,
                               int32_t num_pages, int32_t P, double sm_scale, double* out) {
  if (!q_bf16 || !k_cache || !v_cache || !out || (seq_len > 0 && !block_table_row) || D <= 0 ||
      P <= 0 || seq_len < 0 || kv_head < 0 || kv_head >= Hkv)
    return ORACLE_EINVAL;
  for (int32_t i = 0; i < D; ++i) out[i] = 0.0;
  if (seq_len == 0) return ORACLE_OK;
  double* t = (double*)malloc(sizeof(double) * (size_t)seq_len);
  if (!t) return ORACLE_ENOMEM;
  for (int32_t j = 0; j < seq_len; ++j) {
    const int64_t page = block_table_row[j / P];
    if (page < 0 || page >= num_pages) {
      free(t);
      return ORACLE_EPAGE;
    }
    const uint16_t* kr = k_cache + ((page * Hkv + kv_head) * P + j % P) * D;
    double dot = 0.0;
    for (int32_t i = 0; i < D; ++i) dot += (double)bf16_to_f32(q_bf16[i]) * bf16_to_f32(kr[i]);
    t[j] = sm_scale * dot;
  }
  double m = t[0];
  for (int32_t j = 1; j < seq_len; ++j)
    if (t[j] > m) m = t[j];
  double l = 0.0;
  for (int32_t j = 0; j < seq_len; ++j) {
    const double p = exp(t[j] - m);
    l += p;
    const int64_t page = block_table_row[j / P];
    const uint16_t* vr = v_cache + ((page * Hkv + kv_head) * P + j % P) * D;
    for (int32_t i = 0; i < D; ++i) out[i] += p * bf16_to_f32(vr[i]);
  }
  for (int32_t i = 0; i < D; ++i) out[i] /= l;
  free(t);
  return ORACLE_OK;
}
