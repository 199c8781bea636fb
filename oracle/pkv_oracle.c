/*
 * pkv_oracle.c — the reference (oracle) implementation of paged GQA attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is a plain, slow, deliberately obvious CPU
 * implementation that the GPU library is checked against.  Only the test suite, the
 * package's smoke check and the CPU-baseline leg of the benchmark may load it.  It
 * shares no code, header, table or helper with the CUDA library, and the CUDA library
 * never calls it.
 *
 * What it computes (sources are the pages' titles and sections):
 *   - "Tiny-LLM-Inference Project_Status", feature list: a paged KV cache, chunked
 *     prefill/decode; dtype contract: FP32 KV by default, BF16 KV with its own paged
 *     attention kernel, FP32 operator boundaries.
 *   - "tinyloop Current Status", KV cache modes table: paged attention with 16-token
 *     pages; INT8 KV cache.  Model architecture support table: GQA (fewer KV heads,
 *     MQA too) and chunked prefill.
 * None of the pages writes out the attention formula, so the oracle is the textbook
 * definition of scaled dot-product attention evaluated over the logically reassembled
 * cache:
 *     out[b,h,:] = sum_t softmax_t(scale * q[b,h,:] . K_t[g,:]) * V_t[g,:],  g = h / G
 * in double precision, with max subtraction inside the softmax.  K_t and V_t are the
 * values as stored (FP32 as is, BF16 widened exactly, INT8 as code * scale in double).
 *
 * Physical layout (the library's documented layout, restated here from its
 * specification and not from its code).  Each (page, kv head) pair owns one K block and
 * one V block of 16*D elements; block (page, h) starts at element (page*Hkv + h)*16*D.
 *   FP32 / INT8:  K block [16 tokens][D]     element (t, d) at t*D + d
 *                 V block [D][16 tokens]     element (d, t) at d*16 + t
 *   BF16 (tensor-core tiles of 8x8 "core matrices", each 64 contiguous elements):
 *                 K element (t, d) at ((t/8)*(D/8) + d/8)*64 + (t%8)*8 + d%8
 *                 V element (d, t) at ((d/8)*2  + t/8)*64 + (d%8)*8 + t%8
 *   scales   [num_pages][Hkv][16]  float32     (coded formats; one per token and kv head)
 *   INT8 codes are stored in offset binary: the byte holds code + 128.
 *   slot = page * 16 + offset
 *
 * The INT8 quantiser and the BF16 rounding run in C `float` exactly as specified
 * (IEEE division, round-half-to-even), compiled with -ffp-contract=off and without
 * fast-math, so the stored codes are a function of the inputs alone.
 *
 * One decode step (rotate the new query and key, store the new row, attend) composes
 * these: "tinyloop Current Status", model architecture support table (RoPE with a
 * configurable theta); the rotation convention is a reading (half-split pairs).
 *
 * Parity pins: every function here is pinned by tests that do not re-type it (dense
 * brute force against a library attention, closed forms, permutation invariance,
 * causality, an exhaustive nearest-code search for the quantiser, and the library
 * float->bfloat16 cast for the rounding).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ORACLE_MUTANT selects a deliberately planted mistake; the pin tests build each one
 * and check that some pin fails.  The default build (0) has none. */
#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum { ODT_F32 = 0, ODT_BF16 = 1, ODT_INT8 = 2, ODT_FP8 = 3, ODT_INT4 = 4 };

/* ---------------------------------------------------------------- scalar helpers */

/* bfloat16 -> float: the bf16 bits are the top half of the float32 bits. */
static float bf16_bits_to_float(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* float -> bfloat16 with round-to-nearest, ties to even, on the discarded 16 bits.
 * NaN stays NaN (quiet bit forced). */
uint16_t oracle_f32_to_bf16(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0u)
    return (uint16_t)((u >> 16) | 0x0040u);
  uint32_t lower = u & 0xffffu;
  uint32_t upper = u >> 16;
#if ORACLE_MUTANT == 1 /* ties away from zero */
  if (lower >= 0x8000u) upper += 1u;
#else
  if (lower > 0x8000u || (lower == 0x8000u && (upper & 1u))) upper += 1u;
#endif
  return (uint16_t)upper;
}

/* Read element i of a buffer holding float32 or bfloat16 values. */
static double read_real(const void* p, int dtype, size_t i) {
  if (dtype == ODT_BF16) return (double)bf16_bits_to_float(((const uint16_t*)p)[i]);
  return (double)((const float*)p)[i];
}
static float read_real_f(const void* p, int dtype, size_t i) {
  if (dtype == ODT_BF16) return bf16_bits_to_float(((const uint16_t*)p)[i]);
  return ((const float*)p)[i];
}

/* Symmetric per-row INT8 quantiser: s = max|x| / 127 (float division), code =
 * clamp(round_half_even(x / s), -127, 127); a row of zeros gets s = 0 and codes 0. */
void oracle_quantize_row_int8(const float* x, int n, int8_t* codes, float* scale_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float s = amax / 127.0f;
  for (int i = 0; i < n; ++i) {
    int c = 0;
    if (s != 0.0f) {
#if ORACLE_MUTANT == 2 /* truncation instead of rounding */
      float r = truncf(x[i] / s);
#else
      float r = rintf(x[i] / s);
#endif
      if (r > 127.0f) r = 127.0f;
      if (r < -127.0f) r = -127.0f;
      c = (int)r;
    }
    codes[i] = (int8_t)c;
  }
  *scale_out = s;
}

/*
 * FP8 E4M3, the "fn" member of the OCP 8-bit floating-point formats (named as an option
 * for the KV cache in the TinyInfer review, item 2 "Improve KV cache efficiency"): one
 * sign bit, four exponent bits with bias 7, three mantissa bits; exponent field 0 holds
 * the subnormals m/8 * 2^-6; there is no infinity and S.1111.111 is NaN, so the largest
 * finite magnitude is 1.75 * 2^8 = 448.
 */
double oracle_e4m3_value(uint8_t c) {
  int e = (c >> 3) & 15, m = c & 7;
  double mag;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) mag = ldexp((double)m / 8.0, -6);
  else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
  return (c & 0x80) ? -mag : mag;
}

/* float -> E4M3 code: the nearest finite value, ties to the even code (even mantissa),
 * magnitudes beyond 448 saturating to 448; the sign is kept (a negative value that
 * rounds to zero gives the negative zero 0x80).  Written as a search over the 127
 * finite non-negative codes, whose values increase with the code. */
uint8_t oracle_f32_to_e4m3(float x) {
  double a = fabs((double)x);
  if (a > 448.0) a = 448.0;
  int best = 0;
  double bd = a;  /* distance to code 0 */
  for (int c = 1; c <= 126; ++c) {
    double d = fabs(oracle_e4m3_value((uint8_t)c) - a);
#if ORACLE_MUTANT == 13 /* rounding toward zero */
    if (oracle_e4m3_value((uint8_t)c) <= a) { best = c; bd = d; }
#else
    if (d < bd || (d == bd && (c & 1) == 0)) { best = c; bd = d; }
#endif
  }
  return (uint8_t)(signbit(x) ? (best | 0x80) : best);
}

/* Symmetric per-row FP8 quantiser (the INT8 scheme with the E4M3 range): s = max|x| /
 * 448 (float division), code = e4m3(x / s); a row of zeros gets s = 0 and codes 0. */
void oracle_quantize_row_fp8(const float* x, int n, uint8_t* codes, float* scale_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float s = amax / 448.0f;
  for (int i = 0; i < n; ++i) codes[i] = s != 0.0f ? oracle_f32_to_e4m3(x[i] / s) : 0;
  *scale_out = s;
}

/* Symmetric per-row INT4 quantiser ("tinyloop Current Status", KV cache modes table: an
 * INT4 KV mode, format not given; read as the INT8 scheme with 4-bit codes): s = max|x| / 7
 * (float division), code = clamp(round_half_even(x / s), -7, 7). */
void oracle_quantize_row_int4(const float* x, int n, int8_t* codes, float* scale_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float s = amax / 7.0f;
  for (int i = 0; i < n; ++i) {
    float r = s != 0.0f ? rintf(x[i] / s) : 0.0f;
    if (r > 7.0f) r = 7.0f;
    if (r < -7.0f) r = -7.0f;
    codes[i] = (int8_t)r;
  }
  *scale_out = s;
}

/* ---------------------------------------------------------------- cache addressing */

/*
 * INT4 blocks hold two 4-bit two's-complement codes per byte, D * 8 bytes per block for
 * K and for V of each (page, kv head).
 *   K [16 tokens][D/2 bytes]: along a token's row every 8 consecutive head-dim elements
 *     form one little-endian 32-bit word, in which element e (0..7) occupies the 4 bits
 *     from bit 4 * ((e >> 1) + 4 * (e & 1)): even elements in the low 16 bits, odd ones
 *     in the high 16 bits.
 *   V [D/2 row pairs][16 bytes]: row pair p holds head-dim rows d = 16 (p / 8) + p % 8
 *     (low 4 bits) and d + 8 (high 4 bits); token t sits at byte 4 (t / 4) +
 *     {0, 2, 1, 3}[t % 4] of the pair's 16 bytes.  A token's bytes hold only its codes.
 */
static void int4_place(size_t row_byte0, int e_in_row, size_t* byte, int* shift) {
  int w = e_in_row / 8, e = e_in_row % 8;
#if ORACLE_MUTANT == 14 /* nibbles in plain element order */
  int nib = e;
#else
  int nib = (e >> 1) + 4 * (e & 1);
#endif
  *byte = row_byte0 + 4 * (size_t)w + nib / 2;
  *shift = 4 * (nib % 2);
}
static void int4_k_place(int page, int h, int off, int d, int Hkv, int P, int D, size_t* byte,
                         int* shift) {
  size_t blk = ((size_t)page * Hkv + h) * (size_t)P * D / 2;
  int4_place(blk + (size_t)off * D / 2, d, byte, shift);
}
static void int4_v_place(int page, int h, int off, int d, int Hkv, int P, int D, size_t* byte,
                         int* shift) {
  static const int tpos[4] = {0, 2, 1, 3};
  size_t blk = ((size_t)page * Hkv + h) * (size_t)P * D / 2;
#if ORACLE_MUTANT == 15 /* row pairs (d, d + 1) instead of (d, d + 8) */
  int pair = d / 2, high = d % 2;
#else
  int pair = 8 * (d / 16) + d % 8, high = (d % 16) >= 8;
#endif
  *byte = blk + (size_t)pair * P + 4 * (off / 4) + tpos[off % 4];
  *shift = 4 * high;
}


static size_t k_index(int kv_dtype, int page, int h, int off, int d, int Hkv, int P, int D) {
  size_t blk = ((size_t)page * Hkv + h) * (size_t)P * D;
  if (kv_dtype == ODT_BF16)
    return blk + ((size_t)(off / 8) * (D / 8) + d / 8) * 64 + (off % 8) * 8 + d % 8;
  return blk + (size_t)off * D + d;
}
static size_t v_index(int kv_dtype, int page, int h, int off, int d, int Hkv, int P, int D) {
  size_t blk = ((size_t)page * Hkv + h) * (size_t)P * D;
#if ORACLE_MUTANT == 3 /* V block not transposed */
  (void)kv_dtype;
  return blk + (size_t)off * D + d;
#else
  if (kv_dtype == ODT_BF16)
    return blk + ((size_t)(d / 8) * (P / 8) + off / 8) * 64 + (d % 8) * 8 + off % 8;
  return blk + (size_t)d * P + off;
#endif
}
static size_t s_index(int page, int h, int off, int Hkv, int P) {
  return ((size_t)page * Hkv + h) * P + off;
}

/* Stored K or V element as a double (after dequantisation). */
static double cache_value(const void* cache, const float* scales, int kv_dtype, int is_v,
                          int page, int h, int off, int d, int Hkv, int P, int D) {
  if (kv_dtype == ODT_INT4) {
    size_t byte;
    int shift;
    if (is_v) int4_v_place(page, h, off, d, Hkv, P, D, &byte, &shift);
    else int4_k_place(page, h, off, d, Hkv, P, D, &byte, &shift);
    int c = (((const uint8_t*)cache)[byte] >> shift) & 15;
    if (c >= 8) c -= 16;
    return (double)c * (double)scales[s_index(page, h, off, Hkv, P)];
  }
  size_t i = is_v ? v_index(kv_dtype, page, h, off, d, Hkv, P, D)
                  : k_index(kv_dtype, page, h, off, d, Hkv, P, D);
  if (kv_dtype == ODT_INT8) {
    /* stored in offset binary: the byte holds code + 128 */
#if ORACLE_MUTANT == 16 /* the byte read as a two's-complement code */
    int c = ((const int8_t*)cache)[i];
#else
    int c = (int)((const uint8_t*)cache)[i] - 128;
#endif
    return (double)c * (double)scales[s_index(page, h, off, Hkv, P)];
  }
  if (kv_dtype == ODT_FP8) {
    uint8_t c = ((const uint8_t*)cache)[i];
    return oracle_e4m3_value(c) * (double)scales[s_index(page, h, off, Hkv, P)];
  }
  return read_real(cache, kv_dtype, i);
}

/* ---------------------------------------------------------------- KV append */

/*
 * Write the new tokens' K and V rows into their slots.  Token i goes to
 * slot = slot_mapping[i] (page = slot / P, off = slot % P) for every kv head;
 * slot < 0 means "skip this token" (padding).  The source rows are float32 or
 * bfloat16 [T][Hkv][D].  FP32 cache: stored as the float value; BF16 cache: rounded to
 * nearest even; INT8, FP8 and INT4 caches: quantised per (token, head) with the
 * quantisers above (INT4 codes written into their 4 bits, the rest of the byte kept).
 * Returns the number of tokens whose slot was >= num_pages * P (those are skipped).
 */
int oracle_append(int kv_dtype, int num_pages, int P, int Hkv, int D, void* k_cache,
                  void* v_cache, float* k_scale, float* v_scale, const void* k_new,
                  const void* v_new, int new_dtype, const int32_t* slot_mapping, int T) {
  int bad = 0;
  float* row = (float*)malloc(sizeof(float) * (size_t)D);
  int8_t* codes = (int8_t*)malloc((size_t)D);
  for (int i = 0; i < T; ++i) {
    int slot = slot_mapping[i];
    if (slot < 0) continue;
    if ((long long)slot >= (long long)num_pages * P) { ++bad; continue; }
    int page = slot / P, off = slot % P;
    for (int h = 0; h < Hkv; ++h) {
      for (int is_v = 0; is_v < 2; ++is_v) {
        const void* src = is_v ? v_new : k_new;
        void* dst = is_v ? v_cache : k_cache;
        for (int d = 0; d < D; ++d)
          row[d] = read_real_f(src, new_dtype, ((size_t)i * Hkv + h) * D + d);
        if (kv_dtype == ODT_INT8 || kv_dtype == ODT_FP8) {
          float s;
          if (kv_dtype == ODT_INT8) oracle_quantize_row_int8(row, D, codes, &s);
          else oracle_quantize_row_fp8(row, D, (uint8_t*)codes, &s);
          for (int d = 0; d < D; ++d) {
            size_t j = is_v ? v_index(kv_dtype, page, h, off, d, Hkv, P, D)
                            : k_index(kv_dtype, page, h, off, d, Hkv, P, D);
            /* INT8 codes in offset binary (code + 128); E4M3 codes as they are */
            ((uint8_t*)dst)[j] = kv_dtype == ODT_INT8 ? (uint8_t)(codes[d] + 128)
                                                     : (uint8_t)codes[d];
          }
          (is_v ? v_scale : k_scale)[s_index(page, h, off, Hkv, P)] = s;
        } else if (kv_dtype == ODT_INT4) {
          float s;
          oracle_quantize_row_int4(row, D, codes, &s);
          for (int d = 0; d < D; ++d) {
            size_t byte;
            int shift;
            if (is_v) int4_v_place(page, h, off, d, Hkv, P, D, &byte, &shift);
            else int4_k_place(page, h, off, d, Hkv, P, D, &byte, &shift);
            uint8_t* bp = (uint8_t*)dst + byte;
            *bp = (uint8_t)((*bp & ~(15 << shift)) | ((codes[d] & 15) << shift));
          }
          (is_v ? v_scale : k_scale)[s_index(page, h, off, Hkv, P)] = s;
        } else {
          for (int d = 0; d < D; ++d) {
            size_t j = is_v ? v_index(kv_dtype, page, h, off, d, Hkv, P, D)
                            : k_index(kv_dtype, page, h, off, d, Hkv, P, D);
            if (kv_dtype == ODT_BF16) ((uint16_t*)dst)[j] = oracle_f32_to_bf16(row[d]);
            else ((float*)dst)[j] = row[d];
          }
        }
      }
    }
  }
  free(row);
  free(codes);
  return bad;
}

/* ---------------------------------------------------------------- rotary embedding */

/*
 * Rotary position embedding ("tinyloop Current Status", model architecture support
 * table: RoPE in all forward paths, configurable theta).  The pages give no formula;
 * the reading taken is the half-split form of the Llama / Qwen families: element i and
 * element i + D/2 form a pair rotated by the angle
 *     a_i = pos * theta^(-2i/D),   i = 0 .. D/2 - 1,
 *     y_i = x_i cos a_i - x_{i+D/2} sin a_i,   y_{i+D/2} = x_{i+D/2} cos a_i + x_i sin a_i.
 * Two precisions: queries in double (the definition), and keys that are about to be
 * stored in float with a fixed operation order (angle in double, cos and sin rounded to
 * float, then one float product and one fused multiply-add per output), because the
 * stored bits (BF16 rounding, INT8 codes) are decided by that float arithmetic.
 */
static double rope_angle(int i, int D, int pos, double theta) {
#if ORACLE_MUTANT == 10 /* rotation the wrong way */
  return -(double)pos * pow(theta, -2.0 * (double)i / (double)D);
#else
  return (double)pos * pow(theta, -2.0 * (double)i / (double)D);
#endif
}

static int rope_partner(int i, int D) {
#if ORACLE_MUTANT == 9 /* adjacent pairs (2i, 2i+1) instead of (i, i + D/2) */
  (void)D;
  return 2 * i + 1;
#else
  return i + D / 2;
#endif
}
static int rope_first(int i) {
#if ORACLE_MUTANT == 9
  return 2 * i;
#else
  return i;
#endif
}

void oracle_rope_f64(const double* x, double* y, int D, int pos, double theta) {
  for (int i = 0; i < D / 2; ++i) {
    const double a = rope_angle(i, D, pos, theta), c = cos(a), s = sin(a);
    const int u = rope_first(i), v = rope_partner(i, D);
    y[u] = x[u] * c - x[v] * s;
    y[v] = x[v] * c + x[u] * s;
  }
}

void oracle_rope_f32(const float* x, float* y, int D, int pos, double theta) {
  for (int i = 0; i < D / 2; ++i) {
    const double a = rope_angle(i, D, pos, theta);
    const float c = (float)cos(a), s = (float)sin(a);
    const int u = rope_first(i), v = rope_partner(i, D);
    const float t = x[v] * s, w = x[u] * s;
    y[u] = fmaf(x[u], c, -t);
    y[v] = fmaf(x[v], c, w);
  }
}

/* ---------------------------------------------------------------- attention core */

/*
 * Softmax-weighted sum for one query vector q (length D, already in double) over the
 * logical tokens first_key..n_keys-1 of sequence b, kv head g.  Logical token t lives in
 * physical page block_table[t / P] at offset t % P; no other table entry is read.
 */
static void attend_one(const double* q, int first_key, int n_keys,
                       const int32_t* block_table, int g,
                       const void* k_cache, const void* v_cache, const float* k_scale,
                       const float* v_scale, int kv_dtype, int Hkv, int P, int D,
                       double scale, double* scores, double* out) {
  for (int d = 0; d < D; ++d) out[d] = 0.0;
  if (n_keys <= first_key) return;
  double m = -INFINITY;
  for (int t = first_key; t < n_keys; ++t) {
#if ORACLE_MUTANT == 8 /* pages taken in physical instead of logical order */
    int page = (int)(t / P), off = t % P;
    (void)block_table;
#else
    int page = block_table[t / P], off = t % P;
#endif
    double dot = 0.0;
    for (int d = 0; d < D; ++d)
      dot += q[d] * cache_value(k_cache, k_scale, kv_dtype, 0, page, g, off, d, Hkv, P, D);
#if ORACLE_MUTANT == 4 /* scale dropped */
    scores[t] = dot;
#else
    scores[t] = scale * dot;
#endif
    if (scores[t] > m) m = scores[t];
  }
  double denom = 0.0;
#if ORACLE_MUTANT == 7 /* no max subtraction */
  m = 0.0;
#endif
  for (int t = first_key; t < n_keys; ++t) {
    scores[t] = exp(scores[t] - m);
    denom += scores[t];
  }
  for (int t = first_key; t < n_keys; ++t) {
    int page = block_table[t / P], off = t % P;
    double w = scores[t] / denom;
    for (int d = 0; d < D; ++d)
      out[d] += w * cache_value(v_cache, v_scale, kv_dtype, 1, page, g, off, d, Hkv, P, D);
  }
}

/*
 * Sliding window ("tinyloop Current Status", KV cache modes table: a cache window bounds
 * the KV storage).  Reading: with window W > 0 the query at position pos attends to the
 * keys at positions pos - W + 1 .. pos (the W most recent, its own included); W = 0 (or
 * a window at least as long as the context) is plain causal attention.  Pages wholly
 * before the window are never read, so their table entries may hold anything.
 */
static int window_first_key(int pos, int window) {
  if (window <= 0) return 0;
#if ORACLE_MUTANT == 11 /* window one key short */
  int lo = pos - window + 2;
#else
  int lo = pos - window + 1;
#endif
  return lo > 0 ? lo : 0;
}

/*
 * Batched decode: one query token per sequence.  q is [B][Hq][D] (float32 or
 * bfloat16), out is [B][Hq][D] doubles.  Sequence b attends over its first
 * context_lens[b] logical tokens (the current token included).  GQA: query head h
 * reads kv head h / (Hq / Hkv).  A sequence with context length 0 gets a zero row.
 * With window > 0 it attends to the last `window` of them only (window_first_key).
 * Sequences for which context_lens[b] is negative or above max_blocks * P, or whose
 * block table holds a page outside [0, num_pages) among the pages it reads, get NaN
 * rows; the return value counts them.
 */
int oracle_decode(int kv_dtype, int num_pages, int P, int Hkv, int D, const void* k_cache,
                  const void* v_cache, const float* k_scale, const float* v_scale,
                  const void* q, int q_dtype, int B, int Hq, const int32_t* block_tables,
                  int max_blocks, const int32_t* context_lens, double scale, int window,
                  double* out, int b_begin, int b_end) {
  int G = Hq / Hkv, bad = 0;
  int max_len = max_blocks * P;
  double* qd = (double*)malloc(sizeof(double) * (size_t)D);
  double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  if (b_end > B) b_end = B;
  for (int b = b_begin; b < b_end; ++b) {
    int L = context_lens[b];
    const int32_t* bt = block_tables + (size_t)b * max_blocks;
    int ok = (L >= 0 && L <= max_len);
    int lo = ok ? window_first_key(L - 1, window) : 0;
    for (int j = lo / P; ok && j < (L + P - 1) / P; ++j)
      if (bt[j] < 0 || bt[j] >= num_pages) ok = 0;
    for (int h = 0; h < Hq; ++h) {
      double* o = out + ((size_t)b * Hq + h) * D;
      if (!ok) {
        for (int d = 0; d < D; ++d) o[d] = NAN;
        continue;
      }
      for (int d = 0; d < D; ++d) qd[d] = read_real(q, q_dtype, ((size_t)b * Hq + h) * D + d);
#if ORACLE_MUTANT == 5 /* GQA heads interleaved instead of grouped */
      int g = h % Hkv;
#else
      int g = h / G;
#endif
      attend_one(qd, lo, L, bt, g, k_cache, v_cache, k_scale, v_scale, kv_dtype, Hkv, P, D,
                 scale, scores, o);
    }
    if (!ok) ++bad;
  }
  free(qd);
  free(scores);
  return bad;
}

/*
 * One decode step: for each sequence b whose slot_mapping[b] is >= 0, the new token's
 * key row k_new[b] ([B][Hkv][D], float32 or bfloat16) is rotated (float form) at
 * positions[b] and stored with v_new[b] at slot_mapping[b] exactly as oracle_append
 * stores rows; then every query row q[b] is rotated (double form) at positions[b] and
 * attends over context_lens[b] tokens as in oracle_decode.  positions == NULL means no
 * rotation.  The new token must sit at logical position context_lens[b] - 1: a slot that
 * is not that position's slot (or a length below 1) gives NaN rows for b and nothing is
 * stored.  slot_mapping[b] < 0: nothing is stored and b attends over the cache as is.
 * window as in oracle_decode.  Sequences b_begin .. b_end - 1 only.  Returns the number
 * of sequences given NaN rows.
 */
int oracle_decode_step(int kv_dtype, int num_pages, int P, int Hkv, int D, void* k_cache,
                       void* v_cache, float* k_scale, float* v_scale, const void* q,
                       int q_dtype, const void* k_new, const void* v_new, int new_dtype,
                       const int32_t* slot_mapping, const int32_t* positions, double theta,
                       int B, int Hq, const int32_t* block_tables, int max_blocks,
                       const int32_t* context_lens, double scale, int window, double* out,
                       int b_begin, int b_end) {
  int G = Hq / Hkv, bad = 0;
  int max_len = max_blocks * P;
  double* qd = (double*)malloc(sizeof(double) * (size_t)D);
  double* qr = (double*)malloc(sizeof(double) * (size_t)D);
  double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  float* xk = (float*)malloc(sizeof(float) * (size_t)Hkv * D);
  float* xv = (float*)malloc(sizeof(float) * (size_t)Hkv * D);
  float* row = (float*)malloc(sizeof(float) * (size_t)D);
  if (b_end > B) b_end = B;
  for (int b = b_begin; b < b_end; ++b) {
    int L = context_lens[b];
    const int32_t* bt = block_tables + (size_t)b * max_blocks;
    int ok = (L >= 0 && L <= max_len);
    int lo = ok ? window_first_key(L - 1, window) : 0;
    for (int j = lo / P; ok && j < (L + P - 1) / P; ++j)
      if (bt[j] < 0 || bt[j] >= num_pages) ok = 0;
    const int slot = slot_mapping[b];
    if (ok && slot >= 0 && (L < 1 || slot != bt[(L - 1) / P] * P + (L - 1) % P)) ok = 0;
    const int pos = positions ? positions[b] : 0;
    if (ok && slot >= 0) {
      /* the new row, rotated in float, stored through the append definition */
      for (int h = 0; h < Hkv; ++h) {
        for (int d = 0; d < D; ++d) row[d] = read_real_f(k_new, new_dtype, ((size_t)b * Hkv + h) * D + d);
        if (positions) oracle_rope_f32(row, xk + (size_t)h * D, D, pos, theta);
        else for (int d = 0; d < D; ++d) xk[(size_t)h * D + d] = row[d];
        for (int d = 0; d < D; ++d) xv[(size_t)h * D + d] = read_real_f(v_new, new_dtype, ((size_t)b * Hkv + h) * D + d);
      }
      int32_t one_slot = slot;
      oracle_append(kv_dtype, num_pages, P, Hkv, D, k_cache, v_cache, k_scale, v_scale, xk,
                    xv, 0 /* float32 rows */, &one_slot, 1);
    }
    for (int h = 0; h < Hq; ++h) {
      double* o = out + ((size_t)b * Hq + h) * D;
      if (!ok) {
        for (int d = 0; d < D; ++d) o[d] = NAN;
        continue;
      }
      for (int d = 0; d < D; ++d) qd[d] = read_real(q, q_dtype, ((size_t)b * Hq + h) * D + d);
      if (positions) oracle_rope_f64(qd, qr, D, pos, theta);
      else for (int d = 0; d < D; ++d) qr[d] = qd[d];
      attend_one(qr, lo, L, bt, h / G, k_cache, v_cache, k_scale, v_scale, kv_dtype, Hkv, P,
                 D, scale, scores, o);
    }
    if (!ok) ++bad;
  }
  free(qd);
  free(qr);
  free(scores);
  free(xk);
  free(xv);
  free(row);
  return bad;
}

/*
 * Chunked prefill: sequence b owns query rows q_start_loc[b] .. q_start_loc[b+1]-1 of q
 * ([total_q][Hq][D]).  Its context_lens[b] counts every cached token including the
 * chunk, so query row i of the chunk (Lq = chunk length) sits at absolute position
 * p_i = context_lens[b] - Lq + i and attends to the logical tokens 0..p_i (the causal
 * mask is inclusive of its own position); with window > 0, to p_i - window + 1 .. p_i
 * only (window_first_key).  out is [total_q][Hq][D] doubles.  Sequences with an
 * inconsistent chunk (Lq < 0 or Lq > context length) or a bad page among those their
 * rows read get NaN rows; the return value counts them.
 */
int oracle_prefill(int kv_dtype, int num_pages, int P, int Hkv, int D, const void* k_cache,
                   const void* v_cache, const float* k_scale, const float* v_scale,
                   const void* q, int q_dtype, int B, int Hq, const int32_t* q_start_loc,
                   const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                   double scale, int window, double* out, int b_begin, int b_end) {
  int G = Hq / Hkv, bad = 0;
  int max_len = max_blocks * P;
  double* qd = (double*)malloc(sizeof(double) * (size_t)D);
  double* scores = (double*)malloc(sizeof(double) * (size_t)(max_len > 0 ? max_len : 1));
  if (b_end > B) b_end = B;
  for (int b = b_begin; b < b_end; ++b) {
    int L = context_lens[b];
    int q0 = q_start_loc[b], Lq = q_start_loc[b + 1] - q_start_loc[b];
    const int32_t* bt = block_tables + (size_t)b * max_blocks;
    int ok = (L >= 0 && L <= max_len && Lq >= 0 && Lq <= L);
    /* the chunk's first row has the lowest window start */
    int lo0 = ok ? window_first_key(L - Lq, window) : 0;
    for (int j = lo0 / P; ok && j < (L + P - 1) / P; ++j)
      if (bt[j] < 0 || bt[j] >= num_pages) ok = 0;
    if (!ok) ++bad;
    for (int i = 0; i < (Lq > 0 ? Lq : 0); ++i) {
      int pos = L - Lq + i;
      for (int h = 0; h < Hq; ++h) {
        size_t row = ((size_t)(q0 + i) * Hq + h) * D;
        double* o = out + row;
        if (!ok) {
          for (int d = 0; d < D; ++d) o[d] = NAN;
          continue;
        }
        for (int d = 0; d < D; ++d) qd[d] = read_real(q, q_dtype, row + d);
#if ORACLE_MUTANT == 6 /* causal mask excludes the diagonal */
        int n_keys = pos;
#else
        int n_keys = pos + 1;
#endif
#if ORACLE_MUTANT == 12 /* every row of the chunk takes the window of its last row */
        int first = window_first_key(L - 1, window);
#else
        int first = window_first_key(pos, window);
#endif
        attend_one(qd, first, n_keys, bt, h / G, k_cache, v_cache, k_scale, v_scale,
                   kv_dtype, Hkv, P, D, scale, scores, o);
      }
    }
  }
  free(qd);
  free(scores);
  return bad;
}
