// kvrow.cuh — one K or V row of a kv head, held by a warp as E = D/32 consecutive values
// per lane, converted to the cache's storage format.  Shared by the append kernel and the
// fused decode step, so that both store bit-identical rows.
//
// Quantised rows ("tinyloop Current Status", KV cache modes table: INT8 and INT4 KV
// caches; the TinyInfer review, item 2: INT8 or FP8 KV cache) are symmetric per (token,
// kv head) with an FP32 scale s = max|x| / R computed by IEEE division, R = 127 (INT8),
// 448 (FP8 E4M3) or 7 (INT4); the code is x / s (IEEE division) rounded to nearest with
// ties to even: clamped to [-R, R] for the integer formats, saturating at 448 for E4M3.
// The stored codes are therefore reproducible by any IEEE float implementation.
#pragma once
#include <cuda_fp8.h>

#include <cstdint>

namespace pkv {

// max|x| over the warp's row, then s = amax / range; every lane must call it.
template <int E>
__device__ __forceinline__ float row_scale(const float (&x)[E], float range) {
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  return __fdiv_rn(amax, range);
}

// The stored byte of an INT8 code: offset binary, code + 128 (so that the decode kernel
// widens a code to the f16 value 1024 + byte with a byte permute alone).
__device__ __forceinline__ uint8_t int8_stored(int8_t code) {
  return static_cast<uint8_t>(static_cast<uint8_t>(code) ^ 0x80u);
}

// Returns the row's scale and writes its codes; every lane of the warp must call it.
template <int E>
__device__ __forceinline__ float quantize_row_int8(const float (&x)[E], int8_t (&code)[E]) {
  const float s = row_scale<E>(x, 127.0f);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float r = 0.f;
    if (s != 0.f) r = fminf(fmaxf(rintf(__fdiv_rn(x[e], s)), -127.f), 127.f);
    code[e] = static_cast<int8_t>(static_cast<int>(r));
  }
  return s;
}

template <int E>
__device__ __forceinline__ float quantize_row_int4(const float (&x)[E], int8_t (&code)[E]) {
  const float s = row_scale<E>(x, 7.0f);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float r = 0.f;
    if (s != 0.f) r = fminf(fmaxf(rintf(__fdiv_rn(x[e], s)), -7.f), 7.f);
    code[e] = static_cast<int8_t>(static_cast<int>(r));
  }
  return s;
}

// E4M3 codes by the hardware conversion (round to nearest even, saturating to 448).
template <int E>
__device__ __forceinline__ float quantize_row_fp8(const float (&x)[E], uint8_t (&code)[E]) {
  const float s = row_scale<E>(x, 448.0f);
#pragma unroll
  for (int e = 0; e < E; ++e)
    code[e] = s != 0.f ? static_cast<uint8_t>(__nv_cvt_float_to_fp8(__fdiv_rn(x[e], s),
                                                                    __NV_SATFINITE, __NV_E4M3))
                       : 0;
  return s;
}

// ---- INT4 storage (two 4-bit two's-complement codes per byte)
// K rows: every 8 consecutive head-dim elements form a little-endian 32-bit word; element
// e of the word sits at bit 4 * ((e >> 1) + 4 * (e & 1)) (even elements in the low half).
__device__ __forceinline__ int int4_k_shift(int e) { return 4 * ((e >> 1) + 4 * (e & 1)); }
// V: row pair p holds head-dim rows 16 (p / 8) + p % 8 (low 4 bits) and that + 8 (high 4
// bits); token t of the page sits at byte 4 (t / 4) + {0, 2, 1, 3}[t % 4] of the pair.
__device__ __forceinline__ int int4_v_tpos(int t) {
  return (t & ~3) | ((t & 1) << 1) | ((t >> 1) & 1);
}
__device__ __forceinline__ int int4_v_pair(int d) { return 8 * (d >> 4) + (d & 7); }

// The K row word covering elements 8 (E lane / 8) .. + 7, complete in every lane of the
// group of 8 / E lanes that hold them.
template <int E>
__device__ __forceinline__ uint32_t int4_k_word(const int8_t (&code)[E], int lane) {
  uint32_t w = 0;
#pragma unroll
  for (int e = 0; e < E; ++e)
    w |= (static_cast<uint32_t>(code[e]) & 15u) << int4_k_shift((lane * E + e) & 7);
#pragma unroll
  for (int o = 1; o < 8 / E; o <<= 1) w |= __shfl_xor_sync(0xffffffffu, w, o);
  return w;
}

// The V byte of element e's row pair, meaningful in the lanes whose element is the low
// row of its pair (head-dim index d with d % 16 < 8); the high row's code comes from the
// lane 8 / E further on.
template <int E>
__device__ __forceinline__ uint8_t int4_v_byte(const int8_t (&code)[E], int e) {
  const int hi = __shfl_down_sync(0xffffffffu, static_cast<int>(code[e]), 8 / E);
  return static_cast<uint8_t>((static_cast<uint32_t>(code[e]) & 15u) |
                              ((static_cast<uint32_t>(hi) & 15u) << 4));
}

}  // namespace pkv
