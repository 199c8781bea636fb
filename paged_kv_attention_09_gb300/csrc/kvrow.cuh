// kvrow.cuh — one K or V row of a kv head, held by a warp as E = D/32 consecutive values
// per lane, converted to the cache's storage format.  Shared by the append kernel and the
// fused decode step, so that both store bit-identical rows.
//
// "tinyloop Current Status" (KV cache modes table: INT8 KV cache): rows are quantised
// symmetrically, s = max|x| / 127 with IEEE division and code = clamp(rint(x / s), -127,
// 127) with round-half-to-even, so the stored codes are reproducible by any IEEE float
// implementation.
#pragma once
#include <cstdint>

namespace pkv {

// Returns the row's scale and writes its codes; every lane of the warp must call it.
template <int E>
__device__ __forceinline__ float quantize_row_int8(const float (&x)[E], int8_t (&code)[E]) {
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < E; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.0f);
#pragma unroll
  for (int e = 0; e < E; ++e) {
    float r = 0.f;
    if (s != 0.f) r = fminf(fmaxf(rintf(__fdiv_rn(x[e], s)), -127.f), 127.f);
    code[e] = static_cast<int8_t>(static_cast<int>(r));
  }
  return s;
}

}  // namespace pkv
