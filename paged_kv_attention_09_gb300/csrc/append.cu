// append.cu — KV append: scatter new tokens' K/V rows into their cache slots.
//
// "Tiny-LLM-Inference Project_Status" (feature list: paged KV cache; dtype contract:
// FP32 or BF16 KV), "tinyloop Current Status" (KV cache modes table: INT8 and INT4 KV
// caches) and the TinyInfer review (item 2: INT8 or FP8 KV cache).  One warp per (token,
// kv head) writes both the K row and the V column of that slot; quantised rows go through
// the shared quantisers (kvrow.cuh).  INT4 K rows are written as whole 32-bit words and
// INT4 V bytes belong to one token each, so tokens of one call never share a byte.
#include <cuda_bf16.h>

#include "internal.h"
#include "kvrow.cuh"

namespace pkv {
namespace {

constexpr int kWarps = 8;

template <int NEW_DT>
__device__ __forceinline__ float load_src(const void* p, size_t i) {
  if constexpr (NEW_DT == kBF16) {
    return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  } else {
    return static_cast<const float*>(p)[i];
  }
}

template <int KV_DT, int NEW_DT, int D>
__global__ void __launch_bounds__(kWarps * 32)
    append_kernel(void* __restrict__ k_cache, void* __restrict__ v_cache,
                  float* __restrict__ k_scale, float* __restrict__ v_scale,
                  const void* __restrict__ k_new, const void* __restrict__ v_new,
                  const int32_t* __restrict__ slots, int T, int Hkv, int num_pages,
                  int32_t* dev_status) {
  constexpr int E = D / 32;  // elements per lane
  const int lane = threadIdx.x & 31;
  const long long item = static_cast<long long>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
  if (item >= static_cast<long long>(T) * Hkv) return;
  const int tok = static_cast<int>(item / Hkv), h = static_cast<int>(item % Hkv);
  const int slot = slots[tok];
  if (slot < 0) return;
  if (slot >= num_pages * kPage) {
    if (lane == 0 && dev_status) atomicOr(dev_status, 0x4 /*PKV_DEV_BAD_SLOT*/);
    return;
  }
  const int page = slot / kPage, off = slot % kPage;
  const size_t src_row = (static_cast<size_t>(tok) * Hkv + h) * D;
  const size_t blk = static_cast<size_t>(page) * Hkv + h;  // (page, head) block index
  const size_t k_row = (blk * kPage + off) * D;            // K: [P][D] inside the block
  const size_t v_base = blk * D * kPage + off;             // V: [D][P] inside the block
  // (INT4: D/2 bytes per K row and D/2 row pairs of 16 bytes per V block)

#pragma unroll
  for (int which = 0; which < 2; ++which) {
    const void* src = which ? v_new : k_new;
    float x[E];
#pragma unroll
    for (int e = 0; e < E; ++e) x[e] = load_src<NEW_DT>(src, src_row + lane * E + e);

    if constexpr (KV_DT == kINT4) {
      int8_t code[E];
      const float s = quantize_row_int4<E>(x, code);
      uint8_t* dst = static_cast<uint8_t*>(which ? v_cache : k_cache) + blk * kPage * (D / 2);
      if (which == 0) {
        const uint32_t w = int4_k_word<E>(code, lane);
        if ((lane & (8 / E - 1)) == 0)
          reinterpret_cast<uint32_t*>(dst + off * (D / 2))[lane * E / 8] = w;
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int d = lane * E + e;
          const uint8_t b = int4_v_byte<E>(code, e);
          if ((d & 15) < 8) dst[int4_v_pair(d) * kPage + int4_v_tpos(off)] = b;
        }
      }
      if (lane == 0) (which ? v_scale : k_scale)[blk * kPage + off] = s;
    } else if constexpr (KV_DT == kINT8 || KV_DT == kFP8) {
      uint8_t code[E];
      float s;
      if constexpr (KV_DT == kINT8) {
        int8_t c8[E];
        s = quantize_row_int8<E>(x, c8);
#pragma unroll
        for (int e = 0; e < E; ++e) code[e] = int8_stored(c8[e]);
      } else {
        s = quantize_row_fp8<E>(x, code);
      }
      uint8_t* dst = static_cast<uint8_t*>(which ? v_cache : k_cache);
      if (which == 0) {
#pragma unroll
        for (int e = 0; e < E; ++e) dst[k_row + lane * E + e] = code[e];
      } else {
#pragma unroll
        for (int e = 0; e < E; ++e) dst[v_base + static_cast<size_t>(lane * E + e) * kPage] = code[e];
      }
      if (lane == 0) (which ? v_scale : k_scale)[blk * kPage + off] = s;
    } else if constexpr (KV_DT == kBF16) {
      // tensor-core tile order inside the block (see bf16_k_off / bf16_v_off)
      uint8_t* blkp = static_cast<uint8_t*>(which ? v_cache : k_cache) + blk * kPage * D * 2;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const __nv_bfloat16 b = __float2bfloat16_rn(x[e]);
        const int d = lane * E + e;
        const int off_b = which == 0 ? bf16_k_off(off, d, D) : bf16_v_off(d, off);
        *reinterpret_cast<__nv_bfloat16*>(blkp + off_b) = b;
      }
    } else {
      float* dst = static_cast<float*>(which ? v_cache : k_cache);
#pragma unroll
      for (int e = 0; e < E; ++e) {
        if (which == 0) dst[k_row + lane * E + e] = x[e];
        else dst[v_base + static_cast<size_t>(lane * E + e) * kPage] = x[e];
      }
    }
  }
}

template <int KV_DT, int NEW_DT>
cudaError_t launch_t(int D, dim3 grid, cudaStream_t st, void* k, void* v, float* ks,
                     float* vs, const void* kn, const void* vn, const int32_t* slots, int T,
                     int Hkv, int NP, int32_t* dev_status) {
  if (D == 64)
    append_kernel<KV_DT, NEW_DT, 64><<<grid, kWarps * 32, 0, st>>>(k, v, ks, vs, kn, vn, slots,
                                                                   T, Hkv, NP, dev_status);
  else
    append_kernel<KV_DT, NEW_DT, 128><<<grid, kWarps * 32, 0, st>>>(k, v, ks, vs, kn, vn, slots,
                                                                    T, Hkv, NP, dev_status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const CacheView& c, void* k_cache, void* v_cache, float* ks,
                          float* vs, const void* k_new, const void* v_new, int new_dtype,
                          const int32_t* slots, int T, int32_t* dev_status, cudaStream_t st) {
  const long long items = static_cast<long long>(T) * c.Hkv;
  const dim3 grid(static_cast<unsigned>((items + kWarps - 1) / kWarps));
  const bool nb = new_dtype == kBF16;
  switch (c.dtype) {
    case kF32:
      return nb ? launch_t<kF32, kBF16>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                        slots, T, c.Hkv, c.num_pages, dev_status)
                : launch_t<kF32, kF32>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                       slots, T, c.Hkv, c.num_pages, dev_status);
    case kBF16:
      return nb ? launch_t<kBF16, kBF16>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                         slots, T, c.Hkv, c.num_pages, dev_status)
                : launch_t<kBF16, kF32>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                        slots, T, c.Hkv, c.num_pages, dev_status);
    case kINT8:
      return nb ? launch_t<kINT8, kBF16>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                         slots, T, c.Hkv, c.num_pages, dev_status)
                : launch_t<kINT8, kF32>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                        slots, T, c.Hkv, c.num_pages, dev_status);
    case kFP8:
      return nb ? launch_t<kFP8, kBF16>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                        slots, T, c.Hkv, c.num_pages, dev_status)
                : launch_t<kFP8, kF32>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                       slots, T, c.Hkv, c.num_pages, dev_status);
    case kINT4:
      return nb ? launch_t<kINT4, kBF16>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                         slots, T, c.Hkv, c.num_pages, dev_status)
                : launch_t<kINT4, kF32>(c.D, grid, st, k_cache, v_cache, ks, vs, k_new, v_new,
                                        slots, T, c.Hkv, c.num_pages, dev_status);
    default:
      return cudaErrorInvalidValue;
  }
}

}  // namespace pkv
