// noalloc.cu — decode attention for callers that cannot provide device scratch.
//
// Some programs that embed this library cannot call cudaMalloc or hand it a buffer:
// plugins loaded into an engine whose memory pool already owns all of the device's
// memory and exposes no allocation hook, or steady-state loops whose owners forbid any
// allocation after start-up.  pkv_decode_attn_noalloc serves them: its split-K scratch
// lives in a fixed array in the library's own device memory, reserved when the library
// is loaded, so the call needs nothing from the caller but inputs and outputs.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "internal.h"
#include "pkv.h"

// The scratch every call shares.  Every GPU that loads the library holds these bytes
// until the process exits.  Zero at load; each call clears the part that must start at
// zero (the merge counters) before its kernel runs.
static __device__ __align__(256) unsigned char g_decode_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;
void* g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

// Device address of the scratch array on `device` (the current device).  In host code
// the array's name is only a host-side stand-in, so the address must be asked for once
// per device, with that device current.
pkv_status scratch_address(int device, void** out) {
  if (device < 0 || device >= kMaxDevices) return PKV_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PKV_ERR_DEVICE;
    g_scratch_ptr[device] = p;
  }
  *out = g_scratch_ptr[device];
  return PKV_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" pkv_status pkv_decode_attn_noalloc(const pkv_cache* cache, const void* q,
                                              int32_t q_dtype, int32_t num_seqs,
                                              int32_t num_q_heads, const int32_t* block_tables,
                                              int32_t max_blocks_per_seq,
                                              const int32_t* context_lens, float scale,
                                              float* out, int32_t* dev_status, void* stream) {
  if (!cache || !cache->k_cache || !cache->v_cache) return PKV_ERR_NULL;
  if (cache->kv_dtype < PKV_F32 || cache->kv_dtype > PKV_INT4) return PKV_ERR_DTYPE;
  if (cache->page_size != 16) return PKV_ERR_PAGE_SIZE;
  if (cache->num_pages < 1 || cache->num_kv_heads < 1 || cache->window < 0) return PKV_ERR_SHAPE;
  if (cache->head_dim != 64 && cache->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  const bool coded = pkv::quantised(cache->kv_dtype);
  if (coded && (!cache->k_scale || !cache->v_scale)) return PKV_ERR_NULL;
  if (!aligned16(cache->k_cache) || !aligned16(cache->v_cache)) return PKV_ERR_ALIGN;
  if (coded && (!aligned16(cache->k_scale) || !aligned16(cache->v_scale))) return PKV_ERR_ALIGN;
  if (num_seqs < 0 || num_q_heads < 1 || max_blocks_per_seq < 1) return PKV_ERR_SHAPE;
  if (num_q_heads % cache->num_kv_heads != 0) return PKV_ERR_SHAPE;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;
  if (q_dtype != PKV_F32 && q_dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !block_tables || !context_lens || !out) return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || !aligned4(block_tables) || !aligned4(context_lens))
    return PKV_ERR_ALIGN;
  if (dev_status && !aligned4(dev_status)) return PKV_ERR_ALIGN;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_DEVICE;
  const pkv::CacheView view{cache->k_cache,  cache->v_cache,     cache->k_scale,
                            cache->v_scale,  cache->num_pages,   cache->num_kv_heads,
                            cache->head_dim, cache->kv_dtype,   cache->window};
  pkv::DecodePlan plan{};
  if (!pkv::plan_decode(view, num_seqs, num_q_heads, max_blocks_per_seq, q_dtype, dev,
                        pkv::decode_chunk_override(), &plan))
    return PKV_ERR_DEVICE;
  if (static_cast<long long>(cache->num_kv_heads) * plan.head_groups > 65535)
    return PKV_ERR_UNSUPPORTED;
  if (plan.ws_bytes > sizeof(g_decode_scratch)) return PKV_ERR_WORKSPACE;  // beyond the fixed maximum

  void* scratch = nullptr;
  pkv_status s = scratch_address(dev, &scratch);
  if (s != PKV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (plan.n_splits > 1) {
    // the merge counters lead the scratch and must start at zero
    const size_t counters = static_cast<size_t>(num_seqs) * cache->num_kv_heads * plan.head_groups * 4;
    if (cudaMemsetAsync(scratch, 0, counters, st) != cudaSuccess) return PKV_ERR_LAUNCH;
  }
  pkv::DecodeArgs a{};
  a.c = view;
  a.q = q;
  a.q_dtype = q_dtype;
  a.B = num_seqs;
  a.Hq = num_q_heads;
  a.MB = max_blocks_per_seq;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.scale = scale;
  a.out = out;
  a.ws = scratch;
  a.dev_status = dev_status;
  return pkv::launch_decode(a, plan, st) == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}
