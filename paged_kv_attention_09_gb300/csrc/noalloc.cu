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

#include "abi.h"
#include "internal.h"
#include "nvtx.h"
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

}  // namespace

extern "C" pkv_status pkv_decode_attn_noalloc_ex(const pkv_cache* cache, const void* q,
                                                 int32_t q_dtype, int32_t num_seqs,
                                                 int32_t num_q_heads,
                                                 const int32_t* block_tables,
                                                 int32_t max_blocks_per_seq,
                                                 const int32_t* context_lens, float scale,
                                                 float* out, const pkv_decode_opts* opts,
                                                 int32_t* dev_status, void* stream) {
  PKV_RANGE("pkv_decode_attn_noalloc");
  // the same checks, in the same order, as pkv_decode_attn
  pkv_status s = pkv::check_decode_call(cache, q, q_dtype, num_seqs, num_q_heads, block_tables,
                                        max_blocks_per_seq, context_lens, out, dev_status);
  if (s != PKV_OK) return s;
  int split = 0;
  if (!pkv::split_pages_of(opts, &split)) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_DEVICE;
  const pkv::CacheView view = pkv::view(cache);
  pkv::DecodePlan plan{};
  if (!pkv::plan_decode(view, num_seqs, num_q_heads, max_blocks_per_seq, q_dtype, dev, split,
                        &plan))
    return PKV_ERR_DEVICE;
  if (static_cast<long long>(cache->num_kv_heads) * plan.head_groups > 65535)
    return PKV_ERR_UNSUPPORTED;
  if (plan.ws_bytes > sizeof(g_decode_scratch)) return PKV_ERR_WORKSPACE;  // beyond the fixed maximum

  void* scratch = nullptr;
  s = scratch_address(dev, &scratch);
  if (s != PKV_OK) return s;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (plan.n_splits > 1) {
    // The merge counters lead the scratch and must start at zero.  A caller's workspace
    // is the caller's to keep zeroed (the kernel leaves its counters at zero), but this
    // array is shared by calls of every shape, and a call that stopped before its merge
    // (a failed launch, a wait that gave up) must not leak counts into the next call.
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

extern "C" pkv_status pkv_decode_attn_noalloc(const pkv_cache* cache, const void* q,
                                              int32_t q_dtype, int32_t num_seqs,
                                              int32_t num_q_heads, const int32_t* block_tables,
                                              int32_t max_blocks_per_seq,
                                              const int32_t* context_lens, float scale,
                                              float* out, int32_t* dev_status, void* stream) {
  return pkv_decode_attn_noalloc_ex(cache, q, q_dtype, num_seqs, num_q_heads, block_tables,
                                    max_blocks_per_seq, context_lens, scale, out, nullptr,
                                    dev_status, stream);
}
