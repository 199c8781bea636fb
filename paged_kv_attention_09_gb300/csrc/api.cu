// api.cu — the extern "C" boundary declared in include/pkv.h: argument validation,
// planning and launches.  Allocates nothing; every buffer belongs to the caller
// ("Tiny-LLM-Inference Project_Status", runtime notes: buffers are preallocated from the
// resolved capacity and an oversized request fails fast instead of reallocating).
#include <cstdint>
#include <cuda_runtime.h>

#include "abi.h"
#include "internal.h"
#include "nvtx.h"
#include "pkv.h"

namespace pkv {

pkv_status check_cache(const pkv_cache* c) {
  if (!c || !c->k_cache || !c->v_cache) return PKV_ERR_NULL;
  if (c->kv_dtype < PKV_F32 || c->kv_dtype > PKV_INT4) return PKV_ERR_DTYPE;
  if (c->page_size != 16) return PKV_ERR_PAGE_SIZE;
  if (c->num_pages < 1 || c->num_kv_heads < 1 || c->head_dim < 1) return PKV_ERR_SHAPE;
  if (c->window < 0) return PKV_ERR_SHAPE;
  if (c->head_dim != 64 && c->head_dim != 128) return PKV_ERR_UNSUPPORTED;
  if (quantised(c->kv_dtype) && (!c->k_scale || !c->v_scale)) return PKV_ERR_NULL;
  if (!aligned16(c->k_cache) || !aligned16(c->v_cache)) return PKV_ERR_ALIGN;
  if (quantised(c->kv_dtype) && (!aligned16(c->k_scale) || !aligned16(c->v_scale)))
    return PKV_ERR_ALIGN;
  // every page block must stay addressable with 32-bit slot numbers
  if (static_cast<long long>(c->num_pages) * c->page_size > 0x7fffffffLL) return PKV_ERR_SHAPE;
  return PKV_OK;
}

pkv_status check_decode_shape(const pkv_cache* c, int32_t num_seqs, int32_t Hq, int32_t MB) {
  if (num_seqs < 0 || Hq < 1 || MB < 1) return PKV_ERR_SHAPE;
  if (Hq % c->num_kv_heads != 0) return PKV_ERR_SHAPE;
  if (num_seqs > 65535) return PKV_ERR_UNSUPPORTED;  // grid.y limit
  // token positions over a whole block-table row stay 32-bit
  if (static_cast<long long>(MB) * c->page_size > 0x7fffffffLL) return PKV_ERR_SHAPE;
  return PKV_OK;
}

pkv_status check_decode_call(const pkv_cache* c, const void* q, int32_t q_dtype,
                             int32_t num_seqs, int32_t num_q_heads, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                             const float* out, const int32_t* dev_status) {
  pkv_status s = check_cache(c);
  if (s != PKV_OK) return s;
  s = check_decode_shape(c, num_seqs, num_q_heads, max_blocks_per_seq);
  if (s != PKV_OK) return s;
  if (q_dtype != PKV_F32 && q_dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !block_tables || !context_lens || !out) return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || !aligned4(block_tables) || !aligned4(context_lens))
    return PKV_ERR_ALIGN;
  if (dev_status && !aligned4(dev_status)) return PKV_ERR_ALIGN;
  return PKV_OK;
}

bool split_pages_of(const pkv_decode_opts* opts, int* pages) {
  *pages = opts ? opts->split_pages : 0;
  return *pages >= 0;
}

bool prefill_opts_of(const pkv_prefill_opts* opts, PrefillOpts* out) {
  out->key_split = opts ? opts->key_split : 0;
  return out->key_split >= 0 && out->key_split <= 3;
}

CacheView view(const pkv_cache* c) {
  return CacheView{c->k_cache, c->v_cache, c->k_scale, c->v_scale,
                   c->num_pages, c->num_kv_heads, c->head_dim, c->kv_dtype, c->window};
}

}  // namespace pkv

namespace {

using pkv::aligned16;
using pkv::aligned4;
using pkv::check_cache;
using pkv::check_decode_shape;
using pkv::view;

pkv_status current_device(int* dev) {
  return cudaGetDevice(dev) == cudaSuccess ? PKV_OK : PKV_ERR_DEVICE;
}

// Plans and launches one decode call (a.step: the fused decode step) after the checks.
pkv_status decode_launch(const pkv_cache* cache, pkv::DecodeArgs& a, int split_pages,
                         size_t workspace_bytes, cudaStream_t st) {
  int dev = 0;
  pkv_status s = current_device(&dev);
  if (s != PKV_OK) return s;
  pkv::DecodePlan plan{};
  if (!pkv::plan_decode(a.c, a.B, a.Hq, a.MB, a.q_dtype, dev, split_pages, &plan, a.step))
    return PKV_ERR_DEVICE;
  if (static_cast<long long>(cache->num_kv_heads) * plan.head_groups > 65535)
    return PKV_ERR_UNSUPPORTED;
  if (plan.ws_bytes > 0) {
    if (!a.ws || workspace_bytes < plan.ws_bytes) return PKV_ERR_WORKSPACE;
    if (!aligned16(a.ws)) return PKV_ERR_ALIGN;
  }
  return pkv::launch_decode(a, plan, st) == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

}  // namespace

extern "C" {

pkv_status pkv_append(const pkv_cache* cache, const void* k_new, const void* v_new,
                      int32_t new_dtype, const int32_t* slot_mapping, int32_t num_tokens,
                      int32_t* dev_status, void* stream) {
  PKV_RANGE("pkv_append");
  pkv_status s = check_cache(cache);
  if (s != PKV_OK) return s;
  if (num_tokens < 0) return PKV_ERR_SHAPE;
  if (new_dtype != PKV_F32 && new_dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (num_tokens == 0) return PKV_OK;
  if (!k_new || !v_new || !slot_mapping) return PKV_ERR_NULL;
  if (!aligned16(k_new) || !aligned16(v_new) || !aligned4(slot_mapping)) return PKV_ERR_ALIGN;
  if (dev_status && !aligned4(dev_status)) return PKV_ERR_ALIGN;
  const cudaError_t e = pkv::launch_append(
      view(cache), cache->k_cache, cache->v_cache, cache->k_scale, cache->v_scale, k_new, v_new,
      new_dtype, slot_mapping, num_tokens, dev_status, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

pkv_status pkv_decode_workspace_size_ex(const pkv_cache* cache, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t max_blocks_per_seq,
                                        const pkv_decode_opts* opts, size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  *bytes = 0;
  pkv_status s = check_cache(cache);
  if (s != PKV_OK) return s;
  s = check_decode_shape(cache, num_seqs, num_q_heads, max_blocks_per_seq);
  if (s != PKV_OK) return s;
  int split = 0;
  if (!pkv::split_pages_of(opts, &split)) return PKV_ERR_SHAPE;
  int dev = 0;
  if ((s = current_device(&dev)) != PKV_OK) return s;
  // one size for both pkv_decode_attn and pkv_decode_step (their plans may differ)
  pkv::DecodePlan plan{}, plan_step{};
  if (!pkv::plan_decode(view(cache), num_seqs, num_q_heads, max_blocks_per_seq, PKV_F32, dev,
                        split, &plan) ||
      !pkv::plan_decode(view(cache), num_seqs, num_q_heads, max_blocks_per_seq, PKV_F32, dev,
                        split, &plan_step, true))
    return PKV_ERR_DEVICE;
  *bytes = plan.ws_bytes > plan_step.ws_bytes ? plan.ws_bytes : plan_step.ws_bytes;
  return PKV_OK;
}

pkv_status pkv_decode_workspace_size(const pkv_cache* cache, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t max_blocks_per_seq,
                                     size_t* bytes) {
  return pkv_decode_workspace_size_ex(cache, num_seqs, num_q_heads, max_blocks_per_seq, nullptr,
                                      bytes);
}

pkv_status pkv_decode_attn_ex(const pkv_cache* cache, const void* q, int32_t q_dtype,
                              int32_t num_seqs, int32_t num_q_heads,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, float scale, float* out,
                              void* workspace, size_t workspace_bytes,
                              const pkv_decode_opts* opts, int32_t* dev_status, void* stream) {
  PKV_RANGE("pkv_decode_attn");
  pkv_status s = pkv::check_decode_call(cache, q, q_dtype, num_seqs, num_q_heads, block_tables,
                                        max_blocks_per_seq, context_lens, out, dev_status);
  if (s != PKV_OK) return s;
  int split = 0;
  if (!pkv::split_pages_of(opts, &split)) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;
  pkv::DecodeArgs a{};
  a.c = view(cache);
  a.q = q;
  a.q_dtype = q_dtype;
  a.B = num_seqs;
  a.Hq = num_q_heads;
  a.MB = max_blocks_per_seq;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.scale = scale;
  a.out = out;
  a.ws = workspace;
  a.dev_status = dev_status;
  return decode_launch(cache, a, split, workspace_bytes, static_cast<cudaStream_t>(stream));
}

pkv_status pkv_decode_attn(const pkv_cache* cache, const void* q, int32_t q_dtype,
                           int32_t num_seqs, int32_t num_q_heads, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           float scale, float* out, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream) {
  return pkv_decode_attn_ex(cache, q, q_dtype, num_seqs, num_q_heads, block_tables,
                            max_blocks_per_seq, context_lens, scale, out, workspace,
                            workspace_bytes, nullptr, dev_status, stream);
}

pkv_status pkv_decode_step_ex(const pkv_cache* cache, const void* q, int32_t q_dtype,
                              const void* k_new, const void* v_new, int32_t new_dtype,
                              const int32_t* slot_mapping, const int32_t* positions,
                              double rope_theta, int32_t num_seqs, int32_t num_q_heads,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, float scale, float* out,
                              void* workspace, size_t workspace_bytes,
                              const pkv_decode_opts* opts, int32_t* dev_status, void* stream) {
  PKV_RANGE("pkv_decode_step");
  pkv_status s = check_cache(cache);
  if (s != PKV_OK) return s;
  s = check_decode_shape(cache, num_seqs, num_q_heads, max_blocks_per_seq);
  if (s != PKV_OK) return s;
  if (q_dtype != PKV_F32 && q_dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (new_dtype != PKV_F32 && new_dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (positions && !(rope_theta > 1.0)) return PKV_ERR_SHAPE;
  int split = 0;
  if (!pkv::split_pages_of(opts, &split)) return PKV_ERR_SHAPE;
  if (num_seqs == 0) return PKV_OK;
  if (!q || !k_new || !v_new || !slot_mapping || !block_tables || !context_lens || !out)
    return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || !aligned16(k_new) || !aligned16(v_new) ||
      !aligned4(block_tables) || !aligned4(context_lens) || !aligned4(slot_mapping) ||
      (positions && !aligned4(positions)))
    return PKV_ERR_ALIGN;
  if (dev_status && !aligned4(dev_status)) return PKV_ERR_ALIGN;
  pkv::DecodeArgs a{};
  a.c = view(cache);
  a.q = q;
  a.q_dtype = q_dtype;
  a.B = num_seqs;
  a.Hq = num_q_heads;
  a.MB = max_blocks_per_seq;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.scale = scale;
  a.out = out;
  a.ws = workspace;
  a.dev_status = dev_status;
  a.step = true;
  a.kw = cache->k_cache;
  a.vw = cache->v_cache;
  a.ksw = cache->k_scale;
  a.vsw = cache->v_scale;
  a.k_new = k_new;
  a.v_new = v_new;
  a.new_dtype = new_dtype;
  a.slots = slot_mapping;
  a.positions = positions;
  a.rope_theta = rope_theta;
  return decode_launch(cache, a, split, workspace_bytes, static_cast<cudaStream_t>(stream));
}

pkv_status pkv_decode_step(const pkv_cache* cache, const void* q, int32_t q_dtype,
                           const void* k_new, const void* v_new, int32_t new_dtype,
                           const int32_t* slot_mapping, const int32_t* positions,
                           double rope_theta, int32_t num_seqs, int32_t num_q_heads,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, float scale, float* out,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream) {
  return pkv_decode_step_ex(cache, q, q_dtype, k_new, v_new, new_dtype, slot_mapping, positions,
                            rope_theta, num_seqs, num_q_heads, block_tables, max_blocks_per_seq,
                            context_lens, scale, out, workspace, workspace_bytes, nullptr,
                            dev_status, stream);
}

pkv_status pkv_prefill_workspace_size(const pkv_cache* cache, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t max_q_len,
                                      int32_t max_blocks_per_seq, size_t* bytes) {
  return pkv_prefill_workspace_size_ex(cache, num_seqs, num_q_heads, max_q_len,
                                       max_blocks_per_seq, nullptr, bytes);
}

pkv_status pkv_prefill_workspace_size_ex(const pkv_cache* cache, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t max_q_len,
                                         int32_t max_blocks_per_seq,
                                         const pkv_prefill_opts* opts, size_t* bytes) {
  if (!bytes) return PKV_ERR_NULL;
  *bytes = 0;
  pkv_status s = check_cache(cache);
  if (s != PKV_OK) return s;
  s = check_decode_shape(cache, num_seqs, num_q_heads, max_blocks_per_seq);
  if (s != PKV_OK) return s;
  if (max_q_len < 0) return PKV_ERR_SHAPE;
  pkv::PrefillOpts o{};
  if (!pkv::prefill_opts_of(opts, &o)) return PKV_ERR_SHAPE;
  int dev = 0;
  if ((s = current_device(&dev)) != PKV_OK) return s;
  // the split (hence the scratch) depends on the query type: cover both
  size_t need = 0;
  for (const int32_t qt : {PKV_BF16, PKV_F32}) {
    pkv::PrefillPlan plan{};
    if (!pkv::plan_prefill(view(cache), num_seqs, num_q_heads, max_q_len, max_blocks_per_seq, qt,
                           dev, o, &plan))
      return PKV_ERR_UNSUPPORTED;
    if (plan.ws_bytes > need) need = plan.ws_bytes;
  }
  *bytes = need;
  return PKV_OK;
}

pkv_status pkv_prefill_chunk_attn(const pkv_cache* cache, const void* q, int32_t q_dtype,
                                  int32_t num_seqs, int32_t num_q_heads,
                                  const int32_t* q_start_loc, int32_t max_q_len,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, float scale, float* out,
                                  void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, void* stream) {
  return pkv_prefill_chunk_attn_ex(cache, q, q_dtype, num_seqs, num_q_heads, q_start_loc,
                                   max_q_len, block_tables, max_blocks_per_seq, context_lens,
                                   scale, out, workspace, workspace_bytes, nullptr, dev_status,
                                   stream);
}

pkv_status pkv_prefill_chunk_attn_ex(const pkv_cache* cache, const void* q, int32_t q_dtype,
                                     int32_t num_seqs, int32_t num_q_heads,
                                     const int32_t* q_start_loc, int32_t max_q_len,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, float scale, float* out,
                                     void* workspace, size_t workspace_bytes,
                                     const pkv_prefill_opts* opts, int32_t* dev_status,
                                     void* stream) {
  PKV_RANGE("pkv_prefill_chunk_attn");
  pkv_status s = check_cache(cache);
  if (s != PKV_OK) return s;
  s = check_decode_shape(cache, num_seqs, num_q_heads, max_blocks_per_seq);
  if (s != PKV_OK) return s;
  if (q_dtype != PKV_F32 && q_dtype != PKV_BF16) return PKV_ERR_DTYPE;
  if (max_q_len < 0) return PKV_ERR_SHAPE;
  pkv::PrefillOpts o{};
  if (!pkv::prefill_opts_of(opts, &o)) return PKV_ERR_SHAPE;
  if (num_seqs == 0 || max_q_len == 0) return PKV_OK;
  if (!q || !q_start_loc || !block_tables || !context_lens || !out) return PKV_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || !aligned4(q_start_loc) || !aligned4(block_tables) ||
      !aligned4(context_lens))
    return PKV_ERR_ALIGN;
  if (dev_status && !aligned4(dev_status)) return PKV_ERR_ALIGN;
  int dev = 0;
  if ((s = current_device(&dev)) != PKV_OK) return s;
  pkv::PrefillPlan plan{};
  if (!pkv::plan_prefill(view(cache), num_seqs, num_q_heads, max_q_len, max_blocks_per_seq,
                         q_dtype, dev, o, &plan))
    return PKV_ERR_UNSUPPORTED;
  if (plan.n_row_tiles > 0x7fffffff) return PKV_ERR_UNSUPPORTED;
  if (plan.ws_bytes > 0) {
    if (!workspace || workspace_bytes < plan.ws_bytes) return PKV_ERR_WORKSPACE;
    if (!aligned16(workspace)) return PKV_ERR_ALIGN;
  }
  pkv::PrefillArgs a{};
  a.c = view(cache);
  a.q = q;
  a.q_dtype = q_dtype;
  a.B = num_seqs;
  a.Hq = num_q_heads;
  a.MB = max_blocks_per_seq;
  a.max_q_len = max_q_len;
  a.q_start_loc = q_start_loc;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.scale = scale;
  a.out = out;
  a.ws = workspace;
  a.dev_status = dev_status;
  const cudaError_t e = pkv::launch_prefill(a, plan, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : PKV_ERR_LAUNCH;
}

const char* pkv_status_string(pkv_status status) {
  switch (status) {
    case PKV_OK: return "PKV_OK";
    case PKV_ERR_NULL: return "PKV_ERR_NULL: a required pointer is NULL";
    case PKV_ERR_SHAPE: return "PKV_ERR_SHAPE: invalid size or head counts";
    case PKV_ERR_DTYPE: return "PKV_ERR_DTYPE: unknown dtype code";
    case PKV_ERR_PAGE_SIZE: return "PKV_ERR_PAGE_SIZE: page_size must be 16";
    case PKV_ERR_ALIGN: return "PKV_ERR_ALIGN: pointer not 16-byte aligned";
    case PKV_ERR_WORKSPACE: return "PKV_ERR_WORKSPACE: workspace missing or too small";
    case PKV_ERR_UNSUPPORTED: return "PKV_ERR_UNSUPPORTED: combination not supported";
    case PKV_ERR_LAUNCH: return "PKV_ERR_LAUNCH: CUDA launch failed";
    case PKV_ERR_DEVICE: return "PKV_ERR_DEVICE: no usable CUDA device";
  }
  return "PKV_UNKNOWN_STATUS";
}

}  // extern "C"
