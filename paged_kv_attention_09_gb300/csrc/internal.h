// internal.h — launch-level interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

constexpr int kPage = 16;  // tokens per page (the only supported page size)

enum : int { kF32 = 0, kBF16 = 1, kINT8 = 2 };

struct CacheView {
  const void* k;
  const void* v;
  const float* ks;
  const float* vs;
  int num_pages, Hkv, D, dtype;
};

// ---------------------------------------------------------------- append
cudaError_t launch_append(const CacheView& c, void* k_cache, void* v_cache, float* ks,
                          float* vs, const void* k_new, const void* v_new, int new_dtype,
                          const int32_t* slots, int T, int32_t* dev_status, cudaStream_t st);

// ---------------------------------------------------------------- decode
struct DecodePlan {
  int heads_per_cta;  // q heads handled by one thread block (<= 8)
  int head_groups;    // ceil(G / heads_per_cta)
  int chunk_pages;    // pages per thread block
  int n_splits;       // grid.x = ceil(max_blocks / chunk_pages)
  size_t ws_bytes;    // workspace bytes
};

struct DecodeArgs {
  CacheView c;
  const void* q;
  int q_dtype, B, Hq, MB;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float scale;
  float* out;
  void* ws;
  int32_t* dev_status;
};

// Fills `plan` for this shape on `device`; returns false for unsupported shapes.
bool plan_decode(const CacheView& c, int B, int Hq, int MB, int q_dtype, int device,
                 int chunk_override, DecodePlan* plan);
// The process-wide split override set by pkv_set_decode_chunk_pages (0 = automatic).
int decode_chunk_override();
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st);

// ---------------------------------------------------------------- prefill
struct PrefillPlan {
  int rows_per_cta;   // (token, head) rows per thread block
  int n_row_tiles;    // grid.x
  size_t ws_bytes;
};

struct PrefillArgs {
  CacheView c;
  const void* q;
  int q_dtype, B, Hq, MB, max_q_len;
  const int32_t* q_start_loc;
  const int32_t* block_tables;
  const int32_t* context_lens;
  float scale;
  float* out;
  void* ws;
  int32_t* dev_status;
};

bool plan_prefill(const CacheView& c, int B, int Hq, int max_q_len, int MB, int q_dtype,
                  int device, PrefillPlan* plan);
cudaError_t launch_prefill(const PrefillArgs& a, const PrefillPlan& plan, cudaStream_t st);

}  // namespace pkv
