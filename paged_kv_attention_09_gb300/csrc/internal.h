// internal.h — launch-level interface between the C ABI (api.cu) and the kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

constexpr int kPage = 16;  // tokens per page (the only supported page size)

enum : int { kF32 = 0, kBF16 = 1, kINT8 = 2, kFP8 = 3, kINT4 = 4 };

// Formats stored as codes with one FP32 scale per (token, kv head).
__host__ __device__ constexpr bool quantised(int dtype) {
  return dtype == kINT8 || dtype == kFP8 || dtype == kINT4;
}

// BF16 page blocks are stored as tensor-core tiles: 8 x 8 "core matrices" of 16-byte
// rows, each matrix 128 contiguous bytes, so one bulk copy of a block lands a valid
// MMA operand tile in shared memory.  Byte offsets inside one (page, kv head) block:
//   K (token t, column d): core matrix (t/8, d/8), row t%8, element d%8
//   V (column d, token t): core matrix (d/8, t/8), row d%8, element t%8
__host__ __device__ constexpr int bf16_k_off(int t, int d, int D) {
  return (((t >> 3) * (D >> 3) + (d >> 3)) << 7) + ((t & 7) << 4) + ((d & 7) << 1);
}
__host__ __device__ constexpr int bf16_v_off(int d, int t) {
  return ((((d >> 3) << 1) + (t >> 3)) << 7) + ((d & 7) << 4) + ((t & 7) << 1);
}

struct CacheView {
  const void* k;
  const void* v;
  const float* ks;
  const float* vs;
  int num_pages, Hkv, D, dtype;
  int window;  // sliding-window length in tokens, 0 = none
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
  int cluster;        // 1: the n_splits blocks of a sequence form a cluster and merge on chip
  size_t ws_bytes;    // workspace bytes (0 for on-chip merges)
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
  // the fused decode step (step == true): the new token of each sequence
  bool step = false;
  void* kw = nullptr;  // the cache again, writable (the new rows are stored)
  void* vw = nullptr;
  float* ksw = nullptr;
  float* vsw = nullptr;
  const void* k_new = nullptr;  // [B][Hkv][D]
  const void* v_new = nullptr;
  int new_dtype = 0;
  const int32_t* slots = nullptr;      // [B]; < 0: no new token
  const int32_t* positions = nullptr;  // [B]; nullptr: no rotation
  double rope_theta = 10000.0;
};

// Fills `plan` for this shape on `device`; returns false for unsupported shapes.
// step: plan for the fused decode-step kernels (their shared memory is a little larger).
bool plan_decode(const CacheView& c, int B, int Hq, int MB, int q_dtype, int device,
                 int chunk_override, DecodePlan* plan, bool step = false);
cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st);

// ---------------------------------------------------------------- prefill
struct PrefillPlan {
  int rows_per_cta;   // (token, head) rows per thread block
  int n_row_tiles;    // row tiles per (sequence, kv head)
  int ksplit;         // blocks sharing a row tile's key range (1: no split)
  size_t ws_bytes;    // workspace bytes (partials and tickets of a split; 0 otherwise)
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

// key_split: 0 automatic, else 1..3
struct PrefillOpts {
  int key_split;
};
bool plan_prefill(const CacheView& c, int B, int Hq, int max_q_len, int MB, int q_dtype,
                  int device, const PrefillOpts& opts, PrefillPlan* plan);
cudaError_t launch_prefill(const PrefillArgs& a, const PrefillPlan& plan, cudaStream_t st);
// tcgen05 path (BF16 KV): query rows per block, blocks resident per SM for a query dtype,
// and the launch over n_row_tiles x ksplit blocks per (sequence, kv head).
int prefill_tc_rows();
int prefill_tc_blocks_per_sm(int q_dtype);
cudaError_t launch_prefill_tc(const PrefillArgs& a, int n_row_tiles, int ksplit, cudaStream_t st);

}  // namespace pkv
