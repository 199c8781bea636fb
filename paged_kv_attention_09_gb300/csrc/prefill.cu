// prefill.cu — planning of chunked-prefill attention over a paged BF16 KV cache.
//
// Sources: "Tiny-LLM-Inference Project_Status" (chunked prefill/decode scheduling; the
// chunked-prefill SDPA path; dedicated BF16 paged-attention kernel) and "tinyloop
// Current Status" (chunked prefill, chunk 512; GQA; 16-token pages).  Row i of a chunk
// of length Lq sits at position context_len - Lq + i and attends causally to positions
// 0..that position (the chunk's own K/V are appended first).
//
// The rows of a launch are (chunk token, query head) pairs of one GQA group, token-major
// (row = i * G + head), so the query heads that share a kv head share every K/V tile;
// the tcgen05 kernel (prefill_tc.cu) takes them in tiles of 128.
#include "internal.h"

namespace pkv {

bool plan_prefill(const CacheView& c, int B, int Hq, int max_q_len, int MB, int q_dtype,
                  int device, PrefillPlan* plan) {
  (void)B; (void)MB; (void)device; (void)q_dtype;
  if (c.dtype != kBF16) return false;
  if (c.D != 64 && c.D != 128) return false;
  const int G = Hq / c.Hkv;
  plan->rows_per_cta = prefill_tc_rows();
  const long long rows = static_cast<long long>(max_q_len) * G;
  plan->n_row_tiles = static_cast<int>((rows + plan->rows_per_cta - 1) / plan->rows_per_cta);
  plan->ws_bytes = 0;
  return true;
}

cudaError_t launch_prefill(const PrefillArgs& a, const PrefillPlan& plan, cudaStream_t st) {
  return launch_prefill_tc(a, plan.n_row_tiles, st);
}

}  // namespace pkv
