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
#include <mutex>

#include "internal.h"

namespace pkv {
namespace {

constexpr int kMaxDevices = 64;
int g_sms[kMaxDevices];
std::mutex g_mu;

int sm_count(int device) {
  if (device < 0 || device >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_sms[device] == 0 &&
      cudaDeviceGetAttribute(&g_sms[device], cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    g_sms[device] = 0;
  return g_sms[device];
}

}  // namespace

bool plan_prefill(const CacheView& c, int B, int Hq, int max_q_len, int MB, int q_dtype,
                  int device, const PrefillOpts& opts, PrefillPlan* plan) {
  (void)MB;
  if (c.dtype != kBF16) return false;
  if (c.D != 64 && c.D != 128) return false;
  const int G = Hq / c.Hkv;
  plan->rows_per_cta = prefill_tc_rows();
  const long long rows = static_cast<long long>(max_q_len) * G;
  plan->n_row_tiles = static_cast<int>((rows + plan->rows_per_cta - 1) / plan->rows_per_cta);
  // Key-range split: when the row tiles leave SMs idle (one block per SM: the kernel takes
  // all of an SM's tensor memory), up to 3 blocks share a row tile's keys, as many as keep
  // the launch in one wave; their partial states are merged by the last of them.  (A split
  // into a second wave measured slower than none.)
  const int sms = sm_count(device);
  if (sms <= 0) return false;
  const long long slots = static_cast<long long>(sms) * prefill_tc_blocks_per_sm(q_dtype);
  const long long tiles = static_cast<long long>(plan->n_row_tiles) * c.Hkv * B;
  int best = 1;
  if (opts.key_split > 0) {
    best = opts.key_split;
  } else {
    while (best < 3 && tiles > 0 && tiles * (best + 1) <= slots) ++best;
  }
  if (tiles * best > 0x7fffffffLL / 2) best = 1;
  plan->ksplit = best;
  plan->ws_bytes = 0;
  if (best > 1) {
    const size_t t = static_cast<size_t>(tiles);
    plan->ws_bytes = ((t * 4 + 255) / 256) * 256 +
                     t * best * plan->rows_per_cta * (static_cast<size_t>(c.D) + 2) * 4;
  }
  return true;
}

cudaError_t launch_prefill(const PrefillArgs& a, const PrefillPlan& plan, cudaStream_t st) {
  return launch_prefill_tc(a, plan.n_row_tiles, plan.ksplit, st);
}

}  // namespace pkv
