// abi.h — host-side argument checks shared by every C entry point, so that the entry
// points over one operation validate exactly alike.
#pragma once
#include <cstdint>

#include "internal.h"
#include "pkv.h"

namespace pkv {

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

// The cache descriptor: pointers, dtype, page size, head_dim, alignment, and 32-bit slot
// numbers for every page of the pool.
pkv_status check_cache(const pkv_cache* c);

// A decode-family shape over cache c: sizes, GQA divisibility, grid limits and 32-bit
// token positions over a full block-table row.
pkv_status check_decode_shape(const pkv_cache* c, int32_t num_seqs, int32_t num_q_heads,
                              int32_t max_blocks_per_seq);

// Everything pkv_decode_attn checks before planning (cache, shape, dtypes, pointers,
// alignment), in its order.
pkv_status check_decode_call(const pkv_cache* c, const void* q, int32_t q_dtype,
                             int32_t num_seqs, int32_t num_q_heads, const int32_t* block_tables,
                             int32_t max_blocks_per_seq, const int32_t* context_lens,
                             const float* out, const int32_t* dev_status);

// Split-K pages per block requested by the options (0: automatic); false if invalid.
bool split_pages_of(const pkv_decode_opts* opts, int* pages);
// The prefill options with defaults for NULL; false if a value is out of range.
bool prefill_opts_of(const pkv_prefill_opts* opts, PrefillOpts* out);

CacheView view(const pkv_cache* c);

}  // namespace pkv
