/*
 * pkv.h — C ABI of the GB300 paged-KV attention library (libpkv.so).
 *
 * Three operations make up the hot path of GQA attention over a paged KV cache:
 *
 *   pkv_append              write new tokens' K/V rows into cache pages via a slot map
 *   pkv_decode_attn         one query token per sequence against its paged context
 *   pkv_prefill_chunk_attn  a causal chunk of query tokens against its paged context
 *
 * and around them:
 *
 *   pkv_decode_step         one launch for a whole decode step: rotary embedding of the
 *                           new query and key, append of the new K/V row, attention
 *   pkv_decode_graph_*      a decode step (all layers) captured once per batch-size
 *                           bucket and replayed with one CUDA graph launch
 *   pkv_decode_attn_noalloc decode attention with its split scratch inside the library
 *   *_ex                    the decode calls with per-call options (pkv_decode_opts)
 *   *_workspace_size, pkv_status_string                               host helpers
 *
 * Sources (page title, section):
 *   "Tiny-LLM-Inference Project_Status", feature list and dtype contract: paged KV
 *     cache, chunked prefill/decode scheduling, FP32 KV by default, a dedicated BF16
 *     paged-attention kernel, FP32 operator boundaries, explicit failure instead of a
 *     silent fallback, preallocated buffers that fail fast instead of reallocating.
 *   "tinyloop Current Status", KV cache modes table: paged attention with 16-token
 *     pages and an INT8 KV cache; model architecture support table: GQA/MQA and
 *     chunked prefill.
 *   "mini-llm-inference-engine" README, architectural highlights: true batched decode
 *     (no per-sequence host loop).
 * The attention itself is the textbook definition (the pages do not write it out):
 *     out[h] = sum_t softmax_t(scale * q[h] . K_t[g]) V_t[g],   g = h / (Hq / Hkv).
 *
 * Conventions shared by every call
 *   - Every pointer argument is caller-owned DEVICE memory unless stated otherwise.
 *     The library allocates no device memory and frees none; the only objects it
 *     creates are the host-side CUDA graphs of a pkv_decode_graph, which the caller
 *     destroys with pkv_decode_graph_destroy.
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *   - Host-checkable errors (null pointers, shapes, dtypes, alignment, workspace size)
 *     return a status synchronously and launch nothing.
 *   - Device-detectable errors (a page id outside [0, num_pages), a context length
 *     outside [0, max_blocks_per_seq * page_size], a slot outside the pool, an
 *     inconsistent prefill chunk) are OR-ed into *dev_status as PKV_DEV_* bits; the
 *     affected rows are written as NaN (attention) or skipped (append).  The kernels
 *     never trap or assert.  `dev_status` may be NULL to ignore such reports.
 *   - There is no fallback: an unsupported combination returns PKV_ERR_UNSUPPORTED.
 *   - Only page_size 16 and head_dim 64 or 128 are supported.
 *
 * Cache layout (struct pkv_cache).  Each (page, kv head) pair owns one K block and one
 * V block of page_size * head_dim elements; block (page, h) starts at element
 * (page * num_kv_heads + h) * page_size * head_dim of k_cache / v_cache.
 *   FP32, INT8, FP8:
 *                K element (token t, column d) at t * head_dim + d        (row per token)
 *                V element (token t, column d) at d * page_size + t       (transposed)
 *   INT4 (two codes per byte; a block is page_size * head_dim / 2 bytes):
 *                K: token t's row is head_dim / 2 bytes at t * head_dim / 2; every 8
 *                   consecutive columns form a little-endian 32-bit word in which column
 *                   8w + e sits at bit 4 * ((e >> 1) + 4 * (e & 1)) (even columns in the
 *                   low half-word, odd ones in the high half-word)
 *                V: row pair p (16 bytes at p * 16) holds columns d = 16 (p / 8) + p % 8
 *                   (low 4 bits) and d + 8 (high 4 bits); token t at byte 4 (t / 4) +
 *                   {0, 2, 1, 3}[t % 4] of the pair (a token's bytes hold only its codes)
 *   BF16 (tensor-core tiles: 8 x 8 core matrices of 64 contiguous elements, so a block
 *         is directly an MMA operand tile):
 *                K element (t, d) at ((t/8) * (head_dim/8) + d/8) * 64 + (t%8) * 8 + d%8
 *                V element (t, d) at ((d/8) * 2 + t/8) * 64 + (d%8) * 8 + t%8
 *   k_scale, v_scale  float32 [num_pages][num_kv_heads][page_size]   INT8, FP8, INT4
 *   Token t of a sequence lives in page block_tables[b][t / page_size] at offset
 *   t % page_size; its slot number is page * page_size + offset.
 *   Element types: PKV_F32 float32, PKV_BF16 bfloat16, and three coded formats whose
 *   value is code * scale with one scale per (token, kv head):
 *     PKV_INT8  codes in [-127, 127] stored in offset binary (the byte holds code + 128),
 *               scale = max|x| / 127;
 *     PKV_FP8   E4M3 codes (OCP "fn": bias 7, no infinity, largest finite 448),
 *               scale = max|x| / 448;
 *     PKV_INT4  4-bit two's-complement codes in [-7, 7], scale = max|x| / 7
 *   ("tinyloop Current Status", KV cache modes table: INT8 and INT4 KV caches; the
 *   TinyInfer review, item 2: INT8 or FP8 KV cache).
 *   All cache pointers must be 16-byte aligned.
 *
 * Sliding window (pkv_cache.window; "tinyloop Current Status", KV cache modes table: a
 * cache window bounds the KV storage).  With window W > 0 every attention call lets the
 * query at position pos see the keys at positions pos - W + 1 .. pos only (the W most
 * recent, its own included); 0 means no window.  Pages wholly before a sequence's window
 * are never read, so a cache manager may release them and leave any value (-1 included)
 * in those block-table entries; partly covered pages are read and must hold written
 * rows.  Several block tables may name the same physical pages (prefix sharing): pages
 * are only read by the attention calls.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum { PKV_F32 = 0, PKV_BF16 = 1, PKV_INT8 = 2, PKV_FP8 = 3, PKV_INT4 = 4 } pkv_dtype;

typedef enum {
  PKV_OK = 0,
  PKV_ERR_NULL = 1,        /* a required pointer is NULL */
  PKV_ERR_SHAPE = 2,       /* a size is negative / zero where it must not be, or Hq % Hkv != 0 */
  PKV_ERR_DTYPE = 3,       /* unknown dtype code */
  PKV_ERR_PAGE_SIZE = 4,   /* page_size != 16 */
  PKV_ERR_ALIGN = 5,       /* a pointer is not 16-byte aligned */
  PKV_ERR_WORKSPACE = 6,   /* workspace NULL or smaller than the *_workspace_size answer */
  PKV_ERR_UNSUPPORTED = 7, /* valid but unsupported combination (e.g. head_dim 96) */
  PKV_ERR_LAUNCH = 8,      /* the CUDA launch itself failed */
  PKV_ERR_DEVICE = 9       /* no usable CUDA device / attribute query failed */
} pkv_status;

/* Device-side error bits OR-ed into *dev_status. */
#define PKV_DEV_BAD_PAGE 0x1 /* block table entry outside [0, num_pages) */
#define PKV_DEV_BAD_LEN 0x2  /* context length < 0 or > max_blocks_per_seq * page_size */
#define PKV_DEV_BAD_SLOT 0x4 /* append slot >= num_pages * page_size */
#define PKV_DEV_BAD_CHUNK 0x8 /* prefill chunk length < 0 or > context length */
#define PKV_DEV_TIMEOUT 0x10 /* a bounded wait on an asynchronous copy gave up */

typedef struct pkv_cache {
  void* k_cache;
  void* v_cache;
  float* k_scale; /* INT8, FP8, INT4 only, else NULL */
  float* v_scale; /* INT8, FP8, INT4 only, else NULL */
  int32_t num_pages;
  int32_t page_size;
  int32_t num_kv_heads;
  int32_t head_dim;
  int32_t kv_dtype; /* pkv_dtype */
  int32_t window;   /* sliding-window length in tokens, 0 = none (see above); >= 0 */
} pkv_cache;

/*
 * KV append ("Tiny-LLM-Inference Project_Status": paged KV cache; "tinyloop Current
 * Status": INT8 KV cache).
 *   k_new, v_new   [num_tokens][num_kv_heads][head_dim], element type new_dtype
 *                  (PKV_F32 or PKV_BF16).  FP32 cache: stored as is (BF16 widened
 *                  exactly).  BF16 cache: rounded to nearest even.  INT8 / INT4 cache:
 *                  per (token, kv head) s = max|x| / R (IEEE division, R = 127 / 7),
 *                  code = clamp(rint(x / s), -R, R), s and codes stored.  FP8 cache:
 *                  s = max|x| / 448, code = E4M3(x / s) rounded to nearest even,
 *                  saturating at +-448.  An all-zero row stores s = 0 and zero codes.
 *   slot_mapping   int32 [num_tokens]; slot < 0 skips that token (padding);
 *                  slot >= num_pages * page_size sets PKV_DEV_BAD_SLOT and is skipped.
 *   Slots within one call must be distinct.  num_tokens == 0 is a no-op.
 */
pkv_status pkv_append(const pkv_cache* cache, const void* k_new, const void* v_new,
                      int32_t new_dtype, const int32_t* slot_mapping, int32_t num_tokens,
                      int32_t* dev_status, void* stream);

/*
 * Options of one decode call (pkv_decode_attn_ex, pkv_decode_step_ex,
 * pkv_decode_attn_noalloc_ex, pkv_decode_workspace_size_ex); a NULL pointer means every
 * option at its default.
 *   split_pages  pages of a sequence's context handled by one thread block (split-K);
 *                0 (default) chooses it from the shape and the device's SM count.  The
 *                split only reorders floating-point sums: a fixed value gives
 *                bit-identical results on every device, and bounds the workspace.
 *                Must be >= 0.
 */
typedef struct pkv_decode_opts {
  int32_t split_pages;
} pkv_decode_opts;

/*
 * Scratch bytes pkv_decode_attn (and pkv_decode_step) needs for this shape on the
 * current device (host call, no launch).  The split of long contexts across thread
 * blocks is a fixed function of the shape, the device's SM count and the options, so
 * equal arguments give bit-identical results.  Writes the size to *bytes (0 is possible).
 * The size covers both calls; the _ex form answers for the given options.
 */
pkv_status pkv_decode_workspace_size(const pkv_cache* cache, int32_t num_seqs,
                                     int32_t num_q_heads, int32_t max_blocks_per_seq,
                                     size_t* bytes);
pkv_status pkv_decode_workspace_size_ex(const pkv_cache* cache, int32_t num_seqs,
                                        int32_t num_q_heads, int32_t max_blocks_per_seq,
                                        const pkv_decode_opts* opts, size_t* bytes);

/*
 * Batched decode attention ("mini-llm-inference-engine" README: true batched decode;
 * "tinyloop Current Status": 16-token paged attention, GQA).
 *   q              [num_seqs][num_q_heads][head_dim], q_dtype PKV_F32 or PKV_BF16.
 *   block_tables   int32 [num_seqs][max_blocks_per_seq]; only the first
 *                  ceil(context_lens[b] / page_size) entries of a row are read.
 *   context_lens   int32 [num_seqs]; tokens of sequence b in cache, the current one
 *                  included (append it first).  0 gives a zero output row.
 *   scale          softmax scale (typically 1 / sqrt(head_dim)).
 *   out            float32 [num_seqs][num_q_heads][head_dim].
 *   workspace      device scratch of at least pkv_decode_workspace_size bytes, 16-byte
 *                  aligned.  It must be zero-filled before its first use; every call
 *                  leaves it ready for the next (its counters return to zero).  Calls
 *                  that share a workspace must not run concurrently.
 */
pkv_status pkv_decode_attn(const pkv_cache* cache, const void* q, int32_t q_dtype,
                           int32_t num_seqs, int32_t num_q_heads, const int32_t* block_tables,
                           int32_t max_blocks_per_seq, const int32_t* context_lens,
                           float scale, float* out, void* workspace, size_t workspace_bytes,
                           int32_t* dev_status, void* stream);
/* pkv_decode_attn with options (see pkv_decode_opts; size the workspace with
 * pkv_decode_workspace_size_ex and the same options). */
pkv_status pkv_decode_attn_ex(const pkv_cache* cache, const void* q, int32_t q_dtype,
                              int32_t num_seqs, int32_t num_q_heads,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, float scale, float* out,
                              void* workspace, size_t workspace_bytes,
                              const pkv_decode_opts* opts, int32_t* dev_status, void* stream);

/*
 * One decode step in one launch ("tinyloop Current Status", model architecture support
 * table: RoPE in every forward path with a configurable theta; KV cache modes table:
 * 16-token pages, INT8 KV).  For every sequence b it computes exactly
 *     rotate q[b] and k_new[b] at positions[b];  pkv_append(k_new[b], v_new[b] at
 *     slot_mapping[b]);  pkv_decode_attn over context_lens[b] tokens,
 * with the new token's K/V used straight from registers by the blocks that need it.
 *   q              [num_seqs][num_q_heads][head_dim], PKV_F32 or PKV_BF16 (as decode).
 *   k_new, v_new   [num_seqs][num_kv_heads][head_dim], new_dtype PKV_F32 or PKV_BF16:
 *                  the new token's key (before rotation) and value; stored as
 *                  pkv_append stores rows (BF16 rounding, INT8 codes and scale).
 *   slot_mapping   int32 [num_seqs]: the new token's slot, which must be the slot of
 *                  logical position context_lens[b] - 1 (else PKV_DEV_BAD_SLOT and NaN
 *                  rows for b, nothing stored); < 0: no new token, b attends over the
 *                  cache as it is.  A page being appended to must not be read by another
 *                  sequence of the same call.
 *   positions      int32 [num_seqs] rotation position of each new token, or NULL for no
 *                  rotation.  Rotation: elements i and i + head_dim/2 form a pair turned
 *                  by the angle positions[b] * rope_theta^(-2i/head_dim) (the half-split
 *                  convention); angles, cos and sin in double, rounded to float; the key
 *                  is rotated in float as y_i = fma(x_i, c, -(x_{i+D/2} s)),
 *                  y_{i+D/2} = fma(x_{i+D/2}, c, x_i s) (its bits decide the stored
 *                  values); rope_theta must exceed 1 when positions is not NULL.
 *   Other arguments and the workspace are those of pkv_decode_attn (the size returned
 *   by pkv_decode_workspace_size covers both calls).
 */
pkv_status pkv_decode_step(const pkv_cache* cache, const void* q, int32_t q_dtype,
                           const void* k_new, const void* v_new, int32_t new_dtype,
                           const int32_t* slot_mapping, const int32_t* positions,
                           double rope_theta, int32_t num_seqs, int32_t num_q_heads,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, float scale, float* out,
                           void* workspace, size_t workspace_bytes, int32_t* dev_status,
                           void* stream);
/* pkv_decode_step with options (see pkv_decode_opts). */
pkv_status pkv_decode_step_ex(const pkv_cache* cache, const void* q, int32_t q_dtype,
                              const void* k_new, const void* v_new, int32_t new_dtype,
                              const int32_t* slot_mapping, const int32_t* positions,
                              double rope_theta, int32_t num_seqs, int32_t num_q_heads,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* context_lens, float scale, float* out,
                              void* workspace, size_t workspace_bytes,
                              const pkv_decode_opts* opts, int32_t* dev_status, void* stream);

/*
 * Options of one prefill call (pkv_prefill_chunk_attn_ex, pkv_prefill_workspace_size_ex);
 * a NULL pointer means every option at its default.
 *   key_split  thread blocks that share the key range of one tile of 128 query rows
 *              (each takes a contiguous share of its key tiles; the last of them to
 *              finish merges their partial softmax states, through the workspace): 0
 *              (default) chooses 1..3 from the shape and the device's SM count; otherwise
 *              1, 2 or 3 (other values return PKV_ERR_SHAPE).  The split only reorders
 *              floating-point sums.
 */
typedef struct pkv_prefill_opts {
  int32_t key_split;
} pkv_prefill_opts;

/*
 * Scratch bytes pkv_prefill_chunk_attn needs on the current device (host call, no
 * launch), for either query type; see its workspace argument below.  The _ex form
 * answers for the given options.
 */
pkv_status pkv_prefill_workspace_size(const pkv_cache* cache, int32_t num_seqs,
                                      int32_t num_q_heads, int32_t max_q_len,
                                      int32_t max_blocks_per_seq, size_t* bytes);
pkv_status pkv_prefill_workspace_size_ex(const pkv_cache* cache, int32_t num_seqs,
                                         int32_t num_q_heads, int32_t max_q_len,
                                         int32_t max_blocks_per_seq,
                                         const pkv_prefill_opts* opts, size_t* bytes);

/*
 * Chunked-prefill attention ("Tiny-LLM-Inference Project_Status": chunked prefill,
 * chunked-prefill SDPA path; "tinyloop Current Status": chunked prefill at chunk 512).
 *   q              [total_q][num_q_heads][head_dim] (q_dtype PKV_BF16 or PKV_F32),
 *                  sequence b owning rows q_start_loc[b] .. q_start_loc[b+1]-1.
 *   q_start_loc    int32 [num_seqs + 1], non-decreasing, q_start_loc[0] == 0.
 *   max_q_len      an upper bound of the chunk lengths (sizes the launch).
 *   context_lens   int32 [num_seqs]: cached tokens INCLUDING the chunk (append the
 *                  chunk first).  Chunk row i (chunk length Lq) sits at position
 *                  context_lens[b] - Lq + i and attends to positions 0..that position
 *                  (with a cache window W: position - W + 1 .. position).
 *   out            float32 [total_q][num_q_heads][head_dim].
 *   workspace      as for decode (pkv_prefill_workspace_size bytes, which covers both
 *                  query types; 0 when no row tile's keys are split).
 * The cache must be PKV_BF16 (other formats return PKV_ERR_UNSUPPORTED); the query tile
 * products run on the tcgen05 tensor cores.
 */
pkv_status pkv_prefill_chunk_attn(const pkv_cache* cache, const void* q, int32_t q_dtype,
                                  int32_t num_seqs, int32_t num_q_heads,
                                  const int32_t* q_start_loc, int32_t max_q_len,
                                  const int32_t* block_tables, int32_t max_blocks_per_seq,
                                  const int32_t* context_lens, float scale, float* out,
                                  void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, void* stream);
/* pkv_prefill_chunk_attn with options (see pkv_prefill_opts; size the workspace with
 * pkv_prefill_workspace_size_ex and the same options). */
pkv_status pkv_prefill_chunk_attn_ex(const pkv_cache* cache, const void* q, int32_t q_dtype,
                                     int32_t num_seqs, int32_t num_q_heads,
                                     const int32_t* q_start_loc, int32_t max_q_len,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, float scale, float* out,
                                     void* workspace, size_t workspace_bytes,
                                     const pkv_prefill_opts* opts, int32_t* dev_status,
                                     void* stream);

/*
 * Decode attention without caller-provided scratch.  (The pages describe no such
 * call; it exists for embedding.)  Some host programs cannot call cudaMalloc or lend
 * the library a buffer: a plugin inside an engine whose pool owns all device memory
 * and offers no allocation hook, or a loop whose owner forbids allocation after
 * start-up.  This entry point computes exactly what pkv_decode_attn computes, with the
 * split-K scratch taken from a fixed array of PKV_NOALLOC_SCRATCH_BYTES in the
 * library's own device memory (reserved on every GPU that loads the library, until the
 * process exits).  It allocates nothing and calls no allocating routine.
 *   - Shapes whose split scratch (what pkv_decode_workspace_size_ex reports for the
 *     same options) exceeds PKV_NOALLOC_SCRATCH_BYTES return PKV_ERR_WORKSPACE and
 *     launch nothing.
 *   - The first call on a device looks up the array's device address (once per
 *     device, with that device current) and keeps it for the life of the process; make
 *     that first call before any stream capture.  A cudaDeviceReset of that device
 *     makes the kept address stale: do not call this entry point on it afterwards.
 *   - Every call shares the one array, which keeps the last call's contents: calls
 *     whose work overlaps on the GPU (other streams, other threads) race and must be
 *     serialised by the caller.  Each call first clears, on `stream`, the merge counters
 *     it uses (one small memset): a caller's workspace is the caller's to keep zeroed,
 *     but this array is shared by calls of every shape, and a call that stopped before
 *     its merge (a failed launch, a wait that gave up) must not leak counts into the
 *     next one.
 * Other arguments, errors and results are those of pkv_decode_attn (the _ex form: of
 * pkv_decode_attn_ex), bit for bit.
 */
#define PKV_NOALLOC_SCRATCH_BYTES (4u << 20)
pkv_status pkv_decode_attn_noalloc(const pkv_cache* cache, const void* q, int32_t q_dtype,
                                   int32_t num_seqs, int32_t num_q_heads,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, float scale, float* out,
                                   int32_t* dev_status, void* stream);
pkv_status pkv_decode_attn_noalloc_ex(const pkv_cache* cache, const void* q, int32_t q_dtype,
                                      int32_t num_seqs, int32_t num_q_heads,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, float scale, float* out,
                                      const pkv_decode_opts* opts, int32_t* dev_status,
                                      void* stream);

/*
 * Bucketed CUDA-graph executor for small-batch decode steps ("mini-llm-inference-engine"
 * README, architecture overview, core design principles: CUDA Graph multi-bucket
 * capture; no mechanism is given).  At small batch the kernels of a decode step take a
 * few microseconds each and their launches dominate; this object captures the whole step
 * once per batch-size bucket and replays it with one graph launch.
 *
 * A step runs, for every layer l in order, either
 *     pkv_append(layer l's new rows) then pkv_decode_attn        (fused == 0), or
 *     pkv_decode_step                                            (fused != 0),
 * over the first B sequences of the caller's buffers, B the bucket.  Every pointer is
 * caller-owned device memory captured by address: the caller rewrites the buffers'
 * contents between launches, never their addresses.  Rows num_seqs .. B - 1 of a launch
 * are padding the caller keeps inert: context_lens 0 and slot_mapping -1 (their outputs
 * are zero rows, nothing is stored).  Layers share block_tables, context_lens,
 * slot_mapping, positions, the workspace and dev_status (all layers of a model index the
 * same pages); each layer has its own cache, queries, new rows and output.
 *   layers[l].q      [B_max][num_q_heads][head_dim] (q_dtype)
 *   layers[l].k_new, v_new  [B_max][num_kv_heads][head_dim] (new_dtype); NULL: no append
 *                    (fused == 0 only)
 *   layers[l].out    [B_max][num_q_heads][head_dim] float32
 *   buckets          ascending batch sizes >= 1 (at most PKV_GRAPH_MAX_BUCKETS); B_max is
 *                    the last one
 *   workspace        at least pkv_decode_graph_workspace_size bytes, zero-filled before
 *                    the first launch (the kernels leave it zero)
 * Creation captures and instantiates one graph per bucket on an internal stream of the
 * current device (host objects only; no device memory is allocated by the library).
 * Launches of one executor are ordered on their stream; executors sharing buffers must
 * not run concurrently.  Errors of the captured calls are returned by create.
 */
#define PKV_GRAPH_MAX_BUCKETS 16

typedef struct pkv_graph_layer {
  pkv_cache cache;
  const void* q;
  const void* k_new;
  const void* v_new;
  float* out;
} pkv_graph_layer;

typedef struct pkv_decode_graph_desc {
  int32_t num_layers;
  const pkv_graph_layer* layers; /* host array of num_layers */
  int32_t num_q_heads;
  int32_t q_dtype;
  int32_t new_dtype;
  int32_t fused;                 /* 0: append + decode; else the fused decode step */
  const int32_t* block_tables;   /* [B_max][max_blocks_per_seq] */
  int32_t max_blocks_per_seq;
  const int32_t* context_lens;   /* [B_max] */
  const int32_t* slot_mapping;   /* [B_max]; NULL only when no layer appends */
  const int32_t* positions;      /* fused only: [B_max] or NULL (no rotation) */
  double rope_theta;
  float scale;
  void* workspace;
  size_t workspace_bytes;
  int32_t* dev_status;           /* may be NULL */
  int32_t num_buckets;
  const int32_t* buckets;        /* host array of num_buckets */
} pkv_decode_graph_desc;

typedef struct pkv_decode_graph pkv_decode_graph;

/* Scratch bytes the executor needs (the largest decode workspace over buckets and
 * layers); host call. */
pkv_status pkv_decode_graph_workspace_size(const pkv_decode_graph_desc* desc, size_t* bytes);

/* Validates desc, captures and instantiates one graph per bucket; *out receives the
 * executor (NULL on error). */
pkv_status pkv_decode_graph_create(const pkv_decode_graph_desc* desc, pkv_decode_graph** out);

/* One step for num_seqs sequences (0 <= num_seqs <= B_max; 0 is a no-op): replays the
 * smallest bucket >= num_seqs on `stream` (a stream of the executor's device). */
pkv_status pkv_decode_graph_launch(pkv_decode_graph* graph, int32_t num_seqs, void* stream);

/* The bucket a launch of num_seqs sequences replays (0 if none). */
int32_t pkv_decode_graph_bucket(const pkv_decode_graph* graph, int32_t num_seqs);

/* Releases the executor's graphs (after its launches have completed); NULL is a no-op. */
void pkv_decode_graph_destroy(pkv_decode_graph* graph);

/* Human-readable name of a status code (static storage, never NULL). */
const char* pkv_status_string(pkv_status status);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
