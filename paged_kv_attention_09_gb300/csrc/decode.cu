// decode.cu — batched paged decode attention with split-K over pages.
//
// Sources: "mini-llm-inference-engine" README (true batched decode, one launch for the
// whole batch); "tinyloop Current Status" (paged attention with 16-token pages; GQA;
// INT8 KV cache); "Tiny-LLM-Inference Project_Status" (FP32 default KV, dedicated BF16
// paged kernel, FP32 operator boundaries).  The attention is the textbook
// softmax(scale q.K^T) V, evaluated with a running max / running sum (online softmax)
// so that every K/V byte is read from HBM exactly once.
//
// Thread-block layout: grid (split, sequence, kv-head x head-group).  A block owns up to
// 8 query heads that share one kv head, and a contiguous range of the sequence's
// logical pages.  Each of its 4 warps streams every 4th page of that range
// through its own ring of shared-memory stages filled by 1-D bulk copies (TMA engine,
// one copy per K block, V block and scale vector of a (page, kv-head)).  The producer
// lane validates every page id just before issuing its copies, so the first copies are
// in flight before the queries are even loaded.  Warps merge their (max, sum, acc)
// states at the end; when a sequence is split over several blocks, the block that
// arrives last (an atomic ticket, no waiting) merges the partial states in split order.
//
// Three compute paths:
//   FP32 KV — CUDA cores.  8 lanes per token compute the q.k dot products (3 shuffle
//             steps), lanes own head_dim columns for P.V.
//   BF16 KV — warp-level tensor-core MMA (m16n8k16, BF16).  The query heads of the group
//             form the A rows: the BF16 high part in rows 0-7, the rounding remainder in
//             rows 8-15, so FP32 queries keep ~16 bits; the probabilities use the same
//             hi/lo split for P.V.
//   INT8 KV — f16 MMA for both products.  Codes (stored as code + 128) become the exact
//             f16 values 1152 + code with two byte permutes per 4 codes; the bias is removed
//             afterwards: 1152 * sum(q) from each score, 1152 * sum(P) from the output.
//             FP8 (E4M3) and INT4 KV take the same path: E4M3 codes convert to their exact
//             f16 values (no bias), INT4 codes to (8 + code) / 8 through the hardware
//             FP6 (E2M3) conversion after one mask-and-xor per 4 codes (the TinyInfer
//             review, item 2; "tinyloop Current Status", KV cache modes table).
//             Queries are scaled by a power of two into [0.5, 1) and split hi/lo in f16
//             (rows 0-7 / 8-15); per-token K scales multiply the scores and V scales the
//             probabilities (split hi/lo) in FP32.  (The s8 MMA path is far slower on
//             this part.)
// The order of every floating-point reduction depends only on logical token positions,
// the split size and the warp count, so results are bit-identical under any physical
// page permutation.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <cmath>
#include <mutex>

#include "internal.h"
#include "kvrow.cuh"
#include "ptx.cuh"

namespace pkv {

#ifdef PKV_TEST_HOOKS
// Test builds only (never the product library): while set, the first page wait of every
// warp gives up at once, as a wait that ran out of time would, so that the timeout path
// (error bit, NaN rows, drain of the copies in flight) is exercised with no copy stuck.
__device__ int g_test_fail_first_wait = 0;
#endif

namespace {

constexpr int kMaxHeads = 8;     // query heads per block
constexpr int kMaxHeadDim = 128;

struct DParams {
  const uint8_t* k;
  const uint8_t* v;
  const float* ks;
  const float* vs;
  const void* q;
  const int32_t* bt;
  const int32_t* lens;
  float* out;
  float* ws_o;
  float* ws_m;
  float* ws_l;
  int* ws_ticket;
  int32_t* dev_status;
  int q_dtype, Hkv, Hq, G, hpc, head_groups, MB, B, num_pages, chunk;
  int window;  // sliding window in tokens (0: none)
  int cluster;  // 1: the split blocks of a sequence form a cluster and merge on chip
  float scale_log2;
  // the fused decode step (STEP kernels only)
  uint8_t* kw;
  uint8_t* vw;
  float* ksw;
  float* vsw;
  const void* k_new;
  const void* v_new;
  const int32_t* slots;
  const int32_t* positions;
  int new_dtype;
  // theta^(-2i/D), i < D/2, computed on the host (the rotation angle is pos * inv_freq[i])
  double inv_freq[kMaxHeadDim / 2];
};

// Bytes of one stored K row (one token, one kv head); a V block has as many per token.
template <int KVT, int D>
struct RowBytes {
  static constexpr int value = KVT == kF32 ? 4 * D : KVT == kBF16 ? 2 * D : KVT == kINT4 ? D / 2 : D;
};

// Stages (pages in flight) per warp, and the resident blocks per SM the kernel is
// compiled for.  (Coded formats: 2 stages measured faster than 3 once the scale vectors
// left the bulk-copy engine, 25.8 against 26.2 us at the batch-256 INT8 shapes; 4 stages
// cost a block per SM.)
#ifndef PKV_INT8_STAGES
#define PKV_INT8_STAGES 2
#endif
#ifndef PKV_BF16_STAGES
#define PKV_BF16_STAGES 2
#endif
// (FP32, head_dim 64: 2 stages measured faster than 3, 15.2 against 16.0 us on the
// SmolLM2-shaped workload; 4 cost a block per SM)
#ifndef PKV_F32_STAGES
#define PKV_F32_STAGES 2
#endif
template <int KVT, int D>
struct Tune {
  static constexpr int S = quantised(KVT) ? PKV_INT8_STAGES
                         : KVT == kBF16 ? (D == 64 ? 3 : PKV_BF16_STAGES)
                                        : (D == 64 ? PKV_F32_STAGES : 2);
  // Warps per block.  (Three-warp INT8 blocks, which leave 96 registers at 7 blocks per
  // SM, measured slower than four warps at 72 registers.)
  static constexpr int W = 4;
  static constexpr int minBlocks = (quantised(KVT) && D == 64) ? 7 : (KVT == kBF16 && D == 128) ? 3 : 1;
};

template <int KVT, int D>
struct Layout {
  static constexpr int kBytes = kPage * RowBytes<KVT, D>::value;   // K block of one (page, head)
  static constexpr int vBytes = kBytes;                            // V block of one (page, head)
  static constexpr int sBytes = quantised(KVT) ? kPage * 4 : 0;  // one scale vector
  static constexpr int pageBytes = kBytes + vBytes + 2 * sBytes;
  static constexpr int S = Tune<KVT, D>::S;
  static constexpr int stageBytes = pageBytes;
};

template <int KVT, int D, bool STEP = false>
struct Smem {
  using Lo = Layout<KVT, D>;
  static constexpr int kW = Tune<KVT, D>::W;
  static constexpr int stages = kW * Lo::S * Lo::stageBytes;
  // merge area: per-warp max[8], sum[8], acc[8][D+2], then weights [warp][8] (floats)
  // (+ the block's partial for the on-chip split merge: max[8], sum[8], O[8][D])
  static constexpr int combine =
      (3 * kW * kMaxHeads + kW * kMaxHeads * (D + 2) + 2 * kMaxHeads + kMaxHeads * D) * 4;
  static constexpr int big = stages > combine ? stages : combine;
  static constexpr int probs = KVT == kF32 ? kW * kMaxHeads * kPage * 4 : 0;
  // coded formats: the query fragments (one uint4 per k-step and lane) and per-row constants,
  // built once by warp 0 and read by every warp
  // (+ the raw query rows of the block, bulk-copied at block start, and their barrier)
  // (a fused-step kernel lands the raw rows in its rotated-query area instead: rotation
  // reads the queries itself, so the two are never used in one call)
  static constexpr int auxFrag = (D / 16) * 32 * 16 + 2 * kMaxHeads * 4;
  static constexpr int auxQ = STEP ? 0 : kMaxHeads * D * 4;
  static constexpr int aux = quantised(KVT) ? auxFrag + auxQ + 16 : 0;
  static constexpr int bars = kW * Lo::S * 8;
  // fused step: the block's rotated query rows (float), cos and sin of the rotation
  // angles, the new token's K and V rows in storage format (+ their scales)
  static constexpr int stepQ = STEP ? kMaxHeads * D * 4 : 0;
  static constexpr int stepRope = STEP ? D * 4 : 0;
  static constexpr int stepRow = STEP ? 2 * (RowBytes<KVT, D>::value + 16) : 0;
  static constexpr int step0 = big + probs + aux + bars;
  static constexpr int total = step0 + stepQ + stepRope + stepRow;
  // the coded formats' raw query rows and their barrier (offsets from the base)
  static constexpr int qraw = STEP ? step0 : big + probs + auxFrag;
  static constexpr int qbar = big + probs + auxFrag + auxQ;
};

__device__ __forceinline__ float4 load_q4(const void* q, int q_dtype, size_t i) {
  if (q_dtype == kBF16) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(
        static_cast<const __nv_bfloat16*>(q) + i);
    const float2 a = __bfloat1622float2(p[0]);
    const float2 b = __bfloat1622float2(p[1]);
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(q) + i);
}
__device__ __forceinline__ float2 load_q2(const void* q, int q_dtype, size_t i) {
  if (q_dtype == kBF16)
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(
        static_cast<const __nv_bfloat16*>(q) + i));
  return *reinterpret_cast<const float2*>(static_cast<const float*>(q) + i);
}

// Split two floats into a packed high part and a packed remainder (f16 or bf16).
__device__ __forceinline__ void split_h2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(a, b);
  const float2 f = __half22float2(h);
  const __half2 r = __floats2half2_rn(a - f.x, b - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}
__device__ __forceinline__ void split_b2(float a, float b, uint32_t& hi, uint32_t& lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 f = __bfloat1622float2(h);
  const __nv_bfloat162 r = __floats2bfloat162_rn(a - f.x, b - f.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

// Four stored INT8 bytes (code + 128, a 32-bit word) -> two f16x2 words holding
// 1152 + code exactly: each byte becomes the low byte of the f16 0x64XX = 1024 + byte.
__device__ __forceinline__ void u8x4_to_f16x4_biased(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("prmt.b32 %0, %1, %2, 0x4140;" : "=r"(lo) : "r"(w), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x4342;" : "=r"(hi) : "r"(w), "r"(0x64646464u));
}

// Four E4M3 codes (a 32-bit word) -> two f16x2 words holding their exact values (every
// E4M3 value is an f16 value); byte b lands in half b % 2 of word b / 2.  One conversion
// instruction per 16-bit half of the word, each writing its f16x2 result register
// directly (the two-halves struct of the conversion intrinsic cost extra packing moves:
// FP8 decode at the batch-256 shapes 33.6 -> 27.1 us).
__device__ __forceinline__ void e4m3x4_to_f16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(w));
}

// INT4 codes -> (8 + code) / 8 as f16, exactly.  A nibble with its sign bit flipped
// (code + 8, 0 .. 15) alone in the low bits of a byte is the FP6 E2M3 encoding of
// (code + 8) / 8: exponent field 0 or 1 (bias 1) and three mantissa bits, so codes below
// zero land on the subnormals k / 8 and the rest on 1 + k / 8.  Half H of w (0: the low
// nibbles of its bytes, 1: the high nibbles) -> four such bytes; the hardware conversion
// then turns each 16-bit half into an f16x2 word, byte b into half b % 2.  (Measured at
// the batch-256 shapes against two other forms: (24 + code) / 16 built in the f16 bits
// with a shift and a mask-and-xor per two codes, 31.1 us, and the codes themselves by a
// mask-and-xor plus an f16x2 multiply-add per two codes, 30.3-30.6 us; this form 29.6-29.8.)
template <int H>
__device__ __forceinline__ uint32_t s4x4_to_e2m3x4(uint32_t w) {
  return ((H ? w >> 4 : w) & 0x0F0F0F0Fu) ^ 0x08080808u;
}
__device__ __forceinline__ void e2m3x4_to_f16x4(uint32_t m, uint32_t& lo, uint32_t& hi) {
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
      "cvt.rn.f16x2.e2m3x2 %0, l;\n\tcvt.rn.f16x2.e2m3x2 %1, h;\n\t}"
      : "=r"(lo), "=r"(hi) : "r"(m));
}

// ------------------------------------------------------------------ FP32 (CUDA cores)

// Query heads one FP32 block can hold in registers.
template <int D>
__host__ __device__ constexpr int f32_head_cap() {
  return D == 64 ? kMaxHeads : 4;
}

template <int D>
struct F32Warp {
  static constexpr int NC = D / 32;  // float4 chunks per lane per token row
  static constexpr int HM = f32_head_cap<D>();
  float4 q[HM][NC];
  float m[HM], l[HM];
  float o[HM][NC];

  __device__ void finish(const uint8_t*, int, uint32_t) {}
  // (loading the queries before the first copy measured slower here: they are only
  // consumed by the first page anyway)
  __device__ void prefetch(const DParams&, int, int, int, int, int, uint8_t*, uint8_t*) {}
  // sq: the block's query rows as float in shared memory (the fused step), else nullptr
  __device__ void init(const DParams& p, int b, int h0, int nh, int lane, uint8_t*, int,
                       const float* sq) {
    const int c8 = lane & 7;
#pragma unroll
    for (int h = 0; h < HM; ++h) {
      m[h] = -CUDART_INF_F;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        o[h][i] = 0.f;
        q[h][i] = h >= nh ? make_float4(0.f, 0.f, 0.f, 0.f)
                  : sq    ? *reinterpret_cast<const float4*>(sq + h * D + (c8 + 8 * i) * 4)
                          : load_q4(p.q, p.q_dtype,
                                    (static_cast<size_t>(b) * p.Hq + h0 + h) * D + (c8 + 8 * i) * 4);
      }
    }
  }

  // tokens lo .. valid - 1 of the page are attended (lo > 0 only for the first page of a
  // sliding window)
  template <int NH>
  __device__ void page(const uint8_t* st, float* probs, int valid, int lo, float sl, int lane) {
    const float* Ks = reinterpret_cast<const float*>(st);
    const float* Vs = reinterpret_cast<const float*>(st + Layout<kF32, D>::kBytes);
    const int tq = lane >> 3, c8 = lane & 7;
    float s[4][NH];
#pragma unroll
    for (int ps = 0; ps < 4; ++ps) {
      const int t = ps * 4 + tq;
      const float4* kr = reinterpret_cast<const float4*>(Ks + t * D);
      float acc[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) acc[h] = 0.f;
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        const float4 kv = kr[c8 + 8 * i];
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          acc[h] = fmaf(q[h][i].x, kv.x, acc[h]);
          acc[h] = fmaf(q[h][i].y, kv.y, acc[h]);
          acc[h] = fmaf(q[h][i].z, kv.z, acc[h]);
          acc[h] = fmaf(q[h][i].w, kv.w, acc[h]);
        }
      }
#pragma unroll
      for (int h = 0; h < NH; ++h) {
        float a = acc[h];
        a += __shfl_xor_sync(0xffffffffu, a, 1);
        a += __shfl_xor_sync(0xffffffffu, a, 2);
        a += __shfl_xor_sync(0xffffffffu, a, 4);
        s[ps][h] = t < valid && t >= lo ? a * sl : -CUDART_INF_F;
      }
    }
#pragma unroll
    for (int h = 0; h < NH; ++h) {
      float mx = fmaxf(fmaxf(s[0][h], s[1][h]), fmaxf(s[2][h], s[3][h]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float mn = fmaxf(m[h], mx);
      const float corr = fast_exp2(m[h] - mn);
      m[h] = mn;
      float sum = 0.f;
#pragma unroll
      for (int ps = 0; ps < 4; ++ps) {
        s[ps][h] = fast_exp2(s[ps][h] - mn);
        sum += s[ps][h];
      }
      sum += __shfl_xor_sync(0xffffffffu, sum, 8);
      sum += __shfl_xor_sync(0xffffffffu, sum, 16);
      l[h] = l[h] * corr + sum;
#pragma unroll
      for (int i = 0; i < NC; ++i) o[h][i] *= corr;
      if (c8 == 0) {
#pragma unroll
        for (int ps = 0; ps < 4; ++ps) probs[h * kPage + ps * 4 + tq] = s[ps][h];
      }
    }
    __syncwarp();
    // P.V: lane owns columns d = lane + 32 i; the 4-token chunk order is rotated per
    // lane pair so that the 8 lanes of a shared-memory phase hit distinct banks.
#pragma unroll
    for (int i4 = 0; i4 < 4; ++i4) {
      const int c4 = (i4 + (lane >> 1)) & 3;
      float4 pv[NH];
#pragma unroll
      for (int h = 0; h < NH; ++h) pv[h] = *reinterpret_cast<const float4*>(probs + h * kPage + c4 * 4);
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        float4 vv = *reinterpret_cast<const float4*>(Vs + (lane + 32 * i) * kPage + c4 * 4);
        if (valid < kPage || lo > 0) {  // tokens not attended may hold anything: zero them
          const int t0 = c4 * 4;
          vv.x = t0 + 0 < valid && t0 + 0 >= lo ? vv.x : 0.f;
          vv.y = t0 + 1 < valid && t0 + 1 >= lo ? vv.y : 0.f;
          vv.z = t0 + 2 < valid && t0 + 2 >= lo ? vv.z : 0.f;
          vv.w = t0 + 3 < valid && t0 + 3 >= lo ? vv.w : 0.f;
        }
#pragma unroll
        for (int h = 0; h < NH; ++h) {
          float a = o[h][i];
          a = fmaf(pv[h].x, vv.x, a);
          a = fmaf(pv[h].y, vv.y, a);
          a = fmaf(pv[h].z, vv.z, a);
          a = fmaf(pv[h].w, vv.w, a);
          o[h][i] = a;
        }
      }
    }
    __syncwarp();
  }

  __device__ void store(float* cm, float* cl, float* cO, int lane) {
#pragma unroll
    for (int h = 0; h < HM; ++h) {
      if (lane == 0) {
        cm[h] = m[h];
        cl[h] = l[h];
      }
#pragma unroll
      for (int i = 0; i < NC; ++i) cO[h * (D + 2) + lane + 32 * i] = o[h][i];
    }
  }
};

// ------------------------------------------------------------------ BF16 (MMA)

// Lazy rescale margin of the tensor-core paths' softmax: the running max is raised only
// when a score exceeds it by more than 2^8 (in the exponent's log2 units).
constexpr float kRescaleLog2 = 8.f;

template <int D>
struct Bf16Warp {
  static constexpr int KS = D / 16;  // k-steps of the q.k product
  static constexpr int MT = D / 16;  // m-tiles (16 head-dim rows) of O^T = V^T P^T
  uint32_t qa[KS][4];  // raw query bits from prefetch(), then the A fragments
  // O^T accumulators: lane (r, c) holds head-dim rows 16 mt + r and 16 mt + r + 8 of
  // heads 2c and 2c + 1
  float o[MT][4];
  // per query head r = lane / 4: -(running max) and the running sum, in log2 units (the
  // max is raised only beyond a 2^8 margin), and the head's log2 scale
  float nm, l, row_scale;

  __device__ void finish(const uint8_t*, int, uint32_t) {}
  // Query elements of k-slots {2c, 2c+1} and {2c+8, 2c+9} of every k-step (the standard
  // fragment order), loaded as raw bits: two BF16 or two FP32 values per slot pair.
  __device__ void prefetch(const DParams& p, int b, int h0, int nh, int lane, int, uint8_t*,
                           uint8_t*) {
    const int r = lane >> 2, c = lane & 3;
    const bool has = r < nh;
    const size_t row = (static_cast<size_t>(b) * p.Hq + h0 + r) * D;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const size_t i = row + 16 * ks + 8 * half + 2 * c;
        uint32_t w0 = 0u, w1 = 0u;
        if (has) {
          if (p.q_dtype == kBF16) {
            w0 = *reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(p.q) + i);
          } else {
            const uint2 v = *reinterpret_cast<const uint2*>(static_cast<const float*>(p.q) + i);
            w0 = v.x;
            w1 = v.y;
          }
        }
        qa[ks][2 * half] = w0;
        qa[ks][2 * half + 1] = w1;
      }
    }
  }
  __device__ void init(const DParams& p, int, int, int nh, int lane, uint8_t*, int,
                       const float* sq) {
    const int r = lane >> 2, c = lane & 3;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float2 v;
        if (sq) {  // the fused step's rotated query rows
          v = r < nh ? *reinterpret_cast<const float2*>(sq + r * D + 16 * ks + 8 * half + 2 * c)
                     : make_float2(0.f, 0.f);
        } else if (p.q_dtype == kBF16) {
          v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qa[ks][2 * half]));
        } else {
          v = make_float2(__uint_as_float(qa[ks][2 * half]), __uint_as_float(qa[ks][2 * half + 1]));
        }
        uint32_t hi, lo;
        split_b2(v.x, v.y, hi, lo);
        qa[ks][2 * half] = hi;      // rows 0-7 (a0 / a2): the BF16 high part
        qa[ks][2 * half + 1] = lo;  // rows 8-15 (a1 / a3): the remainder
      }
    }
    row_scale = p.scale_log2;
    nm = CUDART_INF_F;
    l = 0.f;
#pragma unroll
    for (int j = 0; j < MT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  }

  // One page.  K and V arrive as tensor-core tiles, so ldmatrix builds every fragment
  // from whole 16-byte core-matrix rows without bank conflicts.  Scores: n-tile j holds
  // tokens 8j .. 8j+7, lane (r, c) ends up with tokens 2c, 2c+1, 8+2c, 9+2c of head r,
  // which is exactly its B fragment of P^T for the transposed product (k = tokens,
  // n = heads).  Tokens lo .. valid - 1 are attended (lo > 0 only for the first page of a
  // window).
  __device__ void page(const uint8_t* st, int valid, int lo, int lane) {
    using Lo = Layout<kBF16, D>;
    const int c = lane & 3;
    const uint32_t Ks = smem_u32(st);
    const uint32_t Vs = Ks + Lo::kBytes;
    float sacc[2][2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
#pragma unroll
      for (int h = 0; h < 2; ++h) sacc[j][h][0] = sacc[j][h][1] = sacc[j][h][2] = sacc[j][h][3] = 0.f;
#pragma unroll
      for (int s = 0; s < KS / 2; ++s) {
        // matrices: chunks 4s .. 4s+3 of key group j -> b0/b1 of k-steps 2s and 2s+1
        uint32_t f[4];
        ldsm_x4(f, Ks + ((j * (D / 8) + 4 * s + (lane >> 3)) << 7) + ((lane & 7) << 4));
        mma_bf16(sacc[j][0], qa[2 * s + 0], f[0], f[1]);
        mma_bf16(sacc[j][1], qa[2 * s + 1], f[2], f[3]);
      }
    }
    float x[4];
#pragma unroll
    for (int j = 0; j < 2; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e)
        x[2 * j + e] = ((sacc[j][0][e] + sacc[j][0][2 + e]) + (sacc[j][1][e] + sacc[j][1][2 + e])) *
                       row_scale;
    uint32_t vmask0 = 0xffffffffu, vmask1 = 0xffffffffu;
    if (valid < kPage || lo > 0) {  // tokens not attended may hold NaN: mask scores, zero V
      auto in = [&](int t) { return t < valid && t >= lo; };
#pragma unroll
      for (int i = 0; i < 4; ++i) x[i] = in(8 * (i >> 1) + 2 * c + (i & 1)) ? x[i] : -CUDART_INF_F;
      vmask0 = (in(2 * c + 0) ? 0x0000ffffu : 0u) | (in(2 * c + 1) ? 0xffff0000u : 0u);
      vmask1 = (in(2 * c + 8) ? 0x0000ffffu : 0u) | (in(2 * c + 9) ? 0xffff0000u : 0u);
    }
    float mx = fmaxf(fmax3(x[0], x[1], x[2]), x[3]);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // the running max is raised only when a score exceeds it by more than 2^8 (the
    // probabilities then stay below 256, exact enough in BF16 hi + lo and in FP32)
    const bool need = mx + nm > kRescaleLog2;
    if (__any_sync(0xffffffffu, need)) {
      const float nn = need ? -mx : nm;
      const float corr = fast_exp2(nn - nm);  // 0 on the first page (nm = +inf)
      nm = nn;
      l *= corr;
      // this lane's accumulators belong to heads 2c and 2c + 1
      const float ca = __shfl_sync(0xffffffffu, corr, 8 * c);
      const float cb = __shfl_sync(0xffffffffu, corr, 8 * c + 4);
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        o[j][0] *= ca; o[j][1] *= cb; o[j][2] *= ca; o[j][3] *= cb;
      }
    }
    float pr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pr[i] = fast_exp2(x[i] + nm);
    l += (pr[0] + pr[1]) + (pr[2] + pr[3]);
    // B = P^T: tokens {2c, 2c+1} and {8+2c, 9+2c} of head r, high part and remainder
    uint32_t bh0, bl0, bh1, bl1;
    split_b2(pr[0], pr[1], bh0, bl0);
    split_b2(pr[2], pr[3], bh1, bl1);
    // A = V^T rows 16 j .. 16 j + 15 (core matrices of head-dim groups 2j, 2j+1 and token
    // groups 0, 1, handed out in the a0..a3 order), one ldmatrix per m-tile
    const uint32_t vrow = Vs + ((0x3120u >> (4 * (lane >> 3))) & 0xfu) * 128 + ((lane & 7) << 4);
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      uint32_t a[4];
      ldsm_x4(a, vrow + j * 512);
      a[0] &= vmask0; a[1] &= vmask0; a[2] &= vmask1; a[3] &= vmask1;
      mma_bf16(o[j], a, bh0, bh1);
      mma_bf16(o[j], a, bl0, bl1);
    }
  }

  __device__ void store(float* cm, float* cl, float* cO, int lane) {
    const int r = lane >> 2, c = lane & 3;
    float lt = l;
    lt += __shfl_xor_sync(0xffffffffu, lt, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    if (c == 0) {
      cm[r] = -nm;  // the running max in log2 units, as the merge expects
      cl[r] = lt;
    }
    float* oa = cO + (2 * c) * (D + 2);
    float* ob = oa + (D + 2);
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      oa[16 * j + r] = o[j][0];
      ob[16 * j + r] = o[j][1];
      oa[16 * j + r + 8] = o[j][2];
      ob[16 * j + r + 8] = o[j][3];
    }
  }
};

// ------------------------------------------------------------------ INT8 / FP8 / INT4 (f16 MMA)

// One path for the three coded formats: the codes become exact f16 MMA operands.
//   INT8  1152 + code (two byte permutes per 4 stored codes); bias removed afterwards
//   INT4  (8 + code) / 8 (one mask-and-xor per 4 codes, a shift for every second word,
//         then the FP6 conversion, 2 codes per instruction); the factor 8 goes into the
//         score scale and the block's final output, the bias is removed afterwards
//   FP8   the E4M3 value itself (hardware conversion, 2 codes per instruction), no bias
// The per-page path is written against an explicit instruction budget: every shared
// address is a per-lane base plus a constant (the ring of stages is unrolled), the V
// codes arrive with two ldmatrix per 64 head-dim rows, the softmax runs on packed FP32
// pairs, and masking is confined to the few pages that are only partly attended.

// (a, b) -> f16x2 high part and f16x2 remainder: a = hi + lo to ~22 bits.
__device__ __forceinline__ void split_h2x(float2 a, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __float22half2_rn(a);
  const float2 f = __half22float2(h);
  const __half2 r = __float22half2_rn(__fadd2_rn(a, make_float2(-f.x, -f.y)));
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&r);
}

template <int KVT, int D>
struct QuantWarp {
  static constexpr int KS = D / 16;  // k-steps of the q.k product
  static constexpr int MT = D / 16;  // m-tiles (16 head-dim rows) of O^T = V^T P^T
  static constexpr int RB = RowBytes<KVT, D>::value;  // bytes of one stored K row
  // the operands are 2^kMulLog2 (kBias + code)
  static constexpr float kBias = KVT == kINT8 ? 1152.f : KVT == kINT4 ? 8.f : 0.f;
  static constexpr int kMulLog2 = KVT == kINT4 ? -3 : 0;
  static constexpr float kUnit = KVT == kINT4 ? 0.125f : 1.f;  // 2^kMulLog2
  // per-lane shared-window addresses in stage 0 of this warp's ring (a stage adds a
  // constant): scale vectors, the two K rows, the ldmatrix row of the V block, and the
  // first query fragment
  uint32_t a_sc, a_k, a_v, a_q;
  // O^T accumulators: lane (r, c) holds head-dim rows 16 mt + r and 16 mt + r + 8 of
  // heads 2c and 2c + 1 (the C layout of the transposed product)
  float o[MT][4];
  // per query head r = lane / 4, both halves equal: -(running max) in log2 units, and
  // the head's log2 scale (scores stay in raw units; the scale applies in the exponent)
  float2 nm2, rs2;
  float2 l2, sp2;  // running sums of P and of P * s_v, two partial sums each
  float kbias;     // kBias * sum(q) of the head, as the MMA sees q

  // k-slot pair {2c, 2c+1} of k-step ks <-> head_dim 64(ks/4) + 16c + 4(ks%4): each lane's
  // K operand is then one contiguous 16-byte shared-memory load per n-tile.
  __device__ static int kslot_d(int ks, int c) { return 64 * (ks >> 2) + 16 * c + 4 * (ks & 3); }
  // The query values of lane c's k-slots {2c, 2c+1, 2c+8, 2c+9} in k-step ks, from the
  // row at q (shared floats, or the prefetched rows in dtype q_dtype).  INT4 K words hold
  // 8 elements, element e at nibble (e / 2) + 4 (e % 2); the conversion's low-nibble half
  // (even k-steps) gives element pairs (0, 4) and (1, 5) of the word, the high-nibble half
  // (2, 6) and (3, 7), so the slots take elements 2h, 2h + 4, 2h + 1, 2h + 5 of the word
  // 64 (ks / 4) + 16 c + 8 ((ks % 4) / 2), h = ks % 2.
  __device__ static float4 q_slots(const float* sq, const void* q, int q_dtype, int ks, int c) {
    if constexpr (KVT == kINT4) {
      const int d = 64 * (ks >> 2) + 16 * c + 8 * ((ks & 3) >> 1) + 2 * (ks & 1);
      const float2 a = sq ? *reinterpret_cast<const float2*>(sq + d) : load_q2(q, q_dtype, d);
      const float2 b = sq ? *reinterpret_cast<const float2*>(sq + d + 4)
                          : load_q2(q, q_dtype, d + 4);
      return make_float4(a.x, b.x, a.y, b.y);
    } else {
      return sq ? *reinterpret_cast<const float4*>(sq + kslot_d(ks, c))
                : load_q4(q, q_dtype, kslot_d(ks, c));
    }
  }

  // The block's query rows (heads h0 .. h0 + nh - 1 of sequence b, contiguous in q) are
  // requested by one bulk copy at block start, ahead of the block-table and length reads,
  // so that they do not queue behind the first wave of page copies.
  // qraw, qbar: where the rows land (kMaxHeads * D floats at most) and their barrier
  __device__ void prefetch(const DParams& p, int b, int h0, int nh, int lane, int w,
                           uint8_t* qraw, uint8_t* qbar) {
    if (w == 0 && lane == 0) {
      const uint32_t elt = p.q_dtype == kBF16 ? 2u : 4u;
      const uint32_t bytes = static_cast<uint32_t>(nh * D) * elt;
      uint64_t* bar = reinterpret_cast<uint64_t*>(qbar);
      mbar_init(bar, 1);
      fence_barrier_init();
      mbar_arrive_expect_tx(bar, bytes);
      bulk_g2s(qraw,
               static_cast<const uint8_t*>(p.q) + (static_cast<size_t>(b) * p.Hq + h0) * D * elt,
               bytes, bar, l2_evict_first_policy());
    }
    __syncwarp();
  }
  // A block that leaves before init() (a split past its sequence's pages) first lets the
  // query copy land, so that no copy writes into the shared memory of an exited block.
  __device__ void drain_prefetch(uint8_t* qbar, int w) {
    if (w == 0) (void)mbar_wait_warp(smem_u32(qbar), 0);
  }

  // Warp 0 builds the query fragments and the per-row constants in shared memory; the
  // caller synchronises the block before any warp reads them (finish()).  Returns false
  // if the wait for the prefetched rows gave up.
  __device__ bool init(const DParams& p, int b, int h0, int nh, int lane, uint8_t* aux, int w,
                       const float* sq, const uint8_t* qraw, uint8_t* qbar) {
    uint4* frag = reinterpret_cast<uint4*>(aux);
    float* rowc = reinterpret_cast<float*>(aux + KS * 32 * 16);
    bool ok = true;
    if (w == 0) {
      const int r = lane >> 2, c = lane & 3;
      const bool has = r < nh;
      if (!sq) {
        ok = mbar_wait_warp(smem_u32(qbar), 0);
        if (!ok) (void)mbar_wait_warp(smem_u32(qbar), 0);  // drain before reuse
      }
      float4 qv[KS];
      float qmax = 0.f;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qv[ks] = !has ? make_float4(0.f, 0.f, 0.f, 0.f)
                      : q_slots(sq ? sq + r * D : nullptr,
                                qraw + static_cast<size_t>(r) * D * (p.q_dtype == kBF16 ? 2 : 4),
                                p.q_dtype, ks, c);
        qmax = fmaxf(qmax, fmaxf(fmaxf(fabsf(qv[ks].x), fabsf(qv[ks].y)),
                                 fmaxf(fabsf(qv[ks].z), fabsf(qv[ks].w))));
      }
      qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
      qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
      // f16 operands: bring the row's largest |q| into [0.5, 1) by an exact power of two
      // and fold the factor into the score scale; hi + lo keeps ~22 bits.
      int e = 0;
      if (qmax > 0.f) frexpf(qmax, &e);
      float qsum = 0.f;  // sum of the operand values exactly as the MMA sees them
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const float x[4] = {ldexpf(qv[ks].x, -e), ldexpf(qv[ks].y, -e), ldexpf(qv[ks].z, -e),
                            ldexpf(qv[ks].w, -e)};
        uint4 f;
        split_h2(x[0], x[1], f.x, f.y);
        split_h2(x[2], x[3], f.z, f.w);
        frag[ks * 32 + lane] = f;
        const uint32_t fw[4] = {f.x, f.y, f.z, f.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float2 v = __half22float2(*reinterpret_cast<const __half2*>(&fw[h]));
          qsum += v.x + v.y;
        }
      }
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 1);
      qsum += __shfl_xor_sync(0xffffffffu, qsum, 2);
      if (c == 0) {
        rowc[r] = ldexpf(p.scale_log2, e - kMulLog2);
        rowc[kMaxHeads + r] = ldexpf(kBias, kMulLog2) * qsum;  // K entered as 2^m (kBias + code)
      }
    }
    nm2 = make_float2(CUDART_INF_F, CUDART_INF_F);
    l2 = sp2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int j = 0; j < MT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
    (void)b; (void)h0;
    return ok;
  }
  // stage0: shared-window address of stage 0 of this warp's ring
  __device__ void finish(const uint8_t* aux, int lane, uint32_t stage0) {
    using Lo = Layout<KVT, D>;
    const int r = lane >> 2, c = lane & 3;
    const float* rowc = reinterpret_cast<const float*>(aux + KS * 32 * 16);
    const float rs = rowc[r];
    rs2 = make_float2(rs, rs);
    kbias = rowc[kMaxHeads + r];
    a_q = smem_u32(aux) + lane * 16;
    a_sc = stage0 + 2 * Lo::kBytes + c * 16;
    // K rows of n-tile 0: token 4(r/2) + r%2 (n-tile 1: two tokens further)
    a_k = stage0 + (4 * (r >> 1) + (r & 1)) * RB + c * (KVT == kINT4 ? 8 : 16);
    a_v = stage0 + Lo::kBytes + lane * 16;
  }

  // Tokens of a partly attended page (so: its stage offset) that are not attended get
  // score -inf and V scale 0; FP8 V codes of those tokens are also set to zero in shared
  // memory, because a stale E4M3 NaN code would survive a zero probability in the MMA.
  __device__ void mask_v_codes(uint32_t so, int valid, int lo, int lane) {
    if constexpr (KVT == kFP8) {
      using Lo = Layout<KVT, D>;
      // V block: D rows of 16 token bytes; keep bytes t with lo <= t < valid
      const uint32_t keep_lo = (valid >= 16 ? 0xffffu : ((1u << valid) - 1u)) & ~((1u << lo) - 1u);
      uint32_t m[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t bits = (keep_lo >> (4 * q)) & 0xfu;
        m[q] = ((bits & 1u) ? 0xffu : 0u) | ((bits & 2u) ? 0xff00u : 0u) |
               ((bits & 4u) ? 0xff0000u : 0u) | ((bits & 8u) ? 0xff000000u : 0u);
      }
      const uint32_t base = a_v - lane * 16 + so;  // the stage's V block
#pragma unroll
      for (int d = lane; d < D; d += 32) {
        const uint32_t ad = base + d * 16;
        uint4 v = lds_u4(ad);
        v.x &= m[0]; v.y &= m[1]; v.z &= m[2]; v.w &= m[3];
        asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(ad), "r"(v.x), "r"(v.y),
                     "r"(v.z), "r"(v.w) : "memory");
      }
      __syncwarp();
      (void)Lo::kBytes;
    }
  }

  // Two B operands (k-slot pairs of one k-step) of a 32-bit word of stored K codes.
  __device__ static void kcvt(uint32_t w, int half, uint32_t& b0, uint32_t& b1) {
    if constexpr (KVT == kFP8) {
      e4m3x4_to_f16x4(w, b0, b1);
    } else if constexpr (KVT == kINT8) {
      u8x4_to_f16x4_biased(w, b0, b1);
    } else {  // INT4: elements (2 half, 2 half + 4) and (2 half + 1, 2 half + 5) of the word
      e2m3x4_to_f16x4(half ? s4x4_to_e2m3x4<1>(w) : s4x4_to_e2m3x4<0>(w), b0, b1);
    }
  }

  // One page at stage offset `so`.  partial: tokens outside [lo, valid) of this page are
  // not attended (the ragged last page, or the page holding a window's first key).
  __device__ __forceinline__ void page(uint32_t so, bool partial, int valid, int lo, int lane) {
    const int c = lane & 3;
    const float4 k4 = lds_f4(a_sc + so);
    float4 v4 = lds_f4(a_sc + so + kPage * 4);
    // S = Q K^T over the page's 16 tokens: n-tile j column n holds token
    // 4(n/2) + 2j + (n%2), so lane (r, c) ends up with tokens 4c .. 4c+3 of head r.  The
    // accumulators of the hi rows start at -kbias: the code bias cancels in FP32.
    float s0[4], s1[4];
#pragma unroll
    for (int blk = 0; blk < D / 64; ++blk) {
      uint32_t kw0[4], kw1[4];
      if constexpr (KVT == kINT4) {
        const uint2 u = lds_u2(a_k + so + blk * 32);
        const uint2 v = lds_u2(a_k + so + 2 * RB + blk * 32);
        kw0[0] = u.x; kw0[1] = u.y; kw1[0] = v.x; kw1[1] = v.y;
        kw0[2] = kw0[3] = kw1[2] = kw1[3] = 0u;
      } else {
        const uint4 u = lds_u4(a_k + so + blk * 64);
        const uint4 v = lds_u4(a_k + so + 2 * RB + blk * 64);
        kw0[0] = u.x; kw0[1] = u.y; kw0[2] = u.z; kw0[3] = u.w;
        kw1[0] = v.x; kw1[1] = v.y; kw1[2] = v.z; kw1[3] = v.w;
      }
#pragma unroll
      for (int s = 0; s < 4; ++s) {
        const uint4 f = lds_u4(a_q + (4 * blk + s) * 512);
        const uint32_t a[4] = {f.x, f.y, f.z, f.w};
        const int wi = KVT == kINT4 ? (s >> 1) : s;
        uint32_t b0, b1, b2, b3;
        kcvt(kw0[wi], s & 1, b0, b1);
        kcvt(kw1[wi], s & 1, b2, b3);
        if (blk == 0 && s == 0) {
          mma_f16_c(s0, a, b0, b1, -kbias, -kbias, 0.f, 0.f);
          mma_f16_c(s1, a, b2, b3, -kbias, -kbias, 0.f, 0.f);
        } else {
          mma_f16(s0, a, b0, b1);
          mma_f16(s1, a, b2, b3);
        }
      }
    }
    // hi + lo rows, times the tokens' K scales: tokens 4c, 4c+1 and 4c+2, 4c+3
    float2 x01 = __fmul2_rn(__fadd2_rn(make_float2(s0[0], s0[1]), make_float2(s0[2], s0[3])),
                            make_float2(k4.x, k4.y));
    float2 x23 = __fmul2_rn(__fadd2_rn(make_float2(s1[0], s1[1]), make_float2(s1[2], s1[3])),
                            make_float2(k4.z, k4.w));
    if (partial) {  // (padding may hold NaN scales: mask by select)
      const int t = 4 * c;
      const bool o0 = t < valid && t >= lo, o1 = t + 1 < valid && t + 1 >= lo;
      const bool o2 = t + 2 < valid && t + 2 >= lo, o3 = t + 3 < valid && t + 3 >= lo;
      x01.x = o0 ? x01.x : -CUDART_INF_F; x01.y = o1 ? x01.y : -CUDART_INF_F;
      x23.x = o2 ? x23.x : -CUDART_INF_F; x23.y = o3 ? x23.y : -CUDART_INF_F;
      v4.x = o0 ? v4.x : 0.f; v4.y = o1 ? v4.y : 0.f;
      v4.z = o2 ? v4.z : 0.f; v4.w = o3 ? v4.w : 0.f;
      mask_v_codes(so, valid, lo, lane);
    }
    float mx = fmaxf(fmax3(x01.x, x01.y, x23.x), x23.y);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    // The running max is raised only when a score exceeds it by more than 2^8 in the
    // exponent (probabilities then stay below 256, well inside f16 and FP32), so most
    // pages skip the rescale entirely.
    const bool need = fmaf(rs2.x, mx, nm2.x) > kRescaleLog2;
    if (__any_sync(0xffffffffu, need)) {
      const float nn = need ? -rs2.x * mx : nm2.x;
      const float corr = fast_exp2(nn - nm2.x);  // 0 on the first page (nm = +inf)
      nm2 = make_float2(nn, nn);
      const float2 c2 = make_float2(corr, corr);
      l2 = __fmul2_rn(l2, c2);
      sp2 = __fmul2_rn(sp2, c2);
      // this lane's accumulators belong to heads 2c and 2c + 1
      const float ca = __shfl_sync(0xffffffffu, corr, 8 * c);
      const float cb = __shfl_sync(0xffffffffu, corr, 8 * c + 4);
#pragma unroll
      for (int j = 0; j < MT; ++j) {
        o[j][0] *= ca; o[j][1] *= cb; o[j][2] *= ca; o[j][3] *= cb;
      }
    }
    const float2 e01 = __ffma2_rn(x01, rs2, nm2), e23 = __ffma2_rn(x23, rs2, nm2);
    const float2 p01 = make_float2(fast_exp2(e01.x), fast_exp2(e01.y));
    const float2 p23 = make_float2(fast_exp2(e23.x), fast_exp2(e23.y));
    l2 = __fadd2_rn(l2, __fadd2_rn(p01, p23));
    const float2 pv01 = __fmul2_rn(p01, make_float2(v4.x, v4.y));
    const float2 pv23 = __fmul2_rn(p23, make_float2(v4.z, v4.w));
    sp2 = __fadd2_rn(sp2, __fadd2_rn(pv01, pv23));
    // B = P^T (tokens x heads): lane (r, c) holds head r, tokens 4c .. 4c+3, which the
    // k-slot order {2c, 2c+1 | 2c+8, 2c+9} -> tokens {4c, 4c+1 | 4c+2, 4c+3} makes a
    // ready-made fragment (INT4: {4c, 4c+2 | 4c+1, 4c+3}, the order in which its V bytes
    // are stored); the hi and lo parts accumulate into the same C.
    uint32_t bh0, bl0, bh1, bl1;
    if constexpr (KVT == kINT4) {
      split_h2x(make_float2(pv01.x, pv23.x), bh0, bl0);
      split_h2x(make_float2(pv01.y, pv23.y), bh1, bl1);
    } else {
      split_h2x(pv01, bh0, bl0);
      split_h2x(pv23, bh1, bl1);
    }
    // A = V^T rows 16 j + r and 16 j + r + 8, tokens 4c .. 4c+3 (same k-slot order).
    // ldmatrix hands lane (r, c) bytes 4c .. 4c+3 of block rows r + 8 i.
    constexpr int NW = KVT == kINT4 ? MT : 2 * MT;  // words: V rows (pair rows for INT4)
    uint32_t w[NW];
#pragma unroll
    for (int q = 0; q < NW / 4; ++q) {
      uint32_t f[4];
      ldsm_x4(f, a_v + so + q * 512);
      w[4 * q] = f[0]; w[4 * q + 1] = f[1]; w[4 * q + 2] = f[2]; w[4 * q + 3] = f[3];
    }
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      uint32_t a[4];
      if constexpr (KVT == kINT4) {
        // one word: row pair 8 j + r, tokens 4c .. 4c+3 stored in the order 0, 2, 1, 3;
        // low nibbles row 16 j + r, high nibbles row 16 j + r + 8
        e2m3x4_to_f16x4(s4x4_to_e2m3x4<0>(w[j]), a[0], a[2]);
        e2m3x4_to_f16x4(s4x4_to_e2m3x4<1>(w[j]), a[1], a[3]);
      } else if constexpr (KVT == kFP8) {
        e4m3x4_to_f16x4(w[2 * j], a[0], a[2]);
        e4m3x4_to_f16x4(w[2 * j + 1], a[1], a[3]);
      } else {
        u8x4_to_f16x4_biased(w[2 * j], a[0], a[2]);
        u8x4_to_f16x4_biased(w[2 * j + 1], a[1], a[3]);
      }
      mma_f16(o[j], a, bh0, bh1);
      mma_f16(o[j], a, bl0, bl1);
    }
  }

  __device__ void store(float* cm, float* cl, float* cO, int lane) {
    const int r = lane >> 2, c = lane & 3;
    float lt = l2.x + l2.y, st = sp2.x + sp2.y;
    lt += __shfl_xor_sync(0xffffffffu, lt, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    st += __shfl_xor_sync(0xffffffffu, st, 1);
    st += __shfl_xor_sync(0xffffffffu, st, 2);
    if (c == 0) {
      cm[r] = -nm2.x;  // the running max in log2 units, as the merge expects
      cl[r] = lt;
    }
    // V entered the MMA as 2^m (kBias + code) against P s_v: remove 2^m kBias sum(P s_v)
    // of heads 2c and 2c + 1, then the factor 2^m (once here rather than on every page's
    // V scales)
    constexpr float vb = kBias * kUnit, up = 1.f / kUnit;
    const float ba = vb * __shfl_sync(0xffffffffu, st, 8 * c);
    const float bb = vb * __shfl_sync(0xffffffffu, st, 8 * c + 4);
    float* oa = cO + (2 * c) * (D + 2);
    float* ob = oa + (D + 2);
#pragma unroll
    for (int j = 0; j < MT; ++j) {
      oa[16 * j + r] = (o[j][0] - ba) * up;
      ob[16 * j + r] = (o[j][1] - bb) * up;
      oa[16 * j + r + 8] = (o[j][2] - ba) * up;
      ob[16 * j + r + 8] = (o[j][3] - bb) * up;
    }
  }
};

template <int KVT, int D>
struct WarpOf;
template <int D>
struct WarpOf<kF32, D> {
  using type = F32Warp<D>;
};
template <int D>
struct WarpOf<kBF16, D> {
  using type = Bf16Warp<D>;
};
template <int D>
struct WarpOf<kINT8, D> {
  using type = QuantWarp<kINT8, D>;
};
template <int D>
struct WarpOf<kFP8, D> {
  using type = QuantWarp<kFP8, D>;
};
template <int D>
struct WarpOf<kINT4, D> {
  using type = QuantWarp<kINT4, D>;
};

// ------------------------------------------------------------------ the kernel

// Split-K merge on chip, for a sequence whose split blocks form one thread-block cluster
// (rank = split).  Every block has left its partial (max, sum, O of its heads) in its own
// shared memory (`part`); each counts itself done on block 0's counter, and the block that
// finishes last reads every partial through distributed shared memory, writes the output,
// and releases the others, which wait (bounded) so that their shared memory outlives the
// reads.  No global memory is touched and no block waits for another's work.
template <int D, int kThreads>
__device__ __noinline__ void cluster_merge(const DParams& p, const float* part, int nsplit, int b,
                                           int h0, int nh, int tid, int lane, int w,
                                           uint32_t* s_done, uint64_t* s_release, int* s_last) {
  constexpr int kW = kThreads / 32;
  // parameters read once into registers: this function is not inlined, so each use of p
  // would be a load through a generic pointer, repeated after every store
  float* const out = p.out;
  int32_t* const dev_status = p.dev_status;
  const int Hq = p.Hq;
  __syncthreads();        // this block's partial is complete
  cluster_wait_acquire();  // every block's barrier and counter are initialised
  if (tid == 0) {
    fence_acq_rel_cluster();
    const uint32_t old = dsmem_atomic_add(dsmem_addr(smem_u32(s_done), 0), 1);
    *s_last = old == static_cast<uint32_t>(nsplit - 1);
  }
  __syncthreads();
  if (!*s_last) {
    if (tid == 0 && !mbar_wait(s_release, 0) && dev_status)
      atomicOr(dev_status, 0x10);  // PKV_DEV_TIMEOUT
    return;
  }
  fence_acq_rel_cluster();  // the other blocks' partials are visible
  __shared__ float wts[9 * kMaxHeads];  // [split][head] weights, then [head] 1 / total sum
  const uint32_t part_u32 = smem_u32(part);
  for (int r = w; r < nh; r += kW) {
    float ms = -CUDART_INF_F, ls = 0.f;
    if (lane < nsplit) {
      ms = dsmem_ld_f32(dsmem_addr(part_u32 + 4 * r, lane));
      ls = dsmem_ld_f32(dsmem_addr(part_u32 + 4 * (kMaxHeads + r), lane));
    }
    const bool poisoned = __any_sync(0xffffffffu, isnan(ms));
    float M = ms;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    const float f = ms == -CUDART_INF_F ? 0.f : fast_exp2(ms - M);
    float Ls = ls * f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
    if (lane < nsplit) wts[lane * kMaxHeads + r] = f;
    if (lane == 0) wts[8 * kMaxHeads + r] = poisoned ? CUDART_NAN_F : (Ls > 0.f ? 1.f / Ls : 0.f);
  }
  __syncthreads();
  constexpr int D4 = D / 4;
  const size_t row0 = static_cast<size_t>(b) * Hq + h0;
  for (int c = tid; c < nh * D4; c += kThreads) {
    const int r = c / D4;
    const uint32_t src = part_u32 + 4 * (2 * kMaxHeads + r * D) + 16 * (c % D4);
    float4 v[8];
#pragma unroll
    for (int s = 0; s < 8; ++s)
      if (s < nsplit) v[s] = dsmem_ld_f4(dsmem_addr(src, s));
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < 8; ++s) {
      if (s < nsplit) {
        const float wt = wts[s * kMaxHeads + r];
        acc.x += v[s].x * wt; acc.y += v[s].y * wt; acc.z += v[s].z * wt; acc.w += v[s].w * wt;
      }
    }
    const float inv = wts[8 * kMaxHeads + r];
    *reinterpret_cast<float4*>(out + (row0 + r) * D + 4 * (c % D4)) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  __syncthreads();  // every read of another block's shared memory is done
  const uint32_t me = cluster_rank();
  if (tid < nsplit && static_cast<uint32_t>(tid) != me)
    mbar_arrive_remote(dsmem_addr(smem_u32(s_release), tid));
}

// WIN: compiled with the sliding-window range and mask (the kernels without it carry no
// trace of it: the INT8 kernel sits at its register budget)
template <int KVT, int D, bool STEP, bool WIN>
__global__ void __launch_bounds__(Tune<KVT, D>::W * 32, Tune<KVT, D>::minBlocks)
    decode_kernel(const __grid_constant__ DParams p) {
  using Lo = Layout<KVT, D>;
  using Sm = Smem<KVT, D, STEP>;
  constexpr int S = Lo::S;
  constexpr int kW = Tune<KVT, D>::W, kThreads = kW * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  float* probs_all = reinterpret_cast<float*>(smem + Sm::big);
  uint8_t* aux = smem + Sm::big + Sm::probs;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::big + Sm::probs + Sm::aux);
  __shared__ int s_flag, s_last;
  // on-chip split merge: this block's release by the merging block, and (block 0 of the
  // cluster) the count of blocks that finished
  __shared__ __align__(8) uint64_t s_release;
  __shared__ uint32_t s_done;

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int split = blockIdx.x, b = blockIdx.y, z = blockIdx.z;
  if (p.cluster) {
    // Every thread of every block of the cluster arrives here first, before any exit: a
    // block reaches into another's shared memory only after the matching wait.
    if (tid == 0) {
      mbar_init(&s_release, 1);
      s_done = 0;
      fence_barrier_init();
    }
    cluster_arrive_release();
  }
  const int g = z / p.head_groups, hg = z % p.head_groups;
  const int h0 = g * p.G + hg * p.hpc;
  const int nh = min(p.hpc, p.G - hg * p.hpc);

  // The block-table entries of this warp's first 32 pages do not depend on the context
  // length: read them together with it (validated below), so that the first copies wait
  // for one global round trip instead of two.  The warp's page m is the block's logical
  // page pb + w + m kW.  (With a sliding window the block's
  // range starts at the window's first page, known once the length is: a second trip.)
  const int win = WIN ? p.window : 0;
  int pb = split * p.chunk;
  const int32_t* bt = p.bt + static_cast<size_t>(b) * p.MB;
  const int j_off = w + lane * kW;
  int raw_first = win == 0 && pb + j_off < min(p.MB, pb + p.chunk) ? bt[pb + j_off] : -1;
  typename WarpOf<KVT, D>::type st;
  // query loads, in flight with the length and table reads (a fused step with rotation
  // reads its rotated queries from shared memory instead)
  const bool rope = STEP && p.positions != nullptr;
  if (!rope) st.prefetch(p, b, h0, nh, lane, w, smem + Sm::qraw, smem + Sm::qbar);
  // the fused step's loads, raw bits, likewise issued before anything waits: thread t
  // holds query pairs t, t + kThreads, ... (pair (h, i) = elements i and i + D/2 of head
  // h0 + h); the last warp holds the new token's K and V rows, E = D/32 elements per lane
  constexpr int QPT = STEP ? (kMaxHeads * (D / 2) + kThreads - 1) / kThreads : 1;
  constexpr int NE = D / 32;
  uint32_t qr[QPT][2], kr[NE], vr[NE];
  if constexpr (STEP) {
    const bool qb = p.q_dtype == kBF16, nb = p.new_dtype == kBF16;
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int idx = tid + k * kThreads;
      qr[k][0] = qr[k][1] = 0u;
      if (rope && idx < nh * (D / 2)) {
        const size_t qi = (static_cast<size_t>(b) * p.Hq + h0 + idx / (D / 2)) * D + idx % (D / 2);
        if (qb) {
          qr[k][0] = static_cast<const uint16_t*>(p.q)[qi];
          qr[k][1] = static_cast<const uint16_t*>(p.q)[qi + D / 2];
        } else {
          qr[k][0] = static_cast<const uint32_t*>(p.q)[qi];
          qr[k][1] = static_cast<const uint32_t*>(p.q)[qi + D / 2];
        }
      }
    }
    // (the block's last warp takes the new row, so that its quantisation runs beside
    // warp 0's query fragments rather than after them)
    const size_t src = (static_cast<size_t>(b) * p.Hkv + g) * D + lane * NE;
#pragma unroll
    for (int e = 0; e < NE; ++e) {
      kr[e] = vr[e] = 0u;
      if (w == kW - 1) {
        if (nb) {
          kr[e] = static_cast<const uint16_t*>(p.k_new)[src + e];
          vr[e] = static_cast<const uint16_t*>(p.v_new)[src + e];
        } else {
          kr[e] = static_cast<const uint32_t*>(p.k_new)[src + e];
          vr[e] = static_cast<const uint32_t*>(p.v_new)[src + e];
        }
      }
    }
  }
  const int L = p.lens[b];
  const bool len_ok = L >= 0 && L <= p.MB * kPage;
  const int np = len_ok ? (L + kPage - 1) / kPage : 0;
  // first attended key: L - window under a sliding window, else 0; the splits cover the
  // pages from the one that holds it
  const int lo = win > 0 && len_ok && L > win ? L - win : 0;
  const int nsplit = len_ok ? max(1, (np - lo / kPage + p.chunk - 1) / p.chunk) : 1;
  if (split >= nsplit) {
    if constexpr (quantised(KVT)) {
      if (!rope) st.drain_prefetch(smem + Sm::qbar, w);
    }
    return;
  }
  if (win > 0) {
    pb += lo / kPage;
    raw_first = pb + j_off < min(np, pb + p.chunk) ? bt[pb + j_off] : -1;
  }
  const int pe = min(np, pb + p.chunk);
  if (tid == 0) s_flag = len_ok ? 0 : 0x2 /*PKV_DEV_BAD_LEN*/;

  uint8_t* my_stages = stages + static_cast<size_t>(w) * S * Lo::stageBytes;
  uint64_t* my_bars = bars + w * S;
  float* probs = probs_all + w * kMaxHeads * kPage;
  // this warp's iterations: the block's pages w, w + kW, ...
  const int n_my = pe - pb > w ? (pe - pb - w + kW - 1) / kW : 0;

  // ---- page ids: lane l holds the id of this warp's page m = 32 k + l (batch k) for the
  // current and the next batch; the warp's page m is the block's page pb + w + m kW.  An
  // id outside the pool is replaced by page 0 (so every copy stays inside the cache) and
  // flagged: the block's outputs then become NaN.
  int werr = 0;
  auto check_id = [&](int m, int raw) -> int {
    if (m >= n_my) return 0;
    if (raw < 0 || raw >= p.num_pages) {
      werr |= 0x1;  // PKV_DEV_BAD_PAGE
      return 0;
    }
    return raw;
  };
  auto load_ids = [&](int batch) -> int {
    const int m = 32 * batch + lane;
    return check_id(m, m < n_my ? bt[pb + w + m * kW] : -1);
  };
  int ids_cur = check_id(lane, raw_first), ids_nxt = load_ids(1);

  // ---- copy issue: lanes 0 and 1 issue one bulk copy each of the iteration's page (K
  // block, V block), so a whole stage costs one warp instruction; lane 0 posts the byte
  // count.  The coded formats' two 64-byte scale vectors come by per-thread 16-byte async
  // copies of lanes 8..15, whose completion arrives on the same stage barrier: the
  // bulk-copy engine then handles two copies per page instead of four (at the start of a
  // launch, 28 warps of an SM request 3 stages each at once).  The lane's source base,
  // page stride and destination are computed once.
  constexpr int kScaleLanes = quantised(KVT) ? 8 : 0;
  const int ck = lane < 2 ? lane : 0;
  constexpr uint32_t c_bytes = static_cast<uint32_t>(Lo::kBytes);
  const uint32_t c_dst = smem_u32(my_stages) + (ck == 0 ? 0u : c_bytes);
  const uint8_t* c_src = (ck == 0 ? p.k : p.v) + static_cast<size_t>(g) * c_bytes;
  const uint32_t c_stride = static_cast<uint32_t>(p.Hkv) * c_bytes;  // from one page to the next
  const int sl = lane - 8;  // scale lanes: sl / 4 = K or V vector, sl % 4 = 16-byte piece
  const bool s_lane = kScaleLanes > 0 && sl >= 0 && sl < kScaleLanes;
  const uint32_t s_dst = smem_u32(my_stages) + 2 * c_bytes +
                         (s_lane ? static_cast<uint32_t>((sl >> 2) * Lo::sBytes + (sl & 3) * 16) : 0u);
  const float* s_src = s_lane ? (sl >> 2 ? p.vs : p.ks) + static_cast<size_t>(g) * kPage + (sl & 3) * 4 : nullptr;
  const size_t s_stride = static_cast<size_t>(p.Hkv) * kPage;  // floats from one page to the next
  const uint32_t bar0 = smem_u32(my_bars);
  const uint64_t pol = l2_evict_first_policy();  // streamed once: keep L2 for others
  auto issue = [&](int i, int stage) {
    const uint32_t pid = static_cast<uint32_t>(__shfl_sync(0xffffffffu, ids_cur, i & 31));
    const uint32_t bar = bar0 + 8 * stage;
    mbar_arrive_expect_tx_if(lane == 0, bar, 2 * c_bytes);
    bulk_g2s_if(lane < 2, c_dst + stage * Lo::stageBytes, c_src + static_cast<size_t>(pid) * c_stride,
                c_bytes, bar, pol);
    if (s_lane) {
      asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s_dst + stage * Lo::stageBytes),
                   "l"(s_src + static_cast<size_t>(pid) * s_stride) : "memory");
      asm volatile("cp.async.mbarrier.arrive.noinc.shared.b64 [%0];" ::"r"(bar) : "memory");
    }
  };
  if (n_my > 0) {
    if (lane == 0) {
      // one arrival with the bulk bytes, plus one per scale lane when its copy lands
      for (int i = 0; i < S; ++i) mbar_init(&my_bars[i], 1 + kScaleLanes);
      fence_barrier_init();
    }
    __syncwarp();
    // Every stage is requested at once: the launch's first wave keeps HBM busy from the
    // start (measured 0.2-0.3 us faster than requesting the later stages after the first
    // page lands).
    for (int k = 0; k < min(S, n_my); ++k) issue(k, k);
  }

  // ---- the fused decode step: the rotated query rows, and the new token's K and V rows
  // in storage format for the block that holds the sequence's last page (which patches
  // them into that page once it lands, and, for head group 0, stores them in the cache)
  const float* sq = nullptr;
  bool patch = false;
  int t_new = 0;
  uint8_t* const nrow = smem + Sm::step0 + Sm::stepQ + Sm::stepRope;
  if constexpr (STEP) {
    constexpr int RB = RowBytes<KVT, D>::value;
    float* sqw = reinterpret_cast<float*>(smem + Sm::step0);
    float* rc = reinterpret_cast<float*>(smem + Sm::step0 + Sm::stepQ);
    float* rs = rc + D / 2;
    const int slot = p.slots[b];
    const int pos = rope ? p.positions[b] : 0;
    bool slot_ok = true;  // the new token must sit at logical position L - 1
    if (slot >= 0) {
      const int lp = len_ok && L >= 1 ? bt[(L - 1) / kPage] : -1;
      slot_ok = lp >= 0 && lp < p.num_pages && slot == lp * kPage + (L - 1) % kPage;
      if (!slot_ok && tid == 0) atomicOr(&s_flag, 0x4);  // PKV_DEV_BAD_SLOT
    }
    if (rope) {
      // rotation angles pos * theta^(-2i/D) in double, cos and sin rounded to float
      for (int i = tid; i < D / 2; i += kThreads) {
        double sn, cs;
        sincos(static_cast<double>(pos) * p.inv_freq[i], &sn, &cs);
        rc[i] = static_cast<float>(cs);
        rs[i] = static_cast<float>(sn);
      }
      __syncthreads();
    }
    const bool qb = p.q_dtype == kBF16;
#pragma unroll
    for (int k = 0; k < QPT; ++k) {
      const int idx = tid + k * kThreads;
      if (!rope || idx >= nh * (D / 2)) break;
      const int h = idx / (D / 2), i = idx % (D / 2);
      float x0 = __uint_as_float(qb ? qr[k][0] << 16 : qr[k][0]);
      float x1 = __uint_as_float(qb ? qr[k][1] << 16 : qr[k][1]);
      if (rope) {  // pair (i, i + D/2) rotated by angle i
        const float c = rc[i], sn = rs[i];
        const float t = __fmul_rn(x1, sn), u = __fmul_rn(x0, sn);
        x0 = __fmaf_rn(x0, c, -t);
        x1 = __fmaf_rn(x1, c, u);
      }
      sqw[h * D + i] = x0;
      sqw[h * D + i + D / 2] = x1;
    }
    patch = slot >= 0 && slot_ok && np > 0 && pe == np;
    t_new = (L - 1) & (kPage - 1);
    if (patch && w == kW - 1) {
      constexpr int E = NE;  // lane l holds elements E l .. E l + E - 1
      const bool nb = p.new_dtype == kBF16;
      float kx[E], vx[E];
#pragma unroll
      for (int e = 0; e < E; ++e) {
        kx[e] = __uint_as_float(nb ? kr[e] << 16 : kr[e]);
        vx[e] = __uint_as_float(nb ? vr[e] << 16 : vr[e]);
      }
      if (rope) {
        // element d's partner d +- D/2 sits in lane l +- 16 at the same e; the operation
        // order is fixed (it decides the stored bits): two products, then a fused
        // multiply-add per output
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int d = lane * E + e, i = d & (D / 2 - 1);
          const float partner = __shfl_xor_sync(0xffffffffu, kx[e], 16);
          const float c = rc[i], sn = rs[i];
          const float t = __fmul_rn(partner, sn);
          kx[e] = d < D / 2 ? __fmaf_rn(kx[e], c, -t) : __fmaf_rn(kx[e], c, t);
        }
      }
      // storage format, in shared memory (the patch) and, by head group 0, in the cache
      const int page = slot / kPage, off = slot % kPage;
      const size_t blk = static_cast<size_t>(page) * p.Hkv + g;
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const float(&x)[E] = which ? vx : kx;
        uint8_t* nr = nrow + which * (RB + 16);
        uint8_t* cache = which ? p.vw : p.kw;
        if constexpr (KVT == kINT4) {
          // K: the row's words; V: one byte per row pair (the block's V rows 8j + r hold
          // head-dim rows 16j + r and 16j + r + 8) at the token's position
          int8_t code[E];
          const float sc = quantize_row_int4<E>(x, code);
          uint8_t* cb = cache + blk * kPage * (D / 2);
          if (which == 0) {
            const uint32_t wd = int4_k_word<E>(code, lane);
            if ((lane & (8 / E - 1)) == 0) {
              reinterpret_cast<uint32_t*>(nr)[lane * E / 8] = wd;
              if (hg == 0) reinterpret_cast<uint32_t*>(cb + off * (D / 2))[lane * E / 8] = wd;
            }
          } else {
#pragma unroll
            for (int e = 0; e < E; ++e) {
              const int d = lane * E + e;
              const uint8_t by = int4_v_byte<E>(code, e);
              if ((d & 15) < 8) {
                nr[int4_v_pair(d)] = by;
                if (hg == 0) cb[int4_v_pair(d) * kPage + int4_v_tpos(off)] = by;
              }
            }
          }
          if (lane == 0) {
            *reinterpret_cast<float*>(nr + RB) = sc;
            if (hg == 0) (which ? p.vsw : p.ksw)[blk * kPage + off] = sc;
          }
        } else if constexpr (KVT == kINT8 || KVT == kFP8) {
          uint8_t code[E];
          float sc;
          if constexpr (KVT == kINT8) {
            int8_t c8[E];
            sc = quantize_row_int8<E>(x, c8);
#pragma unroll
            for (int e = 0; e < E; ++e) code[e] = int8_stored(c8[e]);
          } else {
            sc = quantize_row_fp8<E>(x, code);
          }
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            nr[d] = code[e];
            if (hg == 0) {
              if (which == 0) cache[(blk * kPage + off) * D + d] = code[e];
              else cache[blk * D * kPage + static_cast<size_t>(d) * kPage + off] = code[e];
            }
          }
          if (lane == 0) {
            *reinterpret_cast<float*>(nr + RB) = sc;
            if (hg == 0) (which ? p.vsw : p.ksw)[blk * kPage + off] = sc;
          }
        } else if constexpr (KVT == kBF16) {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            const __nv_bfloat16 v = __float2bfloat16_rn(x[e]);
            reinterpret_cast<__nv_bfloat16*>(nr)[d] = v;
            if (hg == 0) {
              const int o = which == 0 ? bf16_k_off(off, d, D) : bf16_v_off(d, off);
              *reinterpret_cast<__nv_bfloat16*>(cache + blk * kPage * D * 2 + o) = v;
            }
          }
        } else {
#pragma unroll
          for (int e = 0; e < E; ++e) {
            const int d = lane * E + e;
            reinterpret_cast<float*>(nr)[d] = x[e];
            if (hg == 0) {
              float* cf = reinterpret_cast<float*>(cache);
              if (which == 0) cf[(blk * kPage + off) * D + d] = x[e];
              else cf[blk * D * kPage + static_cast<size_t>(d) * kPage + off] = x[e];
            }
          }
        }
      }
    }
    // rotated queries and the new row are ready (for the coded formats without rotation
    // the block barrier after the query fragments below covers the new row)
    if (rope || !quantised(KVT)) __syncthreads();
    if (rope) sq = sqw;  // (without rotation the queries load as in plain decode)
  }

  if constexpr (quantised(KVT)) {
    if (!st.init(p, b, h0, nh, lane, aux, w, sq, smem + Sm::qraw, smem + Sm::qbar))
      werr |= 0x10;  // PKV_DEV_TIMEOUT
    __syncthreads();  // warp 0 built the shared query fragments
  } else {
    st.init(p, b, h0, nh, lane, aux, w, sq);
  }
  st.finish(aux, lane, smem_u32(my_stages));
  __syncwarp();

  // Partly attended pages: the ragged last page of the sequence (iteration i_tail of the
  // warp that holds it) and, under a window, the page of the window's first key (block
  // 0, warp 0, iteration 0).  Every other page is consumed without masks.
  const int jl = np - 1 - pb - w;
  const int i_tail = (L & (kPage - 1)) != 0 && np == pe && jl >= 0 && jl % kW == 0 ? jl / kW : -1;
  const int i_head = WIN && (lo & (kPage - 1)) != 0 && split == 0 && w == 0 ? 0 : -1;
  // the fused step: the iteration whose page (the sequence's last) takes the new row
  const int i_patch = STEP && patch && jl >= 0 && jl % kW == 0 ? jl / kW : -1;

  // One ring step: wait for stage `stage`, consume its page, refill it with iteration
  // i + S.  For the tensor-core paths the loop below unrolls the ring, so every stage
  // address is a constant.
  auto step = [&](int i, int stage, uint32_t phase) -> bool {
#ifdef PKV_TEST_HOOKS
    if (i == 0 && g_test_fail_first_wait) return false;  // a wait that gives up at once
#endif
    if (!mbar_wait_warp(bar0 + 8 * stage, phase)) return false;
    uint8_t* sp = my_stages + stage * Lo::stageBytes;
    const int j0 = pb + w + i * kW;  // the block's page
    if constexpr (STEP) {
      // the fused step: the new token replaces whatever the cache held at its slot
      if (i == i_patch) {
        constexpr int RB = RowBytes<KVT, D>::value;
        uint8_t* pg = my_stages + stage * Lo::stageBytes;
        const uint8_t* nk = nrow;
        const uint8_t* nv = nrow + RB + 16;
        if constexpr (KVT == kINT4) {
          if (lane < D / 8)
            reinterpret_cast<uint32_t*>(pg + t_new * (D / 2))[lane] = reinterpret_cast<const uint32_t*>(nk)[lane];
          for (int q = lane; q < D / 2; q += 32) pg[Lo::kBytes + q * kPage + int4_v_tpos(t_new)] = nv[q];
        } else {
          for (int d = lane; d < D; d += 32) {
            if constexpr (KVT == kINT8 || KVT == kFP8) {
              pg[t_new * D + d] = nk[d];
              pg[Lo::kBytes + d * kPage + t_new] = nv[d];
            } else if constexpr (KVT == kBF16) {
              *reinterpret_cast<__nv_bfloat16*>(pg + bf16_k_off(t_new, d, D)) =
                  reinterpret_cast<const __nv_bfloat16*>(nk)[d];
              *reinterpret_cast<__nv_bfloat16*>(pg + Lo::kBytes + bf16_v_off(d, t_new)) =
                  reinterpret_cast<const __nv_bfloat16*>(nv)[d];
            } else {
              reinterpret_cast<float*>(pg)[t_new * D + d] = reinterpret_cast<const float*>(nk)[d];
              reinterpret_cast<float*>(pg + Lo::kBytes)[d * kPage + t_new] =
                  reinterpret_cast<const float*>(nv)[d];
            }
          }
        }
        if constexpr (quantised(KVT)) {
          if (lane == 0) {
            reinterpret_cast<float*>(pg + 2 * Lo::kBytes)[t_new] = *reinterpret_cast<const float*>(nk + RB);
            reinterpret_cast<float*>(pg + 2 * Lo::kBytes + Lo::sBytes)[t_new] =
                *reinterpret_cast<const float*>(nv + RB);
          }
        }
        fence_proxy_async_smem();  // ordered before the stage's next bulk copy
        __syncwarp();
      }
    }
    const bool partial = i == i_tail || (WIN && i == i_head);
    if constexpr (quantised(KVT)) {
      int valid = kPage, lo_t = 0;
      if (partial) {
        valid = min(kPage, L - j0 * kPage);
        lo_t = WIN && j0 * kPage < lo ? lo - j0 * kPage : 0;
      }
      st.page(static_cast<uint32_t>(stage * Lo::stageBytes), partial, valid, lo_t, lane);
    } else {
      const int valid = min(kPage, L - j0 * kPage);
      // the window's first page (block 0, warp 0, iteration 0) skips the keys before it
      const int lo_t = WIN && j0 * kPage < lo ? lo - j0 * kPage : 0;
      if constexpr (KVT == kF32) {
        constexpr int HM = f32_head_cap<D>();
        switch (nh) {  // the FP32 path unrolls over the block's head count
          case 1: st.template page<1>(sp, probs, valid, lo_t, p.scale_log2, lane); break;
          case 2: st.template page<2>(sp, probs, valid, lo_t, p.scale_log2, lane); break;
          case 3: st.template page<3>(sp, probs, valid, lo_t, p.scale_log2, lane); break;
          case 4: st.template page<4>(sp, probs, valid, lo_t, p.scale_log2, lane); break;
          default: st.template page<HM>(sp, probs, valid, lo_t, p.scale_log2, lane); break;
        }
      } else {
        st.page(sp, valid, lo_t, lane);
      }
    }
    const int nxt = i + S;
    if (nxt < n_my) {
      if ((nxt & 31) == 0) {
        // the issue index enters a new batch of ids: it becomes the current one
        ids_cur = ids_nxt;
        ids_nxt = load_ids((nxt >> 5) + 1);
      }
      __syncwarp();
      issue(nxt, stage);
    }
    return true;
  };
  int i_fail = -1;  // the iteration whose wait gave up
  if constexpr (KVT == kF32) {
    // (the FP32 page code is large: a rolled ring keeps it in the instruction cache)
    int stage = 0;
    uint32_t phase = 0;
    for (int i = 0; i < n_my; ++i) {
      if (!step(i, stage, phase)) {
        i_fail = i;
        break;
      }
      if (++stage == S) {
        stage = 0;
        phase ^= 1u;
      }
    }
  } else {
    uint32_t ph = 0;
    for (int base = 0; base < n_my; base += S, ph ^= 1u) {
#pragma unroll
      for (int k = 0; k < S; ++k) {
        if (base + k >= n_my) break;
        if (!step(base + k, k, ph)) {
          i_fail = base + k;
          break;
        }
      }
      if (i_fail >= 0) break;
    }
  }
  if (i_fail >= 0) {
    werr |= 0x10;  // PKV_DEV_TIMEOUT
    // Drain (bounded) every copy this warp still has in flight before its stage memory is
    // reused or the block exits: the iteration whose wait gave up and the ones issued
    // after it (iterations i_fail .. i_fail + S - 1).
    const int last = min(n_my, i_fail + S);
    for (int k = i_fail; k < last; ++k)
      (void)mbar_wait_warp(bar0 + 8 * (k % S), static_cast<uint32_t>((k / S) & 1));
  }
  werr = __reduce_or_sync(0xffffffffu, werr);
  if (werr && lane == 0) atomicOr(&s_flag, werr);

  // ---- merge the warps' states (the stage memory is reused once every warp is done)
  __syncthreads();
  float* cm = reinterpret_cast<float*>(stages);
  float* cl = cm + kW * kMaxHeads;
  float* cO = cl + kW * kMaxHeads;
  st.store(cm + w * kMaxHeads, cl + w * kMaxHeads, cO + w * kMaxHeads * (D + 2), lane);
  __syncthreads();
  const int err = s_flag;
  if (tid == 0 && err && p.dev_status) atomicOr(p.dev_status, err);

  // Merge weights, once per (warp, head): exp2(m_w - M), divided by the total sum when
  // this block holds the whole sequence (NaN when the block met an error).
  float* fw = cO + kW * kMaxHeads * (D + 2);
  // on-chip split merge: this block's partial, max[8], sum[8], then O[8][D] (16-byte rows)
  float* part = fw + kW * kMaxHeads;
  const bool single = nsplit == 1;
  if (tid < nh) {
    const int r = tid;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int ww = 0; ww < kW; ++ww) M = fmaxf(M, cm[ww * kMaxHeads + r]);
    float f[kW], Ls = 0.f;
#pragma unroll
    for (int ww = 0; ww < kW; ++ww) {
      const float mw = cm[ww * kMaxHeads + r];
      f[ww] = mw == -CUDART_INF_F ? 0.f : fast_exp2(mw - M);
      Ls += cl[ww * kMaxHeads + r] * f[ww];
    }
    const size_t row = static_cast<size_t>(b) * p.Hq + h0 + r;
    if (single) {
      const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
#pragma unroll
      for (int ww = 0; ww < kW; ++ww) fw[ww * kMaxHeads + r] = err ? CUDART_NAN_F : f[ww] * inv;
    } else {
#pragma unroll
      for (int ww = 0; ww < kW; ++ww) fw[ww * kMaxHeads + r] = f[ww];
      if (p.cluster) {
        part[r] = err ? CUDART_NAN_F : M;
        part[kMaxHeads + r] = Ls;
      } else {
        const size_t prow = static_cast<size_t>(split) * p.B * p.Hq + row;
        p.ws_m[prow] = err ? CUDART_NAN_F : M;
        p.ws_l[prow] = Ls;
      }
    }
  }
  __syncthreads();
  for (int idx = tid; idx < nh * D; idx += kThreads) {
    const int r = idx / D, d = idx % D;
    float O = 0.f;
#pragma unroll
    for (int ww = 0; ww < kW; ++ww) O += cO[(ww * kMaxHeads + r) * (D + 2) + d] * fw[ww * kMaxHeads + r];
    const size_t row = static_cast<size_t>(b) * p.Hq + h0 + r;
    if (single) {
      p.out[row * D + d] = O;
    } else if (p.cluster) {
      part[2 * kMaxHeads + r * D + d] = O;
    } else {
      p.ws_o[(static_cast<size_t>(split) * p.B * p.Hq + row) * D + d] = O;
    }
  }
  if (single) return;
  if (p.cluster) {
    cluster_merge<D, kThreads>(p, part, nsplit, b, h0, nh, tid, lane, w, &s_done, &s_release,
                               &s_last);
    return;
  }

  // ---- split-K: the last block of this (sequence, head group) merges all partials
  __threadfence();
  __syncthreads();
  int* ticket = p.ws_ticket + static_cast<size_t>(b) * p.Hkv * p.head_groups + z;
  if (tid == 0) s_last = atomicAdd(ticket, 1) == nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  // The merge.  Each thread owns 4 consecutive outputs of one or two heads; it issues the
  // 16-byte loads of its first 8 splits' partial outputs first, so that they are in
  // flight together with the (max, sum) loads: warp w reads the (max, sum) of every split
  // for heads w and w + 4 in one round trip and reduces them by shuffles into weights in
  // shared memory.  Further splits follow in batches of 8, added in split order.
  {
    float* wts = reinterpret_cast<float*>(stages);  // [nsplit][8] weights, then [8] 1/L
    float* lsm = wts + (nsplit + 1) * kMaxHeads;    // [nsplit][8] partial sums
    const size_t stride = static_cast<size_t>(p.B) * p.Hq;
    const size_t row0 = static_cast<size_t>(b) * p.Hq + h0;
    constexpr int D4 = D / 4;
    constexpr int CPT = (kMaxHeads * D4 + kThreads - 1) / kThreads;  // chunks per thread
    constexpr int SB = 8;                                             // splits per batch
    const size_t sstride = stride * D4;  // float4s from one split's partial to the next
    const float4* src[CPT];
    int rr[CPT];
    bool act[CPT];
    float4 acc[CPT];
    float4 v[CPT][SB];
    // (the register-bound coded kernels with head_dim 64 issue them after the weights)
    constexpr bool kEarly = !(quantised(KVT) && D == 64);
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int cidx = tid + c * kThreads;
      act[c] = cidx < nh * D4;
      rr[c] = act[c] ? cidx / D4 : 0;
      src[c] = reinterpret_cast<const float4*>(p.ws_o + (row0 + rr[c]) * D) + (act[c] ? cidx % D4 : 0);
      acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      if constexpr (kEarly) {
#pragma unroll
        for (int k = 0; k < SB; ++k)
          v[c][k] = act[c] && k < nsplit ? __ldcg(src[c] + k * sstride) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    __syncthreads();
    for (int r = w; r < nh; r += kW) {
      float M = -CUDART_INF_F;
      bool poisoned = false;
      for (int s = lane; s < nsplit; s += 32) {
        const float ms = __ldcg(p.ws_m + s * stride + row0 + r);
        const float ls = __ldcg(p.ws_l + s * stride + row0 + r);
        poisoned |= isnan(ms);
        M = fmaxf(M, ms);
        wts[s * kMaxHeads + r] = ms;
        lsm[s * kMaxHeads + r] = ls;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
      poisoned = __any_sync(0xffffffffu, poisoned);
      float Ls = 0.f;
      for (int s = lane; s < nsplit; s += 32) {
        const float ms = wts[s * kMaxHeads + r];
        const float f = ms == -CUDART_INF_F ? 0.f : fast_exp2(ms - M);
        wts[s * kMaxHeads + r] = f;
        Ls += lsm[s * kMaxHeads + r] * f;
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) Ls += __shfl_xor_sync(0xffffffffu, Ls, o);
      if (lane == 0) wts[nsplit * kMaxHeads + r] = poisoned ? CUDART_NAN_F : (Ls > 0.f ? 1.f / Ls : 0.f);
    }
    __syncthreads();
    for (int s0 = 0; s0 < nsplit; s0 += SB) {
      if (s0 > 0 || !kEarly) {
#pragma unroll
        for (int c = 0; c < CPT; ++c)
#pragma unroll
          for (int k = 0; k < SB; ++k)
            v[c][k] = act[c] && s0 + k < nsplit ? __ldcg(src[c] + (s0 + k) * sstride)
                                                : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int c = 0; c < CPT; ++c)
#pragma unroll
        for (int k = 0; k < SB; ++k) {
          if (s0 + k < nsplit) {
            const float wt = wts[(s0 + k) * kMaxHeads + rr[c]];
            acc[c].x += v[c][k].x * wt;
            acc[c].y += v[c][k].y * wt;
            acc[c].z += v[c][k].z * wt;
            acc[c].w += v[c][k].w * wt;
          }
        }
    }
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      if (!act[c]) continue;
      const int cidx = tid + c * kThreads;
      const float inv = wts[nsplit * kMaxHeads + rr[c]];
      float* dst = p.out + (row0 + rr[c]) * D + 4 * (cidx % D4);
      dst[0] = acc[c].x * inv;
      dst[1] = acc[c].y * inv;
      dst[2] = acc[c].z * inv;
      dst[3] = acc[c].w * inv;
    }
  }
  if (tid == 0) *ticket = 0;  // leave the counter ready for the next call
}

template <int KVT, int D, bool STEP, bool WIN>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&decode_kernel<KVT, D, STEP, WIN>);
}

struct Variant {
  const void* fn;
  int smem;
  int index;
  int max_splits;  // the last block's merge keeps (2 splits + 1) x 8 floats in shared memory
  int warps;       // warps per block
};

template <int KVT, int D>
constexpr int max_splits_of() {
  return Smem<KVT, D>::big / (2 * kMaxHeads * 4) - 1;
}

#define PKV_VARIANT(T, D, ST, WN, I)                                                        \
  {kernel_ptr<T, D, ST, WN>(), Smem<T, D, ST>::total, I, max_splits_of<T, D>(), \
   Tune<T, D>::W}
// index: dtype-and-head-dim slot (0 .. 9), + 10 for the fused decode step, + 20 for the
// sliding window
constexpr int kVariants = 40;
Variant variant(int dtype, int D, bool step, bool win) {
  switch (dtype * 1000 + D + (step ? 100000 : 0) + (win ? 1000000 : 0)) {
#define PKV_VARIANTS_OF(ST, WN, BASE, KEY)                                                \
    case KEY + kF32 * 1000 + 64: return PKV_VARIANT(kF32, 64, ST, WN, BASE + 0);          \
    case KEY + kF32 * 1000 + 128: return PKV_VARIANT(kF32, 128, ST, WN, BASE + 1);        \
    case KEY + kBF16 * 1000 + 64: return PKV_VARIANT(kBF16, 64, ST, WN, BASE + 2);        \
    case KEY + kBF16 * 1000 + 128: return PKV_VARIANT(kBF16, 128, ST, WN, BASE + 3);      \
    case KEY + kINT8 * 1000 + 64: return PKV_VARIANT(kINT8, 64, ST, WN, BASE + 4);        \
    case KEY + kINT8 * 1000 + 128: return PKV_VARIANT(kINT8, 128, ST, WN, BASE + 5);      \
    case KEY + kFP8 * 1000 + 64: return PKV_VARIANT(kFP8, 64, ST, WN, BASE + 6);          \
    case KEY + kFP8 * 1000 + 128: return PKV_VARIANT(kFP8, 128, ST, WN, BASE + 7);        \
    case KEY + kINT4 * 1000 + 64: return PKV_VARIANT(kINT4, 64, ST, WN, BASE + 8);        \
    case KEY + kINT4 * 1000 + 128: return PKV_VARIANT(kINT4, 128, ST, WN, BASE + 9);
    PKV_VARIANTS_OF(false, false, 0, 0)
    PKV_VARIANTS_OF(true, false, 10, 100000)
    PKV_VARIANTS_OF(false, true, 20, 1000000)
    PKV_VARIANTS_OF(true, true, 30, 1100000)
#undef PKV_VARIANTS_OF
    default: return {nullptr, 0, -1, 1, 4};
  }
}
#undef PKV_VARIANT

// Per-device facts queried once: SM count, and for each kernel variant its resident
// blocks per SM (after raising its dynamic shared-memory limit).
constexpr int kMaxDevices = 64;
constexpr int kMaxCluster = 8;  // portable cluster size: the largest on-chip split merge
struct DevInfo {
  int sms = 0;
  int occ[kVariants] = {};
  // clusters of n blocks of the variant that can be resident at once (-1: not asked yet)
  int clusters[kVariants][kMaxCluster + 1];
  DevInfo() {
    for (auto& v : clusters)
      for (int& c : v) c = -1;
  }
};
DevInfo g_dev[kMaxDevices];
std::mutex g_dev_mu;

bool device_facts(int device, const Variant& v, int* sms, int* occ) {
  if (device < 0 || device >= kMaxDevices || v.index < 0) return false;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DevInfo& d = g_dev[device];
  if (d.sms == 0 &&
      cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return false;
  if (d.occ[v.index] == 0) {
    int o = 0;
    if (cudaFuncSetAttribute(v.fn, cudaFuncAttributeMaxDynamicSharedMemorySize, v.smem) !=
            cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, v.fn, v.warps * 32, v.smem) !=
            cudaSuccess)
      return false;
    d.occ[v.index] = o > 0 ? o : 1;
  }
  *sms = d.sms;
  *occ = d.occ[v.index];
  return true;
}

// How many clusters of n blocks of variant v can be resident at once on `device` (asked
// once; 0 if none can be launched).
int clusters_resident(int device, const Variant& v, int n) {
  if (device < 0 || device >= kMaxDevices || v.index < 0 || n < 2 || n > kMaxCluster) return 0;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  int& c = g_dev[device].clusters[v.index][n];
  if (c < 0) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(n, 1, 1);
    cfg.blockDim = dim3(v.warps * 32);
    cfg.dynamicSmemBytes = v.smem;
    cudaLaunchAttribute attr{};
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = n;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int num = 0;
    if (cudaOccupancyMaxActiveClusters(&num, v.fn, &cfg) != cudaSuccess) {
      (void)cudaGetLastError();
      num = 0;
    }
    c = num;
  }
  return c;
}

}  // namespace

bool plan_decode(const CacheView& c, int B, int Hq, int MB, int q_dtype, int device,
                 int chunk_override, DecodePlan* plan, bool step) {
  (void)q_dtype;
  const Variant v = variant(c.dtype, c.D, step, c.window > 0);
  if (!v.fn) return false;
  const int G = Hq / c.Hkv;
  const int cap = (c.dtype == kF32 && c.D == 128) ? f32_head_cap<128>() : kMaxHeads;
  plan->heads_per_cta = G < cap ? G : cap;
  plan->head_groups = (G + plan->heads_per_cta - 1) / plan->heads_per_cta;
  // pages a sequence's keys can span: the table width, or under a sliding window of W
  // tokens at most ceil((W - 1) / 16) + 1
  int mb = MB > 0 ? MB : 1;
  if (c.window > 0) {
    const long long span = (static_cast<long long>(c.window) + kPage - 2) / kPage + 1;
    if (span < mb) mb = static_cast<int>(span);
  }
  int sms = 0, occ = 0;
  if (!device_facts(device, v, &sms, &occ)) return false;
  int chunk;
  if (chunk_override > 0) {
    chunk = chunk_override;
  } else {
    // When the (sequence, head group) units alone nearly fill the resident block slots,
    // do not split: merges cost more than the last partial wave.  Otherwise aim for
    // about two blocks per slot at full table length, with at least 8 pages per warp and
    // at most 32 splits, so that the partial merge stays short.
    const long long units = static_cast<long long>(B) * c.Hkv * plan->head_groups;
    const long long slots = static_cast<long long>(sms) * occ;
    long long splits = 1;
    if (units > 0 && 4 * units < 3 * slots) {
      splits = (2 * slots + units - 1) / units;
      const long long by_len = mb / (8 * v.warps);
      if (splits > by_len) splits = by_len;
      if (splits > 32) splits = 32;
      if (splits < 1) splits = 1;
    }
    chunk = static_cast<int>((mb + splits - 1) / splits);
  }
  if (chunk < 1) chunk = 1;
  if ((mb + chunk - 1) / chunk > v.max_splits) chunk = (mb + v.max_splits - 1) / v.max_splits;
  plan->chunk_pages = chunk;
  plan->n_splits = (mb + chunk - 1) / chunk;
  // Up to kMaxCluster splits merge on chip (a cluster per sequence and head group, no
  // workspace) when every cluster of the launch is resident at once (a cluster is placed
  // whole on one GPC, so fewer clusters than slots / n fit, and a second wave of clusters
  // costs far more than the merge saves); otherwise the splits merge through the
  // workspace and the last-arriving block.
  const long long units_all = static_cast<long long>(B) * c.Hkv * plan->head_groups;
  plan->cluster = plan->n_splits > 1 && plan->n_splits <= kMaxCluster &&
                  units_all <= clusters_resident(device, v, plan->n_splits);
  size_t ws = 0;
  if (plan->n_splits > 1 && !plan->cluster) {
    const size_t rows = static_cast<size_t>(plan->n_splits) * B * Hq;
    const size_t tickets = static_cast<size_t>(B) * c.Hkv * plan->head_groups;
    ws = ((tickets * 4 + 255) / 256) * 256 + rows * (c.D + 2) * 4;
  }
  plan->ws_bytes = ws;
  return true;
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st) {
  const Variant v = variant(a.c.dtype, a.c.D, a.step, a.c.window > 0);
  if (!v.fn) return cudaErrorInvalidValue;
  DParams p{};
  p.k = static_cast<const uint8_t*>(a.c.k);
  p.v = static_cast<const uint8_t*>(a.c.v);
  p.ks = a.c.ks;
  p.vs = a.c.vs;
  p.q = a.q;
  p.bt = a.block_tables;
  p.lens = a.context_lens;
  p.out = a.out;
  p.dev_status = a.dev_status;
  p.q_dtype = a.q_dtype;
  p.Hkv = a.c.Hkv;
  p.Hq = a.Hq;
  p.G = a.Hq / a.c.Hkv;
  p.hpc = plan.heads_per_cta;
  p.head_groups = plan.head_groups;
  p.MB = a.MB;
  p.B = a.B;
  p.num_pages = a.c.num_pages;
  p.chunk = plan.chunk_pages;
  p.window = a.c.window;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  if (a.step) {
    p.kw = static_cast<uint8_t*>(a.kw);
    p.vw = static_cast<uint8_t*>(a.vw);
    p.ksw = a.ksw;
    p.vsw = a.vsw;
    p.k_new = a.k_new;
    p.v_new = a.v_new;
    p.new_dtype = a.new_dtype;
    p.slots = a.slots;
    p.positions = a.positions;
    if (a.positions) {
      for (int i = 0; i < a.c.D / 2; ++i) p.inv_freq[i] = std::pow(a.rope_theta, -2.0 * i / a.c.D);
    }
  }
  p.cluster = plan.cluster;
  if (plan.n_splits > 1 && !plan.cluster) {
    const size_t tickets = static_cast<size_t>(a.B) * a.c.Hkv * plan.head_groups;
    uint8_t* base = static_cast<uint8_t*>(a.ws);
    p.ws_ticket = reinterpret_cast<int*>(base);
    const size_t rows = static_cast<size_t>(plan.n_splits) * a.B * a.Hq;
    float* f = reinterpret_cast<float*>(base + ((tickets * 4 + 255) / 256) * 256);
    p.ws_o = f;  // [split][seq][head][D]: 16-byte aligned rows for the merge's loads
    p.ws_m = f + rows * a.c.D;
    p.ws_l = p.ws_m + rows;
  }
  // (the shared-memory limit was raised by plan_decode on this device)
  const dim3 grid(plan.n_splits, a.B, a.c.Hkv * plan.head_groups);
  void* args[] = {&p};
  if (!plan.cluster) return cudaLaunchKernel(v.fn, grid, dim3(v.warps * 32), args, v.smem, st);
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(v.warps * 32);
  cfg.dynamicSmemBytes = v.smem;
  cfg.stream = st;
  cudaLaunchAttribute attr{};
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = plan.n_splits;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, v.fn, args);
}

}  // namespace pkv

#ifdef PKV_TEST_HOOKS
// Test builds only: switches the give-up-at-once first wait (see above) on or off.
extern "C" int pkv_test_fail_first_wait(int on) {
  return cudaMemcpyToSymbol(pkv::g_test_fail_first_wait, &on, sizeof(int)) == cudaSuccess ? 0 : 1;
}
#endif
