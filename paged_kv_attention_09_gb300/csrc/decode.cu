// decode.cu — batched paged decode attention with split-K over pages.
//
// Sources: "mini-llm-inference-engine" README (true batched decode, one launch for the
// whole batch); "tinyloop Current Status" (paged attention with 16-token pages; GQA);
// "Tiny-LLM-Inference Project_Status" (FP32 default KV, dedicated BF16 paged kernel,
// FP32 operator boundaries).  The attention is the textbook softmax(scale q.K^T) V,
// evaluated with a running max / running sum (online softmax) so that every K/V byte is
// read from HBM exactly once.
//
// Thread-block layout: grid (split, sequence, kv-head x head-group).  A block owns up to
// 8 query heads that share one kv head, and a contiguous range of the sequence's
// logical pages.  Each of its 4 warps streams every 4th page of that range through its
// own ring of shared-memory stages filled by 1-D bulk copies (TMA engine, one copy per
// K block and per V block of a (page, kv-head)), so each warp keeps several pages in
// flight without any block-wide synchronisation.  Warps merge their (max, sum, acc)
// states at the end; when a sequence is split over several blocks, the block that
// arrives last (an atomic ticket, no waiting) merges the partial states in split order.
//
// Two compute paths:
//   FP32 KV  — CUDA cores.  8 lanes per token compute the q.k dot products (3 shuffle
//              steps), lanes own head_dim columns for P.V.
//   BF16/INT8 KV — warp-level tensor-core MMA (m16n8k16).  The query heads of the group
//              form the A rows (high part in rows 0-7, the rounding remainder in rows
//              8-15, so the product is accurate to ~2^-16 relative), a 16-token page
//              forms two n8 tiles of keys.  INT8 codes are converted exactly to f16
//              (|code| <= 127); per-token scales are applied to the scores (K) and to the
//              probabilities (V) in FP32.
// The order of every floating-point reduction depends only on logical token positions,
// the split size and the warp count, so results are bit-identical under any physical
// page permutation.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kW = 4;            // warps per block
constexpr int kThreads = kW * 32;
constexpr int kMaxHeads = 8;     // query heads per block

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
  float scale_log2;
};

template <int KVT>
struct ElemSize {
  static constexpr int value = KVT == kF32 ? 4 : (KVT == kBF16 ? 2 : 1);
};

template <int KVT, int D>
struct Layout {
  static constexpr int esz = ElemSize<KVT>::value;
  static constexpr int kBytes = kPage * D * esz;          // K block of one (page, head)
  static constexpr int vBytes = kPage * D * esz;          // V block of one (page, head)
  static constexpr int sBytes = KVT == kINT8 ? kPage * 4 : 0;  // one scale vector
  static constexpr int stageBytes = kBytes + vBytes + 2 * sBytes;
};

template <int KVT, int D, int S>
struct Smem {
  using Lo = Layout<KVT, D>;
  static constexpr int stages = kW * S * Lo::stageBytes;
  static constexpr int combine = kW * kMaxHeads * (D + 2) * 4;
  static constexpr int big = stages > combine ? stages : combine;
  static constexpr int probs = KVT == kF32 ? kW * kMaxHeads * kPage * 4 : 0;
  static constexpr int bars = kW * S * 8;
  static constexpr int total = big + probs + bars;
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

  __device__ void init(const DParams& p, int b, int h0, int nh, int lane) {
    const int c8 = lane & 7;
#pragma unroll
    for (int h = 0; h < HM; ++h) {
      m[h] = -CUDART_INF_F;
      l[h] = 0.f;
#pragma unroll
      for (int i = 0; i < NC; ++i) {
        o[h][i] = 0.f;
        q[h][i] = h < nh ? load_q4(p.q, p.q_dtype,
                                   (static_cast<size_t>(b) * p.Hq + h0 + h) * D + (c8 + 8 * i) * 4)
                         : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
  }

  template <int NH>
  __device__ void page(const uint8_t* st, float* probs, int valid, float sl, int lane) {
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
        s[ps][h] = t < valid ? a * sl : -CUDART_INF_F;
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
        if (valid < kPage) {  // padding tokens may hold anything (even NaN): zero them
          const int t0 = c4 * 4;
          vv.x = t0 + 0 < valid ? vv.x : 0.f;
          vv.y = t0 + 1 < valid ? vv.y : 0.f;
          vv.z = t0 + 2 < valid ? vv.z : 0.f;
          vv.w = t0 + 3 < valid ? vv.w : 0.f;
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

// ------------------------------------------------------------------ BF16 / INT8 (MMA)

template <int KVT, int D>
struct MmaWarp {
  static constexpr int KS = D / 16;  // k-steps of the q.k product
  static constexpr int NT = D / 8;   // n-tiles of the P.V product
  uint32_t qa[KS][4];
  float o[NT][4];
  float m, l, row_scale;

  // Which head_dim index the k-slot pair {2c, 2c+1} of k-step ks refers to.  The
  // k-slot -> d map is a permutation chosen so that each lane's K operand is one
  // contiguous 16-byte shared-memory load; q uses the same map.
  __device__ static int kslot_d(int ks, int c) {
    if constexpr (KVT == kINT8) return 64 * (ks >> 2) + 16 * c + 4 * (ks & 3);
    else return 32 * (ks >> 1) + 8 * c + 4 * (ks & 1);
  }

  __device__ void init(const DParams& p, int b, int h0, int nh, int lane) {
    const int r = lane >> 2, c = lane & 3;
    const bool has = r < nh;
    float4 qv[KS];
    float qmax = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      qv[ks] = has ? load_q4(p.q, p.q_dtype,
                             (static_cast<size_t>(b) * p.Hq + h0 + r) * D + kslot_d(ks, c))
                   : make_float4(0.f, 0.f, 0.f, 0.f);
      qmax = fmaxf(qmax, fmaxf(fmaxf(fabsf(qv[ks].x), fabsf(qv[ks].y)),
                               fmaxf(fabsf(qv[ks].z), fabsf(qv[ks].w))));
    }
    row_scale = p.scale_log2;
    if constexpr (KVT == kINT8) {
      // f16 operands: bring the row's largest |q| into [0.5, 1) by an exact power of two
      // and fold the factor into the score scale.
      qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 1));
      qmax = fmaxf(qmax, __shfl_xor_sync(0xffffffffu, qmax, 2));
      int e = 0;
      if (qmax > 0.f) frexpf(qmax, &e);
      row_scale = ldexpf(p.scale_log2, e);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const float x[4] = {ldexpf(qv[ks].x, -e), ldexpf(qv[ks].y, -e), ldexpf(qv[ks].z, -e),
                            ldexpf(qv[ks].w, -e)};
        __half hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          hi[j] = __float2half_rn(x[j]);
          lo[j] = __float2half_rn(x[j] - __half2float(hi[j]));
        }
        qa[ks][0] = pack_half2(hi[0], hi[1]);
        qa[ks][1] = pack_half2(lo[0], lo[1]);
        qa[ks][2] = pack_half2(hi[2], hi[3]);
        qa[ks][3] = pack_half2(lo[2], lo[3]);
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const float x[4] = {qv[ks].x, qv[ks].y, qv[ks].z, qv[ks].w};
        __nv_bfloat16 hi[4], lo[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          hi[j] = __float2bfloat16_rn(x[j]);
          lo[j] = __float2bfloat16_rn(x[j] - __bfloat162float(hi[j]));
        }
        qa[ks][0] = pack_bf162(hi[0], hi[1]);
        qa[ks][1] = pack_bf162(lo[0], lo[1]);
        qa[ks][2] = pack_bf162(hi[2], hi[3]);
        qa[ks][3] = pack_bf162(lo[2], lo[3]);
      }
    }
    m = -CUDART_INF_F;
    l = 0.f;
#pragma unroll
    for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  }

  __device__ void page(const uint8_t* st, int valid, int lane) {
    using Lo = Layout<KVT, D>;
    const int r = lane >> 2, c = lane & 3;
    const uint8_t* Ks = st;
    const uint8_t* Vs = st + Lo::kBytes;
    // ---- S = Q K^T over the page's 16 tokens: n-tile j column n holds token
    //      4(n/2) + 2j + (n%2), so lane (r, c) ends up with tokens 4c .. 4c+3.
    float sacc[2][4];
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      sacc[j][0] = sacc[j][1] = sacc[j][2] = sacc[j][3] = 0.f;
      const int tok = 4 * (r >> 1) + (r & 1) + 2 * j;
      const uint8_t* krow = Ks + tok * D * Lo::esz;
      if constexpr (KVT == kINT8) {
#pragma unroll
        for (int blk = 0; blk < D / 64; ++blk) {
          const uint4 w = *reinterpret_cast<const uint4*>(krow + blk * 64 + c * 16);
          const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
          for (int s = 0; s < 4; ++s) {
            uint32_t b0, b1;
            s8x4_to_f16x4(ws[s], b0, b1);
            mma_f16(sacc[j], qa[4 * blk + s], b0, b1);
          }
        }
      } else {
#pragma unroll
        for (int blk = 0; blk < D / 32; ++blk) {
          const uint4 w = *reinterpret_cast<const uint4*>(krow + (blk * 32 + c * 8) * 2);
          mma_bf16(sacc[j], qa[2 * blk + 0], w.x, w.y);
          mma_bf16(sacc[j], qa[2 * blk + 1], w.z, w.w);
        }
      }
    }
    float x[4];
    x[0] = (sacc[0][0] + sacc[0][2]) * row_scale;
    x[1] = (sacc[0][1] + sacc[0][3]) * row_scale;
    x[2] = (sacc[1][0] + sacc[1][2]) * row_scale;
    x[3] = (sacc[1][1] + sacc[1][3]) * row_scale;
    float vsc[4] = {1.f, 1.f, 1.f, 1.f};
    if constexpr (KVT == kINT8) {
      const float4 k4 = *reinterpret_cast<const float4*>(st + 2 * Lo::kBytes + c * 16);
      const float4 v4 = *reinterpret_cast<const float4*>(st + 2 * Lo::kBytes + Lo::sBytes + c * 16);
      x[0] *= k4.x; x[1] *= k4.y; x[2] *= k4.z; x[3] *= k4.w;
      vsc[0] = v4.x; vsc[1] = v4.y; vsc[2] = v4.z; vsc[3] = v4.w;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) x[i] = (4 * c + i) < valid ? x[i] : -CUDART_INF_F;
    // ---- online softmax (rows r and r+8 both belong to head r)
    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(m, mx);
    const float corr = fast_exp2(m - mn);
    m = mn;
    float pr[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) pr[i] = fast_exp2(x[i] - mn);
    l = l * corr + (pr[0] + pr[1]) + (pr[2] + pr[3]);
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      o[j][0] *= corr; o[j][1] *= corr; o[j][2] *= corr; o[j][3] *= corr;
    }
    // ---- P.V: A rows r = high part, r+8 = remainder; k = the page's 16 tokens.
    uint32_t pa[4];
    if constexpr (KVT == kINT8) {
      __half hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float pp = (4 * c + i) < valid ? pr[i] * vsc[i] : 0.f;
        hi[i] = __float2half_rn(pp);
        lo[i] = __float2half_rn(pp - __half2float(hi[i]));
      }
      pa[0] = pack_half2(hi[0], hi[1]);
      pa[1] = pack_half2(lo[0], lo[1]);
      pa[2] = pack_half2(hi[2], hi[3]);
      pa[3] = pack_half2(lo[2], lo[3]);
    } else {
      __nv_bfloat16 hi[4], lo[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        hi[i] = __float2bfloat16_rn(pr[i]);
        lo[i] = __float2bfloat16_rn(pr[i] - __bfloat162float(hi[i]));
      }
      pa[0] = pack_bf162(hi[0], hi[1]);
      pa[1] = pack_bf162(lo[0], lo[1]);
      pa[2] = pack_bf162(hi[2], hi[3]);
      pa[3] = pack_bf162(lo[2], lo[3]);
    }
    uint32_t vmask0 = 0xffffffffu, vmask1 = 0xffffffffu;
    if constexpr (KVT == kBF16) {
      if (valid < kPage) {  // padding tokens may hold NaN: zero their V entries
        vmask0 = (4 * c + 0 < valid ? 0x0000ffffu : 0u) | (4 * c + 1 < valid ? 0xffff0000u : 0u);
        vmask1 = (4 * c + 2 < valid ? 0x0000ffffu : 0u) | (4 * c + 3 < valid ? 0xffff0000u : 0u);
      }
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      const int d = 8 * j + r;
      if constexpr (KVT == kINT8) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(Vs + d * kPage + 4 * c);
        uint32_t b0, b1;
        s8x4_to_f16x4(w, b0, b1);
        mma_f16(o[j], pa, b0, b1);
      } else {
        const uint2 w = *reinterpret_cast<const uint2*>(Vs + (d * kPage + 4 * c) * 2);
        mma_bf16(o[j], pa, w.x & vmask0, w.y & vmask1);
      }
    }
  }

  __device__ void store(float* cm, float* cl, float* cO, int lane) {
    const int r = lane >> 2, c = lane & 3;
    float lt = l;
    lt += __shfl_xor_sync(0xffffffffu, lt, 1);
    lt += __shfl_xor_sync(0xffffffffu, lt, 2);
    if (c == 0) {
      cm[r] = m;
      cl[r] = lt;
    }
#pragma unroll
    for (int j = 0; j < NT; ++j) {
      cO[r * (D + 2) + 8 * j + 2 * c + 0] = o[j][0] + o[j][2];
      cO[r * (D + 2) + 8 * j + 2 * c + 1] = o[j][1] + o[j][3];
    }
  }
};

template <int KVT, int D>
struct WarpOf {
  using type = MmaWarp<KVT, D>;
};
template <int D>
struct WarpOf<kF32, D> {
  using type = F32Warp<D>;
};

// ------------------------------------------------------------------ the kernel

template <int KVT, int D, int S>
__global__ void __launch_bounds__(kThreads)
    decode_kernel(const __grid_constant__ DParams p) {
  using Lo = Layout<KVT, D>;
  using Sm = Smem<KVT, D, S>;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* stages = smem;
  float* probs_all = reinterpret_cast<float*>(smem + Sm::big);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::big + Sm::probs);
  __shared__ int s_flag, s_last;

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int split = blockIdx.x, b = blockIdx.y, z = blockIdx.z;
  const int g = z / p.head_groups, hg = z % p.head_groups;
  const int h0 = g * p.G + hg * p.hpc;
  const int nh = min(p.hpc, p.G - hg * p.hpc);

  const int L = p.lens[b];
  const bool len_ok = L >= 0 && L <= p.MB * kPage;
  const int np = len_ok ? (L + kPage - 1) / kPage : 0;
  const int nsplit = len_ok ? max(1, (np + p.chunk - 1) / p.chunk) : 1;
  if (split >= nsplit) return;
  const int pb = split * p.chunk, pe = min(np, pb + p.chunk);
  const int32_t* bt = p.bt + static_cast<size_t>(b) * p.MB;

  // Validate this block's page ids before any copy is issued.
  if (tid == 0) s_flag = len_ok ? 0 : 0x2 /*PKV_DEV_BAD_LEN*/;
  __syncthreads();
  for (int j = pb + tid; j < pe; j += kThreads) {
    const int pg = bt[j];
    if (pg < 0 || pg >= p.num_pages) atomicOr(&s_flag, 0x1 /*PKV_DEV_BAD_PAGE*/);
  }
  __syncthreads();
  const int bad = s_flag;

  typename WarpOf<KVT, D>::type st;
  uint8_t* my_stages = stages + static_cast<size_t>(w) * S * Lo::stageBytes;
  uint64_t* my_bars = bars + w * S;
  float* probs = probs_all + w * kMaxHeads * kPage;
  bool timed_out = false;
  st.init(p, b, h0, nh, lane);

  if (!bad) {
    const int span = pe - pb;
    const int n_my = span > w ? (span - w + kW - 1) / kW : 0;
    if (lane == 0) {
      for (int i = 0; i < S; ++i) mbar_init(&my_bars[i], 1);
      fence_barrier_init();
    }
    __syncwarp();
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int i) {
      const int j = pb + w + i * kW;
      const size_t blk = static_cast<size_t>(bt[j]) * p.Hkv + g;
      uint8_t* dst = my_stages + (i % S) * Lo::stageBytes;
      uint64_t* bar = &my_bars[i % S];
      mbar_arrive_expect_tx(bar, Lo::stageBytes);
      bulk_g2s(dst, p.k + blk * Lo::kBytes, Lo::kBytes, bar, pol);
      bulk_g2s(dst + Lo::kBytes, p.v + blk * Lo::vBytes, Lo::vBytes, bar, pol);
      if constexpr (KVT == kINT8) {
        bulk_g2s(dst + 2 * Lo::kBytes, p.ks + blk * kPage, Lo::sBytes, bar, pol);
        bulk_g2s(dst + 2 * Lo::kBytes + Lo::sBytes, p.vs + blk * kPage, Lo::sBytes, bar, pol);
      }
    };
    if (lane == 0) {
      for (int i = 0; i < min(S, n_my); ++i) issue(i);
    }
    int i = 0;
    for (; i < n_my; ++i) {
      const bool ok = mbar_wait(&my_bars[i % S], (i / S) & 1);
      if (!__all_sync(0xffffffffu, ok)) {
        timed_out = true;
        break;
      }
      const int j = pb + w + i * kW;
      const int valid = min(kPage, L - j * kPage);
      const uint8_t* sp = my_stages + (i % S) * Lo::stageBytes;
      if constexpr (KVT == kF32) {
        constexpr int HM = f32_head_cap<D>();
        switch (nh) {  // the FP32 path unrolls over the block's head count
          case 1: st.template page<1>(sp, probs, valid, p.scale_log2, lane); break;
          case 2: st.template page<2>(sp, probs, valid, p.scale_log2, lane); break;
          case 3: st.template page<3>(sp, probs, valid, p.scale_log2, lane); break;
          case 4: st.template page<4>(sp, probs, valid, p.scale_log2, lane); break;
          default: st.template page<HM>(sp, probs, valid, p.scale_log2, lane); break;
        }
      } else {
        st.page(sp, valid, lane);
      }
      __syncwarp();
      if (lane == 0 && i + S < n_my) issue(i + S);
    }
    if (timed_out) {
      // Drain (bounded) whatever this warp still has in flight before leaving.
      for (int k = i + 1; k < min(n_my, i + S); ++k) (void)mbar_wait(&my_bars[k % S], (k / S) & 1);
    }
  }
  if (timed_out && lane == 0) atomicOr(&s_flag, 0x10 /*PKV_DEV_TIMEOUT*/);

  // ---- merge the warps' states (the stage memory is reused once every warp is done)
  __syncthreads();
  float* cm = reinterpret_cast<float*>(stages);
  float* cl = cm + kW * kMaxHeads;
  float* cO = cl + kW * kMaxHeads;
  // Combine area: cm[kW][8], cl[kW][8], cO[kW][8][D+2] (fits in the stage area).
  st.store(cm + w * kMaxHeads, cl + w * kMaxHeads, cO + w * kMaxHeads * (D + 2), lane);
  __syncthreads();
  const int err = s_flag;
  if (tid == 0 && err && p.dev_status) atomicOr(p.dev_status, err);

  const bool single = nsplit == 1;
  for (int idx = tid; idx < nh * D; idx += kThreads) {
    const int r = idx / D, d = idx % D;
    float M = -CUDART_INF_F;
#pragma unroll
    for (int ww = 0; ww < kW; ++ww) M = fmaxf(M, cm[ww * kMaxHeads + r]);
    float Ls = 0.f, O = 0.f;
#pragma unroll
    for (int ww = 0; ww < kW; ++ww) {
      const float mw = cm[ww * kMaxHeads + r];
      const float f = mw == -CUDART_INF_F ? 0.f : fast_exp2(mw - M);
      Ls += cl[ww * kMaxHeads + r] * f;
      O += cO[(ww * kMaxHeads + r) * (D + 2) + d] * f;
    }
    const size_t row = static_cast<size_t>(b) * p.Hq + h0 + r;
    if (single) {
      p.out[row * D + d] = err ? CUDART_NAN_F : (Ls > 0.f ? O / Ls : 0.f);
    } else {
      const size_t prow = static_cast<size_t>(split) * p.B * p.Hq + row;
      p.ws_o[prow * D + d] = O;
      if (d == 0) {
        p.ws_m[prow] = err ? CUDART_NAN_F : M;
        p.ws_l[prow] = Ls;
      }
    }
  }
  if (single) return;

  // ---- split-K: the last block of this (sequence, head group) merges all partials
  __threadfence();
  __syncthreads();
  int* ticket = p.ws_ticket + static_cast<size_t>(b) * p.Hkv * p.head_groups + z;
  if (tid == 0) s_last = atomicAdd(ticket, 1) == nsplit - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  for (int idx = tid; idx < nh * D; idx += kThreads) {
    const int r = idx / D, d = idx % D;
    const size_t row = static_cast<size_t>(b) * p.Hq + h0 + r;
    const size_t stride = static_cast<size_t>(p.B) * p.Hq;
    float M = -CUDART_INF_F;
    bool poisoned = false;
    for (int s = 0; s < nsplit; ++s) {
      const float ms = __ldcg(p.ws_m + s * stride + row);
      poisoned |= isnan(ms);
      M = fmaxf(M, ms);
    }
    float Ls = 0.f, O = 0.f;
    for (int s = 0; s < nsplit; ++s) {
      const float ms = __ldcg(p.ws_m + s * stride + row);
      const float f = ms == -CUDART_INF_F ? 0.f : fast_exp2(ms - M);
      Ls += __ldcg(p.ws_l + s * stride + row) * f;
      O += __ldcg(p.ws_o + (s * stride + row) * D + d) * f;
    }
    p.out[row * D + d] = poisoned ? CUDART_NAN_F : (Ls > 0.f ? O / Ls : 0.f);
  }
  if (tid == 0) *ticket = 0;  // leave the counter ready for the next call
}

template <int KVT, int D>
constexpr int stages_for() {
  return Layout<KVT, D>::stageBytes >= 8192 ? (Layout<KVT, D>::stageBytes >= 16384 ? 2 : 3) : 4;
}

template <int KVT, int D>
const void* kernel_ptr() {
  return reinterpret_cast<const void*>(&decode_kernel<KVT, D, stages_for<KVT, D>()>);
}

template <int KVT, int D>
int smem_bytes() {
  return Smem<KVT, D, stages_for<KVT, D>()>::total;
}

struct Variant {
  const void* fn;
  int smem;
  int index;
};

Variant variant(int dtype, int D) {
  switch (dtype * 1000 + D) {
    case kF32 * 1000 + 64: return {kernel_ptr<kF32, 64>(), smem_bytes<kF32, 64>(), 0};
    case kF32 * 1000 + 128: return {kernel_ptr<kF32, 128>(), smem_bytes<kF32, 128>(), 1};
    case kBF16 * 1000 + 64: return {kernel_ptr<kBF16, 64>(), smem_bytes<kBF16, 64>(), 2};
    case kBF16 * 1000 + 128: return {kernel_ptr<kBF16, 128>(), smem_bytes<kBF16, 128>(), 3};
    case kINT8 * 1000 + 64: return {kernel_ptr<kINT8, 64>(), smem_bytes<kINT8, 64>(), 4};
    case kINT8 * 1000 + 128: return {kernel_ptr<kINT8, 128>(), smem_bytes<kINT8, 128>(), 5};
    default: return {nullptr, 0, -1};
  }
}

// Per-device facts queried once: SM count, and for each kernel variant its resident
// blocks per SM (after raising its dynamic shared-memory limit).
constexpr int kMaxDevices = 64;
struct DevInfo {
  int sms = 0;
  int occ[6] = {0, 0, 0, 0, 0, 0};
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
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, v.fn, kThreads, v.smem) !=
            cudaSuccess)
      return false;
    d.occ[v.index] = o > 0 ? o : 1;
  }
  *sms = d.sms;
  *occ = d.occ[v.index];
  return true;
}

}  // namespace

bool plan_decode(const CacheView& c, int B, int Hq, int MB, int q_dtype, int device,
                 int chunk_override, DecodePlan* plan) {
  (void)q_dtype;
  const Variant v = variant(c.dtype, c.D);
  if (!v.fn) return false;
  const int G = Hq / c.Hkv;
  const int cap = (c.dtype == kF32 && c.D == 128) ? f32_head_cap<128>() : kMaxHeads;
  plan->heads_per_cta = G < cap ? G : cap;
  plan->head_groups = (G + plan->heads_per_cta - 1) / plan->heads_per_cta;
  const int mb = MB > 0 ? MB : 1;
  int sms = 0, occ = 0;
  if (!device_facts(device, v, &sms, &occ)) return false;
  int chunk;
  if (chunk_override > 0) {
    chunk = chunk_override;
  } else {
    // Aim for about two waves of blocks (upper-bound estimate: every sequence at the
    // table's full length), but never fewer than two pages per warp.
    const long long units = static_cast<long long>(B) * c.Hkv * plan->head_groups;
    const long long target = 2LL * sms * occ;
    long long splits = units > 0 ? (target + units - 1) / units : 1;
    const long long max_splits = (mb + 2 * kW - 1) / (2 * kW);
    if (splits > max_splits) splits = max_splits;
    if (splits < 1) splits = 1;
    chunk = static_cast<int>((mb + splits - 1) / splits);
  }
  if (chunk < 1) chunk = 1;
  plan->chunk_pages = chunk;
  plan->n_splits = (mb + chunk - 1) / chunk;
  size_t ws = 0;
  if (plan->n_splits > 1) {
    const size_t rows = static_cast<size_t>(plan->n_splits) * B * Hq;
    const size_t tickets = static_cast<size_t>(B) * c.Hkv * plan->head_groups;
    ws = ((tickets * 4 + 255) / 256) * 256 + rows * (c.D + 2) * 4;
  }
  plan->ws_bytes = ws;
  return true;
}

cudaError_t launch_decode(const DecodeArgs& a, const DecodePlan& plan, cudaStream_t st) {
  const Variant v = variant(a.c.dtype, a.c.D);
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
  p.scale_log2 = a.scale * 1.4426950408889634f;
  if (plan.n_splits > 1) {
    const size_t tickets = static_cast<size_t>(a.B) * a.c.Hkv * plan.head_groups;
    uint8_t* base = static_cast<uint8_t*>(a.ws);
    p.ws_ticket = reinterpret_cast<int*>(base);
    const size_t rows = static_cast<size_t>(plan.n_splits) * a.B * a.Hq;
    float* f = reinterpret_cast<float*>(base + ((tickets * 4 + 255) / 256) * 256);
    p.ws_m = f;
    p.ws_l = f + rows;
    p.ws_o = f + 2 * rows;
  }
  // (the shared-memory limit was raised by plan_decode on this device)
  const dim3 grid(plan.n_splits, a.B, a.c.Hkv * plan.head_groups);
  void* args[] = {&p};
  return cudaLaunchKernel(v.fn, grid, dim3(kThreads), args, v.smem, st);
}

}  // namespace pkv
