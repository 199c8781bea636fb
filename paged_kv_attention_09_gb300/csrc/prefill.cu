// prefill.cu — chunked-prefill attention over a paged BF16 KV cache.
//
// Sources: "Tiny-LLM-Inference Project_Status" (chunked prefill/decode scheduling; the
// chunked-prefill SDPA path; dedicated BF16 paged-attention kernel) and "tinyloop
// Current Status" (chunked prefill, chunk 512; GQA; 16-token pages).  Row i of a chunk
// of length Lq sits at position context_len - Lq + i and attends causally to positions
// 0..that position (the chunk's own K/V are appended first).
//
// Layout: grid (row tile, kv head, sequence).  The rows of a tile are (chunk token,
// query head) pairs of one GQA group, token-major (row = i * G + head), so the query
// heads that share a kv head share every K/V tile.  64 rows per block, 16 per warp.
// K/V stream through a two-stage shared-memory ring in 64-key tiles (4 pages), each page
// block fetched by a 1-D bulk copy.  Q.K^T and P.V run on warp-level tensor-core MMA
// (m16n8k16, BF16 operands, FP32 accumulation); P is split into a BF16 high part and a
// BF16 remainder (two MMAs) so the product keeps ~16 bits and short contexts stay within
// 2e-3 of the exact result.  Online softmax with FP32 running max / sum per row.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"

// 1: tcgen05 kernel (prefill_tc.cu); 0: the warp-level MMA kernel below.
#ifndef PKV_PREFILL_TC
#define PKV_PREFILL_TC 1
#endif

namespace pkv {
namespace {

constexpr int kPW = 4;                 // warps per block
constexpr int kPThreads = kPW * 32;
constexpr int kRows = kPW * 16;        // rows per block
constexpr int kTileKeys = 64;          // keys per pipeline stage
constexpr int kTilePages = kTileKeys / kPage;
constexpr int kPStages = 2;

struct PParams {
  const __nv_bfloat16* k;
  const __nv_bfloat16* v;
  const void* q;
  const int32_t* qsl;
  const int32_t* bt;
  const int32_t* lens;
  float* out;
  int32_t* dev_status;
  int q_dtype, Hkv, Hq, G, MB, num_pages;
  float scale_log2;
};

template <int D>
struct PSmem {
  static constexpr int kBlk = kPage * D * 2;                  // bytes of one page block
  static constexpr int kStage = 2 * kTilePages * kBlk;        // K then V blocks
  static constexpr int total = kPStages * kStage + kPStages * 8;
};

__device__ __forceinline__ float4 load_q4p(const void* q, int q_dtype, size_t i) {
  if (q_dtype == kBF16) {
    const __nv_bfloat162* p = reinterpret_cast<const __nv_bfloat162*>(
        static_cast<const __nv_bfloat16*>(q) + i);
    const float2 a = __bfloat1622float2(p[0]);
    const float2 b = __bfloat1622float2(p[1]);
    return make_float4(a.x, a.y, b.x, b.y);
  }
  return *reinterpret_cast<const float4*>(static_cast<const float*>(q) + i);
}

// QSPLIT: FP32 queries are carried as a BF16 high part plus a BF16 remainder (two
// Q.K^T MMAs); BF16 queries are exact and need one.
template <int D, bool QSPLIT>
__global__ void __launch_bounds__(kPThreads)
    prefill_kernel(const __grid_constant__ PParams p) {
  using Sm = PSmem<D>;
  constexpr int KS = D / 16, NT = D / 8, NQ = QSPLIT ? 2 : 1;
  extern __shared__ __align__(128) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kPStages * Sm::kStage);
  __shared__ int s_flag;

  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int r = lane >> 2, c = lane & 3;
  const int g = blockIdx.y, b = blockIdx.z;
  const int row0 = blockIdx.x * kRows;
  const int q0 = p.qsl[b];
  const int Lq = p.qsl[b + 1] - q0;
  const int L = p.lens[b];
  const int nrows = Lq > 0 ? Lq * p.G : 0;
  if (row0 >= nrows) return;

  int err = 0;
  if (L < 0 || L > p.MB * kPage) err |= 0x2;  // PKV_DEV_BAD_LEN
  if (Lq > L) err |= 0x8;                     // PKV_DEV_BAD_CHUNK
  const int last_row = min(row0 + kRows, nrows) - 1;
  const int p_first = L - Lq + row0 / p.G;
  const int p_last = L - Lq + last_row / p.G;
  const int n_keys = err ? 0 : p_last + 1;
  const int n_pages = (n_keys + kPage - 1) / kPage;
  const int n_tiles = (n_keys + kTileKeys - 1) / kTileKeys;
  const int32_t* bt = p.bt + static_cast<size_t>(b) * p.MB;

  if (tid == 0) s_flag = err;
  __syncthreads();
  for (int j = tid; j < n_pages; j += kPThreads) {
    const int pg = bt[j];
    if (pg < 0 || pg >= p.num_pages) atomicOr(&s_flag, 0x1);  // PKV_DEV_BAD_PAGE
  }
  __syncthreads();
  err = s_flag;

  // ---- this thread's two rows (r and r + 8 of its warp's 16)
  int rowv[2], pos[2];
  bool rvalid[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    rowv[h] = row0 + w * 16 + r + 8 * h;
    rvalid[h] = rowv[h] < nrows;
    pos[h] = rvalid[h] ? L - Lq + rowv[h] / p.G : p_first;
  }
  uint32_t qa[NQ][KS][4];
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    const int d0 = 32 * (ks >> 1) + 8 * c + 4 * (ks & 1);
    float x[2][4];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
      if (rvalid[h] && !err) {
        const int i = rowv[h] / p.G, hh = rowv[h] % p.G;
        v4 = load_q4p(p.q, p.q_dtype,
                      (static_cast<size_t>(q0 + i) * p.Hq + g * p.G + hh) * D + d0);
      }
      x[h][0] = v4.x; x[h][1] = v4.y; x[h][2] = v4.z; x[h][3] = v4.w;
    }
#pragma unroll
    for (int part = 0; part < NQ; ++part) {
      __nv_bfloat16 e[2][4];
#pragma unroll
      for (int h = 0; h < 2; ++h)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const __nv_bfloat16 hi = __float2bfloat16_rn(x[h][j]);
          e[h][j] = part == 0 ? hi : __float2bfloat16_rn(x[h][j] - __bfloat162float(hi));
        }
      qa[part][ks][0] = pack_bf162(e[0][0], e[0][1]);
      qa[part][ks][1] = pack_bf162(e[1][0], e[1][1]);
      qa[part][ks][2] = pack_bf162(e[0][2], e[0][3]);
      qa[part][ks][3] = pack_bf162(e[1][2], e[1][3]);
    }
  }

  float o[NT][4];
#pragma unroll
  for (int j = 0; j < NT; ++j) o[j][0] = o[j][1] = o[j][2] = o[j][3] = 0.f;
  float m[2] = {-CUDART_INF_F, -CUDART_INF_F}, l[2] = {0.f, 0.f};
  bool timed_out = false;

  if (!err) {
    if (tid == 0) {
      for (int i = 0; i < kPStages; ++i) mbar_init(&bars[i], 1);
      fence_barrier_init();
    }
    __syncthreads();
    const uint64_t pol = l2_evict_first_policy();
    auto issue = [&](int t) {
      uint8_t* st = smem + (t % kPStages) * Sm::kStage;
      const int np = min(kTilePages, n_pages - t * kTilePages);
      mbar_arrive_expect_tx(&bars[t % kPStages], np * 2 * Sm::kBlk);
      for (int q = 0; q < np; ++q) {
        const size_t blk = static_cast<size_t>(bt[t * kTilePages + q]) * p.Hkv + g;
        bulk_g2s(st + q * Sm::kBlk, p.k + blk * kPage * D, Sm::kBlk, &bars[t % kPStages], pol);
        bulk_g2s(st + (kTilePages + q) * Sm::kBlk, p.v + blk * kPage * D, Sm::kBlk,
                 &bars[t % kPStages], pol);
      }
    };
    if (tid == 0)
      for (int t = 0; t < min(kPStages, n_tiles); ++t) issue(t);

    for (int t = 0; t < n_tiles; ++t) {
      const bool ok = mbar_wait(&bars[t % kPStages], (t / kPStages) & 1);
      if (__syncthreads_or(!ok)) {
        timed_out = true;
        // drain (bounded) the copies still in flight before leaving
        if (tid == 0)
          for (int k = t + 1; k < min(n_tiles, t + kPStages); ++k)
            (void)mbar_wait(&bars[k % kPStages], (k / kPStages) & 1);
        break;
      }
      const uint8_t* Ks = smem + (t % kPStages) * Sm::kStage;
      const uint8_t* Vs = Ks + kTilePages * Sm::kBlk;
      const int key0 = t * kTileKeys;
      // ---- S = Q K^T for 16 rows x 64 keys: n-tile 2q+j column n = key
      //      16q + 4(n/2) + 2j + (n%2); lane (r, c) holds keys 16q + 4c .. +3.
      float sacc[2 * kTilePages][4];
#pragma unroll
      for (int nt = 0; nt < 2 * kTilePages; ++nt) {
        sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
        const int t = 4 * (r >> 1) + (r & 1) + 2 * (nt & 1);  // token inside page nt/2
        const uint8_t* kpage = Ks + (nt >> 1) * Sm::kBlk;
#pragma unroll
        for (int blk = 0; blk < D / 32; ++blk) {
          const uint4 kw = *reinterpret_cast<const uint4*>(kpage + bf16_k_off(t, blk * 32 + c * 8, D));
#pragma unroll
          for (int part = 0; part < NQ; ++part) {
            mma_bf16(sacc[nt], qa[part][2 * blk + 0], kw.x, kw.y);
            mma_bf16(sacc[nt], qa[part][2 * blk + 1], kw.z, kw.w);
          }
        }
      }
      // ---- causal mask, online softmax for rows r (h=0) and r+8 (h=1)
      float mx[2] = {-CUDART_INF_F, -CUDART_INF_F};
#pragma unroll
      for (int nt = 0; nt < 2 * kTilePages; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int h = e >> 1;
          const int key = key0 + 16 * (nt >> 1) + 4 * c + 2 * (nt & 1) + (e & 1);
          const float s = key <= pos[h] ? sacc[nt][e] * p.scale_log2 : -CUDART_INF_F;
          sacc[nt][e] = s;
          mx[h] = fmaxf(mx[h], s);
        }
      float corr[2];
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float mn = fmaxf(m[h], mx[h]);
        corr[h] = fast_exp2(m[h] - mn);
        m[h] = mn;
        l[h] *= corr[h];
      }
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        o[j][0] *= corr[0]; o[j][1] *= corr[0];
        o[j][2] *= corr[1]; o[j][3] *= corr[1];
      }
      // ---- P.V, one k-step per page; P carried as hi + lo BF16 parts
#pragma unroll
      for (int q = 0; q < kTilePages; ++q) {
        float pr[2][4];  // [row][key 4c + i]
#pragma unroll
        for (int j = 0; j < 2; ++j)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int h = e >> 1;
            const float pv = fast_exp2(sacc[2 * q + j][e] - m[h]);
            pr[h][2 * j + (e & 1)] = pv;
            l[h] += pv;
          }
        uint32_t ahi[4], alo[4];
        {
          __nv_bfloat16 hi[2][4], lo[2][4];
#pragma unroll
          for (int h = 0; h < 2; ++h)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              hi[h][i] = __float2bfloat16_rn(pr[h][i]);
              lo[h][i] = __float2bfloat16_rn(pr[h][i] - __bfloat162float(hi[h][i]));
            }
          ahi[0] = pack_bf162(hi[0][0], hi[0][1]);
          ahi[1] = pack_bf162(hi[1][0], hi[1][1]);
          ahi[2] = pack_bf162(hi[0][2], hi[0][3]);
          ahi[3] = pack_bf162(hi[1][2], hi[1][3]);
          alo[0] = pack_bf162(lo[0][0], lo[0][1]);
          alo[1] = pack_bf162(lo[1][0], lo[1][1]);
          alo[2] = pack_bf162(lo[0][2], lo[0][3]);
          alo[3] = pack_bf162(lo[1][2], lo[1][3]);
        }
        // keys past the block's last query position (page padding, pages not loaded)
        // may hold anything, even NaN: zero their V entries
        const int kb = key0 + 16 * q + 4 * c;
        const uint32_t vm0 =
            (kb + 0 < n_keys ? 0x0000ffffu : 0u) | (kb + 1 < n_keys ? 0xffff0000u : 0u);
        const uint32_t vm1 =
            (kb + 2 < n_keys ? 0x0000ffffu : 0u) | (kb + 3 < n_keys ? 0xffff0000u : 0u);
        const uint8_t* vblk = Vs + q * Sm::kBlk;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
          const int d = 8 * j + r;
          const uint2 vw = *reinterpret_cast<const uint2*>(vblk + bf16_v_off(d, 4 * c));
          mma_bf16(o[j], ahi, vw.x & vm0, vw.y & vm1);
          mma_bf16(o[j], alo, vw.x & vm0, vw.y & vm1);
        }
      }
      __syncthreads();
      if (tid == 0 && t + kPStages < n_tiles) issue(t + kPStages);
    }
  }
  if (timed_out && tid == 0) atomicOr(&s_flag, 0x10);  // PKV_DEV_TIMEOUT
  __syncthreads();
  err = s_flag;
  if (tid == 0 && err && p.dev_status) atomicOr(p.dev_status, err);
  {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      float lt = l[h];
      lt += __shfl_xor_sync(0xffffffffu, lt, 1);
      lt += __shfl_xor_sync(0xffffffffu, lt, 2);
      if (!rvalid[h]) continue;
      const int i = rowv[h] / p.G, hh = rowv[h] % p.G;
      float* dst = p.out + (static_cast<size_t>(q0 + i) * p.Hq + g * p.G + hh) * D;
      const float inv = err ? CUDART_NAN_F : 1.f / lt;
#pragma unroll
      for (int j = 0; j < NT; ++j) {
        const float2 v2 = make_float2(o[j][2 * h] * inv, o[j][2 * h + 1] * inv);
        *reinterpret_cast<float2*>(dst + 8 * j + 2 * c) = v2;
      }
    }
  }
}

template <int D, bool QSPLIT>
const void* pk() {
  return reinterpret_cast<const void*>(&prefill_kernel<D, QSPLIT>);
}

constexpr int kMaxDevices = 64;
bool g_attr_set[kMaxDevices][4];
std::mutex g_mu;

bool raise_smem_limit(int device, int slot, const void* fn, int smem) {
  if (device < 0 || device >= kMaxDevices) return false;
  std::lock_guard<std::mutex> lock(g_mu);
  if (g_attr_set[device][slot]) return true;
  if (cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return false;
  g_attr_set[device][slot] = true;
  return true;
}

}  // namespace

cudaError_t launch_prefill_mma(const PrefillArgs& a, const PrefillPlan& plan, cudaStream_t st);

bool plan_prefill(const CacheView& c, int B, int Hq, int max_q_len, int MB, int q_dtype,
                  int device, PrefillPlan* plan) {
  (void)B; (void)MB; (void)device; (void)q_dtype;
  if (c.dtype != kBF16) return false;
  if (c.D != 64 && c.D != 128) return false;
#if !PKV_PREFILL_TC
  if (c.window > 0) return false;  // the warp-level MMA kernel has no window mask
#endif
  const int G = Hq / c.Hkv;
#if PKV_PREFILL_TC
  plan->rows_per_cta = prefill_tc_rows();
#else
  plan->rows_per_cta = kRows;
#endif
  const long long rows = static_cast<long long>(max_q_len) * G;
  plan->n_row_tiles = static_cast<int>((rows + plan->rows_per_cta - 1) / plan->rows_per_cta);
  plan->ws_bytes = 0;
  return true;
}

cudaError_t launch_prefill(const PrefillArgs& a, const PrefillPlan& plan, cudaStream_t st) {
#if PKV_PREFILL_TC
  return launch_prefill_tc(a, plan.n_row_tiles, st);
#else
  return launch_prefill_mma(a, plan, st);
#endif
}

cudaError_t launch_prefill_mma(const PrefillArgs& a, const PrefillPlan& plan, cudaStream_t st) {
  PParams p{};
  p.k = static_cast<const __nv_bfloat16*>(a.c.k);
  p.v = static_cast<const __nv_bfloat16*>(a.c.v);
  p.q = a.q;
  p.qsl = a.q_start_loc;
  p.bt = a.block_tables;
  p.lens = a.context_lens;
  p.out = a.out;
  p.dev_status = a.dev_status;
  p.q_dtype = a.q_dtype;
  p.Hkv = a.c.Hkv;
  p.Hq = a.Hq;
  p.G = a.Hq / a.c.Hkv;
  p.MB = a.MB;
  p.num_pages = a.c.num_pages;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  const bool split = a.q_dtype == kF32;
  const void* fn;
  int smem;
  if (a.c.D == 64) {
    fn = split ? pk<64, true>() : pk<64, false>();
    smem = PSmem<64>::total;
  } else {
    fn = split ? pk<128, true>() : pk<128, false>();
    smem = PSmem<128>::total;
  }
  if (plan.n_row_tiles == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (!raise_smem_limit(dev, (a.c.D == 64 ? 0 : 2) + (split ? 1 : 0), fn, smem))
    return cudaErrorInvalidValue;
  const dim3 grid(plan.n_row_tiles, a.c.Hkv, a.B);
  void* args[] = {&p};
  return cudaLaunchKernel(fn, grid, dim3(kPThreads), args, smem, st);
}

}  // namespace pkv
