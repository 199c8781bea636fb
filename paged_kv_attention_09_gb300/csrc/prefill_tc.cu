// prefill_tc.cu — chunked-prefill attention on the 5th-generation tensor cores (tcgen05).
//
// Sources: "Tiny-LLM-Inference Project_Status" (chunked prefill/decode scheduling; the
// chunked-prefill SDPA path; BF16 KV with its own paged-attention kernel) and "tinyloop
// Current Status" (chunked prefill, chunk 512; GQA; 16-token pages).  Row i of a chunk
// of length Lq sits at position context_len - Lq + i and attends causally to positions
// 0..that position (the chunk's own K/V are appended first).
//
// One block computes 128 query rows — (chunk token, query head) pairs of one GQA group,
// token-major — against the group's paged K/V in tiles of 64 keys (4 pages):
//   warp 9    producer: one bulk copy per BF16 page block (K and V, already stored as
//             tensor-core tiles) into a two-stage ring;
//   warp 8    MMA issuer: S = Q K^T (M=128, N=64) into a double-buffered TMEM region and
//             O += P V (M=128, N=head_dim) into a TMEM accumulator, one thread issuing
//             tcgen05.mma and tracking completion with tcgen05.commit on mbarriers;
//   warps 0-7 softmax: two threads per row (one TMEM lane, 32 keys each; the row max is
//             exchanged through shared memory): they read S from TMEM, apply the causal
//             mask and the online softmax in FP32, and write P into shared memory as a
//             BF16 high part and a BF16 remainder (two MMAs per page) so that the product
//             keeps ~16 bits.  The running max is only raised when it
//             grows by more than 2^8 (the accumulator in TMEM is rescaled then), so the
//             P.V MMAs accumulate without a per-tile round trip through registers.
// FP32 queries are split the same way into two BF16 tiles (two Q.K^T MMAs per k-step).
// Every operand tile uses the no-swizzle K-major canonical layout of 8 x 16-byte core
// matrices; every wait is bounded.
#include <cuda_bf16.h>
#include <math_constants.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {
namespace {

constexpr int kRowsTC = 128;      // query rows per block (MMA M)
constexpr int kKeysTC = 64;       // keys per tile (MMA N of S)
constexpr int kPagesTC = kKeysTC / kPage;
constexpr int kSoftWarps = 8;           // two threads per query row, 32 keys each
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kThreadsTC = (kSoftWarps + 2) * 32;
constexpr float kRescaleLog2 = 8.f;  // raise the running max only beyond this margin

struct TParams {
  const uint8_t* k;
  const uint8_t* v;
  const void* q;
  const int32_t* qsl;
  const int32_t* bt;
  const int32_t* lens;
  float* out;
  int32_t* dev_status;
  int q_dtype, Hkv, Hq, G, MB, num_pages;
  float scale_log2;
};

template <int D, bool QSPLIT>
struct TSmem {
  static constexpr int kBlk = kPage * D * 2;           // one BF16 page block (K or V)
  static constexpr int qTile = kRowsTC * D * 2;        // one BF16 query tile
  static constexpr int stage = kPagesTC * kBlk;        // the K (or V) blocks of one tile
  static constexpr int KST = QSPLIT ? 2 : 3;           // stages of each of the K and V rings
  static constexpr int pTile = kRowsTC * kKeysTC * 2;  // one BF16 probability tile
  static constexpr int q0 = 0;
  static constexpr int k0 = q0 + (QSPLIT ? 2 : 1) * qTile;
  static constexpr int v0 = k0 + KST * stage;
  static constexpr int p0 = v0 + KST * stage;           // [buffer][hi, lo]
  static constexpr int bar0 = p0 + 2 * 2 * pTile;
  // barriers: k_full[3], k_empty[3], v_full[3], v_empty[3], s_full[2], s_free[2],
  // p_full[2], o_done[2], final, row-max exchange[2], row-sum exchange
  static constexpr int nbars = 24;
  static constexpr int misc0 = bar0 + nbars * 8;        // TMEM base address, flags
  static constexpr int xch0 = misc0 + 16;  // max [2 tiles][2 halves][128], sum [2 halves][128]
  static constexpr int total = xch0 + 3 * 2 * kRowsTC * 4;
  static constexpr int tmemCols = (D + 2 * kKeysTC) <= 256 ? 256 : 512;
};

// Byte offset of element (row, col) in a no-swizzle K-major tile whose K extent is
// kext elements: core matrix (row / 8, col / 8), row % 8, element col % 8.
__device__ __forceinline__ uint32_t tile_off(int row, int col, int kext) {
  return ((((row >> 3) * (kext >> 3)) + (col >> 3)) << 7) + ((row & 7) << 4) + ((col & 7) << 1);
}

template <int D, bool QSPLIT>
__global__ void __launch_bounds__(kThreadsTC, 1)
    prefill_tc_kernel(const __grid_constant__ TParams p) {
  using Sm = TSmem<D, QSPLIT>;
  extern __shared__ __align__(1024) uint8_t smem[];
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + Sm::bar0);
  uint64_t* k_full = bars + 0;
  uint64_t* k_empty = bars + 3;
  uint64_t* v_full = bars + 6;
  uint64_t* v_empty = bars + 9;
  uint64_t* s_full = bars + 12;
  uint64_t* s_free = bars + 14;
  uint64_t* p_full = bars + 16;
  uint64_t* o_done = bars + 18;
  uint64_t* fin = bars + 20;
  uint64_t* xbar = bars + 21;  // [2] row-max exchange, [2] row-sum exchange
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Sm::misc0);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Sm::misc0 + 4);
  __shared__ int s_err;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int row0 = blockIdx.x * kRowsTC;
  const int q0 = p.qsl[b];
  const int Lq = p.qsl[b + 1] - q0;
  const int L = p.lens[b];
  const int nrows = Lq > 0 ? Lq * p.G : 0;
  if (row0 >= nrows) return;

  int err = 0;
  if (L < 0 || L > p.MB * kPage) err |= 0x2;  // PKV_DEV_BAD_LEN
  if (Lq > L) err |= 0x8;                     // PKV_DEV_BAD_CHUNK
  const int last_row = min(row0 + kRowsTC, nrows) - 1;
  const int p_first = L - Lq + row0 / p.G;
  const int p_last = L - Lq + last_row / p.G;
  const int n_keys0 = err ? 0 : p_last + 1;
  const int32_t* bt = p.bt + static_cast<size_t>(b) * p.MB;
  if (tid == 0) s_err = err;
  __syncthreads();
  for (int j = tid; j < (n_keys0 + kPage - 1) / kPage; j += kThreadsTC) {
    const int pg = bt[j];
    if (pg < 0 || pg >= p.num_pages) atomicOr(&s_err, 0x1);  // PKV_DEV_BAD_PAGE
  }
  __syncthreads();
  err = s_err;
  const int n_keys = err ? 0 : n_keys0;
  const int n_pages = (n_keys + kPage - 1) / kPage;
  const int n_tiles = (n_keys + kKeysTC - 1) / kKeysTC;

  // ---- set-up: TMEM, barriers, the query tile(s)
  if (warp == kSoftWarps) {
    tc::tmem_alloc(tmem_slot, Sm::tmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < Sm::nbars; ++i) {
      // s_free, p_full and the exchanges: one arrival per softmax thread
      const bool many = (i >= 14 && i < 18) || i >= 21;
      mbar_init(&bars[i], many ? kSoftThreads : 1);
    }
    fence_barrier_init();
    *abort_flag = 0;
  }
  // softmax threads: row r (= TMEM lane 32 (warp % 4) + lane) and half hf of the keys
  const int r = tid & (kRowsTC - 1);
  const int hf = tid / kRowsTC;
  const int rho = row0 + r;
  const bool valid_row = tid < kSoftThreads && rho < nrows;
  if (tid < kSoftThreads) {
    uint8_t* qhi = smem + Sm::q0;
    uint8_t* qlo = smem + Sm::q0 + Sm::qTile;
    const size_t qrow = valid_row && !err
                            ? (static_cast<size_t>(q0 + rho / p.G) * p.Hq + g * p.G + rho % p.G) * D
                            : 0;
#pragma unroll 4
    for (int kc = hf * (D / 16); kc < (hf + 1) * (D / 16); ++kc) {
      uint4 hi = make_uint4(0u, 0u, 0u, 0u), lo = hi;
      if (valid_row && !err) {
        if (p.q_dtype == kBF16) {
          hi = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(p.q) + qrow + 8 * kc);
        } else {
          const float* qf = static_cast<const float*>(p.q) + qrow + 8 * kc;
          const float4 a = *reinterpret_cast<const float4*>(qf);
          const float4 e = *reinterpret_cast<const float4*>(qf + 4);
          const float x[8] = {a.x, a.y, a.z, a.w, e.x, e.y, e.z, e.w};
          uint32_t h[4], l2[4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const __nv_bfloat162 hv = __floats2bfloat162_rn(x[2 * u], x[2 * u + 1]);
            const float2 hf = __bfloat1622float2(hv);
            const __nv_bfloat162 lv = __floats2bfloat162_rn(x[2 * u] - hf.x, x[2 * u + 1] - hf.y);
            h[u] = *reinterpret_cast<const uint32_t*>(&hv);
            l2[u] = *reinterpret_cast<const uint32_t*>(&lv);
          }
          hi = make_uint4(h[0], h[1], h[2], h[3]);
          lo = make_uint4(l2[0], l2[1], l2[2], l2[3]);
        }
      }
      *reinterpret_cast<uint4*>(qhi + tile_off(r, 8 * kc, D)) = hi;
      if constexpr (QSPLIT) *reinterpret_cast<uint4*>(qlo + tile_off(r, 8 * kc, D)) = lo;
    }
  }
  fence_proxy_async_smem();  // generic writes of Q become visible to the tensor cores
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sbase = smem_u32(smem);

  if (n_tiles > 0 && warp == kSoftWarps + 1) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_last_policy();  // every row tile of the group rereads them
      constexpr int KST = Sm::KST;
      int issued = 0;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % KST, use = j / KST;
        const int np = min(kPagesTC, n_pages - j * kPagesTC);
        if (j >= KST && !mbar_wait(&k_empty[st], (use - 1) & 1)) { *abort_flag = 1; break; }
        if (*abort_flag) break;
        uint8_t* kst = smem + Sm::k0 + st * Sm::stage;
        mbar_arrive_expect_tx(&k_full[st], np * Sm::kBlk);
        for (int q = 0; q < np; ++q) {
          const size_t blk = static_cast<size_t>(bt[j * kPagesTC + q]) * p.Hkv + g;
          bulk_g2s(kst + q * Sm::kBlk, p.k + blk * Sm::kBlk, Sm::kBlk, &k_full[st], pol);
        }
        if (j >= KST && !mbar_wait(&v_empty[st], (use - 1) & 1)) { *abort_flag = 1; issued = -(j + 1); break; }
        uint8_t* vst = smem + Sm::v0 + st * Sm::stage;
        mbar_arrive_expect_tx(&v_full[st], np * Sm::kBlk);
        for (int q = 0; q < np; ++q) {
          const size_t blk = static_cast<size_t>(bt[j * kPagesTC + q]) * p.Hkv + g;
          bulk_g2s(vst + q * Sm::kBlk, p.v + blk * Sm::kBlk, Sm::kBlk, &v_full[st], pol);
        }
        issued = j + 1;
      }
      // leave nothing in flight: the copies of the last issued tiles have landed
      const int kdone = issued >= 0 ? issued : -issued;   // K issued for tiles < kdone
      const int vdone = issued >= 0 ? issued : -issued - 1;
      for (int j = max(0, kdone - KST); j < kdone; ++j) (void)mbar_wait(&k_full[j % KST], (j / KST) & 1);
      for (int j = max(0, vdone - KST); j < vdone; ++j) (void)mbar_wait(&v_full[j % KST], (j / KST) & 1);
    }
  } else if (n_tiles > 0 && warp == kSoftWarps) {
    // ---------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kRowsTC, kKeysTC);
      constexpr uint32_t idO = tc::idesc_bf16_f32(kRowsTC, D);
      constexpr uint32_t sboQK = (D / 8) * 128;  // 8-row groups of Q and of K
      const uint32_t qhi = sbase + Sm::q0, qlo = sbase + Sm::q0 + Sm::qTile;
      constexpr int KST = Sm::KST;
      auto issue_pv = [&](int i) -> bool {
        const int y = i & 1;
        if (!mbar_wait(&p_full[y], (i >> 1) & 1)) return false;
        if (!mbar_wait(&v_full[i % KST], (i / KST) & 1)) return false;
        tc::fence_after_sync();
        const uint32_t vst = sbase + Sm::v0 + (i % KST) * Sm::stage;
        const uint32_t pbuf = sbase + Sm::p0 + y * 2 * Sm::pTile;
#pragma unroll
        for (int q = 0; q < kPagesTC; ++q) {
          const uint64_t bd = tc::smem_desc(vst + q * Sm::kBlk, 128, 256);
#pragma unroll
          for (int part = 0; part < 2; ++part) {
            const uint64_t ad = tc::smem_desc(pbuf + part * Sm::pTile + q * 256, 128, 1024);
            tc::mma_bf16(tmem, ad, bd, idO, !(i == 0 && q == 0 && part == 0));
          }
        }
        tc::commit(&o_done[y]);
        tc::commit(&v_empty[i % KST]);
        return true;
      };
      bool ok = true;
      for (int j = 0; j < n_tiles && ok; ++j) {
        const int x = j & 1;
        ok = mbar_wait(&k_full[j % KST], (j / KST) & 1) &&
             (j < 2 || mbar_wait(&s_free[x], ((j - 2) >> 1) & 1)) && !*abort_flag;
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t kst = sbase + Sm::k0 + (j % KST) * Sm::stage;
        const uint32_t tS = tmem + D + kKeysTC * x;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t bd = tc::smem_desc(kst + ks * 256, 128, sboQK);
          tc::mma_bf16(tS, tc::smem_desc(qhi + ks * 256, 128, sboQK), bd, idS, ks > 0);
          if constexpr (QSPLIT) tc::mma_bf16(tS, tc::smem_desc(qlo + ks * 256, 128, sboQK), bd, idS, true);
        }
        tc::commit(&s_full[x]);
        tc::commit(&k_empty[j % KST]);
        if (j >= 1) ok = issue_pv(j - 1);
      }
      if (ok) ok = issue_pv(n_tiles - 1);
      if (!ok) *abort_flag = 1;
      // every MMA issued above has completed before TMEM is released
      tc::commit(fin);
      (void)mbar_wait(fin, 0);
    }
  } else if (n_tiles > 0) {
    // ---------------------------------------------------------------- softmax rows
    const int pos = valid_row ? L - Lq + rho / p.G : p_first;
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const float sl = p.scale_log2;
    float* xch = reinterpret_cast<float*>(smem + Sm::xch0);  // [tile & 1][half][row]
    float m_used = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int x = j & 1;
      ok = mbar_wait(&s_full[x], (j >> 1) & 1) && !*abort_flag;
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc::fence_after_sync();
      float s[32];
      tc::ld32(tmem + lane_base + D + kKeysTC * x + 32 * hf, s);
      tc::fence_before_sync();
      mbar_arrive(&s_free[x]);
      const int key0 = j * kKeysTC + 32 * hf;
      // raw scores; the scale (> 0) is applied inside the exponent with one FMA
      if (j * kKeysTC + kKeysTC - 1 > p_first || j * kKeysTC + kKeysTC > n_keys) {
#pragma unroll
        for (int k = 0; k < 32; ++k) s[k] = (key0 + k <= pos) ? s[k] : -CUDART_INF_F;
      }
      float mx = s[0];
#pragma unroll
      for (int k = 1; k < 32; ++k) mx = fmaxf(mx, s[k]);
      xch[(x * 2 + hf) * kRowsTC + r] = mx;
      mbar_arrive(&xbar[x]);
      ok = mbar_wait(&xbar[x], (j >> 1) & 1);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      mx = fmaxf(mx, xch[(x * 2 + (hf ^ 1)) * kRowsTC + r]) * sl;
      const bool need = mx > m_used + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_used;
        const float f = need ? fast_exp2(m_used - m_new) : 1.f;
        if (j >= 1) {
          // O holds tiles 0 .. j-1: wait for the last P.V, then rescale this half's columns
          ok = mbar_wait(&o_done[(j - 1) & 1], ((j - 1) >> 1) & 1);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            float o[32];
            const uint32_t ta = tmem + lane_base + (D / 2) * hf + 32 * c;
            tc::ld32(ta, o);
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= f;
            tc::st32(ta, o);
          }
        }
        l *= f;
        m_used = m_new;
      }
      if (j >= 2) {  // the P buffer being rewritten was read by the P.V of tile j-2
        ok = mbar_wait(&o_done[x], ((j - 2) >> 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      uint8_t* phi = smem + Sm::p0 + x * 2 * Sm::pTile;
      uint8_t* plo = phi + Sm::pTile;
      const float nm = -m_used;
#pragma unroll
      for (int kc = 0; kc < 4; ++kc) {
        uint32_t h[4], lo[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float a = fast_exp2(fmaf(s[8 * kc + 2 * u], sl, nm));
          const float e = fast_exp2(fmaf(s[8 * kc + 2 * u + 1], sl, nm));
          l += a + e;
          const __nv_bfloat162 hv = __floats2bfloat162_rn(a, e);
          const float2 hf2 = __bfloat1622float2(hv);
          const __nv_bfloat162 lv = __floats2bfloat162_rn(a - hf2.x, e - hf2.y);
          h[u] = *reinterpret_cast<const uint32_t*>(&hv);
          lo[u] = *reinterpret_cast<const uint32_t*>(&lv);
        }
        const int col = 32 * hf + 8 * kc;
        *reinterpret_cast<uint4*>(phi + tile_off(r, col, kKeysTC)) = make_uint4(h[0], h[1], h[2], h[3]);
        *reinterpret_cast<uint4*>(plo + tile_off(r, col, kKeysTC)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      if (j * kKeysTC + kKeysTC > n_keys) {
        // keys past the last one any row may see: pages not loaded, or page padding
        // that may hold anything (even NaN); zero them in V so that 0 * V stays 0
        // (after this tile's V copies have landed)
        ok = mbar_wait(&v_full[j % Sm::KST], (j / Sm::KST) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        uint8_t* vst = smem + Sm::v0 + (j % Sm::KST) * Sm::stage;
        const int kz = n_keys - j * kKeysTC;
        for (int idx = tid; idx < (kKeysTC - kz) * D; idx += kSoftThreads) {
          const int key = kz + idx / D, d = idx % D;
          *reinterpret_cast<__nv_bfloat16*>(vst + (key >> 4) * Sm::kBlk + bf16_v_off(d, key & 15)) =
              __float2bfloat16_rn(0.f);
        }
      }
      fence_proxy_async_smem();  // P (and zeroed V) become visible to the tensor cores
      tc::fence_before_sync();
      mbar_arrive(&p_full[x]);
    }
    if (ok) {
      ok = mbar_wait(&o_done[(n_tiles - 1) & 1], ((n_tiles - 1) >> 1) & 1);
      ok = __all_sync(0xffffffffu, ok);
    }
    // the row sum is split over the two halves (the max buffers are no longer in use
    // once every thread has passed its last tile's P barrier wait)
    if (ok) {
      float* lx = xch + 2 * 2 * kRowsTC;
      lx[hf * kRowsTC + r] = l;
      mbar_arrive(&xbar[2]);
      ok = __all_sync(0xffffffffu, mbar_wait(&xbar[2], 0));
      l += lx[(hf ^ 1) * kRowsTC + r];
    }
    if (!ok) *abort_flag = 1;
    if (ok) {
      tc::fence_after_sync();
      const float inv = 1.f / l;
      float* dst = valid_row ? p.out + (static_cast<size_t>(q0 + rho / p.G) * p.Hq + g * p.G + rho % p.G) * D
                             : nullptr;
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        float o[32];
        const int col = (D / 2) * hf + 32 * c;
        tc::ld32(tmem + lane_base + col, o);
        if (dst) {
#pragma unroll
          for (int k = 0; k < 32; k += 4)
            *reinterpret_cast<float4*>(dst + col + k) =
                make_float4(o[k] * inv, o[k + 1] * inv, o[k + 2] * inv, o[k + 3] * inv);
        }
      }
    }
  }

  // ---- tear-down: errors become NaN rows; TMEM is released by the warp that took it
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (tid == 0 && *abort_flag) atomicOr(&s_err, 0x10);  // PKV_DEV_TIMEOUT
  __syncthreads();
  err = s_err;
  if (tid == 0 && err && p.dev_status) atomicOr(p.dev_status, err);
  if (err && valid_row) {
    float* dst = p.out + (static_cast<size_t>(q0 + rho / p.G) * p.Hq + g * p.G + rho % p.G) * D;
    for (int d = (D / 2) * hf; d < (D / 2) * (hf + 1); ++d) dst[d] = CUDART_NAN_F;
  }
  if (warp == kSoftWarps) tc::tmem_dealloc(tmem, Sm::tmemCols);
}

template <int D, bool QSPLIT>
const void* tc_kernel() {
  return reinterpret_cast<const void*>(&prefill_tc_kernel<D, QSPLIT>);
}

constexpr int kMaxDevicesTC = 64;
bool g_tc_attr[kMaxDevicesTC][4];
std::mutex g_tc_mu;

}  // namespace

int prefill_tc_rows() { return kRowsTC; }

cudaError_t launch_prefill_tc(const PrefillArgs& a, int n_row_tiles, cudaStream_t st) {
  TParams p{};
  p.k = static_cast<const uint8_t*>(a.c.k);
  p.v = static_cast<const uint8_t*>(a.c.v);
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
  int smem, slot;
  if (a.c.D == 64) {
    fn = split ? tc_kernel<64, true>() : tc_kernel<64, false>();
    smem = split ? TSmem<64, true>::total : TSmem<64, false>::total;
    slot = split ? 1 : 0;
  } else {
    fn = split ? tc_kernel<128, true>() : tc_kernel<128, false>();
    smem = split ? TSmem<128, true>::total : TSmem<128, false>::total;
    slot = split ? 3 : 2;
  }
  if (n_row_tiles == 0) return cudaSuccess;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevicesTC) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(g_tc_mu);
    if (!g_tc_attr[dev][slot]) {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
      if (e != cudaSuccess) return e;
      g_tc_attr[dev][slot] = true;
    }
  }
  const dim3 grid(n_row_tiles, a.c.Hkv, a.B);
  void* args[] = {&p};
  return cudaLaunchKernel(fn, grid, dim3(kThreadsTC), args, smem, st);
}

}  // namespace pkv
