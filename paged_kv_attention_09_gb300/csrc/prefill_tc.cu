// prefill_tc.cu — chunked-prefill attention on the 5th-generation tensor cores (tcgen05).
//
// Sources: "Tiny-LLM-Inference Project_Status" (chunked prefill/decode scheduling; the
// chunked-prefill SDPA path; BF16 KV with its own paged-attention kernel) and "tinyloop
// Current Status" (chunked prefill, chunk 512; GQA; 16-token pages).  Row i of a chunk
// of length Lq sits at position context_len - Lq + i and attends causally to positions
// 0..that position (the chunk's own K/V are appended first); under a sliding window of W
// tokens ("tinyloop Current Status", KV cache modes table) to the last W of them only,
// and the block's tiles start at the page of its lowest window start.
//
// One block computes 128 query rows — (chunk token, query head) pairs of one GQA group,
// token-major — against the group's paged K/V in tiles of 64 keys (4 pages):
//   warps 9, 10  producers of K and of V: one bulk copy per BF16 page block (already
//             stored as tensor-core tiles) into a ring each; two threads, so that K runs
//             ahead of V (the V ring is paced by the P.V products, late in each tile);
//   warp 8    score MMAs: S = Q K^T (M=128, N=64) into one of two TMEM score buffers;
//   warp 11   P.V MMAs: O += P V (M=128, N=head_dim) into one of two TMEM accumulators;
//             one thread each issues tcgen05.mma and tracks completion with
//             tcgen05.commit on mbarriers: two issuers, so that one waits on its barriers
//             while the other keeps the tensor pipe fed;
//   warps 0-7 softmax, two groups of four warps: group g takes key tiles g, g+2, g+4, ...
//             with its own running max and sum, its own score buffer, P buffer and O
//             accumulator, one thread per row (one TMEM lane, 64 keys).  The groups work on
//             two tiles at once and never wait for each other; their (max, sum, O) are
//             merged once at the end.  A thread reads S from TMEM, applies the causal mask
//             and the online softmax in FP32, and writes P back into TMEM as a BF16 high
//             part and a BF16 remainder (two MMAs per page, A operand read from TMEM) so
//             that the product keeps ~16 bits and P never crosses shared memory.  The running max is only raised when it grows by more than 2^8
//             (the group's accumulator in TMEM is rescaled then), so the P.V MMAs
//             accumulate without a per-tile round trip through registers.
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
constexpr int kSoftWarps = 8;           // two groups of 4 warps, one thread per query row
constexpr int kSoftThreads = kSoftWarps * 32;
constexpr int kThreadsTC = (kSoftWarps + 4) * 32;  // + two MMA issuers, K and V producers
constexpr float kRescaleLog2 = 8.f;  // raise the running max only beyond this margin

#ifdef PKV_TEST_HOOKS
// Test builds only: when set, each softmax group's first wait for scores gives up at once
// (as a wait that ran out would), so that the timeout path runs: the other roles' waits
// then run out on their own limits, every copy and product still drains, and the call
// reports PKV_DEV_TIMEOUT with NaN rows.
__device__ int g_test_prefill_fail_first_wait = 0;
#endif

struct TParams {
  const uint8_t* k;
  const uint8_t* v;
  const void* q;
  const int32_t* qsl;
  const int32_t* bt;
  const int32_t* lens;
  float* out;
  int32_t* dev_status;
  // key-range split: each row tile's key tiles are divided among ksplit blocks, which
  // leave partial (max, sum, O) states in the workspace for the last of them to merge
  int ksplit;
  float* ws_o;      // [tile][split][row][D]
  float* ws_m;      // [tile][split][row]
  float* ws_l;      // [tile][split][row]
  int* ws_ticket;   // [tile]
  int q_dtype, Hkv, Hq, G, MB, num_pages;
  int window;  // sliding window in tokens (0: none)
  float scale_log2;
};

template <int D, bool QSPLIT>
struct TSmem {
  static constexpr int kBlk = kPage * D * 2;           // one BF16 page block (K or V)
  static constexpr int qTile = kRowsTC * D * 2;        // one BF16 query tile
  static constexpr int stage = kPagesTC * kBlk;        // the K (or V) blocks of one tile
  static constexpr int KST = QSPLIT ? 2 : 3;           // stages of the V ring (one tile each)
  static constexpr int KSP = 2;                        // stages of the K ring (a tile pair each)
  static constexpr int kStage = 2 * stage;
  static constexpr int q0 = 0;
  static constexpr int k0 = q0 + (QSPLIT ? 2 : 1) * qTile;
  static constexpr int v0 = k0 + KSP * kStage;
  static constexpr int bar0 = v0 + KST * stage;
  // barriers: k_full[2], k_empty[2] (+1 spare each), v_full[3], v_empty[3]; s_full,
  // s_free (+1 spare each); per softmax group p_full[2], o_done[2]; final MMA drain; the
  // groups' final exchange
  static constexpr int nbars = 22;
  static constexpr int misc0 = bar0 + nbars * 8;        // TMEM base address, flags
  static constexpr int xch0 = misc0 + 16;  // final exchange: max [2 groups][128], sum [2][128]
  static constexpr int total = xch0 + 2 * 2 * kRowsTC * 4;
  // TMEM columns: O of group 0 [0, D), O of group 1 [D, 2D), S of a tile pair at 2D
  // (group g's 64 keys at 2D + 64 g),
  // P of group g at 2D + 128 + 64 g (BF16 pairs: high parts in the first 32 columns,
  // remainders in the next 32)
  static constexpr int sCol = 2 * D, pCol = 2 * D + 2 * kKeysTC;
  static constexpr int tmemCols = (2 * D + 4 * kKeysTC) <= 256 ? 256 : 512;
};

// Byte offset of element (row, col) in a no-swizzle K-major tile whose K extent is
// kext elements: core matrix (row / 8, col / 8), row % 8, element col % 8.
__device__ __forceinline__ uint32_t tile_off(int row, int col, int kext) {
  return ((((row >> 3) * (kext >> 3)) + (col >> 3)) << 7) + ((row & 7) << 4) + ((col & 7) << 1);
}

// Index of a row tile of the launch: [sequence][kv head][row tile].
__device__ __forceinline__ int tile_index(const TParams& p, int tile, int g, int b) {
  return (b * p.Hkv + g) * (gridDim.x / p.ksplit) + tile;
}

// Key-range split: the block that takes a row tile's last ticket (an atomic, no waiting)
// merges the ksplit partial states of its 128 rows, in split order, into the output,
// and resets the ticket.  `scratch`: ((ksplit + 1) x 128) floats of shared memory.
template <int D>
__device__ __noinline__ void split_merge(const TParams& p, int tile, int g, int b, int q0, int nrows,
                                         int err, int tid, uint8_t* scratch) {
  __shared__ int s_last;
  // The parameters are read once into registers: this function is not inlined, so each
  // use of p would be a load through a generic pointer, repeated after every store.
  const int KS = p.ksplit, G = p.G, Hq = p.Hq;
  float* const out = p.out;
  const float* const ws_o = p.ws_o;
  const float* const ws_m = p.ws_m;
  const float* const ws_l = p.ws_l;
  const int tix = tile_index(p, tile, g, b);
  __threadfence();
  __syncthreads();
  int* ticket = p.ws_ticket + tix;
  if (tid == 0) s_last = atomicAdd(ticket, 1) == KS - 1;
  __syncthreads();
  if (!s_last) return;
  __threadfence();
  const size_t base = static_cast<size_t>(tix) * KS * kRowsTC;
  const int row0 = tile * kRowsTC;
  float* wts = reinterpret_cast<float*>(scratch);  // [split][row], then [row] 1 / sum
  if (tid < kRowsTC) {
    const int r = tid;
    float m[3], l[3];
#pragma unroll
    for (int s = 0; s < 3; ++s) {  // every load in flight at once
      m[s] = s < KS ? __ldcg(ws_m + base + s * kRowsTC + r) : -CUDART_INF_F;
      l[s] = s < KS ? __ldcg(ws_l + base + s * kRowsTC + r) : 0.f;
    }
    const bool poisoned = isnan(m[0]) || isnan(m[1]) || isnan(m[2]);
    const float M = fmaxf(fmaxf(m[0], m[1]), m[2]);
    float L = 0.f;
#pragma unroll
    for (int s = 0; s < 3; ++s) {
      const float f = m[s] == -CUDART_INF_F ? 0.f : fast_exp2(m[s] - M);
      if (s < KS) wts[s * kRowsTC + r] = f;
      L += l[s] * f;
    }
    wts[KS * kRowsTC + r] = poisoned ? CUDART_NAN_F : 1.f / L;
  }
  __syncthreads();
  if (!err) {
    constexpr int D4 = D / 4;
    constexpr int CH = 4;  // output chunks per thread and round: their loads go out together
    for (int c0 = tid; c0 < kRowsTC * D4; c0 += CH * kThreadsTC) {
      float4 v[CH][3];
#pragma unroll
      for (int u = 0; u < CH; ++u) {
        const int c = c0 + u * kThreadsTC;
        const int r = c / D4, d4 = c % D4;
#pragma unroll
        for (int s = 0; s < 3; ++s)
          v[u][s] = c < kRowsTC * D4 && s < KS
                        ? __ldcg(reinterpret_cast<const float4*>(ws_o + (base + s * kRowsTC + r) * D) + d4)
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < CH; ++u) {
        const int c = c0 + u * kThreadsTC;
        const int r = c / D4, d4 = c % D4;
        const int rho = row0 + r;
        if (c >= kRowsTC * D4 || rho >= nrows) continue;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < 3; ++s) {
          if (s < KS) {
            const float f = wts[s * kRowsTC + r];
            acc.x += v[u][s].x * f; acc.y += v[u][s].y * f; acc.z += v[u][s].z * f; acc.w += v[u][s].w * f;
          }
        }
        const float inv = wts[KS * kRowsTC + r];
        float* dst = out + (static_cast<size_t>(q0 + rho / G) * Hq + g * G + rho % G) * D;
        reinterpret_cast<float4*>(dst)[d4] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      }
    }
  }
  if (tid == 0) *ticket = 0;  // leave the counter ready for the next call
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
  uint64_t* xfin = bars + 21;  // the two softmax groups' final (max, sum) exchange
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Sm::misc0);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + Sm::misc0 + 4);
  __shared__ int s_err;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = blockIdx.y, b = blockIdx.z;
  const int tile = blockIdx.x / p.ksplit, ks = blockIdx.x % p.ksplit;
  const int row0 = tile * kRowsTC;
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
  // Sliding window of W tokens: row position pos sees keys pos - W + 1 .. pos.  Keys
  // below lo_blk are seen by no row of the block, keys below lo_max by some rows only.
  // The block's key range starts at kbase, the first key of the page holding lo_blk;
  // tiles are counted from there.
  const int win = p.window;
  const int lo_blk = win > 0 ? max(0, p_first - win + 1) : 0;
  const int lo_max = win > 0 ? p_last - win + 1 : 0;
  const int kb0 = (lo_blk / kPage) * kPage;
  const int32_t* bt = p.bt + static_cast<size_t>(b) * p.MB;
  if (tid == 0) s_err = err;
  __syncthreads();
  for (int j = kb0 / kPage + tid; j < (n_keys0 + kPage - 1) / kPage; j += kThreadsTC) {
    const int pg = bt[j];
    if (pg < 0 || pg >= p.num_pages) atomicOr(&s_err, 0x1);  // PKV_DEV_BAD_PAGE
  }
  __syncthreads();
  err = s_err;
  // this block's share of the key tiles: [t0, t1) of the row tile's range from kb0
  const int nt_all = err ? 0 : (n_keys0 - kb0 + kKeysTC - 1) / kKeysTC;
  const int t0 = ks * nt_all / p.ksplit, t1 = (ks + 1) * nt_all / p.ksplit;
  const int n_keys = err ? 0 : min(n_keys0, kb0 + t1 * kKeysTC);
  const int kbase = err ? 0 : kb0 + t0 * kKeysTC;
  const int n_pages = max(0, (n_keys - kbase + kPage - 1) / kPage);  // pages from kbase on
  const int n_tiles = t1 - t0;

  // ---- set-up: TMEM, barriers, the query tile(s)
  if (warp == kSoftWarps) {
    tc::tmem_alloc(tmem_slot, Sm::tmemCols);
    tc::tmem_relinquish();
  }
  if (tid == 0) {
    for (int i = 0; i < Sm::nbars; ++i) {
      // p_full: one arrival per thread of the group; s_free and the exchange: every
      // softmax thread; the rest: one arrival (or tcgen05.commit)
      const int count = i == 14 ? kSoftThreads   // s_free: both groups read the pair
                        : (i == 16 || i == 17) ? kSoftThreads / 2
                        : i == 21 ? kSoftThreads
                        : i == 20 ? 2  // the final drain: one commit from each MMA issuer
                        : 1;
      mbar_init(&bars[i], count);
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

  if (n_tiles > 0 && (warp == kSoftWarps + 1 || warp == kSoftWarps + 2)) {
    // ---------------------------------------------------------------- producers
    // warp kSoftWarps + 1 fills the K ring, warp kSoftWarps + 2 the V ring
    if (lane == 0) {
      const bool isK = warp == kSoftWarps + 1;
      const uint64_t pol = l2_evict_last_policy();  // every row tile of the group rereads them
      // K moves a tile pair (8 pages) per stage, V one tile (4 pages) per stage
      const int RS = isK ? Sm::KSP : Sm::KST;
      const int per = isK ? 2 * kPagesTC : kPagesTC;
      const int sbytes = isK ? Sm::kStage : Sm::stage;
      const int n_units = isK ? (n_tiles + 1) / 2 : n_tiles;
      uint64_t* full = isK ? k_full : v_full;
      uint64_t* empty = isK ? k_empty : v_empty;
      const uint8_t* src = isK ? p.k : p.v;
      uint8_t* ring = smem + (isK ? Sm::k0 : Sm::v0);
      const int32_t* btw = bt + kbase / kPage;  // the block's first page
      int issued = 0;
      for (int j = 0; j < n_units; ++j) {
        const int st = j % RS, use = j / RS;
        const int np = min(per, n_pages - j * per);
        if (j >= RS && !mbar_wait(&empty[st], (use - 1) & 1)) { *abort_flag = 1; break; }
        if (*abort_flag) break;
        mbar_arrive_expect_tx(&full[st], np * Sm::kBlk);
        for (int q = 0; q < np; ++q) {
          const size_t blk = static_cast<size_t>(btw[j * per + q]) * p.Hkv + g;
          bulk_g2s(ring + st * sbytes + q * Sm::kBlk, src + blk * Sm::kBlk, Sm::kBlk, &full[st], pol);
        }
        issued = j + 1;
      }
      // leave nothing in flight: the copies of the last issued stages have landed
      for (int j = max(0, issued - RS); j < issued; ++j) (void)mbar_wait(&full[j % RS], (j / RS) & 1);
    }
  } else if (n_tiles > 0 && (warp == kSoftWarps || warp == kSoftWarps + 3)) {
    // ---------------------------------------------------------------- MMA issuers
    if (lane == 0) {
      constexpr uint32_t idS = tc::idesc_bf16_f32(kRowsTC, 2 * kKeysTC);  // a tile pair
      constexpr uint32_t idO = tc::idesc_bf16_f32(kRowsTC, D);
      constexpr uint32_t sboQK = (D / 8) * 128;  // 8-row groups of Q and of K
      const uint32_t qhi = sbase + Sm::q0, qlo = sbase + Sm::q0 + Sm::qTile;
      constexpr int KST = Sm::KST;
      // Operand descriptors are built once and stepped by constant offsets, so that issuing
      // an MMA costs a few instructions.
      const uint64_t dQhi = tc::smem_desc(qhi, 128, sboQK), dQlo = tc::smem_desc(qlo, 128, sboQK);
      const uint64_t dK0 = tc::smem_desc(sbase + Sm::k0, 128, sboQK);
      const uint64_t dV0 = tc::smem_desc(sbase + Sm::v0, 128, 256);
      // S of tile pair pr (tiles 2 pr and 2 pr + 1: 128 keys, one N=128 MMA per k-step)
      // into the score buffer, once both groups have read the previous pair's scores
      constexpr int KSP = Sm::KSP;
      auto issue_s = [&](int pr) -> bool {
        if (!mbar_wait(&k_full[pr % KSP], (pr / KSP) & 1)) return false;
        if (pr >= 1 && !mbar_wait(&s_free[0], (pr - 1) & 1)) return false;
        if (*abort_flag) return false;
        tc::fence_after_sync();
        const uint64_t dK = tc::desc_add(dK0, (pr % KSP) * Sm::kStage);
        const uint32_t tS = tmem + Sm::sCol;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const uint64_t bd = tc::desc_add(dK, ks * 256);
          tc::mma_bf16(tS, tc::desc_add(dQhi, ks * 256), bd, idS, ks > 0);
          if constexpr (QSPLIT) tc::mma_bf16(tS, tc::desc_add(dQlo, ks * 256), bd, idS, true);
        }
        tc::commit(&s_full[0]);
        tc::commit(&k_empty[pr % KSP]);
        return true;
      };
      // O_y += P_i V_i into the accumulator of group y = i & 1 (its first tile starts it)
      auto issue_pv = [&](int i) -> bool {
        const int y = i & 1;
        if (!mbar_wait(&p_full[y], (i >> 1) & 1)) return false;
        if (!mbar_wait(&v_full[i % KST], (i / KST) & 1)) return false;
        tc::fence_after_sync();
        const uint64_t dV = tc::desc_add(dV0, (i % KST) * Sm::stage);
        const uint32_t tP = tmem + Sm::pCol + kKeysTC * y;  // A = P straight from TMEM
#pragma unroll
        for (int q = 0; q < kPagesTC; ++q) {
          const uint64_t bd = tc::desc_add(dV, q * Sm::kBlk);
#pragma unroll
          for (int part = 0; part < 2; ++part)
            tc::mma_bf16_ts(tmem + D * y, tP + 32 * part + 8 * q, bd, idO, !(i < 2 && q == 0 && part == 0));
        }
        tc::commit(&o_done[y]);
        tc::commit(&v_empty[i % KST]);
        return true;
      };
      // Warp 8 runs ahead through the tile pairs (bounded by the one score buffer);
      // warp 11 follows the softmax groups with the P.V products.
      bool ok = true;
      if (warp == kSoftWarps) {
        for (int pr = 0; pr < (n_tiles + 1) / 2 && ok; ++pr) ok = issue_s(pr);
      } else {
        for (int i = 0; i < n_tiles && ok; ++i) ok = issue_pv(i);
      }
      if (!ok) *abort_flag = 1;
      // every MMA either issuer started has completed before TMEM is released
      tc::commit(fin);
      (void)mbar_wait(fin, 0);
    }
  } else if (n_tiles > 0) {
    // ---------------------------------------------------------------- softmax rows
    // group grp (= hf) owns tiles grp, grp + 2, ...: score buffer, P buffer and O
    // accumulator grp; thread = row r (TMEM lane 32 (warp % 4) + lane)
    const int grp = hf;
    const int pos = valid_row ? L - Lq + rho / p.G : p_first;
    const int lo_row = win > 0 ? pos - win + 1 : 0;  // first key of the row's window
    const uint32_t lane_base = static_cast<uint32_t>(32 * (warp & 3)) << 16;
    const uint32_t tO = tmem + lane_base + D * grp;
    const float sl = p.scale_log2;
    float m_used = -CUDART_INF_F, l = 0.f;
    bool ok = true;
    int n_mine = 0;  // tiles this group has finished
    for (int j = grp; j < n_tiles; j += 2, ++n_mine) {
      const int k = j >> 1;  // this group's k-th tile
      ok = mbar_wait(&s_full[0], k & 1) && !*abort_flag;  // the scores of pair k
#ifdef PKV_TEST_HOOKS
      if (k == 0 && g_test_prefill_fail_first_wait) ok = false;  // a wait that gives up
#endif
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      tc::fence_after_sync();
      float s[64];
      {
        float t0[32], t1[32];
        tc::ld32(tmem + lane_base + Sm::sCol + kKeysTC * grp, t0);
        tc::ld32(tmem + lane_base + Sm::sCol + kKeysTC * grp + 32, t1);
#pragma unroll
        for (int u = 0; u < 32; ++u) { s[u] = t0[u]; s[32 + u] = t1[u]; }
      }
      tc::fence_before_sync();
      mbar_arrive(&s_free[0]);
      const int key0 = kbase + j * kKeysTC;
      // raw scores; the scale (> 0) is applied inside the exponent with one FMA
      if (key0 + kKeysTC - 1 > p_first || key0 + kKeysTC > n_keys || key0 < lo_max) {
#pragma unroll
        for (int u = 0; u < 64; ++u)
          s[u] = (key0 + u <= pos && key0 + u >= lo_row) ? s[u] : -CUDART_INF_F;
      }
      float t[32];  // pairwise max tree (a flat chain would be 63 dependent steps)
#pragma unroll
      for (int u = 0; u < 32; ++u) t[u] = fmaxf(s[u], s[u + 32]);
#pragma unroll
      for (int w2 = 16; w2 >= 1; w2 >>= 1)
#pragma unroll
        for (int u = 0; u < w2; ++u) t[u] = fmaxf(t[u], t[u + w2]);
      const float mx = t[0] * sl;
      const bool need = mx > m_used + kRescaleLog2;
      if (__any_sync(0xffffffffu, need)) {
        const float m_new = need ? mx : m_used;
        const float f = need ? fast_exp2(m_used - m_new) : 1.f;
        if (k >= 1) {
          // O holds this group's earlier tiles: wait for their last P.V, then rescale
          ok = mbar_wait(&o_done[grp], (k - 1) & 1);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          tc::fence_after_sync();
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tc::ld32(tO + 32 * c, o);
#pragma unroll
            for (int u = 0; u < 32; ++u) o[u] *= f;
            tc::st32(tO + 32 * c, o);
          }
        }
        l *= f;
        m_used = m_new;
      }
      if (k >= 1) {  // P buffer grp was read by the P.V of this group's previous tile
        ok = mbar_wait(&o_done[grp], (k - 1) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      }
      // (a group can meet a row's keys only in a later tile: while its max is still -inf,
      // every probability is 0, not exp2(-inf + inf))
      const float nm = m_used == -CUDART_INF_F ? 0.f : -m_used;
      const uint32_t tP = tmem + lane_base + Sm::pCol + kKeysTC * grp;
      float2 ls[2];
      const float2 sl2 = make_float2(sl, sl), nm2 = make_float2(nm, nm);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {  // keys 32 hh .. 32 hh + 31 -> P columns 16 hh ..
        uint32_t h[16], lo[16];
#pragma unroll
        for (int u = 0; u < 16; ++u) {
          const float2 x = __ffma2_rn(make_float2(s[32 * hh + 2 * u], s[32 * hh + 2 * u + 1]), sl2, nm2);
          const float2 pe = make_float2(fast_exp2(x.x), fast_exp2(x.y));
          if (u == 0) ls[hh] = pe;
          else ls[hh] = __fadd2_rn(ls[hh], pe);
          const __nv_bfloat162 hv = __floats2bfloat162_rn(pe.x, pe.y);
          const float2 hf2 = __bfloat1622float2(hv);
          const float2 r2 = __fadd2_rn(pe, make_float2(-hf2.x, -hf2.y));
          const __nv_bfloat162 lv = __floats2bfloat162_rn(r2.x, r2.y);
          h[u] = *reinterpret_cast<const uint32_t*>(&hv);
          lo[u] = *reinterpret_cast<const uint32_t*>(&lv);
        }
        tc::st16_nowait(tP + 16 * hh, h);
        tc::st16_nowait(tP + 32 + 16 * hh, lo);
      }
      tc::st_wait();
      l += (ls[0].x + ls[0].y) + (ls[1].x + ls[1].y);
      const int kz = min(kKeysTC, n_keys - key0);      // tile keys kz .. 63: past the end
      const int hz = j == 0 && ks == 0 ? lo_blk - kbase : 0;  // tile keys 0 .. hz - 1: before the window
      if (kz < kKeysTC || hz > 0) {
        // keys no row may see: pages not loaded, page padding, or keys of the first page
        // before every row's window; they may hold anything (even NaN), so zero them in V
        // so that 0 * V stays 0 (after this tile's V copies have landed)
        ok = mbar_wait(&v_full[j % Sm::KST], (j / Sm::KST) & 1);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        uint8_t* vst = smem + Sm::v0 + (j % Sm::KST) * Sm::stage;
        for (int idx = r; idx < (kKeysTC - kz + hz) * D; idx += kRowsTC) {
          const int u = idx / D, d = idx % D;
          const int key = u < hz ? u : kz + (u - hz);
          *reinterpret_cast<__nv_bfloat16*>(vst + (key >> 4) * Sm::kBlk + bf16_v_off(d, key & 15)) =
              __float2bfloat16_rn(0.f);
        }
      }
      fence_proxy_async_smem();  // zeroed V becomes visible to the tensor cores
      tc::fence_before_sync();   // and so does P in TMEM
      mbar_arrive(&p_full[grp]);
    }
    if (ok && n_mine > 0) {  // this group's last P.V
      ok = __all_sync(0xffffffffu, mbar_wait(&o_done[grp], (n_mine - 1) & 1));
    }
    tc::fence_before_sync();
    // the two groups' (max, sum) of this row, exchanged once
    float* xm = reinterpret_cast<float*>(smem + Sm::xch0);  // [group][row]
    float* xl = xm + 2 * kRowsTC;
    xm[grp * kRowsTC + r] = m_used;
    xl[grp * kRowsTC + r] = l;
    mbar_arrive(xfin);
    ok = __all_sync(0xffffffffu, mbar_wait(xfin, 0) && ok);
    if (!ok) *abort_flag = 1;
    if (ok) {
      tc::fence_after_sync();
      const float m_o = xm[(grp ^ 1) * kRowsTC + r], l_o = xl[(grp ^ 1) * kRowsTC + r];
      const float M = fmaxf(m_used, m_o);
      const float a_me = m_used == -CUDART_INF_F ? 0.f : fast_exp2(m_used - M);
      const float a_ot = m_o == -CUDART_INF_F ? 0.f : fast_exp2(m_o - M);
      const float lsum = l * a_me + l_o * a_ot;
      // a split block leaves its unnormalised partial for the merge
      const bool partial = p.ksplit > 1;
      const float inv = partial ? 1.f : 1.f / lsum;
      const float wA = (grp == 0 ? a_me : a_ot) * inv, wB = (grp == 0 ? a_ot : a_me) * inv;
      const bool hasB = n_tiles > 1;  // group 1's accumulator holds data
      const size_t pidx = (static_cast<size_t>(tile_index(p, tile, g, b)) * p.ksplit + ks) * kRowsTC + r;
      float* dst = !valid_row ? nullptr
                   : partial ? p.ws_o + pidx * D
                             : p.out + (static_cast<size_t>(q0 + rho / p.G) * p.Hq + g * p.G + rho % p.G) * D;
      if (partial && valid_row && grp == 0) {
        p.ws_m[pidx] = M;
        p.ws_l[pidx] = lsum;
      }
      // group grp writes head_dim columns [grp D/2, (grp + 1) D/2) of its row
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const int col = (D / 2) * grp + 32 * c;
        float oa[32], ob[32];
        tc::ld32(tmem + lane_base + col, oa);
        if (hasB) {
          tc::ld32(tmem + lane_base + D + col, ob);
        } else {
#pragma unroll
          for (int u = 0; u < 32; ++u) ob[u] = 0.f;
        }
        if (dst) {
#pragma unroll
          for (int u = 0; u < 32; u += 4)
            *reinterpret_cast<float4*>(dst + col + u) =
                make_float4(oa[u] * wA + ob[u] * wB, oa[u + 1] * wA + ob[u + 1] * wB,
                            oa[u + 2] * wA + ob[u + 2] * wB, oa[u + 3] * wA + ob[u + 3] * wB);
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
    if (p.ksplit > 1 && hf == 0)  // a poisoned partial turns the merged row into NaN
      p.ws_m[(static_cast<size_t>(tile_index(p, tile, g, b)) * p.ksplit + ks) * kRowsTC + r] = CUDART_NAN_F;
  }
  if (warp == kSoftWarps) tc::tmem_dealloc(tmem, Sm::tmemCols);
  if (p.ksplit > 1) {
    // a block with no key tiles (a short row range split more ways than it has tiles)
    // leaves an empty partial
    if (n_tiles == 0 && !err && valid_row && hf == 0) {
      const size_t pidx = (static_cast<size_t>(tile_index(p, tile, g, b)) * p.ksplit + ks) * kRowsTC + r;
      p.ws_m[pidx] = -CUDART_INF_F;
      p.ws_l[pidx] = 0.f;
      for (int d = 0; d < D; d += 4)
        *reinterpret_cast<float4*>(p.ws_o + pidx * D + d) = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    split_merge<D>(p, tile, g, b, q0, nrows, err, tid, smem + Sm::xch0);
  }
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

int prefill_tc_blocks_per_sm(int q_dtype) {
  (void)q_dtype;
  return 1;  // the kernel takes all of an SM's tensor memory
}

cudaError_t launch_prefill_tc(const PrefillArgs& a, int n_row_tiles, int ksplit, cudaStream_t st) {
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
  p.window = a.c.window;
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
  p.ksplit = ksplit;
  if (ksplit > 1) {
    const size_t tiles = static_cast<size_t>(n_row_tiles) * a.c.Hkv * a.B;
    uint8_t* base = static_cast<uint8_t*>(a.ws);
    p.ws_ticket = reinterpret_cast<int*>(base);
    float* f = reinterpret_cast<float*>(base + ((tiles * 4 + 255) / 256) * 256);
    const size_t rows = tiles * ksplit * kRowsTC;
    p.ws_o = f;
    p.ws_m = f + rows * a.c.D;
    p.ws_l = p.ws_m + rows;
  }
  const dim3 grid(n_row_tiles * ksplit, a.c.Hkv, a.B);
  void* args[] = {&p};
  return cudaLaunchKernel(fn, grid, dim3(kThreadsTC), args, smem, st);
}

}  // namespace pkv

#ifdef PKV_TEST_HOOKS
// Test builds only: switches the give-up-at-once first score wait (see above) on or off.
extern "C" int pkv_test_prefill_fail_first_wait(int on) {
  return cudaMemcpyToSymbol(pkv::g_test_prefill_fail_first_wait, &on, sizeof(int)) == cudaSuccess ? 0 : 1;
}
#endif
