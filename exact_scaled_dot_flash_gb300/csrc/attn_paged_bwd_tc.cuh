// attn_paged_bwd_tc.cuh - the backward over a paged cache on the tcgen05
// tensor cores (F16/BF16, D in {64, 128}, page_size a multiple of 8 that
// divides 128 or a multiple of 128).
//
// Source: ruDNN user guide, section 11 (backward of paged attention): dq for
// the packed queries and the history gradients dk, dv in the cache's shape,
// the probabilities recomputed from the forward's statistics; ordered, no
// atomics.
//
// The two kernels are the dense backward's (attn_bwd_tc.cuh: 384 threads, 8
// elementwise warps, a TMA producer, an MMA issuer; the same MMA order, TMEM
// map and packing) with paged addressing:
//  - rows and columns of the query side are (query, head) pairs of one
//    sequence and of a block of gp query heads sharing a kv head (gp = Hq/Hkv
//    when it divides 128, else 1), packed query-major: pair = query * gp +
//    head-in-block; a tile of 128 pairs is one TMA box of the 4-D view
//    [queries, Hq/gp, gp, D] (the paged forward's view), so a decode step's
//    gp heads share one tile;
//  - a K/V tile of 128 keys of a sequence is gathered page by page through
//    the 4-D view [pages, page_size, Hkv, D] of the cache (boxes of
//    min(page_size, 128) rows; a page id outside the cache loads zeros);
//  - pair p sees key j when p's query exists in the sequence, j < seq_len and,
//    causal, j <= its position (explicit, or the newest-token default);
//  - paged_dkdv_tc_kernel: CTA = (sequence, 128-key block, kv head), K and V
//    resident, the (Q, dO) tiles of every head block of the group streamed.
//    Its key rows are stored straight into the cache gradients only for the
//    physical pages with exactly one reader (the reverse index's count); pages
//    read by several sequences (or blocks), or by none, are left to the fp32
//    FMA key-major kernel, which sums their readers in the index order;
//  - paged_dq_tc_kernel: CTA = (sequence, head block, 128 pairs), Q and dO
//    resident, the sequence's K/V tiles streamed; the rows of its sequence
//    are stored directly.
#pragma once

#include <atomic>

#include "attn_bwd_tc.cuh"
#include "paged_bwd.h"
#include "params.h"
#include "ptx.cuh"

namespace attn {
namespace pbwd {
namespace tc {

using bwdtc::BR;
using bwdtc::Cfg;
using bwdtc::DqCfg;
using bwdtc::NUM_THREADS;
using bwdtc::REG_EW;
using bwdtc::REG_OTHER;
using bwdtc::TMEM_COLS;
using bwdtc::WARP_MMA;
using bwdtc::WARP_TMA;
using bwdtc::kstep16;
using bwdtc::store_row16;
using bwdtc::tmem_a_kstep;
using bwdtc::tmem_ld64;
using bwdtc::tmem_st_packed64;

__device__ __forceinline__ int seq_keys(const PagedParams& pp, int s) {
  const int64_t cap = static_cast<int64_t>(pp.max_pages) * pp.page_size;
  const int L = __ldg(pp.seq_lens + s);
  return L < 0 ? 0 : (L > cap ? static_cast<int>(cap) : L);
}

__device__ __forceinline__ void seq_rows(const PagedParams& pp, int s, int& q0, int& n) {
  int a = __ldg(pp.q_offsets + s), b = __ldg(pp.q_offsets + s + 1);
  a = a < 0 ? 0 : (a > pp.num_queries ? pp.num_queries : a);
  b = b < 0 ? 0 : (b > pp.num_queries ? pp.num_queries : b);
  q0 = a;
  n = b > a ? b - a : 0;
}

// Load the 128 keys [key0, key0 + 128) of a sequence's page table into a
// swizzled tile (one box per page, or one box inside a page of >= 128 keys).
template <int D>
__device__ __forceinline__ void load_kv_tile(uint32_t dst, const CUtensorMap* m, uint32_t bar, const int32_t* table,
                                             const PagedParams& pp, int key0, int hk) {
  using C = Cfg<D>;
  const int box_rows = pp.page_size < BR ? pp.page_size : BR;
  const int boxes = BR / box_rows;
  for (int i = 0; i < boxes; ++i) {
    const int key = key0 + i * box_rows;
    const int pidx = key / pp.page_size;
    const int page = pidx < pp.max_pages ? __ldg(table + pidx) : -1;  // -1: a zero-filled box
    // checked build: the box lands inside its chunk of the tile (a skipped
    // copy leaves the tile's barrier to time out)
    if (!range_in_bounds(pp.status, i * box_rows, box_rows, BR)) continue;
    for (int c = 0; c < C::NCHUNK; ++c)
      tma_load_4d(dst + c * C::CHUNK_BYTES + i * box_rows * 128, m, bar, c * C::BOX_D, hk, key % pp.page_size,
                  page);
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    paged_dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                         const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const PagedParams pp, const TcArgs a, int kblocks, int gp) {
  using C = Cfg<D>;
  // ---- work: key block kb of sequence s, kv head hk
  const int lin = static_cast<int>(blockIdx.x);
  const int kb = lin % kblocks;
  const int rest = lin / kblocks;
  const int hk = rest % pp.Hkv, s = rest / pp.Hkv;
  const int L = seq_keys(pp, s);
  int q0, n;
  seq_rows(pp, s, q0, n);
  const int P = pp.page_size;
  const int used = (L + P - 1) / P;  // pages the sequence reads
  const int key0 = kb * BR;
  if (n == 0 || key0 >= used * P) return;  // not a block of this sequence's pages (uniform)
  const int group = pp.Hq / pp.Hkv;
  const int hblocks = group / gp;
  const int ptiles = (n * gp + BR - 1) / BR;  // tiles of 128 (query, head) pairs per head block
  const int diag = L - n;                      // default positions: query qi sits at diag + qi
  const bool dflt = pp.positions == nullptr;
  const int t_lo = (pp.causal && dflt) ? (max(0, key0 - diag) * gp) / BR : 0;
  const int per_hb = key0 < L ? max(0, ptiles - t_lo) : 0;
  const int N = per_hb * hblocks;
  const int32_t* table = pp.block_table + static_cast<size_t>(s) * pp.max_pages;

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < C::STAGES; ++st) {
      mbar_init(bar(C::BAR_FULL + st), 1);
      mbar_init(bar(C::BAR_EMPTY + st), 1);
    }
    mbar_init(bar(C::BAR_RES), 1);
    mbar_init(bar(C::BAR_S), 1);
    mbar_init(bar(C::BAR_S + 1), 1);
    mbar_init(bar(C::BAR_DP), 1);
    mbar_init(bar(C::BAR_P), 256);
    mbar_init(bar(C::BAR_DS), 256);
    mbar_init(bar(C::BAR_DONE), 1);
    mbar_init_fence();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    if (pp.status) atomicOr(pp.status, STATUS_TIMEOUT);
  };

  if (warp >= 8) {
    setmaxnreg_dec<REG_OTHER>();
    if (warp == WARP_TMA && lane == 0 && N > 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar(C::BAR_RES), 2 * C::TILE_BYTES);
      load_kv_tile<D>(sb, &tm_k, bar(C::BAR_RES), table, pp, key0, hk);
      load_kv_tile<D>(sb + C::TILE_BYTES, &tm_v, bar(C::BAR_RES), table, pp, key0, hk);
      int it = 0;
      for (; it < N; ++it) {
        const int st = it % C::STAGES;
        if (!mbar_wait(bar(C::BAR_EMPTY + st), ((it / C::STAGES) & 1) ^ 1)) { fail(); break; }
        const int hb = it / per_hb, t = t_lo + (it - hb * per_hb);
        const int hh = hk * hblocks + hb;  // head block in [0, Hq / gp)
        const int qs = q0 + t * (BR / gp);
        const uint32_t dst = sb + C::OFF_RING + st * 2 * C::TILE_BYTES;
        mbar_arrive_expect_tx(bar(C::BAR_FULL + st), 2 * C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_4d(dst + c * C::CHUNK_BYTES, &tm_q, bar(C::BAR_FULL + st), c * C::BOX_D, 0, hh, qs);
          tma_load_4d(dst + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_do, bar(C::BAR_FULL + st), c * C::BOX_D, 0, hh,
                      qs);
        }
      }
      for (int st = 0; st < C::STAGES && st < it; ++st) {
        const int fills = (it - st + C::STAGES - 1) / C::STAGES;
        if (!mbar_wait(bar(C::BAR_FULL + st), (fills - 1) & 1)) fail();
      }
      if (!mbar_wait(bar(C::BAR_RES), 0)) fail();
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer (the dense kernel's)
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_s = make_idesc_f16(BF16, BR, BR, false);
      constexpr uint32_t idesc_o = make_idesc_f16(BF16, BR, D, true);
      constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
      constexpr uint32_t RSTEP16 = (16 * 128) >> 4;
      const uint64_t dk_a = smem_desc(sb, 16, C::SBO, C::LAYOUT);
      const uint64_t dv_a = smem_desc(sb + C::TILE_BYTES, 16, C::SBO, C::LAYOUT);
      const uint64_t ring_k = smem_desc(sb + C::OFF_RING, 16, C::SBO, C::LAYOUT);
      const uint64_t ring_mn = smem_desc(sb + C::OFF_RING, C::CHUNK_BYTES, C::SBO, C::LAYOUT);
      bool ok = true;
      auto issue_s = [&](int it) {
        const int st = it % C::STAGES;
        if (!warp_wait(bar(C::BAR_FULL + st), (it / C::STAGES) & 1)) return false;
        tc_fence_after();
        const uint64_t q = ring_k + st * 2 * TILE16;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::KSTEPS_D; ++k)
            umma_ss(tmem + 0, dk_a + kstep16<D>(k), q + kstep16<D>(k), idesc_s, k > 0 ? 1u : 0u);
          umma_commit(bar(C::BAR_S));
        }
        __syncwarp();
        return true;
      };
      auto issue_dp = [&](int it) {
        const int st = it % C::STAGES;
        const uint64_t g = ring_k + st * 2 * TILE16 + TILE16;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::KSTEPS_D; ++k)
            umma_ss(tmem + BR, dv_a + kstep16<D>(k), g + kstep16<D>(k), idesc_s, k > 0 ? 1u : 0u);
          umma_commit(bar(C::BAR_DP));
        }
        __syncwarp();
      };
      if (N > 0) {
        if (!warp_wait(bar(C::BAR_RES), 0)) ok = false;
        tc_fence_after();
        if (ok && !issue_s(0)) ok = false;
        if (ok) issue_dp(0);
        for (int it = 0; it < N && ok; ++it) {
          const int st = it % C::STAGES;
          if (!warp_wait(bar(C::BAR_P), it & 1)) { ok = false; break; }
          tc_fence_after();
          {
            const uint64_t g = ring_mn + st * 2 * TILE16 + TILE16;
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < C::KSTEPS_R; ++k)
                umma_ts(tmem + 256, tmem + tmem_a_kstep(k), g + k * RSTEP16, idesc_o, (it > 0 || k > 0) ? 1u : 0u);
            }
            __syncwarp();
          }
          if (it + 1 < N && !issue_s(it + 1)) { ok = false; break; }
          if (!warp_wait(bar(C::BAR_DS), it & 1)) { ok = false; break; }
          tc_fence_after();
          {
            const uint64_t q = ring_mn + st * 2 * TILE16;
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < C::KSTEPS_R; ++k)
                umma_ts(tmem + 256 + D, tmem + BR + tmem_a_kstep(k), q + k * RSTEP16, idesc_o,
                        (it > 0 || k > 0) ? 1u : 0u);
            }
            __syncwarp();
          }
          if (elect_one()) {
            umma_commit(bar(C::BAR_EMPTY + st));
          }
          __syncwarp();
          if (it + 1 < N) issue_dp(it + 1);
        }
      }
      if (!ok && lane == 0) fail();
      if (elect_one()) {
        umma_commit(bar(C::BAR_DONE));
      }
      __syncwarp();
      if (!warp_wait(bar(C::BAR_DONE), 0) && lane == 0) fail();
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- elementwise
    setmaxnreg_inc<REG_EW>();
    const int half = warp >> 2;                // pair columns [64 half, +64) of the tile
    const int row = ((warp & 3) << 5) + lane;  // key row = TMEM lane
    const int key = key0 + row;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_off, tDP = tS + BR;
    const float sc = pp.scale_log2;
    // this warp's copy of the tile's column statistics
    float* st_l2 = reinterpret_cast<float*>(smem + C::OFF_STATS) + warp * C::STATS_PER_WARP;
    float* st_ds = st_l2 + 64;
    int* st_lim = reinterpret_cast<int*>(st_l2 + 128);
    // keys past the sequence see nothing: their limit test always fails
    const int kcmp = key < L ? key : 0x7fffffff;
    // pair columns lane and lane + 32 of this warpgroup's 64 of tile `it`:
    // lse2, D and the largest visible key (-1 for a pair with no query or no
    // visible key); loaded one tile ahead so their latency hides behind a tile
    float l2v[2], dsv[2];
    int limv[2];
    auto load_stats = [&](int it) {
      const int hb = it / per_hb, t = t_lo + (it - hb * per_hb);
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int pair = t * BR + 64 * half + 32 * u + lane;
        const int qi = pair / gp;
        const int hq = hk * group + hb * gp + (pair - qi * gp);
        const size_t ri = static_cast<size_t>(q0 + (qi < n ? qi : 0)) * pp.Hq + hq;
        const bool in = qi < n && in_bounds(pp.status, static_cast<int64_t>(ri),
                                            static_cast<int64_t>(pp.num_queries) * pp.Hq);
        l2v[u] = in ? __ldg(a.lse2 + ri) : -INFINITY;
        dsv[u] = in ? __ldg(a.dsum + ri) : 0.f;
        limv[u] = 0x7ffffffe;
        if (pp.causal)
          limv[u] = dflt ? diag + qi
                         : ((in && in_bounds(pp.status, q0 + qi, pp.num_queries))
                                ? min(__ldg(pp.positions + q0 + qi), 0x7ffffffe) : -1);
      }
    };
    if (N > 0) load_stats(0);
    bool failed = false;
    for (int it = 0; it < N; ++it) {
      __syncwarp();
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const bool live = l2v[u] != -INFINITY;
        st_l2[32 * u + lane] = live ? l2v[u] : 0.f;
        st_ds[32 * u + lane] = live ? dsv[u] : 0.f;
        st_lim[32 * u + lane] = live ? limv[u] : -1;
      }
      if (it + 1 < N) load_stats(it + 1);
      __syncwarp();
      float x[64];
      const bool ok = mbar_wait(bar(C::BAR_S), it & 1);
      if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
      tc_fence_after();
      tmem_ld64<BF16>(tS + 64 * half, x);
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 l4 = reinterpret_cast<const float4*>(st_l2)[c4];
        const int4 m4 = reinterpret_cast<const int4*>(st_lim)[c4];
        x[4 * c4 + 0] = kcmp <= m4.x ? fast_exp2(x[4 * c4 + 0] * sc - l4.x) : 0.f;
        x[4 * c4 + 1] = kcmp <= m4.y ? fast_exp2(x[4 * c4 + 1] * sc - l4.y) : 0.f;
        x[4 * c4 + 2] = kcmp <= m4.z ? fast_exp2(x[4 * c4 + 2] * sc - l4.z) : 0.f;
        x[4 * c4 + 3] = kcmp <= m4.w ? fast_exp2(x[4 * c4 + 3] * sc - l4.w) : 0.f;
      }
      tmem_st_packed64<BF16>(tS + 64 * half, x);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::BAR_P));
      const bool ok2 = mbar_wait(bar(C::BAR_DP), it & 1);
      if (__any_sync(0xffffffffu, !ok2)) { failed = true; break; }
      tc_fence_after();
      float dp[64];
      tmem_ld64<BF16>(tDP + 64 * half, dp);
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 d4 = reinterpret_cast<const float4*>(st_ds)[c4];
        dp[4 * c4 + 0] = x[4 * c4 + 0] * (dp[4 * c4 + 0] - d4.x);
        dp[4 * c4 + 1] = x[4 * c4 + 1] * (dp[4 * c4 + 1] - d4.y);
        dp[4 * c4 + 2] = x[4 * c4 + 2] * (dp[4 * c4 + 2] - d4.z);
        dp[4 * c4 + 3] = x[4 * c4 + 3] * (dp[4 * c4 + 3] - d4.w);
      }
      tmem_st_packed64<BF16>(tDP + 64 * half, dp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::BAR_DS));
    }
    // ---------------------------------------------------------------- epilogue
    // warpgroup 0 writes dK (scaled), warpgroup 1 dV; a key row goes to its
    // physical slot when its page has exactly one reader
    if (failed) {
      if (lane == 0) fail();
    } else {
      bool ok = true;
      if (N > 0) {
        ok = mbar_wait(bar(C::BAR_DONE), 0);
        if (__any_sync(0xffffffffu, !ok)) { ok = false; if (lane == 0) fail(); }
      }
      const int pidx = key / P;
      int page = (pidx < used && in_bounds(pp.status, static_cast<int64_t>(s) * pp.max_pages + pidx,
                                           static_cast<int64_t>(pp.num_seqs) * pp.max_pages))
                     ? __ldg(table + pidx) : -1;
      if (page >= pp.num_pages || (page >= 0 && __ldg(a.offsets + page + 1) - __ldg(a.offsets + page) != 1))
        page = -1;
      // the key row in the cache gradient: [pages, page_size, Hkv, D]
      const int64_t crow = ((static_cast<int64_t>(page < 0 ? 0 : page) * P + key % P) * pp.Hkv + hk) * D;
      if (page >= 0 && !range_in_bounds(pp.status, crow, D, static_cast<int64_t>(pp.num_pages) * P * pp.Hkv * D))
        page = -1;
      void* dst = half == 0 ? a.dk : a.dv;
      if (ok) {
        tc_fence_after();
        const uint32_t src = tmem + lane_off + 256 + (half == 0 ? D : 0);
        const float mul = half == 0 ? a.scale : 1.f;
        uint8_t* rowp = static_cast<uint8_t*>(dst) +
                        ((static_cast<size_t>(page < 0 ? 0 : page) * P + key % P) * pp.Hkv + hk) * D * 2;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          float v[32];
          if (N > 0) {
            uint32_t r[32];
            tmem_ld32(src + 32 * c, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0.f;
          }
          if (page >= 0 && dst) store_row16<BF16, 32>(rowp + c * 64, v, mul);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Key blocks per CTA of the streaming key-major kernel.
constexpr int KPC = 8;

// The key-major kernel for calls whose query side per (sequence, kv head) is
// one tile (one head block and at most 128 (query, head) pairs: a decode step,
// or a short chunk). CTA = (sequence, kv head, run of KPC 128-key blocks):
// the query and dout tile stays resident while the key blocks stream through
// the two-stage ring (K and V of a block in one stage), so the setup, the
// query loads and the row statistics are paid once per run instead of once per
// 128 keys, and the epilogue of a block overlaps the S and dP MMAs of the next.
// Per block: S^T = K Q^T and dP^T = V dO^T (SS), P^T and dS'^T by the
// elementwise warps (packed into S^T's and dP^T's columns), dV = P^T dO and
// dK = dS'^T Q (TS, one query tile: no accumulation across tiles), then the
// elementwise warps store the block's dK and dV rows of single-reader pages
// and compute the next block's P^T. The order makes every TMEM reuse safe: the
// MMA issues the next block's S and dP after dK (the tensor pipe runs in
// order), and the elementwise warps finish reading dK and dV before they
// release the next block's P^T for the dV MMA.
template <int D, bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    paged_dkdv_stream_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                             const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                             const PagedParams pp, const TcArgs a, int chunks) {
  using C = Cfg<D>;
  constexpr int BAR_KVFULL = C::BAR_FULL, BAR_KVEMPTY = C::BAR_EMPTY;  // the ring holds K, V pairs
  constexpr int BAR_ACC = C::BAR_S + 1;                                 // dK, dV of the block complete
  static_assert(C::STAGES >= 2, "two ring stages");
  constexpr int NST = 2;
  // ---- work: key blocks [kb0, kb0 + nb) of sequence s, kv head hk
  const int lin = static_cast<int>(blockIdx.x);
  const int ch = lin % chunks;
  const int rest = lin / chunks;
  const int hk = rest % pp.Hkv, s = rest / pp.Hkv;
  const int L = seq_keys(pp, s);
  int q0, n;
  seq_rows(pp, s, q0, n);
  const int P = pp.page_size;
  const int used = (L + P - 1) / P;
  const int kblocks_used = (used * P + BR - 1) / BR;
  const int kb0 = ch * KPC;
  const int nb = min(KPC, kblocks_used - kb0);
  if (n == 0 || nb <= 0) return;  // uniform
  const int group = pp.Hq / pp.Hkv;  // = the head block: one tile of (query, head) pairs
  const int diag = L - n;
  const bool dflt = pp.positions == nullptr;
  const int32_t* table = pp.block_table + static_cast<size_t>(s) * pp.max_pages;

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(bar(BAR_KVFULL + st), 1);
      mbar_init(bar(BAR_KVEMPTY + st), 1);
    }
    mbar_init(bar(C::BAR_RES), 1);
    mbar_init(bar(C::BAR_S), 1);
    mbar_init(bar(BAR_ACC), 1);
    mbar_init(bar(C::BAR_DP), 1);
    mbar_init(bar(C::BAR_P), 256);
    mbar_init(bar(C::BAR_DS), 256);
    mbar_init(bar(C::BAR_DONE), 1);
    mbar_init_fence();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    if (pp.status) atomicOr(pp.status, STATUS_TIMEOUT);
  };

  if (warp >= 8) {
    setmaxnreg_dec<REG_OTHER>();
    if (warp == WARP_TMA && lane == 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(C::BAR_RES), 2 * C::TILE_BYTES);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_4d(sb + c * C::CHUNK_BYTES, &tm_q, bar(C::BAR_RES), c * C::BOX_D, 0, hk, q0);
        tma_load_4d(sb + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_do, bar(C::BAR_RES), c * C::BOX_D, 0, hk, q0);
      }
      int i = 0;
      for (; i < nb; ++i) {
        const int st = i % NST;
        if (!mbar_wait(bar(BAR_KVEMPTY + st), ((i / NST) & 1) ^ 1)) { fail(); break; }
        const uint32_t dst = sb + C::OFF_RING + st * 2 * C::TILE_BYTES;
        mbar_arrive_expect_tx(bar(BAR_KVFULL + st), 2 * C::TILE_BYTES);
        load_kv_tile<D>(dst, &tm_k, bar(BAR_KVFULL + st), table, pp, (kb0 + i) * BR, hk);
        load_kv_tile<D>(dst + C::TILE_BYTES, &tm_v, bar(BAR_KVFULL + st), table, pp, (kb0 + i) * BR, hk);
      }
      for (int st = 0; st < NST && st < i; ++st) {
        const int fills = (i - st + NST - 1) / NST;
        if (!mbar_wait(bar(BAR_KVFULL + st), (fills - 1) & 1)) fail();
      }
      if (!mbar_wait(bar(C::BAR_RES), 0)) fail();
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_s = make_idesc_f16(BF16, BR, BR, false);
      constexpr uint32_t idesc_o = make_idesc_f16(BF16, BR, D, true);
      constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
      constexpr uint32_t RSTEP16 = (16 * 128) >> 4;
      const uint64_t res_k = smem_desc(sb, 16, C::SBO, C::LAYOUT);                  // Q, dO as K-major B
      const uint64_t res_mn = smem_desc(sb, C::CHUNK_BYTES, C::SBO, C::LAYOUT);     // Q, dO as MN-major B
      const uint64_t ring_k = smem_desc(sb + C::OFF_RING, 16, C::SBO, C::LAYOUT);  // K, V as K-major A
      bool ok = warp_wait(bar(C::BAR_RES), 0);
      tc_fence_after();
      for (int i = 0; i < nb && ok; ++i) {
        const int st = i % NST;
        if (!warp_wait(bar(BAR_KVFULL + st), (i / NST) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kk = ring_k + st * 2 * TILE16;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::KSTEPS_D; ++k)
            umma_ss(tmem + 0, kk + kstep16<D>(k), res_k + kstep16<D>(k), idesc_s, k > 0 ? 1u : 0u);
          umma_commit(bar(C::BAR_S));
#pragma unroll
          for (int k = 0; k < C::KSTEPS_D; ++k)
            umma_ss(tmem + BR, kk + TILE16 + kstep16<D>(k), res_k + TILE16 + kstep16<D>(k), idesc_s,
                    k > 0 ? 1u : 0u);
          umma_commit(bar(C::BAR_DP));
          umma_commit(bar(BAR_KVEMPTY + st));  // K and V of the block are no longer read
        }
        __syncwarp();
        if (!warp_wait(bar(C::BAR_P), i & 1)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::KSTEPS_R; ++k)
            umma_ts(tmem + 256, tmem + tmem_a_kstep(k), res_mn + TILE16 + k * RSTEP16, idesc_o, k > 0 ? 1u : 0u);
        }
        __syncwarp();
        if (!warp_wait(bar(C::BAR_DS), i & 1)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::KSTEPS_R; ++k)
            umma_ts(tmem + 256 + D, tmem + BR + tmem_a_kstep(k), res_mn + k * RSTEP16, idesc_o, k > 0 ? 1u : 0u);
          umma_commit(bar(BAR_ACC));
        }
        __syncwarp();
      }
      if (!ok && lane == 0) fail();
      if (elect_one()) {
        umma_commit(bar(C::BAR_DONE));
      }
      __syncwarp();
      if (!warp_wait(bar(C::BAR_DONE), 0) && lane == 0) fail();
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- elementwise
    setmaxnreg_inc<REG_EW>();
    const int half = warp >> 2;                // pair columns [64 half, +64) of the tile
    const int row = ((warp & 3) << 5) + lane;  // key row of the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_off, tDP = tS + BR;
    const float sc = pp.scale_log2;
    float* st_l2 = reinterpret_cast<float*>(smem + C::OFF_STATS) + warp * C::STATS_PER_WARP;
    float* st_ds = st_l2 + 64;
    int* st_lim = reinterpret_cast<int*>(st_l2 + 128);
    // the tile's column statistics, once: lse2, D and the largest visible key
    // (-1 for a pair with no query or no visible key)
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int pair = 64 * half + 32 * u + lane;
      const int qi = pair / group;
      const int hq = hk * group + (pair - qi * group);
      const size_t ri = static_cast<size_t>(q0 + (qi < n ? qi : 0)) * pp.Hq + hq;
      const bool in = qi < n && in_bounds(pp.status, static_cast<int64_t>(ri),
                                          static_cast<int64_t>(pp.num_queries) * pp.Hq);
      const float l2 = in ? __ldg(a.lse2 + ri) : -INFINITY;
      const float dsm = in ? __ldg(a.dsum + ri) : 0.f;
      int lim = 0x7ffffffe;
      if (pp.causal)
        lim = dflt ? diag + qi
                   : ((in && in_bounds(pp.status, q0 + qi, pp.num_queries))
                          ? min(__ldg(pp.positions + q0 + qi), 0x7ffffffe) : -1);
      const bool live = l2 != -INFINITY;
      st_l2[32 * u + lane] = live ? l2 : 0.f;
      st_ds[32 * u + lane] = live ? dsm : 0.f;
      st_lim[32 * u + lane] = live ? lim : -1;
    }
    __syncwarp();
    void* dst = half == 0 ? a.dk : a.dv;
    const float mul = half == 0 ? a.scale : 1.f;
    bool failed = false;
    for (int i = 0; i < nb && !failed; ++i) {
      const int key = (kb0 + i) * BR + row;
      const int kcmp = key < L ? key : 0x7fffffff;  // keys past the sequence see nothing
      float x[64];
      const bool ok = mbar_wait(bar(C::BAR_S), i & 1);
      if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
      tc_fence_after();
      tmem_ld64<BF16>(tS + 64 * half, x);
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 l4 = reinterpret_cast<const float4*>(st_l2)[c4];
        const int4 m4 = reinterpret_cast<const int4*>(st_lim)[c4];
        x[4 * c4 + 0] = kcmp <= m4.x ? fast_exp2(x[4 * c4 + 0] * sc - l4.x) : 0.f;
        x[4 * c4 + 1] = kcmp <= m4.y ? fast_exp2(x[4 * c4 + 1] * sc - l4.y) : 0.f;
        x[4 * c4 + 2] = kcmp <= m4.z ? fast_exp2(x[4 * c4 + 2] * sc - l4.z) : 0.f;
        x[4 * c4 + 3] = kcmp <= m4.w ? fast_exp2(x[4 * c4 + 3] * sc - l4.w) : 0.f;
      }
      tmem_st_packed64<BF16>(tS + 64 * half, x);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::BAR_P));
      const bool ok2 = mbar_wait(bar(C::BAR_DP), i & 1);
      if (__any_sync(0xffffffffu, !ok2)) { failed = true; break; }
      tc_fence_after();
      float dp[64];
      tmem_ld64<BF16>(tDP + 64 * half, dp);
#pragma unroll
      for (int c4 = 0; c4 < 16; ++c4) {
        const float4 d4 = reinterpret_cast<const float4*>(st_ds)[c4];
        dp[4 * c4 + 0] = x[4 * c4 + 0] * (dp[4 * c4 + 0] - d4.x);
        dp[4 * c4 + 1] = x[4 * c4 + 1] * (dp[4 * c4 + 1] - d4.y);
        dp[4 * c4 + 2] = x[4 * c4 + 2] * (dp[4 * c4 + 2] - d4.z);
        dp[4 * c4 + 3] = x[4 * c4 + 3] * (dp[4 * c4 + 3] - d4.w);
      }
      tmem_st_packed64<BF16>(tDP + 64 * half, dp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::BAR_DS));
      // ---- the block's rows: warpgroup 0 writes dK (scaled), warpgroup 1 dV;
      // a key row goes to its physical slot when its page has exactly one reader
      const int pidx = key / P;
      int page = (pidx < used && in_bounds(pp.status, static_cast<int64_t>(s) * pp.max_pages + pidx,
                                           static_cast<int64_t>(pp.num_seqs) * pp.max_pages))
                     ? __ldg(table + pidx) : -1;
      if (page >= pp.num_pages || (page >= 0 && __ldg(a.offsets + page + 1) - __ldg(a.offsets + page) != 1))
        page = -1;
      const int64_t crow = ((static_cast<int64_t>(page < 0 ? 0 : page) * P + key % P) * pp.Hkv + hk) * D;
      if (page >= 0 && !range_in_bounds(pp.status, crow, D, static_cast<int64_t>(pp.num_pages) * P * pp.Hkv * D))
        page = -1;
      const bool ok3 = mbar_wait(bar(BAR_ACC), i & 1);
      if (__any_sync(0xffffffffu, !ok3)) { failed = true; break; }
      tc_fence_after();
      const uint32_t src = tmem + lane_off + 256 + (half == 0 ? D : 0);
      uint8_t* rowp = static_cast<uint8_t*>(dst) + crow * 2;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(src + 32 * c, r);
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
        if (page >= 0 && dst) store_row16<BF16, 32>(rowp + c * 64, v, mul);
      }
      tc_fence_before();
    }
    if (failed && lane == 0) fail();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// The streaming key-major kernel for a query side of at most NPN (query, head)
// pairs (a decode step with a group of up to 32 heads, or a few queries): S^T
// and dP^T are 128 keys x NPN pairs (MMA N = NPN instead of 128), dV and dK
// contract over NPN pairs (2 K-steps instead of 8), one warpgroup computes P
// and dS' for all NPN pairs of its key rows, and the small resident tiles leave
// room for three K/V stages.
constexpr int NPN = 32;

template <int D>
struct NarrowCfg {
  using C = Cfg<D>;
  static constexpr int QCHUNK = NPN * 128;  // one NPN-row x 64-column box
  static constexpr int QTILE = C::NCHUNK * QCHUNK;
  static constexpr int OFF_RING = (2 * QTILE + 1023) / 1024 * 1024;
  static constexpr int KVSTAGE = 2 * C::TILE_BYTES;
  static constexpr int NST = 3;
  static constexpr int OFF_BAR = OFF_RING + NST * KVSTAGE;
  static constexpr int BAR_FULL = 0, BAR_EMPTY = NST, BAR_RES = 2 * NST, BAR_S = BAR_RES + 1, BAR_DP = BAR_S + 1,
                       BAR_P = BAR_DP + 1, BAR_DS = BAR_P + 1, BAR_ACC = BAR_DS + 1, BAR_DONE = BAR_ACC + 1,
                       NUM_BARS = BAR_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_STATS = (OFF_MISC + 16 + 15) / 16 * 16;
  static constexpr int STATS_PER_WARP = 3 * NPN;  // lse2, D, limit of each pair column
  static constexpr int SMEM_BYTES = OFF_STATS + 4 * STATS_PER_WARP * 4 + 1024;
  static_assert(SMEM_BYTES <= 232448, "narrow streaming kernel shared memory");
};

template <int D, bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    paged_dkdv_narrow_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                             const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                             const PagedParams pp, const TcArgs a, int chunks) {
  using C = Cfg<D>;
  using X = NarrowCfg<D>;
  constexpr int NST = X::NST;
  // ---- work: key blocks [kb0, kb0 + nb) of sequence s, kv head hk
  const int lin = static_cast<int>(blockIdx.x);
  const int ch = lin % chunks;
  const int rest = lin / chunks;
  const int hk = rest % pp.Hkv, s = rest / pp.Hkv;
  const int L = seq_keys(pp, s);
  int q0, n;
  seq_rows(pp, s, q0, n);
  const int P = pp.page_size;
  const int used = (L + P - 1) / P;
  const int kblocks_used = (used * P + BR - 1) / BR;
  const int kb0 = ch * KPC;
  const int nb = min(KPC, kblocks_used - kb0);
  if (n == 0 || nb <= 0) return;  // uniform
  const int group = pp.Hq / pp.Hkv;
  const int diag = L - n;
  const bool dflt = pp.positions == nullptr;
  const int32_t* table = pp.block_table + static_cast<size_t>(s) * pp.max_pages;

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + X::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + X::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < NST; ++st) {
      mbar_init(bar(X::BAR_FULL + st), 1);
      mbar_init(bar(X::BAR_EMPTY + st), 1);
    }
    mbar_init(bar(X::BAR_RES), 1);
    mbar_init(bar(X::BAR_S), 1);
    mbar_init(bar(X::BAR_DP), 1);
    // P: warpgroup 0 has written P^T, warpgroup 1 has read the previous block's dV
    mbar_init(bar(X::BAR_P), 256);
    mbar_init(bar(X::BAR_DS), 128);
    mbar_init(bar(X::BAR_ACC), 1);
    mbar_init(bar(X::BAR_DONE), 1);
    mbar_init_fence();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    if (pp.status) atomicOr(pp.status, STATUS_TIMEOUT);
  };

  if (warp >= 8) {
    setmaxnreg_dec<REG_OTHER>();
    if (warp == WARP_TMA && lane == 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(X::BAR_RES), 2 * X::QTILE);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_4d(sb + c * X::QCHUNK, &tm_q, bar(X::BAR_RES), c * C::BOX_D, 0, hk, q0);
        tma_load_4d(sb + X::QTILE + c * X::QCHUNK, &tm_do, bar(X::BAR_RES), c * C::BOX_D, 0, hk, q0);
      }
      int i = 0;
      for (; i < nb; ++i) {
        const int st = i % NST;
        if (!mbar_wait(bar(X::BAR_EMPTY + st), ((i / NST) & 1) ^ 1)) { fail(); break; }
        const uint32_t dst = sb + X::OFF_RING + st * X::KVSTAGE;
        mbar_arrive_expect_tx(bar(X::BAR_FULL + st), X::KVSTAGE);
        load_kv_tile<D>(dst, &tm_k, bar(X::BAR_FULL + st), table, pp, (kb0 + i) * BR, hk);
        load_kv_tile<D>(dst + C::TILE_BYTES, &tm_v, bar(X::BAR_FULL + st), table, pp, (kb0 + i) * BR, hk);
      }
      for (int st = 0; st < NST && st < i; ++st) {
        const int fills = (i - st + NST - 1) / NST;
        if (!mbar_wait(bar(X::BAR_FULL + st), (fills - 1) & 1)) fail();
      }
      if (!mbar_wait(bar(X::BAR_RES), 0)) fail();
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_s = make_idesc_f16(BF16, BR, NPN, false);
      constexpr uint32_t idesc_o = make_idesc_f16(BF16, BR, D, true);
      constexpr uint32_t QTILE16 = X::QTILE >> 4, QCHUNK16 = X::QCHUNK >> 4;
      constexpr uint32_t KV16 = X::KVSTAGE >> 4, TILE16 = C::TILE_BYTES >> 4;
      constexpr uint32_t RSTEP16 = (16 * 128) >> 4;
      const uint64_t res_k = smem_desc(sb, 16, C::SBO, C::LAYOUT);              // Q, dO as K-major B
      const uint64_t res_mn = smem_desc(sb, X::QCHUNK, C::SBO, C::LAYOUT);      // Q, dO as MN-major B
      const uint64_t ring_k = smem_desc(sb + X::OFF_RING, 16, C::SBO, C::LAYOUT);  // K, V as K-major A
      auto qstep = [](int k) -> uint32_t { return (k / 4) * QCHUNK16 + (k % 4) * 2; };
      bool ok = warp_wait(bar(X::BAR_RES), 0);
      tc_fence_after();
      for (int i = 0; i < nb && ok; ++i) {
        const int st = i % NST;
        if (!warp_wait(bar(X::BAR_FULL + st), (i / NST) & 1)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kk = ring_k + st * KV16;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::KSTEPS_D; ++k)
            umma_ss(tmem + 0, kk + kstep16<D>(k), res_k + qstep(k), idesc_s, k > 0 ? 1u : 0u);
          umma_commit(bar(X::BAR_S));
#pragma unroll
          for (int k = 0; k < C::KSTEPS_D; ++k)
            umma_ss(tmem + BR, kk + TILE16 + kstep16<D>(k), res_k + QTILE16 + qstep(k), idesc_s, k > 0 ? 1u : 0u);
          umma_commit(bar(X::BAR_DP));
          umma_commit(bar(X::BAR_EMPTY + st));  // K and V of the block are no longer read
        }
        __syncwarp();
        if (!warp_wait(bar(X::BAR_P), i & 1)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < NPN / 16; ++k)
            umma_ts(tmem + 256, tmem + k * 8, res_mn + QTILE16 + k * RSTEP16, idesc_o, k > 0 ? 1u : 0u);
        }
        __syncwarp();
        if (!warp_wait(bar(X::BAR_DS), i & 1)) { ok = false; break; }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < NPN / 16; ++k)
            umma_ts(tmem + 256 + D, tmem + BR + k * 8, res_mn + k * RSTEP16, idesc_o, k > 0 ? 1u : 0u);
          umma_commit(bar(X::BAR_ACC));
        }
        __syncwarp();
      }
      if (!ok && lane == 0) fail();
      if (elect_one()) {
        umma_commit(bar(X::BAR_DONE));
      }
      __syncwarp();
      if (!warp_wait(bar(X::BAR_DONE), 0) && lane == 0) fail();
    }
    __syncwarp();
  } else {
    setmaxnreg_inc<REG_EW>();
    const int row = ((warp & 3) << 5) + lane;  // key row of the block = TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const bool ew = warp < 4;                  // warpgroup 0: P, dS' and the dK rows; 1: the dV rows
    const float sc = pp.scale_log2;
    float* st_l2 = reinterpret_cast<float*>(smem + X::OFF_STATS) + (warp & 3) * X::STATS_PER_WARP;
    float* st_ds = st_l2 + NPN;
    int* st_lim = reinterpret_cast<int*>(st_l2 + 2 * NPN);
    if (ew) {
      // pair column `lane`: lse2, D and the largest visible key (-1: no query or no key)
      const int pair = lane;
      const int qi = pair / group;
      const int hq = hk * group + (pair - qi * group);
      const size_t ri = static_cast<size_t>(q0 + (qi < n ? qi : 0)) * pp.Hq + hq;
      const bool in = qi < n && in_bounds(pp.status, static_cast<int64_t>(ri),
                                          static_cast<int64_t>(pp.num_queries) * pp.Hq);
      const float l2 = in ? __ldg(a.lse2 + ri) : -INFINITY;
      const float dsm = in ? __ldg(a.dsum + ri) : 0.f;
      int lim = 0x7ffffffe;
      if (pp.causal)
        lim = dflt ? diag + qi
                   : ((in && in_bounds(pp.status, q0 + qi, pp.num_queries))
                          ? min(__ldg(pp.positions + q0 + qi), 0x7ffffffe) : -1);
      const bool live = l2 != -INFINITY;
      st_l2[lane] = live ? l2 : 0.f;
      st_ds[lane] = live ? dsm : 0.f;
      st_lim[lane] = live ? lim : -1;
      __syncwarp();
    }
    void* dst = ew ? a.dk : a.dv;
    const float mul = ew ? a.scale : 1.f;
    bool failed = false;
    for (int i = 0; i < nb && !failed; ++i) {
      const int key = (kb0 + i) * BR + row;
      // warpgroup 1: the previous block's dV rows are read, the next dV MMA may overwrite them
      if (!ew) mbar_arrive(bar(X::BAR_P));
      if (ew) {
        const int kcmp = key < L ? key : 0x7fffffff;  // keys past the sequence see nothing
        const bool ok = mbar_wait(bar(X::BAR_S), i & 1);
        if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
        tc_fence_after();
        float x[NPN];
        {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off, r);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < NPN; ++c) x[c] = __uint_as_float(r[c]);
        }
#pragma unroll
        for (int c4 = 0; c4 < NPN / 4; ++c4) {
          const float4 l4 = reinterpret_cast<const float4*>(st_l2)[c4];
          const int4 m4 = reinterpret_cast<const int4*>(st_lim)[c4];
          x[4 * c4 + 0] = kcmp <= m4.x ? fast_exp2(x[4 * c4 + 0] * sc - l4.x) : 0.f;
          x[4 * c4 + 1] = kcmp <= m4.y ? fast_exp2(x[4 * c4 + 1] * sc - l4.y) : 0.f;
          x[4 * c4 + 2] = kcmp <= m4.z ? fast_exp2(x[4 * c4 + 2] * sc - l4.z) : 0.f;
          x[4 * c4 + 3] = kcmp <= m4.w ? fast_exp2(x[4 * c4 + 3] * sc - l4.w) : 0.f;
        }
        {
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) pk[c] = pack2<BF16>(x[2 * c], x[2 * c + 1]);
          tmem_st16(tmem + lane_off, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(X::BAR_P));
        const bool ok2 = mbar_wait(bar(X::BAR_DP), i & 1);
        if (__any_sync(0xffffffffu, !ok2)) { failed = true; break; }
        tc_fence_after();
        {
          uint32_t r[32];
          tmem_ld32(tmem + lane_off + BR, r);
          tmem_wait_ld();
          uint32_t pk[16];
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float d0 = x[2 * c] * (__uint_as_float(r[2 * c]) - st_ds[2 * c]);
            const float d1 = x[2 * c + 1] * (__uint_as_float(r[2 * c + 1]) - st_ds[2 * c + 1]);
            pk[c] = pack2<BF16>(d0, d1);
          }
          tmem_st16(tmem + lane_off + BR, pk);
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(X::BAR_DS));
      }
      // ---- the block's rows (dK by warpgroup 0, dV by warpgroup 1); a key row
      // goes to its physical slot when its page has exactly one reader
      const int pidx = key / P;
      int page = (pidx < used && in_bounds(pp.status, static_cast<int64_t>(s) * pp.max_pages + pidx,
                                           static_cast<int64_t>(pp.num_seqs) * pp.max_pages))
                     ? __ldg(table + pidx) : -1;
      if (page >= pp.num_pages || (page >= 0 && __ldg(a.offsets + page + 1) - __ldg(a.offsets + page) != 1))
        page = -1;
      const int64_t crow = ((static_cast<int64_t>(page < 0 ? 0 : page) * P + key % P) * pp.Hkv + hk) * D;
      if (page >= 0 && !range_in_bounds(pp.status, crow, D, static_cast<int64_t>(pp.num_pages) * P * pp.Hkv * D))
        page = -1;
      const bool ok3 = mbar_wait(bar(X::BAR_ACC), i & 1);
      if (__any_sync(0xffffffffu, !ok3)) { failed = true; break; }
      tc_fence_after();
      const uint32_t src = tmem + lane_off + 256 + (ew ? D : 0);
      uint8_t* rowp = static_cast<uint8_t*>(dst) + crow * 2;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t r[32];
        tmem_ld32(src + 32 * c, r);
        tmem_wait_ld();
        float v[32];
#pragma unroll
        for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
        if (page >= 0 && dst) store_row16<BF16, 32>(rowp + c * 64, v, mul);
      }
      tc_fence_before();
    }
    if (failed && lane == 0) fail();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    paged_dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                       const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const PagedParams pp, const TcArgs a, int qtiles, int gp) {
  using C = Cfg<D>;
  using Q = DqCfg<D>;
  // ---- work: 128 (query, head) pairs of head block hh of sequence s
  const int lin = static_cast<int>(blockIdx.x);
  const int t = lin % qtiles;
  const int rest = lin / qtiles;
  const int nhb = pp.Hq / gp;
  const int hh = rest % nhb, s = rest / nhb;
  int q0, n;
  seq_rows(pp, s, q0, n);
  if (t * BR >= n * gp) return;  // uniform
  const int L = seq_keys(pp, s);
  const int group = pp.Hq / pp.Hkv;
  const int hk = hh * gp / group;
  const int diag = L - n;
  const bool dflt = pp.positions == nullptr;
  int hi = L;  // keys past every row's causal limit are not visited (default positions)
  if (pp.causal && dflt) hi = min(hi, max(0, diag + min(n - 1, ((t + 1) * BR - 1) / gp) + 1));
  const int N = hi > 0 ? (hi + BR - 1) / BR : 0;
  const int32_t* table = pp.block_table + static_cast<size_t>(s) * pp.max_pages;

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + Q::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Q::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int st = 0; st < Q::KST; ++st) {
      mbar_init(bar(Q::BAR_KFULL + st), 1);
      mbar_init(bar(Q::BAR_KEMPTY + st), 1);
    }
    for (int st = 0; st < Q::VST; ++st) {
      mbar_init(bar(Q::BAR_VFULL + st), 1);
      mbar_init(bar(Q::BAR_VEMPTY + st), 1);
    }
    mbar_init(bar(Q::BAR_RES), 1);
    mbar_init(bar(Q::BAR_S), 1);
    mbar_init(bar(Q::BAR_S + 1), 1);
    mbar_init(bar(Q::BAR_DP), 1);
    mbar_init(bar(Q::BAR_DS), 256);
    mbar_init(bar(Q::BAR_DONE), 1);
    mbar_init_fence();
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    if (pp.status) atomicOr(pp.status, STATUS_TIMEOUT);
  };

  if (warp >= 8) {
    setmaxnreg_dec<REG_OTHER>();
    if (warp == WARP_TMA && lane == 0 && N > 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      const int qs = q0 + t * (BR / gp);
      mbar_arrive_expect_tx(bar(Q::BAR_RES), 2 * C::TILE_BYTES);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_4d(sb + c * C::CHUNK_BYTES, &tm_q, bar(Q::BAR_RES), c * C::BOX_D, 0, hh, qs);
        tma_load_4d(sb + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_do, bar(Q::BAR_RES), c * C::BOX_D, 0, hh, qs);
      }
      int nk = 0, nv = 0;
      bool ok = true;
      for (int j = 0; j < N && ok; ++j) {
        const int ks = j % Q::KST, vs = j % Q::VST;
        if (!mbar_wait(bar(Q::BAR_KEMPTY + ks), ((j / Q::KST) & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(Q::BAR_KFULL + ks), C::TILE_BYTES);
        load_kv_tile<D>(sb + Q::OFF_K + ks * C::TILE_BYTES, &tm_k, bar(Q::BAR_KFULL + ks), table, pp, j * BR, hk);
        ++nk;
        if (!mbar_wait(bar(Q::BAR_VEMPTY + vs), ((j / Q::VST) & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(Q::BAR_VFULL + vs), C::TILE_BYTES);
        load_kv_tile<D>(sb + Q::OFF_V + vs * C::TILE_BYTES, &tm_v, bar(Q::BAR_VFULL + vs), table, pp, j * BR, hk);
        ++nv;
      }
      if (!ok) fail();
      for (int st = 0; st < Q::KST && st < nk; ++st)
        if (!mbar_wait(bar(Q::BAR_KFULL + st), (((nk - st + Q::KST - 1) / Q::KST) - 1) & 1)) fail();
      for (int st = 0; st < Q::VST && st < nv; ++st)
        if (!mbar_wait(bar(Q::BAR_VFULL + st), (((nv - st + Q::VST - 1) / Q::VST) - 1) & 1)) fail();
      if (!mbar_wait(bar(Q::BAR_RES), 0)) fail();
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer (the dense kernel's)
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_s = make_idesc_f16(BF16, BR, BR, false);
      constexpr uint32_t idesc_o = make_idesc_f16(BF16, BR, D, true);
      constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
      constexpr uint32_t RSTEP16 = (16 * 128) >> 4;
      const uint64_t q_a = smem_desc(sb, 16, C::SBO, C::LAYOUT);
      const uint64_t do_a = smem_desc(sb + C::TILE_BYTES, 16, C::SBO, C::LAYOUT);
      const uint64_t k_b = smem_desc(sb + Q::OFF_K, 16, C::SBO, C::LAYOUT);
      const uint64_t k_mn = smem_desc(sb + Q::OFF_K, C::CHUNK_BYTES, C::SBO, C::LAYOUT);
      const uint64_t v_b = smem_desc(sb + Q::OFF_V, 16, C::SBO, C::LAYOUT);
      bool ok = true;
      auto issue_s = [&](int j) {
        const int ks = j % Q::KST;
        if (!warp_wait(bar(Q::BAR_KFULL + ks), (j / Q::KST) & 1)) return false;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::KSTEPS_D; ++k)
            umma_ss(tmem + BR * (j & 1), q_a + kstep16<D>(k), k_b + ks * TILE16 + kstep16<D>(k), idesc_s,
                    k > 0 ? 1u : 0u);
          umma_commit(bar(Q::BAR_S + (j & 1)));
        }
        __syncwarp();
        return true;
      };
      auto issue_dp = [&](int j) {
        const int vs = j % Q::VST;
        if (!warp_wait(bar(Q::BAR_VFULL + vs), (j / Q::VST) & 1)) return false;
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::KSTEPS_D; ++k)
            umma_ss(tmem + 2 * BR, do_a + kstep16<D>(k), v_b + vs * TILE16 + kstep16<D>(k), idesc_s,
                    k > 0 ? 1u : 0u);
          umma_commit(bar(Q::BAR_DP));
          umma_commit(bar(Q::BAR_VEMPTY + vs));
        }
        __syncwarp();
        return true;
      };
      if (N > 0) {
        if (!warp_wait(bar(Q::BAR_RES), 0)) ok = false;
        tc_fence_after();
        if (ok && !issue_s(0)) ok = false;
        if (ok && !issue_dp(0)) ok = false;
        if (ok && N > 1 && !issue_s(1)) ok = false;
        for (int j = 0; j < N && ok; ++j) {
          if (!warp_wait(bar(Q::BAR_DS), j & 1)) { ok = false; break; }
          tc_fence_after();
          const int ks = j % Q::KST;
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < C::KSTEPS_R; ++k)
              umma_ts(tmem + 3 * BR, tmem + 2 * BR + tmem_a_kstep(k), k_mn + ks * TILE16 + k * RSTEP16, idesc_o,
                      (j > 0 || k > 0) ? 1u : 0u);
            umma_commit(bar(Q::BAR_KEMPTY + ks));
          }
          __syncwarp();
          if (j + 1 < N && !issue_dp(j + 1)) { ok = false; break; }
          if (j + 2 < N && !issue_s(j + 2)) { ok = false; break; }
        }
      }
      if (!ok && lane == 0) fail();
      if (elect_one()) {
        umma_commit(bar(Q::BAR_DONE));
      }
      __syncwarp();
      if (!warp_wait(bar(Q::BAR_DONE), 0) && lane == 0) fail();
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- elementwise
    setmaxnreg_inc<REG_EW>();
    const int half = warp >> 2;                // key columns [64 half, +64)
    const int row = ((warp & 3) << 5) + lane;  // pair row = TMEM lane
    const int pair = t * BR + row;
    const int qi = pair / gp;
    const int hq = hh * gp + (pair - qi * gp);
    const bool row_ok = qi < n;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const size_t ri = static_cast<size_t>(q0 + (row_ok ? qi : 0)) * pp.Hq + hq;
    const int64_t nrows = static_cast<int64_t>(pp.num_queries) * pp.Hq;  // extent for the checked build
    const bool stat_ok = row_ok && in_bounds(pp.status, static_cast<int64_t>(ri), nrows);
    const float l2 = stat_ok ? __ldg(a.lse2 + ri) : -INFINITY;
    const bool live = l2 != -INFINITY;
    const float dsi = live ? __ldg(a.dsum + ri) : 0.f;
    const int pos = row_ok ? (dflt ? diag + qi
                                   : (in_bounds(pp.status, q0 + qi, pp.num_queries) ? __ldg(pp.positions + q0 + qi)
                                                                                    : -1))
                           : -1;
    const int causal_lim = pp.causal ? pos : 0x7fffffff;
    // the smallest visibility limit of this warp's live rows: a 64-key slice at or
    // below it (and inside the sequence) needs no per-element test; a dead row takes
    // lse2 = +inf there, so its p is exactly 0
    const int warp_lim = __reduce_min_sync(0xffffffffu, live ? causal_lim : 0x7fffffff);
    const float l2f = live ? l2 : INFINITY;
    const float sc = pp.scale_log2;
    bool failed = false;
    for (int j = 0; j < N; ++j) {
      float x[64];
      const bool ok = mbar_wait(bar(Q::BAR_S + (j & 1)), (j >> 1) & 1);
      if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
      tc_fence_after();
      tmem_ld64<BF16>(tmem + lane_off + BR * (j & 1) + 64 * half, x);
      const int kc0 = j * BR + 64 * half;
      if (kc0 + 63 < L && kc0 + 63 <= warp_lim) {
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = fast_exp2(x[c] * sc - l2f);
      } else {
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int key = kc0 + c;
          const bool vis = live && key < L && key <= causal_lim;
          x[c] = vis ? fast_exp2(x[c] * sc - l2) : 0.f;
        }
      }
      const bool ok2 = mbar_wait(bar(Q::BAR_DP), j & 1);
      if (__any_sync(0xffffffffu, !ok2)) { failed = true; break; }
      tc_fence_after();
      float dp[64];
      tmem_ld64<BF16>(tmem + lane_off + 2 * BR + 64 * half, dp);
#pragma unroll
      for (int c = 0; c < 64; ++c) dp[c] = x[c] * (dp[c] - dsi);
      tmem_st_packed64<BF16>(tmem + lane_off + 2 * BR + 64 * half, dp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(Q::BAR_DS));
    }
    // ---------------------------------------------------------------- epilogue
    if (failed) {
      if (lane == 0) fail();
    } else {
      bool ok = true;
      if (N > 0) {
        ok = mbar_wait(bar(Q::BAR_DONE), 0);
        if (__any_sync(0xffffffffu, !ok)) { ok = false; if (lane == 0) fail(); }
      }
      if (ok) {
        tc_fence_after();
        uint8_t* rowp = static_cast<uint8_t*>(a.dq) + (ri * D + half * (D / 2)) * 2;
        const bool row_in =
            stat_ok && range_in_bounds(pp.status, static_cast<int64_t>(ri) * D + half * (D / 2), D / 2, nrows * D);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          float v[32];
          if (N > 0) {
            uint32_t r[32];
            tmem_ld32(tmem + lane_off + 3 * BR + half * (D / 2) + 32 * c, r);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(r[e]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0.f;
          }
          if (row_in) store_row16<BF16, 32>(rowp + c * 64, v, a.scale);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

}  // namespace tc

template <int D, bool BF16>
cudaError_t launch_paged_bwd_tc(EncodeTiledFn enc, const PagedParams& pp, const void* q, const void* k,
                                const void* v, const void* dout, const TcArgs& a, cudaStream_t st) {
  using namespace tc;
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  const int group = pp.Hq / pp.Hkv;
  const int gp = BR % group == 0 ? group : 1;
  CUtensorMap tq, tdo, tk, tv;
  {  // q, dout viewed as [queries, Hq/gp, gp, D]; boxes of 128 (query, head) pairs
    const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(gp),
                                static_cast<cuuint64_t>(pp.Hq / gp), static_cast<cuuint64_t>(pp.num_queries)};
    const cuuint64_t gstride[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(gp) * D * 2,
                                   static_cast<cuuint64_t>(pp.Hq) * D * 2};
    const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(gp), 1u, static_cast<cuuint32_t>(BR / gp)};
    for (int i = 0; i < 2; ++i)
      if (enc(i == 0 ? &tq : &tdo, dt, 4, const_cast<void*>(i == 0 ? q : dout), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
  }
  {  // k, v viewed as [pages, page_size, Hkv, D]
    const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(pp.Hkv),
                                static_cast<cuuint64_t>(pp.page_size), static_cast<cuuint64_t>(pp.num_pages)};
    const cuuint64_t gstride[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(pp.Hkv) * D * 2,
                                   static_cast<cuuint64_t>(pp.page_size) * pp.Hkv * D * 2};
    const cuuint32_t box[4] = {64u, 1u, static_cast<cuuint32_t>(pp.page_size < BR ? pp.page_size : BR), 1u};
    for (int i = 0; i < 2; ++i)
      if (enc(i == 0 ? &tk : &tv, dt, 4, const_cast<void*>(i == 0 ? k : v), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
  }
  // q, dout again with boxes of NPN (query, head) pairs, for the narrow kernel
  CUtensorMap tqn, tdon;
  const bool narrow_ok = gp == group && NPN % gp == 0;
  if (narrow_ok) {
    const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(gp),
                                static_cast<cuuint64_t>(pp.Hq / gp), static_cast<cuuint64_t>(pp.num_queries)};
    const cuuint64_t gstride[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(gp) * D * 2,
                                   static_cast<cuuint64_t>(pp.Hq) * D * 2};
    const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(gp), 1u, static_cast<cuuint32_t>(NPN / gp)};
    for (int i = 0; i < 2; ++i)
      if (enc(i == 0 ? &tqn : &tdon, dt, 4, const_cast<void*>(i == 0 ? q : dout), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
  }
  auto kv = paged_dkdv_tc_kernel<D, BF16>;
  auto kvs = paged_dkdv_stream_kernel<D, BF16>;
  auto kvn = paged_dkdv_narrow_kernel<D, BF16>;
  constexpr int smem_kvn = NarrowCfg<D>::SMEM_BYTES;
  auto kq = paged_dq_tc_kernel<D, BF16>;
  constexpr int smem_kv = Cfg<D>::SMEM_BYTES;
  constexpr int smem_q = DqCfg<D>::SMEM_BYTES;
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = pp.device >= 0 && pp.device < 64 ? 1ull << pp.device : 0ull;
  if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kvs, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kvn, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kvn);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  if (a.dk || a.dv) {
    const int64_t kblocks = (static_cast<int64_t>(pp.max_pages) * pp.page_size + BR - 1) / BR;
    // one tile of (query, head) pairs per (sequence, kv head): stream the key blocks
    const bool stream = gp == group && static_cast<int64_t>(pp.max_queries) * gp <= BR;
    const int64_t chunks = (kblocks + KPC - 1) / KPC;
    const int64_t ctas = static_cast<int64_t>(pp.num_seqs) * pp.Hkv * (stream ? chunks : kblocks);
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    // at most NPN pairs: the narrow streaming kernel
    const bool narrow = stream && narrow_ok && static_cast<int64_t>(pp.max_queries) * gp <= NPN;
    if (ctas > 0 && narrow)
      kvn<<<static_cast<unsigned>(ctas), NUM_THREADS, smem_kvn, st>>>(tqn, tdon, tk, tv, pp, a,
                                                                      static_cast<int>(chunks));
    else if (ctas > 0 && stream)
      kvs<<<static_cast<unsigned>(ctas), NUM_THREADS, smem_kv, st>>>(tq, tdo, tk, tv, pp, a,
                                                                     static_cast<int>(chunks));
    else if (ctas > 0)
      kv<<<static_cast<unsigned>(ctas), NUM_THREADS, smem_kv, st>>>(tq, tdo, tk, tv, pp, a,
                                                                    static_cast<int>(kblocks), gp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (a.dq) {
    const int64_t qtiles = (static_cast<int64_t>(pp.max_queries) * gp + BR - 1) / BR;
    const int64_t ctas = static_cast<int64_t>(pp.num_seqs) * (pp.Hq / gp) * qtiles;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (ctas > 0)
      kq<<<static_cast<unsigned>(ctas), NUM_THREADS, smem_q, st>>>(tq, tdo, tk, tv, pp, a,
                                                                   static_cast<int>(qtiles), gp);
  }
  return cudaGetLastError();
}

}  // namespace pbwd
}  // namespace attn
