// attn_paged_tc.cuh - attention over a paged key/value cache with packed
// variable-length queries on the tcgen05 tensor cores (F16/BF16, D in
// {64, 128}): attn_paged_fwd's prefill- and decode-shaped calls.
//
// Source: ruDNN user guide, section 9 (paged attention): physical pages
// K, V [pages, page_size, Hkv, D] read through per-sequence page tables,
// packed queries [queries, Hq, D], GQA, causal mask by absolute position,
// split key history merged from FP32 partial statistics.
//
// The pipeline is the dense forward's (attn_tc.cuh: 384 threads, two query
// tiles of 128 rows per CTA sharing every K/V tile, S and P in tensor memory,
// MMA order S_0 PV_1 S_1 PV_0, lazy rescale); what changes is the addressing:
//  - the rows of a CTA are (query, head) pairs of one sequence and one block
//    of gp query heads that share a kv head (gp = Hq/Hkv when that divides
//    128, else 1), packed as row = query * gp + head-in-block, so every K/V
//    tile serves all the heads of a GQA group; a decode step (one query) is
//    gp rows of a 128-row tile;
//  - a CTA is (sequence, 256 packed rows, head block, key split);
//  - a Q tile of 128 packed rows is one TMA box of a 4-D view
//    [queries, Hq/gp, gp, D] of q (box 64 x gp x 1 x 128/gp);
//  - a K/V tile of 128 keys is gathered page by page through a 4-D view
//    [pages, page_size, Hkv, D] of the cache (box 64 x 1 x min(page_size, 128)
//    x 1): one box per page inside the tile, at the page the table names; a
//    page index outside the cache loads zeros (TMA fills out-of-range boxes);
//  - row i of the CTA sees key j when j < seq_len and, causal, j <= its
//    position (explicit, or the newest-token default);
//  - rows are stored directly (their sequence's rows only) in the input dtype;
//    with num_splits > 1 the CTA covers a contiguous run of the key tiles and
//    stores its unnormalised output and (m, l) for launch_split_merge.
// Requires page_size a multiple of 8 that divides 128 or is a multiple of 128.
#pragma once

#include <atomic>

#include "params.h"
#include "ptx.cuh"
#include "seq_order.cuh"

namespace attn {
namespace pagedtc {

constexpr int BM = 128;
constexpr int BN = 128;
constexpr int NQ = 2;
constexpr int NUM_THREADS = 384;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int TMEM_COLS = 512;
constexpr int REG_SOFTMAX = 200;
constexpr int REG_OTHER = 96;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.0f;

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "paged tensor-core head dims are 64 and 128");
  static constexpr int BOX_D = 64;
  static constexpr int NCHUNK = D / BOX_D;
  static constexpr int CHUNK_BYTES = BN * 128;
  static constexpr int TILE_BYTES = NCHUNK * CHUNK_BYTES;
  static constexpr int STAGES = D == 128 ? 4 : 8;
  static constexpr uint32_t LAYOUT = 2u;  // SW128
  static constexpr int SBO = 1024;
  static constexpr int KSTEPS_QK = D / 16;
  static constexpr int KSTEPS_PV = BN / 16;
  static constexpr int COL_P = 64;
  static constexpr int OFF_KV = NQ * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_KV + STAGES * TILE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 4 * NQ + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = (SMEM_USED + 1024) > 120 * 1024 ? (SMEM_USED + 1024) : 120 * 1024;
  static constexpr int BAR_FULL = 0, BAR_EMPTY = STAGES, BAR_Q = 2 * STAGES, BAR_S = BAR_Q + NQ;
  static constexpr int BAR_P = BAR_S + NQ, BAR_O = BAR_P + NQ, BAR_DONE = BAR_O + NQ;
};

struct PWork {
  int s, hh, hk, sp, q_lo, nq, row0, L, j0;
  int n[NQ], nfull[NQ], nmax;  // n, nmax: key tiles j0 .. j0+n-1 of this CTA's split
};

// blockIdx.x -> (sequence, 256-row block, split, head block; the head block
// fastest, so that the CTAs reading the same K/V tiles run side by side). LPT:
// the sequences longest first, for calls with one row block per sequence
// (decode); prefill keeps the batch order, and a kernel without the ranking
// code at all (its presence alone measured 15% slower on prefill).
// Empty when the row block lies past the sequence's rows.
template <bool LPT>
__device__ __forceinline__ PWork make_pwork(const PagedParams& pp, int qblocks, int gp) {
  PWork w;
  int item = static_cast<int>(blockIdx.x);
  const int nhh = pp.Hq / gp;
  w.hh = item % nhh;
  item /= nhh;
  w.sp = item % pp.num_splits;
  item /= pp.num_splits;
  const int qb = item % qblocks;
  if constexpr (LPT) w.s = seq_by_rank(pp, item / qblocks);  // longest sequences first
  else w.s = item / qblocks;
  w.hk = (w.hh * gp) / (pp.Hq / pp.Hkv);
  w.q_lo = min(max(__ldg(pp.q_offsets + w.s), 0), pp.num_queries);
  const int q_hi = min(max(__ldg(pp.q_offsets + w.s + 1), w.q_lo), pp.num_queries);
  w.nq = q_hi - w.q_lo;
  w.row0 = qb * NQ * BM;
  w.L = min(max(__ldg(pp.seq_lens + w.s), 0), pp.max_pages * pp.page_size);
  const int rows = w.nq * gp;
  int ntot[NQ], nall = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int r0 = w.row0 + t * BM;
    ntot[t] = 0;
    w.nfull[t] = 0;
    if (r0 < rows) {
      const int first_q = r0 / gp, last_q = min(w.nq - 1, (r0 + BM - 1) / gp);
      int hi = w.L, lo = w.L;
      if (pp.causal) {
        if (pp.positions) {
          lo = 0;  // arbitrary positions: every tile is masked element by element
        } else {
          hi = min(hi, w.L - w.nq + last_q + 1);
          lo = min(lo, w.L - w.nq + first_q + 1);
        }
      }
      ntot[t] = hi > 0 ? (hi + BN - 1) / BN : 0;
      w.nfull[t] = lo > 0 ? lo / BN : 0;
    }
    nall = max(nall, ntot[t]);
  }
  w.j0 = static_cast<int>(static_cast<int64_t>(nall) * w.sp / pp.num_splits);
  const int j1 = static_cast<int>(static_cast<int64_t>(nall) * (w.sp + 1) / pp.num_splits);
  w.nmax = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    w.n[t] = max(0, min(ntot[t], j1) - w.j0);
    w.nmax = max(w.nmax, w.n[t]);
  }
  return w;
}

template <int D, bool BF16, bool LPT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    paged_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const PagedParams pp, void* out, float* lse,
                    int qblocks, int gp) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const PWork w = make_pwork<LPT>(pp, qblocks, gp);
  if (w.row0 >= w.nq * gp) return;  // no rows here (CTA-uniform); rows without keys still get NaN
  const bool partial = pp.num_splits > 1;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::BAR_FULL + s), 1);
      mbar_init(bar(C::BAR_EMPTY + s), 1);
    }
    for (int t = 0; t < NQ; ++t) {
      mbar_init(bar(C::BAR_Q + t), 1);
      mbar_init(bar(C::BAR_S + t), 1);
      mbar_init(bar(C::BAR_P + t), BM);
      mbar_init(bar(C::BAR_O + t), 1);
    }
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
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      for (int t = 0; t < NQ; ++t) {
        if (w.n[t] == 0) continue;
        mbar_arrive_expect_tx(bar(C::BAR_Q + t), C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_4d(sb + t * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_q, bar(C::BAR_Q + t), c * C::BOX_D, 0,
                      w.hh, w.q_lo + (w.row0 + t * BM) / gp);
      }
      const int32_t* table = pp.block_table + static_cast<size_t>(w.s) * pp.max_pages;
      const int box_rows = pp.page_size < BN ? pp.page_size : BN;
      const int boxes = BN / box_rows;
      int it = 0;
      bool ok = true;
      for (int jj = 0; jj < w.nmax && ok; ++jj) {
        const int j = w.j0 + jj;  // key tile
        for (int kv = 0; kv < 2; ++kv, ++it) {
          const int st = it % C::STAGES;
          if (!mbar_wait(bar(C::BAR_EMPTY + st), ((it / C::STAGES) & 1) ^ 1)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(C::BAR_FULL + st), C::TILE_BYTES);
          const CUtensorMap* m = kv == 0 ? &tm_k : &tm_v;
          for (int i = 0; i < boxes; ++i) {
            const int key = j * BN + i * box_rows;
            const int pidx = key / pp.page_size;
            const int page = pidx < pp.max_pages ? __ldg(table + pidx) : -1;  // -1: zero-filled box
            // checked build: the box lands inside its chunk of the ring slot (a
            // skipped copy leaves the slot's barrier to time out)
            if (!range_in_bounds(pp.status, i * box_rows, box_rows, BN)) continue;
            for (int c = 0; c < C::NCHUNK; ++c)
              tma_load_4d(sb + C::OFF_KV + st * C::TILE_BYTES + c * C::CHUNK_BYTES + i * box_rows * 128, m,
                          bar(C::BAR_FULL + st), c * C::BOX_D, w.hk, key % pp.page_size, page);
          }
        }
      }
      if (!ok) fail();
      for (int st = 0; st < C::STAGES && st < it; ++st) {
        const int fills = (it - st + C::STAGES - 1) / C::STAGES;
        if (!mbar_wait(bar(C::BAR_FULL + st), (fills - 1) & 1)) fail();
      }
      for (int t = 0; t < NQ; ++t)
        if (w.n[t] > 0 && !mbar_wait(bar(C::BAR_Q + t), 0)) fail();
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_qk = make_idesc_f16(BF16, BM, BN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, BM, D, true);
      constexpr int ST = C::STAGES;
      const int n0 = w.n[0], n1 = w.n[1], nmax = w.nmax;
      bool ok = true;
      for (int t = 0; t < NQ && ok; ++t)
        if ((t ? n1 : n0) > 0 && !warp_wait(bar(C::BAR_Q + t), 0)) ok = false;
      const uint64_t dq0 = smem_desc(sb, 16, C::SBO, C::LAYOUT);
      const uint64_t dk0 = smem_desc(sb + C::OFF_KV, 16, C::SBO, C::LAYOUT);
      const uint64_t dv0 = smem_desc(sb + C::OFF_KV, C::CHUNK_BYTES, C::SBO, C::LAYOUT);
      constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
      constexpr uint32_t CHUNK16 = C::CHUNK_BYTES >> 4;
      constexpr uint32_t VSTEP16 = (16 * 128) >> 4;
      auto kstep = [](int k) -> uint32_t { return (k / 4) * CHUNK16 + (k % 4) * 2; };
      auto wait_full = [&](int idx) { return warp_wait(bar(C::BAR_FULL + idx % ST), (idx / ST) & 1); };
      auto issue_s = [&](int t, int j) {
        const uint64_t a = dq0 + t * TILE16;
        const uint64_t b = dk0 + ((2 * j) % ST) * TILE16;
        if (elect_one()) {
#pragma unroll
          for (int k = 0; k < C::KSTEPS_QK; ++k)
            umma_ss(tmem + t * BN, a + kstep(k), b + kstep(k), idesc_qk, k > 0 ? 1u : 0u);
          umma_commit(bar(C::BAR_S + t));
        }
        __syncwarp();
      };
      auto issue_pv = [&](int t, int j) {
        const uint64_t b = dv0 + ((2 * j + 1) % ST) * TILE16;
        const uint32_t d = tmem + 256 + t * D;
        const uint32_t a = tmem + t * BN + C::COL_P;
        if (elect_one()) {
          umma_ts(d, a, b, idesc_pv, j > 0 ? 1u : 0u);
#pragma unroll
          for (int k = 1; k < C::KSTEPS_PV; ++k) umma_ts(d, a + k * 8, b + k * VSTEP16, idesc_pv, 1u);
          if (j == (t ? n1 : n0) - 1) umma_commit(bar(C::BAR_O + t));
        }
        __syncwarp();
      };
      // no abort-flag polling here: every wait below is bounded
      for (int j = 0; j <= nmax && ok; ++j) {
        if (j < nmax) {
          if (!wait_full(2 * j)) { ok = false; break; }
          tc_fence_after();
          if (j < n0) issue_s(0, j);
        }
        if (j >= 1 && j - 1 < n1) {
          if (j - 1 >= n0 && !wait_full(2 * (j - 1) + 1)) { ok = false; break; }
          if (!warp_wait(bar(C::BAR_P + 1), (j - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          issue_pv(1, j - 1);
        }
        if (j >= 1) {
          if (elect_one()) umma_commit(bar(C::BAR_EMPTY + (2 * (j - 1) + 1) % ST));
          __syncwarp();
        }
        if (j < nmax) {
          if (j < n1) issue_s(1, j);
          if (elect_one()) umma_commit(bar(C::BAR_EMPTY + (2 * j) % ST));
          __syncwarp();
          if (j < n0) {
            if (!wait_full(2 * j + 1) || !warp_wait(bar(C::BAR_P + 0), j & 1)) { ok = false; break; }
            tc_fence_after();
            issue_pv(0, j);
          }
        }
      }
      if (!ok && lane == 0) fail();
      if (elect_one()) umma_commit(bar(C::BAR_DONE));
      __syncwarp();
      if (!warp_wait(bar(C::BAR_DONE), 0) && lane == 0) fail();
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    setmaxnreg_inc<REG_SOFTMAX>();
    const int t = warp >> 2;
    const int row = ((warp & 3) << 5) + lane;
    const int pr = w.row0 + t * BM + row;  // packed row: query * gp + head in block
    const int tq = pr / gp;                // query within the sequence
    const bool row_ok = tq < w.nq;
    const int head = w.hh * gp + (pr - tq * gp);
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_off + t * BN;
    const uint32_t tP = tS + C::COL_P;
    const uint32_t tO = tmem + lane_off + 256 + t * D;
    const int n_t = t ? w.n[1] : w.n[0];
    const int nfull_t = t ? w.nfull[1] : w.nfull[0];
    const float sc = pp.scale_log2;
    const int pos = !row_ok ? -1
                            : (pp.positions ? (in_bounds(pp.status, w.q_lo + tq, pp.num_queries)
                                                   ? __ldg(pp.positions + w.q_lo + tq) : -1)
                                            : w.L - w.nq + tq);
    const int causal_lim = pp.causal ? pos : 0x7fffffff;
    const int key_lim = w.L;
    float m_run = -INFINITY, l_run = 0.f;
    bool failed = false;
    for (int j = 0; j < n_t; ++j) {
      const bool ok = mbar_wait(bar(C::BAR_S + t), j & 1);
      if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
      tc_fence_after();
      float s[128];
      {
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, sr[c]);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 128; ++i) s[i] = __uint_as_float(sr[i >> 5][i & 31]);
      }
      const int key0 = (w.j0 + j) * BN;
      if (w.j0 + j >= nfull_t) {
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          const int key = key0 + i;
          if (key >= key_lim || key > causal_lim) s[i] = -INFINITY;
        }
      }
      float c0 = fmax3(s[0], s[1], s[2]), c1 = fmax3(s[3], s[4], s[5]);
      float c2 = fmax3(s[6], s[7], s[8]), c3 = fmax3(s[9], s[10], s[11]);
#pragma unroll
      for (int i = 12; i < 124; i += 8) {
        c0 = fmax3(c0, s[i], s[i + 1]);
        c1 = fmax3(c1, s[i + 2], s[i + 3]);
        c2 = fmax3(c2, s[i + 4], s[i + 5]);
        c3 = fmax3(c3, s[i + 6], s[i + 7]);
      }
      c0 = fmax3(c0, s[124], s[125]);
      c1 = fmax3(c1, s[126], s[127]);
      const float m_tile = fmax3(c0, c1, fmaxf(c2, c3)) * sc;
      const bool need = m_tile > m_run + RESCALE_LOG2;
      float alpha = 1.f;
      if (need) {
        alpha = fast_exp2(m_run - m_tile);
        m_run = m_tile;
        l_run *= alpha;
      }
      const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
      float2 sum_a = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
#pragma unroll
      for (int hh = 0; hh < 2; ++hh) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int i = 64 * hh + 2 * c;
          const float2 xa = ffma2(make_float2(s[i], s[i + 1]), make_float2(sc, sc), make_float2(neg_m, neg_m));
          const float2 xb = ffma2(make_float2(s[i + 2], s[i + 3]), make_float2(sc, sc), make_float2(neg_m, neg_m));
          const float2 pa = make_float2(fast_exp2(xa.x), fast_exp2(xa.y));
          const float2 pb = make_float2(fast_exp2(xb.x), fast_exp2(xb.y));
          sum_a = fadd2(sum_a, pa);
          sum_b = fadd2(sum_b, pb);
          pk[c] = pack2<BF16>(pa.x, pa.y);
          pk[c + 1] = pack2<BF16>(pb.x, pb.y);
        }
        tmem_st32(tP + 32 * hh, pk);
      }
      l_run += (sum_a.x + sum_a.y) + (sum_b.x + sum_b.y);
      if (j > 0 && __any_sync(0xffffffffu, need)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 x = fmul2(make_float2(__uint_as_float(o[i]), __uint_as_float(o[i + 1])),
                                   make_float2(alpha, alpha));
            o[i] = __float_as_uint(x.x);
            o[i + 1] = __float_as_uint(x.y);
          }
          tmem_st32(tO + 32 * c, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::BAR_P + t));
    }
    // ---------------------------------------------------------------- epilogue
    const bool have = n_t > 0;
    if (!failed && have) {
      const bool ok = mbar_wait(bar(C::BAR_O + t), 0);
      if (__any_sync(0xffffffffu, !ok)) failed = true;
    }
    if (failed) {
      if (lane == 0) fail();
    } else if (w.row0 + t * BM < w.nq * gp) {
      tc_fence_after();
      const bool live = have && l_run > 0.f;
      const size_t orow = static_cast<size_t>(w.q_lo + (row_ok ? tq : 0)) * pp.Hq + (row_ok ? head : 0);
      const int64_t nrows = static_cast<int64_t>(pp.num_queries) * pp.Hq;  // extents for the checked build
      if (partial) {  // unnormalised output of this key run and its (m, l)
        const size_t prow = static_cast<size_t>(w.sp) * pp.num_queries * pp.Hq + orow;
        float4* dst = reinterpret_cast<float4*>(pp.ws_o + prow * D);
        const bool row_in = row_ok && in_bounds(pp.status, static_cast<int64_t>(prow), pp.num_splits * nrows);
        if (have) {
#pragma unroll
          for (int c = 0; c < D / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
            if (row_in) {
#pragma unroll
              for (int u = 0; u < 8; ++u)
                dst[c * 8 + u] = make_float4(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1]),
                                             __uint_as_float(o[4 * u + 2]), __uint_as_float(o[4 * u + 3]));
            }
          }
        }
        if (row_in) pp.ws_ml[prow] = make_float2(live ? m_run : -INFINITY, live ? l_run : 0.f);
      } else {
        const float inv = live ? 1.f / l_run : __int_as_float(0x7fc00000);
        uint8_t* dst = static_cast<uint8_t*>(out) + orow * D * 2;
        const bool row_in = row_ok && in_bounds(pp.status, static_cast<int64_t>(orow), nrows);
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          if (have) {
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = 0u;
          }
          if (row_in) {
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float2 x = fmul2(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])),
                                     make_float2(inv, inv));
              pk[i] = pack2<BF16>(x.x, x.y);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              reinterpret_cast<uint4*>(dst + c * 64)[u] =
                  make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
        if (row_in && lse) lse[orow] = live ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
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


template <int D, bool BF16>
cudaError_t launch_paged_tc(EncodeTiledFn enc, const PagedParams& pp, const void* q, const void* k, const void* v,
                            void* out, float* lse, cudaStream_t stream) {
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint32_t estride[4] = {1, 1, 1, 1};
  CUtensorMap tq, tk, tv;
  // gp query heads share each CTA's rows: the kv group when it divides 128
  const int group = pp.Hq / pp.Hkv;
  const int gp = BM % group == 0 ? group : 1;
  {  // q viewed as [queries, Hq/gp, gp, D]
    const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(gp),
                                static_cast<cuuint64_t>(pp.Hq / gp), static_cast<cuuint64_t>(pp.num_queries)};
    const cuuint64_t gstride[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(gp) * D * 2,
                                   static_cast<cuuint64_t>(pp.Hq) * D * 2};
    const cuuint32_t box[4] = {64u, static_cast<cuuint32_t>(gp), 1u, static_cast<cuuint32_t>(BM / gp)};
    if (enc(&tq, dt, 4, const_cast<void*>(q), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  {  // k, v viewed as [pages, page_size, Hkv, D]
    const cuuint64_t gdim[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(pp.Hkv),
                                static_cast<cuuint64_t>(pp.page_size), static_cast<cuuint64_t>(pp.num_pages)};
    const cuuint64_t gstride[3] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(pp.Hkv) * D * 2,
                                   static_cast<cuuint64_t>(pp.page_size) * pp.Hkv * D * 2};
    const cuuint32_t box[4] = {64u, 1u, static_cast<cuuint32_t>(pp.page_size < BN ? pp.page_size : BN), 1u};
    for (int i = 0; i < 2; ++i)
      if (enc(i == 0 ? &tk : &tv, dt, 4, const_cast<void*>(i == 0 ? k : v), gdim, gstride, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorInvalidValue;
  }
  const int64_t qblocks = (static_cast<int64_t>(pp.max_queries) * gp + NQ * BM - 1) / (NQ * BM);
  const bool lpt = qblocks == 1;
  auto kern = lpt ? paged_tc_kernel<D, BF16, true> : paged_tc_kernel<D, BF16, false>;
  constexpr int smem = Cfg<D>::SMEM_BYTES;
  static std::atomic<unsigned long long> configured[2] = {{0}, {0}};
  const unsigned long long bit = pp.device >= 0 && pp.device < 64 ? 1ull << pp.device : 0ull;
  if (!bit || !(configured[lpt].load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[lpt].fetch_or(bit, std::memory_order_acq_rel);
  }
  const int64_t ctas = static_cast<int64_t>(pp.num_seqs) * qblocks * (pp.Hq / gp) * pp.num_splits;
  if (ctas == 0) return cudaSuccess;
  if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(ctas), NUM_THREADS, smem, stream>>>(tq, tk, tv, pp, out, lse,
                                                                   static_cast<int>(qblocks), gp);
  return cudaGetLastError();
}

}  // namespace pagedtc
}  // namespace attn
