// attn_mla_tc.cuh - multi-head latent attention (absorbed projections) over a
// paged latent cache on the tcgen05 tensor cores (F16/BF16, R in {256, 512},
// Pd in {0, 64}).
//
// Source: ruDNN user guide, section 9 (MLA): q [queries, H, R] with the key
// projection absorbed, a positional query qp [queries, H, Pd], one latent row
// c_j [R] and one positional key kp_j [Pd] per token shared by every head;
//   s_j = scale (q . c_j + qp . kp_j),   out = sum_j softmax_j(s) c_j,
// paging, packed queries, positions and the causal mask as for paged attention.
//
// Shape of the work: the rows of a sequence are its (query, head) pairs,
// row = query * H + head, so a decode step with H = 128 heads is one 128-row
// tile. A key row [c_j | kp_j] is R + Pd wide (576 for R = 512, Pd = 64) and
// the output R wide. Each 128-row block is run by R/128 CTAs, one per
// 128-column slice of the output: every CTA computes the full scores
// S = [q | qp] [c | kp]^T of its rows (the same MMAs, so the same P, in each
// CTA) and its own slice of P . c. With only 128 output columns the whole
// query fits in tensor memory next to the scores, so shared memory holds
// nothing but a ring of 64-key tiles, and the score MMAs are 64 keys wide: a
// 128 x N x 16 MMA costs about the same for N = 16..64, so the width halves
// the score cost per key against 32-key tiles.
//
// Tensor memory (512 columns): the query chunks (64 dims = 32 packed 16-bit
// columns each, at most nine), S (64 fp32 columns), P (32 packed columns), the
// 128-column output slice. The S MMA reads its A operand (the query) from
// tensor memory and the key chunk from the ring; P . V reads P from tensor
// memory and this slice's two latent chunks of the same ring tile as V (the
// values are the latent rows, so no separate value load exists).
//
// Warps: 0-3 softmax (one row per thread: loads the 64 scores, frees S for the
// next tile's MMA, masks, online softmax, waits for the previous P . V before
// writing P and, rarely, rescaling O), 4 TMA producer (the query once through
// ring stages 1.., then key tiles gathered page by page through 3-D views
// [pages, page_size, R] and [pages, page_size, Pd] of the caches; an invalid
// page id loads zeros), 5 MMA issuer, order S_0 S_1 PV_0 S_2 PV_1 ...
//
// Key-range splits: the CTA's key tiles are cut into num_splits balanced runs;
// with more than one run each CTA writes its unnormalised partial output and
// (m, l) and launch_split_merge combines them (the split of attn_fwd_split).
// Requires page_size a multiple of 8 that divides 64 or is a multiple of 64.
#pragma once

#include <atomic>

#include "params.h"
#include "ptx.cuh"
#include "seq_order.cuh"

namespace attn {
namespace mlatc {

constexpr int BM = 128;           // (query, head) rows per CTA
constexpr int BN = 64;            // keys per tile
constexpr int OC = 128;           // output columns per CTA
constexpr int NUM_THREADS = 192;  // warps 0-3 softmax, 4 TMA, 5 MMA
constexpr int WARP_TMA = 4;
constexpr int WARP_MMA = 5;
constexpr int TMEM_COLS = 512;
constexpr int COL_Q = 0;          // query chunks: columns [0, 32 NCH), NCH <= 9
constexpr int COL_S = 288;        // S: 64 fp32 columns
constexpr int COL_P = 352;        // P: 64 keys as 32 packed columns
constexpr int COL_O = 384;        // output slice: columns [384, 512)
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.0f;

template <int R, int PD>
struct Cfg {
  static_assert(R == 256 || R == 512, "tensor-core MLA latent ranks are 256 and 512");
  static_assert(PD == 0 || PD == 64, "tensor-core MLA positional widths are 0 and 64");
  static constexpr int NH = R / OC;          // CTAs per row block (output slices)
  static constexpr int NCH = (R + PD) / 64;  // 64-wide chunks of a key row
  static constexpr int NCH_LAT = R / 64;     // ... of which latent
  static constexpr int QCH_BYTES = BM * 128;
  static constexpr int KCH_BYTES = BN * 128;
  static constexpr int STAGE_BYTES = NCH * KCH_BYTES;
  static constexpr int RESERVE = 1024 + 256;  // base alignment + barriers
  static constexpr int ST_FIT = (SMEM_LIMIT - RESERVE) / STAGE_BYTES;
  static constexpr int STAGES = ST_FIT > 6 ? 6 : ST_FIT;
  // the query passes through ring stages 1.. on its way to tensor memory
  static constexpr int OFF_STAGING = STAGE_BYTES;
  static_assert(STAGES >= 3, "ring too small");
  static_assert(OFF_STAGING + NCH * QCH_BYTES <= STAGES * STAGE_BYTES, "staging overflows the ring");
  static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr int BAR_FULL = 0, BAR_EMPTY = STAGES, BAR_QST = 2 * STAGES, BAR_QT = BAR_QST + 1,
                       BAR_S = BAR_QST + 2, BAR_SFREE = BAR_S + 1, BAR_P = BAR_S + 2, BAR_PV = BAR_S + 3,
                       BAR_DONE = BAR_S + 4, NUM_BARS = BAR_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");
  static_assert(COL_Q + NCH * 32 <= COL_S && COL_O + OC <= TMEM_COLS, "tensor memory");
};

struct MWork {
  int s, sp, h, q_lo, nq, row0, L, t0, n, nfull;
};

// blockIdx.x -> (sequence, 128-row block, split, output slice); the slice is
// fastest so that the CTAs sharing key tiles run side by side. LPT: the
// sequences longest first, for calls with one row block per sequence (decode).
template <int NH, bool LPT>
__device__ __forceinline__ MWork make_mwork(const PagedParams& pp, int rblocks) {
  MWork w;
  int item = static_cast<int>(blockIdx.x);
  w.h = item % NH;
  item /= NH;
  w.sp = item % pp.num_splits;
  item /= pp.num_splits;
  const int rb = item % rblocks;
  if constexpr (LPT) w.s = seq_by_rank(pp, item / rblocks);  // longest sequences first
  else w.s = item / rblocks;
  const int H = pp.Hq;
  w.q_lo = min(max(__ldg(pp.q_offsets + w.s), 0), pp.num_queries);
  const int q_hi = min(max(__ldg(pp.q_offsets + w.s + 1), w.q_lo), pp.num_queries);
  w.nq = q_hi - w.q_lo;
  w.row0 = rb * BM;
  w.L = min(max(__ldg(pp.seq_lens + w.s), 0), pp.max_pages * pp.page_size);
  w.t0 = w.n = w.nfull = 0;
  if (w.row0 >= w.nq * H) return w;
  int hi = w.L, lo = w.L;
  if (pp.causal) {
    if (pp.positions) {
      lo = 0;  // arbitrary positions: every tile is masked element by element
    } else {
      const int first_q = w.row0 / H, last_q = min(w.nq - 1, (w.row0 + BM - 1) / H);
      hi = min(hi, w.L - w.nq + last_q + 1);
      lo = min(lo, w.L - w.nq + first_q + 1);
    }
  }
  const int T = hi > 0 ? (hi + BN - 1) / BN : 0;
  w.nfull = lo > 0 ? lo / BN : 0;
  w.t0 = static_cast<int>(static_cast<int64_t>(T) * w.sp / pp.num_splits);
  w.n = static_cast<int>(static_cast<int64_t>(T) * (w.sp + 1) / pp.num_splits) - w.t0;
  return w;
}

template <int R, int PD, bool BF16, bool LPT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                  const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_kp,
                  const PagedParams pp, void* out, float* lse, int rblocks) {
  using C = Cfg<R, PD>;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = pp.Hq;
  const MWork w = make_mwork<C::NH, LPT>(pp, rblocks);
  const int rows_seq = w.nq * H;
  if (w.row0 >= rows_seq) return;  // no rows here (CTA-uniform)
  const int64_t rows_total = static_cast<int64_t>(pp.num_queries) * H;
  const int64_t grow0 = static_cast<int64_t>(w.q_lo) * H + w.row0;  // first global row of the CTA
  const bool partial = pp.num_splits > 1;

  if (w.n == 0) {  // no key tile in this run (CTA-uniform): the rows see no key here
    if (warp < 4) {
      const int r = warp * 32 + lane;
      const int64_t grow = grow0 + r;
      if (w.row0 + r < rows_seq && in_bounds(pp.status, grow, rows_total)) {
        if (partial) {
          if (w.h == 0) pp.ws_ml[w.sp * rows_total + grow] = make_float2(-INFINITY, 0.f);
        } else {
          const uint16_t nan16 = BF16 ? 0x7fc0u : 0x7e00u;
          const uint32_t nn = static_cast<uint32_t>(nan16) * 0x10001u;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + (grow * R + w.h * OC) * 2);
#pragma unroll 4
          for (int u = 0; u < OC / 8; ++u) dst[u] = make_uint4(nn, nn, nn, nn);
          if (lse && w.h == 0) lse[grow] = -INFINITY;
        }
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::BAR_FULL + s), 1);
      mbar_init(bar(C::BAR_EMPTY + s), 1);
    }
    mbar_init(bar(C::BAR_QST), 1);
    mbar_init(bar(C::BAR_QT), BM);
    mbar_init(bar(C::BAR_S), 1);
    mbar_init(bar(C::BAR_SFREE), BM);
    mbar_init(bar(C::BAR_P), BM);
    mbar_init(bar(C::BAR_PV), 1);
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
  const int n = w.n;

  if (warp == WARP_TMA) {
    if (lane == 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_lat);
      if constexpr (PD > 0) {
        tma_prefetch_desc(&tm_qp);
        tma_prefetch_desc(&tm_kp);
      }
      const int gy = static_cast<int>(grow0);
      mbar_arrive_expect_tx(bar(C::BAR_QST), C::NCH * C::QCH_BYTES);
      for (int c = 0; c < C::NCH; ++c) {
        const uint32_t dst = sb + C::OFF_STAGING + c * C::QCH_BYTES;
        if (c < C::NCH_LAT) tma_load_2d(dst, &tm_q, bar(C::BAR_QST), c * 64, gy);
        else tma_load_2d(dst, &tm_qp, bar(C::BAR_QST), (c - C::NCH_LAT) * 64, gy);
      }
      const int32_t* table = pp.block_table + static_cast<size_t>(w.s) * pp.max_pages;
      const int P = pp.page_size;
      const int box_rows = P < BN ? P : BN;
      const int boxes = BN / box_rows;
      bool ok = true;
      int issued = 0;
      for (int i = 0; i < n && ok; ++i, ++issued) {
        const int st = i % C::STAGES;
        // stages 1.. hold the staged query until it is in tensor memory
        if (i == 1 && !mbar_wait(bar(C::BAR_QT), 0)) { ok = false; break; }
        if (!mbar_wait(bar(C::BAR_EMPTY + st), ((i / C::STAGES) & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(C::BAR_FULL + st), C::STAGE_BYTES);
        const uint32_t base = sb + st * C::STAGE_BYTES;
        for (int b = 0; b < boxes; ++b) {
          const int key = (w.t0 + i) * BN + b * box_rows;
          const int pidx = key / P;
          const int page = pidx < pp.max_pages ? __ldg(table + pidx) : -1;  // -1: zero-filled box
          const int y = key - pidx * P;
          // checked build: the box lands inside its chunk of the ring stage (a
          // skipped copy leaves the stage's barrier to time out)
          if (!range_in_bounds(pp.status, b * box_rows, box_rows, BN)) continue;
          for (int c = 0; c < C::NCH; ++c) {
            const uint32_t dst = base + c * C::KCH_BYTES + b * box_rows * 128;
            if (c < C::NCH_LAT) tma_load_3d(dst, &tm_lat, bar(C::BAR_FULL + st), c * 64, y, page);
            else tma_load_3d(dst, &tm_kp, bar(C::BAR_FULL + st), (c - C::NCH_LAT) * 64, y, page);
          }
        }
      }
      if (!ok) fail();
      // the CTA must not retire with copies in flight
      for (int st = 0; st < C::STAGES && st < issued; ++st) {
        const int fills = (issued - st + C::STAGES - 1) / C::STAGES;
        if (!mbar_wait(bar(C::BAR_FULL + st), (fills - 1) & 1)) fail();
      }
      if (!mbar_wait(bar(C::BAR_QST), 0)) fail();
    }
    __syncwarp();
  } else if (warp == WARP_MMA) {
    if (lane == 0) {
      // ------------------------------------------------------------ MMA issuer
      constexpr uint32_t idesc_s = make_idesc_f16(BF16, BM, BN, false);
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, BM, OC, true);
      constexpr int ST = C::STAGES;
      constexpr uint32_t STAGE16 = C::STAGE_BYTES >> 4;
      constexpr uint32_t KCH16 = C::KCH_BYTES >> 4;
      constexpr uint32_t VSTEP16 = (16 * 128) >> 4;
      bool ok = mbar_wait(bar(C::BAR_QT), 0);
      tc_fence_after();
      const uint64_t dk = smem_desc(sb, 16, 1024, 2u);
      const uint64_t dv = smem_desc(sb + w.h * (OC / 64) * C::KCH_BYTES, C::KCH_BYTES, 1024, 2u);
      for (int i = 0; i <= n && ok; ++i) {
        if (i < n) {
          const int st = i % ST;
          if (!mbar_wait(bar(C::BAR_FULL + st), (i / ST) & 1)) { ok = false; break; }
          // S is single-buffered: the softmax must have read S(i-1)
          if (i > 0 && !mbar_wait(bar(C::BAR_SFREE), (i - 1) & 1)) { ok = false; break; }
          tc_fence_after();
          const uint64_t b0 = dk + st * STAGE16;
#pragma unroll
          for (int c = 0; c < C::NCH; ++c) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ts(tmem + COL_S, tmem + COL_Q + c * 32 + kk * 8, b0 + c * KCH16 + kk * 2, idesc_s,
                      (c | kk) ? 1u : 0u);
          }
          umma_commit(bar(C::BAR_S));
        }
        if (i >= 1) {
          const int j = i - 1;
          if (!mbar_wait(bar(C::BAR_P), j & 1)) { ok = false; break; }
          tc_fence_after();
          const uint64_t b0 = dv + (j % ST) * STAGE16;
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_ts(tmem + COL_O, tmem + COL_P + kk * 8, b0 + kk * VSTEP16, idesc_pv, (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(C::BAR_PV));
          umma_commit(bar(C::BAR_EMPTY + j % ST));
        }
      }
      if (!ok) fail();
      umma_commit(bar(C::BAR_DONE));
      if (!mbar_wait(bar(C::BAR_DONE), 0)) fail();
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- softmax
    const int r = warp * 32 + lane;  // row within the CTA = tensor-memory lane
    const bool row_ok = w.row0 + r < rows_seq;
    const int64_t grow = grow0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tQ = tmem + lane_off + COL_Q;
    const uint32_t tS = tmem + lane_off + COL_S;
    const uint32_t tP = tmem + lane_off + COL_P;
    const uint32_t tO = tmem + lane_off + COL_O;
    const int tq = (w.row0 + r) / H;
    const int pos = !row_ok ? -1
                            : (pp.positions ? (in_bounds(pp.status, w.q_lo + tq, pp.num_queries)
                                                   ? __ldg(pp.positions + w.q_lo + tq) : -1)
                                            : w.L - w.nq + tq);
    const int causal_lim = pp.causal ? pos : 0x7fffffff;
    const int key_lim = w.L;
    const float sc = pp.scale_log2;
    bool failed = false;
    // the query: staged shared memory (128-byte swizzled rows) -> tensor memory
    {
      const bool ok = mbar_wait(bar(C::BAR_QST), 0);
      if (__any_sync(0xffffffffu, !ok)) failed = true;
      if (!failed) {
        const uint8_t* row = smem + C::OFF_STAGING + r * 128;
#pragma unroll 1
        for (int c = 0; c < C::NCH; ++c) {
          uint32_t wd[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const uint4 v = *reinterpret_cast<const uint4*>(row + c * C::QCH_BYTES + ((u ^ (r & 7)) << 4));
            wd[4 * u] = v.x;
            wd[4 * u + 1] = v.y;
            wd[4 * u + 2] = v.z;
            wd[4 * u + 3] = v.w;
          }
          tmem_st32(tQ + c * 32, wd);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::BAR_QT));
    }
    float m_run = -INFINITY, l_run = 0.f;
    for (int i = 0; i < n && !failed; ++i) {
      const bool ok = mbar_wait(bar(C::BAR_S), i & 1);
      if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
      tc_fence_after();
      float s[BN];
      {
        uint32_t sr[2][32];
        tmem_ld32(tS, sr[0]);
        tmem_ld32(tS + 32, sr[1]);
        tmem_wait_ld();
#pragma unroll
        for (int k = 0; k < BN; ++k) s[k] = __uint_as_float(sr[k >> 5][k & 31]);
      }
      tc_fence_before();
      mbar_arrive(bar(C::BAR_SFREE));  // the next tile's scores may overwrite S
      const int tile = w.t0 + i;
      if (tile >= w.nfull) {
        const int key0 = tile * BN;
#pragma unroll
        for (int k = 0; k < BN; ++k) {
          const int key = key0 + k;
          if (key >= key_lim || key > causal_lim) s[k] = -INFINITY;
        }
      }
      float c0 = fmax3(s[0], s[1], s[2]), c1 = fmax3(s[3], s[4], s[5]);
#pragma unroll
      for (int k = 6; k < 62; k += 4) {
        c0 = fmax3(c0, s[k], s[k + 1]);
        c1 = fmax3(c1, s[k + 2], s[k + 3]);
      }
      const float m_tile = fmax3(c0, c1, fmaxf(s[62], s[63])) * sc;
      const bool need = m_tile > m_run + RESCALE_LOG2;
      float alpha = 1.f;
      if (need) {
        alpha = fast_exp2(m_run - m_tile);
        m_run = m_tile;
        l_run *= alpha;
      }
      const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
      float2 sum_a = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
      uint32_t pk[32];
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const float2 xa = ffma2(make_float2(s[2 * k], s[2 * k + 1]), make_float2(sc, sc), make_float2(neg_m, neg_m));
        const float2 xb =
            ffma2(make_float2(s[2 * k + 2], s[2 * k + 3]), make_float2(sc, sc), make_float2(neg_m, neg_m));
        const float2 pa = make_float2(fast_exp2(xa.x), fast_exp2(xa.y));
        const float2 pb = make_float2(fast_exp2(xb.x), fast_exp2(xb.y));
        sum_a = fadd2(sum_a, pa);
        sum_b = fadd2(sum_b, pb);
        pk[k] = pack2<BF16>(pa.x, pa.y);
        pk[k + 1] = pack2<BF16>(pb.x, pb.y);
      }
      l_run += (sum_a.x + sum_a.y) + (sum_b.x + sum_b.y);
      // P is single-buffered and O is read by P . V: wait for the previous one
      if (i > 0) {
        const bool pv = mbar_wait(bar(C::BAR_PV), (i - 1) & 1);
        if (__any_sync(0xffffffffu, !pv)) { failed = true; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need)) {  // O holds earlier tiles relative to the old maximum
#pragma unroll 1
          for (int c = 0; c < OC / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; k += 2) {
              const float2 x = fmul2(make_float2(__uint_as_float(o[k]), __uint_as_float(o[k + 1])),
                                     make_float2(alpha, alpha));
              o[k] = __float_as_uint(x.x);
              o[k + 1] = __float_as_uint(x.y);
            }
            tmem_st32(tO + 32 * c, o);
          }
        }
      }
      tmem_st32(tP, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::BAR_P));
    }
    // ---------------------------------------------------------------- epilogue
    if (!failed) {
      const bool ok = mbar_wait(bar(C::BAR_DONE), 0);
      if (__any_sync(0xffffffffu, !ok)) failed = true;
    }
    if (failed) {
      if (lane == 0) fail();
    } else {
      tc_fence_after();
      const bool live = l_run > 0.f;
      const bool row_in = row_ok && in_bounds(pp.status, grow, rows_total);  // checked build
      if (partial) {
        float4* dst = reinterpret_cast<float4*>(pp.ws_o + (w.sp * rows_total + grow) * R + w.h * OC);
#pragma unroll 1
        for (int c = 0; c < OC / 32; ++c) {
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
        if (row_in && w.h == 0)
          pp.ws_ml[w.sp * rows_total + grow] = make_float2(live ? m_run : -INFINITY, live ? l_run : 0.f);
      } else {
        const float inv = live ? 1.f / l_run : __int_as_float(0x7fc00000);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + (grow * R + w.h * OC) * 2);
#pragma unroll 1
        for (int c = 0; c < OC / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_wait_ld();
          if (row_in) {
            uint32_t pkd[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
              const float2 x = fmul2(make_float2(__uint_as_float(o[2 * k]), __uint_as_float(o[2 * k + 1])),
                                     make_float2(inv, inv));
              pkd[k] = pack2<BF16>(x.x, x.y);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[c * 4 + u] = make_uint4(pkd[4 * u], pkd[4 * u + 1], pkd[4 * u + 2], pkd[4 * u + 3]);
          }
        }
        if (row_in && lse && w.h == 0) lse[grow] = live ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
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

template <int R, int PD, bool BF16>
cudaError_t launch_mla_tc(EncodeTiledFn enc, const PagedParams& pp, const void* q, const void* qp, const void* lat,
                          const void* kp, void* out, float* lse, cudaStream_t stream) {
  using C = Cfg<R, PD>;
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint32_t estride[3] = {1, 1, 1};
  const cuuint64_t rows = static_cast<cuuint64_t>(pp.num_queries) * pp.Hq;
  CUtensorMap tq, tqp, tlat, tkp;
  auto enc2 = [&](CUtensorMap* m, const void* base, int width) {  // [rows, width], box 64 x 128
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(width), rows};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(width) * 2};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(BM)};
    return enc(m, dt, 2, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  auto enc3 = [&](CUtensorMap* m, const void* base, int width) {  // [pages, page_size, width]
    const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(pp.page_size),
                                static_cast<cuuint64_t>(pp.num_pages)};
    const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(width) * 2,
                                   static_cast<cuuint64_t>(pp.page_size) * width * 2};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(pp.page_size < BN ? pp.page_size : BN), 1u};
    return enc(m, dt, 3, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  if (enc2(&tq, q, R) != CUDA_SUCCESS || enc3(&tlat, lat, R) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  if constexpr (PD > 0) {
    if (enc2(&tqp, qp, PD) != CUDA_SUCCESS || enc3(&tkp, kp, PD) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  } else {
    tqp = tq;  // unused
    tkp = tlat;
  }
  const int64_t rblocks = (static_cast<int64_t>(pp.max_queries) * pp.Hq + BM - 1) / BM;
  const bool lpt = rblocks == 1;
  auto kern = lpt ? mla_tc_kernel<R, PD, BF16, true> : mla_tc_kernel<R, PD, BF16, false>;
  constexpr int smem = C::SMEM_BYTES;
  static std::atomic<unsigned long long> configured[2] = {{0}, {0}};
  const unsigned long long bit = pp.device >= 0 && pp.device < 64 ? 1ull << pp.device : 0ull;
  if (!bit || !(configured[lpt].load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[lpt].fetch_or(bit, std::memory_order_acq_rel);
  }
  const int64_t ctas = static_cast<int64_t>(pp.num_seqs) * rblocks * pp.num_splits * C::NH;
  if (ctas == 0) return cudaSuccess;
  if (ctas > 0x7fffffffLL || rblocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(ctas), NUM_THREADS, smem, stream>>>(tq, tqp, tlat, tkp, pp, out, lse,
                                                                   static_cast<int>(rblocks));
  return cudaGetLastError();
}

}  // namespace mlatc
}  // namespace attn
