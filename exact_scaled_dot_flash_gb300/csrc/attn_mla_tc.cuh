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
// block. A key row [c_j | kp_j] is R + Pd wide (576 for R = 512, Pd = 64) and
// the output R wide; 128 x R fp32 does not fit in tensor memory next to the
// query and the scores, so a cluster of NH = R/128 CTAs runs each row block,
// CTA h accumulating output columns [128 h, 128 h + 128).
//
// The scores are computed once per row block. The block's 64-key tiles are
// dealt round-robin to the cluster: the CTA that owns tile t (t mod NH = h)
// issues its 36 score MMAs (the query, resident in tensor memory, times the
// tile's nine 64-wide key chunks streamed through a ring), runs the softmax,
// writes the 16-bit P tile and every row's (reference maximum, row sum) into
// P slot t mod 8 of its shared memory and copies both into the same slot of
// every other CTA of the cluster (cp.async.bulk shared::cta -> shared::cluster,
// completing on the receiver's mbarrier). Every CTA multiplies every P tile by
// its own two latent chunks of the tile (P from shared memory, the chunks from
// a second ring). A CTA therefore issues 36 / NH score MMAs and 4 output MMAs
// per tile, where computing the scores in every CTA would take 36 + 4.
//
// One reference maximum per row for the whole cluster. P of a tile is
// exp2(s' - m) for the reference m its owner chose; the output accumulator of
// every CTA is relative to that CTA's current reference m_O. Before the first
// P, the CTAs exchange the row maxima of their first tiles through distributed
// shared memory and all start from their maximum (a cluster barrier orders
// the exchange). An owner then keeps m = m_O unless the tile's maximum exceeds
// it by more than 8 (log2 units; then m = that maximum), so that in the common
// case every tile arrives with the receiver's own reference. A receiver
// reconciles each tile row by row: equal references add the tile's row sum; a
// larger one rescales the row of the accumulator (after the previous P . V)
// and the row sum and adopts it; a smaller one scales the row of P in its own
// slot down (for its own tile only after every peer has received the copy) and
// adds the scaled sum. Numerically this is the online softmax with lazy
// rescaling; which reference a tile used only changes rounding.
//
// Tensor memory (512 columns): the query chunks (64 dims = 32 packed 16-bit
// columns each, at most nine), S (64 fp32 columns), the 128-column output slice.
// Shared memory: 8 P slots (16 KB), 8 (m, l) vectors (1 KB), 2 value stages
// (this CTA's two latent chunks of a tile, 16 KB), a 6-slot ring of score
// chunks (8 KB), the first tiles' row maxima of every CTA. The query passes
// through the P slots and value stages on its way to tensor memory. (Fewer P
// slots for a deeper score ring measured slower: a slot is reused only once
// every CTA has multiplied its tile.)
//
// Warps: 0-3 softmax (one row per thread; each own tile's scores, then the
// reconciliation of every tile up to it, in tile order), 4 TMA (the query, then
// the score chunks of this CTA's tiles), 6 TMA (this CTA's two value chunks of
// every tile), 5 score-MMA issuer (the next own tile's 36 MMAs, chunk by chunk,
// once the softmax has read the previous S), 7 P . V issuer (every tile in order
// as its P arrives). Every issuing warp runs its loop as a whole and issues
// from one elected lane (from a lane-0-only region the copies and MMAs issued
// 5-7% slower). A tcgen05.mma took ~70 cycles of its issuing thread and a
// commit ~45 there: one issuer for both streams spent ~4000 cycles per 4 tiles
// issuing and made the next own score tile wait behind the P . V of the peers'
// tiles (one thread in order: a third slower; one thread polling both streams:
// 25 % slower than two threads). The producers read each tile's page ids one tile ahead: a table
// read in front of every copy put a global-load latency on each chunk. Key
// tiles are gathered page by page through 3-D views [pages, page_size, R] and
// [pages, page_size, Pd] of the caches; an invalid page id loads zeros. Every
// wait is bounded; a cluster barrier after the barrier setup, one for the
// exchange of first-tile maxima and one before exit keep the CTAs resident
// while a peer may still write to them.
//
// Key-range splits: the block's key tiles are cut into num_splits balanced
// runs (one cluster each); with more than one run each CTA writes its
// unnormalised partial output and (m, l) and launch_split_merge combines them.
// Requires page_size a multiple of 8 that divides 64 or is a multiple of 64.
#pragma once

#include <atomic>

#include "params.h"
#include "ptx.cuh"
#include "seq_order.cuh"

namespace attn {
namespace mlatc {

constexpr int BM = 128;           // (query, head) rows per cluster
constexpr int BN = 64;            // keys per tile
constexpr int OC = 128;           // output columns per CTA
constexpr int NUM_THREADS = 256;  // warps 0-3 softmax, 4 TMA (query, scores), 5 score MMA, 6 TMA (values), 7 P.V MMA
constexpr int WARP_KEY = 4;
constexpr int WARP_MMA = 5;
constexpr int WARP_VAL = 6;
constexpr int WARP_PV = 7;
constexpr int TMEM_COLS = 512;
constexpr int COL_Q = 0;          // query chunks: columns [0, 32 NCH), NCH <= 9
constexpr int COL_S = 288;        // S: 64 fp32 columns
constexpr int COL_O = 384;        // output slice: columns [384, 512)
constexpr int NPS = 8;            // P slots (a multiple of NH: slot t mod 8 has one writer)
constexpr int NVS = 2;            // value stages
constexpr int NSR = 6;            // score-chunk ring slots
constexpr int BAR_SOFTMAX = 1;    // named barrier of the 128 softmax threads
constexpr int SMEM_LIMIT = 227 * 1024;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.0f;

template <int R, int PD>
struct Cfg {
  static_assert(R == 256 || R == 512, "tensor-core MLA latent ranks are 256 and 512");
  static_assert(PD == 0 || PD == 64, "tensor-core MLA positional widths are 0 and 64");
  static constexpr int NH = R / OC;          // CTAs per cluster (output slices)
  static constexpr int NCH = (R + PD) / 64;  // 64-wide chunks of a key row
  static constexpr int NCH_LAT = R / 64;     // ... of which latent
  static constexpr int QCH_BYTES = BM * 128;
  static constexpr int KCH_BYTES = BN * 128;
  static constexpr int P_BYTES = BM * BN * 2;
  static constexpr int ML_BYTES = BM * 8;
  static constexpr int V_BYTES = (OC / 64) * KCH_BYTES;
  static constexpr int OFF_P = 0;
  static constexpr int OFF_V = OFF_P + NPS * P_BYTES;
  static constexpr int OFF_SR = OFF_V + NVS * V_BYTES;
  static constexpr int OFF_ML = OFF_SR + NSR * KCH_BYTES;
  static constexpr int OFF_M0 = OFF_ML + NPS * ML_BYTES;
  static constexpr int OFF_BAR = OFF_M0 + NH * BM * 4;
  // the staged query may cover the P slots and the value stages, not the score ring
  static_assert(NCH * QCH_BYTES <= OFF_SR, "query staging overlaps the score ring");
  static_assert(NPS % NH == 0, "a P slot has one writer");
  enum : int {
    BAR_QST = 0,
    BAR_QT,
    BAR_S,
    BAR_SFREE,
    BAR_DONE,
    BAR_SR_FULL,
    BAR_SR_EMPTY = BAR_SR_FULL + NSR,
    BAR_V_FULL = BAR_SR_EMPTY + NSR,
    BAR_P_ARR = BAR_V_FULL + NVS,      // a peer's P tile and (m, l) have landed in the slot
    BAR_P_READY = BAR_P_ARR + NPS,      // the slot's tile is reconciled: P . V may read it
    BAR_PV_DONE = BAR_P_READY + NPS,    // this CTA's P . V of the slot's tile is complete
    BAR_SLOT_FREE = BAR_PV_DONE + NPS,  // every CTA's P . V of the slot's tile is complete
    BAR_RECV = BAR_SLOT_FREE + NPS,     // every peer has received this CTA's tile in the slot
    NUM_BARS = BAR_RECV + NPS
  };
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static_assert(SMEM_BYTES + 4 * (kMaxRanked + 1) <= SMEM_LIMIT, "shared memory");
  static_assert(COL_Q + NCH * 32 <= COL_S && COL_S + BN <= COL_O && COL_O + OC <= TMEM_COLS, "tensor memory");
};

struct MWork {
  int s, sp, q_lo, nq, row0, L, t0, n, nfull;
};

// cluster -> (sequence, 128-row block, split). LPT: the sequences longest
// first, for calls with one row block per sequence (decode).
template <int NH, bool LPT>
__device__ __forceinline__ MWork make_mwork(const PagedParams& pp, int rblocks) {
  MWork w;
  int item = static_cast<int>(blockIdx.x) / NH;
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
__global__ void __cluster_dims__(R / OC, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                  const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_kp,
                  const PagedParams pp, void* out, float* lse, int rblocks) {
  using C = Cfg<R, PD>;
  constexpr int NH = C::NH;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = pp.Hq;
  const int h = static_cast<int>(cluster_rank());  // output slice
  const MWork w = make_mwork<NH, LPT>(pp, rblocks);
  const int rows_seq = w.nq * H;
  // every CTA of the cluster has the same work: they take the same exits,
  // before any traffic between them
  if (w.row0 >= rows_seq) return;
  const int64_t rows_total = static_cast<int64_t>(pp.num_queries) * H;
  const int64_t grow0 = static_cast<int64_t>(w.q_lo) * H + w.row0;  // first global row of the block
  const bool partial = pp.num_splits > 1;

  if (w.n == 0) {  // no key tile in this run: the rows see no key here
    if (warp < 4) {
      const int r = warp * 32 + lane;
      const int64_t grow = grow0 + r;
      if (w.row0 + r < rows_seq && in_bounds(pp.status, grow, rows_total)) {
        if (partial) {
          if (h == 0) pp.ws_ml[w.sp * rows_total + grow] = make_float2(-INFINITY, 0.f);
        } else {
          const uint16_t nan16 = BF16 ? 0x7fc0u : 0x7e00u;
          const uint32_t nn = static_cast<uint32_t>(nan16) * 0x10001u;
          uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + (grow * R + h * OC) * 2);
#pragma unroll 4
          for (int u = 0; u < OC / 8; ++u) dst[u] = make_uint4(nn, nn, nn, nn);
          if (lse && h == 0) lse[grow] = -INFINITY;
        }
      }
    }
    return;
  }

  if (threadIdx.x == 0) {
    mbar_init(bar(C::BAR_QST), 1);
    mbar_init(bar(C::BAR_QT), BM);
    mbar_init(bar(C::BAR_S), 1);
    mbar_init(bar(C::BAR_SFREE), BM);
    mbar_init(bar(C::BAR_DONE), 2);  // both MMA issuers
    for (int i = 0; i < NSR; ++i) {
      mbar_init(bar(C::BAR_SR_FULL + i), 1);
      mbar_init(bar(C::BAR_SR_EMPTY + i), 1);
    }
    for (int i = 0; i < NVS; ++i) {
      mbar_init(bar(C::BAR_V_FULL + i), 1);
    }
    for (int i = 0; i < NPS; ++i) {
      mbar_init(bar(C::BAR_P_ARR + i), 1);  // the local expect_tx arrival + the peer's bytes
      mbar_init(bar(C::BAR_P_READY + i), BM);
      mbar_init(bar(C::BAR_PV_DONE + i), 1);
      mbar_init(bar(C::BAR_SLOT_FREE + i), NH);  // one commit from every CTA of the cluster
      mbar_init(bar(C::BAR_RECV + i), NH - 1);   // one arrival from every peer
    }
    mbar_init_fence();
    // the first delivery into every slot a peer writes
    for (int i = 0; i < NPS; ++i)
      if (i % NH != h) mbar_arrive_expect_tx(bar(C::BAR_P_ARR + i), C::P_BYTES + C::ML_BYTES);
  }
  if (warp == WARP_MMA) {
    tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_arrive();  // every CTA's barriers exist before any remote access
  cluster_wait();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  auto fail = [&]() {
    if (pp.status) atomicOr(pp.status, STATUS_TIMEOUT);
  };
  const int n = w.n;
  const int32_t* table = pp.block_table + static_cast<size_t>(w.s) * pp.max_pages;
  const int P = pp.page_size;
  const int box_rows = P < BN ? P : BN;
  const int boxes = BN / box_rows;

  if (warp >= 4) {
    cluster_arrive();  // the exchange of first-tile maxima: nothing to send from these warps
    if (warp == WARP_KEY) {
      // ------------------------------------------------ TMA: query, own score chunks
      // (the whole warp waits; one elected lane issues the copies)
      const int gy = static_cast<int>(grow0);
      if (elect_one()) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_lat);
        if constexpr (PD > 0) {
          tma_prefetch_desc(&tm_qp);
          tma_prefetch_desc(&tm_kp);
        }
        mbar_arrive_expect_tx(bar(C::BAR_QST), C::NCH * C::QCH_BYTES);
        for (int c = 0; c < C::NCH; ++c) {
          const uint32_t dst = sb + c * C::QCH_BYTES;
          if (c < C::NCH_LAT) tma_load_2d(dst, &tm_q, bar(C::BAR_QST), c * 64, gy);
          else tma_load_2d(dst, &tm_qp, bar(C::BAR_QST), (c - C::NCH_LAT) * 64, gy);
        }
      }
      __syncwarp();
      bool ok = true;
      int cnt = 0;
      // page ids of the own tile being loaded (cur) and of the next one (nxt),
      // read one own tile ahead so that no table read stalls a load; -1 (past
      // the table) loads zeros
      int cur[8], nxt[8];
      auto read_pages = [&](int d, int (&dst)[8]) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          dst[b] = -1;
          if (b < boxes && d < n) {
            const int pidx = ((w.t0 + d) * BN + b * box_rows) / P;
            if (pidx < pp.max_pages) dst[b] = __ldg(table + pidx);
          }
        }
      };
      read_pages(h, nxt);
      for (int d = h; d < n && ok; d += NH) {
#pragma unroll
        for (int b = 0; b < 8; ++b) cur[b] = nxt[b];
        read_pages(d + NH, nxt);
        for (int c = 0; c < C::NCH; ++c, ++cnt) {
          const int slot = cnt % NSR;
          if (!warp_wait(bar(C::BAR_SR_EMPTY + slot), ((cnt / NSR) & 1) ^ 1)) {
            ok = false;
            break;
          }
          if (elect_one()) {
            mbar_arrive_expect_tx(bar(C::BAR_SR_FULL + slot), C::KCH_BYTES);
            const uint32_t base = sb + C::OFF_SR + slot * C::KCH_BYTES;
#pragma unroll
            for (int b = 0; b < 8; ++b) {
              if (b >= boxes) break;
              const int key = (w.t0 + d) * BN + b * box_rows;
              const int y = key - (key / P) * P;
              // checked build: the box lands inside its ring slot (a skipped copy
              // leaves the slot's barrier to time out)
              if (!range_in_bounds(pp.status, b * box_rows, box_rows, BN)) continue;
              const uint32_t dst = base + b * box_rows * 128;
              if (c < C::NCH_LAT) tma_load_3d(dst, &tm_lat, bar(C::BAR_SR_FULL + slot), c * 64, y, cur[b]);
              else tma_load_3d(dst, &tm_kp, bar(C::BAR_SR_FULL + slot), (c - C::NCH_LAT) * 64, y, cur[b]);
            }
          }
          __syncwarp();
        }
      }
      if (!ok && lane == 0) fail();
      // the CTA must not retire with copies in flight
      for (int slot = 0; slot < NSR && slot < cnt; ++slot) {
        const int fills = (cnt - slot + NSR - 1) / NSR;
        if (!warp_wait(bar(C::BAR_SR_FULL + slot), (fills - 1) & 1) && lane == 0) fail();
      }
      if (!warp_wait(bar(C::BAR_QST), 0) && lane == 0) fail();
    } else if (warp == WARP_VAL) {
      // ------------------------------------------------ TMA: own value chunks of every tile
      // page ids of tiles i (cur), i + 1 and i + 2: read two tiles ahead
      int cur[8], nx1[8], nx2[8];
      auto read_pages = [&](int i, int (&dst)[8]) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          dst[b] = -1;
          if (b < boxes && i < n) {
            const int pidx = ((w.t0 + i) * BN + b * box_rows) / P;
            if (pidx < pp.max_pages) dst[b] = __ldg(table + pidx);
          }
        }
      };
      read_pages(0, nx1);
      read_pages(1, nx2);
      bool ok = warp_wait(bar(C::BAR_QT), 0);  // the staged query covers the value stages
      int issued = 0;
      for (int i = 0; i < n && ok; ++i, ++issued) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          cur[b] = nx1[b];
          nx1[b] = nx2[b];
        }
        read_pages(i + 2, nx2);
        const int st = i % NVS;
        // the stage's previous tile, i - NVS, has been multiplied (this CTA's P . V;
        // its phase is the (i - NVS) / NPS-th of that slot's barrier, and the one
        // before completed when this producer refilled the stage for i - NVS)
        if (i >= NVS && !warp_wait(bar(C::BAR_PV_DONE + (i - NVS) % NPS), ((i - NVS) / NPS) & 1)) {
          ok = false;
          break;
        }
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(C::BAR_V_FULL + st), C::V_BYTES);
          const uint32_t base = sb + C::OFF_V + st * C::V_BYTES;
#pragma unroll
          for (int b = 0; b < 8; ++b) {
            if (b >= boxes) break;
            const int key = (w.t0 + i) * BN + b * box_rows;
            const int y = key - (key / P) * P;
            if (!range_in_bounds(pp.status, b * box_rows, box_rows, BN)) continue;
#pragma unroll
            for (int c2 = 0; c2 < OC / 64; ++c2)
              tma_load_3d(base + c2 * C::KCH_BYTES + b * box_rows * 128, &tm_lat, bar(C::BAR_V_FULL + st),
                          (h * (OC / 64) + c2) * 64, y, cur[b]);
          }
        }
        __syncwarp();
      }
      if (!ok && lane == 0) fail();
      for (int st = 0; st < NVS && st < issued; ++st) {
        const int fills = (issued - st + NVS - 1) / NVS;
        if (!warp_wait(bar(C::BAR_V_FULL + st), (fills - 1) & 1) && lane == 0) fail();
      }
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ score MMA issuer
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_s = make_idesc_f16(BF16, BM, BN, false);
      constexpr uint32_t KCH16 = C::KCH_BYTES >> 4;
      const uint64_t d_sr = smem_desc(sb + C::OFF_SR, 16, 1024, 2u);
      // score MMAs of the own tiles, chunk by chunk (once the softmax has read
      // the previous own S); P . V is issued by another warp (WARP_PV)
      bool ok = warp_wait(bar(C::BAR_QT), 0);
      tc_fence_after();
      int cnt = 0;
      for (int d = h, k = 0; d < n && ok; d += NH, ++k) {
        if (k > 0 && !warp_wait(bar(C::BAR_SFREE), (k - 1) & 1)) { ok = false; break; }
        for (int c = 0; c < C::NCH; ++c, ++cnt) {
          const int slot = cnt % NSR;
          if (!warp_wait(bar(C::BAR_SR_FULL + slot), (cnt / NSR) & 1)) { ok = false; break; }
          tc_fence_after();
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ts(tmem + COL_S, tmem + COL_Q + c * 32 + kk * 8, d_sr + slot * KCH16 + kk * 2, idesc_s,
                      (c | kk) ? 1u : 0u);
            umma_commit(bar(C::BAR_SR_EMPTY + slot));
          }
          __syncwarp();
        }
        if (elect_one()) {
          if (ok) umma_commit(bar(C::BAR_S));
        }
        __syncwarp();
      }
      if (!ok && lane == 0) fail();
      if (elect_one()) {
        umma_commit(bar(C::BAR_DONE));
      }
      __syncwarp();
      if (!warp_wait(bar(C::BAR_DONE), 0) && lane == 0) fail();
    } else if (warp == WARP_PV) {
      // ------------------------------------------------------------ P . V issuer
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_pv = make_idesc_f16(BF16, BM, OC, true);
      constexpr uint32_t P16 = C::P_BYTES >> 4;
      constexpr uint32_t V16 = C::V_BYTES >> 4;
      constexpr uint32_t VSTEP16 = (16 * 128) >> 4;  // 16 keys of an MN-major value chunk
      const uint64_t d_p = smem_desc(sb + C::OFF_P, 16, 1024, 2u);
      const uint64_t d_v = smem_desc(sb + C::OFF_V, C::KCH_BYTES, 1024, 2u);
      constexpr uint16_t all = static_cast<uint16_t>((1u << NH) - 1u);
      bool ok = true;
      for (int j = 0; j < n && ok; ++j) {
        const int slot = j % NPS, st = j % NVS;
        if (!warp_wait(bar(C::BAR_P_READY + slot), (j / NPS) & 1) ||
            !warp_wait(bar(C::BAR_V_FULL + st), (j / NVS) & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (elect_one()) {
#pragma unroll
          for (int kk = 0; kk < BN / 16; ++kk)
            umma_ss(tmem + COL_O, d_p + slot * P16 + kk * 2, d_v + st * V16 + kk * VSTEP16, idesc_pv,
                    (j > 0 || kk > 0) ? 1u : 0u);
          umma_commit(bar(C::BAR_PV_DONE + slot));
          umma_commit_mc(bar(C::BAR_SLOT_FREE + slot), all);
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
    cluster_wait();
  } else {
    // -------------------------------------------------------------- softmax
    const int r = warp * 32 + lane;  // row within the block = tensor-memory lane
    const bool row_ok = w.row0 + r < rows_seq;
    const int64_t grow = grow0 + r;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tQ = tmem + lane_off + COL_Q;
    const uint32_t tS = tmem + lane_off + COL_S;
    const uint32_t tO = tmem + lane_off + COL_O;
    const int tq = (w.row0 + r) / H;
    const int pos = !row_ok ? -1
                            : (pp.positions ? (in_bounds(pp.status, w.q_lo + tq, pp.num_queries)
                                                   ? __ldg(pp.positions + w.q_lo + tq) : -1)
                                            : w.L - w.nq + tq);
    const int causal_lim = pp.causal ? pos : 0x7fffffff;
    const int key_lim = w.L;
    const float sc = pp.scale_log2;
    float2* ml = reinterpret_cast<float2*>(smem + C::OFF_ML);
    bool failed = false;
    // the query: staged shared memory (128-byte swizzled rows) -> tensor memory
    {
      const bool ok = mbar_wait(bar(C::BAR_QST), 0);
      if (__any_sync(0xffffffffu, !ok)) failed = true;
      if (!failed) {
        const uint8_t* row = smem + r * 128;
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
    float s[BN];
    float tmax = -INFINITY;
    // scores of own tile d (the k-th): load, free S for the next own tile, mask; max
    auto load_scores = [&](int d, int k) {
      if (!failed) {
        const bool ok = mbar_wait(bar(C::BAR_S), k & 1);
        if (__any_sync(0xffffffffu, !ok)) failed = true;
      }
      if (!failed) {
        tc_fence_after();
        uint32_t sr[2][32];
        tmem_ld32(tS, sr[0]);
        tmem_ld32(tS + 32, sr[1]);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < BN; ++e) s[e] = __uint_as_float(sr[e >> 5][e & 31]);
      }
      tc_fence_before();
      mbar_arrive(bar(C::BAR_SFREE));
      if (failed) return;
      const int tile = w.t0 + d;
      if (tile >= w.nfull) {
        const int key0 = tile * BN;
#pragma unroll
        for (int e = 0; e < BN; ++e) {
          const int key = key0 + e;
          if (key >= key_lim || key > causal_lim) s[e] = -INFINITY;
        }
      }
      float c0 = fmax3(s[0], s[1], s[2]), c1 = fmax3(s[3], s[4], s[5]);
#pragma unroll
      for (int e = 6; e < 62; e += 4) {
        c0 = fmax3(c0, s[e], s[e + 1]);
        c1 = fmax3(c1, s[e + 2], s[e + 3]);
      }
      tmax = fmax3(c0, c1, fmaxf(s[62], s[63])) * sc;
    };
    if (h < n) load_scores(h, 0);
    // the row maxima of every CTA's first tile -> a common starting reference
    __syncwarp();
    for (int c = 0; c < NH; ++c)
      st_cluster_f32(peer_addr(sb + C::OFF_M0 + (h * BM + r) * 4, c), failed ? -INFINITY : tmax);
    cluster_arrive();
    cluster_wait();
    float m_O = -INFINITY, l = 0.f;
    {
      const float* m0 = reinterpret_cast<const float*>(smem + C::OFF_M0);
#pragma unroll
      for (int c = 0; c < NH; ++c) m_O = fmaxf(m_O, m0[c * BM + r]);
    }

    // own tile d: P and (m, l) into slot d % NPS here, then copied to the peers
    auto own_tile = [&](int d, int k) {
      if (k > 0) load_scores(d, k);
      const int slot = d % NPS;
      float m_ref = -INFINITY, l_src = 0.f;
      uint32_t pk[32];
      if (!failed) {
        m_ref = (m_O == -INFINITY || tmax > m_O + RESCALE_LOG2) ? tmax : m_O;
        const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;
        float2 sum_a = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const float2 xa =
              ffma2(make_float2(s[2 * e], s[2 * e + 1]), make_float2(sc, sc), make_float2(neg_m, neg_m));
          const float2 xb =
              ffma2(make_float2(s[2 * e + 2], s[2 * e + 3]), make_float2(sc, sc), make_float2(neg_m, neg_m));
          const float2 pa = make_float2(fast_exp2(xa.x), fast_exp2(xa.y));
          const float2 pb = make_float2(fast_exp2(xb.x), fast_exp2(xb.y));
          sum_a = fadd2(sum_a, pa);
          sum_b = fadd2(sum_b, pb);
          pk[e] = pack2<BF16>(pa.x, pa.y);
          pk[e + 1] = pack2<BF16>(pb.x, pb.y);
        }
        l_src = (sum_a.x + sum_a.y) + (sum_b.x + sum_b.y);
        // the slot's previous tile has been multiplied in every CTA
        if (d >= NPS) {
          const bool ok = mbar_wait_cluster(bar(C::BAR_SLOT_FREE + slot), ((d / NPS) - 1) & 1);
          if (__any_sync(0xffffffffu, !ok)) failed = true;
        }
      }
      if (!failed) {
        uint8_t* prow = smem + C::OFF_P + slot * C::P_BYTES + r * 128;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          *reinterpret_cast<uint4*>(prow + ((u ^ (r & 7)) << 4)) =
              make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        ml[slot * BM + r] = make_float2(m_ref, l_src);
        fence_proxy_async_smem();  // for this CTA's MMA and the copies to the peers
      }
      if (bar_red_or(BAR_SOFTMAX, BM, failed)) failed = true;
      if (!failed && r == 0) {
        const uint32_t src_p = sb + C::OFF_P + slot * C::P_BYTES;
        const uint32_t src_ml = sb + C::OFF_ML + slot * C::ML_BYTES;
        for (int c = 1; c < NH; ++c) {
          const uint32_t peer = static_cast<uint32_t>((h + c) % NH);
          const uint32_t pbar = peer_addr(bar(C::BAR_P_ARR + slot), peer);
          bulk_copy_to_peer(peer_addr(src_p, peer), src_p, C::P_BYTES, pbar);
          bulk_copy_to_peer(peer_addr(src_ml, peer), src_ml, C::ML_BYTES, pbar);
        }
      }
    };

    // tile j: take its reference and row sum into this CTA's (m_O, l)
    auto reconcile = [&](int j) {
      const int slot = j % NPS, wr = j % NH;
      if (wr != h && !failed) {
        const bool ok = mbar_wait_cluster(bar(C::BAR_P_ARR + slot), (j / NPS) & 1);
        if (__any_sync(0xffffffffu, !ok)) failed = true;
        if (!failed && r == 0) {
          if (j + NPS < n) mbar_arrive_expect_tx(bar(C::BAR_P_ARR + slot), C::P_BYTES + C::ML_BYTES);
          mbar_arrive_peer_relaxed(peer_addr(bar(C::BAR_RECV + slot), static_cast<uint32_t>(wr)));
        }
      }
      bool need_o = false, need_p = false;
      float alpha = 1.f, beta = 1.f;
      if (!failed) {
        const float2 v = ml[slot * BM + r];
        const float ms = v.x, ls = v.y;
        if (ls > 0.f) {
          if (l == 0.f) {  // nothing accumulated yet: the tile's reference becomes the row's
            m_O = ms;
            l = ls;
          } else if (ms > m_O) {
            alpha = fast_exp2(m_O - ms);
            l = l * alpha + ls;
            m_O = ms;
            need_o = true;
          } else if (ms < m_O) {
            beta = fast_exp2(ms - m_O);
            l += ls * beta;
            need_p = true;
          } else {
            l += ls;
          }
        }
      }
      if (__any_sync(0xffffffffu, need_o)) {
        // O holds tiles < j relative to the old reference: after this CTA's P . V of tile j - 1
        const int pj = j - 1;  // >= 0: a row with l > 0 has reconciled an earlier tile
        const bool ok = mbar_wait(bar(C::BAR_PV_DONE + pj % NPS), (pj / NPS) & 1);
        if (__any_sync(0xffffffffu, !ok)) failed = true;
        if (!failed) {
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < OC / 32; ++c) {
            uint32_t o[32];
            tmem_ld32(tO + 32 * c, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              const float2 x = fmul2(make_float2(__uint_as_float(o[e]), __uint_as_float(o[e + 1])),
                                     make_float2(alpha, alpha));
              o[e] = __float_as_uint(x.x);
              o[e + 1] = __float_as_uint(x.y);
            }
            tmem_st32(tO + 32 * c, o);
          }
          tmem_wait_st();
          tc_fence_before();
        }
      }
      bool bad = false;
      if (need_p && !failed) {
        // this row of P was computed against a smaller reference: scale it down;
        // an own tile only once every peer's copy has landed
        bool ok = true;
        if (wr == h) ok = mbar_wait_cluster(bar(C::BAR_RECV + slot), (j / NPS) & 1);
        if (ok) {
          uint8_t* prow = smem + C::OFF_P + slot * C::P_BYTES + r * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            uint4* q4 = reinterpret_cast<uint4*>(prow + (u << 4));
            uint4 v = *q4;
            uint32_t* wv = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float lo, hi;
              if constexpr (BF16) {
                const __nv_bfloat162 b2 = *reinterpret_cast<const __nv_bfloat162*>(&wv[e]);
                lo = __low2float(b2);
                hi = __high2float(b2);
              } else {
                const __half2 b2 = *reinterpret_cast<const __half2*>(&wv[e]);
                lo = __low2float(b2);
                hi = __high2float(b2);
              }
              wv[e] = pack2<BF16>(lo * beta, hi * beta);
            }
            *q4 = v;
          }
          fence_proxy_async_smem();
        } else {
          bad = true;
        }
      }
      if (__any_sync(0xffffffffu, bad)) failed = true;
      mbar_arrive(bar(C::BAR_P_READY + slot));
    };

    // own tiles in order, each followed by the reconciliation of every tile up to it
    int last = -1;
    for (int d = h, k = 0; last < n - 1; d += NH, ++k) {
      if (d < n) own_tile(d, k);
      const int upto = d < n ? d : n - 1;
      for (int j = last + 1; j <= upto; ++j) reconcile(j);
      last = upto;
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
      const bool live = l > 0.f;
      const bool row_in = row_ok && in_bounds(pp.status, grow, rows_total);  // checked build
      if (partial) {
        float4* dst = reinterpret_cast<float4*>(pp.ws_o + (w.sp * rows_total + grow) * R + h * OC);
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
        if (row_in && h == 0)
          pp.ws_ml[w.sp * rows_total + grow] = make_float2(live ? m_O : -INFINITY, live ? l : 0.f);
      } else {
        const float inv = live ? 1.f / l : __int_as_float(0x7fc00000);
        uint4* dst = reinterpret_cast<uint4*>(static_cast<uint8_t*>(out) + (grow * R + h * OC) * 2);
#pragma unroll 1
        for (int c = 0; c < OC / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(tO + 32 * c, o);
          tmem_wait_ld();
          if (row_in) {
            uint32_t pkd[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float2 x = fmul2(make_float2(__uint_as_float(o[2 * e]), __uint_as_float(o[2 * e + 1])),
                                     make_float2(inv, inv));
              pkd[e] = pack2<BF16>(x.x, x.y);
            }
#pragma unroll
            for (int u = 0; u < 4; ++u)
              dst[c * 4 + u] = make_uint4(pkd[4 * u], pkd[4 * u + 1], pkd[4 * u + 2], pkd[4 * u + 3]);
          }
        }
        if (row_in && lse && h == 0) lse[grow] = live ? (m_O + log2f(l)) * LN2 : -INFINITY;
      }
    }
  }
  // no CTA leaves while a peer may still copy into it or arrive on its barriers
  tc_fence_before();
  __syncwarp();
  cluster_arrive();
  cluster_wait();
  if (warp == WARP_MMA) {
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
