// attn_mla_bwd_tc.cuh - backward of paged MLA (absorbed projections) on the
// tcgen05 tensor cores: F16/BF16, latent rank R in {256, 512}, positional
// width Pd in {0, 64}, page_size a multiple of 8 that divides 128 or a
// multiple of 128.
//
// Source: ruDNN user guide, section 11 (the MLA backward returns dq, dqp, the
// latent gradient with its key and value parts, and dkp, recomputing the
// probabilities from the forward's statistics; the history gradients are
// reduced in a fixed order). With the forward's lse_r and D_r = dout_r . out_r,
// for every row r (a (query, head) pair of a sequence) and visible key j:
//   s = scale (q_r . c_j + qp_r . kp_j),   p = exp(s - lse_r),
//   dp = dout_r . c_j,                      ds' = scale p (dp - D_r),
//   dlatent_j = sum_r (p dout_r + ds' q_r),  dkp_j = sum_r ds' qp_r,
//   dq_r = sum_j ds' c_j,                    dqp_r = sum_j ds' kp_j.
// The rows of a sequence are contiguous in q, qp, dout and dq.
//
// An R-wide gradient accumulator does not fit in tensor memory beside S and
// dP, so, as in the forward, every 128-column slice h of it is a CTA of its
// own that recomputes S and dP (the same MMAs in the same order, so the same
// P in every slice). Both kernels stream 64-dimension chunks of their
// operands (128 rows x 128 bytes, 128-byte swizzle) through a ring of shared-
// memory slots and keep the chunks their gradient MMAs read in keep slots:
//  - key-major (KM): CTA = (sequence, 128-key block, slice h); for every
//    128-row tile of the sequence that can see the block:
//      S^T  = [c | kp] [q | qp]^T,  dP^T = c dout^T      (SS, keys = M)
//      P^T, dS'^T by the elementwise warps (16-bit, into S^T's and dP^T's
//      columns)
//      dlatent_h += P^T dout_h + dS'^T q_h,  dkp += dS'^T qp (h = 0)
//    (TS; dout_h, q_h, qp held in keep slots). Its key rows go straight to
//    the pages with exactly one reader; the ordered fp32 FMA pass writes the
//    pages read by several sequences (or blocks) and zeroes unread ones.
//  - query-major (QM): CTA = (sequence, 128-row tile, slice h); for every key
//    block the tile can see:  S = [q | qp] [c | kp]^T,  dP = dout c^T,  dS',
//    then dq_h += dS' c_h,  dqp += dS' kp (h = 0), with c_h and kp in keep
//    slots (two sets, so the next block's load overlaps this block's MMAs).
//    Decode-shaped calls (one row tile per sequence) take the sequences
//    longest first.
// Tensor memory: S [0, 128), dP [128, 256), the slice accumulator [256, 384),
// the positional accumulator [384, 448). 384 threads: 8 elementwise warps
// (two warpgroups, each owning 64 of the 128 columns of every TMEM lane), a
// TMA producer warp, an MMA-issuer warp, two warps whose registers go to the
// elementwise ones. Every mbarrier wait is bounded.
#pragma once

#include <atomic>

#include "attn_bwd_tc.cuh"
#include "paged_bwd.h"
#include "params.h"
#include "ptx.cuh"
#include "seq_order.cuh"

namespace attn {
namespace mlabwd {

using bwdtc::REG_EW;
using bwdtc::REG_OTHER;
using bwdtc::store_row16;
using bwdtc::tmem_a_kstep;
using bwdtc::tmem_ld64;
using bwdtc::tmem_st_packed64;

constexpr int BR = 128;                 // keys of a block, rows of a tile, TMEM lanes
constexpr int CHUNK_BYTES = BR * 128;   // one 128-row x 64-dimension 16-bit chunk
constexpr int NUM_THREADS = 384;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int TMEM_COLS = 512;
constexpr int COL_S = 0, COL_DP = 128, COL_ACC = 256, COL_ACCP = 384;
constexpr int SMEM_LIMIT = 227 * 1024;

// Row statistics and reverse index of the workspace, the outputs (any may be
// nullptr) and the natural scale.
struct MlaArgs {
  const float* lse2;   // [queries * H] lse in log2 units
  const float* dsum;   // [queries * H] D_r
  const int* offsets;  // [pages + 1] the reverse index's per-page offsets (reader counts)
  void* dq;            // [queries, H, R]
  void* dqp;           // [queries, H, Pd]
  void* dlat;          // [pages, page_size, R]
  void* dkp;           // [pages, page_size, Pd]
  float scale;
};

template <int R, int PD, bool KM>
struct Cfg {
  static_assert(R == 256 || R == 512, "tensor-core MLA backward latent ranks are 256 and 512");
  static_assert(PD == 0 || PD == 64, "tensor-core MLA backward positional widths are 0 and 64");
  static constexpr int NCL = R / 64;          // latent chunks of a row
  static constexpr int NCP = PD / 64;         // positional chunks (0 or 1)
  static constexpr int NCH = NCL + NCP;
  static constexpr int NH = R / 128;          // CTAs per block or tile: 128-column output slices
  static constexpr int KEEP = KM ? 4 + NCP : 2 + NCP;  // chunks the gradient MMAs read
  static constexpr int KBUF = KM ? 1 : 2;     // keep sets (query-major: double buffered)
  static constexpr int RESERVE = 2048;        // base alignment + barriers
  static constexpr int RING_FIT = (SMEM_LIMIT - RESERVE) / CHUNK_BYTES - KBUF * KEEP;
  static constexpr int RING = RING_FIT > 12 ? 12 : RING_FIT;
  static_assert(RING >= 4, "ring too small");
  static constexpr int OFF_KEEP = 0;
  static constexpr int OFF_RING = KBUF * KEEP * CHUNK_BYTES;
  static constexpr int OFF_BAR = OFF_RING + RING * CHUNK_BYTES;
  static constexpr int BAR_FULL = 0, BAR_EMPTY = RING, BAR_KFULL = 2 * RING, BAR_KFREE = BAR_KFULL + KBUF,
                       BAR_SDP = BAR_KFREE + KBUF, BAR_PDS = BAR_SDP + 1, BAR_DONE = BAR_PDS + 1,
                       NUM_BARS = BAR_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;
  static_assert(SMEM_BYTES <= SMEM_LIMIT, "shared memory");

  // Keep slot of chunk c in role `role` (0: key chunk, 1: query chunk, 2: dout
  // chunk) for slice h, or -1 when the chunk streams through the ring.
  __device__ static __forceinline__ int keep_slot(int c, int role, int h) {
    if constexpr (KM) {
      if (role == 1) return c == 2 * h ? 0 : (c == 2 * h + 1 ? 1 : (NCP && c == NCL ? 4 : -1));
      if (role == 2) return c == 2 * h ? 2 : (c == 2 * h + 1 ? 3 : -1);
      return -1;
    } else {
      if (role == 0) return c == 2 * h ? 0 : (c == 2 * h + 1 ? 1 : (NCP && c == NCL ? 2 : -1));
      return -1;
    }
  }
};

__device__ __forceinline__ int mla_keys(const PagedParams& pp, int s) {
  return min(max(__ldg(pp.seq_lens + s), 0), pp.max_pages * pp.page_size);
}

// A 128-key block [key0, key0 + 128) of chunk `x` (64 dimensions) of a
// paged [pages, page_size, width] cache into a ring or keep slot, page by page.
__device__ __forceinline__ void load_key_chunk(uint32_t dst, const CUtensorMap* m, uint32_t bar,
                                               const int32_t* table, const PagedParams& pp, int key0, int x) {
  const int P = pp.page_size;
  const int box_rows = P < BR ? P : BR;
  const int boxes = BR / box_rows;
  for (int i = 0; i < boxes; ++i) {
    const int key = key0 + i * box_rows;
    const int pidx = key / P;
    const int page = pidx < pp.max_pages ? __ldg(table + pidx) : -1;  // -1: a zero-filled box
    // checked build: the box lands inside the chunk (a skipped copy leaves the
    // slot's barrier to time out)
    if (!range_in_bounds(pp.status, i * box_rows, box_rows, BR)) continue;
    tma_load_3d(dst + i * box_rows * 128, m, bar, x, key % P, page);
  }
}

// Work of a CTA. Key-major: the key block and its rows' tiles [t_lo, t_hi);
// query-major: the row tile and its key blocks [0, n). In both, `n` counts
// the loop's iterations.
struct BWork {
  int s, h, q_lo, nq, L, rows_seq;
  int key0;        // key-major: first key of the block
  int tile;        // query-major: the row tile
  int t_lo, n;     // key-major: first row tile; both: iterations
};

template <int R, int PD, bool KM, bool LPT>
__device__ __forceinline__ BWork make_bwork(const PagedParams& pp, int nblk) {
  using C = Cfg<R, PD, KM>;
  BWork w;
  int lin = static_cast<int>(blockIdx.x);
  w.h = lin % C::NH;
  lin /= C::NH;
  const int blk = lin % nblk;  // key block (KM) or row tile (QM)
  const int sr = lin / nblk;
  if constexpr (LPT) w.s = seq_by_rank(pp, sr);  // decode-shaped query-major calls: longest first
  else w.s = sr;
  const int H = pp.Hq;
  w.q_lo = min(max(__ldg(pp.q_offsets + w.s), 0), pp.num_queries);
  const int q_hi = min(max(__ldg(pp.q_offsets + w.s + 1), w.q_lo), pp.num_queries);
  w.nq = q_hi - w.q_lo;
  w.rows_seq = w.nq * H;
  w.L = mla_keys(pp, w.s);
  w.key0 = w.tile = w.t_lo = w.n = 0;
  const bool dflt = pp.positions == nullptr;
  if constexpr (KM) {
    w.key0 = blk * BR;
    const int used = (w.L + pp.page_size - 1) / pp.page_size;  // pages the sequence reads
    if (w.nq == 0 || w.key0 >= used * pp.page_size) {  // not a block of this sequence's pages
      w.key0 = -1;
      return w;
    }
    if (w.key0 >= w.L) return w;  // slots past the last key: zeros
    const int ntiles = (w.rows_seq + BR - 1) / BR;
    // default positions: query qi sits at L - nq + qi and sees key0 when qi >= key0 - (L - nq)
    w.t_lo = (pp.causal && dflt) ? (max(0, w.key0 - (w.L - w.nq)) * H) / BR : 0;
    w.n = max(0, ntiles - w.t_lo);
  } else {
    w.tile = blk;
    const int row0 = blk * BR;
    if (row0 >= w.rows_seq) {
      w.tile = -1;
      return w;
    }
    int hi = w.L;
    if (pp.causal && dflt) {
      const int last_q = min(w.nq - 1, (row0 + BR - 1) / H);
      hi = min(hi, w.L - w.nq + last_q + 1);
    }
    w.n = hi > 0 ? (hi + BR - 1) / BR : 0;
  }
  return w;
}

template <int R, int PD, bool BF16, bool KM, bool LPT>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    mla_bwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_qp,
                      const __grid_constant__ CUtensorMap tm_do, const __grid_constant__ CUtensorMap tm_lat,
                      const __grid_constant__ CUtensorMap tm_kp, const PagedParams pp, const MlaArgs a,
                      int nblk) {
  using C = Cfg<R, PD, KM>;
  const BWork w = make_bwork<R, PD, KM, LPT>(pp, nblk);
  if (KM ? w.key0 < 0 : w.tile < 0) return;  // CTA-uniform: nothing of this sequence here
  const int H = pp.Hq;
  const int P = pp.page_size;
  const int32_t* table = pp.block_table + static_cast<size_t>(w.s) * pp.max_pages;

  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int N = w.n;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::RING; ++i) {
      mbar_init(bar(C::BAR_FULL + i), 1);
      mbar_init(bar(C::BAR_EMPTY + i), 1);
    }
    for (int i = 0; i < C::KBUF; ++i) {
      mbar_init(bar(C::BAR_KFULL + i), 1);
      mbar_init(bar(C::BAR_KFREE + i), 1);
    }
    mbar_init(bar(C::BAR_SDP), 1);
    mbar_init(bar(C::BAR_PDS), 256);
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
  // first global row of the rows tile of iteration it (KM) or of the CTA (QM)
  auto tile_row0 = [&](int it) -> int {
    return w.q_lo * H + (KM ? (w.t_lo + it) : w.tile) * BR;
  };
  auto key_base = [&](int it) -> int { return KM ? w.key0 : it * BR; };

  if (warp >= 8) {
    setmaxnreg_dec<REG_OTHER>();
    if (warp == WARP_TMA && N > 0) {
      // ------------------------------------------------------------ producer
      // (the whole warp waits; one elected lane issues the copies)
      if (elect_one()) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_do);
        tma_prefetch_desc(&tm_lat);
        if constexpr (PD > 0) {
          tma_prefetch_desc(&tm_qp);
          tma_prefetch_desc(&tm_kp);
        }
      }
      __syncwarp();
      // chunk c of role `role` of iteration it into dst, completing on b
      auto load = [&](int it, int c, int role, uint32_t dst, uint32_t b) {
        if (role == 0) {
          if (c < C::NCL) load_key_chunk(dst, &tm_lat, b, table, pp, key_base(it), 64 * c);
          else load_key_chunk(dst, &tm_kp, b, table, pp, key_base(it), 0);
        } else if (role == 1) {
          if (c < C::NCL) tma_load_2d(dst, &tm_q, b, 64 * c, tile_row0(it));
          else tma_load_2d(dst, &tm_qp, b, 0, tile_row0(it));
        } else {
          tma_load_2d(dst, &tm_do, b, 64 * c, tile_row0(it));
        }
      };
      bool ok = true;
      int rc = 0;   // ring loads issued
      int nit = 0;  // iterations whose keep loads were issued
      for (int it = 0; it < N && ok; ++it) {
        // the keep set of this iteration: free once the gradient MMAs of the
        // iteration that last used it completed
        const int kb = it % C::KBUF;
        if (it >= C::KBUF && !warp_wait(bar(C::BAR_KFREE + kb), ((it / C::KBUF) - 1) & 1)) { ok = false; break; }
        if (elect_one()) {
          mbar_arrive_expect_tx(bar(C::BAR_KFULL + kb), C::KEEP * CHUNK_BYTES);
          for (int c = 0; c < C::NCH; ++c)
            for (int role = 0; role < 3; ++role) {
              if (role == 2 && c >= C::NCL) continue;
              const int k = C::keep_slot(c, role, w.h);
              if (k >= 0)
                load(it, c, role, sb + C::OFF_KEEP + (kb * C::KEEP + k) * CHUNK_BYTES, bar(C::BAR_KFULL + kb));
            }
        }
        __syncwarp();
        ++nit;
        for (int c = 0; c < C::NCH && ok; ++c)
          for (int role = 0; role < 3; ++role) {
            if (role == 2 && c >= C::NCL) continue;
            if (C::keep_slot(c, role, w.h) >= 0) continue;
            const int slot = rc % C::RING;
            if (!warp_wait(bar(C::BAR_EMPTY + slot), ((rc / C::RING) & 1) ^ 1)) { ok = false; break; }
            if (elect_one()) {
              mbar_arrive_expect_tx(bar(C::BAR_FULL + slot), CHUNK_BYTES);
              load(it, c, role, sb + C::OFF_RING + slot * CHUNK_BYTES, bar(C::BAR_FULL + slot));
            }
            __syncwarp();
            ++rc;
          }
      }
      if (!ok && lane == 0) fail();
      // drain: every copy issued has landed before the CTA exits
      for (int i = 0; i < C::RING && i < rc; ++i) {
        const int fills = (rc - i + C::RING - 1) / C::RING;
        if (!warp_wait(bar(C::BAR_FULL + i), (fills - 1) & 1) && lane == 0) fail();
      }
      for (int kb = 0; kb < C::KBUF && kb < nit; ++kb) {
        const int fills = (nit - kb + C::KBUF - 1) / C::KBUF;
        if (!warp_wait(bar(C::BAR_KFULL + kb), (fills - 1) & 1) && lane == 0) fail();
      }
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_a = make_idesc_f16(BF16, BR, BR, false);   // S, dP: both K-major
      constexpr uint32_t idesc_g = make_idesc_f16(BF16, BR, 128, true);   // gradient slice, B MN-major
      constexpr uint32_t idesc_p = make_idesc_f16(BF16, BR, 64, true);    // positional gradient
      constexpr uint32_t CH16 = CHUNK_BYTES >> 4;
      constexpr uint32_t RSTEP16 = (16 * 128) >> 4;  // 16 rows of an MN-major chunk
      const uint64_t ring_k = smem_desc(sb + C::OFF_RING, 16, 1024, 2u);
      const uint64_t keep_k = smem_desc(sb + C::OFF_KEEP, 16, 1024, 2u);
      const uint64_t keep_mn = smem_desc(sb + C::OFF_KEEP, CHUNK_BYTES, 1024, 2u);
      bool ok = true;
      int rc = 0;
      for (int it = 0; it < N && ok; ++it) {
        const int kb = it % C::KBUF;
        if (!warp_wait(bar(C::BAR_KFULL + kb), (it / C::KBUF) & 1)) { ok = false; break; }
        // S and dP, chunk by chunk (descriptors of chunk c's three operands)
        for (int c = 0; c < C::NCH && ok; ++c) {
          uint64_t d[3];
          int used[3] = {-1, -1, -1};
          for (int role = 0; role < 3; ++role) {
            if (role == 2 && c >= C::NCL) continue;
            const int k = C::keep_slot(c, role, w.h);
            if (k >= 0) {
              d[role] = keep_k + (kb * C::KEEP + k) * CH16;
            } else {
              const int slot = rc % C::RING;
              if (!warp_wait(bar(C::BAR_FULL + slot), (rc / C::RING) & 1)) { ok = false; break; }
              d[role] = ring_k + slot * CH16;
              used[role] = slot;
              ++rc;
            }
          }
          if (!ok) break;
          tc_fence_after();
          // key-major: keys are M (A = key chunk); query-major: rows are M
          const uint64_t sa = KM ? d[0] : d[1], sbd = KM ? d[1] : d[0];
          if (elect_one()) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_ss(tmem + COL_S, sa + kk * 2, sbd + kk * 2, idesc_a, (c | kk) ? 1u : 0u);
          }
          __syncwarp();
          if (c < C::NCL) {
            const uint64_t pa = KM ? d[0] : d[2], pb = KM ? d[2] : d[0];
            if (elect_one()) {
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                umma_ss(tmem + COL_DP, pa + kk * 2, pb + kk * 2, idesc_a, (c | kk) ? 1u : 0u);
            }
            __syncwarp();
          }
          if (elect_one()) {
            for (int role = 0; role < 3; ++role)
              if (used[role] >= 0) umma_commit(bar(C::BAR_EMPTY + used[role]));
          }
          __syncwarp();
        }
        if (!ok) break;
        if (elect_one()) {
          umma_commit(bar(C::BAR_SDP));
        }
        __syncwarp();
        // the gradient slice, once the elementwise warps have written P and dS'
        if (!warp_wait(bar(C::BAR_PDS), it & 1)) { ok = false; break; }
        tc_fence_after();
        const uint64_t kmn = keep_mn + kb * C::KEEP * CH16;
        if constexpr (KM) {
          // dlatent_h += P^T dout_h  (keep 2, 3)  +  dS'^T q_h  (keep 0, 1)
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              umma_ts(tmem + COL_ACC, tmem + COL_S + tmem_a_kstep(k), kmn + 2 * CH16 + k * RSTEP16, idesc_g,
                      (it > 0 || k > 0) ? 1u : 0u);
#pragma unroll
            for (int k = 0; k < 8; ++k)
              umma_ts(tmem + COL_ACC, tmem + COL_DP + tmem_a_kstep(k), kmn + k * RSTEP16, idesc_g, 1u);
          }
          __syncwarp();
          if (C::NCP && w.h == 0) {  // dkp += dS'^T qp  (keep 4)
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < 8; ++k)
                umma_ts(tmem + COL_ACCP, tmem + COL_DP + tmem_a_kstep(k), kmn + 4 * CH16 + k * RSTEP16, idesc_p,
                        (it > 0 || k > 0) ? 1u : 0u);
            }
            __syncwarp();
          }
        } else {
          // dq_h += dS' c_h  (keep 0, 1);  dqp += dS' kp  (keep 2)
          if (elect_one()) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
              umma_ts(tmem + COL_ACC, tmem + COL_DP + tmem_a_kstep(k), kmn + k * RSTEP16, idesc_g,
                      (it > 0 || k > 0) ? 1u : 0u);
          }
          __syncwarp();
          if (C::NCP && w.h == 0) {
            if (elect_one()) {
#pragma unroll
              for (int k = 0; k < 8; ++k)
                umma_ts(tmem + COL_ACCP, tmem + COL_DP + tmem_a_kstep(k), kmn + 2 * CH16 + k * RSTEP16, idesc_p,
                        (it > 0 || k > 0) ? 1u : 0u);
            }
            __syncwarp();
          }
        }
        if (elect_one()) {
          umma_commit(bar(C::BAR_KFREE + kb));
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
    const int half = warp >> 2;                // columns [64 half, +64) of every lane
    const int lrow = ((warp & 3) << 5) + lane;  // TMEM lane: key (KM) or row (QM) of the tile
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_off + COL_S, tDP = tmem + lane_off + COL_DP;
    const float sc = pp.scale_log2;
    const float scale = a.scale;
    const bool dflt = pp.positions == nullptr;
    const int64_t nrows = static_cast<int64_t>(pp.num_queries) * H;  // extent for the checked build
    // statistics of one row of the sequence (its tile-local index r): lse2, D
    // and the largest key it sees (-1: no row, or no visible key)
    auto row_stats = [&](int r, float& l2, float& ds, int& lim) {
      l2 = -INFINITY;
      ds = 0.f;
      lim = -1;
      if (r >= w.rows_seq) return;
      const int64_t g = static_cast<int64_t>(w.q_lo) * H + r;
      if (!in_bounds(pp.status, g, nrows)) return;
      l2 = __ldg(a.lse2 + g);
      if (l2 == -INFINITY) return;
      ds = __ldg(a.dsum + g);
      const int qi = r / H;
      int pos = w.L - 1;
      if (pp.causal)
        pos = dflt ? w.L - w.nq + qi
                   : (in_bounds(pp.status, w.q_lo + qi, pp.num_queries) ? __ldg(pp.positions + w.q_lo + qi) : -1);
      lim = min(pos, w.L - 1);
    };
    bool failed = false;
    if constexpr (KM) {
      const int key = w.key0 + lrow;
      for (int it = 0; it < N; ++it) {
        // rows 64 half + lane and 64 half + 32 + lane of the tile, shuffled out below
        const int rbase = (w.t_lo + it) * BR + 64 * half;
        float l2a, l2b, dsa, dsb;
        int lima, limb;
        row_stats(rbase + lane, l2a, dsa, lima);
        row_stats(rbase + 32 + lane, l2b, dsb, limb);
        const bool ok = mbar_wait(bar(C::BAR_SDP), it & 1);
        if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
        tc_fence_after();
        float x[64], dp[64];
        tmem_ld64<BF16>(tS + 64 * half, x);
        tmem_ld64<BF16>(tDP + 64 * half, dp);
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const float l2 = __shfl_sync(0xffffffffu, c < 32 ? l2a : l2b, c & 31);
          const float dsi = __shfl_sync(0xffffffffu, c < 32 ? dsa : dsb, c & 31);
          const int lim = __shfl_sync(0xffffffffu, c < 32 ? lima : limb, c & 31);
          const bool vis = key <= lim;
          const float pr = vis ? fast_exp2(x[c] * sc - l2) : 0.f;
          x[c] = pr;
          dp[c] = pr * (dp[c] - dsi) * scale;
        }
        tmem_st_packed64<BF16>(tS + 64 * half, x);
        tmem_st_packed64<BF16>(tDP + 64 * half, dp);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(C::BAR_PDS));
      }
    } else {
      float l2, dsi;
      int lim;
      row_stats(w.tile * BR + lrow, l2, dsi, lim);
      for (int it = 0; it < N; ++it) {
        const bool ok = mbar_wait(bar(C::BAR_SDP), it & 1);
        if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
        tc_fence_after();
        float x[64], dp[64];
        tmem_ld64<BF16>(tS + 64 * half, x);
        tmem_ld64<BF16>(tDP + 64 * half, dp);
        const int kc0 = it * BR + 64 * half;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const bool vis = kc0 + c <= lim;
          const float pr = vis ? fast_exp2(x[c] * sc - l2) : 0.f;
          dp[c] = pr * (dp[c] - dsi) * scale;
        }
        tmem_st_packed64<BF16>(tDP + 64 * half, dp);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(C::BAR_PDS));
      }
    }
    // ---------------------------------------------------------------- epilogue
    if (failed) {
      if (lane == 0) fail();
    } else {
      bool ok = true;
      if (N > 0) {
        ok = mbar_wait(bar(C::BAR_DONE), 0);
        if (__any_sync(0xffffffffu, !ok)) { ok = false; if (lane == 0) fail(); }
      }
      if (ok) {
        tc_fence_after();
        // destination rows: key-major, the key's slot of a page with exactly
        // one reader; query-major, the sequence's row
        int64_t drow = -1;
        if constexpr (KM) {
          const int key = w.key0 + lrow;
          const int pidx = key / P;
          const int used = (w.L + P - 1) / P;
          int page = (pidx < used && in_bounds(pp.status, static_cast<int64_t>(w.s) * pp.max_pages + pidx,
                                               static_cast<int64_t>(pp.num_seqs) * pp.max_pages))
                         ? __ldg(table + pidx) : -1;
          if (page >= pp.num_pages ||
              (page >= 0 && __ldg(a.offsets + page + 1) - __ldg(a.offsets + page) != 1))
            page = -1;
          if (page >= 0) drow = static_cast<int64_t>(page) * P + key % P;
          if (drow >= 0 && !in_bounds(pp.status, drow, static_cast<int64_t>(pp.num_pages) * P)) drow = -1;
        } else {
          const int r = w.tile * BR + lrow;
          if (r < w.rows_seq) drow = static_cast<int64_t>(w.q_lo) * H + r;
          if (drow >= 0 && !in_bounds(pp.status, drow, nrows)) drow = -1;
        }
        void* dst = KM ? a.dlat : a.dq;   // the slice's gradient rows
        void* dstp = KM ? a.dkp : a.dqp;  // the positional gradient rows (slice 0)
        if (dst != nullptr) {
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            float v[32];
            if (N > 0) {
              uint32_t rr[32];
              tmem_ld32(tmem + lane_off + COL_ACC + 64 * half + 32 * c, rr);
              tmem_wait_ld();
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(rr[e]);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) v[e] = 0.f;
            }
            if (drow >= 0)
              store_row16<BF16, 32>(static_cast<uint8_t*>(dst) + (drow * R + 128 * w.h + 64 * half + 32 * c) * 2, v,
                                    1.f);
          }
        }
        if (C::NCP && w.h == 0 && dstp != nullptr) {
          float v[32];
          if (N > 0) {
            uint32_t rr[32];
            tmem_ld32(tmem + lane_off + COL_ACCP + 32 * half, rr);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = __uint_as_float(rr[e]);
          } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) v[e] = 0.f;
          }
          if (drow >= 0) store_row16<BF16, 32>(static_cast<uint8_t*>(dstp) + (drow * PD + 32 * half) * 2, v, 1.f);
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

}  // namespace mlabwd
}  // namespace attn

namespace attn {
namespace mlabwd {

// Encode the five tensor maps and launch the key-major kernel (when dlatent
// or dkpos is wanted) and the query-major one (when dq or dqp is).
template <int R, int PD, bool BF16>
cudaError_t launch_mla_bwd_tc(EncodeTiledFn enc, const PagedParams& pp, const void* q, const void* qp,
                              const void* lat, const void* kp, const void* dout, const MlaArgs& a,
                              cudaStream_t stream) {
  const CUtensorMapDataType dt = BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const cuuint32_t estride[3] = {1, 1, 1};
  const cuuint64_t rows = static_cast<cuuint64_t>(pp.num_queries) * pp.Hq;
  CUtensorMap tq, tqp, tdo, tlat, tkp;
  auto enc2 = [&](CUtensorMap* m, const void* base, int width) {  // [rows, width], boxes of 64 x 128
    const cuuint64_t gdim[2] = {static_cast<cuuint64_t>(width), rows};
    const cuuint64_t gstride[1] = {static_cast<cuuint64_t>(width) * 2};
    const cuuint32_t box[2] = {64u, static_cast<cuuint32_t>(BR)};
    return enc(m, dt, 2, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  auto enc3 = [&](CUtensorMap* m, const void* base, int width) {  // [pages, page_size, width]
    const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(width), static_cast<cuuint64_t>(pp.page_size),
                                static_cast<cuuint64_t>(pp.num_pages)};
    const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(width) * 2,
                                   static_cast<cuuint64_t>(pp.page_size) * width * 2};
    const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(pp.page_size < BR ? pp.page_size : BR), 1u};
    return enc(m, dt, 3, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  };
  if (enc2(&tq, q, R) != CUDA_SUCCESS || enc2(&tdo, dout, R) != CUDA_SUCCESS || enc3(&tlat, lat, R) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  if constexpr (PD > 0) {
    if (enc2(&tqp, qp, PD) != CUDA_SUCCESS || enc3(&tkp, kp, PD) != CUDA_SUCCESS) return cudaErrorInvalidValue;
  } else {
    tqp = tq;  // unused
    tkp = tlat;
  }
  const unsigned long long bit = pp.device >= 0 && pp.device < 64 ? 1ull << pp.device : 0ull;
  // shared-memory opt-in once per kernel and device
  auto opt_in = [&](auto kern, int smem, std::atomic<unsigned long long>& done) -> cudaError_t {
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
  };
  static std::atomic<unsigned long long> configured[3] = {{0}, {0}, {0}};
  if (a.dlat || a.dkp) {
    using C = Cfg<R, PD, true>;
    const int64_t kblocks = (static_cast<int64_t>(pp.max_pages) * pp.page_size + BR - 1) / BR;
    const int64_t ctas = static_cast<int64_t>(pp.num_seqs) * kblocks * C::NH;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (ctas > 0) {
      auto kern = mla_bwd_tc_kernel<R, PD, BF16, true, false>;
      cudaError_t e = opt_in(kern, C::SMEM_BYTES, configured[0]);
      if (e != cudaSuccess) return e;
      kern<<<static_cast<unsigned>(ctas), NUM_THREADS, C::SMEM_BYTES, stream>>>(tq, tqp, tdo, tlat, tkp, pp, a,
                                                                                 static_cast<int>(kblocks));
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  if (a.dq || a.dqp) {
    using C = Cfg<R, PD, false>;
    const int64_t rtiles = (static_cast<int64_t>(pp.max_queries) * pp.Hq + BR - 1) / BR;
    const int64_t ctas = static_cast<int64_t>(pp.num_seqs) * rtiles * C::NH;
    if (ctas > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    if (ctas > 0) {
      const bool lpt = rtiles == 1;  // decode-shaped: the sequences longest first
      auto kern = lpt ? mla_bwd_tc_kernel<R, PD, BF16, false, true> : mla_bwd_tc_kernel<R, PD, BF16, false, false>;
      cudaError_t e = opt_in(kern, C::SMEM_BYTES, configured[lpt ? 2 : 1]);
      if (e != cudaSuccess) return e;
      kern<<<static_cast<unsigned>(ctas), NUM_THREADS, C::SMEM_BYTES, stream>>>(tq, tqp, tdo, tlat, tkp, pp, a,
                                                                                 static_cast<int>(rtiles));
      e = cudaGetLastError();
      if (e != cudaSuccess) return e;
    }
  }
  return cudaSuccess;
}

}  // namespace mlabwd
}  // namespace attn
