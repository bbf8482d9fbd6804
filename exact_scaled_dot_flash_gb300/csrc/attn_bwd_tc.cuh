// attn_bwd_tc.cuh - attention backward on the tcgen05 tensor cores (F16/BF16,
// D in {64, 128}), the ordered path: no atomics, a fixed summation order.
//
// Source: ruDNN user guide, section 11: the backward returns dq, dk, dv and
// recomputes the probabilities from the inputs and the forward's row
// log-sum-exp instead of storing the score matrix. For visible (i, j):
//   p = exp2(s2_ij - lse2_i),  s2 = (scale q_i.k_j + bias_ij) log2 e,
//   ds = p (dp - D_i),  dp = dout_i . v_j,  D_i = dout_i . o_i,
//   dv_j = sum_i p dout_i,  dk_j = scale sum_i ds q_i,  dq_i = scale sum_j ds k_j.
//
// Two kernels, 384 threads each (8 elementwise warps, a TMA producer warp,
// an MMA-issuer warp, two idle warps whose registers go to the first eight):
//
// dkdv_tc_kernel: one CTA per (b, kv head, 128 keys). K and V stay in shared
// memory; (Q, dO) tiles of 128 rows of every query head of the group stream
// through a ring. Per query tile i, with keys as the MMA's M (TMEM lanes):
//   S^T  = K Q_i^T      (SS)           -> TMEM [0, 128)
//   dP^T = V dO_i^T     (SS)           -> TMEM [128, 256)
//   P^T  = exp2(S^T * c - lse2)        written as 16-bit into S^T's columns
//   dV  += P^T dO_i     (TS, dO_i MN-major)   TMEM [256, 256 + D)
//   dS^T = P^T (dP^T - D)              written as 16-bit into dP^T's columns
//   dK  += dS^T Q_i     (TS, Q_i MN-major)    TMEM [256 + D, 256 + 2D)
// issued as S(i) dP(i) | dV(i) S(i+1) | dK(i) dP(i+1) | ..., so each
// elementwise step overlaps an MMA. Warpgroup w of the eight warps handles
// query columns [64w, 64w + 64) of every key row.
//
// dq_tc_kernel: one CTA per (b, query head, 128 rows); (K, V) tiles stream
// through a ring. Per key tile j, rows as M:
//   S   = Q K_j^T   (SS) -> TMEM [128 (j & 1), +128)   (double buffered)
//   dP  = dO V_j^T  (SS) -> TMEM [256, 384)
//   dS  = P (dP - D)   16-bit into dP's columns
//   dQ += dS K_j    (TS, K_j MN-major) -> TMEM [384, 384 + D)
// issued as S(0) dP(0) S(1) | dQ(0) dP(1) S(2) | dQ(1) dP(2) S(3) | ...
//
// Each row is shared by two warps (one per warpgroup), each owning 64 of the
// 128 columns. A warp packs its 64 16-bit results into the first 32 columns of
// its own 64: never into columns the other warp may still have to read. The
// TS MMA then takes K-steps 0-3 from columns [0, 32) and K-steps 4-7 from
// columns [64, 96) of the region (tmem_a_kstep).
//
// The same 128B-swizzled tile serves as a K-major operand (rows = M or N,
// K = D) and as an MN-major one (rows = K, N = D). Every mbarrier wait is
// bounded; on expiry a CTA records STATUS_TIMEOUT, drains and exits.
#pragma once

#include <atomic>

#include "params.h"
#include "ptx.cuh"

namespace attn {
namespace bwdtc {

constexpr int BR = 128;           // rows of every tile (TMEM lanes)
constexpr int NUM_THREADS = 384;
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int TMEM_COLS = 512;
constexpr int REG_EW = 200;       // elementwise warps (2 x 128 x 200 + 128 x 96 <= 384 x 168)
constexpr int REG_OTHER = 96;
constexpr float LOG2E = 1.4426950408889634f;

template <int D>
struct Cfg {
  static_assert(D == 64 || D == 128, "tensor-core backward head dims are 64 and 128");
  static constexpr int BOX_D = 64;                      // 128-byte swizzled rows of 16-bit values
  static constexpr int NCHUNK = D / BOX_D;
  static constexpr int CHUNK_BYTES = BR * 128;          // one 128-row x 64-column box
  static constexpr int TILE_BYTES = NCHUNK * CHUNK_BYTES;
  static constexpr int STAGES = D == 128 ? 2 : 4;       // ring slots, each two tiles
  static constexpr int SBO = 1024;
  static constexpr uint32_t LAYOUT = 2u;                // SW128
  static constexpr int KSTEPS_D = D / 16;               // K = D contractions
  static constexpr int KSTEPS_R = BR / 16;              // K = 128 rows contractions
  // shared memory: two resident tiles, then the ring
  static constexpr int OFF_RING = 2 * TILE_BYTES;
  static constexpr int OFF_BAR = OFF_RING + STAGES * 2 * TILE_BYTES;
  static constexpr int NUM_BARS = 2 * STAGES + 8;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  // per elementwise warp, the current query tile's column statistics (lse2, D,
  // visibility limit) of the paged key-major kernel, read with broadcast loads
  // (the dense kernel shuffles them: staging them measured no faster there)
  static constexpr int OFF_STATS = (OFF_MISC + 16 + 15) / 16 * 16;
  static constexpr int STATS_PER_WARP = 3 * 64;  // floats
  static constexpr int SMEM_BYTES = OFF_STATS + 8 * STATS_PER_WARP * 4 + 1024;
  static_assert(SMEM_BYTES <= 232448, "key-major kernel shared memory");
  static constexpr int BAR_FULL = 0, BAR_EMPTY = STAGES;
  static constexpr int BAR_RES = 2 * STAGES;            // resident tiles loaded
  static constexpr int BAR_S = BAR_RES + 1;             // 2 (dq kernel double-buffers S)
  static constexpr int BAR_DP = BAR_S + 2;
  static constexpr int BAR_P = BAR_DP + 1;              // dkdv: P^T written
  static constexpr int BAR_DS = BAR_P + 1;
  static constexpr int BAR_DONE = BAR_DS + 1;
};

// TMEM column of K-step k (16 rows of K = 8 packed columns) of an A operand
// written by the two warpgroups into [0, 32) and [64, 96) of a 128-column region
__device__ __forceinline__ uint32_t tmem_a_kstep(int k) { return (k < 4 ? 0 : 64) + (k & 3) * 8; }

// 16-byte-unit offset of K-step k inside a K-major 128B-swizzled tile
template <int D>
__device__ __forceinline__ uint32_t kstep16(int k) {
  return (k / 4) * (Cfg<D>::CHUNK_BYTES >> 4) + (k % 4) * 2;
}

template <bool BF16>
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float* x) {
  uint32_t r[2][32];
  tmem_ld32(taddr, r[0]);
  tmem_ld32(taddr + 32, r[1]);
  tmem_wait_ld();
#pragma unroll
  for (int i = 0; i < 64; ++i) x[i] = __uint_as_float(r[i >> 5][i & 31]);
}

// 64 fp32 values -> 32 packed 16-bit pairs -> tensor memory columns [taddr, +32)
template <bool BF16>
__device__ __forceinline__ void tmem_st_packed64(uint32_t taddr, const float* x) {
  uint32_t pk[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) pk[i] = pack2<BF16>(x[2 * i], x[2 * i + 1]);
  tmem_st32(taddr, pk);
}

// Store D/2 fp32 values (one thread's half row) to global memory in 16-bit.
// Linear CTA index -> (tile rank, head) over a grid of (tiles, heads): heads
// are taken HEAD_GROUP at a time, and inside a group the tiles of all its heads
// are interleaved by rank, rank 0 first. The kernels map rank 0 to their
// heaviest causal tile, so the longest CTAs start first across the whole grid
// while the tiles a group's CTAs share stay in L2.
constexpr int HEAD_GROUP = 16;
__device__ __forceinline__ void cta_order(int& rank, int& head) {
  const int ntiles = static_cast<int>(gridDim.x), nheads = static_cast<int>(gridDim.y);
  const int lin = static_cast<int>(blockIdx.y) * ntiles + static_cast<int>(blockIdx.x);
  const int per_group = ntiles * HEAD_GROUP;
  const int g = lin / per_group;
  const int within = lin - g * per_group;
  const int hg = min(HEAD_GROUP, nheads - g * HEAD_GROUP);
  rank = within / hg;
  head = g * HEAD_GROUP + (within - rank * hg);
}

template <bool BF16, int N>
__device__ __forceinline__ void store_row16(void* dst, const float* x, float mul) {
  uint4* d = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int i = 0; i < N / 8; ++i)
    d[i] = make_uint4(pack2<BF16>(x[8 * i] * mul, x[8 * i + 1] * mul), pack2<BF16>(x[8 * i + 2] * mul, x[8 * i + 3] * mul),
                      pack2<BF16>(x[8 * i + 4] * mul, x[8 * i + 5] * mul), pack2<BF16>(x[8 * i + 6] * mul, x[8 * i + 7] * mul));
}



template <int D, bool BF16, bool BIAS>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    dkdv_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                   const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                   const KernelParams p, const BwdArgs a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work: 128 keys of one (b, kv head); every query tile that sees them
  // (causal: the first key blocks see the most query tiles, so they start first)
  int kb, bhk;
  cta_order(kb, bhk);
  const int b = bhk / p.Hkv, hk = bhk - b * p.Hkv;
  const int key0 = kb * BR;
  int lim = p.Sk;
  if (p.padding) {
    const int L = __ldg(p.kv_lens + b);
    lim = L < 0 ? 0 : (L > p.Sk ? p.Sk : L);
  }
  const int diag = p.Sk - p.Sq;
  const int nqt = (p.Sq + BR - 1) / BR;
  const int qt_lo = p.causal ? max(0, key0 - diag) / BR : 0;
  const int per_head = key0 < lim ? max(0, nqt - qt_lo) : 0;
  const int N = per_head * p.group;  // iterations: (query head of the group, query tile)

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(bar(C::BAR_FULL + s), 1);
      mbar_init(bar(C::BAR_EMPTY + s), 1);
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
    if (p.status) atomicOr(p.status, STATUS_TIMEOUT);
  };

  if (warp >= 8) {
    setmaxnreg_dec<REG_OTHER>();
    if (warp == WARP_TMA && lane == 0 && N > 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      mbar_arrive_expect_tx(bar(C::BAR_RES), 2 * C::TILE_BYTES);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d(sb + c * C::CHUNK_BYTES, &tm_k, bar(C::BAR_RES), c * C::BOX_D, key0, bhk);
        tma_load_3d(sb + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_v, bar(C::BAR_RES), c * C::BOX_D, key0, bhk);
      }
      int it = 0;
      for (; it < N; ++it) {
        const int s = it % C::STAGES;
        if (!mbar_wait(bar(C::BAR_EMPTY + s), ((it / C::STAGES) & 1) ^ 1)) { fail(); break; }
        const int g = it / per_head, qt = qt_lo + (it - g * per_head);
        const int bhq = b * p.Hq + hk * p.group + g;
        const uint32_t dst = sb + C::OFF_RING + s * 2 * C::TILE_BYTES;
        mbar_arrive_expect_tx(bar(C::BAR_FULL + s), 2 * C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c) {
          tma_load_3d(dst + c * C::CHUNK_BYTES, &tm_q, bar(C::BAR_FULL + s), c * C::BOX_D, qt * BR, bhq);
          tma_load_3d(dst + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_do, bar(C::BAR_FULL + s), c * C::BOX_D,
                      qt * BR, bhq);
        }
      }
      // drain: every copy issued has landed before the CTA exits
      for (int s = 0; s < C::STAGES && s < it; ++s) {
        const int fills = (it - s + C::STAGES - 1) / C::STAGES;
        if (!mbar_wait(bar(C::BAR_FULL + s), (fills - 1) & 1)) fail();
      }
      if (!mbar_wait(bar(C::BAR_RES), 0)) fail();
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_s = make_idesc_f16(BF16, BR, BR, false);  // M = keys, N = query rows
      constexpr uint32_t idesc_o = make_idesc_f16(BF16, BR, D, true);    // N = D, B MN-major
      constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
      constexpr uint32_t RSTEP16 = (16 * 128) >> 4;  // 16 rows of an MN-major tile
      const uint64_t dk_a = smem_desc(sb, 16, C::SBO, C::LAYOUT);
      const uint64_t dv_a = smem_desc(sb + C::TILE_BYTES, 16, C::SBO, C::LAYOUT);
      const uint64_t ring_k = smem_desc(sb + C::OFF_RING, 16, C::SBO, C::LAYOUT);           // K-major views
      const uint64_t ring_mn = smem_desc(sb + C::OFF_RING, C::CHUNK_BYTES, C::SBO, C::LAYOUT);  // MN-major views
      bool ok = true;
      auto issue_s = [&](int it) {  // S^T = K Q_i^T, dP^T = V dO_i^T
        const int s = it % C::STAGES;
        if (!warp_wait(bar(C::BAR_FULL + s), (it / C::STAGES) & 1)) return false;
        tc_fence_after();
        const uint64_t q = ring_k + s * 2 * TILE16;
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
        const int s = it % C::STAGES;
        const uint64_t g = ring_k + s * 2 * TILE16 + TILE16;
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
          const int s = it % C::STAGES;
          // dV += P^T dO_i   (P^T: 16-bit in S^T's columns)
          if (!warp_wait(bar(C::BAR_P), it & 1)) { ok = false; break; }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t g = ring_mn + s * 2 * TILE16 + TILE16;
#pragma unroll
            for (int k = 0; k < C::KSTEPS_R; ++k)
              umma_ts(tmem + 256, tmem + tmem_a_kstep(k), g + k * RSTEP16, idesc_o, (it > 0 || k > 0) ? 1u : 0u);
          }
          __syncwarp();
          if (it + 1 < N && !issue_s(it + 1)) { ok = false; break; }
          // dK += dS^T Q_i   (dS^T: 16-bit in dP^T's columns)
          if (!warp_wait(bar(C::BAR_DS), it & 1)) { ok = false; break; }
          tc_fence_after();
          if (elect_one()) {
            const uint64_t q = ring_mn + s * 2 * TILE16;
#pragma unroll
            for (int k = 0; k < C::KSTEPS_R; ++k)
              umma_ts(tmem + 256 + D, tmem + BR + tmem_a_kstep(k), q + k * RSTEP16, idesc_o,
                      (it > 0 || k > 0) ? 1u : 0u);
            umma_commit(bar(C::BAR_EMPTY + s));
          }
          __syncwarp();
          if (it + 1 < N) issue_dp(it + 1);
        }
      }
      if (!ok && lane == 0) fail();
      if (elect_one()) umma_commit(bar(C::BAR_DONE));
      __syncwarp();
      if (!warp_wait(bar(C::BAR_DONE), 0) && lane == 0) fail();
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- elementwise
    setmaxnreg_inc<REG_EW>();
    const int half = warp >> 2;                      // query columns [64 half, +64)
    const int row = ((warp & 3) << 5) + lane;        // key row = TMEM lane
    const int key = key0 + row;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_off, tDP = tS + BR;
    const float sc = p.scale_log2;
    bool failed = false;
    for (int it = 0; it < N; ++it) {
      const int g = it / per_head, qt = qt_lo + (it - g * per_head);
      const int hq = hk * p.group + g;
      const size_t bhq = static_cast<size_t>(b) * p.Hq + hq;
      const int i0 = qt * BR + 64 * half;
      const float* bcol = nullptr;
      if constexpr (BIAS) {
        const int bb = p.bias_b == 1 ? 0 : b;
        const int bh = p.bias_h == 1 ? 0 : hq;
        bcol = p.bias + (static_cast<size_t>(bb) * p.bias_h + bh) * p.Sq * static_cast<size_t>(p.Sk) + key;
      }
      // lse2 and D of this warpgroup's 64 query rows: lane l holds rows l and
      // l + 32 (coalesced loads, issued before the wait), shuffled out below
      const int ia = i0 + lane, ib = i0 + 32 + lane;
      const int64_t nrows = static_cast<int64_t>(p.B) * p.Hq * p.Sq;  // extents for the checked build
      const bool oka = ia < p.Sq && in_bounds(p.status, static_cast<int64_t>(bhq) * p.Sq + ia, nrows);
      const bool okb = ib < p.Sq && in_bounds(p.status, static_cast<int64_t>(bhq) * p.Sq + ib, nrows);
      const float l2a = oka ? __ldg(a.lse2 + bhq * p.Sq + ia) : -INFINITY;
      const float l2b = okb ? __ldg(a.lse2 + bhq * p.Sq + ib) : -INFINITY;
      const float dsa = oka ? __ldg(a.dsum + bhq * p.Sq + ia) : 0.f;
      const float dsb = okb ? __ldg(a.dsum + bhq * p.Sq + ib) : 0.f;
      float x[64];
      const bool ok = mbar_wait(bar(C::BAR_S), it & 1);
      if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
      tc_fence_after();
      tmem_ld64<BF16>(tS + 64 * half, x);
      // every (key, query) pair of this warp's block visible: no per-element mask;
      // a query row without a visible key takes lse2 = +inf, so its p is exactly 0
      const bool interior = !BIAS && key0 + BR - 1 < lim && (!p.causal || key0 + BR - 1 <= i0 + diag);
      if (interior) {
        const float l2fa = l2a == -INFINITY ? INFINITY : l2a, l2fb = l2b == -INFINITY ? INFINITY : l2b;
#pragma unroll
        for (int c = 0; c < 64; ++c)
          x[c] = fast_exp2(x[c] * sc - __shfl_sync(0xffffffffu, c < 32 ? l2fa : l2fb, c & 31));
      } else {
        const bool key_vis = key < lim;
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          const int i = i0 + c;
          const float l2 = __shfl_sync(0xffffffffu, c < 32 ? l2a : l2b, c & 31);
          const bool vis = key_vis && (!p.causal || key <= i + diag) && l2 != -INFINITY;
          float s2 = x[c] * sc - l2;
          if constexpr (BIAS) {
            const int64_t bi = (bcol - p.bias) + static_cast<int64_t>(i) * p.Sk;
            if (vis && in_bounds(p.status, bi, static_cast<int64_t>(p.bias_b) * p.bias_h * p.Sq * p.Sk))
              s2 = fmaf(__ldg(p.bias + bi), LOG2E, s2);
          }
          x[c] = vis ? fast_exp2(s2) : 0.f;
        }
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
      for (int c = 0; c < 64; ++c) {
        const float dsi = __shfl_sync(0xffffffffu, c < 32 ? dsa : dsb, c & 31);
        dp[c] = x[c] * (dp[c] - dsi);
      }
      tmem_st_packed64<BF16>(tDP + 64 * half, dp);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar(C::BAR_DS));
    }
    // ---------------------------------------------------------------- epilogue
    // warpgroup 0 writes dK (scaled), warpgroup 1 dV, one key row per thread
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
        const uint32_t src = tmem + lane_off + 256 + (half == 0 ? D : 0);
        void* dst = half == 0 ? a.dk : a.dv;
        const float mul = half == 0 ? a.scale : 1.f;
        uint8_t* rowp = static_cast<uint8_t*>(dst) + (static_cast<size_t>(bhk) * p.Sk + key) * D * 2;
        const bool row_in = key < p.Sk && range_in_bounds(p.status, (static_cast<int64_t>(bhk) * p.Sk + key) * D, D,
                                                          static_cast<int64_t>(p.B) * p.Hkv * p.Sk * D);
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
          if (row_in) store_row16<BF16, 32>(rowp + c * 64, v, mul);
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


// Shared-memory plan of the dq kernel: Q and dO resident, then separate rings
// for K (held until dQ(j) completes) and V (released after dP(j)).
template <int D>
struct DqCfg {
  using C = Cfg<D>;
  static constexpr int KST = D == 128 ? 3 : 4;
  static constexpr int VST = D == 128 ? 2 : 4;
  static constexpr int OFF_K = 2 * C::TILE_BYTES;
  static constexpr int OFF_V = OFF_K + KST * C::TILE_BYTES;
  static constexpr int OFF_BAR = OFF_V + VST * C::TILE_BYTES;
  static constexpr int BAR_KFULL = 0, BAR_KEMPTY = KST, BAR_VFULL = 2 * KST, BAR_VEMPTY = 2 * KST + VST;
  static constexpr int BAR_RES = 2 * KST + 2 * VST;
  static constexpr int BAR_S = BAR_RES + 1;  // two: S is double buffered
  static constexpr int BAR_DP = BAR_S + 2;
  static constexpr int BAR_DS = BAR_DP + 1;
  static constexpr int BAR_DONE = BAR_DS + 1;
  static constexpr int NUM_BARS = BAR_DONE + 1;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
  static_assert(SMEM_BYTES <= 232448, "dq kernel shared memory");
};

template <int D, bool BF16, bool BIAS>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    dq_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                 const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                 const KernelParams p, const BwdArgs a) {
  using C = Cfg<D>;
  using Q = DqCfg<D>;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + Q::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + Q::OFF_MISC);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // ---- work: 128 query rows of one (b, query head); the key tiles they see
  // causal: the last query tiles see the most keys, so they start first
  int rank, bh;
  cta_order(rank, bh);
  const int qt = p.causal ? static_cast<int>(gridDim.x) - 1 - rank : rank;
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int bhk = b * p.Hkv + hq / p.group;
  const int q0 = qt * BR;
  int lim = p.Sk;
  if (p.padding) {
    const int L = __ldg(p.kv_lens + b);
    lim = L < 0 ? 0 : (L > p.Sk ? p.Sk : L);
  }
  const int diag = p.Sk - p.Sq;
  int hi = lim;
  if (p.causal) hi = min(hi, min(q0 + BR - 1, p.Sq - 1) + diag + 1);
  const int N = hi > 0 ? (hi + BR - 1) / BR : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < Q::KST; ++s) {
      mbar_init(bar(Q::BAR_KFULL + s), 1);
      mbar_init(bar(Q::BAR_KEMPTY + s), 1);
    }
    for (int s = 0; s < Q::VST; ++s) {
      mbar_init(bar(Q::BAR_VFULL + s), 1);
      mbar_init(bar(Q::BAR_VEMPTY + s), 1);
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
    if (p.status) atomicOr(p.status, STATUS_TIMEOUT);
  };

  if (warp >= 8) {
    setmaxnreg_dec<REG_OTHER>();
    if (warp == WARP_TMA && lane == 0 && N > 0) {
      // ------------------------------------------------------------ producer
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar(Q::BAR_RES), 2 * C::TILE_BYTES);
      for (int c = 0; c < C::NCHUNK; ++c) {
        tma_load_3d(sb + c * C::CHUNK_BYTES, &tm_q, bar(Q::BAR_RES), c * C::BOX_D, q0, bh);
        tma_load_3d(sb + C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_do, bar(Q::BAR_RES), c * C::BOX_D, q0, bh);
      }
      int nk = 0, nv = 0;  // K and V tiles issued
      bool ok = true;
      for (int j = 0; j < N && ok; ++j) {
        const int ks = j % Q::KST, vs = j % Q::VST;
        if (!mbar_wait(bar(Q::BAR_KEMPTY + ks), ((j / Q::KST) & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(Q::BAR_KFULL + ks), C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sb + Q::OFF_K + ks * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_k, bar(Q::BAR_KFULL + ks),
                      c * C::BOX_D, j * BR, bhk);
        ++nk;
        if (!mbar_wait(bar(Q::BAR_VEMPTY + vs), ((j / Q::VST) & 1) ^ 1)) { ok = false; break; }
        mbar_arrive_expect_tx(bar(Q::BAR_VFULL + vs), C::TILE_BYTES);
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_load_3d(sb + Q::OFF_V + vs * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_v, bar(Q::BAR_VFULL + vs),
                      c * C::BOX_D, j * BR, bhk);
        ++nv;
      }
      if (!ok) fail();
      // drain: every copy issued has landed before the CTA exits
      for (int s = 0; s < Q::KST && s < nk; ++s)
        if (!mbar_wait(bar(Q::BAR_KFULL + s), (((nk - s + Q::KST - 1) / Q::KST) - 1) & 1)) fail();
      for (int s = 0; s < Q::VST && s < nv; ++s)
        if (!mbar_wait(bar(Q::BAR_VFULL + s), (((nv - s + Q::VST - 1) / Q::VST) - 1) & 1)) fail();
      if (!mbar_wait(bar(Q::BAR_RES), 0)) fail();
    } else if (warp == WARP_MMA) {
      // ------------------------------------------------------------ MMA issuer
      // (the whole warp waits; one elected lane issues the MMAs and commits)
      constexpr uint32_t idesc_s = make_idesc_f16(BF16, BR, BR, false);  // M = rows, N = keys
      constexpr uint32_t idesc_o = make_idesc_f16(BF16, BR, D, true);    // N = D, B MN-major
      constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
      constexpr uint32_t RSTEP16 = (16 * 128) >> 4;
      const uint64_t q_a = smem_desc(sb, 16, C::SBO, C::LAYOUT);
      const uint64_t do_a = smem_desc(sb + C::TILE_BYTES, 16, C::SBO, C::LAYOUT);
      const uint64_t k_b = smem_desc(sb + Q::OFF_K, 16, C::SBO, C::LAYOUT);
      const uint64_t k_mn = smem_desc(sb + Q::OFF_K, C::CHUNK_BYTES, C::SBO, C::LAYOUT);
      const uint64_t v_b = smem_desc(sb + Q::OFF_V, 16, C::SBO, C::LAYOUT);
      bool ok = true;
      auto issue_s = [&](int j) {  // S = Q K_j^T into buffer j & 1
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
      auto issue_dp = [&](int j) {  // dP = dO V_j^T
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
          // dQ += dS K_j   (dS: 16-bit in dP's columns; K_j as an MN-major operand)
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
      if (elect_one()) umma_commit(bar(Q::BAR_DONE));
      __syncwarp();
      if (!warp_wait(bar(Q::BAR_DONE), 0) && lane == 0) fail();
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- elementwise
    setmaxnreg_inc<REG_EW>();
    const int half = warp >> 2;                      // key columns [64 half, +64)
    const int row = ((warp & 3) << 5) + lane;        // query row = TMEM lane
    const int i = q0 + row;
    const bool row_ok = i < p.Sq;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const size_t ri = static_cast<size_t>(bh) * p.Sq + i;
    const int64_t nrows = static_cast<int64_t>(p.B) * p.Hq * p.Sq;  // extent for the checked build
    const bool stat_ok = row_ok && in_bounds(p.status, static_cast<int64_t>(ri), nrows);
    const float l2 = stat_ok ? __ldg(a.lse2 + ri) : -INFINITY;
    const float dsi = stat_ok ? __ldg(a.dsum + ri) : 0.f;
    const bool live = row_ok && l2 != -INFINITY;
    const float l2f = live ? l2 : INFINITY;  // interior tiles: exp2(s - inf) = 0 for a dead row
    const int causal_lim = p.causal ? i + diag : 0x7fffffff;
    const float sc = p.scale_log2;
    const float* brow = nullptr;
    if constexpr (BIAS) {
      if (row_ok) {
        const int bb = p.bias_b == 1 ? 0 : b;
        const int bhb = p.bias_h == 1 ? 0 : hq;
        brow = p.bias + ((static_cast<size_t>(bb) * p.bias_h + bhb) * p.Sq + i) * static_cast<size_t>(p.Sk);
      }
    }
    bool failed = false;
    for (int j = 0; j < N; ++j) {
      float x[64];
      const bool ok = mbar_wait(bar(Q::BAR_S + (j & 1)), (j >> 1) & 1);
      if (__any_sync(0xffffffffu, !ok)) { failed = true; break; }
      tc_fence_after();
      tmem_ld64<BF16>(tmem + lane_off + BR * (j & 1) + 64 * half, x);
      const int kc0 = j * BR + 64 * half;
      // every key of this warp's 64 visible to every row of the block: no
      // per-element mask (a dead row has lse2 = +inf here, so its p is 0)
      if (!BIAS && kc0 + 63 < lim && (!p.causal || kc0 + 63 <= q0 + diag)) {
#pragma unroll
        for (int c = 0; c < 64; ++c) x[c] = fast_exp2(x[c] * sc - l2f);
      } else
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const int key = kc0 + c;
        const bool vis = live && key < lim && key <= causal_lim;
        float s2 = x[c] * sc - l2;
        if constexpr (BIAS) {
          if (vis && in_bounds(p.status, (brow - p.bias) + key,
                               static_cast<int64_t>(p.bias_b) * p.bias_h * p.Sq * p.Sk))
            s2 = fmaf(__ldg(brow + key), LOG2E, s2);
        }
        x[c] = vis ? fast_exp2(s2) : 0.f;
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
        const bool row_in = row_ok && range_in_bounds(p.status, static_cast<int64_t>(ri) * D + half * (D / 2), D / 2,
                                                      nrows * D);
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


// Host side. Q/dO viewed as [B*Hq, Sq, D], K/V as [B*Hkv, Sk, D]; boxes of
// 64 columns x 128 rows, 128-byte swizzle; rows past S are zero-filled.
template <int D>
static CUresult encode_bwd(EncodeTiledFn enc, CUtensorMap* m, bool bf16, const void* ptr, uint64_t S,
                           uint64_t BH) {
  const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(D), S, BH};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(D) * 2, S * D * 2};
  const cuuint32_t box[3] = {64u, static_cast<cuuint32_t>(BR), 1u};
  const cuuint32_t estride[3] = {1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void*>(ptr),
             gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int D, bool BF16, bool BIAS>
cudaError_t launch_bwd_tc_instance(EncodeTiledFn enc, const void* q, const void* k, const void* v,
                                   const void* dout, const KernelParams& p, const BwdArgs& a,
                                   cudaStream_t stream) {
  CUtensorMap tq, tdo, tk, tv;
  const uint64_t bhq = static_cast<uint64_t>(p.B) * p.Hq, bhk = static_cast<uint64_t>(p.B) * p.Hkv;
  if (encode_bwd<D>(enc, &tq, BF16, q, p.Sq, bhq) != CUDA_SUCCESS ||
      encode_bwd<D>(enc, &tdo, BF16, dout, p.Sq, bhq) != CUDA_SUCCESS ||
      encode_bwd<D>(enc, &tk, BF16, k, p.Sk, bhk) != CUDA_SUCCESS ||
      encode_bwd<D>(enc, &tv, BF16, v, p.Sk, bhk) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  auto kv = dkdv_tc_kernel<D, BF16, BIAS>;
  auto kq = dq_tc_kernel<D, BF16, BIAS>;
  constexpr int smem_kv = Cfg<D>::SMEM_BYTES;
  constexpr int smem_q = DqCfg<D>::SMEM_BYTES;
  // the shared-memory opt-in is per device and per kernel: set it once
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = p.device >= 0 && p.device < 64 ? 1ull << p.device : 0ull;
  if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kv, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_kv);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kq, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_q);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const unsigned nkb = static_cast<unsigned>((p.Sk + BR - 1) / BR);
  const unsigned nqt = static_cast<unsigned>((p.Sq + BR - 1) / BR);
  if (nkb > 0 && bhk > 0)
    kv<<<dim3(nkb, static_cast<unsigned>(bhk)), NUM_THREADS, smem_kv, stream>>>(tq, tdo, tk, tv, p, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  if (nqt > 0 && bhq > 0)
    kq<<<dim3(nqt, static_cast<unsigned>(bhq)), NUM_THREADS, smem_q, stream>>>(tq, tdo, tk, tv, p, a);
  return cudaGetLastError();
}

}  // namespace bwdtc
}  // namespace attn
