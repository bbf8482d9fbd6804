// attn_tc.cuh - exact attention forward on the 5th-generation tensor cores
// (tcgen05) of sm_103a, F16/BF16 inputs, fp32 statistics and accumulation.
//
// Algorithm: the tiled, single-pass exact attention that the FlashAttention
// paper describes (cited by "HOF cognitive Flash Attention in Rust", sections
// 2 and 4, as computing the same exact result as the dense kernel without the
// n x n score matrix in HBM): for each query tile, stream K/V tiles, keep a
// running row maximum m and row sum l, rescale the output accumulator when m
// grows, and divide by l at the end. The scores never leave the SM.
//
// One CTA owns NQ = 2 query tiles of BM = 128 rows of one (batch, query head)
// and streams the key/value tiles they need once for both. 384 threads:
//   warpgroup 0, 1  softmax for query tile 0 / 1: thread r owns TMEM lane r =
//                   query row r. It pulls its 128 scores of the tile with
//                   tcgen05.ld, applies scale, bias and mask, keeps m and l
//                   in registers, writes P (16-bit) back into tensor memory,
//                   rescales its O row when needed, and in the end normalises
//                   O, stages it in shared memory and stores it with TMA.
//   warp 8          TMA producer: Q tiles once, then K_j, V_j in order into a
//                   ring of STAGES shared-memory slots (full/empty mbarriers).
//   warp 9          MMA issuer (the whole warp waits, one elected lane issues);
//                   allocates the 512 TMEM columns.
//   warps 10, 11    idle (they complete the third warpgroup, whose registers
//                   are handed to the softmax warpgroups with setmaxnreg).
// MMA issue order per K/V tile j:  S_0(j), PV_1(j-1), S_1(j), PV_0(j), with
// S_t = Q_t K_j^T (SS form) and O_t += P_t V_j (P_t read from tensor memory,
// TS form). Softmax t therefore has two MMA slots (the other tile's PV and S)
// to turn S_t into P_t before the tensor core needs it.
// Tensor-memory map (fp32 columns): S_0 [0,128), S_1 [128,256), O_0 at 256,
// O_1 at 256 + D; P_t (16-bit pairs) aliases columns [64,128) of S_t. The MMA
// that next overwrites S_t is issued after the PV MMA that reads P_t, and
// tcgen05 MMAs from one thread execute in issue order.
// Rescaling is lazy: a row's reference maximum moves only when the tile max
// exceeds it by more than 2^8; probabilities are then at most 256, well inside
// the 16-bit and fp32 ranges, and the final O / l uses the same reference, so
// the result is unchanged.
// Every mbarrier wait is bounded; on expiry the CTA records STATUS_TIMEOUT in
// the device status word, drains its own copies and MMAs, frees TMEM and exits.
// Split-KV: with num_splits > 1 the grid has one CTA per (work item, split);
// a CTA runs the key tiles of its split only (tile counters stay local to the
// split, key positions absolute) and writes its unnormalised O rows with their
// (m, l) to the workspace instead of O; launch_split_merge combines them. With
// one split the epilogue writes O, and with EPI_O_LSE also the row log-sum-exp
// (a separate instance: the extra store costs the O-only kernel registers).
#pragma once

#include <atomic>

#include "params.h"
#include "ptx.cuh"

namespace attn {
namespace tc {

constexpr int BM = 128;           // query rows per Q tile = TMEM lanes
constexpr int BN = 128;           // keys per K/V tile
constexpr int NQ = 2;             // Q tiles per CTA
constexpr int NUM_THREADS = 384;  // 2 softmax warpgroups + producer/MMA warpgroup
constexpr int WARP_TMA = 8;
constexpr int WARP_MMA = 9;
constexpr int TMEM_COLS = 512;
constexpr int REG_SOFTMAX = 200;  // 2*128*200 + 128*96 <= 384 * 168 (launch allocation)
constexpr int REG_OTHER = 96;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_LOG2 = 8.0f;  // lazy-rescale threshold (log2 units)
constexpr int HEAD_GROUP = 16;        // heads scheduled together so their K/V stay in L2
constexpr int BIAS_CHUNK = 32;                     // keys per staged bias chunk
constexpr int BIAS_SLOTS = BN / BIAS_CHUNK;        // ring slots per query tile (one K/V tile)
constexpr int BIAS_SLOT_BYTES = BM * BIAS_CHUNK * 4;  // 16 KB, 128-byte rows

template <int D, int BMODE = BIAS_NONE>
struct Cfg {
  static_assert(D == 32 || D == 64 || D == 128, "compiled head dims are 32, 64, 128");
  static_assert(BMODE != BIAS_STAGED || D <= 64, "the staged bias ring fits for D <= 64");
  static constexpr int SWIZZLE = D >= 64 ? 128 : 64;  // bytes per swizzled smem row
  static constexpr int BOX_D = SWIZZLE / 2;           // 16-bit elements per TMA box row
  static constexpr int NCHUNK = D / BOX_D;            // boxes per tile along D
  static constexpr int ROW_BYTES = SWIZZLE;
  static constexpr int CHUNK_BYTES = BN * ROW_BYTES;  // one box: 128 rows
  static constexpr int TILE_BYTES = NCHUNK * CHUNK_BYTES;
  static constexpr int STAGES =
      BMODE == BIAS_STAGED ? (D == 64 ? 4 : 6) : (D == 128 ? 4 : (D == 64 ? 8 : 12));
  static constexpr uint32_t LAYOUT = SWIZZLE == 128 ? 2u : 4u;  // UMMA swizzle code
  static constexpr int SBO = 8 * ROW_BYTES;                      // 8-row group stride
  static constexpr int KSTEPS_QK = D / 16;
  static constexpr int KSTEPS_PER_CHUNK = BOX_D / 16;
  static constexpr int KSTEPS_PV = BN / 16;
  static constexpr int COL_P = 64;  // P_t at S_t + 64 (16-bit pairs, 64 columns)
  static constexpr int OFF_KV = NQ * TILE_BYTES;
  static constexpr int OFF_BIAS = OFF_KV + STAGES * TILE_BYTES;
  static constexpr int BIAS_RING_BYTES = BMODE == BIAS_STAGED ? NQ * BIAS_SLOTS * BIAS_SLOT_BYTES : 0;
  static constexpr int OFF_BAR = OFF_BIAS + BIAS_RING_BYTES;
  static constexpr int NUM_BIAS_BARS = BMODE == BIAS_STAGED ? 2 * NQ * BIAS_SLOTS : 0;
  static constexpr int NUM_BARS = 2 * STAGES + 4 * NQ + 1 + NUM_BIAS_BARS;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int SMEM_USED = OFF_MISC + 16;
  // +1024 for aligning the dynamic window; at least 120 KB so that one CTA
  // (which takes all 512 TMEM columns) is resident per SM.
  static constexpr int SMEM_BYTES =
      (SMEM_USED + 1024) > 120 * 1024 ? (SMEM_USED + 1024) : 120 * 1024;
  static constexpr int BAR_FULL = 0;
  static constexpr int BAR_EMPTY = STAGES;
  static constexpr int BAR_Q = 2 * STAGES;
  static constexpr int BAR_S = BAR_Q + NQ;
  static constexpr int BAR_P = BAR_S + NQ;
  static constexpr int BAR_O = BAR_P + NQ;
  static constexpr int BAR_DONE = BAR_O + NQ;
  static constexpr int BAR_BFULL = BAR_DONE + 1;                  // bias slot loaded
  static constexpr int BAR_BEMPTY = BAR_BFULL + NQ * BIAS_SLOTS;  // bias slot read by softmax
};

// Per-CTA work description, computed identically by every thread.
struct Work {
  int b, hq, bh, bhk, q0;
  int key_limit;   // keys >= key_limit are padding (<= Sk)
  int diag;        // Sk - Sq: causal offset (bottom-right alignment)
  int n[NQ];       // K/V tiles Q tile t needs (0: no visible key at all)
  int nfull[NQ];   // leading K/V tiles of Q tile t with no masked element
  int nmax;
  int j0;          // first K/V tile of this CTA's split (tile indices above are relative)
};

// Linear CTA index -> (head, query block). Heads are taken HEAD_GROUP at a
// time; inside a group the query blocks of all its heads are interleaved,
// heaviest causal block first, so the K/V of the heads in flight stay in L2
// and the long blocks start before the short ones.
// With split-KV (SPLIT) the splits of one work item are adjacent CTAs.
template <bool SPLIT>
__device__ __forceinline__ Work make_work(const KernelParams& p) {
  Work w;
  const int qblocks = (p.Sq + NQ * BM - 1) / (NQ * BM);
  const int bhq = p.B * p.Hq;
  const int per_group = qblocks * HEAD_GROUP;
  const int item = SPLIT ? static_cast<int>(blockIdx.x) / p.num_splits : static_cast<int>(blockIdx.x);
  const int split = SPLIT ? static_cast<int>(blockIdx.x) - item * p.num_splits : 0;
  const int g = item / per_group;
  const int within = item - g * per_group;
  const int hg = min(HEAD_GROUP, bhq - g * HEAD_GROUP);
  const int rank = within / hg;
  w.bh = g * HEAD_GROUP + (within - rank * hg);
  const int qb = p.causal ? (qblocks - 1 - rank) : rank;
  w.b = w.bh / p.Hq;
  w.hq = w.bh - w.b * p.Hq;
  w.bhk = w.b * p.Hkv + w.hq / p.group;
  w.q0 = qb * (NQ * BM);
  w.diag = p.Sk - p.Sq;
  int lim = p.Sk;
  if (p.padding) {
    int L = __ldg(p.kv_lens + w.b);
    lim = L < 0 ? 0 : (L > p.Sk ? p.Sk : L);
  }
  w.key_limit = lim;
  w.nmax = 0;
#pragma unroll
  for (int t = 0; t < NQ; ++t) {
    const int r0 = w.q0 + t * BM;
    w.n[t] = 0;
    w.nfull[t] = 0;
    if (r0 < p.Sq) {
      const int rlast = min(r0 + BM - 1, p.Sq - 1);
      int hi = lim;   // keys [0, hi) are visible to some row of the tile
      int lo = lim;   // keys [0, lo) are visible to every row of the tile
      if (p.causal) {
        hi = min(hi, rlast + w.diag + 1);
        lo = min(lo, r0 + w.diag + 1);
      }
      w.n[t] = hi > 0 ? (hi + BN - 1) / BN : 0;
      w.nfull[t] = lo > 0 ? lo / BN : 0;
    }
    w.nmax = max(w.nmax, w.n[t]);
  }
  w.j0 = 0;
  if constexpr (SPLIT) {
    // balanced contiguous runs of the item's tiles [0, nmax)
    const int jlo = static_cast<int>(static_cast<int64_t>(split) * w.nmax / p.num_splits);
    const int jhi = static_cast<int>(static_cast<int64_t>(split + 1) * w.nmax / p.num_splits);
#pragma unroll
    for (int t = 0; t < NQ; ++t) {
      w.n[t] = max(0, min(jhi, w.n[t]) - jlo);
      w.nfull[t] = max(0, w.nfull[t] - jlo);
    }
    w.j0 = jlo;
    w.nmax = jhi - jlo;
  }
  return w;
}

template <int D, bool BF16, int BMODE, int EPI>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    attn_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_q,
                       const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v,
                       const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_b, const KernelParams p) {
  using C = Cfg<D, BMODE>;
  constexpr bool BIAS = BMODE != BIAS_NONE;
  constexpr bool SPLIT = EPI == EPI_PARTIAL;
  extern __shared__ uint8_t smem_dyn[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~static_cast<uintptr_t>(1023));
  const uint32_t sb = smem_u32(smem);
  auto bar = [&](int i) -> uint32_t { return sb + C::OFF_BAR + 8 * i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::OFF_MISC);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const Work w = make_work<SPLIT>(p);

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
    if constexpr (BMODE == BIAS_STAGED) {
      for (int i = 0; i < NQ * BIAS_SLOTS; ++i) {
        mbar_init(bar(C::BAR_BFULL + i), 1);
        mbar_init(bar(C::BAR_BEMPTY + i), BM);
      }
    }
    *abort_flag = 0;
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
    *abort_flag = 1;
    if (p.status) atomicOr(p.status, STATUS_TIMEOUT);
  };

  if (warp >= 2 * 4) {
    setmaxnreg_dec<REG_OTHER>();
    if (warp == WARP_TMA) {
      // -------------------------------------------------------------- producer
      if (lane == 0) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        tma_prefetch_desc(&tm_v);
        tma_prefetch_desc(&tm_o);
        for (int t = 0; t < NQ; ++t) {
          if (w.n[t] == 0) continue;
          mbar_arrive_expect_tx(bar(C::BAR_Q + t), C::TILE_BYTES);
          for (int c = 0; c < C::NCHUNK; ++c)
            tma_load_3d(sb + t * C::TILE_BYTES + c * C::CHUNK_BYTES, &tm_q, bar(C::BAR_Q + t),
                        c * C::BOX_D, w.q0 + t * BM, w.bh);
        }
        int it = 0;  // ring position: K_j at 2j, V_j at 2j + 1
        for (int j = 0; j < w.nmax && !*abort_flag; ++j) {
          for (int kv = 0; kv < 2; ++kv, ++it) {
            const int s = it % C::STAGES;
            const uint32_t ph = (it / C::STAGES) & 1;
            if (!mbar_wait(bar(C::BAR_EMPTY + s), ph ^ 1)) {
              fail();
              break;
            }
            mbar_arrive_expect_tx(bar(C::BAR_FULL + s), C::TILE_BYTES);
            const CUtensorMap* m = kv == 0 ? &tm_k : &tm_v;
            for (int c = 0; c < C::NCHUNK; ++c)
              tma_load_3d(sb + C::OFF_KV + s * C::TILE_BYTES + c * C::CHUNK_BYTES, m,
                          bar(C::BAR_FULL + s), c * C::BOX_D, (w.j0 + j) * BN, w.bhk);
          }
        }
        // Drain: every copy this thread issued has landed before the CTA exits.
        for (int s = 0; s < C::STAGES && s < it; ++s) {
          const int fills = (it - s + C::STAGES - 1) / C::STAGES;
          if (!mbar_wait(bar(C::BAR_FULL + s), (fills - 1) & 1)) fail();
        }
        for (int t = 0; t < NQ; ++t)
          if (w.n[t] > 0 && !mbar_wait(bar(C::BAR_Q + t), 0)) fail();
      }
      __syncwarp();
    } else if (BMODE == BIAS_STAGED && warp == WARP_MMA + 1) {
      // -------------------------------------------------------------- bias producer
      // Chunk c of key tile j for query tile t: bias rows [r0, r0+128), keys
      // [128j + 32c, +32), into ring slot (count_t mod 4) of tile t's ring.
      if (lane == 0) {
        const int bz = (p.bias_b == 1 ? 0 : w.b) * p.bias_h + (p.bias_h == 1 ? 0 : w.hq);
        int cnt[NQ] = {0, 0};
        bool ok = true;
        for (int j = 0; j < w.nmax && ok; ++j) {
          for (int t = 0; t < NQ && ok; ++t) {
            if (j >= w.n[t]) continue;
            for (int c = 0; c < BIAS_SLOTS; ++c, ++cnt[t]) {
              if (*abort_flag) { ok = false; break; }
              const int slot = t * BIAS_SLOTS + cnt[t] % BIAS_SLOTS;
              if (!mbar_wait(bar(C::BAR_BEMPTY + slot), ((cnt[t] / BIAS_SLOTS) & 1) ^ 1)) {
                ok = false;
                break;
              }
              mbar_arrive_expect_tx(bar(C::BAR_BFULL + slot), BIAS_SLOT_BYTES);
              tma_load_3d(sb + C::OFF_BIAS + slot * BIAS_SLOT_BYTES, &tm_b, bar(C::BAR_BFULL + slot),
                          (w.j0 + j) * BN + c * BIAS_CHUNK, w.q0 + t * BM, bz);
            }
          }
        }
        if (!ok) fail();
        // Drain: every bias copy issued has landed before the CTA exits.
        for (int t = 0; t < NQ; ++t)
          for (int s2 = 0; s2 < BIAS_SLOTS && s2 < cnt[t]; ++s2) {
            const int fills = (cnt[t] - s2 + BIAS_SLOTS - 1) / BIAS_SLOTS;
            if (!mbar_wait(bar(C::BAR_BFULL + t * BIAS_SLOTS + s2), (fills - 1) & 1)) fail();
          }
      }
      __syncwarp();
    } else if (warp == WARP_MMA) {
      // -------------------------------------------------------------- MMA issuer
      // The whole warp runs the loop and takes every wait; one elected lane
      // issues the MMAs and commits.
      {
        constexpr uint32_t idesc_qk = make_idesc_f16(BF16, BM, BN, false);
        constexpr uint32_t idesc_pv = make_idesc_f16(BF16, BM, D, true);
        constexpr int ST = C::STAGES;
        const int n0 = w.n[0], n1 = w.n[1], nmax = w.nmax;
        bool ok = true;
        for (int t = 0; t < NQ && ok; ++t)
          if (w.n[t] > 0 && !warp_wait(bar(C::BAR_Q + t), 0)) ok = false;

        // Descriptors of the first K-step of Q_0, of ring stage 0 as a K tile
        // (K-major) and as a V tile (MN-major). Other tiles, stages and K-steps
        // only move the start address, a plain addition to the low field.
        const uint64_t dq0 = smem_desc(sb, 16, C::SBO, C::LAYOUT);
        const uint64_t dk0 = smem_desc(sb + C::OFF_KV, 16, C::SBO, C::LAYOUT);
        const uint64_t dv0 = smem_desc(sb + C::OFF_KV, C::CHUNK_BYTES, C::SBO, C::LAYOUT);
        constexpr uint32_t TILE16 = C::TILE_BYTES >> 4;
        constexpr uint32_t CHUNK16 = C::CHUNK_BYTES >> 4;
        constexpr uint32_t VSTEP16 = (16 * C::ROW_BYTES) >> 4;  // 16 keys of V
        auto kstep = [](int k) -> uint32_t {
          return (k / C::KSTEPS_PER_CHUNK) * CHUNK16 + (k % C::KSTEPS_PER_CHUNK) * 2;
        };
        auto wait_full = [&](int idx) {
          return warp_wait(bar(C::BAR_FULL + idx % ST), (idx / ST) & 1);
        };
        // S_t = Q_t K_j^T
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
        // O_t += P_t V_j (P_t of tile j is in tensor memory)
        auto issue_pv = [&](int t, int j) {
          const uint64_t b = dv0 + ((2 * j + 1) % ST) * TILE16;
          const uint32_t d = tmem + 256 + t * D;
          const uint32_t a = tmem + t * BN + C::COL_P;
          if (elect_one()) {
            umma_ts(d, a, b, idesc_pv, j > 0 ? 1u : 0u);
#pragma unroll
            for (int k = 1; k < C::KSTEPS_PV; ++k) umma_ts(d, a + k * 8, b + k * VSTEP16, idesc_pv, 1u);
            if (j == w.n[t] - 1) umma_commit(bar(C::BAR_O + t));
          }
          __syncwarp();
        };

        // No abort-flag read in this loop: a shared-memory load between MMA
        // groups stalls the MMA stream (measured: 9% on the causal S=4096
        // D=128 workload). If another role fails, the next bounded wait here
        // expires instead and this warp takes the same exit.
        for (int j = 0; j <= nmax && ok; ++j) {
          if (j < nmax) {
            if (!wait_full(2 * j)) { ok = false; break; }  // K_j
            tc_fence_after();
            if (j < n0) issue_s(0, j);
          }
          if (j >= 1 && j - 1 < n1) {
            // V_{j-1} was already waited for by PV_0(j-1) unless tile 0 skipped it
            if (j - 1 >= n0 && !wait_full(2 * (j - 1) + 1)) { ok = false; break; }
            if (!warp_wait(bar(C::BAR_P + 1), (j - 1) & 1)) { ok = false; break; }
            tc_fence_after();
            issue_pv(1, j - 1);
          }
          if (j >= 1) {
            if (elect_one()) umma_commit(bar(C::BAR_EMPTY + (2 * (j - 1) + 1) % ST));  // V_{j-1} free
            __syncwarp();
          }
          if (j < nmax) {
            if (j < n1) issue_s(1, j);
            if (elect_one()) umma_commit(bar(C::BAR_EMPTY + (2 * j) % ST));  // K_j free
            __syncwarp();
            if (j < n0) {
              if (!wait_full(2 * j + 1) || !warp_wait(bar(C::BAR_P + 0), j & 1)) { ok = false; break; }
              tc_fence_after();
              issue_pv(0, j);
            }
          }
        }
        if (!ok && lane == 0) fail();
        // Drain: all MMAs issued above have completed before TMEM is freed.
        if (elect_one()) umma_commit(bar(C::BAR_DONE));
        __syncwarp();
        if (!warp_wait(bar(C::BAR_DONE), 0) && lane == 0) fail();
      }
      __syncwarp();
    }
  } else {
    // ---------------------------------------------------------------- softmax
    setmaxnreg_inc<REG_SOFTMAX>();
    const int t = warp >> 2;                   // query tile of this warpgroup
    const int row = ((warp & 3) << 5) + lane;  // TMEM lane = row within the tile
    const int r0 = w.q0 + t * BM;
    const int row_g = r0 + row;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) << 5) << 16;
    const uint32_t tS = tmem + lane_off + t * BN;
    const uint32_t tP = tS + C::COL_P;
    const uint32_t tO = tmem + lane_off + 256 + t * D;
    const int n_t = w.n[t];
    const int nfull_t = w.nfull[t];
    const float sc = p.scale_log2;

    const float* brow = nullptr;
    if constexpr (BIAS) {
      if (row_g < p.Sq) {
        const int bb = p.bias_b == 1 ? 0 : w.b;
        const int bh = p.bias_h == 1 ? 0 : w.hq;
        brow = p.bias + ((static_cast<size_t>(bb) * p.bias_h + bh) * p.Sq + row_g) *
                            static_cast<size_t>(p.Sk);
      }
    }
    const int causal_lim = p.causal ? row_g + w.diag : 0x7fffffff;  // last visible key
    const int key_lim = w.key_limit;

    bool bias_failed = false;  // a staged bias chunk never arrived
    float m_run = -INFINITY;  // reference max of the row (log2 domain)
    float l_run = 0.f;        // sum of 2^(s - m_run) over the keys seen
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
      if constexpr (BMODE == BIAS_STAGED) {
        // bias chunks from the shared-memory ring (128-byte swizzled rows)
        const uint8_t* ring = smem + C::OFF_BIAS + t * BIAS_SLOTS * BIAS_SLOT_BYTES;
#pragma unroll
        for (int c = 0; c < BIAS_SLOTS; ++c) {
          const int cnt = j * BIAS_SLOTS + c;
          const int slot = cnt % BIAS_SLOTS;
          if (!mbar_wait(bar(C::BAR_BFULL + t * BIAS_SLOTS + slot), (cnt / BIAS_SLOTS) & 1))
            bias_failed = true;
          const uint8_t* rowp = ring + slot * BIAS_SLOT_BYTES + row * 128;
          float bv[32];
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const float4 b4 = *reinterpret_cast<const float4*>(rowp + ((q ^ (row & 7)) << 4));
            bv[4 * q] = b4.x; bv[4 * q + 1] = b4.y; bv[4 * q + 2] = b4.z; bv[4 * q + 3] = b4.w;
          }
          mbar_arrive(bar(C::BAR_BEMPTY + t * BIAS_SLOTS + slot));
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float2 x = ffma2(make_float2(s[32 * c + i], s[32 * c + i + 1]), make_float2(sc, sc),
                                   fmul2(make_float2(bv[i], bv[i + 1]), make_float2(LOG2E, LOG2E)));
            s[32 * c + i] = x.x;
            s[32 * c + i + 1] = x.y;
          }
        }
      } else if constexpr (BIAS) {
        // scores -> log2 domain with the bias folded in
        if (brow != nullptr) {
          const float* bp = brow + key0;
          const int64_t nbias = static_cast<int64_t>(p.bias_b) * p.bias_h * p.Sq * p.Sk;  // checked build
          if (j < nfull_t && p.bias_vec4 && range_in_bounds(p.status, bp - p.bias, 128, nbias)) {
#pragma unroll
            for (int i = 0; i < 128; i += 4) {
              const float4 b4 = __ldg(reinterpret_cast<const float4*>(bp + i));
              const float2 lo = ffma2(make_float2(s[i], s[i + 1]), make_float2(sc, sc),
                                      fmul2(make_float2(b4.x, b4.y), make_float2(LOG2E, LOG2E)));
              const float2 hi = ffma2(make_float2(s[i + 2], s[i + 3]), make_float2(sc, sc),
                                      fmul2(make_float2(b4.z, b4.w), make_float2(LOG2E, LOG2E)));
              s[i] = lo.x; s[i + 1] = lo.y; s[i + 2] = hi.x; s[i + 3] = hi.y;
            }
          } else {
#pragma unroll
            for (int i = 0; i < 128; ++i) {
              const float bv =
                  (key0 + i < key_lim && in_bounds(p.status, (bp - p.bias) + i, nbias)) ? __ldg(bp + i) : 0.f;
              s[i] = fmaf(s[i], sc, bv * LOG2E);
            }
          }
        } else {
#pragma unroll
          for (int i = 0; i < 128; i += 2) {
            const float2 x = fmul2(make_float2(s[i], s[i + 1]), make_float2(sc, sc));
            s[i] = x.x; s[i + 1] = x.y;
          }
        }
      }
      if (j >= nfull_t) {
#pragma unroll
        for (int i = 0; i < 128; ++i) {
          const int key = key0 + i;
          if (key >= key_lim || key > causal_lim) s[i] = -INFINITY;
        }
      }
      // row max: four independent chains of 3-input max
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
      const float mx = fmax3(c0, c1, fmaxf(c2, c3));
      const float m_tile = BIAS ? mx : mx * sc;
      // lazy rescale: move the reference max only when it grew by > 2^8
      const bool need = m_tile > m_run + RESCALE_LOG2;
      float alpha = 1.f;
      if (need) {
        alpha = fast_exp2(m_run - m_tile);  // 0 when m_run is -inf
        m_run = m_tile;
        l_run *= alpha;
      }
      const float neg_m = (m_run == -INFINITY) ? 0.f : -m_run;
      float2 sum_a = make_float2(0.f, 0.f), sum_b = make_float2(0.f, 0.f);
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t pk[32];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int i = 64 * h + 2 * c;
          float2 xa, xb;
          if constexpr (BIAS) {
            xa = fadd2(make_float2(s[i], s[i + 1]), make_float2(neg_m, neg_m));
            xb = fadd2(make_float2(s[i + 2], s[i + 3]), make_float2(neg_m, neg_m));
          } else {
            xa = ffma2(make_float2(s[i], s[i + 1]), make_float2(sc, sc), make_float2(neg_m, neg_m));
            xb = ffma2(make_float2(s[i + 2], s[i + 3]), make_float2(sc, sc),
                       make_float2(neg_m, neg_m));
          }
          const float2 pa = make_float2(fast_exp2(xa.x), fast_exp2(xa.y));
          const float2 pb = make_float2(fast_exp2(xb.x), fast_exp2(xb.y));
          sum_a = fadd2(sum_a, pa);
          sum_b = fadd2(sum_b, pb);
          pk[c] = pack2<BF16>(pa.x, pa.y);
          pk[c + 1] = pack2<BF16>(pb.x, pb.y);
        }
        tmem_st32(tP + 32 * h, pk);
      }
      l_run += (sum_a.x + sum_a.y) + (sum_b.x + sum_b.y);
      // O_t was last written by PV of tile j-1, complete before S_t of tile j
      // was signalled; rescale it before PV of tile j is issued.
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
      if (__any_sync(0xffffffffu, bias_failed)) { failed = true; break; }
    }

    // ---------------------------------------------------------------- epilogue
    // Every warp of the warpgroup reaches the named barrier, failed or not, so
    // that a timeout in one warp can never leave the others waiting on it.
    if (SPLIT && r0 < p.Sq) {
      // split partial: unnormalised O row and (m, l), straight to the workspace
      const bool have = n_t > 0;
      if (!failed && have) {
        const bool ok = mbar_wait(bar(C::BAR_O + t), 0);
        if (__any_sync(0xffffffffu, !ok)) failed = true;
      }
      const size_t rr =
          (static_cast<size_t>(blockIdx.x % p.num_splits) * p.B * p.Hq + w.bh) * p.Sq +
          static_cast<size_t>(row_g);
      // bounds-checked build: the partial row lies inside the workspace
      const bool rr_ok = row_g < p.Sq &&
                         in_bounds(p.status, static_cast<int64_t>(rr),
                                   static_cast<int64_t>(p.num_splits) * p.B * p.Hq * p.Sq);
      if (failed) {
        if (lane == 0) fail();
        // m = +inf, l = NaN: the merge makes the row NaN whatever the other
        // parts (or an earlier call's scratch) hold
        if (rr_ok) p.ws_ml[rr] = make_float2(INFINITY, __int_as_float(0x7fc00000));
      } else {
        tc_fence_after();
        float4* wrow = reinterpret_cast<float4*>(p.ws_o + rr * D);
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
          if (rr_ok) {
#pragma unroll
            for (int i = 0; i < 8; ++i)
              wrow[8 * c + i] = make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                            __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
          }
        }
        if (rr_ok) p.ws_ml[rr] = have ? make_float2(m_run, l_run) : make_float2(-INFINITY, 0.f);
      }
    } else if (!SPLIT && r0 < p.Sq) {
      const bool have = n_t > 0;
      if (!failed && have) {
        const bool ok = mbar_wait(bar(C::BAR_O + t), 0);
        if (__any_sync(0xffffffffu, !ok)) failed = true;
      }
      if (failed) {
        if (lane == 0) fail();
      } else {
        tc_fence_after();
        // rows with no visible key have an undefined softmax: NaN
        const float inv = (have && l_run > 0.f) ? 1.f / l_run : __int_as_float(0x7fc00000);
        if (EPI == EPI_O_LSE && row_g < p.Sq &&
            in_bounds(p.status, static_cast<int64_t>(w.bh) * p.Sq + row_g, static_cast<int64_t>(p.B) * p.Hq * p.Sq))
          p.lse[static_cast<size_t>(w.bh) * p.Sq + row_g] =
              (have && l_run > 0.f) ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
        uint8_t* stage = smem + t * C::TILE_BYTES;  // Q_t is dead: reuse it for O_t
        const int swz = C::SWIZZLE == 128 ? (row & 7) : ((row >> 1) & 3);
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
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const float2 x = fmul2(make_float2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])),
                                   make_float2(inv, inv));
            pk[i] = pack2<BF16>(x.x, x.y);
          }
          const int col0 = 32 * c;
          const int box = col0 / C::BOX_D;
          const int ch0 = ((col0 % C::BOX_D) * 2) / 16;
          uint8_t* rowp = stage + box * C::CHUNK_BYTES + row * C::ROW_BYTES;
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int ch = (ch0 + u) ^ swz;
            *reinterpret_cast<uint4*>(rowp + ch * 16) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
          }
        }
        fence_proxy_async_smem();
      }
      named_bar_sync(1 + t, BM);
      if (row == 0 && !*abort_flag) {
        for (int c = 0; c < C::NCHUNK; ++c)
          tma_store_3d(&tm_o, sb + t * C::TILE_BYTES + c * C::CHUNK_BYTES, c * C::BOX_D, r0,
                       w.bh);
        tma_store_commit();
        tma_store_wait_all();
      }
    } else if (failed && lane == 0) {
      fail();
    }
  }

  // ------------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == WARP_MMA) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, TMEM_COLS);
  }
}

// Host side: encode the four 3-D tensor maps and launch. Q/O are viewed as
// [B*Hq, Sq, D] and K/V as [B*Hkv, Sk, D] (x = D innermost), so a box that
// runs past S is zero-filled on load and clipped on store, per head.
template <int D>
static CUresult encode_3d(EncodeTiledFn enc, CUtensorMap* m, bool bf16, const void* ptr,
                          uint64_t S, uint64_t BH) {
  using C = Cfg<D>;
  const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(D), S, BH};
  const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(D) * 2, S * D * 2};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(C::BOX_D), static_cast<cuuint32_t>(BM), 1};
  const cuuint32_t estride[3] = {1, 1, 1};
  return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
             const_cast<void*>(ptr), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
             C::SWIZZLE == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
}

template <int D, bool BF16, int BMODE, int EPI>
cudaError_t launch_tc_instance(EncodeTiledFn enc, const void* q, const void* k, const void* v,
                               void* out, const KernelParams& p, cudaStream_t stream) {
  CUtensorMap tq, tk, tv, to, tb;
  const uint64_t bhq = static_cast<uint64_t>(p.B) * p.Hq, bhk = static_cast<uint64_t>(p.B) * p.Hkv;
  if (encode_3d<D>(enc, &tq, BF16, q, p.Sq, bhq) != CUDA_SUCCESS ||
      encode_3d<D>(enc, &tk, BF16, k, p.Sk, bhk) != CUDA_SUCCESS ||
      encode_3d<D>(enc, &tv, BF16, v, p.Sk, bhk) != CUDA_SUCCESS ||
      encode_3d<D>(enc, &to, BF16, out, p.Sq, bhq) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  tb = tq;  // placeholder unless the bias is staged
  if constexpr (BMODE == BIAS_STAGED) {
    // bias viewed as [bias_b * bias_h, Sq, Sk] fp32; boxes of 32 keys x 128 rows
    const cuuint64_t gdim[3] = {static_cast<cuuint64_t>(p.Sk), static_cast<cuuint64_t>(p.Sq),
                                static_cast<cuuint64_t>(p.bias_b) * p.bias_h};
    const cuuint64_t gstride[2] = {static_cast<cuuint64_t>(p.Sk) * 4,
                                   static_cast<cuuint64_t>(p.Sq) * p.Sk * 4};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(BIAS_CHUNK), static_cast<cuuint32_t>(BM), 1};
    const cuuint32_t estride[3] = {1, 1, 1};
    if (enc(&tb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(p.bias), gdim, gstride, box,
            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cudaErrorInvalidValue;
  }
  auto kern = attn_fwd_tc_kernel<D, BF16, BMODE, EPI>;
  constexpr int smem = Cfg<D, BMODE>::SMEM_BYTES;
  // The shared-memory opt-in is per device and per kernel: set it once.
  static std::atomic<unsigned long long> configured{0};
  const unsigned long long bit = p.device >= 0 && p.device < 64 ? 1ull << p.device : 0ull;
  if (!bit || !(configured.load(std::memory_order_acquire) & bit)) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured.fetch_or(bit, std::memory_order_acq_rel);
  }
  const uint64_t qblocks = (static_cast<uint64_t>(p.Sq) + NQ * BM - 1) / (NQ * BM);
  const uint64_t ctas = bhq * qblocks * static_cast<uint64_t>(p.num_splits);
  if (ctas > 0x7fffffffull) return cudaErrorInvalidConfiguration;
  kern<<<static_cast<unsigned>(ctas), NUM_THREADS, smem, stream>>>(tq, tk, tv, to, tb, p);
  return cudaGetLastError();
}

}  // namespace tc
}  // namespace attn
