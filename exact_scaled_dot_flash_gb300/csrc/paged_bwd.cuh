// paged_bwd.cuh - kernels of the backward over a paged cache (paged attention
// and paged MLA), fp32 FMA arithmetic for every dtype, ordered: no atomics
// in any gradient, one fixed summation order, so repeated calls return the
// same bits.
//
// Source: ruDNN user guide, section 11 (backward of paged attention and
// ordered history gradients): dq for the packed queries and dk, dv in the
// shape of the physical caches, the probabilities recomputed from the forward's
// statistics; an ordered variant reduces the history (cache) gradients
// without atomics, using a workspace that holds row statistics and a reverse
// index from physical pages to the table entries that read them. For MLA the
// latent gradient holds both its key and its value contribution.
//
// With the forward's lse_i and D_i = dout_i . out_i, for every visible (i, j):
//   p_ij = exp(s_ij - lse_i),  dp_ij = dout_i . v_j,  ds_ij = p_ij (dp_ij - D_i)
//   dq_i = scale sum_j ds_ij k_j,  dk_j = scale sum_i ds_ij q_i,  dv_j = sum_i p_ij dout_i
// paged attention: s_ij = scale q_i . k_j, v_j its own cache;
// MLA:             s_ij = scale (q_i . c_j + qp_i . kp_j), k_j = v_j = c_j, so
//                  dc_j = sum_i (p_ij dout_i + scale ds_ij q_i), dkp_j = scale
//                  sum_i ds_ij qp_i, dqp_i = scale sum_j ds_ij kp_j.
//
// Two kernels after the preprocess and the page index:
//  - key-major (dkdv_kernel): a CTA owns up to ROWS key slots of one physical
//    page and key/value head, keeps their rows in registers, and walks the
//    table entries that read the page (ascending), and for each the (query,
//    head) rows of that sequence (ascending) staged through shared memory;
//    slots of a page nobody reads are written as zeros. After the tensor-core
//    kernels it runs only over the index's list of pages whose reader count is
//    not one, its CTAs striding over the list;
//  - query-major (dq_kernel): a CTA owns ROWS (query, head) rows of one
//    sequence and key/value head and streams the sequence's keys, gathered
//    through the page table, through shared memory.
// TPK threads share a row (or key), each owning DK/TPK elements; the dot
// products are reduced with log2(TPK) xor shuffles.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <atomic>

#include "paged_bwd.h"
#include "params.h"
#include "ptx.cuh"
#include "simt.cuh"

namespace attn {
namespace pbwd {

using simt::axpy4;
using simt::dot4;
using simt::load4;
using simt::store4;

constexpr int THREADS = 256;

// DK: width of q, k, v, dout (D, or the latent rank R); PD: positional width
// (MLA only); TPK: threads per row or key.
template <int DK, int PD, int TPK>
struct Cfg {
  static constexpr int G = DK / 4, PG = PD / 4;
  static constexpr int GPT = G / TPK;                // float4 groups of a main vector per thread
  static constexpr int PPT = (PG + TPK - 1) / TPK;   // positional groups per thread (some idle)
  static constexpr int ROWS = THREADS / TPK;         // keys (key-major) or rows (query-major) per CTA
  static constexpr int RT = DK <= 128 ? 32 : 16;     // rows or keys per shared-memory tile
  static_assert(G % TPK == 0 && GPT >= 1, "DK must split evenly over TPK threads");
  static constexpr size_t dkdv_smem(bool) { return static_cast<size_t>(RT) * (2 * G + PG) * 16 + RT * 12; }
  static constexpr size_t dq_smem(bool mla) { return static_cast<size_t>(RT) * ((mla ? 1 : 2) * G + PG) * 16; }
};

template <int TPK>
__device__ __forceinline__ float quad_sum(float x) {
#pragma unroll
  for (int o = 1; o < TPK; o <<= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
  return x;
}

__device__ __forceinline__ int keys_of(const PagedParams& pp, int s) {
  const int64_t cap = static_cast<int64_t>(pp.max_pages) * pp.page_size;
  const int L = __ldg(pp.seq_lens + s);
  return L < 0 ? 0 : (L > cap ? static_cast<int>(cap) : L);
}

__device__ __forceinline__ int clamp_off(const PagedParams& pp, int s) {
  const int o = __ldg(pp.q_offsets + s);
  return o < 0 ? 0 : (o > pp.num_queries ? pp.num_queries : o);
}

// The query rows of sequence s: [q0, q0 + n).
__device__ __forceinline__ void rows_of(const PagedParams& pp, int s, int& q0, int& n) {
  q0 = clamp_off(pp, s);
  const int q1 = clamp_off(pp, s + 1);
  n = q1 > q0 ? q1 - q0 : 0;
}

__device__ __forceinline__ int position_of(const PagedParams& pp, int row, int q0, int n, int L) {
  return pp.positions ? __ldg(pp.positions + row) : L - n + (row - q0);
}

// The key slots [blockIdx.y * kpc, +kpc) of one physical page and kv head.
template <int DK, int PD, int TPK, int DT, bool MLA>
__device__ __forceinline__ void dkdv_page(const void* __restrict__ q, const void* __restrict__ qp,
                                          const void* __restrict__ k, const void* __restrict__ kp,
                                          const void* __restrict__ v, const void* __restrict__ dout,
                                          const Buffers& b, void* __restrict__ dk, void* __restrict__ dkp,
                                          void* __restrict__ dv, const PagedParams& pp, float scale, int kpc,
                                          int page, int hk) {
  using C = Cfg<DK, PD, TPK>;
  constexpr int G = C::G, PG = C::PG, GPT = C::GPT, PPT = C::PPT, RT = C::RT;
  extern __shared__ float4 smem[];
  float4* qs = smem;             // [RT][G]
  float4* gs = qs + RT * G;      // [RT][G]
  float4* qps = gs + RT * G;     // [RT][PG]
  float* ls = reinterpret_cast<float*>(qps + RT * PG);
  float* dss = ls + RT;
  int* ps = reinterpret_cast<int*>(dss + RT);

  const int tid = threadIdx.x, part = tid % TPK, kl = tid / TPK;
  const int group = pp.Hq / pp.Hkv;
  const int P = pp.page_size;
  // extents (float4 groups, rows, entries) for the bounds-checked build
  int* const st = pp.status;
  const size_t nq4 = static_cast<size_t>(pp.num_queries) * pp.Hq * G, nqp4 = static_cast<size_t>(pp.num_queries) * pp.Hq * PG;
  const size_t nk4 = static_cast<size_t>(pp.num_pages) * P * pp.Hkv * G, nkp4 = static_cast<size_t>(pp.num_pages) * P * PG;
  const int64_t nrows = static_cast<int64_t>(pp.num_queries) * pp.Hq;
  const int64_t nrefs = static_cast<int64_t>(pp.num_seqs) * pp.max_pages;
  const int t0 = blockIdx.y * kpc;
  const int t = t0 + kl;
  const bool key_ok = kl < kpc && t < P;
  const size_t slot = static_cast<size_t>(page) * P + (key_ok ? t : 0);
  const size_t krow = (slot * pp.Hkv + hk) * G;

  const bool page_ok = in_bounds(st, page, pp.num_pages);
  const int r_lo = page_ok ? __ldg(b.offsets + page) : 0, r_hi = page_ok ? __ldg(b.offsets + page + 1) : 0;

  float4 kr[GPT], vr[GPT], dka[GPT], dva[GPT], kpr[PPT > 0 ? PPT : 1], dkpa[PPT > 0 ? PPT : 1];
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
  for (int c = 0; c < GPT; ++c) {
    kr[c] = key_ok ? load4<DT>(k, krow + part + TPK * c, nk4, st) : z;
    if constexpr (!MLA) vr[c] = key_ok ? load4<DT>(v, krow + part + TPK * c, nk4, st) : z;
    dka[c] = dva[c] = z;
  }
#pragma unroll
  for (int c = 0; c < PPT; ++c) {
    const int gi = part + TPK * c;
    kpr[c] = (key_ok && gi < PG) ? load4<DT>(kp, slot * PG + gi, nkp4, st) : z;
    dkpa[c] = z;
  }

  for (int ri = r_lo; ri < r_hi; ++ri) {
    if (!in_bounds(st, ri, nrefs)) break;
    const int code = __ldg(b.refs + ri);
    const int s = code / pp.max_pages, blk = code - s * pp.max_pages;
    const int L = keys_of(pp, s);
    const int kmin = blk * P + t0;  // first key position of this CTA in sequence s
    if (kmin >= L) continue;
    int q0, n;
    rows_of(pp, s, q0, n);
    const int kpos = blk * P + t;
    const bool key_vis = key_ok && kpos < L;
    const int npairs = n * group;
    int e_lo = 0;  // rows before e_lo see none of these keys (default positions only)
    if (pp.causal && !pp.positions) e_lo = max(0, kmin - (L - n)) * group;
    // the (query, head) rows of tile e0 of this sequence: element idx of the
    // tile is column c of row r (q, then dout, then qp); row r's statistics
    auto row_of = [&](int e, size_t& rr) {
      const bool in = e < npairs;
      const int qi = in ? e / group : 0;
      rr = static_cast<size_t>(q0 + qi) * pp.Hq + hk * group + (in ? e - qi * group : 0);
      return in;
    };
    auto element = [&](int e0, int idx) {
      const int r = idx / (2 * G + PG), c = idx - r * (2 * G + PG);
      size_t rr;
      if (!row_of(e0 + r, rr)) return z;
      return c < G ? load4<DT>(q, rr * G + c, nq4, st)
                   : (c < 2 * G ? load4<DT>(dout, rr * G + c - G, nq4, st)
                                : load4<DT>(qp, rr * PG + c - 2 * G, nqp4, st));
    };
    auto put = [&](int idx, float4 v) {
      const int r = idx / (2 * G + PG), c = idx - r * (2 * G + PG);
      if (c < G) {
        if (in_bounds(st, r * G + c, RT * G)) qs[r * G + c] = v;
      } else if (c < 2 * G) {
        if (in_bounds(st, r * G + c - G, RT * G)) gs[r * G + c - G] = v;
      } else if (in_bounds(st, r * PG + c - 2 * G, RT * PG)) {
        qps[r * PG + c - 2 * G] = v;
      }
    };
    // the row statistics of row rr (and its position) for the staged tile
    auto stats = [&](size_t rr, float& l2v, float& dsv, int& posv) {
      const bool ok = in_bounds(st, static_cast<int64_t>(rr), nrows);
      l2v = ok ? b.lse2[rr] : -INFINITY;
      dsv = ok ? b.dsum[rr] : 0.f;
      const int qrow = static_cast<int>(rr / pp.Hq);
      posv = (!pp.positions || in_bounds(st, qrow, pp.num_queries)) ? position_of(pp, qrow, q0, n, L) : -1;
    };
    // full 256-thread CTAs load the next tile into registers while computing
    // this one (its latency would otherwise be paid once per tile)
    constexpr int TOT = RT * (2 * G + PG);
    constexpr int NPT = (TOT + THREADS - 1) / THREADS;
    const bool pf = blockDim.x == THREADS;
    float4 pre[NPT];
    float pre_l2 = -INFINITY, pre_ds = 0.f;
    int pre_pos = -1;
    auto fetch = [&](int e0) {
#pragma unroll
      for (int k = 0; k < NPT; ++k) {
        const int idx = tid + k * THREADS;
        pre[k] = idx < TOT ? element(e0, idx) : z;
      }
      if (tid < RT) {
        size_t rr;
        if (row_of(e0 + tid, rr)) {
          stats(rr, pre_l2, pre_ds, pre_pos);
        } else {
          pre_l2 = -INFINITY;
          pre_ds = 0.f;
          pre_pos = -1;
        }
      }
    };
    if (pf && e_lo < npairs) fetch(e_lo);
    for (int e0 = e_lo; e0 < npairs; e0 += RT) {
      __syncthreads();
      if (pf) {
#pragma unroll
        for (int k = 0; k < NPT; ++k)
          if (tid + k * THREADS < TOT) put(tid + k * THREADS, pre[k]);
      } else {
        for (int idx = tid; idx < TOT; idx += blockDim.x) put(idx, element(e0, idx));
        if (tid < RT) {
          size_t rr;
          if (row_of(e0 + tid, rr)) {
            stats(rr, pre_l2, pre_ds, pre_pos);
          } else {
            pre_l2 = -INFINITY;
            pre_ds = 0.f;
            pre_pos = -1;
          }
        }
      }
      if (tid < RT) {
        ls[tid] = pre_l2;
        dss[tid] = pre_l2 != -INFINITY ? pre_ds : 0.f;
        ps[tid] = pre_pos;
      }
      __syncthreads();
      if (pf && e0 + RT < npairs) fetch(e0 + RT);
      const int rows_here = min(RT, npairs - e0);  // rows past the sequence's last are not visited
#pragma unroll 2
      for (int r = 0; r < rows_here; ++r) {
        // two independent partial sums per dot product (shorter FMA chains)
        float sa = 0.f, sb = 0.f, pa = 0.f, pb = 0.f;
#pragma unroll
        for (int c = 0; c < GPT; ++c) {
          if (c & 1) {
            sb = dot4(qs[r * G + part + TPK * c], kr[c], sb);
            pb = dot4(gs[r * G + part + TPK * c], MLA ? kr[c] : vr[c], pb);
          } else {
            sa = dot4(qs[r * G + part + TPK * c], kr[c], sa);
            pa = dot4(gs[r * G + part + TPK * c], MLA ? kr[c] : vr[c], pa);
          }
        }
#pragma unroll
        for (int c = 0; c < PPT; ++c)
          if (part + TPK * c < PG) sb = dot4(qps[r * PG + part + TPK * c], kpr[c], sb);
        const float sd = quad_sum<TPK>(sa + sb);
        const float pd = quad_sum<TPK>(pa + pb);
        const float l2 = ls[r];
        const bool vis = key_vis && l2 != -INFINITY && (!pp.causal || kpos <= ps[r]);
        const float pr = vis ? fast_exp2(sd * pp.scale_log2 - l2) : 0.f;
        const float ds = vis ? pr * (pd - dss[r]) : 0.f;
#pragma unroll
        for (int c = 0; c < GPT; ++c) {
          if constexpr (MLA) {
            dka[c] = axpy4(pr, gs[r * G + part + TPK * c], dka[c]);
            dka[c] = axpy4(ds * scale, qs[r * G + part + TPK * c], dka[c]);
          } else {
            dva[c] = axpy4(pr, gs[r * G + part + TPK * c], dva[c]);
            dka[c] = axpy4(ds, qs[r * G + part + TPK * c], dka[c]);
          }
        }
#pragma unroll
        for (int c = 0; c < PPT; ++c)
          if (part + TPK * c < PG) dkpa[c] = axpy4(ds, qps[r * PG + part + TPK * c], dkpa[c]);
      }
    }
  }
  if (!key_ok) return;
#pragma unroll
  for (int c = 0; c < GPT; ++c) {
    const float4 a = dka[c];
    if constexpr (MLA) {
      if (dk) store4<DT>(dk, krow + part + TPK * c, nk4, st, a);
    } else {
      if (dk)
        store4<DT>(dk, krow + part + TPK * c, nk4, st, make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale));
      if (dv) store4<DT>(dv, krow + part + TPK * c, nk4, st, dva[c]);
    }
  }
#pragma unroll
  for (int c = 0; c < PPT; ++c) {
    const int gi = part + TPK * c;
    const float4 a = dkpa[c];
    if (dkp && gi < PG)
      store4<DT>(dkp, slot * PG + gi, nkp4, st, make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale));
  }
}

// Every page (one CTA per page and kv head), or, with `listed`, the pages of
// the index's list of pages whose reader count is not one (after the
// tensor-core kernel has written the others), the CTAs striding over it.
template <int DK, int PD, int TPK, int DT, bool MLA>
__global__ void __launch_bounds__(THREADS) dkdv_kernel(const void* __restrict__ q, const void* __restrict__ qp,
                                                       const void* __restrict__ k, const void* __restrict__ kp,
                                                       const void* __restrict__ v, const void* __restrict__ dout,
                                                       const Buffers b, void* __restrict__ dk,
                                                       void* __restrict__ dkp, void* __restrict__ dv,
                                                       const PagedParams pp, float scale, int kpc, int listed) {
  const int unit = blockIdx.x / pp.Hkv, hk = blockIdx.x - unit * pp.Hkv;
  if (!listed) {
    dkdv_page<DK, PD, TPK, DT, MLA>(q, qp, k, kp, v, dout, b, dk, dkp, dv, pp, scale, kpc, unit, hk);
    return;
  }
  const int n = *b.list;  // uniform over the CTA
  const int stride = gridDim.x / pp.Hkv;
  for (int li = unit; li < n; li += stride) {
    __syncthreads();  // the previous page's shared-memory rows are no longer read
    if (!in_bounds(pp.status, 1 + li, static_cast<int64_t>(pp.num_pages) + 1)) break;
    dkdv_page<DK, PD, TPK, DT, MLA>(q, qp, k, kp, v, dout, b, dk, dkp, dv, pp, scale, kpc, b.list[1 + li], hk);
  }
}

template <int DK, int PD, int TPK, int DT, bool MLA>
__global__ void __launch_bounds__(THREADS) dq_kernel(const void* __restrict__ q, const void* __restrict__ qp,
                                                     const void* __restrict__ k, const void* __restrict__ kp,
                                                     const void* __restrict__ v, const void* __restrict__ dout,
                                                     const Buffers b, void* __restrict__ dq,
                                                     void* __restrict__ dqp, const PagedParams pp, float scale) {
  using C = Cfg<DK, PD, TPK>;
  constexpr int G = C::G, PG = C::PG, GPT = C::GPT, PPT = C::PPT, RT = C::RT, ROWS = C::ROWS;
  constexpr int VG = MLA ? 0 : G;  // value groups staged (MLA reuses the latent)
  extern __shared__ float4 smem[];
  float4* ks = smem;           // [RT][G]
  float4* vs = ks + RT * G;    // [RT][VG]
  float4* kps = vs + RT * VG;  // [RT][PG]
  __shared__ int hi_s;

  const int tid = threadIdx.x, part = tid % TPK, rl = tid / TPK;
  const int s = blockIdx.x / pp.Hkv, hk = blockIdx.x - s * pp.Hkv;
  const int group = pp.Hq / pp.Hkv;
  const int P = pp.page_size;
  // extents (float4 groups, rows, entries) for the bounds-checked build
  int* const st = pp.status;
  const size_t nq4 = static_cast<size_t>(pp.num_queries) * pp.Hq * G, nqp4 = static_cast<size_t>(pp.num_queries) * pp.Hq * PG;
  const size_t nk4 = static_cast<size_t>(pp.num_pages) * P * pp.Hkv * G, nkp4 = static_cast<size_t>(pp.num_pages) * P * PG;
  const int64_t nrows = static_cast<int64_t>(pp.num_queries) * pp.Hq;
  const int64_t ntab = static_cast<int64_t>(pp.num_seqs) * pp.max_pages;
  int q0, n;
  rows_of(pp, s, q0, n);
  const int npairs = n * group;
  const int e = blockIdx.y * ROWS + rl;
  if (blockIdx.y * ROWS >= npairs) return;  // uniform over the CTA
  const int L = keys_of(pp, s);
  const bool row_ok = e < npairs;
  const int qi = row_ok ? e / group : 0;
  const size_t rr = static_cast<size_t>(q0 + qi) * pp.Hq + hk * group + (row_ok ? e - qi * group : 0);

  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  float4 qr[GPT], gr[GPT], acc[GPT], qpr[PPT > 0 ? PPT : 1], accp[PPT > 0 ? PPT : 1];
#pragma unroll
  for (int c = 0; c < GPT; ++c) {
    qr[c] = row_ok ? load4<DT>(q, rr * G + part + TPK * c, nq4, st) : z;
    gr[c] = row_ok ? load4<DT>(dout, rr * G + part + TPK * c, nq4, st) : z;
    acc[c] = z;
  }
#pragma unroll
  for (int c = 0; c < PPT; ++c) {
    const int gi = part + TPK * c;
    qpr[c] = (row_ok && gi < PG) ? load4<DT>(qp, rr * PG + gi, nqp4, st) : z;
    accp[c] = z;
  }
  const bool stat_ok = row_ok && in_bounds(st, static_cast<int64_t>(rr), nrows);
  const float l2 = stat_ok ? b.lse2[rr] : -INFINITY;
  const bool live = l2 != -INFINITY;
  const float dsi = live ? b.dsum[rr] : 0.f;
  const int pos = (row_ok && (!pp.positions || in_bounds(st, q0 + qi, pp.num_queries)))
                      ? position_of(pp, q0 + qi, q0, n, L) : -1;
  // keys past every row's causal limit are not visited
  if (tid == 0) hi_s = 0;
  __syncthreads();
  if (live && part == 0) atomicMax(&hi_s, pp.causal ? min(L, max(pos + 1, 0)) : L);
  __syncthreads();
  const int hi = hi_s;

  // the key tile at key0, gathered through the page table into registers one
  // tile ahead (its load latency hides behind the current tile), then stored
  // to shared memory: element idx is column c of key row r (k, then v, then kp)
  constexpr int TOT = RT * (G + VG + PG);
  constexpr int NPT = (TOT + THREADS - 1) / THREADS;
  float4 pre[NPT];
  auto fetch = [&](int key0) {
#pragma unroll
    for (int u = 0; u < NPT; ++u) {
      const int idx = tid + u * THREADS;
      const int r = idx / (G + VG + PG), c = idx - r * (G + VG + PG);
      const int j = key0 + r;
      int pg = -1;
      const int64_t te = static_cast<int64_t>(s) * pp.max_pages + j / P;
      if (idx < TOT && j < hi && in_bounds(st, te, ntab)) pg = __ldg(pp.block_table + te);
      const bool ok = pg >= 0 && pg < pp.num_pages;  // entries outside the cache read as zero keys
      const size_t sl = ok ? static_cast<size_t>(pg) * P + j % P : 0;
      float4 x = z;
      if (ok) {
        if (c < G) x = load4<DT>(k, (sl * pp.Hkv + hk) * G + c, nk4, st);
        else if (c < G + VG) x = load4<DT>(v, (sl * pp.Hkv + hk) * G + c - G, nk4, st);
        else x = load4<DT>(kp, sl * PG + c - G - VG, nkp4, st);
      }
      pre[u] = x;
    }
  };
  if (hi > 0) fetch(0);
  for (int key0 = 0; key0 < hi; key0 += RT) {
    __syncthreads();
#pragma unroll
    for (int u = 0; u < NPT; ++u) {
      const int idx = tid + u * THREADS;
      if (idx < TOT) {
        const int r = idx / (G + VG + PG), c = idx - r * (G + VG + PG);
        if (c < G) {
          if (in_bounds(st, r * G + c, RT * G)) ks[r * G + c] = pre[u];
        } else if (c < G + VG) {
          if (in_bounds(st, r * VG + c - G, RT * VG)) vs[r * VG + c - G] = pre[u];
        } else if (in_bounds(st, r * PG + c - G - VG, RT * PG)) {
          kps[r * PG + c - G - VG] = pre[u];
        }
      }
    }
    __syncthreads();
    if (key0 + RT < hi) fetch(key0 + RT);
#pragma unroll 2
    for (int c2 = 0; c2 < RT; ++c2) {
      const int j = key0 + c2;
      // two independent partial sums per dot product (shorter FMA chains)
      float sa = 0.f, sb = 0.f, pa = 0.f, pb = 0.f;
#pragma unroll
      for (int c = 0; c < GPT; ++c) {
        const float4 kv = ks[c2 * G + part + TPK * c];
        const float4 vv = MLA ? kv : vs[c2 * VG + part + TPK * c];
        if (c & 1) {
          sb = dot4(qr[c], kv, sb);
          pb = dot4(gr[c], vv, pb);
        } else {
          sa = dot4(qr[c], kv, sa);
          pa = dot4(gr[c], vv, pa);
        }
      }
#pragma unroll
      for (int c = 0; c < PPT; ++c)
        if (part + TPK * c < PG) sb = dot4(qpr[c], kps[c2 * PG + part + TPK * c], sb);
      const float sd = quad_sum<TPK>(sa + sb);
      const float pd = quad_sum<TPK>(pa + pb);
      const bool vis = live && j < L && (!pp.causal || j <= pos);
      const float pr = vis ? fast_exp2(sd * pp.scale_log2 - l2) : 0.f;
      const float ds = vis ? pr * (pd - dsi) : 0.f;
#pragma unroll
      for (int c = 0; c < GPT; ++c) acc[c] = axpy4(ds, ks[c2 * G + part + TPK * c], acc[c]);
#pragma unroll
      for (int c = 0; c < PPT; ++c)
        if (part + TPK * c < PG) accp[c] = axpy4(ds, kps[c2 * PG + part + TPK * c], accp[c]);
    }
  }
  if (!row_ok) return;
#pragma unroll
  for (int c = 0; c < GPT; ++c) {
    const float4 a = acc[c];
    if (dq)
      store4<DT>(dq, rr * G + part + TPK * c, nq4, st, make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale));
  }
#pragma unroll
  for (int c = 0; c < PPT; ++c) {
    const int gi = part + TPK * c;
    const float4 a = accp[c];
    if (dqp && gi < PG)
      store4<DT>(dqp, rr * PG + gi, nqp4, st, make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale));
  }
}

// Opts a kernel into `smem` bytes of dynamic shared memory when that is above
// the default 48 KB, once per device (`done`: the kernel's own device mask).
template <typename Kernel>
cudaError_t allow_smem(Kernel kern, size_t smem, int device, std::atomic<unsigned long long>& done) {
  if (smem <= 48 * 1024) return cudaSuccess;
  const unsigned long long bit = device >= 0 && device < 64 ? 1ull << device : 0ull;
  if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
  return e;
}

// Launch both kernels of one instance (either may be skipped by passing no
// outputs for it).
template <int DK, int PD, int TPK, int DT, bool MLA>
cudaError_t launch_instance(const PagedParams& pp, const void* q, const void* qp, const void* k, const void* kp,
                            const void* v, const void* dout, const Buffers& b, void* dq, void* dqp, void* dk,
                            void* dkp, void* dv, float scale, cudaStream_t st, bool skip_single = false) {
  using C = Cfg<DK, PD, TPK>;
  static std::atomic<unsigned long long> smem_done[2] = {{0}, {0}};  // this instance's two kernels
  const int group = pp.Hq / pp.Hkv;
  if (dk || dkp || dv) {
    // keys per CTA: the page's slots, rounded up so that a CTA is whole warps;
    // over the listed pages (usually few), 128 page slots of CTAs stride the list
    const int unit = 32 / TPK;
    const int kpc = pp.page_size >= C::ROWS ? C::ROWS : (pp.page_size + unit - 1) / unit * unit;
    const unsigned units = static_cast<unsigned>(skip_single ? std::min(pp.num_pages, 128) : pp.num_pages);
    const dim3 grid(units * pp.Hkv, static_cast<unsigned>((pp.page_size + kpc - 1) / kpc));
    const size_t smem = C::dkdv_smem(MLA);
    auto kern = dkdv_kernel<DK, PD, TPK, DT, MLA>;
    cudaError_t e = allow_smem(kern, smem, pp.device, smem_done[0]);
    if (e != cudaSuccess) return e;
    if (grid.x > 0) kern<<<grid, kpc * TPK, smem, st>>>(q, qp, k, kp, v, dout, b, dk, dkp, dv, pp, scale, kpc,
                                                      skip_single ? 1 : 0);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  if (dq || dqp) {
    const int64_t blocks = (static_cast<int64_t>(pp.max_queries) * group + C::ROWS - 1) / C::ROWS;
    const dim3 grid(static_cast<unsigned>(pp.num_seqs) * pp.Hkv, static_cast<unsigned>(blocks));
    const size_t smem = C::dq_smem(MLA);
    auto kern = dq_kernel<DK, PD, TPK, DT, MLA>;
    cudaError_t e = allow_smem(kern, smem, pp.device, smem_done[1]);
    if (e != cudaSuccess) return e;
    if (grid.x > 0 && grid.y > 0) kern<<<grid, THREADS, smem, st>>>(q, qp, k, kp, v, dout, b, dq, dqp, pp, scale);
  }
  return cudaGetLastError();
}

}  // namespace pbwd
}  // namespace attn
