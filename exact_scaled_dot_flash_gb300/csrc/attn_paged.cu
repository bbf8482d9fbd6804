// attn_paged.cu - attention over a paged key/value cache with packed
// variable-length queries, fp32 FMA arithmetic: the calls the tensor-core
// kernel (attn_paged_tc.cuh) does not take (F32, D in {16, 32}, page sizes
// its tile gathers do not cover).
//
// Source: ruDNN user guide, section 9 (paged attention): the kernel reads the
// physical cache pages directly (K and V [pages, page_size, Hkv, D]) through
// per-sequence page tables, handles packed prefill and decode queries
// ([queries, Hq, D], output likewise), and compares absolute positions for
// the causal mask. Key j of sequence s is row j % page_size of page
// table[s][j / page_size]; the queries of sequence s are rows
// q_offsets[s] .. q_offsets[s+1]-1; a query at position pos sees keys
// j < seq_len[s] (and j <= pos when causal); without explicit positions the
// n queries of a sequence of length L sit at L - n .. L - 1.
//
// CTA = one (sequence, kv head) and 64 rows, a row being a (query, query
// head of the GQA group) pair, so every key/value row gathered into shared
// memory serves all the heads that share it. 4 threads per row, as in the
// F32 kernel; keys stream 32 at a time.
//
// Metadata is trusted only as far as memory safety: a page index outside
// [0, num_pages) reads as zeros, lengths are clamped to the table's capacity
// and query offsets to [0, num_queries].
#include "params.h"
#include "ptx.cuh"
#include "simt.cuh"

namespace attn {
namespace paged {

using simt::axpy4;
using simt::dot4;
using simt::load4;
using simt::store4;

constexpr int ROWS = 64;
constexpr int THREADS = 256;
constexpr int KT = 32;
constexpr float LN2 = 0.6931471805599453f;

template <int D, int DT>
__global__ void __launch_bounds__(THREADS) paged_fwd_kernel(const void* __restrict__ q,
                                                            const void* __restrict__ kc,
                                                            const void* __restrict__ vc,
                                                            void* __restrict__ out, float* __restrict__ lse,
                                                            const PagedParams pp) {
  constexpr int G = D / 4;
  constexpr int GPT = G / 4;
  __shared__ float4 ks[KT][G];
  __shared__ float4 vs[KT][G];

  const int tid = threadIdx.x, part = tid & 3, rl = tid >> 2;
  const int s = blockIdx.x / pp.Hkv, hk = blockIdx.x - s * pp.Hkv;
  const int group = pp.Hq / pp.Hkv;
  const int q_lo = min(max(__ldg(pp.q_offsets + s), 0), pp.num_queries);
  const int q_hi = min(max(__ldg(pp.q_offsets + s + 1), q_lo), pp.num_queries);
  const int nq = q_hi - q_lo;
  const int r = blockIdx.y * ROWS + rl;  // row = (query, head of the group)
  if (blockIdx.y * ROWS >= nq * group) return;  // CTA-uniform
  const int tq = r / group;
  const int h = hk * group + (r - tq * group);
  const bool row_ok = tq < nq;
  const int t = q_lo + (row_ok ? tq : 0);
  const int L = min(max(__ldg(pp.seq_lens + s), 0), pp.max_pages * pp.page_size);
  // extents (float4 groups, rows) for the bounds-checked build
  int* const st = pp.status;
  const size_t nq4 = static_cast<size_t>(pp.num_queries) * pp.Hq * G;
  const size_t nk4 = static_cast<size_t>(pp.num_pages) * pp.page_size * pp.Hkv * G;
  const int pos = pp.positions ? (in_bounds(st, t, pp.num_queries) ? __ldg(pp.positions + t) : -1) : L - nq + tq;
  const int key_hi_row = pp.causal ? min(L, pos + 1) : L;  // keys [0, key_hi_row) are visible to this row
  // keys any row of this CTA may see
  int key_hi = L;
  if (pp.causal && !pp.positions) {
    const int last = min(nq - 1, (blockIdx.y * ROWS + ROWS - 1) / group);
    key_hi = min(L, L - nq + last + 1);
  }

  const size_t qrow = (static_cast<size_t>(t) * pp.Hq + h) * G;
  float4 qr[GPT], acc[GPT];
#pragma unroll
  for (int i = 0; i < GPT; ++i) {
    qr[i] = row_ok ? load4<DT>(q, qrow + part + 4 * i, nq4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
    acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int32_t* table = pp.block_table + static_cast<size_t>(s) * pp.max_pages;
  const int64_t ntab = static_cast<int64_t>(pp.num_seqs) * pp.max_pages;
  float m_run = -INFINITY, l_run = 0.f;
  for (int key0 = 0; key0 < key_hi; key0 += KT) {
    __syncthreads();
    for (int e = tid; e < KT * G; e += THREADS) {
      const int kr = e / G, c = e - (e / G) * G;
      const int j = key0 + kr;
      float4 kv = make_float4(0.f, 0.f, 0.f, 0.f), vv = kv;
      if (j < key_hi && in_bounds(st, static_cast<int64_t>(s) * pp.max_pages + j / pp.page_size, ntab)) {
        const int page = __ldg(table + j / pp.page_size);
        if (page >= 0 && page < pp.num_pages) {
          const size_t idx = ((static_cast<size_t>(page) * pp.page_size + j % pp.page_size) * pp.Hkv + hk) * G + c;
          kv = load4<DT>(kc, idx, nk4, st);
          vv = load4<DT>(vc, idx, nk4, st);
        }
      }
      if (in_bounds(st, kr * G + c, KT * G)) {
        ks[kr][c] = kv;
        vs[kr][c] = vv;
      }
    }
    __syncthreads();
    float sreg[KT];
#pragma unroll
    for (int c = 0; c < KT; ++c) {
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < GPT; ++i) d = dot4(qr[i], ks[c][part + 4 * i], d);
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      sreg[c] = (row_ok && key0 + c < key_hi_row) ? d * pp.scale_log2 : -INFINITY;
    }
    float mx = sreg[0];
#pragma unroll
    for (int c = 1; c < KT; ++c) mx = fmaxf(mx, sreg[c]);
    const float m_new = fmaxf(m_run, mx);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = fast_exp2(m_run - m_use);
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < KT; ++c) {
      sreg[c] = fast_exp2(sreg[c] - m_use);
      sum += sreg[c];
    }
    l_run = l_run * alpha + sum;
    m_run = m_new;
#pragma unroll
    for (int i = 0; i < GPT; ++i) {
      float4 a = acc[i];
      a.x *= alpha; a.y *= alpha; a.z *= alpha; a.w *= alpha;
#pragma unroll
      for (int c = 0; c < KT; ++c) a = axpy4(sreg[c], vs[c][part + 4 * i], a);
      acc[i] = a;
    }
  }
  if (!row_ok) return;
  const float inv = l_run > 0.f ? 1.f / l_run : __int_as_float(0x7fc00000);
#pragma unroll
  for (int i = 0; i < GPT; ++i) {
    const float4 a = acc[i];
    store4<DT>(out, qrow + part + 4 * i, nq4, st, make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv));
  }
  if (lse && part == 0 && in_bounds(st, static_cast<int64_t>(t) * pp.Hq + h, static_cast<int64_t>(pp.num_queries) * pp.Hq))
    lse[static_cast<size_t>(t) * pp.Hq + h] = l_run > 0.f ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
}

// Decode-shaped calls (at most RMAX rows = queries x group heads per
// (sequence, kv head)): one CTA of DEC_WARPS warps per (sequence, kv head,
// split). Each lane
// owns one key of a 32-key chunk and computes its scores against every row
// (queries in shared memory, broadcast reads); each row keeps an online
// softmax per warp (warp max and sum by shuffles); P V then runs with lanes
// over dimensions, the probabilities shuffled out key by key and the value
// rows read coalesced, VB rows per batch of independent loads. The warps take
// interleaved chunks and are combined through shared memory at the end.
// Bandwidth-bound: every key row is read once for all the heads of its group.
// With num_splits > 1, CTA (., z) takes the z-th balanced run of 32-key
// chunks and writes its unnormalised partial (m, l, O) for launch_split_merge.
constexpr int RMAX = 8;
constexpr int DEC_WARPS = 8;
constexpr int VB = 8;  // value rows loaded together in P V

template <int D, int DT>
__global__ void __launch_bounds__(DEC_WARPS * 32) paged_decode_kernel(const void* __restrict__ q,
                                                                      const void* __restrict__ kc,
                                                                      const void* __restrict__ vc,
                                                                      void* __restrict__ out,
                                                                      float* __restrict__ lse,
                                                                      const PagedParams pp) {
  constexpr int G = D / 4;             // float4 groups of a row
  constexpr int LG = (G + 31) / 32;    // float4 groups of a row per lane in P V
  __shared__ float4 qs[RMAX][G];
  __shared__ float sm_m[DEC_WARPS][RMAX], sm_l[DEC_WARPS][RMAX];
  __shared__ float4 sm_acc[DEC_WARPS][RMAX][G];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int s = blockIdx.x / pp.Hkv, hk = blockIdx.x - s * pp.Hkv;
  const int group = pp.Hq / pp.Hkv;
  const int q_lo = min(max(__ldg(pp.q_offsets + s), 0), pp.num_queries);
  const int q_hi = min(max(__ldg(pp.q_offsets + s + 1), q_lo), pp.num_queries);
  const int nq = q_hi - q_lo;
  // rows of this CTA: <= RMAX when max_queries bounds every sequence, as the
  // call requires; clamped so that a wrong bound cannot index past RMAX
  const int R = min(nq * group, RMAX);
  if (R <= 0) return;
  const int L = min(max(__ldg(pp.seq_lens + s), 0), pp.max_pages * pp.page_size);
  // extents (float4 groups, rows, entries) for the bounds-checked build
  int* const st = pp.status;
  const int64_t nrows = static_cast<int64_t>(pp.num_queries) * pp.Hq;
  const size_t nq4 = static_cast<size_t>(nrows) * G;
  const size_t nk4 = static_cast<size_t>(pp.num_pages) * pp.page_size * pp.Hkv * G;
  const int64_t ntab = static_cast<int64_t>(pp.num_seqs) * pp.max_pages;
  // rows' positions and the CTA's key range
  int pos[RMAX];
  int key_hi = 0;
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    const int tq = r / group;
    pos[r] = r < R ? (pp.positions ? (in_bounds(st, q_lo + tq, pp.num_queries) ? __ldg(pp.positions + q_lo + tq) : -1)
                                   : L - nq + tq)
                   : -1;
    if (r < R) key_hi = max(key_hi, pp.causal ? min(L, pos[r] + 1) : L);
  }
  for (int e = threadIdx.x; e < RMAX * G; e += DEC_WARPS * 32) {
    const int r = e / G, c = e - (e / G) * G;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (r < R) {
      const int t = q_lo + r / group, h = hk * group + r % group;
      v = load4<DT>(q, (static_cast<size_t>(t) * pp.Hq + h) * G + c, nq4, st);
    }
    if (in_bounds(st, r * G + c, RMAX * G)) qs[r][c] = v;
  }
  __syncthreads();

  const int32_t* table = pp.block_table + static_cast<size_t>(s) * pp.max_pages;
  float m_w[RMAX], l_w[RMAX];
  float4 acc[RMAX][LG];
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    m_w[r] = -INFINITY;
    l_w[r] = 0.f;
#pragma unroll
    for (int i = 0; i < LG; ++i) acc[r][i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int nchunks = (key_hi + 31) / 32;
  const int c_lo = static_cast<int>(static_cast<int64_t>(blockIdx.y) * nchunks / pp.num_splits);
  const int c_hi = static_cast<int>(static_cast<int64_t>(blockIdx.y + 1) * nchunks / pp.num_splits);
  for (int c = c_lo + warp; c < c_hi; c += DEC_WARPS) {
    const int j = c * 32 + lane;
    const bool in = j < key_hi;
    int page = (in && in_bounds(st, static_cast<int64_t>(s) * pp.max_pages + j / pp.page_size, ntab))
                   ? __ldg(table + j / pp.page_size) : -1;
    const bool ok = in && page >= 0 && page < pp.num_pages;
    const size_t krow = ok ? ((static_cast<size_t>(page) * pp.page_size + j % pp.page_size) * pp.Hkv + hk) * G : 0;
    // scores of this lane's key against every row
    float sc[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) sc[r] = 0.f;
    if (ok) {  // the lane's key row, 8 values per load
#pragma unroll 4
      for (int g2 = 0; g2 < G / 2; ++g2) {
        float4 k0, k1;
        simt::load8<DT>(kc, krow / 2 + g2, nk4 / 2, st, k0, k1);
#pragma unroll
        for (int r = 0; r < RMAX; ++r) sc[r] = dot4(qs[r][2 * g2 + 1], k1, dot4(qs[r][2 * g2], k0, sc[r]));
      }
    }
    float p[RMAX];
#pragma unroll
    for (int r = 0; r < RMAX; ++r) {
      const bool vis = in && r < R && (!pp.causal || j <= pos[r]);
      float x = vis ? sc[r] * pp.scale_log2 : -INFINITY;
      float mx = x;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
      const float m_new = fmaxf(m_w[r], mx);
      const float m_use = m_new == -INFINITY ? 0.f : m_new;
      const float alpha = fast_exp2(m_w[r] - m_use);
      p[r] = fast_exp2(x - m_use);
      float sum = p[r];
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      l_w[r] = l_w[r] * alpha + sum;
      m_w[r] = m_new;
#pragma unroll
      for (int i = 0; i < LG; ++i) {
        acc[r][i].x *= alpha; acc[r][i].y *= alpha; acc[r][i].z *= alpha; acc[r][i].w *= alpha;
      }
    }
    // P V: lanes over dimensions, VB keys per batch (loads first, then FMAs)
    const int kmax = min(32, key_hi - c * 32);
    for (int k0 = 0; k0 < kmax; k0 += VB) {
      float4 vv[VB][LG];
#pragma unroll
      for (int b = 0; b < VB; ++b) {
        const int k = k0 + b;
        const int pg = __shfl_sync(0xffffffffu, page, k & 31);
        const bool use = k < kmax && pg >= 0 && pg < pp.num_pages;  // warp-uniform
        const int jk = c * 32 + k;
        const size_t vrow = use ? ((static_cast<size_t>(pg) * pp.page_size + jk % pp.page_size) * pp.Hkv + hk) * G : 0;
#pragma unroll
        for (int i = 0; i < LG; ++i) {
          const int g = lane + 32 * i;
          vv[b][i] = (use && g < G) ? load4<DT>(vc, vrow + g, nk4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
      }
#pragma unroll
      for (int b = 0; b < VB; ++b) {
        const int k = (k0 + b) & 31;
#pragma unroll
        for (int r = 0; r < RMAX; ++r) {
          const float pk = __shfl_sync(0xffffffffu, p[r], k);  // 0 for a key past kmax (masked)
#pragma unroll
          for (int i = 0; i < LG; ++i) acc[r][i] = axpy4(pk, vv[b][i], acc[r][i]);
        }
      }
    }
  }
  // combine the warps
#pragma unroll
  for (int r = 0; r < RMAX; ++r) {
    if (lane == 0) {
      sm_m[warp][r] = m_w[r];
      sm_l[warp][r] = l_w[r];
    }
#pragma unroll
    for (int i = 0; i < LG; ++i)
      if (lane + 32 * i < G) sm_acc[warp][r][lane + 32 * i] = acc[r][i];
  }
  __syncthreads();
  for (int e = threadIdx.x; e < R * G; e += DEC_WARPS * 32) {
    const int r = e / G, g = e - (e / G) * G;
    float M = -INFINITY;
#pragma unroll
    for (int wv = 0; wv < DEC_WARPS; ++wv) M = fmaxf(M, sm_m[wv][r]);
    float Ls = 0.f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
#pragma unroll
      for (int wv = 0; wv < DEC_WARPS; ++wv) {
        const float f = fast_exp2(sm_m[wv][r] - M);  // 0 for a warp that saw no key
        Ls = fmaf(f, sm_l[wv][r], Ls);
        o = axpy4(f, sm_acc[wv][r][g], o);
      }
    }
    const int t = q_lo + r / group, h = hk * group + r % group;
    const size_t row = static_cast<size_t>(t) * pp.Hq + h;
    if (pp.num_splits > 1) {  // partial of this split, relative to 2^M
      const size_t rr = static_cast<size_t>(blockIdx.y) * pp.num_queries * pp.Hq + row;
      if (!in_bounds(st, static_cast<int64_t>(rr), pp.num_splits * nrows)) continue;
      reinterpret_cast<float4*>(pp.ws_o)[rr * G + g] = o;
      if (g == 0) pp.ws_ml[rr] = make_float2(M, Ls);
      continue;
    }
    const float inv = Ls > 0.f ? 1.f / Ls : __int_as_float(0x7fc00000);
    store4<DT>(out, row * G + g, nq4, st, make_float4(o.x * inv, o.y * inv, o.z * inv, o.w * inv));
    if (lse && g == 0 && in_bounds(st, static_cast<int64_t>(row), nrows))
      lse[row] = Ls > 0.f ? (M + log2f(Ls)) * LN2 : -INFINITY;
  }
}

template <int DT>
static cudaError_t launch_dt(int D, const PagedParams& pp, const void* q, const void* k, const void* v,
                             void* out, float* lse, cudaStream_t st, int* unsupported) {
  const int group = pp.Hq / pp.Hkv;
  if (paged_is_decode(pp.max_queries, group)) {  // a CTA per (sequence, kv head, split)
    const dim3 grid(static_cast<unsigned>(pp.num_seqs) * pp.Hkv, static_cast<unsigned>(pp.num_splits));
    switch (D) {
      case 16: paged_decode_kernel<16, DT><<<grid, DEC_WARPS * 32, 0, st>>>(q, k, v, out, lse, pp); break;
      case 32: paged_decode_kernel<32, DT><<<grid, DEC_WARPS * 32, 0, st>>>(q, k, v, out, lse, pp); break;
      case 64: paged_decode_kernel<64, DT><<<grid, DEC_WARPS * 32, 0, st>>>(q, k, v, out, lse, pp); break;
      case 128: paged_decode_kernel<128, DT><<<grid, DEC_WARPS * 32, 0, st>>>(q, k, v, out, lse, pp); break;
      default: *unsupported = 1; return cudaSuccess;
    }
    return cudaGetLastError();
  }
  const int64_t ry = (static_cast<int64_t>(pp.max_queries) * group + ROWS - 1) / ROWS;
  const dim3 grid(static_cast<unsigned>(pp.num_seqs) * pp.Hkv, static_cast<unsigned>(ry > 0 ? ry : 1));
  switch (D) {
    case 16: paged_fwd_kernel<16, DT><<<grid, THREADS, 0, st>>>(q, k, v, out, lse, pp); break;
    case 32: paged_fwd_kernel<32, DT><<<grid, THREADS, 0, st>>>(q, k, v, out, lse, pp); break;
    case 64: paged_fwd_kernel<64, DT><<<grid, THREADS, 0, st>>>(q, k, v, out, lse, pp); break;
    case 128: paged_fwd_kernel<128, DT><<<grid, THREADS, 0, st>>>(q, k, v, out, lse, pp); break;
    default: *unsupported = 1; return cudaSuccess;
  }
  return cudaGetLastError();
}

}  // namespace paged

cudaError_t launch_paged_simt(int D, int dtype, const PagedParams& pp, const void* q, const void* k,
                              const void* v, void* out, float* lse, cudaStream_t stream, int* unsupported) {
  *unsupported = 0;
  if (dtype == 0) return paged::launch_dt<0>(D, pp, q, k, v, out, lse, stream, unsupported);
  if (dtype == 1) return paged::launch_dt<1>(D, pp, q, k, v, out, lse, stream, unsupported);
  return paged::launch_dt<2>(D, pp, q, k, v, out, lse, stream, unsupported);
}

}  // namespace attn
