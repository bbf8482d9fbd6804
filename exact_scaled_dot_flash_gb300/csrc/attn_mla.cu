// attn_mla.cu - multi-head latent attention (MLA) with absorbed projections
// over a paged latent cache, fp32 FMA arithmetic for every dtype.
//
// Source: ruDNN user guide, section 9 (paged attention and MLA): the query
// arrives with the key projection absorbed, q [queries, H, R], plus a
// positional query qp [queries, H, P]; the cache holds one latent row c_j
// [pages, page_size, 1, R] and one positional key kp_j [pages, page_size, 1,
// P] per token, shared by every head; the output is the compressed context
// [queries, H, R]:
//   s_j = scale (q . c_j + qp . kp_j),   out = sum_j softmax_j(s) c_j.
// Paging, packed queries, positions and the causal mask are those of
// attn_paged.cu.
//
// CTA = one sequence and 256 / (R/16) rows, a row being a (query, head) pair;
// every latent row gathered into shared memory serves all the heads. R/16
// threads share a row: each holds 16 values of q and of the accumulator and a
// share of the Pd positional values, and the dot products are reduced with
// log2(R/16) xor shuffles. Keys stream 8 at a time as fp32
// [latent | positional] rows.
#include "params.h"
#include "ptx.cuh"
#include "simt.cuh"

namespace attn {
namespace mla {

using simt::axpy4;
using simt::dot4;
using simt::load4;
using simt::store4;

constexpr int THREADS = 256;
constexpr int KT = 8;
template <int R>
struct RowMap {
  static constexpr int TPR = R / 16;  // threads per row
  static constexpr int ROWS = THREADS / TPR;
};
constexpr float LN2 = 0.6931471805599453f;

template <int R, int PD, int DT>
__global__ void __launch_bounds__(THREADS) mla_fwd_kernel(const void* __restrict__ q, const void* __restrict__ qp,
                                                          const void* __restrict__ lat,
                                                          const void* __restrict__ kpos, void* __restrict__ out,
                                                          float* __restrict__ lse, const PagedParams pp) {
  constexpr int TPR = RowMap<R>::TPR;
  constexpr int ROWS = RowMap<R>::ROWS;
  constexpr int GR = R / 4;             // float4 groups of a latent row
  constexpr int GRT = GR / TPR;         // ... per thread (4)
  constexpr int GP = PD / 4;            // float4 groups of a positional row
  constexpr int GPT = (GP + TPR - 1) / TPR;
  static_assert(GR % TPR == 0, "R must be a multiple of 32");
  __shared__ float4 cs[KT][GR];
  __shared__ float4 ps[KT][GP > 0 ? GP : 1];

  const int tid = threadIdx.x, part = tid & (TPR - 1), rl = tid / TPR;
  const int s = blockIdx.x;
  const int H = pp.Hq;
  const int q_lo = min(max(__ldg(pp.q_offsets + s), 0), pp.num_queries);
  const int q_hi = min(max(__ldg(pp.q_offsets + s + 1), q_lo), pp.num_queries);
  const int nq = q_hi - q_lo;
  if (static_cast<int>(blockIdx.y) * ROWS >= nq * H) return;  // CTA-uniform
  const int r = blockIdx.y * ROWS + rl;
  const int tq = r / H, h = r - (r / H) * H;
  const bool row_ok = tq < nq;
  const int t = q_lo + (row_ok ? tq : 0);
  const int L = min(max(__ldg(pp.seq_lens + s), 0), pp.max_pages * pp.page_size);
  // extents (float4 groups, rows, entries) for the bounds-checked build
  int* const st = pp.status;
  const int64_t nrows = static_cast<int64_t>(pp.num_queries) * H;
  const size_t ntok = static_cast<size_t>(pp.num_pages) * pp.page_size;
  const int64_t ntab = static_cast<int64_t>(pp.num_seqs) * pp.max_pages;
  const int pos = pp.positions ? (in_bounds(st, t, pp.num_queries) ? __ldg(pp.positions + t) : -1) : L - nq + tq;
  const int key_hi_row = pp.causal ? min(L, pos + 1) : L;
  int key_hi = L;
  if (pp.causal && !pp.positions) {
    const int last = min(nq - 1, (static_cast<int>(blockIdx.y) * ROWS + ROWS - 1) / H);
    key_hi = min(L, L - nq + last + 1);
  }

  const size_t row = static_cast<size_t>(t) * H + h;
  float4 qr[GRT], acc[GRT];
#pragma unroll
  for (int i = 0; i < GRT; ++i) {
    qr[i] = row_ok ? load4<DT>(q, row * GR + part + TPR * i, nrows * GR, st) : make_float4(0.f, 0.f, 0.f, 0.f);
    acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  float4 qpr[GPT > 0 ? GPT : 1];
#pragma unroll
  for (int i = 0; i < GPT; ++i) {
    const int g = part + TPR * i;
    qpr[i] = (row_ok && g < GP) ? load4<DT>(qp, row * GP + g, nrows * GP, st) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const int32_t* table = pp.block_table + static_cast<size_t>(s) * pp.max_pages;
  float m_run = -INFINITY, l_run = 0.f;
  for (int key0 = 0; key0 < key_hi; key0 += KT) {
    __syncthreads();
    for (int e = tid; e < KT * (GR + GP); e += THREADS) {
      const int kr = e / (GR + GP), c = e - kr * (GR + GP);
      const int j = key0 + kr;
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (j < key_hi && in_bounds(st, static_cast<int64_t>(s) * pp.max_pages + j / pp.page_size, ntab)) {
        const int page = __ldg(table + j / pp.page_size);
        if (page >= 0 && page < pp.num_pages) {
          const size_t tok = static_cast<size_t>(page) * pp.page_size + j % pp.page_size;
          v = c < GR ? load4<DT>(lat, tok * GR + c, ntok * GR, st) : load4<DT>(kpos, tok * GP + (c - GR), ntok * GP, st);
        }
      }
      if (c < GR) {
        if (in_bounds(st, kr * GR + c, KT * GR)) cs[kr][c] = v;
      } else if (in_bounds(st, kr * GP + c - GR, KT * GP)) {
        ps[kr][c - GR] = v;
      }
    }
    __syncthreads();
    float sreg[KT];
#pragma unroll
    for (int c = 0; c < KT; ++c) {
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < GRT; ++i) d = dot4(qr[i], cs[c][part + TPR * i], d);
#pragma unroll
      for (int i = 0; i < GPT; ++i)
        if (part + TPR * i < GP) d = dot4(qpr[i], ps[c][part + TPR * i], d);
#pragma unroll
      for (int o = 1; o < TPR; o <<= 1) d += __shfl_xor_sync(0xffffffffu, d, o);
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
    for (int i = 0; i < GRT; ++i) {
      float4 a = acc[i];
      a.x *= alpha; a.y *= alpha; a.z *= alpha; a.w *= alpha;
#pragma unroll
      for (int c = 0; c < KT; ++c) a = axpy4(sreg[c], cs[c][part + TPR * i], a);
      acc[i] = a;
    }
  }
  if (!row_ok) return;
  const float inv = l_run > 0.f ? 1.f / l_run : __int_as_float(0x7fc00000);
#pragma unroll
  for (int i = 0; i < GRT; ++i) {
    const float4 a = acc[i];
    store4<DT>(out, row * GR + part + TPR * i, nrows * GR, st, make_float4(a.x * inv, a.y * inv, a.z * inv, a.w * inv));
  }
  if (lse && part == 0 && in_bounds(st, static_cast<int64_t>(row), nrows))
    lse[row] = l_run > 0.f ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
}

template <int R, int PD>
static cudaError_t launch_rp(int dtype, const PagedParams& pp, const void* q, const void* qp, const void* lat,
                             const void* kp, void* out, float* lse, cudaStream_t st) {
  constexpr int ROWS = RowMap<R>::ROWS;
  const int64_t ry = (static_cast<int64_t>(pp.max_queries) * pp.Hq + ROWS - 1) / ROWS;
  const dim3 grid(static_cast<unsigned>(pp.num_seqs), static_cast<unsigned>(ry > 0 ? ry : 1));
  if (dtype == 0) mla_fwd_kernel<R, PD, 0><<<grid, THREADS, 0, st>>>(q, qp, lat, kp, out, lse, pp);
  else if (dtype == 1) mla_fwd_kernel<R, PD, 1><<<grid, THREADS, 0, st>>>(q, qp, lat, kp, out, lse, pp);
  else mla_fwd_kernel<R, PD, 2><<<grid, THREADS, 0, st>>>(q, qp, lat, kp, out, lse, pp);
  return cudaGetLastError();
}

template <int R>
static cudaError_t launch_r(int Pd, int dtype, const PagedParams& pp, const void* q, const void* qp, const void* lat,
                            const void* kp, void* out, float* lse, cudaStream_t st, int* unsupported) {
  switch (Pd) {
    case 0: return launch_rp<R, 0>(dtype, pp, q, qp, lat, kp, out, lse, st);
    case 16: return launch_rp<R, 16>(dtype, pp, q, qp, lat, kp, out, lse, st);
    case 32: return launch_rp<R, 32>(dtype, pp, q, qp, lat, kp, out, lse, st);
    case 64: return launch_rp<R, 64>(dtype, pp, q, qp, lat, kp, out, lse, st);
    default: *unsupported = 1; return cudaSuccess;
  }
}

}  // namespace mla

cudaError_t launch_mla_simt(int R, int Pd, int dtype, const PagedParams& pp, const void* q, const void* qp,
                            const void* lat, const void* kp, void* out, float* lse, cudaStream_t stream,
                            int* unsupported) {
  *unsupported = 0;
  switch (R) {
    case 128: return mla::launch_r<128>(Pd, dtype, pp, q, qp, lat, kp, out, lse, stream, unsupported);
    case 256: return mla::launch_r<256>(Pd, dtype, pp, q, qp, lat, kp, out, lse, stream, unsupported);
    case 512: return mla::launch_r<512>(Pd, dtype, pp, q, qp, lat, kp, out, lse, stream, unsupported);
    default: *unsupported = 1; return cudaSuccess;
  }
}

}  // namespace attn
