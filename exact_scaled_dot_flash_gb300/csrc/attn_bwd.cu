// attn_bwd.cu - attention backward (dq, dk, dv) with fp32 FMA arithmetic, for
// every dtype: the ordered path, with no atomics and a fixed summation order.
//
// Source: ruDNN user guide, section 11: the backward returns dq, dk, dv,
// recomputes the probabilities from the inputs instead of storing the score
// matrix, and has an ordered variant without atomic accumulation. With the
// forward's row log-sum-exp lse_i (natural log), for every visible (i, j):
//
//   p_ij  = exp(scale * q_i.k_j + bias_ij - lse_i)
//   dp_ij = dout_i . v_j,      D_i = dout_i . o_i  (= sum_j p_ij dp_ij)
//   ds_ij = p_ij * (dp_ij - D_i)
//   dv_j  = sum_i p_ij dout_i,   dk_j = scale * sum_i ds_ij q_i,
//   dq_i  = scale * sum_j ds_ij k_j
//
// GQA: dk, dv of a key/value head sum over its query heads. Rows with
// lse = -inf (no visible key) contribute nothing and get dq = 0.
//
// Three kernels: a per-row preprocess (D_i and lse in log2 units; the paged
// backward's row-statistics kernel), a
// key-major kernel for dk, dv (each CTA owns 64 keys of one (b, kv head) and
// walks every query row of the group that can see them), and a query-major
// kernel for dq (64 rows per CTA, keys streamed through shared memory).
// 4 threads share a row (or key): each owns D/4 of its vectors, and the dot
// products are reduced with two xor shuffles.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "paged_bwd.h"
#include "params.h"
#include "ptx.cuh"
#include "simt.cuh"

namespace attn {
namespace bwd {

using simt::load4;
using simt::store4;
using simt::dot4;
using simt::axpy4;

constexpr int ROWS = 64;     // keys (dk/dv kernel) or query rows (dq kernel) per CTA
constexpr int THREADS = 256;
constexpr int RT = 32;       // query rows (or keys) per shared-memory tile
constexpr float LOG2E = 1.4426950408889634f;

// dk, dv: CTA = 64 keys of one (b, kv head); all query heads of its group.
template <int D, int DT, bool BIAS>
__global__ void __launch_bounds__(THREADS) dkdv_kernel(const void* __restrict__ q,
                                                       const void* __restrict__ k,
                                                       const void* __restrict__ v,
                                                       const void* __restrict__ dout,
                                                       const float* __restrict__ dsum,
                                                       const float* __restrict__ lse2,
                                                       void* __restrict__ dk, void* __restrict__ dv,
                                                       const KernelParams p, float scale) {
  constexpr int G = D / 4;    // float4 groups per vector
  constexpr int GPT = G / 4;  // groups per thread
  __shared__ float4 qs[RT][G];
  __shared__ float4 gs[RT][G];
  __shared__ float ls[RT], dss[RT];

  const int tid = threadIdx.x, part = tid & 3, kl = tid >> 2;
  const int bhk = blockIdx.x;
  const int b = bhk / p.Hkv, hk = bhk - b * p.Hkv;
  const int key0 = blockIdx.y * ROWS;
  const int key = key0 + kl;
  const bool key_ok = key < p.Sk;
  int lim = p.Sk;
  if (p.padding) {
    const int L = __ldg(p.kv_lens + b);
    lim = L < 0 ? 0 : (L > p.Sk ? p.Sk : L);
  }
  const int diag = p.Sk - p.Sq;
  // extents (float4 groups, rows, elements) for the bounds-checked build
  int* const st = p.status;
  const size_t nq4 = static_cast<size_t>(p.B) * p.Hq * p.Sq * G, nk4 = static_cast<size_t>(p.B) * p.Hkv * p.Sk * G;
  const int64_t nrows = static_cast<int64_t>(p.B) * p.Hq * p.Sq;
  const int64_t nbias = static_cast<int64_t>(p.bias_b) * p.bias_h * p.Sq * p.Sk;

  float4 kr[GPT], vr[GPT], dka[GPT], dva[GPT];
  const size_t kvrow = (static_cast<size_t>(bhk) * p.Sk + (key_ok ? key : 0)) * G;
#pragma unroll
  for (int i = 0; i < GPT; ++i) {
    kr[i] = key_ok ? load4<DT>(k, kvrow + part + 4 * i, nk4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
    vr[i] = key_ok ? load4<DT>(v, kvrow + part + 4 * i, nk4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
    dka[i] = dva[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // query rows that can see some key of this CTA (causal: i >= key0 - diag)
  const int row_lo = p.causal ? max(0, key0 - diag) : 0;
  const bool any_key = key0 < lim;
  for (int g = 0; g < p.group && any_key; ++g) {
    const int hq = hk * p.group + g;
    const size_t bh = static_cast<size_t>(b) * p.Hq + hq;
    const float* brow0 = nullptr;
    if constexpr (BIAS) {
      const int bb = p.bias_b == 1 ? 0 : b;
      const int bhb = p.bias_h == 1 ? 0 : hq;
      brow0 = p.bias + (static_cast<size_t>(bb) * p.bias_h + bhb) * p.Sq * static_cast<size_t>(p.Sk);
    }
    for (int r0 = row_lo; r0 < p.Sq; r0 += RT) {
      __syncthreads();
      for (int e = tid; e < RT * G; e += THREADS) {
        const int r = e / G, c = e - (e / G) * G;
        const bool in = r0 + r < p.Sq;
        const size_t idx = (bh * p.Sq + (in ? r0 + r : 0)) * G + c;
        qs[r][c] = in ? load4<DT>(q, idx, nq4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
        gs[r][c] = in ? load4<DT>(dout, idx, nq4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
      if (tid < RT) {
        const bool in = r0 + tid < p.Sq && in_bounds(st, static_cast<int64_t>(bh * p.Sq + r0 + tid), nrows);
        ls[tid] = in ? lse2[bh * p.Sq + r0 + tid] : -INFINITY;
        dss[tid] = in ? dsum[bh * p.Sq + r0 + tid] : 0.f;
      }
      __syncthreads();
#pragma unroll 2
      for (int r = 0; r < RT; ++r) {
        const int i = r0 + r;
        float sd = 0.f, pd = 0.f;
#pragma unroll
        for (int c = 0; c < GPT; ++c) {
          sd = dot4(qs[r][part + 4 * c], kr[c], sd);
          pd = dot4(gs[r][part + 4 * c], vr[c], pd);
        }
        sd += __shfl_xor_sync(0xffffffffu, sd, 1);
        sd += __shfl_xor_sync(0xffffffffu, sd, 2);
        pd += __shfl_xor_sync(0xffffffffu, pd, 1);
        pd += __shfl_xor_sync(0xffffffffu, pd, 2);
        const float l2 = ls[r];
        const bool vis = key_ok && i < p.Sq && key < lim && (!p.causal || key <= i + diag) && l2 != -INFINITY;
        float x = sd * p.scale_log2 - l2;
        if constexpr (BIAS) {
          const int64_t bi = (brow0 - p.bias) + static_cast<int64_t>(i) * p.Sk + key;
          if (vis && in_bounds(st, bi, nbias)) x = fmaf(__ldg(p.bias + bi), LOG2E, x);
        }
        const float pr = vis ? fast_exp2(x) : 0.f;
        const float ds = pr * (pd - dss[r]);
#pragma unroll
        for (int c = 0; c < GPT; ++c) {
          dva[c] = axpy4(pr, gs[r][part + 4 * c], dva[c]);
          dka[c] = axpy4(ds, qs[r][part + 4 * c], dka[c]);
        }
      }
    }
  }
  if (!key_ok) return;
#pragma unroll
  for (int c = 0; c < GPT; ++c) {
    const float4 a = dka[c];
    store4<DT>(dk, kvrow + part + 4 * c, nk4, st, make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale));
    store4<DT>(dv, kvrow + part + 4 * c, nk4, st, dva[c]);
  }
}

// dq: CTA = 64 query rows of one (b, hq); keys streamed 32 at a time.
template <int D, int DT, bool BIAS>
__global__ void __launch_bounds__(THREADS) dq_kernel(const void* __restrict__ q,
                                                     const void* __restrict__ k,
                                                     const void* __restrict__ v,
                                                     const void* __restrict__ dout,
                                                     const float* __restrict__ dsum,
                                                     const float* __restrict__ lse2,
                                                     void* __restrict__ dq, const KernelParams p,
                                                     float scale) {
  constexpr int G = D / 4;
  constexpr int GPT = G / 4;
  __shared__ float4 ks[RT][G];
  __shared__ float4 vs[RT][G];

  const int tid = threadIdx.x, part = tid & 3, rl = tid >> 2;
  const int bh = blockIdx.x;
  const int b = bh / p.Hq, hq = bh - b * p.Hq;
  const int bhk = b * p.Hkv + hq / p.group;
  const int q0 = blockIdx.y * ROWS;
  const int i = q0 + rl;
  const bool row_ok = i < p.Sq;
  int lim = p.Sk;
  if (p.padding) {
    const int L = __ldg(p.kv_lens + b);
    lim = L < 0 ? 0 : (L > p.Sk ? p.Sk : L);
  }
  const int diag = p.Sk - p.Sq;
  int hi = lim;
  if (p.causal) hi = min(hi, min(q0 + ROWS - 1, p.Sq - 1) + diag + 1);
  // extents (float4 groups, rows, elements) for the bounds-checked build
  int* const st = p.status;
  const size_t nq4 = static_cast<size_t>(p.B) * p.Hq * p.Sq * G, nk4 = static_cast<size_t>(p.B) * p.Hkv * p.Sk * G;
  const int64_t nrows = static_cast<int64_t>(p.B) * p.Hq * p.Sq;
  const int64_t nbias = static_cast<int64_t>(p.bias_b) * p.bias_h * p.Sq * p.Sk;

  const size_t qrow = (static_cast<size_t>(bh) * p.Sq + (row_ok ? i : 0)) * G;
  float4 qr[GPT], gr[GPT], acc[GPT];
#pragma unroll
  for (int c = 0; c < GPT; ++c) {
    qr[c] = row_ok ? load4<DT>(q, qrow + part + 4 * c, nq4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
    gr[c] = row_ok ? load4<DT>(dout, qrow + part + 4 * c, nq4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
    acc[c] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const bool stat_ok = row_ok && in_bounds(st, static_cast<int64_t>(bh) * p.Sq + i, nrows);
  const float l2 = stat_ok ? lse2[static_cast<size_t>(bh) * p.Sq + i] : -INFINITY;
  const float dsi = stat_ok ? dsum[static_cast<size_t>(bh) * p.Sq + i] : 0.f;
  const float* brow = nullptr;
  if constexpr (BIAS) {
    if (row_ok) {
      const int bb = p.bias_b == 1 ? 0 : b;
      const int bhb = p.bias_h == 1 ? 0 : hq;
      brow = p.bias + ((static_cast<size_t>(bb) * p.bias_h + bhb) * p.Sq + i) * static_cast<size_t>(p.Sk);
    }
  }
  const int causal_lim = p.causal ? i + diag : 0x7fffffff;
  const bool live = row_ok && l2 != -INFINITY;

  for (int key0 = 0; key0 < hi; key0 += RT) {
    __syncthreads();
    for (int e = tid; e < RT * G; e += THREADS) {
      const int r = e / G, c = e - (e / G) * G;
      const bool in = key0 + r < hi;
      const size_t idx = (static_cast<size_t>(bhk) * p.Sk + (in ? key0 + r : 0)) * G + c;
      ks[r][c] = in ? load4<DT>(k, idx, nk4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
      vs[r][c] = in ? load4<DT>(v, idx, nk4, st) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
#pragma unroll 2
    for (int c2 = 0; c2 < RT; ++c2) {
      const int key = key0 + c2;
      float sd = 0.f, pd = 0.f;
#pragma unroll
      for (int c = 0; c < GPT; ++c) {
        sd = dot4(qr[c], ks[c2][part + 4 * c], sd);
        pd = dot4(gr[c], vs[c2][part + 4 * c], pd);
      }
      sd += __shfl_xor_sync(0xffffffffu, sd, 1);
      sd += __shfl_xor_sync(0xffffffffu, sd, 2);
      pd += __shfl_xor_sync(0xffffffffu, pd, 1);
      pd += __shfl_xor_sync(0xffffffffu, pd, 2);
      const bool vis = live && key < lim && key <= causal_lim;
      float x = sd * p.scale_log2 - l2;
      if constexpr (BIAS) {
        if (vis && in_bounds(st, (brow - p.bias) + key, nbias)) x = fmaf(__ldg(brow + key), LOG2E, x);
      }
      const float pr = vis ? fast_exp2(x) : 0.f;
      const float ds = pr * (pd - dsi);
#pragma unroll
      for (int c = 0; c < GPT; ++c) acc[c] = axpy4(ds, ks[c2][part + 4 * c], acc[c]);
    }
  }
  if (!row_ok) return;
#pragma unroll
  for (int c = 0; c < GPT; ++c) {
    const float4 a = acc[c];
    store4<DT>(dq, qrow + part + 4 * c, nq4, st, make_float4(a.x * scale, a.y * scale, a.z * scale, a.w * scale));
  }
}

template <int D, int DT>
static cudaError_t launch_d(const KernelParams& p, const void* q, const void* k, const void* v,
                            const void* out, const void* dout, const float* lse, float* dsum,
                            float* lse2, void* dq, void* dk, void* dv, float scale,
                            cudaStream_t st) {
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.Sq;
  cudaError_t e = launch_bwd_preprocess(D, DT, out, dout, lse, dsum, lse2, rows, st, p.status);
  if (e != cudaSuccess) return e;
  const dim3 g_kv(static_cast<unsigned>(p.B) * p.Hkv, static_cast<unsigned>((p.Sk + ROWS - 1) / ROWS));
  const dim3 g_q(static_cast<unsigned>(p.B) * p.Hq, static_cast<unsigned>((p.Sq + ROWS - 1) / ROWS));
  if (p.bias) {
    dkdv_kernel<D, DT, true><<<g_kv, THREADS, 0, st>>>(q, k, v, dout, dsum, lse2, dk, dv, p, scale);
    dq_kernel<D, DT, true><<<g_q, THREADS, 0, st>>>(q, k, v, dout, dsum, lse2, dq, p, scale);
  } else {
    dkdv_kernel<D, DT, false><<<g_kv, THREADS, 0, st>>>(q, k, v, dout, dsum, lse2, dk, dv, p, scale);
    dq_kernel<D, DT, false><<<g_q, THREADS, 0, st>>>(q, k, v, dout, dsum, lse2, dq, p, scale);
  }
  return cudaGetLastError();
}

template <int DT>
static cudaError_t launch_dt(int D, const KernelParams& p, const void* q, const void* k,
                             const void* v, const void* out, const void* dout, const float* lse,
                             float* dsum, float* lse2, void* dq, void* dk, void* dv, float scale,
                             cudaStream_t st, int* unsupported) {
  switch (D) {
    case 16: return launch_d<16, DT>(p, q, k, v, out, dout, lse, dsum, lse2, dq, dk, dv, scale, st);
    case 32: return launch_d<32, DT>(p, q, k, v, out, dout, lse, dsum, lse2, dq, dk, dv, scale, st);
    case 64: return launch_d<64, DT>(p, q, k, v, out, dout, lse, dsum, lse2, dq, dk, dv, scale, st);
    case 128: return launch_d<128, DT>(p, q, k, v, out, dout, lse, dsum, lse2, dq, dk, dv, scale, st);
    default: *unsupported = 1; return cudaSuccess;
  }
}

}  // namespace bwd

// D_i = dout_i . o_i and lse_i in log2 units (the paged backward's row
// statistics kernel: rows of D elements, 16-byte loads, D_i = 0 for a row
// with no visible key).
cudaError_t launch_bwd_preprocess(int D, int dtype, const void* out, const void* dout, const float* lse,
                                  float* dsum, float* lse2, int64_t rows, cudaStream_t st, int* status) {
  if (!(D == 16 || D == 32 || D == 64 || D == 128)) return cudaErrorInvalidValue;
  const pbwd::Buffers b{dsum, lse2, nullptr, nullptr, nullptr, nullptr};
  return pbwd::launch_preprocess(dtype, D, out, dout, lse, b, rows, st, status);
}

cudaError_t launch_bwd_simt(int D, int dtype, const KernelParams& p, const void* q, const void* k,
                            const void* v, const void* out, const void* dout, const float* lse,
                            float* dsum, float* lse2, void* dq, void* dk, void* dv, float scale,
                            cudaStream_t stream, int* unsupported) {
  *unsupported = 0;
  if (dtype == 0)
    return bwd::launch_dt<0>(D, p, q, k, v, out, dout, lse, dsum, lse2, dq, dk, dv, scale, stream, unsupported);
  if (dtype == 1)
    return bwd::launch_dt<1>(D, p, q, k, v, out, dout, lse, dsum, lse2, dq, dk, dv, scale, stream, unsupported);
  return bwd::launch_dt<2>(D, p, q, k, v, out, dout, lse, dsum, lse2, dq, dk, dv, scale, stream, unsupported);
}

}  // namespace attn
