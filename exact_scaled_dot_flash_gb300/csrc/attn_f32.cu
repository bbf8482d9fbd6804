// attn_f32.cu - exact attention forward for F32 inputs: fp32 FMA throughout
// (no TF32 tensor cores, whose 10-bit mantissa would miss an fp32-level
// tolerance), same tiled online-softmax algorithm as the tensor-core path.
//
// CTA = 64 query rows of one (batch, query head), 256 threads; a quad of 4
// threads owns one row: each thread holds a quarter of q and of the output
// accumulator (float4 groups g with g % 4 == part, so a warp's shared-memory
// reads of a K/V row hit 4 distinct 16-byte words, broadcast across rows).
// Keys stream through shared memory 32 at a time; for each key tile every
// thread computes its quad's 32 scores (partial dot products reduced with two
// xor shuffles), keeps the running max m and sum l in the log2 domain, and
// rescales its accumulator when m grows.
// Split-KV (blockIdx.z = split): the CTA's visible key range is cut into
// num_splits runs of whole key tiles; a split CTA writes its unnormalised
// accumulator and (m, l) to the workspace for the merge kernel.
#include "params.h"
#include "ptx.cuh"

namespace attn {
namespace f32 {

constexpr int ROWS = 64;
constexpr int THREADS = 256;
constexpr int KT = 32;  // keys per shared-memory tile
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

template <int D, bool BIAS>
__global__ void __launch_bounds__(THREADS)
    attn_fwd_f32_kernel(const float* __restrict__ q, const float* __restrict__ k,
                        const float* __restrict__ v, float* __restrict__ out,
                        const KernelParams p) {
  static_assert(D % 16 == 0 && D <= 128, "head dim");
  constexpr int G = D / 4;       // float4 groups per row
  constexpr int GPT = G / 4;     // groups per thread
  __shared__ float4 ks[KT][G];
  __shared__ float4 vs[KT][G];

  const int tid = threadIdx.x;
  const int part = tid & 3;
  const int row = tid >> 2;
  const int bh = blockIdx.x;
  const int b = bh / p.Hq;
  const int hq = bh - b * p.Hq;
  const int bhk = b * p.Hkv + hq / p.group;
  const int q0 = blockIdx.y * ROWS;
  const int row_g = q0 + row;
  const bool row_ok = row_g < p.Sq;

  int key_lim = p.Sk;
  if (p.padding) {
    const int L = __ldg(p.kv_lens + b);
    key_lim = L < 0 ? 0 : (L > p.Sk ? p.Sk : L);
  }
  const int diag = p.Sk - p.Sq;
  int hi = key_lim;  // keys any row of this CTA may see
  if (p.causal) hi = min(hi, min(q0 + ROWS - 1, p.Sq - 1) + diag + 1);
  const int causal_lim = p.causal ? row_g + diag : 0x7fffffff;
  // this split's keys: whole tiles [klo, khi) of the CTA's range [0, hi)
  int klo = 0, khi = hi;
  if (p.num_splits > 1) {
    const int64_t nt = hi > 0 ? (hi + KT - 1) / KT : 0;
    const int64_t split = blockIdx.z;
    klo = static_cast<int>(split * nt / p.num_splits) * KT;
    khi = min(hi, static_cast<int>((split + 1) * nt / p.num_splits) * KT);
  }

  float4 qr[GPT], acc[GPT];
  const float4* qrow = reinterpret_cast<const float4*>(q + ((size_t)bh * p.Sq + row_g) * D);
#pragma unroll
  for (int i = 0; i < GPT; ++i) {
    qr[i] = row_ok ? __ldg(qrow + part + 4 * i) : make_float4(0.f, 0.f, 0.f, 0.f);
    acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  const float* brow = nullptr;
  if constexpr (BIAS) {
    if (row_ok) {
      const int bb = p.bias_b == 1 ? 0 : b;
      const int bhh = p.bias_h == 1 ? 0 : hq;
      brow = p.bias + (((size_t)bb * p.bias_h + bhh) * p.Sq + row_g) * (size_t)p.Sk;
    }
  }
  const float4* kh = reinterpret_cast<const float4*>(k + (size_t)bhk * p.Sk * D);
  const float4* vh = reinterpret_cast<const float4*>(v + (size_t)bhk * p.Sk * D);

  float m_run = -INFINITY, l_run = 0.f;
  for (int key0 = klo; key0 < khi; key0 += KT) {
    __syncthreads();
    for (int e = tid; e < KT * G; e += THREADS) {
      const int r = e / G, g = e - (e / G) * G;
      const bool in = key0 + r < khi;
      ks[r][g] = in ? __ldg(kh + (size_t)(key0 + r) * G + g) : make_float4(0.f, 0.f, 0.f, 0.f);
      vs[r][g] = in ? __ldg(vh + (size_t)(key0 + r) * G + g) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    __syncthreads();
    float s[KT];
#pragma unroll
    for (int c = 0; c < KT; ++c) {
      float d = 0.f;
#pragma unroll
      for (int i = 0; i < GPT; ++i) {
        const float4 kk = ks[c][part + 4 * i];
        d = fmaf(qr[i].x, kk.x, d);
        d = fmaf(qr[i].y, kk.y, d);
        d = fmaf(qr[i].z, kk.z, d);
        d = fmaf(qr[i].w, kk.w, d);
      }
      d += __shfl_xor_sync(0xffffffffu, d, 1);
      d += __shfl_xor_sync(0xffffffffu, d, 2);
      const int key = key0 + c;
      float x = d * p.scale_log2;
      if constexpr (BIAS) {
        if (brow != nullptr && key < key_lim) x = fmaf(__ldg(brow + key), LOG2E, x);
      }
      s[c] = (key >= key_lim || key > causal_lim) ? -INFINITY : x;
    }
    float mx = s[0];
#pragma unroll
    for (int c = 1; c < KT; ++c) mx = fmaxf(mx, s[c]);
    const float m_new = fmaxf(m_run, mx);
    const float m_use = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = fast_exp2(m_run - m_use);
    float sum = 0.f;
#pragma unroll
    for (int c = 0; c < KT; ++c) {
      s[c] = fast_exp2(s[c] - m_use);
      sum += s[c];
    }
    l_run = l_run * alpha + sum;
    m_run = m_new;
#pragma unroll
    for (int i = 0; i < GPT; ++i) {
      float4 a = acc[i];
      a.x *= alpha; a.y *= alpha; a.z *= alpha; a.w *= alpha;
#pragma unroll
      for (int c = 0; c < KT; ++c) {
        const float4 vv = vs[c][part + 4 * i];
        a.x = fmaf(s[c], vv.x, a.x);
        a.y = fmaf(s[c], vv.y, a.y);
        a.z = fmaf(s[c], vv.z, a.z);
        a.w = fmaf(s[c], vv.w, a.w);
      }
      acc[i] = a;
    }
  }
  if (!row_ok) return;
  const int64_t nrows = static_cast<int64_t>(p.B) * p.Hq * p.Sq;  // extent for the checked build
  if (p.num_splits > 1) {
    // partial result: accumulator relative to 2^m_run, and (m_run, l_run)
    const size_t r = (static_cast<size_t>(blockIdx.z) * p.B * p.Hq + bh) * p.Sq + row_g;
    if (!in_bounds(p.status, static_cast<int64_t>(r), p.num_splits * nrows)) return;
    float4* wrow = reinterpret_cast<float4*>(p.ws_o + r * D);
#pragma unroll
    for (int i = 0; i < GPT; ++i) wrow[part + 4 * i] = acc[i];
    if (part == 0) p.ws_ml[r] = make_float2(m_run, l_run);
    return;
  }
  if (!in_bounds(p.status, static_cast<int64_t>(bh) * p.Sq + row_g, nrows)) return;
  if (p.lse != nullptr && part == 0)
    p.lse[static_cast<size_t>(bh) * p.Sq + row_g] =
        l_run > 0.f ? (m_run + log2f(l_run)) * LN2 : -INFINITY;
  const float inv = l_run > 0.f ? 1.f / l_run : __int_as_float(0x7fc00000);
  float4* orow = reinterpret_cast<float4*>(out + ((size_t)bh * p.Sq + row_g) * D);
#pragma unroll
  for (int i = 0; i < GPT; ++i) {
    float4 a = acc[i];
    a.x *= inv; a.y *= inv; a.z *= inv; a.w *= inv;
    orow[part + 4 * i] = a;
  }
}

template <int D, bool BIAS>
static cudaError_t launch_one(const KernelParams& p, const float* q, const float* k,
                              const float* v, float* out, cudaStream_t stream) {
  dim3 grid(static_cast<unsigned>(p.B) * static_cast<unsigned>(p.Hq),
            static_cast<unsigned>((p.Sq + ROWS - 1) / ROWS), static_cast<unsigned>(p.num_splits));
  attn_fwd_f32_kernel<D, BIAS><<<grid, THREADS, 0, stream>>>(q, k, v, out, p);
  return cudaGetLastError();
}

__global__ void nan_fill_kernel(uint8_t* out, int64_t count, int elem_bytes) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride) {
    if (elem_bytes == 4)
      reinterpret_cast<uint32_t*>(out)[i] = 0x7fc00000u;
    else if (elem_bytes == 2)
      reinterpret_cast<uint16_t*>(out)[i] = 0x7e00u;  // f16 quiet NaN (bf16 uses 0x7fc0)
  }
}

__global__ void nan_fill_bf16_kernel(uint16_t* out, int64_t count) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count; i += stride)
    out[i] = 0x7fc0u;
}

}  // namespace f32

cudaError_t launch_f32(int D, bool has_bias, const KernelParams& p, const float* q,
                       const float* k, const float* v, float* out, cudaStream_t stream,
                       int* unsupported) {
  *unsupported = 0;
#define ATTN_F32_CASE(DD)                                                                    \
  case DD:                                                                                   \
    return has_bias ? f32::launch_one<DD, true>(p, q, k, v, out, stream)                     \
                    : f32::launch_one<DD, false>(p, q, k, v, out, stream);
  switch (D) {
    ATTN_F32_CASE(16)
    ATTN_F32_CASE(32)
    ATTN_F32_CASE(64)
    ATTN_F32_CASE(128)
    default:
      *unsupported = 1;
      return cudaSuccess;
  }
#undef ATTN_F32_CASE
}

// elem_bytes: 4 = f32, 2 = f16, 3 = bf16 (16-bit storage with the bf16 NaN pattern).
cudaError_t launch_nan_fill(void* out, int64_t count, int elem_bytes, cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  const int threads = 256;
  int64_t blocks = (count + threads - 1) / threads;
  if (blocks > 4096) blocks = 4096;
  if (elem_bytes == 3)
    f32::nan_fill_bf16_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        static_cast<uint16_t*>(out), count);
  else
    f32::nan_fill_kernel<<<(unsigned)blocks, threads, 0, stream>>>(static_cast<uint8_t*>(out),
                                                                   count, elem_bytes);
  return cudaGetLastError();
}

}  // namespace attn
