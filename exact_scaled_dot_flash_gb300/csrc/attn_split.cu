// attn_split.cu - the merge step of split-KV attention, and a float fill.
//
// Split-KV follows the ruDNN user guide, section 9: the key history is split,
// each part keeps FP32 partial statistics, and the parts are merged. Part s of
// row r holds its running maximum m_s (log2 units), its sum
// l_s = sum_j 2^(x_j - m_s) and its unnormalised output
// O_s = sum_j 2^(x_j - m_s) V_j over the keys j it saw (x_j the log2-domain
// score). With M = max_s m_s and w_s = 2^(m_s - M) (0 for an empty part):
//   O = sum_s w_s O_s / sum_s w_s l_s,   lse = (M + log2 sum_s w_s l_s) ln 2,
// which is the softmax over the union of the parts. A row whose parts are all
// empty has no visible key: O is NaN and lse is -inf. A part whose kernel gave
// up on a bounded wait stores m = +inf, l = NaN, which makes O and lse NaN.
#include "params.h"
#include "ptx.cuh"

namespace attn {
namespace split {

constexpr float LN2 = 0.6931471805599453f;

// One thread per (row, group of 4 output columns); the (m, l) pairs of a row
// are read by all its threads (same address within a warp: one transaction).
template <int D, int DT>
__global__ void __launch_bounds__(256) merge_kernel(const KernelParams p, void* out) {
  constexpr int G = D / 4;
  const int64_t rows = static_cast<int64_t>(p.B) * p.Hq * p.Sq;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= rows * G) return;
  const int64_t r = idx / G;
  const int g = static_cast<int>(idx - r * G);
  const int ns = p.num_splits;
  // the bounds-checked build tests every workspace, output and lse index
  if (!range_in_bounds(p.status, (static_cast<int64_t>(ns) - 1) * rows + r, 1, ns * rows)) return;
  float M = -INFINITY;
  for (int s = 0; s < ns; ++s) M = fmaxf(M, p.ws_ml[s * rows + r].x);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float L = 0.f;
  if (M != -INFINITY) {
    const float4* wo = reinterpret_cast<const float4*>(p.ws_o);
    for (int s = 0; s < ns; ++s) {
      const float2 ml = p.ws_ml[s * rows + r];
      const float w = exp2f(ml.x - M);  // 0 for an empty part (m = -inf)
      if (w == 0.f) continue;
      L = fmaf(w, ml.y, L);
      const float4 o = wo[(s * rows + r) * G + g];
      acc.x = fmaf(w, o.x, acc.x);
      acc.y = fmaf(w, o.y, acc.y);
      acc.z = fmaf(w, o.z, acc.z);
      acc.w = fmaf(w, o.w, acc.w);
    }
  }
  const float inv = L > 0.f ? 1.f / L : __int_as_float(0x7fc00000);
  acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
  if (!in_bounds(p.status, r * G + g, rows * G)) return;
  if constexpr (DT == 0) {
    reinterpret_cast<float4*>(out)[r * G + g] = acc;
  } else {
    constexpr bool BF16 = DT == 2;
    reinterpret_cast<uint2*>(out)[r * G + g] =
        make_uint2(pack2<BF16>(acc.x, acc.y), pack2<BF16>(acc.z, acc.w));
  }
  // L is NaN only when a part reported a failed kernel wait (m = +inf, l = NaN)
  if (g == 0 && p.lse != nullptr)
    p.lse[r] = L > 0.f ? (M + log2f(L)) * LN2 : (L == 0.f ? -INFINITY : __int_as_float(0x7fc00000));
}

__global__ void fill_kernel(float* out, int64_t count, float value) {
  const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < count; i += stride)
    out[i] = value;
}

template <int D>
static cudaError_t launch_d(const KernelParams& p, int dtype, void* out, cudaStream_t stream) {
  const int64_t threads_total = static_cast<int64_t>(p.B) * p.Hq * p.Sq * (D / 4);
  const int64_t blocks = (threads_total + 255) / 256;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned nb = static_cast<unsigned>(blocks);
  if (dtype == 0) merge_kernel<D, 0><<<nb, 256, 0, stream>>>(p, out);
  else if (dtype == 1) merge_kernel<D, 1><<<nb, 256, 0, stream>>>(p, out);
  else merge_kernel<D, 2><<<nb, 256, 0, stream>>>(p, out);
  return cudaGetLastError();
}

}  // namespace split

cudaError_t launch_split_merge(const KernelParams& p, int D, int dtype, void* out,
                               cudaStream_t stream) {
  switch (D) {
    case 16: return split::launch_d<16>(p, dtype, out, stream);
    case 32: return split::launch_d<32>(p, dtype, out, stream);
    case 64: return split::launch_d<64>(p, dtype, out, stream);
    case 128: return split::launch_d<128>(p, dtype, out, stream);
    case 256: return split::launch_d<256>(p, dtype, out, stream);
    case 512: return split::launch_d<512>(p, dtype, out, stream);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_f32_fill(float* out, int64_t count, float value, cudaStream_t stream) {
  if (count <= 0) return cudaSuccess;
  int64_t blocks = (count + 255) / 256;
  if (blocks > 4096) blocks = 4096;
  split::fill_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(out, count, value);
  return cudaGetLastError();
}

}  // namespace attn
