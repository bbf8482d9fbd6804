// simt.cuh - vector load/store and fp32 FMA helpers of the SIMT (non tensor
// core) kernels: 4 consecutive elements of an F32/F16/BF16 array as a float4.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace attn {
namespace simt {

// dtype: 0 f32, 1 f16, 2 bf16
template <int DT>
__device__ __forceinline__ float4 load4(const void* base, size_t idx4) {
  if constexpr (DT == 0) {
    return __ldg(reinterpret_cast<const float4*>(base) + idx4);
  } else {
    const uint2 u = __ldg(reinterpret_cast<const uint2*>(base) + idx4);
    float2 a, b;
    if constexpr (DT == 1) {
      a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
      b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
    } else {
      a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
    }
    return make_float4(a.x, a.y, b.x, b.y);
  }
}

// 8 consecutive elements (float4 pair idx8 of the array) with one 16-byte
// load for 16-bit types (two for F32).
template <int DT>
__device__ __forceinline__ void load8(const void* base, size_t idx8, float4& lo, float4& hi) {
  if constexpr (DT == 0) {
    lo = __ldg(reinterpret_cast<const float4*>(base) + 2 * idx8);
    hi = __ldg(reinterpret_cast<const float4*>(base) + 2 * idx8 + 1);
  } else {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(base) + idx8);
    float2 a, b, c, d;
    if constexpr (DT == 1) {
      a = __half22float2(*reinterpret_cast<const __half2*>(&u.x));
      b = __half22float2(*reinterpret_cast<const __half2*>(&u.y));
      c = __half22float2(*reinterpret_cast<const __half2*>(&u.z));
      d = __half22float2(*reinterpret_cast<const __half2*>(&u.w));
    } else {
      a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
      b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
      c = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.z));
      d = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.w));
    }
    lo = make_float4(a.x, a.y, b.x, b.y);
    hi = make_float4(c.x, c.y, d.x, d.y);
  }
}

template <int DT>
__device__ __forceinline__ void store4(void* base, size_t idx4, float4 v) {
  if constexpr (DT == 0) {
    reinterpret_cast<float4*>(base)[idx4] = v;
  } else {
    reinterpret_cast<uint2*>(base)[idx4] = make_uint2(pack2<DT == 2>(v.x, v.y), pack2<DT == 2>(v.z, v.w));
  }
}

// Bounds-checked forms (see in_bounds): n4 is the number of float4 groups in
// the array; an index outside it is recorded in *status and skipped.
template <int DT>
__device__ __forceinline__ float4 load4(const void* base, size_t idx4, size_t n4, int* status) {
  return in_bounds(status, static_cast<int64_t>(idx4), static_cast<int64_t>(n4))
             ? load4<DT>(base, idx4)
             : make_float4(0.f, 0.f, 0.f, 0.f);
}

template <int DT>
__device__ __forceinline__ void store4(void* base, size_t idx4, size_t n4, int* status, float4 v) {
  if (in_bounds(status, static_cast<int64_t>(idx4), static_cast<int64_t>(n4))) store4<DT>(base, idx4, v);
}

// idx8 counts 8-element groups; n8 is their number in the array
template <int DT>
__device__ __forceinline__ void load8(const void* base, size_t idx8, size_t n8, int* status, float4& lo,
                                      float4& hi) {
  if (in_bounds(status, static_cast<int64_t>(idx8), static_cast<int64_t>(n8))) {
    load8<DT>(base, idx8, lo, hi);
  } else {
    lo = hi = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

__device__ __forceinline__ float dot4(float4 a, float4 b, float acc) {
  acc = fmaf(a.x, b.x, acc);
  acc = fmaf(a.y, b.y, acc);
  acc = fmaf(a.z, b.z, acc);
  return fmaf(a.w, b.w, acc);
}

__device__ __forceinline__ float4 axpy4(float a, float4 x, float4 y) {
  return make_float4(fmaf(a, x.x, y.x), fmaf(a, x.y, y.y), fmaf(a, x.z, y.z), fmaf(a, x.w, y.w));
}

}  // namespace simt
}  // namespace attn
