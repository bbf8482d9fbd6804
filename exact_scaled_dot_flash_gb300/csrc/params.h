// params.h - per-launch scalar parameters shared by the host launcher and the
// kernels (internal to libattn.so; not part of the C ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace attn {

struct KernelParams {
  int B, Hq, Hkv, Sq, Sk;
  int group;              // Hq / Hkv: query heads per key/value head
  int causal;             // bottom-right causal mask
  int padding;            // key-padding mask from kv_lens
  const int32_t* kv_lens; // [B] or nullptr
  const float* bias;      // [bias_b, bias_h, Sq, Sk] or nullptr
  int bias_b, bias_h;
  int bias_vec4;          // bias rows may be read as float4
  float scale_log2;       // scale * log2(e): scores are kept in the log2 domain
  int* status;            // device status word (STATUS_* bits)
  int device;             // CUDA device the launch runs on
};

// cuTensorMapEncodeTiled, resolved at run time through the runtime's
// driver entry-point query (no link-time dependency on libcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

namespace tc {
// How the additive bias reaches the softmax: none; read by each thread from
// global memory; or staged by TMA through a shared-memory ring (D <= 64).
constexpr int BIAS_NONE = 0, BIAS_DIRECT = 1, BIAS_STAGED = 2;
template <int D, bool BF16, int BMODE>
cudaError_t launch_tc_instance(EncodeTiledFn enc, const void* q, const void* k, const void* v,
                               void* out, const KernelParams& p, cudaStream_t stream);
}  // namespace tc

// Launchers. Return a cudaError_t; *unsupported is set when D has no kernel.
cudaError_t launch_f32(int D, bool has_bias, const KernelParams& p, const float* q,
                       const float* k, const float* v, float* out, cudaStream_t stream,
                       int* unsupported);
cudaError_t launch_nan_fill(void* out, int64_t count, int elem_bytes, cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(int* status, unsigned long long limit_ns,
                                      cudaStream_t stream);

}  // namespace attn
