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
  // Split-KV: the visible key range of every work item is cut into
  // num_splits contiguous parts, one CTA each. With num_splits == 1 the
  // kernel writes O (and lse, when set) itself; otherwise it writes the
  // unnormalised partial output and its (m, l) statistics, and
  // launch_split_merge combines them.
  int num_splits;
  float* ws_o;            // [num_splits, B*Hq, Sq, D] fp32 partial O (relative to m)
  float2* ws_ml;          // [num_splits, B*Hq, Sq] (m in log2 units, l)
  float* lse;             // [B*Hq*Sq] natural-log row log-sum-exp, or nullptr
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
// What the epilogue writes: O; O and the row log-sum-exp; or, for split-KV
// (p.num_splits > 1), the unnormalised partials for launch_split_merge.
constexpr int EPI_O = 0, EPI_O_LSE = 1, EPI_PARTIAL = 2;
template <int D, bool BF16, int BMODE, int EPI>
cudaError_t launch_tc_instance(EncodeTiledFn enc, const void* q, const void* k, const void* v,
                               void* out, const KernelParams& p, cudaStream_t stream);
}  // namespace tc

// Launchers. Return a cudaError_t; *unsupported is set when D has no kernel.
cudaError_t launch_f32(int D, bool has_bias, const KernelParams& p, const float* q,
                       const float* k, const float* v, float* out, cudaStream_t stream,
                       int* unsupported);
cudaError_t launch_nan_fill(void* out, int64_t count, int elem_bytes, cudaStream_t stream);
cudaError_t launch_f32_fill(float* out, int64_t count, float value, cudaStream_t stream);
// Arguments of the backward kernels beyond KernelParams.
struct BwdArgs {
  const float* lse2;  // [B*Hq*Sq] row log-sum-exp in log2 units
  const float* dsum;  // [B*Hq*Sq] D_i = dout_i . o_i
  void* dq;
  void* dk;
  void* dv;
  float scale;        // natural scale (dk and dq are scaled by it)
};
namespace bwdtc {
// Tensor-core backward (F16/BF16, D in {64, 128}): dk/dv then dq; the
// preprocess (launch_bwd_preprocess) must have filled lse2 and dsum.
template <int D, bool BF16, bool BIAS>
cudaError_t launch_bwd_tc_instance(EncodeTiledFn enc, const void* q, const void* k, const void* v,
                                   const void* dout, const KernelParams& p, const BwdArgs& a,
                                   cudaStream_t stream);
}  // namespace bwdtc
cudaError_t launch_bwd_preprocess(int D, int dtype, const void* out, const void* dout, const float* lse,
                                  float* dsum, float* lse2, int64_t rows, cudaStream_t stream,
                                  int* status = nullptr);

// Paged key/value cache with packed variable-length queries.
struct PagedParams {
  int num_seqs, num_queries, Hq, Hkv, page_size, num_pages, max_pages, max_queries;
  const int32_t* block_table;  // [num_seqs, max_pages] physical page of each key block
  const int32_t* seq_lens;     // [num_seqs] keys of each sequence
  const int32_t* q_offsets;    // [num_seqs + 1] query rows of sequence s: [q_offsets[s], q_offsets[s+1])
  const int32_t* positions;    // [num_queries] absolute positions, or nullptr (the newest tokens)
  int causal;
  float scale_log2;
  int* status;
  int device;
  // decode-shaped paged calls and tensor-core MLA: key-range splits, each
  // writing an unnormalised partial (rows r = query * Hq + head) that
  // launch_split_merge combines
  int num_splits;
  float* ws_o;    // [num_splits, num_queries * Hq, D] (D = R for MLA)
  float2* ws_ml;  // [num_splits, num_queries * Hq] (m in log2 units, l)
};
namespace pagedtc {
// Tensor-core paged kernel (F16/BF16, D in {64, 128}, page_size a multiple of
// 8 dividing 128 or a multiple of 128); splits by pp.num_splits.
template <int D, bool BF16>
cudaError_t launch_paged_tc(EncodeTiledFn enc, const PagedParams& pp, const void* q, const void* k, const void* v,
                            void* out, float* lse, cudaStream_t stream);
}  // namespace pagedtc
// True for decode-shaped attn_paged_fwd calls (the only ones that split).
inline bool paged_is_decode(int max_queries, int group) { return static_cast<long long>(max_queries) * group <= 8; }
// MLA over a paged latent cache (PagedParams with Hq = heads, Hkv = 1).
namespace mlatc {
// Tensor-core MLA (F16/BF16, R in {256, 512}, Pd in {0, 64}, page_size a
// multiple of 8 dividing 64 or a multiple of 64); splits by pp.num_splits.
template <int R, int PD, bool BF16>
cudaError_t launch_mla_tc(EncodeTiledFn enc, const PagedParams& pp, const void* q, const void* qp, const void* lat,
                          const void* kp, void* out, float* lse, cudaStream_t stream);
}  // namespace mlatc
cudaError_t launch_mla_simt(int R, int Pd, int dtype, const PagedParams& pp, const void* q, const void* qp,
                            const void* lat, const void* kp, void* out, float* lse, cudaStream_t stream,
                            int* unsupported);
cudaError_t launch_paged_simt(int D, int dtype, const PagedParams& pp, const void* q, const void* k,
                              const void* v, void* out, float* lse, cudaStream_t stream, int* unsupported);

// Backward, fp32 FMA path for every dtype (dtype: 0 f32, 1 f16, 2 bf16): the
// preprocess (dsum = rowsum(dout * out), lse2 = lse * log2 e), then dk/dv and dq.
cudaError_t launch_bwd_simt(int D, int dtype, const KernelParams& p, const void* q, const void* k,
                            const void* v, const void* out, const void* dout, const float* lse,
                            float* dsum, float* lse2, void* dq, void* dk, void* dv, float scale,
                            cudaStream_t stream, int* unsupported);
// O[r,:] = sum_s 2^(m_s - M) O_s[r,:] / sum_s 2^(m_s - M) l_s,  M = max_s m_s;
// lse[r] = (M + log2 sum_s 2^(m_s - M) l_s) ln 2.  dtype: 0 f32, 1 f16, 2 bf16.
cudaError_t launch_split_merge(const KernelParams& p, int D, int dtype, void* out,
                               cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(int* status, unsigned long long limit_ns,
                                      cudaStream_t stream);
// Records a failed CUDA call for attn_last_cuda_error(); returns ATTN_ERR_CUDA.
int record_cuda_error(cudaError_t e);
// Unique id of the calling thread's current CUDA context, 0 if there is none.
// Caches of device addresses are keyed on it: a device reset reloads the
// module and may move every __device__ variable.
unsigned long long current_context_id();

}  // namespace attn
