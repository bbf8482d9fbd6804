// attn_noalloc.cu - attn_fwd_split_noalloc: split-KV attention whose scratch
// lives in a fixed array inside the library instead of a caller workspace.
//
// Some callers cannot call cudaMalloc: plugin code that its host application
// hands device buffers for inputs and outputs but no allocator, or services
// that allow no device allocation after start-up because cudaMalloc and
// cudaFree can block and synchronise the whole device. They still want the
// split-KV path, which needs scratch for its partial results. This entry
// point takes that scratch from g_split_scratch, a file-scope device array of
// ATTN_NOALLOC_SCRATCH_BYTES that every GPU loading the library holds until
// the process exits, and allocates nothing itself.
#include <mutex>

#include "attn.h"
#include "params.h"

namespace {

constexpr size_t kScratchBytes = ATTN_NOALLOC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch of every attn_fwd_split_noalloc call on a device. The split
// kernel writes every partial (O, m, l) the merge kernel reads before it is
// read, so nothing has to be cleared between calls; a split CTA whose bounded
// wait expired writes (m = +inf, l = NaN) for its rows, which the merge turns
// into NaN rows, so another call's partials never pass as a result.
static __device__ __align__(256) unsigned char g_split_scratch[kScratchBytes];

// In host code g_split_scratch names a host-side shadow, not device memory:
// the device address comes from cudaGetSymbolAddress, called while the device
// is current. It is cached per device together with the id of the CUDA
// context it was looked up in; a later call in another context (after a
// device or primary-context reset, which reloads the module and may move the
// array) looks it up again. A failed lookup is not cached: the next call
// retries, and the error is recorded for attn_last_cuda_error().
struct ScratchState {
  std::mutex mu;
  unsigned long long ctx_id = 0;
  void* ptr = nullptr;
};
ScratchState g_scratch[kMaxDevices];

int scratch_ptr(int dev, void** out) {
  if (dev < 0 || dev >= kMaxDevices) return attn::record_cuda_error(cudaErrorInvalidDevice);
  ScratchState& st = g_scratch[dev];
  unsigned long long id = attn::current_context_id();
  std::lock_guard<std::mutex> lock(st.mu);
  if (st.ptr != nullptr && id != 0 && st.ctx_id == id) {
    *out = st.ptr;
    return ATTN_OK;
  }
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_split_scratch);
  if (e != cudaSuccess || p == nullptr)
    return attn::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
  if (id == 0) id = attn::current_context_id();  // the lookup may have made the context current
  st.ptr = p;
  st.ctx_id = id;
  *out = p;
  return ATTN_OK;
}

}  // namespace

extern "C" int attn_fwd_split_noalloc(const attn_shape_t* shape, const void* q, const void* k,
                                      const void* v, int mask_kind, const int32_t* kv_lens,
                                      const float* bias, float scale, attn_dtype_t dtype,
                                      int num_splits, void* out, float* lse, void* stream) {
  if (!shape) return ATTN_ERR_NULL;
  size_t need = 0;
  const int rc = attn_split_workspace_bytes(shape, num_splits, &need);
  if (rc != ATTN_OK) return rc;
  if (need > kScratchBytes) return ATTN_ERR_SCRATCH;
  if (need == 0)  // one split: no scratch at all
    return attn_fwd_split(shape, q, k, v, mask_kind, kv_lens, bias, scale, dtype, num_splits,
                          nullptr, 0, out, lse, stream);
  int dev = 0;
  const cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn::record_cuda_error(e);
  void* ws = nullptr;
  const int sr = scratch_ptr(dev, &ws);
  if (sr != ATTN_OK) return sr;
  return attn_fwd_split(shape, q, k, v, mask_kind, kv_lens, bias, scale, dtype, num_splits, ws,
                        kScratchBytes, out, lse, stream);
}
