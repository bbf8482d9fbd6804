// attn_api.cu - the C ABI of libattn.so (declared in include/attn.h):
// argument validation, per-device state, and dispatch to the kernels.
//
// Contract sources (page title, section): ruDNN user guide section 2 (the
// attention entry takes query, key, value, an optional mask and an optional
// attn_bias and returns a setup error instead of failing later) and section 9
// (contiguous F32/F16/BF16 inputs of one dtype, Hq divisible by Hkv, a finite
// positive scale); section 7 (statistics in FP32, output in the input dtype).
#include <math.h>
#include <stdint.h>

#include <initializer_list>
#include <mutex>

#include "attn.h"
#include "paged_bwd.h"
#include "params.h"

namespace {

constexpr int kVersion = 1 * 10000 + 0 * 100 + 0;
constexpr int kMaxDevices = 64;

thread_local int g_last_cuda_error = 0;

// Sticky per-device status word that kernels OR STATUS_* bits into.
__device__ int g_status_word;

// The status word's device address, per device and per CUDA context: after a
// device or primary-context reset the module is loaded again and the address
// may move, so a cached address is used only while the context it was looked
// up in is still the current one.
struct DeviceState {
  std::mutex mu;
  unsigned long long ctx_id = 0;
  int* status = nullptr;
};
DeviceState g_devices[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);
std::once_flag g_ctx_once;
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

std::once_flag g_encode_once;
attn::EncodeTiledFn g_encode = nullptr;

attn::EncodeTiledFn encode_fn() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult qres = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &qres) == cudaSuccess &&
        qres == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<attn::EncodeTiledFn>(fn);
  });
  return g_encode;
}

}  // namespace

// Unique id of the calling thread's current CUDA context (0 when there is
// none yet, or the driver cannot tell).
unsigned long long attn::current_context_id() {
  std::call_once(g_ctx_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
    fn = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess && q == cudaDriverEntryPointSuccess)
      g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(fn);
  });
  if (!g_ctx_get_current || !g_ctx_get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return 0;
  if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

namespace {

// Device address of g_status_word on the current device `dev`, looked up
// again whenever the current context differs from the one the cached address
// came from; a failed lookup is not cached (the next call retries).
int* status_ptr(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  DeviceState& st = g_devices[dev];
  unsigned long long id = attn::current_context_id();
  std::lock_guard<std::mutex> lock(st.mu);
  if (st.status != nullptr && id != 0 && st.ctx_id == id) return st.status;
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_status_word);
  if (e != cudaSuccess) {
    g_last_cuda_error = static_cast<int>(e);
    return nullptr;
  }
  if (id == 0) id = attn::current_context_id();  // the lookup may have made the context current
  st.status = static_cast<int*>(p);
  st.ctx_id = id;
  return st.status;
}

int fail_cuda(cudaError_t e) {
  g_last_cuda_error = static_cast<int>(e);
  return ATTN_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

int attn::record_cuda_error(cudaError_t e) { return fail_cuda(e); }

namespace {

bool overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  if (!a || !b || na <= 0 || nb <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

int elem_size(attn_dtype_t d) { return d == ATTN_F32 ? 4 : 2; }


// Workspace of a split-KV call: fp32 partial O [num_splits, B*Hq, Sq, D], then
// (at the next 256-byte boundary) the (m, l) float pairs [num_splits, B*Hq, Sq].
struct SplitLayout {
  int64_t o_bytes = 0, ml_offset = 0, total = 0;
};
SplitLayout split_layout(const attn_shape_t& s, int num_splits) {
  SplitLayout L;
  if (num_splits <= 1) return L;
  const int64_t rows = static_cast<int64_t>(num_splits) * s.B * s.Hq * s.Sq;
  L.o_bytes = rows * s.D * 4;
  L.ml_offset = (L.o_bytes + 255) / 256 * 256;
  L.total = L.ml_offset + rows * 8;
  return L;
}

int run(const attn_shape_t* shape, const void* q, const void* k, const void* v, int mask_kind,
        const int32_t* kv_lens, const float* bias, float scale, attn_dtype_t dtype,
        int num_splits, void* workspace, size_t workspace_bytes, void* out, float* lse,
        void* stream);

}  // namespace

extern "C" {

int attn_version(void) { return kVersion; }

int attn_last_cuda_error(void) { return g_last_cuda_error; }

const char* attn_strerror(int code) {
  switch (code) {
    case ATTN_OK: return "success";
    case ATTN_ERR_NULL: return "a required pointer is NULL";
    case ATTN_ERR_SHAPE: return "invalid shape (dims, Hq % Hkv, or bias dims)";
    case ATTN_ERR_DTYPE: return "unknown dtype";
    case ATTN_ERR_HEAD_DIM: return "head dim D has no compiled kernel for this dtype";
    case ATTN_ERR_ALIGN: return "a pointer is not 16-byte aligned";
    case ATTN_ERR_SCALE: return "scale must be finite and positive";
    case ATTN_ERR_MASK: return "invalid mask_kind, or key padding without kv_lens";
    case ATTN_ERR_OVERLAP: return "out overlaps an input";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_TIMEOUT: return "a kernel wait timed out";
    case ATTN_ERR_SPLITS: return "num_splits must be in [1, 32]";
    case ATTN_ERR_WORKSPACE: return "workspace is NULL or smaller than its *_workspace_bytes query";
    case ATTN_ERR_SCRATCH:
      return "problem needs more split scratch than ATTN_NOALLOC_SCRATCH_BYTES (use fewer splits or a workspace)";
    default: return "unknown status code";
  }
}

int attn_device_status(int device, int* flags, int clear) {
  if (!flags) return ATTN_ERR_NULL;
  int old = 0;
  cudaError_t e = cudaGetDevice(&old);
  if (e != cudaSuccess) return fail_cuda(e);
  if (device != old && (e = cudaSetDevice(device)) != cudaSuccess) return fail_cuda(e);
  int v = 0;
  e = cudaMemcpyFromSymbol(&v, g_status_word, sizeof(int));
  if (e == cudaSuccess && clear) {
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_status_word, &zero, sizeof(int));
  }
  if (device != old) cudaSetDevice(old);
  if (e != cudaSuccess) return fail_cuda(e);
  *flags = v;
  return ATTN_OK;
}

int attn_selftest_wait_timeout(unsigned int limit_us, void* stream) {
  if (limit_us == 0 || limit_us > 5000000u) return ATTN_ERR_SHAPE;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  int* st = status_ptr(dev);
  if (!st) return fail_cuda(cudaErrorInvalidDevice);
  e = attn::launch_wait_timeout_probe(st, 1000ull * limit_us, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
}

int attn_fwd(const attn_shape_t* shape, const void* q, const void* k, const void* v,
             int mask_kind, const int32_t* kv_lens, const float* bias, float scale,
             attn_dtype_t dtype, void* out, void* stream) {
  return run(shape, q, k, v, mask_kind, kv_lens, bias, scale, dtype, 1, nullptr, 0, out, nullptr,
             stream);
}

int attn_split_workspace_bytes(const attn_shape_t* shape, int num_splits, size_t* bytes) {
  if (!shape || !bytes) return ATTN_ERR_NULL;
  const attn_shape_t s = *shape;
  if (s.B < 0 || s.Sq < 0 || s.Hq <= 0 || s.D <= 0) return ATTN_ERR_SHAPE;
  if (num_splits < 1 || num_splits > ATTN_MAX_SPLITS) return ATTN_ERR_SPLITS;
  *bytes = static_cast<size_t>(split_layout(s, num_splits).total);
  return ATTN_OK;
}

int attn_fwd_split(const attn_shape_t* shape, const void* q, const void* k, const void* v,
                   int mask_kind, const int32_t* kv_lens, const float* bias, float scale,
                   attn_dtype_t dtype, int num_splits, void* workspace, size_t workspace_bytes,
                   void* out, float* lse, void* stream) {
  return run(shape, q, k, v, mask_kind, kv_lens, bias, scale, dtype, num_splits, workspace,
             workspace_bytes, out, lse, stream);
}

}  // extern "C"

namespace {

int run(const attn_shape_t* shape, const void* q, const void* k, const void* v, int mask_kind,
        const int32_t* kv_lens, const float* bias, float scale, attn_dtype_t dtype,
        int num_splits, void* workspace, size_t workspace_bytes, void* out, float* lse,
        void* stream) {
  // ---- validation: everything is checked before any CUDA call
  if (!shape) return ATTN_ERR_NULL;
  const attn_shape_t s = *shape;
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  if (s.B < 0 || s.Sq < 0 || s.Sk < 0 || s.Hq <= 0 || s.Hkv <= 0 || s.D <= 0)
    return ATTN_ERR_SHAPE;
  if (s.Hq % s.Hkv != 0) return ATTN_ERR_SHAPE;
  if (mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_KEY_PADDING)) return ATTN_ERR_MASK;
  if ((mask_kind & ATTN_MASK_KEY_PADDING) && !kv_lens) return ATTN_ERR_MASK;
  if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_SCALE;
  if (bias && !((s.bias_b == 1 || s.bias_b == s.B) && (s.bias_h == 1 || s.bias_h == s.Hq)))
    return ATTN_ERR_SHAPE;
  const bool tensor_core = dtype != ATTN_F32;
  if (tensor_core ? !(s.D == 32 || s.D == 64 || s.D == 128)
                  : !(s.D == 16 || s.D == 32 || s.D == 64 || s.D == 128))
    return ATTN_ERR_HEAD_DIM;
  // grid limits: x = B*Hq (< 2^31), y = query blocks (<= 65535)
  const int64_t bhq = static_cast<int64_t>(s.B) * s.Hq;
  const int64_t bhk = static_cast<int64_t>(s.B) * s.Hkv;
  if (bhq > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  const int rows_per_cta = tensor_core ? 256 : 64;
  if ((static_cast<int64_t>(s.Sq) + rows_per_cta - 1) / rows_per_cta > 65535) return ATTN_ERR_SHAPE;
  if (num_splits < 1 || num_splits > ATTN_MAX_SPLITS) return ATTN_ERR_SPLITS;
  if (tensor_core && bhq * ((static_cast<int64_t>(s.Sq) + 255) / 256) * num_splits > 0x7fffffffLL)
    return ATTN_ERR_SHAPE;
  if (num_splits > 1 && bhq * s.Sq * (s.D / 4) / 256 >= 0x7fffffffLL) return ATTN_ERR_SHAPE;
  if (s.B == 0 || s.Sq == 0) return ATTN_OK;  // nothing to compute
  if (!q || !out || (s.Sk > 0 && (!k || !v))) return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return ATTN_ERR_ALIGN;
  if (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) return ATTN_ERR_ALIGN;
  if (kv_lens && (reinterpret_cast<uintptr_t>(kv_lens) & 3u)) return ATTN_ERR_ALIGN;
  const int es = elem_size(dtype);
  const int64_t out_bytes = bhq * s.Sq * s.D * es;
  const int64_t kv_bytes = bhk * s.Sk * s.D * es;
  const int64_t bias_bytes =
      bias ? static_cast<int64_t>(s.bias_b) * s.bias_h * s.Sq * static_cast<int64_t>(s.Sk) * 4 : 0;
  if (overlaps(out, out_bytes, q, out_bytes) || overlaps(out, out_bytes, k, kv_bytes) ||
      overlaps(out, out_bytes, v, kv_bytes) || overlaps(out, out_bytes, bias, bias_bytes) ||
      overlaps(out, out_bytes, kv_lens, static_cast<int64_t>(s.B) * 4))
    return ATTN_ERR_OVERLAP;
  // every buffer the call writes (out, lse, workspace) is disjoint from every
  // other buffer it touches
  const int64_t lse_bytes = lse ? bhq * s.Sq * 4 : 0;
  if (lse) {
    if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_ERR_ALIGN;
    if (overlaps(lse, lse_bytes, q, out_bytes) || overlaps(lse, lse_bytes, k, kv_bytes) ||
        overlaps(lse, lse_bytes, v, kv_bytes) || overlaps(lse, lse_bytes, bias, bias_bytes) ||
        overlaps(lse, lse_bytes, kv_lens, static_cast<int64_t>(s.B) * 4) ||
        overlaps(lse, lse_bytes, out, out_bytes))
      return ATTN_ERR_OVERLAP;
  }
  const SplitLayout lay = split_layout(s, num_splits);
  if (num_splits > 1 && s.Sk > 0) {
    if (!workspace || workspace_bytes < static_cast<size_t>(lay.total)) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
    const int64_t wb = lay.total;
    if (overlaps(workspace, wb, q, out_bytes) || overlaps(workspace, wb, k, kv_bytes) ||
        overlaps(workspace, wb, v, kv_bytes) || overlaps(workspace, wb, bias, bias_bytes) ||
        overlaps(workspace, wb, kv_lens, static_cast<int64_t>(s.B) * 4) ||
        overlaps(workspace, wb, out, out_bytes) || overlaps(workspace, wb, lse, lse_bytes))
      return ATTN_ERR_OVERLAP;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (s.Sk == 0) {  // no key at all: every row is undefined
    cudaError_t e = attn::launch_nan_fill(out, bhq * s.Sq * s.D,
                                          dtype == ATTN_F32 ? 4 : (dtype == ATTN_F16 ? 2 : 3), st);
    if (e == cudaSuccess && lse) e = attn::launch_f32_fill(lse, bhq * s.Sq, -INFINITY, st);
    return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);

  attn::KernelParams p;
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.Sq = s.Sq;
  p.Sk = s.Sk;
  p.group = s.Hq / s.Hkv;
  p.causal = (mask_kind & ATTN_MASK_CAUSAL) ? 1 : 0;
  p.padding = (mask_kind & ATTN_MASK_KEY_PADDING) ? 1 : 0;
  p.kv_lens = p.padding ? kv_lens : nullptr;
  p.bias = bias;
  p.bias_b = bias ? s.bias_b : 1;
  p.bias_h = bias ? s.bias_h : 1;
  p.bias_vec4 = bias && aligned16(bias) && (s.Sk % 4 == 0);
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status_ptr(dev);
  p.device = dev;
  p.num_splits = num_splits;
  p.ws_o = num_splits > 1 ? static_cast<float*>(workspace) : nullptr;
  p.ws_ml = num_splits > 1
                ? reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + lay.ml_offset)
                : nullptr;
  p.lse = lse;
  // after the partial kernel, the merge: O and lse from the split partials
  auto finish = [&](cudaError_t err) -> int {
    if (err == cudaSuccess && num_splits > 1)
      err = attn::launch_split_merge(p, s.D, static_cast<int>(dtype), out, st);
    return err == cudaSuccess ? ATTN_OK : fail_cuda(err);
  };

  if (!tensor_core) {
    int unsupported = 0;
    e = attn::launch_f32(s.D, bias != nullptr, p, static_cast<const float*>(q),
                         static_cast<const float*>(k), static_cast<const float*>(v),
                         static_cast<float*>(out), st, &unsupported);
    if (unsupported) return ATTN_ERR_HEAD_DIM;
    return finish(e);
  }

  attn::EncodeTiledFn enc = encode_fn();
  if (!enc) return fail_cuda(cudaErrorNotSupported);
  const bool bf16 = dtype == ATTN_BF16;
  // bias: none; staged through shared memory by TMA when D <= 64 and the rows
  // allow 16-byte TMA strides; otherwise read directly by the softmax threads
  const int bmode = !bias ? 0 : ((s.D <= 64 && p.bias_vec4) ? 2 : 1);
  using namespace attn::tc;
#define ATTN_TC_CALL(DD, BB, MM)                                                                \
  (num_splits > 1 ? launch_tc_instance<DD, BB, MM, EPI_PARTIAL>(enc, q, k, v, out, p, st)      \
   : lse          ? launch_tc_instance<DD, BB, MM, EPI_O_LSE>(enc, q, k, v, out, p, st)        \
                  : launch_tc_instance<DD, BB, MM, EPI_O>(enc, q, k, v, out, p, st))
#define ATTN_TC_DISPATCH(DD, STAGED)                                                           \
  case DD:                                                                                     \
    if (bmode == 2)                                                                            \
      e = bf16 ? ATTN_TC_CALL(DD, true, STAGED) : ATTN_TC_CALL(DD, false, STAGED);             \
    else if (bmode == 1)                                                                       \
      e = bf16 ? ATTN_TC_CALL(DD, true, BIAS_DIRECT) : ATTN_TC_CALL(DD, false, BIAS_DIRECT);   \
    else                                                                                       \
      e = bf16 ? ATTN_TC_CALL(DD, true, BIAS_NONE) : ATTN_TC_CALL(DD, false, BIAS_NONE);       \
    break;
  switch (s.D) {
    ATTN_TC_DISPATCH(32, BIAS_STAGED)
    ATTN_TC_DISPATCH(64, BIAS_STAGED)
    ATTN_TC_DISPATCH(128, BIAS_DIRECT)
    default:
      return ATTN_ERR_HEAD_DIM;
  }
#undef ATTN_TC_CALL
#undef ATTN_TC_DISPATCH
  return finish(e);
}

}  // namespace

// ---------------------------------------------------------------- backward
namespace {

int64_t bwd_workspace_total(const attn_shape_t& s) {
  const int64_t rows = static_cast<int64_t>(s.B) * s.Hq * s.Sq;
  return ((rows * 4 + 255) / 256 * 256) * 2;  // D_i, then lse_i in log2 units
}

}  // namespace

extern "C" {

int attn_bwd_workspace_bytes(const attn_shape_t* shape, size_t* bytes) {
  if (!shape || !bytes) return ATTN_ERR_NULL;
  const attn_shape_t s = *shape;
  if (s.B < 0 || s.Sq < 0 || s.Hq <= 0) return ATTN_ERR_SHAPE;
  *bytes = static_cast<size_t>(bwd_workspace_total(s));
  return ATTN_OK;
}

int attn_bwd(const attn_shape_t* shape, const void* q, const void* k, const void* v,
             const void* out, const void* dout, const float* lse, int mask_kind,
             const int32_t* kv_lens, const float* bias, float scale, attn_dtype_t dtype,
             void* workspace, size_t workspace_bytes, void* dq, void* dk, void* dv,
             void* stream) {
  // ---- validation: everything is checked before any CUDA call
  if (!shape) return ATTN_ERR_NULL;
  const attn_shape_t s = *shape;
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  if (s.B < 0 || s.Sq < 0 || s.Sk < 0 || s.Hq <= 0 || s.Hkv <= 0 || s.D <= 0) return ATTN_ERR_SHAPE;
  if (s.Hq % s.Hkv != 0) return ATTN_ERR_SHAPE;
  if (mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_KEY_PADDING)) return ATTN_ERR_MASK;
  if ((mask_kind & ATTN_MASK_KEY_PADDING) && !kv_lens) return ATTN_ERR_MASK;
  if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_SCALE;
  if (bias && !((s.bias_b == 1 || s.bias_b == s.B) && (s.bias_h == 1 || s.bias_h == s.Hq)))
    return ATTN_ERR_SHAPE;
  if (!(s.D == 16 || s.D == 32 || s.D == 64 || s.D == 128)) return ATTN_ERR_HEAD_DIM;
  const int64_t bhq = static_cast<int64_t>(s.B) * s.Hq;
  const int64_t bhk = static_cast<int64_t>(s.B) * s.Hkv;
  if (bhq > 0x7fffffffLL) return ATTN_ERR_SHAPE;
  if ((static_cast<int64_t>(s.Sq) + 63) / 64 > 65535 || (static_cast<int64_t>(s.Sk) + 63) / 64 > 65535)
    return ATTN_ERR_SHAPE;
  if (s.B == 0) return ATTN_OK;
  const int es = elem_size(dtype);
  const int64_t q_bytes = bhq * s.Sq * s.D * es;
  const int64_t kv_bytes = bhk * s.Sk * s.D * es;
  const int64_t lse_bytes = bhq * s.Sq * 4;
  const int64_t bias_bytes =
      bias ? static_cast<int64_t>(s.bias_b) * s.bias_h * s.Sq * static_cast<int64_t>(s.Sk) * 4 : 0;
  const bool rows = s.Sq > 0, keys = s.Sk > 0;
  if ((rows && (!q || !out || !dout || !lse || !dq)) || (keys && (!k || !v || !dk || !dv)))
    return ATTN_ERR_NULL;
  if ((rows && (!aligned16(q) || !aligned16(out) || !aligned16(dout) || !aligned16(dq))) ||
      (keys && (!aligned16(k) || !aligned16(v) || !aligned16(dk) || !aligned16(dv))))
    return ATTN_ERR_ALIGN;
  if ((lse && (reinterpret_cast<uintptr_t>(lse) & 3u)) || (bias && (reinterpret_cast<uintptr_t>(bias) & 3u)) ||
      (kv_lens && (reinterpret_cast<uintptr_t>(kv_lens) & 3u)))
    return ATTN_ERR_ALIGN;
  const int64_t ws_need = (rows && keys) ? bwd_workspace_total(s) : 0;
  if (ws_need > 0) {
    if (!workspace || workspace_bytes < static_cast<size_t>(ws_need)) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  }
  // every buffer the call writes is disjoint from every other buffer it touches
  struct Buf { const void* p; int64_t n; };
  const Buf ins[] = {{q, q_bytes}, {k, kv_bytes}, {v, kv_bytes}, {out, q_bytes}, {dout, q_bytes},
                     {lse, lse_bytes}, {bias, bias_bytes}, {kv_lens, static_cast<int64_t>(s.B) * 4}};
  const Buf outs[] = {{dq, q_bytes}, {dk, kv_bytes}, {dv, kv_bytes}, {ws_need ? workspace : nullptr, ws_need}};
  for (int a = 0; a < 4; ++a) {
    for (const Buf& b : ins)
      if (overlaps(outs[a].p, outs[a].n, b.p, b.n)) return ATTN_ERR_OVERLAP;
    for (int c = a + 1; c < 4; ++c)
      if (overlaps(outs[a].p, outs[a].n, outs[c].p, outs[c].n)) return ATTN_ERR_OVERLAP;
  }

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (!rows || !keys) {  // no query rows: dk = dv = 0; no keys: dq = 0
    if (keys) {
      if ((e = cudaMemsetAsync(dk, 0, static_cast<size_t>(kv_bytes), st)) == cudaSuccess)
        e = cudaMemsetAsync(dv, 0, static_cast<size_t>(kv_bytes), st);
    }
    if (rows && e == cudaSuccess) e = cudaMemsetAsync(dq, 0, static_cast<size_t>(q_bytes), st);
    return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
  }
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return fail_cuda(e);
  attn::KernelParams p{};
  p.B = s.B;
  p.Hq = s.Hq;
  p.Hkv = s.Hkv;
  p.Sq = s.Sq;
  p.Sk = s.Sk;
  p.group = s.Hq / s.Hkv;
  p.causal = (mask_kind & ATTN_MASK_CAUSAL) ? 1 : 0;
  p.padding = (mask_kind & ATTN_MASK_KEY_PADDING) ? 1 : 0;
  p.kv_lens = p.padding ? kv_lens : nullptr;
  p.bias = bias;
  p.bias_b = bias ? s.bias_b : 1;
  p.bias_h = bias ? s.bias_h : 1;
  p.bias_vec4 = 0;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.status = status_ptr(dev);
  p.device = dev;
  p.num_splits = 1;
  float* dsum = static_cast<float*>(workspace);
  float* lse2 = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + ws_need / 2);
  // F16/BF16 with D in {64, 128}: tensor cores; otherwise the fp32 FMA path
  const bool tc = dtype != ATTN_F32 && (s.D == 64 || s.D == 128) && bhq <= 65535 && bhk <= 65535;
  if (tc) {
    attn::EncodeTiledFn enc = encode_fn();
    if (!enc) return fail_cuda(cudaErrorNotSupported);
    e = attn::launch_bwd_preprocess(s.D, static_cast<int>(dtype), out, dout, lse, dsum, lse2, bhq * s.Sq, st,
                                    p.status);
    if (e != cudaSuccess) return fail_cuda(e);
    attn::BwdArgs a{lse2, dsum, dq, dk, dv, scale};
    const bool bf = dtype == ATTN_BF16;
    using namespace attn::bwdtc;
#define ATTN_BWD_TC(DD, BB) \
  (bias ? launch_bwd_tc_instance<DD, BB, true>(enc, q, k, v, dout, p, a, st) \
        : launch_bwd_tc_instance<DD, BB, false>(enc, q, k, v, dout, p, a, st))
    if (s.D == 128) e = bf ? ATTN_BWD_TC(128, true) : ATTN_BWD_TC(128, false);
    else e = bf ? ATTN_BWD_TC(64, true) : ATTN_BWD_TC(64, false);
#undef ATTN_BWD_TC
    return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
  }
  int unsupported = 0;
  e = attn::launch_bwd_simt(s.D, static_cast<int>(dtype), p, q, k, v, out, dout, lse, dsum, lse2, dq,
                            dk, dv, scale, st, &unsupported);
  if (unsupported) return ATTN_ERR_HEAD_DIM;
  return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
}

}  // extern "C"

// ---------------------------------------------------------------- paged cache
extern "C" {

int attn_paged_workspace_bytes(const attn_paged_shape_t* shape, int num_splits, size_t* bytes) {
  if (!shape || !bytes) return ATTN_ERR_NULL;
  const attn_paged_shape_t s = *shape;
  if (s.num_queries < 0 || s.Hq <= 0 || s.Hkv <= 0 || s.D <= 0 || s.max_queries < 0) return ATTN_ERR_SHAPE;
  if (num_splits < 1 || num_splits > ATTN_MAX_SPLITS) return ATTN_ERR_SPLITS;
  const bool dec = attn::paged_is_decode(s.max_queries, s.Hq / s.Hkv);
  attn_shape_t rows{1, 1, 1, s.num_queries * s.Hq, 0, s.D, 1, 1};
  *bytes = (dec && num_splits > 1) ? static_cast<size_t>(split_layout(rows, num_splits).total) : 0;
  return ATTN_OK;
}

int attn_paged_fwd(const attn_paged_shape_t* shape, const void* q, const void* k_cache,
                   const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                   const int32_t* q_offsets, const int32_t* positions, int causal, float scale,
                   attn_dtype_t dtype, int num_splits, void* workspace, size_t workspace_bytes,
                   void* out, float* lse, void* stream) {
  if (!shape) return ATTN_ERR_NULL;
  const attn_paged_shape_t s = *shape;
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  if (s.num_seqs < 0 || s.num_queries < 0 || s.Hq <= 0 || s.Hkv <= 0 || s.D <= 0 || s.page_size <= 0 ||
      s.num_pages < 0 || s.max_pages < 0 || s.max_queries < 0 || s.Hq % s.Hkv != 0)
    return ATTN_ERR_SHAPE;
  if (causal != 0 && causal != 1) return ATTN_ERR_MASK;
  if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_SCALE;
  if (!(s.D == 16 || s.D == 32 || s.D == 64 || s.D == 128)) return ATTN_ERR_HEAD_DIM;
  if (num_splits < 1 || num_splits > ATTN_MAX_SPLITS) return ATTN_ERR_SPLITS;
  const int64_t group = s.Hq / s.Hkv;
  // splits apply to decode-shaped calls (the only kernel that splits)
  const int splits = attn::paged_is_decode(s.max_queries, static_cast<int>(group)) ? num_splits : 1;
  attn_shape_t rows_shape{1, 1, 1, s.num_queries * s.Hq, 0, s.D, 1, 1};
  const SplitLayout lay = split_layout(rows_shape, splits);
  if (static_cast<int64_t>(s.num_seqs) * s.Hkv > 0x7fffffffLL ||
      (static_cast<int64_t>(s.max_queries) * group + 63) / 64 > 65535 ||
      static_cast<int64_t>(s.max_pages) * s.page_size > 0x7fffffffLL)
    return ATTN_ERR_SHAPE;
  if (s.num_queries == 0 || s.num_seqs == 0) return ATTN_OK;
  if (!q || !out || !seq_lens || !q_offsets || (s.max_pages > 0 && !block_table) ||
      (s.num_pages > 0 && (!k_cache || !v_cache)))
    return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || (k_cache && !aligned16(k_cache)) || (v_cache && !aligned16(v_cache)))
    return ATTN_ERR_ALIGN;
  for (const void* pi : {static_cast<const void*>(block_table), static_cast<const void*>(seq_lens),
                         static_cast<const void*>(q_offsets), static_cast<const void*>(positions),
                         static_cast<const void*>(lse)})
    if (pi && (reinterpret_cast<uintptr_t>(pi) & 3u)) return ATTN_ERR_ALIGN;
  const int es = elem_size(dtype);
  const int64_t q_bytes = static_cast<int64_t>(s.num_queries) * s.Hq * s.D * es;
  const int64_t kv_bytes = static_cast<int64_t>(s.num_pages) * s.page_size * s.Hkv * s.D * es;
  const int64_t lse_bytes = lse ? static_cast<int64_t>(s.num_queries) * s.Hq * 4 : 0;
  struct Buf { const void* p; int64_t n; };
  const Buf ins[] = {{q, q_bytes}, {k_cache, kv_bytes}, {v_cache, kv_bytes},
                     {block_table, static_cast<int64_t>(s.num_seqs) * s.max_pages * 4},
                     {seq_lens, static_cast<int64_t>(s.num_seqs) * 4},
                     {q_offsets, static_cast<int64_t>(s.num_seqs + 1) * 4},
                     {positions, positions ? static_cast<int64_t>(s.num_queries) * 4 : 0}};
  for (const Buf& b : ins)
    if (overlaps(out, q_bytes, b.p, b.n) || overlaps(lse, lse_bytes, b.p, b.n)) return ATTN_ERR_OVERLAP;
  if (overlaps(out, q_bytes, lse, lse_bytes)) return ATTN_ERR_OVERLAP;
  if (splits > 1) {
    if (!workspace || workspace_bytes < static_cast<size_t>(lay.total)) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
    for (const Buf& b : ins)
      if (overlaps(workspace, lay.total, b.p, b.n)) return ATTN_ERR_OVERLAP;
    if (overlaps(workspace, lay.total, out, q_bytes) || overlaps(workspace, lay.total, lse, lse_bytes))
      return ATTN_ERR_OVERLAP;
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  attn::PagedParams pp{};
  pp.num_splits = splits;
  pp.ws_o = splits > 1 ? static_cast<float*>(workspace) : nullptr;
  pp.ws_ml = splits > 1 ? reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + lay.ml_offset) : nullptr;
  pp.num_seqs = s.num_seqs;
  pp.num_queries = s.num_queries;
  pp.Hq = s.Hq;
  pp.Hkv = s.Hkv;
  pp.page_size = s.page_size;
  pp.num_pages = s.num_pages;
  pp.max_pages = s.max_pages;
  pp.max_queries = s.max_queries;
  pp.block_table = block_table;
  pp.seq_lens = seq_lens;
  pp.q_offsets = q_offsets;
  pp.positions = positions;
  pp.causal = causal;
  pp.scale_log2 = scale * 1.4426950408889634f;
  pp.status = status_ptr(dev);
  pp.device = dev;
  int unsupported = 0;
  // F16/BF16 calls with D in {64, 128} and a page size the tile gathers
  // cover take the tensor cores; the rest the fp32 FMA kernels
  const bool pow_ok = s.page_size % 8 == 0 && (128 % s.page_size == 0 || s.page_size % 128 == 0);
  if (dtype != ATTN_F32 && (s.D == 64 || s.D == 128) && pow_ok && s.num_pages > 0) {
    attn::EncodeTiledFn enc = encode_fn();
    if (!enc) return fail_cuda(cudaErrorNotSupported);
    const bool bf = dtype == ATTN_BF16;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    using namespace attn::pagedtc;
    if (s.D == 128) e = bf ? launch_paged_tc<128, true>(enc, pp, q, k_cache, v_cache, out, lse, st)
                           : launch_paged_tc<128, false>(enc, pp, q, k_cache, v_cache, out, lse, st);
    else e = bf ? launch_paged_tc<64, true>(enc, pp, q, k_cache, v_cache, out, lse, st)
                : launch_paged_tc<64, false>(enc, pp, q, k_cache, v_cache, out, lse, st);
  } else {
    e = attn::launch_paged_simt(s.D, static_cast<int>(dtype), pp, q, k_cache, v_cache, out, lse,
                                static_cast<cudaStream_t>(stream), &unsupported);
    if (unsupported) return ATTN_ERR_HEAD_DIM;
  }
  if (e == cudaSuccess && splits > 1) {  // merge the partials of rows r = query * Hq + head
    attn::KernelParams mp{};
    mp.B = 1;
    mp.Hq = 1;
    mp.Sq = s.num_queries * s.Hq;
    mp.num_splits = splits;
    mp.ws_o = pp.ws_o;
    mp.ws_ml = pp.ws_ml;
    mp.lse = lse;
    e = attn::launch_split_merge(mp, s.D, static_cast<int>(dtype), out, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
}

}  // extern "C"

// ---------------------------------------------------------------- MLA
extern "C" {

int attn_paged_mla_workspace_bytes(const attn_mla_shape_t* shape, int num_splits, size_t* bytes) {
  if (!shape || !bytes) return ATTN_ERR_NULL;
  const attn_mla_shape_t s = *shape;
  if (s.num_queries < 0 || s.H <= 0 || s.R <= 0 || static_cast<int64_t>(s.num_queries) * s.H > 0x7fffffffLL)
    return ATTN_ERR_SHAPE;
  if (num_splits < 1 || num_splits > ATTN_MAX_SPLITS) return ATTN_ERR_SPLITS;
  attn_shape_t rows{1, 1, 1, s.num_queries * s.H, 0, s.R, 1, 1};
  *bytes = num_splits > 1 ? static_cast<size_t>(split_layout(rows, num_splits).total) : 0;
  return ATTN_OK;
}

int attn_paged_mla(const attn_mla_shape_t* shape, const void* q, const void* qp, const void* latent,
                   const void* kpos, const int32_t* block_table, const int32_t* seq_lens,
                   const int32_t* q_offsets, const int32_t* positions, int causal, float scale,
                   attn_dtype_t dtype, int num_splits, void* workspace, size_t workspace_bytes,
                   void* out, float* lse, void* stream) {
  if (!shape) return ATTN_ERR_NULL;
  const attn_mla_shape_t s = *shape;
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  if (s.num_seqs < 0 || s.num_queries < 0 || s.H <= 0 || s.R <= 0 || s.Pd < 0 || s.page_size <= 0 ||
      s.num_pages < 0 || s.max_pages < 0 || s.max_queries < 0)
    return ATTN_ERR_SHAPE;
  if (causal != 0 && causal != 1) return ATTN_ERR_MASK;
  if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_SCALE;
  if (!(s.R == 128 || s.R == 256 || s.R == 512) || !(s.Pd == 0 || s.Pd == 16 || s.Pd == 32 || s.Pd == 64))
    return ATTN_ERR_HEAD_DIM;
  if (num_splits < 1 || num_splits > ATTN_MAX_SPLITS) return ATTN_ERR_SPLITS;
  if ((static_cast<int64_t>(s.max_queries) * s.H + 7) / 8 > 65535 ||
      static_cast<int64_t>(s.max_pages) * s.page_size > 0x7fffffffLL ||
      static_cast<int64_t>(s.num_queries) * s.H > 0x7fffffffLL)
    return ATTN_ERR_SHAPE;
  if (s.num_queries == 0 || s.num_seqs == 0) return ATTN_OK;
  if (!q || !out || !seq_lens || !q_offsets || (s.max_pages > 0 && !block_table) ||
      (s.num_pages > 0 && !latent) || (s.Pd > 0 && (!qp || (s.num_pages > 0 && !kpos))))
    return ATTN_ERR_NULL;
  if (!aligned16(q) || !aligned16(out) || (qp && !aligned16(qp)) || (latent && !aligned16(latent)) ||
      (kpos && !aligned16(kpos)))
    return ATTN_ERR_ALIGN;
  for (const void* pi : {static_cast<const void*>(block_table), static_cast<const void*>(seq_lens),
                         static_cast<const void*>(q_offsets), static_cast<const void*>(positions),
                         static_cast<const void*>(lse)})
    if (pi && (reinterpret_cast<uintptr_t>(pi) & 3u)) return ATTN_ERR_ALIGN;
  const int es = elem_size(dtype);
  const int64_t rows = static_cast<int64_t>(s.num_queries) * s.H;
  const int64_t out_bytes = rows * s.R * es;
  const int64_t lse_bytes = lse ? rows * 4 : 0;
  const int64_t tok = static_cast<int64_t>(s.num_pages) * s.page_size;
  struct Buf { const void* p; int64_t n; };
  const Buf ins[] = {{q, out_bytes}, {qp, rows * s.Pd * es}, {latent, tok * s.R * es}, {kpos, tok * s.Pd * es},
                     {block_table, static_cast<int64_t>(s.num_seqs) * s.max_pages * 4},
                     {seq_lens, static_cast<int64_t>(s.num_seqs) * 4},
                     {q_offsets, static_cast<int64_t>(s.num_seqs + 1) * 4},
                     {positions, positions ? static_cast<int64_t>(s.num_queries) * 4 : 0}};
  for (const Buf& b : ins)
    if (overlaps(out, out_bytes, b.p, b.n) || overlaps(lse, lse_bytes, b.p, b.n)) return ATTN_ERR_OVERLAP;
  if (overlaps(out, out_bytes, lse, lse_bytes)) return ATTN_ERR_OVERLAP;
  attn_shape_t rows_shape{1, 1, 1, s.num_queries * s.H, 0, s.R, 1, 1};
  const SplitLayout lay = split_layout(rows_shape, num_splits);
  if (num_splits > 1) {
    if (!workspace || workspace_bytes < static_cast<size_t>(lay.total)) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
    for (const Buf& b : ins)
      if (overlaps(workspace, lay.total, b.p, b.n)) return ATTN_ERR_OVERLAP;
    if (overlaps(workspace, lay.total, out, out_bytes) || overlaps(workspace, lay.total, lse, lse_bytes))
      return ATTN_ERR_OVERLAP;
  }

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e);
  attn::PagedParams pp{};
  pp.num_splits = 1;
  pp.num_seqs = s.num_seqs;
  pp.num_queries = s.num_queries;
  pp.Hq = s.H;
  pp.Hkv = 1;
  pp.page_size = s.page_size;
  pp.num_pages = s.num_pages;
  pp.max_pages = s.max_pages;
  pp.max_queries = s.max_queries;
  pp.block_table = block_table;
  pp.seq_lens = seq_lens;
  pp.q_offsets = q_offsets;
  pp.positions = positions;
  pp.causal = causal;
  pp.scale_log2 = scale * 1.4426950408889634f;
  pp.status = status_ptr(dev);
  pp.device = dev;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  // F16/BF16 with R in {256, 512}, Pd in {0, 64} and a page size the 64-key
  // tile gathers cover take the tensor cores (and the key-range splits)
  const bool page_ok = s.page_size % 8 == 0 && (64 % s.page_size == 0 || s.page_size % 64 == 0);
  if (dtype != ATTN_F32 && (s.R == 256 || s.R == 512) && (s.Pd == 0 || s.Pd == 64) && page_ok &&
      s.num_pages > 0) {
    attn::EncodeTiledFn enc = encode_fn();
    if (!enc) return fail_cuda(cudaErrorNotSupported);
    pp.num_splits = num_splits;
    pp.ws_o = num_splits > 1 ? static_cast<float*>(workspace) : nullptr;
    pp.ws_ml = num_splits > 1 ? reinterpret_cast<float2*>(static_cast<uint8_t*>(workspace) + lay.ml_offset)
                              : nullptr;
    const bool bf = dtype == ATTN_BF16;
    using attn::mlatc::launch_mla_tc;
#define ATTN_MLA_TC(R, PD)                                                                         \
  (bf ? launch_mla_tc<R, PD, true>(enc, pp, q, qp, latent, kpos, out, lse, st)                     \
      : launch_mla_tc<R, PD, false>(enc, pp, q, qp, latent, kpos, out, lse, st))
    if (s.R == 512) e = s.Pd == 64 ? ATTN_MLA_TC(512, 64) : ATTN_MLA_TC(512, 0);
    else e = s.Pd == 64 ? ATTN_MLA_TC(256, 64) : ATTN_MLA_TC(256, 0);
#undef ATTN_MLA_TC
    if (e == cudaSuccess && num_splits > 1) {  // merge the partials of rows r = query * H + head
      attn::KernelParams mp{};
      mp.B = 1;
      mp.Hq = 1;
      mp.Sq = s.num_queries * s.H;
      mp.num_splits = num_splits;
      mp.ws_o = pp.ws_o;
      mp.ws_ml = pp.ws_ml;
      mp.lse = lse;
      e = attn::launch_split_merge(mp, s.R, static_cast<int>(dtype), out, st);
    }
    return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
  }
  int unsupported = 0;
  e = attn::launch_mla_simt(s.R, s.Pd, static_cast<int>(dtype), pp, q, qp, latent, kpos, out, lse, st,
                            &unsupported);
  if (unsupported) return ATTN_ERR_HEAD_DIM;
  return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
}

}  // extern "C"

// ---------------------------------------------------------------- paged backward
namespace {

// Grid limits and required pointers shared by both paged backward calls;
// `rows_per_cta` is the query-major kernel's (query, head) rows per CTA.
int check_paged_bwd_shape(int num_seqs, int num_queries, int heads, int Hkv, int page_size, int num_pages,
                          int max_pages, int max_queries, int rows_per_cta) {
  if (num_seqs < 0 || num_queries < 0 || heads <= 0 || Hkv <= 0 || heads % Hkv != 0 || page_size <= 0 ||
      num_pages < 0 || max_pages < 0 || max_queries < 0)
    return ATTN_ERR_SHAPE;
  const int64_t group = heads / Hkv;
  if (static_cast<int64_t>(num_seqs) * Hkv > 0x7fffffffLL || static_cast<int64_t>(num_pages) * Hkv > 0x7fffffffLL ||
      (static_cast<int64_t>(max_queries) * group + rows_per_cta - 1) / rows_per_cta > 65535 ||
      (static_cast<int64_t>(page_size) + rows_per_cta - 1) / rows_per_cta > 65535 ||
      static_cast<int64_t>(max_pages) * page_size > 0x7fffffffLL ||
      static_cast<int64_t>(num_seqs) * max_pages > 0x7fffffffLL)
    return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

attn::pbwd::Layout paged_bwd_layout(int num_seqs, int num_queries, int heads, int num_pages, int max_pages) {
  return attn::pbwd::layout(static_cast<int64_t>(num_queries) * heads, num_pages,
                            static_cast<int64_t>(num_seqs) * max_pages);
}

attn::PagedParams paged_bwd_params(int dev, int num_seqs, int num_queries, int heads, int Hkv, int page_size,
                                   int num_pages, int max_pages, int max_queries, const int32_t* block_table,
                                   const int32_t* seq_lens, const int32_t* q_offsets, const int32_t* positions,
                                   int causal, float scale) {
  attn::PagedParams pp{};
  pp.num_splits = 1;
  pp.num_seqs = num_seqs;
  pp.num_queries = num_queries;
  pp.Hq = heads;
  pp.Hkv = Hkv;
  pp.page_size = page_size;
  pp.num_pages = num_pages;
  pp.max_pages = max_pages;
  pp.max_queries = max_queries;
  pp.block_table = block_table;
  pp.seq_lens = seq_lens;
  pp.q_offsets = q_offsets;
  pp.positions = positions;
  pp.causal = causal;
  pp.scale_log2 = scale * 1.4426950408889634f;
  pp.status = status_ptr(dev);
  pp.device = dev;
  return pp;
}

struct Buf { const void* p; int64_t n; };

// Every written buffer is disjoint from every read buffer and from the others.
bool any_overlap(const Buf* outs, int n_out, const Buf* ins, int n_in) {
  for (int a = 0; a < n_out; ++a) {
    for (int i = 0; i < n_in; ++i)
      if (overlaps(outs[a].p, outs[a].n, ins[i].p, ins[i].n)) return true;
    for (int c = a + 1; c < n_out; ++c)
      if (overlaps(outs[a].p, outs[a].n, outs[c].p, outs[c].n)) return true;
  }
  return false;
}

bool misaligned4(std::initializer_list<const void*> ps) {
  for (const void* p : ps)
    if (p && (reinterpret_cast<uintptr_t>(p) & 3u)) return true;
  return false;
}

}  // namespace

extern "C" {

int attn_paged_bwd_workspace_bytes(const attn_paged_shape_t* shape, size_t* bytes) {
  if (!shape || !bytes) return ATTN_ERR_NULL;
  const attn_paged_shape_t s = *shape;
  if (s.num_seqs < 0 || s.num_queries < 0 || s.Hq <= 0 || s.num_pages < 0 || s.max_pages < 0)
    return ATTN_ERR_SHAPE;
  *bytes = static_cast<size_t>(paged_bwd_layout(s.num_seqs, s.num_queries, s.Hq, s.num_pages, s.max_pages).total);
  return ATTN_OK;
}

int attn_paged_bwd(const attn_paged_shape_t* shape, const void* q, const void* k_cache, const void* v_cache,
                   const int32_t* block_table, const int32_t* seq_lens, const int32_t* q_offsets,
                   const int32_t* positions, int causal, float scale, attn_dtype_t dtype, const void* out,
                   const void* dout, const float* lse, void* workspace, size_t workspace_bytes, void* dq,
                   void* dk_cache, void* dv_cache, void* stream) {
  if (!shape) return ATTN_ERR_NULL;
  const attn_paged_shape_t s = *shape;
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  int rc = check_paged_bwd_shape(s.num_seqs, s.num_queries, s.Hq, s.Hkv, s.page_size, s.num_pages, s.max_pages,
                                 s.max_queries, 64);
  if (rc != ATTN_OK) return rc;
  if (s.D <= 0) return ATTN_ERR_SHAPE;
  if (causal != 0 && causal != 1) return ATTN_ERR_MASK;
  if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_SCALE;
  if (!(s.D == 16 || s.D == 32 || s.D == 64 || s.D == 128)) return ATTN_ERR_HEAD_DIM;
  const bool work = s.num_queries > 0 && s.num_seqs > 0 && (dq || dk_cache || dv_cache);
  if (work && (!q || !out || !dout || !lse || !seq_lens || !q_offsets || (s.max_pages > 0 && !block_table) ||
               (s.num_pages > 0 && (!k_cache || !v_cache))))
    return ATTN_ERR_NULL;
  for (const void* p16 : {q, k_cache, v_cache, out, dout, static_cast<const void*>(dq),
                          static_cast<const void*>(dk_cache), static_cast<const void*>(dv_cache)})
    if (p16 && !aligned16(p16)) return ATTN_ERR_ALIGN;
  if (misaligned4({block_table, seq_lens, q_offsets, positions, lse})) return ATTN_ERR_ALIGN;
  const int es = elem_size(dtype);
  const int64_t q_bytes = static_cast<int64_t>(s.num_queries) * s.Hq * s.D * es;
  const int64_t kv_bytes = static_cast<int64_t>(s.num_pages) * s.page_size * s.Hkv * s.D * es;
  const attn::pbwd::Layout lay = paged_bwd_layout(s.num_seqs, s.num_queries, s.Hq, s.num_pages, s.max_pages);
  if (work) {
    if (!workspace || workspace_bytes < static_cast<size_t>(lay.total)) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  }
  const Buf ins[] = {{q, q_bytes}, {k_cache, kv_bytes}, {v_cache, kv_bytes}, {out, q_bytes}, {dout, q_bytes},
                     {lse, static_cast<int64_t>(s.num_queries) * s.Hq * 4},
                     {block_table, static_cast<int64_t>(s.num_seqs) * s.max_pages * 4},
                     {seq_lens, static_cast<int64_t>(s.num_seqs) * 4},
                     {q_offsets, static_cast<int64_t>(s.num_seqs + 1) * 4},
                     {positions, positions ? static_cast<int64_t>(s.num_queries) * 4 : 0}};
  const Buf outs[] = {{dq, q_bytes}, {dk_cache, kv_bytes}, {dv_cache, kv_bytes},
                      {work ? workspace : nullptr, lay.total}};
  if (any_overlap(outs, 4, ins, 10)) return ATTN_ERR_OVERLAP;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (!work) {  // no query: the cache gradients are zero
    if (dk_cache && kv_bytes) e = cudaMemsetAsync(dk_cache, 0, static_cast<size_t>(kv_bytes), st);
    if (e == cudaSuccess && dv_cache && kv_bytes) e = cudaMemsetAsync(dv_cache, 0, static_cast<size_t>(kv_bytes), st);
    return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
  }
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return fail_cuda(e);
  const attn::PagedParams pp =
      paged_bwd_params(dev, s.num_seqs, s.num_queries, s.Hq, s.Hkv, s.page_size, s.num_pages, s.max_pages,
                       s.max_queries, block_table, seq_lens, q_offsets, positions, causal, scale);
  const attn::pbwd::Buffers b = attn::pbwd::carve(workspace, lay);
  e = attn::pbwd::launch_preprocess(static_cast<int>(dtype), s.D, out, dout, lse, b,
                                    static_cast<int64_t>(s.num_queries) * s.Hq, st, pp.status);
  if (e == cudaSuccess && (dk_cache || dv_cache)) e = attn::pbwd::launch_page_index(pp, b, st);
  // F16/BF16 with D in {64, 128} and a page size the 128-key tile gathers
  // cover take the tensor cores; the pages that do not have exactly one reader
  // then go through the fp32 FMA key-major kernel
  const bool page_ok = s.page_size % 8 == 0 && (128 % s.page_size == 0 || s.page_size % 128 == 0);
  if (e == cudaSuccess && dtype != ATTN_F32 && (s.D == 64 || s.D == 128) && page_ok && s.num_pages > 0) {
    attn::EncodeTiledFn enc = encode_fn();
    if (!enc) return fail_cuda(cudaErrorNotSupported);
    const attn::pbwd::TcArgs ta{b.lse2, b.dsum, b.offsets, dq, dk_cache, dv_cache, scale};
    const bool bf = dtype == ATTN_BF16;
    using attn::pbwd::launch_paged_bwd_tc;
    if (s.D == 128) e = bf ? launch_paged_bwd_tc<128, true>(enc, pp, q, k_cache, v_cache, dout, ta, st)
                           : launch_paged_bwd_tc<128, false>(enc, pp, q, k_cache, v_cache, dout, ta, st);
    else e = bf ? launch_paged_bwd_tc<64, true>(enc, pp, q, k_cache, v_cache, dout, ta, st)
                : launch_paged_bwd_tc<64, false>(enc, pp, q, k_cache, v_cache, dout, ta, st);
    if (e == cudaSuccess && (dk_cache || dv_cache))
      e = attn::pbwd::launch_paged_dkdv_shared(s.D, static_cast<int>(dtype), pp, q, k_cache, v_cache, dout, b,
                                               dk_cache, dv_cache, scale, st);
    return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
  }
  if (e == cudaSuccess)
    e = attn::pbwd::launch_paged_bwd(s.D, static_cast<int>(dtype), pp, q, k_cache, v_cache, dout, b, dq, dk_cache,
                                     dv_cache, scale, st);
  return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
}

int attn_paged_mla_bwd_workspace_bytes(const attn_mla_shape_t* shape, size_t* bytes) {
  if (!shape || !bytes) return ATTN_ERR_NULL;
  const attn_mla_shape_t s = *shape;
  if (s.num_seqs < 0 || s.num_queries < 0 || s.H <= 0 || s.num_pages < 0 || s.max_pages < 0) return ATTN_ERR_SHAPE;
  *bytes = static_cast<size_t>(paged_bwd_layout(s.num_seqs, s.num_queries, s.H, s.num_pages, s.max_pages).total);
  return ATTN_OK;
}

int attn_paged_mla_bwd(const attn_mla_shape_t* shape, const void* q, const void* qp, const void* latent,
                       const void* kpos, const int32_t* block_table, const int32_t* seq_lens,
                       const int32_t* q_offsets, const int32_t* positions, int causal, float scale,
                       attn_dtype_t dtype, const void* out, const void* dout, const float* lse, void* workspace,
                       size_t workspace_bytes, void* dq, void* dqp, void* dlatent, void* dkpos, void* stream) {
  if (!shape) return ATTN_ERR_NULL;
  const attn_mla_shape_t s = *shape;
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  if (s.R <= 0 || s.Pd < 0) return ATTN_ERR_SHAPE;
  if (!(s.R == 128 || s.R == 256 || s.R == 512) || !(s.Pd == 0 || s.Pd == 16 || s.Pd == 32 || s.Pd == 64))
    return ATTN_ERR_HEAD_DIM;
  int rc = check_paged_bwd_shape(s.num_seqs, s.num_queries, s.H, 1, s.page_size, s.num_pages, s.max_pages,
                                 s.max_queries, 8192 / s.R);
  if (rc != ATTN_OK) return rc;
  if (causal != 0 && causal != 1) return ATTN_ERR_MASK;
  if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_SCALE;
  if (s.Pd == 0) dqp = dkpos = nullptr;  // nothing to compute
  const bool work = s.num_queries > 0 && s.num_seqs > 0 && (dq || dqp || dlatent || dkpos);
  if (work && (!q || !out || !dout || !lse || !seq_lens || !q_offsets || (s.max_pages > 0 && !block_table) ||
               (s.num_pages > 0 && !latent) || (s.Pd > 0 && (!qp || (s.num_pages > 0 && !kpos)))))
    return ATTN_ERR_NULL;
  for (const void* p16 : {q, qp, latent, kpos, out, dout, static_cast<const void*>(dq), static_cast<const void*>(dqp),
                          static_cast<const void*>(dlatent), static_cast<const void*>(dkpos)})
    if (p16 && !aligned16(p16)) return ATTN_ERR_ALIGN;
  if (misaligned4({block_table, seq_lens, q_offsets, positions, lse})) return ATTN_ERR_ALIGN;
  const int es = elem_size(dtype);
  const int64_t rows = static_cast<int64_t>(s.num_queries) * s.H;
  const int64_t tok = static_cast<int64_t>(s.num_pages) * s.page_size;
  const attn::pbwd::Layout lay = paged_bwd_layout(s.num_seqs, s.num_queries, s.H, s.num_pages, s.max_pages);
  if (work) {
    if (!workspace || workspace_bytes < static_cast<size_t>(lay.total)) return ATTN_ERR_WORKSPACE;
    if (!aligned16(workspace)) return ATTN_ERR_ALIGN;
  }
  const Buf ins[] = {{q, rows * s.R * es}, {qp, rows * s.Pd * es}, {latent, tok * s.R * es},
                     {kpos, tok * s.Pd * es}, {out, rows * s.R * es}, {dout, rows * s.R * es}, {lse, rows * 4},
                     {block_table, static_cast<int64_t>(s.num_seqs) * s.max_pages * 4},
                     {seq_lens, static_cast<int64_t>(s.num_seqs) * 4},
                     {q_offsets, static_cast<int64_t>(s.num_seqs + 1) * 4},
                     {positions, positions ? static_cast<int64_t>(s.num_queries) * 4 : 0}};
  const Buf outs[] = {{dq, rows * s.R * es}, {dqp, rows * s.Pd * es}, {dlatent, tok * s.R * es},
                      {dkpos, tok * s.Pd * es}, {work ? workspace : nullptr, lay.total}};
  if (any_overlap(outs, 5, ins, 11)) return ATTN_ERR_OVERLAP;

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (!work) {
    if (dlatent && tok) e = cudaMemsetAsync(dlatent, 0, static_cast<size_t>(tok * s.R * es), st);
    if (e == cudaSuccess && dkpos && tok) e = cudaMemsetAsync(dkpos, 0, static_cast<size_t>(tok * s.Pd * es), st);
    return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
  }
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return fail_cuda(e);
  const attn::PagedParams pp =
      paged_bwd_params(dev, s.num_seqs, s.num_queries, s.H, 1, s.page_size, s.num_pages, s.max_pages,
                       s.max_queries, block_table, seq_lens, q_offsets, positions, causal, scale);
  const attn::pbwd::Buffers b = attn::pbwd::carve(workspace, lay);
  e = attn::pbwd::launch_preprocess(static_cast<int>(dtype), s.R, out, dout, lse, b, rows, st, pp.status);
  if (e == cudaSuccess && (dlatent || dkpos)) e = attn::pbwd::launch_page_index(pp, b, st);
  // F16/BF16 with R in {256, 512}, Pd in {0, 64} and a page size the 128-key
  // gathers cover take the tensor cores; the pages that do not have exactly
  // one reader then go through the fp32 FMA key-major kernel
  const bool page_ok = s.page_size % 8 == 0 && (128 % s.page_size == 0 || s.page_size % 128 == 0);
  if (e == cudaSuccess && dtype != ATTN_F32 && (s.R == 256 || s.R == 512) && (s.Pd == 0 || s.Pd == 64) &&
      page_ok && s.num_pages > 0) {
    attn::EncodeTiledFn enc = encode_fn();
    if (!enc) return fail_cuda(cudaErrorNotSupported);
    e = attn::pbwd::launch_mla_bwd_tc(enc, s.R, s.Pd, dtype == ATTN_BF16, pp, q, qp, latent, kpos, dout, b, dq, dqp,
                                      dlatent, dkpos, scale, st);
    if (e == cudaSuccess && (dlatent || dkpos))
      e = attn::pbwd::launch_mla_dkdv_shared(s.R, s.Pd, static_cast<int>(dtype), pp, q, qp, latent, kpos, dout, b,
                                             dlatent, dkpos, scale, st);
    return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
  }
  if (e == cudaSuccess)
    e = attn::pbwd::launch_mla_bwd(s.R, s.Pd, static_cast<int>(dtype), pp, q, qp, latent, kpos, dout, b, dq, dqp,
                                   dlatent, dkpos, scale, st);
  return e == cudaSuccess ? ATTN_OK : fail_cuda(e);
}

}  // extern "C"
