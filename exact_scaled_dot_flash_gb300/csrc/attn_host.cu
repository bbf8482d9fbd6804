// attn_host.cu - attn_fwd_host: attention on tensors that live in host memory,
// with the transfers overlapped with the computation.
//
// The pages' attention entry computes on device tensors; a caller whose q, k,
// v and output live in host memory otherwise pays the upload, the kernel and
// the download one after the other. Here the problem is cut into chunks of
// whole (batch, kv head) units: chunk = batch index b and kv heads
// [h0, h0 + nh) with their Hq/Hkv query heads each. Its Q, K, V and O are
// contiguous ranges of the [B, H, S, D] tensors and its bias the matching rows
// of [bias_b, bias_h, Sq, Sk], so each moves with one copy. Two device slots
// (in the caller's workspace) hold a chunk's inputs and output; three streams
// carry the work:
//   upload c     (library stream U): after the attention of c-2 has read slot c%2
//   attention c  (the caller's stream): after upload c and download c-2
//   download c   (library stream D): after attention c
// so the upload of c+1, the attention of c and the download of c-1 overlap.
// Every chunk runs attn_fwd on its own (B = 1) shape: each output row is
// computed by the same kernel code from the same inputs as in one whole-problem
// call, so the result is identical. The caller's stream is ordered after all of
// it when the call returns.
#include <math.h>

#include <mutex>

#include "attn.h"
#include "params.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr int kTargetChunks = 8;  // enough chunks to overlap; 16 measured no better

int64_t up256(int64_t x) { return (x + 255) / 256 * 256; }

struct HostPlan {
  int nh = 0;  // kv heads of the largest chunk
  int64_t q_bytes = 0, kv_bytes = 0, bias_bytes = 0;  // of the largest chunk
  int64_t off_q = 0, off_k = 0, off_v = 0, off_o = 0, off_bias = 0;  // within a slot
  int64_t off_lens = 0, off_slot[2] = {0, 0}, slot_bytes = 0, total = 0;
};

// Workspace: kv_lens (B int32), then two slots of [Q | K | V | O | bias] for the
// largest chunk, every piece starting on a 256-byte boundary.
HostPlan make_plan(const attn_shape_t& s, int es, bool bias) {
  HostPlan p;
  const int g = s.Hq / s.Hkv;
  int want = (kTargetChunks + s.B - 1) / s.B;
  want = want < 1 ? 1 : (want > s.Hkv ? s.Hkv : want);
  p.nh = (s.Hkv + want - 1) / want;
  p.q_bytes = static_cast<int64_t>(p.nh) * g * s.Sq * s.D * es;
  p.kv_bytes = static_cast<int64_t>(p.nh) * s.Sk * s.D * es;
  p.bias_bytes = bias ? static_cast<int64_t>(s.bias_h == 1 ? 1 : p.nh * g) * s.Sq * s.Sk * 4 : 0;
  p.off_q = 0;
  p.off_k = up256(p.q_bytes);
  p.off_v = p.off_k + up256(p.kv_bytes);
  p.off_o = p.off_v + up256(p.kv_bytes);
  p.off_bias = p.off_o + up256(p.q_bytes);
  p.slot_bytes = p.off_bias + up256(p.bias_bytes);
  p.off_lens = 0;
  p.off_slot[0] = up256(static_cast<int64_t>(s.B) * 4);
  p.off_slot[1] = p.off_slot[0] + p.slot_bytes;
  p.total = p.off_slot[1] + p.slot_bytes;
  return p;
}

// Shape checks shared by the call and its workspace query (attn_fwd's rules).
int check_shape(const attn_shape_t& s, attn_dtype_t dtype, bool bias) {
  if (dtype != ATTN_F32 && dtype != ATTN_F16 && dtype != ATTN_BF16) return ATTN_ERR_DTYPE;
  if (s.B < 0 || s.Sq < 0 || s.Sk < 0 || s.Hq <= 0 || s.Hkv <= 0 || s.D <= 0 || s.Hq % s.Hkv != 0)
    return ATTN_ERR_SHAPE;
  if (bias && !((s.bias_b == 1 || s.bias_b == s.B) && (s.bias_h == 1 || s.bias_h == s.Hq)))
    return ATTN_ERR_SHAPE;
  return ATTN_OK;
}

bool host_overlaps(const void* a, int64_t na, const void* b, int64_t nb) {
  if (!a || !b || na <= 0 || nb <= 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + static_cast<uintptr_t>(nb) && b0 < a0 + static_cast<uintptr_t>(na);
}

// The library's copy streams and events of one device, created on first use;
// the mutex serialises the enqueueing of calls on that device.
struct HostExec {
  std::mutex mu;
  bool ready = false;
  cudaStream_t up = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, in[2] = {nullptr, nullptr}, comp[2] = {nullptr, nullptr},
              out[2] = {nullptr, nullptr};
};
HostExec g_exec[kMaxDevices];

cudaError_t exec_init(HostExec& x) {
  if (x.ready) return cudaSuccess;
  cudaError_t e = cudaStreamCreateWithFlags(&x.up, cudaStreamNonBlocking);
  if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&x.down, cudaStreamNonBlocking);
  cudaEvent_t* evs[] = {&x.start, &x.in[0], &x.in[1], &x.comp[0], &x.comp[1], &x.out[0], &x.out[1]};
  for (cudaEvent_t* ev : evs)
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
  if (e == cudaSuccess) x.ready = true;
  return e;
}

}  // namespace

extern "C" {

int attn_fwd_host_workspace_bytes(const attn_shape_t* shape, attn_dtype_t dtype, int with_bias, size_t* bytes) {
  if (!shape || !bytes) return ATTN_ERR_NULL;
  const attn_shape_t s = *shape;
  const int rc = check_shape(s, dtype, with_bias != 0);
  if (rc != ATTN_OK) return rc;
  *bytes = (s.B == 0 || s.Sq == 0) ? 0 : static_cast<size_t>(make_plan(s, dtype == ATTN_F32 ? 4 : 2, with_bias != 0).total);
  return ATTN_OK;
}

int attn_fwd_host(const attn_shape_t* shape, const void* q, const void* k, const void* v, int mask_kind,
                  const int32_t* kv_lens, const float* bias, float scale, attn_dtype_t dtype, void* workspace,
                  size_t workspace_bytes, void* out, void* stream) {
  // ---- validation, before any CUDA call (the chunk calls repeat attn_fwd's own)
  if (!shape) return ATTN_ERR_NULL;
  const attn_shape_t s = *shape;
  int rc = check_shape(s, dtype, bias != nullptr);
  if (rc != ATTN_OK) return rc;
  if (mask_kind & ~(ATTN_MASK_CAUSAL | ATTN_MASK_KEY_PADDING)) return ATTN_ERR_MASK;
  if ((mask_kind & ATTN_MASK_KEY_PADDING) && !kv_lens) return ATTN_ERR_MASK;
  if (!(scale > 0.f) || !isfinite(scale)) return ATTN_ERR_SCALE;
  const bool tensor_core = dtype != ATTN_F32;
  if (tensor_core ? !(s.D == 32 || s.D == 64 || s.D == 128) : !(s.D == 16 || s.D == 32 || s.D == 64 || s.D == 128))
    return ATTN_ERR_HEAD_DIM;
  if (s.B == 0 || s.Sq == 0) return ATTN_OK;
  if (!q || !out || (s.Sk > 0 && (!k || !v))) return ATTN_ERR_NULL;
  const int es = dtype == ATTN_F32 ? 4 : 2;
  const HostPlan p = make_plan(s, es, bias != nullptr);
  if (!workspace || workspace_bytes < static_cast<size_t>(p.total)) return ATTN_ERR_WORKSPACE;
  if (reinterpret_cast<uintptr_t>(workspace) & 15u) return ATTN_ERR_ALIGN;
  const int64_t bhq = static_cast<int64_t>(s.B) * s.Hq;
  const int64_t out_bytes = bhq * s.Sq * s.D * es;
  const int64_t kv_bytes = static_cast<int64_t>(s.B) * s.Hkv * s.Sk * s.D * es;
  const int64_t bias_bytes = bias ? static_cast<int64_t>(s.bias_b) * s.bias_h * s.Sq * static_cast<int64_t>(s.Sk) * 4 : 0;
  if (host_overlaps(out, out_bytes, q, out_bytes) || host_overlaps(out, out_bytes, k, kv_bytes) ||
      host_overlaps(out, out_bytes, v, kv_bytes) || host_overlaps(out, out_bytes, bias, bias_bytes) ||
      host_overlaps(out, out_bytes, kv_lens, static_cast<int64_t>(s.B) * 4))
    return ATTN_ERR_OVERLAP;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return attn::record_cuda_error(e);
  if (dev < 0 || dev >= kMaxDevices) return attn::record_cuda_error(cudaErrorInvalidDevice);
  HostExec& x = g_exec[dev];
  std::lock_guard<std::mutex> lock(x.mu);
  e = exec_init(x);
  if (e != cudaSuccess) return attn::record_cuda_error(e);

  cudaStream_t st_main = static_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  const int g = s.Hq / s.Hkv;
  const int64_t row_q = static_cast<int64_t>(s.Sq) * s.D * es;  // one head of Q or O
  const int64_t row_kv = static_cast<int64_t>(s.Sk) * s.D * es;
  const int64_t row_bias = static_cast<int64_t>(s.Sq) * s.Sk * 4;
  int32_t* d_lens = kv_lens ? reinterpret_cast<int32_t*>(ws + p.off_lens) : nullptr;
  auto cp = [](void* dst, const void* src, int64_t n, cudaMemcpyKind kind, cudaStream_t st) {
    return n > 0 ? cudaMemcpyAsync(dst, src, static_cast<size_t>(n), kind, st) : cudaSuccess;
  };

  rc = ATTN_OK;
  e = cudaEventRecord(x.start, st_main);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(x.up, x.start, 0);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(x.down, x.start, 0);
  if (e == cudaSuccess && d_lens) e = cp(d_lens, kv_lens, static_cast<int64_t>(s.B) * 4, cudaMemcpyHostToDevice, x.up);
  int c = 0;
  for (int b = 0; b < s.B && e == cudaSuccess && rc == ATTN_OK; ++b) {
    // chunks of p.nh kv heads; in the last batch index they taper (p.nh, p.nh/2,
    // then p.nh/4 each) so that the compute and download left after the last
    // upload are short
    int step = p.nh;
    for (int h0 = 0; h0 < s.Hkv && e == cudaSuccess && rc == ATTN_OK; h0 += step, ++c) {
      if (b == s.B - 1 && h0 > 0) step = step / 2 > (p.nh + 3) / 4 ? step / 2 : (p.nh + 3) / 4;
      const int nh = (h0 + step <= s.Hkv) ? step : s.Hkv - h0;
      const int sl = c & 1;
      uint8_t* slot = ws + p.off_slot[sl];
      const int64_t qoff = (static_cast<int64_t>(b) * s.Hq + static_cast<int64_t>(h0) * g) * row_q;
      const int64_t kvoff = (static_cast<int64_t>(b) * s.Hkv + h0) * row_kv;
      const int64_t qn = static_cast<int64_t>(nh) * g * row_q, kvn = static_cast<int64_t>(nh) * row_kv;
      attn_shape_t cs{1, nh * g, nh, s.Sq, s.Sk, s.D, 1, 1};
      const float* hb = nullptr;
      int64_t bn = 0;
      if (bias) {
        const int bb = s.bias_b == 1 ? 0 : b;
        if (s.bias_h == 1) {
          hb = bias + static_cast<int64_t>(bb) * row_bias / 4;
          bn = row_bias;
        } else {
          hb = bias + (static_cast<int64_t>(bb) * s.Hq + static_cast<int64_t>(h0) * g) * row_bias / 4;
          bn = static_cast<int64_t>(nh) * g * row_bias;
          cs.bias_h = nh * g;
        }
      }
      // upload c: slot sl is free once the attention of c-2 has read it
      if (c >= 2) e = cudaStreamWaitEvent(x.up, x.comp[sl], 0);
      if (e == cudaSuccess) e = cp(slot + p.off_q, static_cast<const uint8_t*>(q) + qoff, qn, cudaMemcpyHostToDevice, x.up);
      if (e == cudaSuccess) e = cp(slot + p.off_k, static_cast<const uint8_t*>(k) + kvoff, kvn, cudaMemcpyHostToDevice, x.up);
      if (e == cudaSuccess) e = cp(slot + p.off_v, static_cast<const uint8_t*>(v) + kvoff, kvn, cudaMemcpyHostToDevice, x.up);
      if (e == cudaSuccess && bias) e = cp(slot + p.off_bias, hb, bn, cudaMemcpyHostToDevice, x.up);
      if (e == cudaSuccess) e = cudaEventRecord(x.in[sl], x.up);
      // attention c, on the caller's stream: after its upload and after the
      // download of c-2 has read the slot's output
      if (e == cudaSuccess) e = cudaStreamWaitEvent(st_main, x.in[sl], 0);
      if (e == cudaSuccess && c >= 2) e = cudaStreamWaitEvent(st_main, x.out[sl], 0);
      if (e != cudaSuccess) break;
      rc = attn_fwd(&cs, slot + p.off_q, slot + p.off_k, slot + p.off_v, mask_kind, d_lens ? d_lens + b : nullptr,
                    bias ? reinterpret_cast<const float*>(slot + p.off_bias) : nullptr, scale, dtype,
                    slot + p.off_o, st_main);
      if (rc != ATTN_OK) break;
      e = cudaEventRecord(x.comp[sl], st_main);
      // download c
      if (e == cudaSuccess) e = cudaStreamWaitEvent(x.down, x.comp[sl], 0);
      if (e == cudaSuccess) e = cp(static_cast<uint8_t*>(out) + qoff, slot + p.off_o, qn, cudaMemcpyDeviceToHost, x.down);
      if (e == cudaSuccess) e = cudaEventRecord(x.out[sl], x.down);
    }
  }
  // the caller's stream follows everything enqueued, on success or not, so
  // that the caller may release the buffers once it has synchronised
  cudaError_t e2 = cudaEventRecord(x.in[0], x.up);
  if (e2 == cudaSuccess) e2 = cudaEventRecord(x.out[0], x.down);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st_main, x.in[0], 0);
  if (e2 == cudaSuccess) e2 = cudaStreamWaitEvent(st_main, x.out[0], 0);
  if (rc != ATTN_OK) return rc;
  if (e != cudaSuccess) return attn::record_cuda_error(e);
  if (e2 != cudaSuccess) return attn::record_cuda_error(e2);
  return ATTN_OK;
}

}  // extern "C"
