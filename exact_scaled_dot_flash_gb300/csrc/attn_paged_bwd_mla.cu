// attn_paged_bwd_mla.cu - the paged MLA instances of the backward kernels in
// paged_bwd.cuh: one latent head shared by all heads (Hkv = 1), the latent row
// serving as key and value, an optional positional part. R/32 threads share a
// row or key, so each thread holds 32 latent elements whatever the rank.
#include "paged_bwd.cuh"

namespace attn {
namespace pbwd {

namespace {

template <int R, int PD>
cudaError_t launch_rp(int dtype, const PagedParams& pp, const void* q, const void* qp, const void* lat,
                      const void* kp, const void* dout, const Buffers& b, void* dq, void* dqp, void* dlat,
                      void* dkp, float scale, cudaStream_t st) {
  constexpr int TPK = R / 32;
  if (dtype == 0)
    return launch_instance<R, PD, TPK, 0, true>(pp, q, qp, lat, kp, lat, dout, b, dq, dqp, dlat, dkp, nullptr,
                                                scale, st);
  if (dtype == 1)
    return launch_instance<R, PD, TPK, 1, true>(pp, q, qp, lat, kp, lat, dout, b, dq, dqp, dlat, dkp, nullptr,
                                                scale, st);
  return launch_instance<R, PD, TPK, 2, true>(pp, q, qp, lat, kp, lat, dout, b, dq, dqp, dlat, dkp, nullptr, scale,
                                              st);
}

template <int R>
cudaError_t launch_r(int Pd, int dtype, const PagedParams& pp, const void* q, const void* qp, const void* lat,
                     const void* kp, const void* dout, const Buffers& b, void* dq, void* dqp, void* dlat, void* dkp,
                     float scale, cudaStream_t st) {
  switch (Pd) {
    case 0: return launch_rp<R, 0>(dtype, pp, q, qp, lat, kp, dout, b, dq, dqp, dlat, dkp, scale, st);
    case 16: return launch_rp<R, 16>(dtype, pp, q, qp, lat, kp, dout, b, dq, dqp, dlat, dkp, scale, st);
    case 32: return launch_rp<R, 32>(dtype, pp, q, qp, lat, kp, dout, b, dq, dqp, dlat, dkp, scale, st);
    case 64: return launch_rp<R, 64>(dtype, pp, q, qp, lat, kp, dout, b, dq, dqp, dlat, dkp, scale, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_mla_bwd(int R, int Pd, int dtype, const PagedParams& pp, const void* q, const void* qp,
                           const void* lat, const void* kp, const void* dout, const Buffers& b, void* dq,
                           void* dqp, void* dlat, void* dkp, float scale, cudaStream_t st) {
  switch (R) {
    case 128: return launch_r<128>(Pd, dtype, pp, q, qp, lat, kp, dout, b, dq, dqp, dlat, dkp, scale, st);
    case 256: return launch_r<256>(Pd, dtype, pp, q, qp, lat, kp, dout, b, dq, dqp, dlat, dkp, scale, st);
    case 512: return launch_r<512>(Pd, dtype, pp, q, qp, lat, kp, dout, b, dq, dqp, dlat, dkp, scale, st);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_mla_dkdv_shared(int R, int Pd, int dtype, const PagedParams& pp, const void* q, const void* qp,
                                   const void* lat, const void* kp, const void* dout, const Buffers& b, void* dlat,
                                   void* dkp, float scale, cudaStream_t st) {
#define ATTN_MLA_SHARED(RR, PP, TT)                                                                                \
  launch_instance<RR, PP, RR / 32, TT, true>(pp, q, qp, lat, kp, lat, dout, b, nullptr, nullptr, dlat, dkp, nullptr, \
                                             scale, st, true)
#define ATTN_MLA_SHARED_P(RR)                                                                  \
  if (Pd == 0) return dtype == 1 ? ATTN_MLA_SHARED(RR, 0, 1) : ATTN_MLA_SHARED(RR, 0, 2);     \
  if (Pd == 64) return dtype == 1 ? ATTN_MLA_SHARED(RR, 64, 1) : ATTN_MLA_SHARED(RR, 64, 2); \
  return cudaErrorInvalidValue;
  if (dtype != 1 && dtype != 2) return cudaErrorInvalidValue;
  if (R == 256) { ATTN_MLA_SHARED_P(256) }
  if (R == 512) { ATTN_MLA_SHARED_P(512) }
  return cudaErrorInvalidValue;
#undef ATTN_MLA_SHARED_P
#undef ATTN_MLA_SHARED
}

}  // namespace pbwd
}  // namespace attn
