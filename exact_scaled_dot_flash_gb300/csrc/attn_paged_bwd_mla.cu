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

}  // namespace pbwd
}  // namespace attn
