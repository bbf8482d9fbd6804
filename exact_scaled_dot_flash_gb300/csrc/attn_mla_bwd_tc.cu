// attn_mla_bwd_tc.cu - explicit instantiations of the tensor-core MLA
// backward (latent ranks 256 and 512, positional widths 0 and 64, F16 and BF16).
#include "attn_mla_bwd_tc.cuh"

namespace attn {
namespace mlabwd {

#define ATTN_MLA_BWD_INST(R, PD, BF)                                                                                 \
  template cudaError_t launch_mla_bwd_tc<R, PD, BF>(EncodeTiledFn, const PagedParams&, const void*, const void*,     \
                                                    const void*, const void*, const void*, const MlaArgs&,          \
                                                    cudaStream_t);
ATTN_MLA_BWD_INST(256, 0, true)
ATTN_MLA_BWD_INST(256, 64, true)
ATTN_MLA_BWD_INST(512, 0, true)
ATTN_MLA_BWD_INST(512, 64, true)
ATTN_MLA_BWD_INST(256, 0, false)
ATTN_MLA_BWD_INST(256, 64, false)
ATTN_MLA_BWD_INST(512, 0, false)
ATTN_MLA_BWD_INST(512, 64, false)
#undef ATTN_MLA_BWD_INST

}  // namespace mlabwd

cudaError_t pbwd::launch_mla_bwd_tc(EncodeTiledFn enc, int R, int Pd, bool bf16, const PagedParams& pp,
                                    const void* q, const void* qp, const void* lat, const void* kp, const void* dout,
                                    const Buffers& b, void* dq, void* dqp, void* dlat, void* dkp, float scale,
                                    cudaStream_t st) {
  const mlabwd::MlaArgs a{b.lse2, b.dsum, b.offsets, dq, dqp, dlat, dkp, scale};
  using mlabwd::launch_mla_bwd_tc;
  if (R == 512 && Pd == 64)
    return bf16 ? launch_mla_bwd_tc<512, 64, true>(enc, pp, q, qp, lat, kp, dout, a, st)
                : launch_mla_bwd_tc<512, 64, false>(enc, pp, q, qp, lat, kp, dout, a, st);
  if (R == 512 && Pd == 0)
    return bf16 ? launch_mla_bwd_tc<512, 0, true>(enc, pp, q, qp, lat, kp, dout, a, st)
                : launch_mla_bwd_tc<512, 0, false>(enc, pp, q, qp, lat, kp, dout, a, st);
  if (R == 256 && Pd == 64)
    return bf16 ? launch_mla_bwd_tc<256, 64, true>(enc, pp, q, qp, lat, kp, dout, a, st)
                : launch_mla_bwd_tc<256, 64, false>(enc, pp, q, qp, lat, kp, dout, a, st);
  if (R == 256 && Pd == 0)
    return bf16 ? launch_mla_bwd_tc<256, 0, true>(enc, pp, q, qp, lat, kp, dout, a, st)
                : launch_mla_bwd_tc<256, 0, false>(enc, pp, q, qp, lat, kp, dout, a, st);
  return cudaErrorInvalidValue;
}

}  // namespace attn
