// attn_bwd_tc_bf16.cu - explicit instantiations of the tensor-core backward for
// BF16 inputs: head dims 64 and 128, with and without an additive bias.
#include "attn_bwd_tc.cuh"

namespace attn {
namespace bwdtc {

#define ATTN_BWD_INST(D, BIAS)                                                                 \
  template cudaError_t launch_bwd_tc_instance<D, true, BIAS>(EncodeTiledFn, const void*, const void*, \
                                                          const void*, const void*,             \
                                                          const KernelParams&, const BwdArgs&,  \
                                                          cudaStream_t);
ATTN_BWD_INST(64, false)
ATTN_BWD_INST(64, true)
ATTN_BWD_INST(128, false)
ATTN_BWD_INST(128, true)
#undef ATTN_BWD_INST

}  // namespace bwdtc
}  // namespace attn
