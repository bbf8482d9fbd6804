// attn_tc_f16.cu - explicit instantiations of the tensor-core kernel for
// F16 inputs, writing O: head dims 32, 64, 128; no bias, bias read
// directly, bias staged through shared memory for D <= 64.
#include "attn_tc.cuh"

namespace attn {
namespace tc {

#define ATTN_TC_INST(D, MODE)                                                             \
  template cudaError_t launch_tc_instance<D, false, MODE, EPI_O>(                       \
      EncodeTiledFn, const void*, const void*, const void*, void*, const KernelParams&,  \
      cudaStream_t);
ATTN_TC_INST(32, BIAS_NONE)
ATTN_TC_INST(32, BIAS_DIRECT)
ATTN_TC_INST(32, BIAS_STAGED)
ATTN_TC_INST(64, BIAS_NONE)
ATTN_TC_INST(64, BIAS_DIRECT)
ATTN_TC_INST(64, BIAS_STAGED)
ATTN_TC_INST(128, BIAS_NONE)
ATTN_TC_INST(128, BIAS_DIRECT)
#undef ATTN_TC_INST

}  // namespace tc
}  // namespace attn
