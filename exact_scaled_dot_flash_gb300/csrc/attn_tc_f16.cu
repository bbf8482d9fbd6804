// attn_tc_f16.cu - explicit instantiations of the tensor-core kernel for
// F16 inputs (head dims 32, 64, 128; with and without bias).
#include "attn_tc.cuh"

namespace attn {
namespace tc {

#define ATTN_TC_INST(D, BIAS)                                                             \
  template cudaError_t launch_tc_instance<D, false, BIAS>(                                  \
      EncodeTiledFn, const void*, const void*, const void*, void*, const KernelParams&,  \
      cudaStream_t);
ATTN_TC_INST(32, false)
ATTN_TC_INST(32, true)
ATTN_TC_INST(64, false)
ATTN_TC_INST(64, true)
ATTN_TC_INST(128, false)
ATTN_TC_INST(128, true)
#undef ATTN_TC_INST

}  // namespace tc
}  // namespace attn
