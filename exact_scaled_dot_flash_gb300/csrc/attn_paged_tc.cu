// attn_paged_tc.cu - explicit instantiations of the tensor-core paged kernel
// (F16/BF16, head dims 64 and 128).
#include "attn_paged_tc.cuh"

namespace attn {
namespace pagedtc {

#define ATTN_PAGED_INST(D, BF)                                                                        \
  template cudaError_t launch_paged_tc<D, BF>(EncodeTiledFn, const PagedParams&, const void*, const void*, \
                                              const void*, void*, float*, cudaStream_t);
ATTN_PAGED_INST(64, true)
ATTN_PAGED_INST(64, false)
ATTN_PAGED_INST(128, true)
ATTN_PAGED_INST(128, false)
#undef ATTN_PAGED_INST

}  // namespace pagedtc
}  // namespace attn
