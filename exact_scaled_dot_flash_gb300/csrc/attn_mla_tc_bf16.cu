// attn_mla_tc_bf16.cu - explicit instantiations of the tensor-core MLA kernel
// for BF16 (latent ranks 256 and 512, positional widths 0 and 64).
#include "attn_mla_tc.cuh"

namespace attn {
namespace mlatc {

#define ATTN_MLA_INST(R, PD)                                                                                 \
  template cudaError_t launch_mla_tc<R, PD, true>(EncodeTiledFn, const PagedParams&, const void*, const void*, \
                                                 const void*, const void*, void*, float*, cudaStream_t);
ATTN_MLA_INST(256, 0)
ATTN_MLA_INST(256, 64)
ATTN_MLA_INST(512, 0)
ATTN_MLA_INST(512, 64)
#undef ATTN_MLA_INST

}  // namespace mlatc
}  // namespace attn
