// attn_paged_bwd_tc.cu - instances of the tensor-core paged backward
// (attn_paged_bwd_tc.cuh): F16 and BF16, D in {64, 128}.
#include "attn_paged_bwd_tc.cuh"

namespace attn {
namespace pbwd {

template cudaError_t launch_paged_bwd_tc<64, false>(EncodeTiledFn, const PagedParams&, const void*, const void*,
                                                    const void*, const void*, const TcArgs&, cudaStream_t);
template cudaError_t launch_paged_bwd_tc<64, true>(EncodeTiledFn, const PagedParams&, const void*, const void*,
                                                   const void*, const void*, const TcArgs&, cudaStream_t);
template cudaError_t launch_paged_bwd_tc<128, false>(EncodeTiledFn, const PagedParams&, const void*, const void*,
                                                     const void*, const void*, const TcArgs&, cudaStream_t);
template cudaError_t launch_paged_bwd_tc<128, true>(EncodeTiledFn, const PagedParams&, const void*, const void*,
                                                    const void*, const void*, const TcArgs&, cudaStream_t);

}  // namespace pbwd
}  // namespace attn
