// paged_bwd.h - launchers of the paged-cache backward (attn_paged_bwd) and
// of the paged MLA backward (attn_paged_mla_bwd); kernels in attn_paged_bwd.cu.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "params.h"

namespace attn {
namespace pbwd {

// Device scratch of one backward call, carved from the caller's workspace:
// per-row D_i and lse_i (log2 units), then the reverse page index (per
// physical page its count, its offset into refs, and refs: the table entries
// s * max_pages + b that read it, ascending), then the list of the pages whose
// reader count is not one (list[0] = their number, list[1..] the pages).
struct Layout {
  int64_t dsum, lse2, count, offsets, refs, list, total;  // byte offsets, total size
};
Layout layout(int64_t rows, int64_t num_pages, int64_t table_entries);

struct Buffers {
  float* dsum;
  float* lse2;
  int* count;
  int* offsets;
  int* refs;
  int* list;
};
Buffers carve(void* workspace, const Layout& lay);

// Row statistics of the nq * heads rows of out/dout ([rows, width] in dtype);
// `status`: the device status word (bounds-checked build).
cudaError_t launch_preprocess(int dtype, int width, const void* out, const void* dout, const float* lse,
                              const Buffers& b, int64_t rows, cudaStream_t st, int* status = nullptr);

// The reverse page index of every table entry that a sequence with queries
// reads (block b < ceil(seq_len / page_size), page id in [0, num_pages)).
cudaError_t launch_page_index(const PagedParams& pp, const Buffers& b, cudaStream_t st);

// Paged attention: dq [nq, Hq, D], dk/dv [pages, page_size, Hkv, D]; any
// output may be nullptr (not computed). D in {16, 32, 64, 128}.
cudaError_t launch_paged_bwd(int D, int dtype, const PagedParams& pp, const void* q, const void* k,
                             const void* v, const void* dout, const Buffers& b, void* dq, void* dk, void* dv,
                             float scale, cudaStream_t st);

// Key-major pass of the fp32 FMA kernels over the pages whose reader count
// is not one (no reader: zeros; shared: every reader in order), after the
// tensor-core pass has written the pages with exactly one reader.
cudaError_t launch_paged_dkdv_shared(int D, int dtype, const PagedParams& pp, const void* q, const void* k,
                                     const void* v, const void* dout, const Buffers& b, void* dk, void* dv,
                                     float scale, cudaStream_t st);

// Tensor-core paged backward (F16/BF16, D in {64, 128}, page_size a multiple
// of 8 dividing 128 or a multiple of 128): dq for every row, and dk/dv for the
// pages with exactly one reader (when dk or dv is given).
struct TcArgs {
  const float* lse2;
  const float* dsum;
  const int* offsets;  // the reverse index's per-page offsets (reader counts)
  void* dq;
  void* dk;
  void* dv;
  float scale;
};
template <int D, bool BF16>
cudaError_t launch_paged_bwd_tc(EncodeTiledFn enc, const PagedParams& pp, const void* q, const void* k,
                                const void* v, const void* dout, const TcArgs& a, cudaStream_t st);

// Tensor-core paged MLA backward (F16/BF16: bf16 selects BF16; R in {256,
// 512}, Pd in {0, 64}, page_size a multiple of 8 dividing 128 or a multiple of
// 128): dq, dqp for every row and dlatent, dkpos for the pages with exactly
// one reader (b's reverse index; outputs may be nullptr).
cudaError_t launch_mla_bwd_tc(EncodeTiledFn enc, int R, int Pd, bool bf16, const PagedParams& pp, const void* q,
                              const void* qp, const void* lat, const void* kp, const void* dout, const Buffers& b,
                              void* dq, void* dqp, void* dlat, void* dkp, float scale, cudaStream_t st);

// Key-major fp32 FMA pass of paged MLA over the pages whose reader count is
// not one, after the tensor-core kernels (R in {256, 512}, Pd in {0, 64},
// dtype 1 f16 or 2 bf16).
cudaError_t launch_mla_dkdv_shared(int R, int Pd, int dtype, const PagedParams& pp, const void* q, const void* qp,
                                   const void* lat, const void* kp, const void* dout, const Buffers& b, void* dlat,
                                   void* dkp, float scale, cudaStream_t st);

// Paged MLA (Hq = heads, Hkv = 1): dq [nq, H, R], dqp [nq, H, Pd], dlatent
// [pages, page_size, R], dkpos [pages, page_size, Pd]; outputs may be nullptr.
// R in {128, 256, 512}, Pd in {0, 16, 32, 64}.
cudaError_t launch_mla_bwd(int R, int Pd, int dtype, const PagedParams& pp, const void* q, const void* qp,
                           const void* lat, const void* kp, const void* dout, const Buffers& b, void* dq,
                           void* dqp, void* dlat, void* dkp, float scale, cudaStream_t st);

}  // namespace pbwd
}  // namespace attn
