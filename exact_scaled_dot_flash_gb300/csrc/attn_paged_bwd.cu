// attn_paged_bwd.cu - the backward over a paged cache: workspace layout, row
// statistics, the reverse page index, and the paged-attention instances of
// the kernels in paged_bwd.cuh (the MLA instances are in
// attn_paged_bwd_mla.cu).
//
// Reverse page index (ruDNN user guide, section 11: the ordered history
// reduction keeps a reverse index from physical pages to their readers in
// its workspace). A table entry (s, b) is live when sequence s has queries,
// b < ceil(seq_len / page_size) and its page id lies in [0, num_pages); the
// index lists, per physical page, its live entries s * max_pages + b in
// ascending order. Built in four steps: count per page (integer atomics, whose
// result does not depend on their order), an exclusive scan into offsets, a
// scatter of each entry into its page's segment, and a sort of every segment,
// so the final order, and with it the summation order of the key-major
// kernel, is fixed.
#include "paged_bwd.cuh"

namespace attn {
namespace pbwd {

namespace {

constexpr float LOG2E = 1.4426950408889634f;

int64_t round256(int64_t x) { return (x + 255) / 256 * 256; }

// D_i = dout_i . out_i (0 for a row with no visible key) and lse_i * log2(e);
// 2^tpr_log2 threads per row of groups8 x 8 elements, 16-byte loads.
template <int DT>
__global__ void __launch_bounds__(256) preprocess_kernel(const void* out, const void* dout, const float* lse,
                                                         float* dsum, float* lse2, int64_t rows, int groups8,
                                                         int tpr_log2, int* status) {
  const int64_t r = (static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x) >> tpr_log2;
  const int tpr = 1 << tpr_log2;
  const int sub = threadIdx.x & (tpr - 1);
  float acc = 0.f;
  if (r < rows) {
    for (int g = sub; g < groups8; g += tpr) {
      float4 a0, a1, b0, b1;
      simt::load8<DT>(out, r * groups8 + g, rows * groups8, status, a0, a1);
      simt::load8<DT>(dout, r * groups8 + g, rows * groups8, status, b0, b1);
      acc = simt::dot4(a1, b1, simt::dot4(a0, b0, acc));
    }
  }
  for (int o = tpr >> 1; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (r < rows && sub == 0) {
    const float l = lse[r];
    dsum[r] = l == -INFINITY ? 0.f : acc;
    lse2[r] = l * LOG2E;
  }
}

__device__ __forceinline__ int live_page(const PagedParams& pp, int64_t entry) {
  const int s = static_cast<int>(entry / pp.max_pages);
  const int blk = static_cast<int>(entry - static_cast<int64_t>(s) * pp.max_pages);
  int q0, n;
  rows_of(pp, s, q0, n);
  if (n == 0 || static_cast<int64_t>(blk) * pp.page_size >= keys_of(pp, s)) return -1;
  const int pg = __ldg(pp.block_table + entry);
  return (pg >= 0 && pg < pp.num_pages) ? pg : -1;
}

__global__ void count_kernel(const PagedParams pp, int* count) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(pp.num_seqs) * pp.max_pages) return;
  const int pg = live_page(pp, e);
  if (pg >= 0 && in_bounds(pp.status, pg, pp.num_pages)) atomicAdd(count + pg, 1);
}

// offsets[p] = sum of count[0..p), offsets[n] = the total; one CTA.
__global__ void __launch_bounds__(1024) scan_kernel(const int* count, int* offsets, int n) {
  constexpr int ITEMS = 4;
  __shared__ int warp_sums[32];
  __shared__ int carry;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base < n; base += 1024 * ITEMS) {
    const int i0 = base + threadIdx.x * ITEMS;
    int v[ITEMS], sum = 0;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      v[k] = i0 + k < n ? count[i0 + k] : 0;
      sum += v[k];
    }
    int x = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, x, o);
      if (lane >= o) x += y;
    }
    if (lane == 31) warp_sums[warp] = x;
    __syncthreads();
    if (warp == 0) {
      int w = warp_sums[lane];
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, w, o);
        if (lane >= o) w += y;
      }
      warp_sums[lane] = w;
    }
    __syncthreads();
    int excl = carry + (warp ? warp_sums[warp - 1] : 0) + x - sum;
#pragma unroll
    for (int k = 0; k < ITEMS; ++k) {
      if (i0 + k < n) offsets[i0 + k] = excl;
      excl += v[k];
    }
    __syncthreads();  // every thread has read carry and warp_sums
    if (threadIdx.x == 1023) carry = excl;
    __syncthreads();
  }
  if (threadIdx.x == 0) offsets[n] = carry;
}

// Each live entry takes a slot of its page's segment (count runs down to 0).
__global__ void fill_kernel(const PagedParams pp, int* count, const int* offsets, int* refs) {
  const int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (e >= static_cast<int64_t>(pp.num_seqs) * pp.max_pages) return;
  const int pg = live_page(pp, e);
  if (pg < 0) return;
  if (!in_bounds(pp.status, pg, pp.num_pages)) return;
  const int c = atomicSub(count + pg, 1);
  const int slot = offsets[pg + 1] - c;  // inside [offsets[pg], offsets[pg + 1])
  if (in_bounds(pp.status, slot, static_cast<int64_t>(pp.num_seqs) * pp.max_pages)) refs[slot] = static_cast<int>(e);
}

// Insertion sort of every page's segment (segments are short: one entry per
// sequence or block that reads the page); pages whose reader count is not one
// join the list (in any order: each is computed on its own).
__global__ void sort_kernel(const int* offsets, int* refs, int* list, int pages, int64_t nrefs, int* status) {
  const int p = blockIdx.x * blockDim.x + threadIdx.x;
  if (p >= pages) return;
  const int lo = offsets[p], hi = offsets[p + 1];
  if (!range_in_bounds(status, lo, hi - lo, nrefs)) return;
  if (hi - lo != 1) {
    const int li = 1 + atomicAdd(list, 1);
    if (in_bounds(status, li, static_cast<int64_t>(pages) + 1)) list[li] = p;
  }
  for (int i = lo + 1; i < hi; ++i) {
    const int x = refs[i];
    int j = i - 1;
    while (j >= lo && refs[j] > x) {
      refs[j + 1] = refs[j];
      --j;
    }
    refs[j + 1] = x;
  }
}

}  // namespace

Layout layout(int64_t rows, int64_t num_pages, int64_t table_entries) {
  Layout l{};
  l.dsum = 0;
  l.lse2 = round256(rows * 4);
  l.count = l.lse2 + round256(rows * 4);
  l.offsets = l.count + round256(num_pages * 4);
  l.refs = l.offsets + round256((num_pages + 1) * 4);
  l.list = l.refs + round256(table_entries * 4);
  l.total = l.list + round256((num_pages + 1) * 4);
  return l;
}

Buffers carve(void* workspace, const Layout& lay) {
  uint8_t* w = static_cast<uint8_t*>(workspace);
  return Buffers{reinterpret_cast<float*>(w + lay.dsum), reinterpret_cast<float*>(w + lay.lse2),
                 reinterpret_cast<int*>(w + lay.count), reinterpret_cast<int*>(w + lay.offsets),
                 reinterpret_cast<int*>(w + lay.refs), reinterpret_cast<int*>(w + lay.list)};
}

cudaError_t launch_preprocess(int dtype, int width, const void* out, const void* dout, const float* lse,
                              const Buffers& b, int64_t rows, cudaStream_t st, int* status) {
  const int groups8 = width / 8;  // widths are multiples of 16
  int tpr_log2 = 0;
  while ((2 << tpr_log2) <= groups8 && (2 << tpr_log2) <= 32) ++tpr_log2;
  const int64_t blocks = ((rows << tpr_log2) + 255) / 256;
  if (blocks <= 0) return cudaSuccess;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned nb = static_cast<unsigned>(blocks);
  if (dtype == 0)
    preprocess_kernel<0><<<nb, 256, 0, st>>>(out, dout, lse, b.dsum, b.lse2, rows, groups8, tpr_log2, status);
  else if (dtype == 1)
    preprocess_kernel<1><<<nb, 256, 0, st>>>(out, dout, lse, b.dsum, b.lse2, rows, groups8, tpr_log2, status);
  else
    preprocess_kernel<2><<<nb, 256, 0, st>>>(out, dout, lse, b.dsum, b.lse2, rows, groups8, tpr_log2, status);
  return cudaGetLastError();
}

cudaError_t launch_page_index(const PagedParams& pp, const Buffers& b, cudaStream_t st) {
  if (pp.num_pages <= 0) return cudaSuccess;
  cudaError_t e = cudaMemsetAsync(b.count, 0, static_cast<size_t>(pp.num_pages) * 4, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(b.list, 0, 4, st);
  if (e != cudaSuccess) return e;
  const int64_t entries = static_cast<int64_t>(pp.num_seqs) * pp.max_pages;
  const unsigned eb = static_cast<unsigned>((entries + 255) / 256);
  if (eb > 0) count_kernel<<<eb, 256, 0, st>>>(pp, b.count);
  scan_kernel<<<1, 1024, 0, st>>>(b.count, b.offsets, pp.num_pages);
  if (eb > 0) fill_kernel<<<eb, 256, 0, st>>>(pp, b.count, b.offsets, b.refs);
  sort_kernel<<<static_cast<unsigned>((pp.num_pages + 255) / 256), 256, 0, st>>>(b.offsets, b.refs, b.list,
                                                                                  pp.num_pages, entries, pp.status);
  return cudaGetLastError();
}

cudaError_t launch_paged_bwd(int D, int dtype, const PagedParams& pp, const void* q, const void* k,
                             const void* v, const void* dout, const Buffers& b, void* dq, void* dk, void* dv,
                             float scale, cudaStream_t st) {
#define ATTN_PBWD(DD, TT) \
  launch_instance<DD, 0, 4, TT, false>(pp, q, nullptr, k, nullptr, v, dout, b, dq, nullptr, dk, nullptr, dv, scale, st)
#define ATTN_PBWD_D(DD) \
  case DD: return dtype == 0 ? ATTN_PBWD(DD, 0) : dtype == 1 ? ATTN_PBWD(DD, 1) : ATTN_PBWD(DD, 2);
  switch (D) {
    ATTN_PBWD_D(16)
    ATTN_PBWD_D(32)
    ATTN_PBWD_D(64)
    ATTN_PBWD_D(128)
    default: return cudaErrorInvalidValue;
  }
#undef ATTN_PBWD_D
#undef ATTN_PBWD
}

cudaError_t launch_paged_dkdv_shared(int D, int dtype, const PagedParams& pp, const void* q, const void* k,
                                     const void* v, const void* dout, const Buffers& b, void* dk, void* dv,
                                     float scale, cudaStream_t st) {
#define ATTN_PBWD(DD, TT)                                                                                   \
  launch_instance<DD, 0, 4, TT, false>(pp, q, nullptr, k, nullptr, v, dout, b, nullptr, nullptr, dk, nullptr, dv, \
                                       scale, st, true)
  switch (D) {
    case 64: return dtype == 1 ? ATTN_PBWD(64, 1) : ATTN_PBWD(64, 2);
    case 128: return dtype == 1 ? ATTN_PBWD(128, 1) : ATTN_PBWD(128, 2);
    default: return cudaErrorInvalidValue;
  }
#undef ATTN_PBWD
}

}  // namespace pbwd
}  // namespace attn
