// seq_order.cuh - longest-first order of the sequences of a paged call.
//
// The CTAs of a paged kernel are launched sequence by sequence, and the
// sequences of a serving batch differ in length by up to an order of
// magnitude; launched in batch order, the last waves can hold the longest
// sequences and leave most SMs idle at the end. In a decode-shaped call (one
// row block per sequence) a CTA's duration follows its sequence's key count,
// so every CTA ranks the sequences by key count (descending; ties by index)
// and takes the sequence of the rank it was launched for: the longest CTAs
// start first. Ranking costs each CTA one read of the metadata and
// num_seqs^2 / threads comparisons in shared memory; above kMaxRanked
// sequences the batch order is kept.
#pragma once

#include "params.h"

namespace attn {

constexpr int kMaxRanked = 256;

__device__ __forceinline__ int seq_keys(const PagedParams& pp, int s) {
  return min(max(__ldg(pp.seq_lens + s), 0), pp.max_pages * pp.page_size);
}

// The sequence of rank `rank` (0 = most keys). Every thread of the CTA must
// call it: it stages the key counts in shared memory and synchronises.
__device__ __forceinline__ int seq_by_rank(const PagedParams& pp, int rank) {
  if (pp.num_seqs > kMaxRanked) return rank;
  __shared__ int work[kMaxRanked];
  __shared__ int chosen;
  for (int i = threadIdx.x; i < pp.num_seqs; i += blockDim.x) work[i] = seq_keys(pp, i);
  if (threadIdx.x == 0) chosen = rank;  // every rank is held by exactly one sequence
  __syncthreads();
  for (int i = threadIdx.x; i < pp.num_seqs; i += blockDim.x) {
    const int wi = work[i];
    int r = 0;
    for (int j = 0; j < pp.num_seqs; ++j) r += (work[j] > wi) || (work[j] == wi && j < i);
    if (r == rank) chosen = i;
  }
  __syncthreads();
  return chosen;
}

}  // namespace attn
