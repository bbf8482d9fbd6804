/*
 * attn.h - C ABI of the exact scaled-dot-product attention library
 * (libattn.so) for GB300 / sm_103a: the dense forward (attn_fwd, with key
 * splits and the log-sum-exp in attn_fwd_split, on host buffers in
 * attn_fwd_host), its backward (attn_bwd), attention and MLA over a paged
 * cache (attn_paged_fwd, attn_paged_mla) and their backward (attn_paged_bwd,
 * attn_paged_mla_bwd). Each entry below states its own definition and source.
 *
 * The operation, per batch b, query head hq and query row i:
 *
 *   s_j = scale * dot(Q[b,hq,i,:], K[b,hk,j,:]) + bias[b,hq,i,j]   (visible j)
 *   s_j = -inf                                                      (masked j)
 *   O[b,hq,i,:] = sum_j softmax_j(s) * V[b,hk,j,:],   hk = hq / (Hq / Hkv)
 *
 * Definition sources (page title, section):
 *  - "RustによるHOF認知Flash Attention実装の手引き" (HOF cognitive Flash
 *    Attention in Rust), section 4 "Kernel": exact scaled dot-product
 *    attention; exp of the scores divided by the row sum gives row-stochastic
 *    weights A; the output is A.V. Sections 2 and 4: a tiled FlashAttention
 *    kernel gives the same exact result without materialising the n x n
 *    score matrix in HBM (this library never writes it).
 *  - tensai autograd guide, "Attention の組み立て": (batch, head, seq,
 *    headDim) layout; scale Q.K^T, then add the mask, then softmax over the
 *    last axis; causal mask 0 on/below the diagonal, -inf above.
 *  - ruDNN user guide, section 2 (Attention): query, key, value, optional
 *    mask, optional attn_bias, options; errors are returned, not raised.
 *    Section 9: contiguous unquantised F32/F16/BF16 inputs of one dtype,
 *    Hq divisible by Hkv, a finite positive scale. Section 7: statistics in
 *    FP32, the output cast to the input dtype.
 *
 * Readings where the pages are silent: the causal diagonal is aligned
 * bottom-right (key j visible to row i when j <= i + Sk - Sq); key padding
 * masks keys j >= clamp(kv_lens[b], 0, Sk) and never query rows; a masked
 * position stays -inf whatever the bias; a row with no visible key has an
 * undefined softmax and its output is NaN.
 */
#ifndef ATTN_H_
#define ATTN_H_

#include <stddef.h>
#include <stdint.h>

/* The library is built with hidden visibility; only these entry points are
 * exported, so two copies of it loaded in one process never resolve each
 * other's internal (kernel) symbols. */
#if defined(__GNUC__)
#define ATTN_API __attribute__((visibility("default")))
#else
#define ATTN_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of Q, K, V and O. */
typedef enum { ATTN_F32 = 0, ATTN_F16 = 1, ATTN_BF16 = 2 } attn_dtype_t;

/* Mask kinds: bit flags, ATTN_MASK_CAUSAL | ATTN_MASK_KEY_PADDING = both. */
enum {
  ATTN_MASK_NONE = 0,
  ATTN_MASK_CAUSAL = 1,
  ATTN_MASK_KEY_PADDING = 2
};

/* Status codes: 0 is success, errors are negative. */
enum {
  ATTN_OK = 0,
  ATTN_ERR_NULL = -1,      /* a required pointer is NULL                              */
  ATTN_ERR_SHAPE = -2,     /* a dimension is out of range, Hq % Hkv != 0, bad bias dims */
  ATTN_ERR_DTYPE = -3,     /* unknown dtype                                           */
  ATTN_ERR_HEAD_DIM = -4,  /* D has no compiled kernel for this dtype                 */
  ATTN_ERR_ALIGN = -5,     /* a pointer is not 16-byte aligned                        */
  ATTN_ERR_SCALE = -6,     /* scale is not finite and positive                        */
  ATTN_ERR_MASK = -7,      /* unknown mask bits, or KEY_PADDING with kv_lens == NULL  */
  ATTN_ERR_OVERLAP = -8,   /* out overlaps q, k, v, kv_lens or bias                   */
  ATTN_ERR_CUDA = -9,      /* a CUDA call failed; see attn_last_cuda_error()          */
  ATTN_ERR_TIMEOUT = -10,  /* a kernel gave up on a bounded wait (see attn_device_status) */
  ATTN_ERR_SPLITS = -11,   /* num_splits outside [1, ATTN_MAX_SPLITS]                 */
  ATTN_ERR_WORKSPACE = -12,/* split workspace NULL or smaller than required           */
  ATTN_ERR_SCRATCH = -13   /* attn_fwd_split_noalloc: problem needs more scratch than
                              ATTN_NOALLOC_SCRATCH_BYTES                              */
};

/* Largest num_splits attn_fwd_split accepts. */
#define ATTN_MAX_SPLITS 32

/* Problem shape. All counts are elements.
 *   Q   [B, Hq,  Sq, D]   contiguous, row-major
 *   K,V [B, Hkv, Sk, D]   contiguous, row-major
 *   O   [B, Hq,  Sq, D]   contiguous, row-major
 *   bias (fp32) [bias_b, bias_h, Sq, Sk] with bias_b in {1, B}, bias_h in {1, Hq};
 *   a size-1 axis broadcasts. bias_b / bias_h are read only when bias != NULL. */
typedef struct {
  int32_t B, Hq, Hkv, Sq, Sk, D;
  int32_t bias_b, bias_h;
} attn_shape_t;

/* attn_fwd - exact attention forward on the GPU, asynchronous on `stream`.
 *
 * q, k, v, out: device pointers to contiguous tensors of `dtype` (layouts
 *   above), each 16-byte aligned. `out` is written entirely (rows with no
 *   visible key become NaN) and must not overlap any input.
 * mask_kind: ATTN_MASK_* bits. ATTN_MASK_KEY_PADDING needs kv_lens.
 * kv_lens: device int32[B] valid key counts (clamped to [0, Sk] on the
 *   device), or NULL without ATTN_MASK_KEY_PADDING.
 * bias: device fp32 [bias_b, bias_h, Sq, Sk] (16-byte aligned) or NULL; it is
 *   added to the scaled scores and indexed by the query head.
 * scale: multiplies Q.K^T; finite and > 0 (typically 1/sqrt(D)).
 * stream: a cudaStream_t, or NULL for the legacy default stream.
 *
 * Supported head dims: D in {32, 64, 128} for F16/BF16 (tensor-core path),
 * D in {16, 32, 64, 128} for F32 (fp32 FMA path). B or Sq equal to 0 is a
 * no-op; Sk equal to 0 gives NaN rows. Hq, Hkv, D must be positive.
 *
 * Ownership: the caller owns every buffer; the library keeps no pointer after
 * returning and allocates no device memory. The call does not synchronise;
 * argument errors are reported before anything is launched. Thread-safe.
 * Returns ATTN_OK or a negative ATTN_ERR_* code. */
ATTN_API int attn_fwd(const attn_shape_t* shape,
             const void* q, const void* k, const void* v,
             int mask_kind, const int32_t* kv_lens,
             const float* bias,
             float scale, attn_dtype_t dtype,
             void* out,
             void* stream);

/* attn_fwd_split - attn_fwd with the key range of each query row cut into
 * `num_splits` parts that run as separate CTAs, and an optional row
 * log-sum-exp output.
 *
 * Source: ruDNN user guide, section 9: a long key history is split into
 * parts, each part keeps FP32 partial statistics, and the parts are merged.
 * Part s of a row keeps its running maximum m_s, its exp-sum l_s and its
 * unnormalised output O_s; the merge rescales each part by exp(m_s - M),
 * M = max_s m_s, and divides by the rescaled sum, which equals the softmax
 * over all keys. Splitting gives the GPU enough CTAs when B*Hq*ceil(Sq/256)
 * is small (few long rows: chunked prefill, decode).
 *
 * Arguments are those of attn_fwd, plus:
 * num_splits: 1..ATTN_MAX_SPLITS. Each (batch, head, 256-row query block)
 *   cuts its visible key tiles into num_splits balanced contiguous runs
 *   (a run may be empty when there are fewer tiles than splits). 1 runs the
 *   attn_fwd kernel unchanged and needs no workspace.
 * workspace, workspace_bytes: device scratch of at least
 *   attn_split_workspace_bytes(shape, num_splits) bytes, 16-byte aligned,
 *   owned by the caller, disjoint from every other buffer; ignored (may be
 *   NULL) when num_splits == 1. Its contents on entry do not matter and are
 *   meaningless afterwards; two calls in flight at once need two workspaces.
 * lse: NULL, or device float [B, Hq, Sq] (4-byte aligned, disjoint from the
 *   rest) that receives the natural-log row log-sum-exp
 *   lse = log sum_j exp(s_j) over the visible keys (-inf for a row with no
 *   visible key, whose output is NaN).
 *
 * With num_splits > 1 the result is the same softmax evaluated in a
 * different summation order, so it agrees with attn_fwd to rounding, not
 * bit for bit. Asynchronous on `stream` (two kernels when num_splits > 1).
 * Returns ATTN_OK or a negative ATTN_ERR_* code (ATTN_ERR_SPLITS,
 * ATTN_ERR_WORKSPACE in addition to attn_fwd's). */
ATTN_API int attn_fwd_split(const attn_shape_t* shape,
                   const void* q, const void* k, const void* v,
                   int mask_kind, const int32_t* kv_lens,
                   const float* bias,
                   float scale, attn_dtype_t dtype,
                   int num_splits, void* workspace, size_t workspace_bytes,
                   void* out, float* lse,
                   void* stream);

/* attn_split_workspace_bytes - bytes of workspace attn_fwd_split needs for
 * `shape` and `num_splits` (0 when num_splits == 1):
 * num_splits*B*Hq*Sq*(4*D + 8) plus up to 255 bytes of alignment padding.
 * Writes *bytes. Returns ATTN_OK, ATTN_ERR_NULL, ATTN_ERR_SHAPE or
 * ATTN_ERR_SPLITS. */
ATTN_API int attn_split_workspace_bytes(const attn_shape_t* shape, int num_splits, size_t* bytes);

/* attn_bwd - gradients of attention: dq, dk, dv for a loss whose gradient
 * with respect to the output is `dout`. Asynchronous on `stream`.
 *
 * Source: ruDNN user guide, section 11: the backward returns dq, dk and dv and
 * recomputes the probabilities instead of storing the score matrix; its
 * ordered variant accumulates without atomics in a fixed order, which this
 * call does (bit-identical results on repeated calls). With the forward's row
 * log-sum-exp lse_i, for every visible (i, j):
 *   p_ij = exp(scale*q_i.k_j + bias_ij - lse_i),  dp_ij = dout_i . v_j,
 *   D_i = dout_i . out_i,  ds_ij = p_ij * (dp_ij - D_i),
 *   dv_j = sum_i p_ij dout_i,  dk_j = scale * sum_i ds_ij q_i,
 *   dq_i = scale * sum_j ds_ij k_j,
 * dk and dv summed over the query heads that share a key/value head (GQA).
 * The bias is a constant (no bias gradient). A row with no visible key
 * (lse = -inf) contributes nothing and gets dq = 0.
 *
 * shape, q, k, v, mask_kind, kv_lens, bias, scale, dtype: exactly as given to
 *   the forward call.
 * out: the forward output O [B, Hq, Sq, D] (dtype); dout: dL/dO, same layout.
 * lse: the forward's row log-sum-exp, float [B, Hq, Sq] (from attn_fwd_split).
 * workspace, workspace_bytes: device scratch of at least
 *   attn_bwd_workspace_bytes(shape) bytes, 16-byte aligned, caller-owned.
 * dq [B, Hq, Sq, D], dk, dv [B, Hkv, Sk, D]: outputs in dtype, 16-byte aligned,
 *   written entirely, disjoint from every input, each other and the workspace.
 *
 * Head dims: D in {16, 32, 64, 128} for every dtype. B = 0 is a no-op; Sq = 0
 * gives dk = dv = 0; Sk = 0 gives dq = 0. Returns ATTN_OK or a negative
 * ATTN_ERR_* code (validation before any launch). */
ATTN_API int attn_bwd(const attn_shape_t* shape,
                      const void* q, const void* k, const void* v,
                      const void* out, const void* dout, const float* lse,
                      int mask_kind, const int32_t* kv_lens,
                      const float* bias,
                      float scale, attn_dtype_t dtype,
                      void* workspace, size_t workspace_bytes,
                      void* dq, void* dk, void* dv,
                      void* stream);

/* attn_bwd_workspace_bytes - workspace attn_bwd needs for `shape`: two float
 * arrays of B*Hq*Sq, each rounded up to 256 bytes. Writes *bytes. Returns
 * ATTN_OK, ATTN_ERR_NULL or ATTN_ERR_SHAPE. */
ATTN_API int attn_bwd_workspace_bytes(const attn_shape_t* shape, size_t* bytes);

/* Shape of a paged-cache call. Counts are elements.
 *   q, out  [num_queries, Hq, D]           packed queries, sequence by sequence
 *   k_cache, v_cache [num_pages, page_size, Hkv, D]   physical pages
 *   block_table [num_seqs, max_pages] int32   physical page of key block b of sequence s
 *   max_queries: an upper bound on the queries of one sequence (sizes the grid;
 *   a call with at most 8 rows of queries x (Hq/Hkv) heads per sequence and kv
 *   head is decode-shaped, the only shape that splits). Rows beyond a bound
 *   that is too small are not written.
 * F16/BF16 calls with D in {64, 128} and a page size that is a multiple of 8
 * dividing 128 or a multiple of 128 run on the tensor cores, the query heads
 * of a GQA group packed into the rows of one tile; the rest on fp32 FMA
 * kernels. */
typedef struct {
  int32_t num_seqs, num_queries, Hq, Hkv, D;
  int32_t page_size, num_pages, max_pages, max_queries;
} attn_paged_shape_t;

/* attn_paged_fwd - attention of packed variable-length queries over a paged
 * key/value cache (prefill chunks and decode steps in one call).
 *
 * Source: ruDNN user guide, section 9 (paged attention): the call reads the
 * physical cache pages through per-sequence page tables, handles packed
 * prefill and decode, maps query head hq to key/value head hq / (Hq / Hkv),
 * and applies the causal mask by absolute position.
 *
 * Key j of sequence s is row j % page_size of page block_table[s][j / page_size];
 * sequence s has seq_lens[s] keys (clamped to [0, max_pages * page_size]). Its
 * queries are rows q_offsets[s] .. q_offsets[s+1]-1 of q (offsets clamped to
 * [0, num_queries]); a query row outside every range is not written. With
 * causal = 1 the query at position p sees keys j <= p; positions (int32
 * [num_queries], zero-based, absolute within the sequence) may be NULL, which
 * places the n queries of a sequence of length L at L - n .. L - 1. A row that
 * sees no key is NaN (lse -inf). lse: NULL or float [num_queries, Hq] natural
 * log-sum-exp.
 *
 * num_splits (1..ATTN_MAX_SPLITS) cuts the keys of every sequence and head
 * of a decode-shaped call (max_queries * Hq/Hkv <= 8) into that many runs,
 * one CTA each, merged afterwards from FP32 partial statistics (the split of
 * attn_fwd_split); it needs a 16-byte-aligned workspace of
 * attn_paged_workspace_bytes(shape, num_splits) bytes, disjoint from every
 * other buffer; other calls ignore num_splits and the workspace. With splits,
 * a query row outside every sequence range gets unspecified values.
 *
 * All pointers are device pointers: q, k_cache, v_cache, out 16-byte aligned;
 * the int32 arrays and lse 4-byte aligned; out and lse disjoint from every
 * input. Page-table entries outside [0, num_pages) read as zero keys and
 * values (no out-of-bounds access). D in {16, 32, 64, 128}, every dtype.
 * Asynchronous on `stream`; returns ATTN_OK or a negative ATTN_ERR_* code
 * (ATTN_ERR_MASK for causal not in {0, 1}). */
ATTN_API int attn_paged_fwd(const attn_paged_shape_t* shape,
                            const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_table, const int32_t* seq_lens,
                            const int32_t* q_offsets, const int32_t* positions,
                            int causal, float scale, attn_dtype_t dtype,
                            int num_splits, void* workspace, size_t workspace_bytes,
                            void* out, float* lse,
                            void* stream);

/* attn_paged_workspace_bytes - workspace attn_paged_fwd needs for `shape` and
 * `num_splits` (0 when the call does not split). Returns ATTN_OK,
 * ATTN_ERR_NULL, ATTN_ERR_SHAPE or ATTN_ERR_SPLITS. */
ATTN_API int attn_paged_workspace_bytes(const attn_paged_shape_t* shape, int num_splits, size_t* bytes);

/* Shape of an MLA call: q [num_queries, H, R], qp [num_queries, H, Pd],
 * latent [num_pages, page_size, 1, R], kpos [num_pages, page_size, 1, Pd],
 * out [num_queries, H, R]; block_table [num_seqs, max_pages]. */
typedef struct {
  int32_t num_seqs, num_queries, H, R, Pd;
  int32_t page_size, num_pages, max_pages, max_queries;
} attn_mla_shape_t;

/* attn_paged_mla - multi-head latent attention with absorbed projections over
 * a paged latent cache.
 *
 * Source: ruDNN user guide, section 9 (MLA): the query with the key
 * projection absorbed (q, width R, the latent rank) and a positional query
 * (qp, width Pd) attend over a cache of one shared latent row c_j and one
 * positional key kp_j per token; the output is the compressed context
 * out = sum_j softmax_j(scale * (q . c_j + qp . kp_j)) c_j, width R. Position
 * encoding is applied by the caller before the call, the value and output
 * projections after it; scale is the original model's QK scale.
 *
 * Paging, packed queries, positions (NULL = the newest tokens), the causal
 * mask, empty rows (NaN, lse -inf) and the trust in metadata are those of
 * attn_paged_fwd, with one key/value head shared by all H heads.
 * Supported: R in {128, 256, 512}, Pd in {0, 16, 32, 64}; every dtype. q, qp,
 * latent, kpos, out 16-byte aligned device pointers (qp, kpos may be NULL when
 * Pd == 0); lse NULL or float [num_queries, H]; num_queries * H < 2^31.
 *
 * num_splits (1..ATTN_MAX_SPLITS) cuts the key tiles of every 128-row block of
 * (query, head) rows into that many runs, one CTA each, merged afterwards
 * from FP32 partial statistics (the split of attn_fwd_split). With
 * num_splits > 1 a workspace of attn_paged_mla_workspace_bytes(shape,
 * num_splits) bytes is required (16-byte aligned, disjoint from every other
 * buffer); calls that run on the fp32 FMA kernel (F32, R = 128, Pd in
 * {16, 32}, or page sizes that are not a multiple of 8 dividing 64 or a
 * multiple of 64) ignore the splits. Asynchronous on `stream`; returns ATTN_OK
 * or a negative ATTN_ERR_* code. */
ATTN_API int attn_paged_mla(const attn_mla_shape_t* shape,
                            const void* q, const void* qp,
                            const void* latent, const void* kpos,
                            const int32_t* block_table, const int32_t* seq_lens,
                            const int32_t* q_offsets, const int32_t* positions,
                            int causal, float scale, attn_dtype_t dtype,
                            int num_splits, void* workspace, size_t workspace_bytes,
                            void* out, float* lse,
                            void* stream);

/* attn_paged_mla_workspace_bytes - workspace attn_paged_mla needs for `shape`
 * and `num_splits`: 0 when num_splits == 1, else
 * num_splits * num_queries * H * (4 R + 8) plus up to 255 bytes of padding.
 * Returns ATTN_OK, ATTN_ERR_NULL, ATTN_ERR_SHAPE or ATTN_ERR_SPLITS. */
ATTN_API int attn_paged_mla_workspace_bytes(const attn_mla_shape_t* shape, int num_splits, size_t* bytes);

/* attn_paged_bwd - gradients of attn_paged_fwd for a loss whose gradient with
 * respect to its output is `dout`: dq for the packed queries and the history
 * gradients dk_cache, dv_cache in the shape of the physical caches.
 * Asynchronous on `stream`.
 *
 * Source: ruDNN user guide, section 11 (backward of paged attention and
 * ordered history gradients): the backward returns dq, dk, dv, recomputes the
 * probabilities instead of storing the score matrix, may skip any gradient
 * the caller does not want, and has an ordered variant that reduces the cache
 * gradients without atomics through a workspace holding row statistics and a
 * reverse page index. This call is that ordered variant: every gradient is
 * summed in one fixed order (the readers of a page by ascending (sequence,
 * block), their query rows and heads ascending), so repeated calls give
 * identical bits. Per visible (query row i, key j), with the forward's lse_i:
 *   p_ij = exp(scale q_i.k_j - lse_i),  dp_ij = dout_i . v_j,
 *   D_i = dout_i . out_i,  ds_ij = p_ij (dp_ij - D_i),
 *   dq_i = scale sum_j ds_ij k_j,  dk_j = scale sum_i ds_ij q_i,  dv_j = sum_i p_ij dout_i.
 * A physical page read by several sequences (a shared prefix), or by one
 * sequence at several blocks, receives the sum of every read; a page that no
 * sequence with queries reads gets zeros. A row with no visible key (lse
 * -inf) contributes nothing and gets dq = 0.
 *
 * shape, q, k_cache, v_cache, block_table, seq_lens, q_offsets, positions,
 *   causal, scale, dtype: exactly as given to attn_paged_fwd (same metadata
 *   rules; page-table entries outside [0, num_pages) read as zero keys and
 *   receive nothing).
 * out, dout: the forward output and dL/dO, [num_queries, Hq, D] in dtype.
 * lse: the forward's float [num_queries, Hq] natural log-sum-exp.
 * workspace: at least attn_paged_bwd_workspace_bytes(shape) bytes, 16-byte
 *   aligned, caller-owned, disjoint from every other buffer.
 * dq [num_queries, Hq, D], dk_cache, dv_cache [num_pages, page_size, Hkv, D]:
 *   outputs in dtype, 16-byte aligned device pointers; each may be NULL (not
 *   computed). dk_cache and dv_cache are written entirely; dq rows outside
 *   every sequence's range (or beyond max_queries) are not written.
 * D in {16, 32, 64, 128}, every dtype. F16/BF16 calls with D in {64, 128} and a
 * page size that is a multiple of 8 dividing 128 or a multiple of 128 run on
 * the tensor cores (pages with exactly one reader written by them, the others
 * by an fp32 FMA pass over those pages); the rest on fp32 FMA kernels.
 * Returns ATTN_OK or a negative ATTN_ERR_* code (validation before any
 * launch). */
ATTN_API int attn_paged_bwd(const attn_paged_shape_t* shape,
                            const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_table, const int32_t* seq_lens,
                            const int32_t* q_offsets, const int32_t* positions,
                            int causal, float scale, attn_dtype_t dtype,
                            const void* out, const void* dout, const float* lse,
                            void* workspace, size_t workspace_bytes,
                            void* dq, void* dk_cache, void* dv_cache,
                            void* stream);

/* attn_paged_bwd_workspace_bytes - workspace attn_paged_bwd needs: two float
 * arrays of num_queries * Hq (row statistics), num_pages + num_pages + 1 ints
 * (reverse index counts and offsets), num_seqs * max_pages ints (the index)
 * and num_pages + 1 ints (the pages that do not have exactly one reader), each
 * rounded up to 256 bytes. Returns ATTN_OK, ATTN_ERR_NULL or ATTN_ERR_SHAPE. */
ATTN_API int attn_paged_bwd_workspace_bytes(const attn_paged_shape_t* shape, size_t* bytes);

/* attn_paged_mla_bwd - gradients of attn_paged_mla: dq [num_queries, H, R],
 * dqp [num_queries, H, Pd], and the cache-shaped dlatent [num_pages,
 * page_size, 1, R] and dkpos [num_pages, page_size, 1, Pd].
 *
 * Source: ruDNN user guide, section 11: the MLA backward returns dq, dqp,
 * dlatent and dkp, dlatent holding both the key and the value contribution of
 * each latent row. With s_ij = scale (q_i . c_j + qp_i . kp_j) and v_j = c_j:
 *   dc_j = sum_i (p_ij dout_i + scale ds_ij q_i),  dkp_j = scale sum_i ds_ij qp_i,
 *   dq_i = scale sum_j ds_ij c_j,  dqp_i = scale sum_j ds_ij kp_j.
 * Everything else (ordered summation, shared pages, skipped outputs, the
 * workspace of attn_paged_mla_bwd_workspace_bytes, edge cases) is as for
 * attn_paged_bwd with one latent head shared by all H heads. R in {128, 256,
 * 512}, Pd in {0, 16, 32, 64}, every dtype (fp32 FMA arithmetic); with Pd == 0,
 * qp, kpos, dqp and dkpos are ignored. */
ATTN_API int attn_paged_mla_bwd(const attn_mla_shape_t* shape,
                                const void* q, const void* qp,
                                const void* latent, const void* kpos,
                                const int32_t* block_table, const int32_t* seq_lens,
                                const int32_t* q_offsets, const int32_t* positions,
                                int causal, float scale, attn_dtype_t dtype,
                                const void* out, const void* dout, const float* lse,
                                void* workspace, size_t workspace_bytes,
                                void* dq, void* dqp, void* dlatent, void* dkpos,
                                void* stream);

/* attn_paged_mla_bwd_workspace_bytes - workspace attn_paged_mla_bwd needs (the
 * layout of attn_paged_bwd_workspace_bytes with Hq = H). Returns ATTN_OK,
 * ATTN_ERR_NULL or ATTN_ERR_SHAPE. */
ATTN_API int attn_paged_mla_bwd_workspace_bytes(const attn_mla_shape_t* shape, size_t* bytes);

/* Size of the device scratch array built into the library for
 * attn_fwd_split_noalloc (32 MiB per GPU that loads the library). */
#define ATTN_NOALLOC_SCRATCH_BYTES (32u << 20)

/* attn_fwd_split_noalloc - attn_fwd_split for callers that cannot allocate
 * device memory. (The pages have no counterpart; this is a calling
 * convention of this library.)
 *
 * Who needs it: code that may not call cudaMalloc, such as a plugin whose host
 * application passes it input and output buffers but no allocator, or a
 * service that forbids device allocation after start-up because cudaMalloc
 * and cudaFree can block and synchronise the device. Such a caller cannot
 * provide the workspace attn_fwd_split needs for num_splits > 1.
 *
 * Arguments and results are those of attn_fwd_split without the workspace:
 * the split partials go to a static device array of
 * ATTN_NOALLOC_SCRATCH_BYTES inside the library, which every GPU that loads
 * the library holds until the process exits. The call allocates nothing.
 * The caller still owns and passes q, k, v, kv_lens, bias, out and lse.
 *
 * Limit: problems with attn_split_workspace_bytes(shape, num_splits) above
 * ATTN_NOALLOC_SCRATCH_BYTES are rejected with ATTN_ERR_SCRATCH before
 * anything runs; lower num_splits, or use attn_fwd_split with a workspace.
 * num_splits == 1 uses no scratch.
 *
 * Shared state: all calls on a device use the same array, which keeps what
 * the last call wrote. Nothing in it has to start at zero: each call writes
 * every partial it later reads. Two calls whose kernels overlap on the GPU
 * (different streams, or different host threads, without ordering between
 * them) race on the array and may return wrong results; order them, for
 * example on one stream.
 *
 * Set-up: the first call with num_splits > 1 on a device looks up the
 * array's device address (cudaGetSymbolAddress, with that device current)
 * and caches it with the id of the current CUDA context; make that first
 * call before any stream capture begins. A call made in another context
 * than the cached one (after cudaDeviceReset or a primary-context reset,
 * which reload the library's device module and may move the array) looks
 * the address up again, as does every call after a failed lookup.
 *
 * A split CTA whose bounded wait expired (a nonzero attn_device_status
 * word) writes partials that make its rows NaN in out (and
 * their lse NaN), so a failed call never returns another call's partials.
 *
 * Returns ATTN_OK, ATTN_ERR_SCRATCH, ATTN_ERR_CUDA if the set-up fails (the
 * CUDA error code is then in attn_last_cuda_error), or any code of
 * attn_fwd_split. */
ATTN_API int attn_fwd_split_noalloc(const attn_shape_t* shape,
                                    const void* q, const void* k, const void* v,
                                    int mask_kind, const int32_t* kv_lens,
                                    const float* bias,
                                    float scale, attn_dtype_t dtype,
                                    int num_splits,
                                    void* out, float* lse,
                                    void* stream);

/* attn_strerror - static English text for a status code (never NULL). */
ATTN_API const char* attn_strerror(int code);

/* attn_last_cuda_error - the cudaError_t value of the last CUDA failure seen
 * by attn_fwd on the calling thread (0 if none). */
ATTN_API int attn_last_cuda_error(void);

/* Bits of the device status word (attn_device_status). */
#define ATTN_STATUS_TIMEOUT 1 /* a kernel gave up on a bounded wait and unwound */
#define ATTN_STATUS_BOUNDS 2  /* bounds-checked build only (libattn_checked.so, compiled
                                 with ATTN_CHECKED): a computed global or shared-memory
                                 index of a paged, MLA, split or backward kernel fell
                                 outside its buffer; the access was skipped */

/* attn_device_status - read (and, when clear != 0, reset) the sticky error
 * word that kernels on `device` set when a bounded wait expires (and, in the
 * bounds-checked build, when an index falls outside its buffer). Writes the
 * flags to *flags (0 = no failure seen; ATTN_STATUS_* bits otherwise).
 * Synchronises with the device. Each build of the library (libattn.so,
 * libattn_checked.so) has its own word. Returns ATTN_OK, ATTN_ERR_NULL or
 * ATTN_ERR_CUDA. */
ATTN_API int attn_device_status(int device, int* flags, int clear);

/* attn_fwd_host - attn_fwd on tensors in HOST memory: q, k, v, kv_lens, bias
 * and out are host pointers with attn_fwd's layouts and rules; the result is
 * identical to attn_fwd on device copies of the same inputs. (The pages have
 * no counterpart; this is the library's executor for host-resident tensors.)
 *
 * The problem is cut into chunks of whole (batch, kv head) units (about 8 in
 * all); two chunk slots live in `workspace` (device memory of at least
 * attn_fwd_host_workspace_bytes(shape, dtype, bias != NULL) bytes, 16-byte
 * aligned, owned by the caller). The upload of chunk c+1 (a library copy
 * stream), the attention of chunk c (on `stream`) and the download of chunk
 * c-1 (a second library copy stream) run at the same time; `stream` is
 * ordered after every copy when the call returns, so `out` is complete, and
 * the inputs may be released, once `stream` has completed. Pinned (page-locked)
 * host buffers make the copies asynchronous DMA; pageable ones work but the
 * copies then block the calling thread.
 *
 * Calls on one device are enqueued one at a time (a per-device lock); calls in
 * flight at once need separate workspaces. Allocates no device memory; creates
 * two streams and seven events per device on first use, kept until the
 * process exits. Returns ATTN_OK or a negative ATTN_ERR_* code (argument
 * errors before anything is enqueued; ATTN_ERR_WORKSPACE for a missing or
 * small workspace). */
ATTN_API int attn_fwd_host(const attn_shape_t* shape,
                           const void* q, const void* k, const void* v,
                           int mask_kind, const int32_t* kv_lens,
                           const float* bias,
                           float scale, attn_dtype_t dtype,
                           void* workspace, size_t workspace_bytes,
                           void* out,
                           void* stream);

/* attn_fwd_host_workspace_bytes - device workspace attn_fwd_host needs for
 * `shape`, `dtype` and whether a bias is passed (0 when B or Sq is 0): the
 * kv_lens array and two slots for the largest chunk's Q, K, V, O and bias.
 * Returns ATTN_OK, ATTN_ERR_NULL, ATTN_ERR_DTYPE or ATTN_ERR_SHAPE. */
ATTN_API int attn_fwd_host_workspace_bytes(const attn_shape_t* shape, attn_dtype_t dtype, int with_bias,
                                           size_t* bytes);

/* attn_selftest_wait_timeout - failure-path self-test (the pages have no
 * counterpart; it checks this library's own error reporting). Launches, on
 * `stream`, a one-thread kernel that waits on an mbarrier phase nothing
 * completes, with the same bounded-wait code the attention kernels use but a
 * limit of `limit_us` microseconds (1..5,000,000). On expiry the kernel sets
 * the timeout bit of the device status word (read it with attn_device_status)
 * and returns; the GPU context stays usable. Asynchronous; returns ATTN_OK,
 * ATTN_ERR_SHAPE for an out-of-range limit, or ATTN_ERR_CUDA. */
ATTN_API int attn_selftest_wait_timeout(unsigned int limit_us, void* stream);

/* attn_version - library version as major*10000 + minor*100 + patch. */
ATTN_API int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_H_ */
