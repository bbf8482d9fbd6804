/*
 * Float64 CPU oracle for exact scaled-dot-product attention (forward, and
 * the first-order backward at the end of this file).
 *
 * TEST INFRASTRUCTURE ONLY. This file is the slow, plain definition that the
 * GPU kernels are checked against. Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark may load it. It shares no code,
 * header, table or helper with the CUDA library, and it never reads a value
 * produced by the CUDA path.
 *
 * What it computes, for every batch b, query head hq and query row i:
 *
 *   s_j = scale * sum_d Q[b,hq,i,d] * K[b,hk,j,d] + bias[b,hq,i,j]   (visible j)
 *   s_j = -inf                                                        (masked j)
 *   w_j = exp(s_j - max_j s_j) / sum_j exp(s_j - max_j s_j)
 *   O[b,hq,i,:] = sum_j w_j * V[b,hk,j,:]
 *
 * Sources (by page title and section):
 *  - "RustによるHOF認知Flash Attention実装の手引き" (HOF cognitive Flash
 *    Attention in Rust), section 4 "Kernel": scores are Q.K^T times a scale,
 *    exponentiated, divided by the row sum to give row-stochastic weights A,
 *    and the result is A.V. Section 2 and section 4: the FlashAttention
 *    tiling computes the same exact result, so the oracle is the untiled
 *    definition.
 *  - tensai autograd guide, "Attention の組み立て" (assembling attention):
 *    layout (batch, head, seq, headDim); the scale is applied to Q.K^T before
 *    the additive mask; softmax over the last axis; the causal mask is 0 on
 *    and below the diagonal and -Inf above it.
 *  - ruDNN user guide, section 9 (paged attention and MLA): Hq must be a
 *    multiple of Hkv (GQA); inputs are F32/F16/BF16; scale finite and
 *    positive. Section 2: the attention op takes an optional mask and an
 *    optional additive attn_bias.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - the row maximum is subtracted before exp (softmax is shift invariant, so
 *    this is the same value as the page's raw exp, without overflow);
 *  - scale multiplies Q.K^T only; the fp32 bias is added after scaling;
 *  - a masked position is -inf whatever the bias;
 *  - causal alignment is bottom-right: key j is visible to row i when
 *    j <= i + (Sk - Sq);
 *  - key padding masks keys j >= clamp(kv_lens[b], 0, Sk); query rows are
 *    not masked;
 *  - GQA maps query head hq to key/value head hq / (Hq / Hkv);
 *  - the bias has shape [bias_b, bias_h, Sq, Sk] with bias_b in {1, B} and
 *    bias_h in {1, Hq}, broadcast over the size-1 axes;
 *  - a row with no visible key has undefined weights: the oracle returns NaN
 *    for its weights and its output (exp(-inf - (-inf)) in the plain form).
 *
 * Log-sum-exp of a row (ruDNN user guide, section 9: a split history keeps
 * FP32 partial statistics that are merged afterwards; the statistic that makes
 * two partial softmaxes mergeable is the log of the row's exp-sum):
 *
 *   lse = log(sum_j exp(s_j))  over the visible j,   -inf for an empty row.
 *
 * Inputs are float64 arrays holding the already dtype-rounded values,
 * widened exactly; accumulation is in float64 throughout.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_MASK_CAUSAL 1
#define ORACLE_MASK_KEY_PADDING 2

typedef struct {
  int64_t B, Hq, Hkv, Sq, Sk, D;
  int64_t bias_b, bias_h; /* ignored when bias == NULL */
} oracle_shape;

typedef struct {
  const oracle_shape* s;
  const double *q, *k, *v, *bias;
  const int32_t* kv_lens;
  int mask;
  double scale;
} problem;

/* One output row (b, hq, i): writes D outputs, Sk weights when w != NULL and
 * the row's log-sum-exp when lse != NULL. `sc` is caller scratch of Sk doubles. */
static void attention_row(const problem* P, int64_t b, int64_t hq, int64_t i,
                          double* o, double* w, double* lse, double* sc) {
  const oracle_shape* s = P->s;
  const int64_t D = s->D, Sk = s->Sk, Sq = s->Sq;
  const int64_t group = s->Hq / s->Hkv;
  const int64_t hk = hq / group;

  int64_t key_limit = Sk;
  if (P->mask & ORACLE_MASK_KEY_PADDING) {
    int64_t L = P->kv_lens[b];
    key_limit = L < 0 ? 0 : (L > Sk ? Sk : L);
  }
  const double* qi = P->q + ((b * s->Hq + hq) * Sq + i) * D;
  const double* kh = P->k + (b * s->Hkv + hk) * Sk * D;
  const double* vh = P->v + (b * s->Hkv + hk) * Sk * D;
  const double* brow = NULL;
  if (P->bias) {
    int64_t bb = (s->bias_b == 1) ? 0 : b;
    int64_t bh = (s->bias_h == 1) ? 0 : hq;
    brow = P->bias + ((bb * s->bias_h + bh) * Sq + i) * Sk;
  }

  /* scores, with the mask as -inf */
  double m = -INFINITY;
  for (int64_t j = 0; j < Sk; ++j) {
    int visible = j < key_limit;
    if ((P->mask & ORACLE_MASK_CAUSAL) && !(j <= i + (Sk - Sq))) visible = 0;
    double sj = -INFINITY;
    if (visible) {
      double dot = 0.0;
      for (int64_t d = 0; d < D; ++d) dot += qi[d] * kh[j * D + d];
      sj = P->scale * dot + (brow ? brow[j] : 0.0);
    }
    sc[j] = sj;
    if (sj > m) m = sj;
  }

  if (m == -INFINITY) { /* no visible key: undefined softmax -> NaN */
    for (int64_t d = 0; d < D; ++d) o[d] = NAN;
    if (w) for (int64_t j = 0; j < Sk; ++j) w[j] = NAN;
    if (lse) *lse = -INFINITY;
    return;
  }

  /* exp and row sum */
  double l = 0.0;
  for (int64_t j = 0; j < Sk; ++j) {
    double p = exp(sc[j] - m); /* exp(-inf) == 0 for masked keys */
    sc[j] = p;
    l += p;
  }
  if (lse) *lse = m + log(l);
  /* row-stochastic weights and the weighted sum of V */
  for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
  for (int64_t j = 0; j < Sk; ++j) {
    double wj = sc[j] / l;
    if (w) w[j] = wj;
    for (int64_t d = 0; d < D; ++d) o[d] += wj * vh[j * D + d];
  }
}

/* ---- threading: a shared counter hands out work items ---- */
typedef struct {
  const problem* P;
  int64_t n_items;
  const int64_t* rows; /* NULL: items are (b, hq) heads; else (b, hq, i) triples */
  double* out;
  double* weights;
  double* lse;
  int64_t next;
  pthread_mutex_t lock;
  int failed;
} job;

static int64_t take(job* J) {
  pthread_mutex_lock(&J->lock);
  int64_t t = J->next++;
  pthread_mutex_unlock(&J->lock);
  return t;
}

static void* worker(void* arg) {
  job* J = (job*)arg;
  const oracle_shape* s = J->P->s;
  double* sc = (double*)malloc(sizeof(double) * (size_t)(s->Sk > 0 ? s->Sk : 1));
  if (!sc) {
    pthread_mutex_lock(&J->lock);
    J->failed = 1;
    pthread_mutex_unlock(&J->lock);
    return NULL;
  }
  for (int64_t t = take(J); t < J->n_items; t = take(J)) {
    if (J->rows) {
      const int64_t* r = J->rows + 3 * t;
      attention_row(J->P, r[0], r[1], r[2], J->out + t * s->D, NULL, J->lse ? J->lse + t : NULL, sc);
    } else {
      int64_t b = t / s->Hq, hq = t % s->Hq;
      for (int64_t i = 0; i < s->Sq; ++i) {
        int64_t row = (b * s->Hq + hq) * s->Sq + i;
        attention_row(J->P, b, hq, i, J->out + row * s->D,
                      J->weights ? J->weights + row * s->Sk : NULL, J->lse ? J->lse + row : NULL, sc);
      }
    }
  }
  free(sc);
  return NULL;
}

static int run(job* J, int nthreads) {
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  if (nthreads > J->n_items) nthreads = J->n_items > 0 ? (int)J->n_items : 1;
  J->next = 0;
  J->failed = 0;
  pthread_mutex_init(&J->lock, NULL);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) return -2;
  int started = 0;
  for (int t = 0; t < nthreads; ++t)
    if (pthread_create(&th[t], NULL, worker, J) == 0) ++started;
  if (started == 0) worker(J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  pthread_mutex_destroy(&J->lock);
  return J->failed ? -2 : 0;
}

static int check_shape(const oracle_shape* s, int mask, const int32_t* kv_lens) {
  if (!s) return -1;
  if (s->B < 0 || s->Hq <= 0 || s->Hkv <= 0 || s->Sq < 0 || s->Sk < 0 || s->D <= 0) return -1;
  if (s->Hq % s->Hkv) return -1;
  if ((mask & ORACLE_MASK_KEY_PADDING) && !kv_lens) return -1;
  if (mask & ~(ORACLE_MASK_CAUSAL | ORACLE_MASK_KEY_PADDING)) return -1;
  return 0;
}

/* Full problem. out: [B,Hq,Sq,D]; weights (optional): [B,Hq,Sq,Sk]; lse
 * (optional): [B,Hq,Sq]. Returns 0, -1 on a bad argument, -2 when memory runs out. */
int oracle_attention(const oracle_shape* s, const double* q, const double* k, const double* v,
                     int mask, const int32_t* kv_lens, const double* bias, double scale,
                     double* out, double* weights, double* lse, int nthreads) {
  if (check_shape(s, mask, kv_lens)) return -1;
  if (bias && !((s->bias_b == 1 || s->bias_b == s->B) && (s->bias_h == 1 || s->bias_h == s->Hq)))
    return -1;
  problem P = {s, q, k, v, bias, kv_lens, mask, scale};
  job J;
  memset(&J, 0, sizeof J);
  J.P = &P;
  J.n_items = s->B * s->Hq;
  J.out = out;
  J.weights = weights;
  J.lse = lse;
  return run(&J, nthreads);
}

/* Selected rows only. rows: nrows triples (b, hq, i); out: [nrows, D]; lse
 * (optional): [nrows]. */
int oracle_attention_rows(const oracle_shape* s, const double* q, const double* k, const double* v,
                          int mask, const int32_t* kv_lens, const double* bias, double scale,
                          int64_t nrows, const int64_t* rows, double* out, double* lse,
                          int nthreads) {
  if (check_shape(s, mask, kv_lens)) return -1;
  if (bias && !((s->bias_b == 1 || s->bias_b == s->B) && (s->bias_h == 1 || s->bias_h == s->Hq)))
    return -1;
  for (int64_t t = 0; t < nrows; ++t) {
    const int64_t* r = rows + 3 * t;
    if (r[0] < 0 || r[0] >= s->B || r[1] < 0 || r[1] >= s->Hq || r[2] < 0 || r[2] >= s->Sq) return -1;
  }
  problem P = {s, q, k, v, bias, kv_lens, mask, scale};
  job J;
  memset(&J, 0, sizeof J);
  J.P = &P;
  J.n_items = nrows;
  J.rows = rows;
  J.out = out;
  J.lse = lse;
  return run(&J, nthreads);
}

/*
 * Backward (first-order gradients) of the same operation, in float64.
 *
 * Source: ruDNN user guide, section 11 (backward of paged attention): the
 * backward returns dq, dk and dv and recomputes the probabilities instead of
 * storing the score matrix. The oracle writes out the chain rule of the
 * forward definition above for a loss L with dL/dO = dout, row by row:
 *
 *   w_j   = softmax weights of the row (as in the forward)
 *   dv_j += w_j * dout_i                       (O_i = sum_j w_j v_j)
 *   dw_j  = dout_i . v_j
 *   ds_j  = w_j * (dw_j - sum_k w_k dw_k)      (Jacobian of the softmax)
 *   dq_i  = scale * sum_j ds_j k_j             (s_j = scale q_i.k_j + bias)
 *   dk_j += scale * ds_j q_i
 *
 * with GQA summing dk and dv over the query heads that share a key/value
 * head. The bias is a constant (the page's backward returns no bias
 * gradient). Reading where the pages are silent: a row with no visible key
 * (output NaN in the forward) contributes nothing; its dq row is 0.
 */
typedef struct {
  const problem* P;
  const double* dout;
  double *dq, *dk, *dv;
  int64_t next;
  pthread_mutex_t lock;
  int failed;
} bwd_job;

static int64_t bwd_take(bwd_job* J) {
  pthread_mutex_lock(&J->lock);
  int64_t t = J->next++;
  pthread_mutex_unlock(&J->lock);
  return t;
}

/* One (b, hk): every query row of the heads that share hk. */
static void backward_group(const problem* P, const double* dout, double* dq, double* dk,
                           double* dv, int64_t b, int64_t hk, double* w, double* sc, double* o,
                           double* dw) {
  const oracle_shape* s = P->s;
  const int64_t D = s->D, Sk = s->Sk, Sq = s->Sq;
  const int64_t group = s->Hq / s->Hkv;
  const double* kh = P->k + (b * s->Hkv + hk) * Sk * D;
  const double* vh = P->v + (b * s->Hkv + hk) * Sk * D;
  double* dkh = dk + (b * s->Hkv + hk) * Sk * D;
  double* dvh = dv + (b * s->Hkv + hk) * Sk * D;
  for (int64_t x = 0; x < Sk * D; ++x) dkh[x] = dvh[x] = 0.0;
  for (int64_t hq = hk * group; hq < (hk + 1) * group; ++hq) {
    for (int64_t i = 0; i < Sq; ++i) {
      const int64_t row = (b * s->Hq + hq) * Sq + i;
      const double* qi = P->q + row * D;
      const double* gi = dout + row * D;
      double* dqi = dq + row * D;
      for (int64_t d = 0; d < D; ++d) dqi[d] = 0.0;
      attention_row(P, b, hq, i, o, w, NULL, sc);
      if (Sk == 0 || isnan(w[0])) continue; /* no visible key: no contribution */
      double wdw = 0.0;
      for (int64_t j = 0; j < Sk; ++j) {
        double g = 0.0;
        for (int64_t d = 0; d < D; ++d) g += gi[d] * vh[j * D + d];
        dw[j] = g;
        wdw += w[j] * g;
      }
      for (int64_t j = 0; j < Sk; ++j) {
        if (w[j] == 0.0) continue; /* masked, or exp underflow: zero weight, zero terms */
        const double ds = w[j] * (dw[j] - wdw);
        for (int64_t d = 0; d < D; ++d) {
          dqi[d] += P->scale * ds * kh[j * D + d];
          dkh[j * D + d] += P->scale * ds * qi[d];
          dvh[j * D + d] += w[j] * gi[d];
        }
      }
    }
  }
}

static void* bwd_worker(void* arg) {
  bwd_job* J = (bwd_job*)arg;
  const oracle_shape* s = J->P->s;
  const size_t sk = (size_t)(s->Sk > 0 ? s->Sk : 1);
  double* w = (double*)malloc(sizeof(double) * sk);
  double* sc = (double*)malloc(sizeof(double) * sk);
  double* dw = (double*)malloc(sizeof(double) * sk);
  double* o = (double*)malloc(sizeof(double) * (size_t)s->D);
  if (!w || !sc || !dw || !o) {
    pthread_mutex_lock(&J->lock);
    J->failed = 1;
    pthread_mutex_unlock(&J->lock);
  } else {
    for (int64_t t = bwd_take(J); t < s->B * s->Hkv; t = bwd_take(J))
      backward_group(J->P, J->dout, J->dq, J->dk, J->dv, t / s->Hkv, t % s->Hkv, w, sc, o, dw);
  }
  free(w);
  free(sc);
  free(dw);
  free(o);
  return NULL;
}

/* dout: [B,Hq,Sq,D]; writes dq [B,Hq,Sq,D], dk and dv [B,Hkv,Sk,D].
 * Returns 0, -1 on a bad argument, -2 when memory runs out. */
int oracle_attention_bwd(const oracle_shape* s, const double* q, const double* k, const double* v,
                         int mask, const int32_t* kv_lens, const double* bias, double scale,
                         const double* dout, double* dq, double* dk, double* dv, int nthreads) {
  if (check_shape(s, mask, kv_lens) || !dout || !dq || !dk || !dv) return -1;
  if (bias && !((s->bias_b == 1 || s->bias_b == s->B) && (s->bias_h == 1 || s->bias_h == s->Hq)))
    return -1;
  problem P = {s, q, k, v, bias, kv_lens, mask, scale};
  bwd_job J;
  memset(&J, 0, sizeof J);
  J.P = &P;
  J.dout = dout;
  J.dq = dq;
  J.dk = dk;
  J.dv = dv;
  const int64_t items = s->B * s->Hkv;
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  if (nthreads > items) nthreads = items > 0 ? (int)items : 1;
  pthread_mutex_init(&J.lock, NULL);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  if (!th) {
    pthread_mutex_destroy(&J.lock);
    return -2;
  }
  int started = 0;
  for (int t = 0; t < nthreads; ++t)
    if (pthread_create(&th[t], NULL, bwd_worker, &J) == 0) ++started;
  if (started == 0) bwd_worker(&J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  pthread_mutex_destroy(&J.lock);
  return J.failed ? -2 : 0;
}

/*
 * Paged key/value cache, packed variable-length queries.
 *
 * Source: ruDNN user guide, section 9 (paged attention): keys and values live
 * in physical pages K [pages, page_size, Hkv, D] and V [pages, page_size, Hkv,
 * D]; each sequence has a page table, a key length and queries at zero-based
 * absolute positions; queries are packed as Q [queries, Hq, D] and the output
 * is [queries, Hq, D]; causal attention compares absolute positions.
 *
 * Readings: the queries of sequence s are rows q_off[s] .. q_off[s+1]-1 of Q
 * (packed in sequence order); key j of sequence s is row j % page_size of page
 * table[s * max_pages + j / page_size]; keys j < seq_len[s] exist; under the
 * causal mask the query at position pos sees keys j <= pos. When `positions`
 * is NULL, the n queries of a sequence of length L are its newest tokens, at
 * positions L - n .. L - 1. Everything else (max subtraction, GQA mapping, an
 * empty row giving NaN and lse = -inf) is as in the dense definition above.
 */
int oracle_paged_attention(int64_t num_seqs, int64_t Hq, int64_t Hkv, int64_t D, int64_t page_size,
                           int64_t max_pages, const double* q, const double* kc, const double* vc,
                           const int32_t* table, const int32_t* seq_len, const int32_t* q_off,
                           const int32_t* positions, int causal, double scale, double* out,
                           double* lse) {
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || page_size <= 0 || max_pages < 0)
    return -1;
  const int64_t group = Hq / Hkv;
  int64_t cap = 1;
  for (int64_t s = 0; s < num_seqs; ++s)
    if (seq_len[s] > cap) cap = seq_len[s];
  double* sc = (double*)malloc(sizeof(double) * (size_t)cap);
  if (!sc) return -2;
  for (int64_t s = 0; s < num_seqs; ++s) {
    const int64_t L = seq_len[s];
    const int64_t n = q_off[s + 1] - q_off[s];
    if (L < 0 || n < 0 || L > max_pages * page_size) {
      free(sc);
      return -1;
    }
    for (int64_t t = q_off[s]; t < q_off[s + 1]; ++t) {
      const int64_t pos = positions ? positions[t] : L - n + (t - q_off[s]);
      for (int64_t h = 0; h < Hq; ++h) {
        const int64_t hk = h / group;
        const double* qi = q + (t * Hq + h) * D;
        double* o = out + (t * Hq + h) * D;
        double m = -INFINITY;
        for (int64_t j = 0; j < L; ++j) {
          double sj = -INFINITY;
          if (!causal || j <= pos) {
            const int64_t page = table[s * max_pages + j / page_size];
            const double* kj = kc + ((page * page_size + j % page_size) * Hkv + hk) * D;
            double dot = 0.0;
            for (int64_t d = 0; d < D; ++d) dot += qi[d] * kj[d];
            sj = scale * dot;
          }
          sc[j] = sj;
          if (sj > m) m = sj;
        }
        if (m == -INFINITY) {
          for (int64_t d = 0; d < D; ++d) o[d] = NAN;
          if (lse) lse[t * Hq + h] = -INFINITY;
          continue;
        }
        double l = 0.0;
        for (int64_t j = 0; j < L; ++j) {
          sc[j] = exp(sc[j] - m);
          l += sc[j];
        }
        if (lse) lse[t * Hq + h] = m + log(l);
        for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
        for (int64_t j = 0; j < L; ++j) {
          if (sc[j] == 0.0) continue;
          const int64_t page = table[s * max_pages + j / page_size];
          const double* vj = vc + ((page * page_size + j % page_size) * Hkv + hk) * D;
          const double w = sc[j] / l;
          for (int64_t d = 0; d < D; ++d) o[d] += w * vj[d];
        }
      }
    }
  }
  free(sc);
  return 0;
}

/*
 * Multi-head latent attention (MLA) with absorbed projections over a paged
 * latent cache.
 *
 * Source: ruDNN user guide, section 9 (paged attention and MLA): the query is
 * given with the key projection absorbed, q [queries, H, R], plus a positional
 * query qp [queries, H, P]; the cache holds one shared latent row c_j
 * [pages, page_size, 1, R] and one positional key row kp_j [pages, page_size,
 * 1, P] per token; the output is the compressed context [queries, H, R]
 * (value and output projections are applied by the caller); the scale is the
 * original model's QK scale. So, for query t, head h and visible key j:
 *
 *   s_j = scale * (q_t,h . c_j + qp_t,h . kp_j),   out_t,h = sum_j softmax_j(s) c_j.
 *
 * Paging, packing, positions, the causal mask and empty rows are as in
 * oracle_paged_attention (every head reads the same single latent head).
 */
int oracle_paged_mla(int64_t num_seqs, int64_t H, int64_t R, int64_t Pd, int64_t page_size, int64_t max_pages,
                     const double* q, const double* qp, const double* lat, const double* kp, const int32_t* table,
                     const int32_t* seq_len, const int32_t* q_off, const int32_t* positions, int causal,
                     double scale, double* out, double* lse) {
  if (num_seqs < 0 || H <= 0 || R <= 0 || Pd < 0 || page_size <= 0 || max_pages < 0) return -1;
  int64_t cap = 1;
  for (int64_t s = 0; s < num_seqs; ++s)
    if (seq_len[s] > cap) cap = seq_len[s];
  double* sc = (double*)malloc(sizeof(double) * (size_t)cap);
  if (!sc) return -2;
  for (int64_t s = 0; s < num_seqs; ++s) {
    const int64_t L = seq_len[s];
    const int64_t n = q_off[s + 1] - q_off[s];
    if (L < 0 || n < 0 || L > max_pages * page_size) {
      free(sc);
      return -1;
    }
    for (int64_t t = q_off[s]; t < q_off[s + 1]; ++t) {
      const int64_t pos = positions ? positions[t] : L - n + (t - q_off[s]);
      for (int64_t h = 0; h < H; ++h) {
        const double* qi = q + (t * H + h) * R;
        const double* qpi = qp + (t * H + h) * Pd;
        double* o = out + (t * H + h) * R;
        double m = -INFINITY;
        for (int64_t j = 0; j < L; ++j) {
          double sj = -INFINITY;
          if (!causal || j <= pos) {
            const int64_t row = table[s * max_pages + j / page_size] * page_size + j % page_size;
            double dot = 0.0;
            for (int64_t d = 0; d < R; ++d) dot += qi[d] * lat[row * R + d];
            for (int64_t d = 0; d < Pd; ++d) dot += qpi[d] * kp[row * Pd + d];
            sj = scale * dot;
          }
          sc[j] = sj;
          if (sj > m) m = sj;
        }
        if (m == -INFINITY) {
          for (int64_t d = 0; d < R; ++d) o[d] = NAN;
          if (lse) lse[t * H + h] = -INFINITY;
          continue;
        }
        double l = 0.0;
        for (int64_t j = 0; j < L; ++j) {
          sc[j] = exp(sc[j] - m);
          l += sc[j];
        }
        if (lse) lse[t * H + h] = m + log(l);
        for (int64_t d = 0; d < R; ++d) o[d] = 0.0;
        for (int64_t j = 0; j < L; ++j) {
          if (sc[j] == 0.0) continue;
          const int64_t row = table[s * max_pages + j / page_size] * page_size + j % page_size;
          const double w = sc[j] / l;
          for (int64_t d = 0; d < R; ++d) o[d] += w * lat[row * R + d];
        }
      }
    }
  }
  free(sc);
  return 0;
}

/*
 * Backward of the paged-cache attention and of paged MLA, in float64.
 *
 * Source: ruDNN user guide, section 11 (backward of paged attention and
 * ordered history gradients): the paged backward returns dq for the packed
 * queries and dk, dv in the shape of the physical caches (the "history"
 * gradients); the MLA backward returns dq, dqp and the cache-shaped dlatent,
 * dkp, where dlatent holds both the key and the value contribution of each
 * latent row. Per query row the chain rule is that of oracle_attention_bwd
 * above (w = softmax weights, dw_j = dout . v_j, ds_j = w_j (dw_j - sum_k w_k
 * dw_k)), with key j of sequence s at row j % page_size of page
 * table[s][j / page_size], and for MLA s_j = scale (q . c_j + qp . kp_j),
 * v_j = c_j.
 *
 * Readings where the pages are silent: a physical page read by several
 * sequences (a shared prefix), or by one sequence at several logical blocks,
 * receives the sum of the contributions of every read; a page that no query
 * reads gets zero gradients; a query row with no visible key contributes
 * nothing and gets dq = 0; query rows outside every sequence's range get 0.
 */
static int paged_check(int64_t num_seqs, int64_t page_size, int64_t max_pages, int64_t num_pages,
                       int64_t num_queries, const int32_t* table, const int32_t* seq_len,
                       const int32_t* q_off, int64_t* cap) {
  *cap = 1;
  for (int64_t s = 0; s < num_seqs; ++s) {
    const int64_t L = seq_len[s];
    if (L < 0 || L > max_pages * page_size) return -1;
    if (q_off[s] < 0 || q_off[s + 1] < q_off[s] || q_off[s + 1] > num_queries) return -1;
    for (int64_t b = 0; b < (L + page_size - 1) / page_size; ++b) {
      const int32_t pg = table[s * max_pages + b];
      if (pg < 0 || pg >= num_pages) return -1;
    }
    if (L > *cap) *cap = L;
  }
  return 0;
}

int oracle_paged_attention_bwd(int64_t num_seqs, int64_t Hq, int64_t Hkv, int64_t D, int64_t page_size,
                               int64_t max_pages, int64_t num_pages, int64_t num_queries, const double* q,
                               const double* kc, const double* vc, const int32_t* table,
                               const int32_t* seq_len, const int32_t* q_off, const int32_t* positions,
                               int causal, double scale, const double* dout, double* dq, double* dk,
                               double* dv) {
  if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || D <= 0 || page_size <= 0 || max_pages < 0 ||
      num_pages < 0 || num_queries < 0)
    return -1;
  int64_t cap;
  if (paged_check(num_seqs, page_size, max_pages, num_pages, num_queries, table, seq_len, q_off, &cap))
    return -1;
  const int64_t group = Hq / Hkv;
  for (int64_t x = 0; x < num_queries * Hq * D; ++x) dq[x] = 0.0;
  for (int64_t x = 0; x < num_pages * page_size * Hkv * D; ++x) dk[x] = dv[x] = 0.0;
  double* w = (double*)malloc(sizeof(double) * (size_t)cap);
  double* dw = (double*)malloc(sizeof(double) * (size_t)cap);
  if (!w || !dw) {
    free(w);
    free(dw);
    return -2;
  }
  for (int64_t s = 0; s < num_seqs; ++s) {
    const int64_t L = seq_len[s];
    const int64_t n = q_off[s + 1] - q_off[s];
    for (int64_t t = q_off[s]; t < q_off[s + 1]; ++t) {
      const int64_t p_t = positions ? positions[t] : L - n + (t - q_off[s]);
      for (int64_t h = 0; h < Hq; ++h) {
        const int64_t hk = h / group;
        const double* qi = q + (t * Hq + h) * D;
        const double* gi = dout + (t * Hq + h) * D;
        double* dqi = dq + (t * Hq + h) * D;
        /* the forward's weights of this row */
        double m = -INFINITY;
        for (int64_t j = 0; j < L; ++j) {
          w[j] = -INFINITY;
          if (!causal || j <= p_t) {
            const int64_t row = (table[s * max_pages + j / page_size] * page_size + j % page_size) * Hkv + hk;
            double acc = 0.0;
            for (int64_t d = 0; d < D; ++d) acc += qi[d] * kc[row * D + d];
            w[j] = scale * acc;
          }
          if (w[j] > m) m = w[j];
        }
        if (m == -INFINITY) continue; /* no visible key: no contribution */
        double l = 0.0;
        for (int64_t j = 0; j < L; ++j) {
          w[j] = exp(w[j] - m);
          l += w[j];
        }
        double wdw = 0.0;
        for (int64_t j = 0; j < L; ++j) {
          w[j] /= l;
          dw[j] = 0.0;
          if (w[j] == 0.0) continue;
          const int64_t row = (table[s * max_pages + j / page_size] * page_size + j % page_size) * Hkv + hk;
          for (int64_t d = 0; d < D; ++d) dw[j] += gi[d] * vc[row * D + d];
          wdw += w[j] * dw[j];
        }
        for (int64_t j = 0; j < L; ++j) {
          if (w[j] == 0.0) continue; /* masked, or exp underflow: zero weight, zero terms */
          const int64_t row = (table[s * max_pages + j / page_size] * page_size + j % page_size) * Hkv + hk;
          const double dsj = w[j] * (dw[j] - wdw);
          for (int64_t d = 0; d < D; ++d) {
            dqi[d] += scale * dsj * kc[row * D + d];
            dk[row * D + d] += scale * dsj * qi[d];
            dv[row * D + d] += w[j] * gi[d];
          }
        }
      }
    }
  }
  free(w);
  free(dw);
  return 0;
}

int oracle_paged_mla_bwd(int64_t num_seqs, int64_t H, int64_t R, int64_t Pd, int64_t page_size,
                         int64_t max_pages, int64_t num_pages, int64_t num_queries, const double* q,
                         const double* qp, const double* lat, const double* kp, const int32_t* table,
                         const int32_t* seq_len, const int32_t* q_off, const int32_t* positions, int causal,
                         double scale, const double* dout, double* dq, double* dqp, double* dlat,
                         double* dkp) {
  if (num_seqs < 0 || H <= 0 || R <= 0 || Pd < 0 || page_size <= 0 || max_pages < 0 || num_pages < 0 ||
      num_queries < 0)
    return -1;
  int64_t cap;
  if (paged_check(num_seqs, page_size, max_pages, num_pages, num_queries, table, seq_len, q_off, &cap))
    return -1;
  for (int64_t x = 0; x < num_queries * H * R; ++x) dq[x] = 0.0;
  for (int64_t x = 0; x < num_queries * H * Pd; ++x) dqp[x] = 0.0;
  for (int64_t x = 0; x < num_pages * page_size * R; ++x) dlat[x] = 0.0;
  for (int64_t x = 0; x < num_pages * page_size * Pd; ++x) dkp[x] = 0.0;
  double* w = (double*)malloc(sizeof(double) * (size_t)cap);
  double* dw = (double*)malloc(sizeof(double) * (size_t)cap);
  if (!w || !dw) {
    free(w);
    free(dw);
    return -2;
  }
  for (int64_t s = 0; s < num_seqs; ++s) {
    const int64_t L = seq_len[s];
    const int64_t n = q_off[s + 1] - q_off[s];
    for (int64_t t = q_off[s]; t < q_off[s + 1]; ++t) {
      const int64_t p_t = positions ? positions[t] : L - n + (t - q_off[s]);
      for (int64_t h = 0; h < H; ++h) {
        const double* qi = q + (t * H + h) * R;
        const double* qpt = qp + (t * H + h) * Pd;
        const double* gi = dout + (t * H + h) * R;
        double* dqi = dq + (t * H + h) * R;
        double* dqpi = dqp + (t * H + h) * Pd;
        double m = -INFINITY;
        for (int64_t j = 0; j < L; ++j) {
          w[j] = -INFINITY;
          if (!causal || j <= p_t) {
            const int64_t row = table[s * max_pages + j / page_size] * page_size + j % page_size;
            double acc = 0.0;
            for (int64_t d = 0; d < R; ++d) acc += qi[d] * lat[row * R + d];
            for (int64_t d = 0; d < Pd; ++d) acc += qpt[d] * kp[row * Pd + d];
            w[j] = scale * acc;
          }
          if (w[j] > m) m = w[j];
        }
        if (m == -INFINITY) continue;
        double l = 0.0;
        for (int64_t j = 0; j < L; ++j) {
          w[j] = exp(w[j] - m);
          l += w[j];
        }
        double wdw = 0.0;
        for (int64_t j = 0; j < L; ++j) {
          w[j] /= l;
          dw[j] = 0.0;
          if (w[j] == 0.0) continue;
          const int64_t row = table[s * max_pages + j / page_size] * page_size + j % page_size;
          for (int64_t d = 0; d < R; ++d) dw[j] += gi[d] * lat[row * R + d];
          wdw += w[j] * dw[j];
        }
        for (int64_t j = 0; j < L; ++j) {
          if (w[j] == 0.0) continue;
          const int64_t row = table[s * max_pages + j / page_size] * page_size + j % page_size;
          const double dsj = w[j] * (dw[j] - wdw);
          for (int64_t d = 0; d < R; ++d) {
            dqi[d] += scale * dsj * lat[row * R + d];
            dlat[row * R + d] += scale * dsj * qi[d] + w[j] * gi[d]; /* key and value parts */
          }
          for (int64_t d = 0; d < Pd; ++d) {
            dqpi[d] += scale * dsj * kp[row * Pd + d];
            dkp[row * Pd + d] += scale * dsj * qpt[d];
          }
        }
      }
    }
  }
  free(w);
  free(dw);
  return 0;
}
