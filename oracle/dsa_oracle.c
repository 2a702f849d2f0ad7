/*
 * dsa_oracle.c -- plain, slow, fp64 CPU oracle of the DeepSeek Sparse Attention
 * hot path.  TEST INFRASTRUCTURE ONLY: it is loaded by the tests, by the smoke
 * check and by the CPU-baseline leg of the benchmark, never by the product path.
 * It shares no code, header or constant with the CUDA library.
 *
 * Pages followed (cited by title and section):
 *  [DSA-blog]  "Accelerating GLM-5.2 Long-Context Training with cuDNN Fused DSA
 *              Kernels ..." (Megatron-Bridge discussion 4957), section "How DSA works".
 *  [NoPE-PR]   SkyRL PR 2388 "NoPE / unaligned top-k for SparseMLA", sections
 *              "Why" and "Change".
 *  [cudnn_dsa] NeMo AutoModel API page glm_moe_dsa.kernels.cudnn_dsa: entries
 *              cudnn_indexer_topk, cudnn_sparse_attention,
 *              prepare_cudnn_dsa_packed_metadata, _compact_and_sort_indices.
 *  [Chunk-PR]  SkyRL PR 2423 "query-chunked sparse attention", section "Summary".
 *
 * Every floating-point input arrives already widened to double by the caller,
 * so the oracle computes in fp64 throughout.  Where the pages leave a step
 * open, the reading taken is written next to the step.
 */
#include <math.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* THD packing metadata                                                      */
/* [cudnn_dsa] prepare_cudnn_dsa_packed_metadata: per query, the start of its */
/* packed sequence and its real causal length.  Reading: with no context      */
/* parallelism the query coordinates are the identity, so for token t in     */
/* sequence i, start = cu[i] and causal length = t - cu[i] + 1 (the diagonal  */
/* is included, "s <= t").                                                    */
/* Returns 0 on success, -1 if cu_seqlens is not a non-decreasing cover of    */
/* [0, T].                                                                    */
/* ------------------------------------------------------------------------ */
int oracle_packed_metadata(const int32_t *cu_seqlens, int num_seqs, int T,
                           int32_t *seq_start, int32_t *causal_len,
                           int32_t *max_seqlen, int32_t *all_rows_nonempty) {
  if (num_seqs < 1 || cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != T) return -1;
  int mx = 0;
  for (int i = 0; i < num_seqs; ++i) {
    int a = cu_seqlens[i], b = cu_seqlens[i + 1];
    if (b < a) return -1;
    if (b - a > mx) mx = b - a;
    for (int t = a; t < b; ++t) {
      seq_start[t] = a;
      causal_len[t] = t - a + 1;
    }
  }
  *max_seqlen = mx;
  /* every real token sees at least itself, so every row is nonempty */
  *all_rows_nonempty = (T > 0) ? 1 : 0;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* THD packing metadata with context parallelism                              */
/* [cudnn_dsa] prepare_cudnn_dsa_packed_metadata: metadata for rank-local     */
/* queries and gathered global keys.  query_indices holds the global padded-  */
/* storage coordinate of each local query row (absent: the identity, i.e. the */
/* queries cover every global key token); cu_seqlens_padded holds the padded  */
/* storage boundaries (absent: cu_seqlens is also the storage); padding_mask  */
/* marks local padding rows and stays authoritative; the result holds, per    */
/* query, the global padded-storage start and the real causal length.         */
/* Readings: with P the storage boundaries and L_i = cu[i+1] - cu[i], a row   */
/* with coordinate g lies in sequence i when P[i] <= g < P[i+1]; its position */
/* is p = g - P[i]; start = P[i] and causal length = p + 1 when p < L_i and   */
/* the row is not masked, else 0 (a padding row).  A row outside every        */
/* sequence's storage gets start = g and length 0.  A nonzero mask byte marks */
/* padding.  max_seqlen = max_i L_i; all_rows_nonempty = every length > 0.    */
/* Returns 0, or -1 when cu_seqlens / cu_seqlens_padded are not non-decreasing*/
/* from 0, a sequence's real length exceeds its storage, the storage exceeds  */
/* total_key_tokens, or a coordinate lies outside [0, total_key_tokens).      */
/* ------------------------------------------------------------------------ */
int oracle_packed_metadata_cp(const int32_t *cu_seqlens, const int32_t *cu_padded, int num_seqs,
                              int total_key_tokens, const int32_t *query_idx, const uint8_t *pad_mask,
                              int Tq, int32_t *seq_start, int32_t *causal_len, int32_t *max_seqlen,
                              int32_t *all_rows_nonempty) {
  const int32_t *P = cu_padded ? cu_padded : cu_seqlens;
  if (num_seqs < 1 || cu_seqlens[0] != 0 || P[0] != 0 || P[num_seqs] > total_key_tokens) return -1;
  int mx = 0;
  for (int i = 0; i < num_seqs; ++i) {
    int L = cu_seqlens[i + 1] - cu_seqlens[i];
    if (L < 0 || P[i + 1] < P[i] || L > P[i + 1] - P[i]) return -1;
    if (L > mx) mx = L;
  }
  int nonempty = 1;
  for (int r = 0; r < Tq; ++r) {
    int g = query_idx ? query_idx[r] : r;
    if (g < 0 || g >= total_key_tokens) return -1;
    int start = g, len = 0;
    for (int i = 0; i < num_seqs; ++i) {
      if (P[i] <= g && g < P[i + 1]) {
        int pos = g - P[i];
        start = P[i];
        if (pos < cu_seqlens[i + 1] - cu_seqlens[i] && !(pad_mask && pad_mask[r])) len = pos + 1;
        break;
      }
    }
    seq_start[r] = start;
    causal_len[r] = len;
    if (len == 0) nonempty = 0;
  }
  *max_seqlen = mx;
  *all_rows_nonempty = (Tq > 0) ? nonempty : 0;
  return 0;
}

/* ------------------------------------------------------------------------ */
/* Lightning-indexer score                                                   */
/* [cudnn_dsa] cudnn_indexer_topk: index_q [T, H_index, 128], one shared      */
/* index_k [T_k, 128], already-scaled head weights [T, H_index] ("the caller  */
/* owns both scalings").  The pages do not print the formula; the reading is  */
/*   score(t, s) = sum_h w[t,h] * max(0, sum_d q[t,h,d] * k[s,d]).            */
/* ------------------------------------------------------------------------ */
static double indexer_score(const double *q_t /*[Hi,Di]*/, const double *k_s /*[Di]*/,
                            const double *w_t /*[Hi]*/, int Hi, int Di, double *mag) {
  double score = 0.0, m = 0.0;
  for (int h = 0; h < Hi; ++h) {
    double dot = 0.0, adot = 0.0;
    for (int d = 0; d < Di; ++d) {
      dot += q_t[(size_t)h * Di + d] * k_s[d];
      adot += fabs(q_t[(size_t)h * Di + d] * k_s[d]);
    }
    double relu = dot > 0.0 ? dot : 0.0;
    score += w_t[h] * relu;
    m += fabs(w_t[h]) * adot;
  }
  if (mag) *mag = m;
  return score;
}

/* Scores for explicit (row, key) pairs.  q_rows holds the query rows named by
 * pair_row (indices into q_rows), k holds all keys.  mag_out (nullable) gets
 * sum_h |w| sum_d |q k|, the scale of the rounding error of any fp32
 * evaluation of the same score. */
void oracle_indexer_scores(const double *q_rows, const double *k, const double *w_rows,
                           int Hi, int Di, const int64_t *pair_row, const int64_t *pair_key,
                           int64_t npairs, double *out, double *mag_out) {
#pragma omp parallel for schedule(static)
  for (int64_t p = 0; p < npairs; ++p) {
    const double *q_t = q_rows + (size_t)pair_row[p] * Hi * Di;
    const double *w_t = w_rows + (size_t)pair_row[p] * Hi;
    double mag;
    out[p] = indexer_score(q_t, k + (size_t)pair_key[p] * Di, w_t, Hi, Di, &mag);
    if (mag_out) mag_out[p] = mag;
  }
}

/* ------------------------------------------------------------------------ */
/* Per-query causal top-k                                                    */
/* [DSA-blog] "How DSA works": the indexer emits the top-k key indices per    */
/* query.  [cudnn_dsa] cudnn_indexer_topk returns int32 global indices; the   */
/* canonical form (cudnn_sparse_attention, topk_length) is a compact,         */
/* ascending valid prefix followed by -1.                                     */
/* Readings: candidates are the causal keys s in [start(t), t]; n = min(K, c);*/
/* order by score descending, ties to the lower index; the n winners are     */
/* written ascending, then K - n copies of -1; len[t] = n.                    */
/* ------------------------------------------------------------------------ */
typedef struct { double score; int32_t idx; } cand_t;

static int cand_cmp(const void *a, const void *b) {
  const cand_t *x = (const cand_t *)a, *y = (const cand_t *)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}
static int int_cmp(const void *a, const void *b) {
  int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
  return (x > y) - (x < y);
}

/* Top-k of one query row over the window [b, b + c - 1] of keys. */
static void topk_window(const double *q_row, const double *k, const double *w_row, int64_t b, int64_t c,
                        int Hi, int Di, int K, int32_t *row, int32_t *len_out, double *kth_out) {
  cand_t *cand = (cand_t *)malloc(sizeof(cand_t) * (size_t)(c > 0 ? c : 1));
  for (int64_t s = b; s < b + c; ++s) {
    cand[s - b].score = indexer_score(q_row, k + (size_t)s * Di, w_row, Hi, Di, NULL);
    cand[s - b].idx = (int32_t)s;
  }
  qsort(cand, (size_t)(c > 0 ? c : 0), sizeof(cand_t), cand_cmp); /* full sort: plain definition */
  int n = (int)(c < K ? c : K);
  if (n < 0) n = 0;
  for (int j = 0; j < n; ++j) row[j] = cand[j].idx;
  qsort(row, (size_t)n, sizeof(int32_t), int_cmp);
  for (int j = n; j < K; ++j) row[j] = -1;
  *len_out = n;
  if (kth_out) *kth_out = n > 0 ? cand[n - 1].score : -INFINITY;
  free(cand);
}

/* q_rows/w_rows hold only the nrows requested rows; row_t[r] is the global
 * token of row r (its causal window is [seq_start[row_t[r]], row_t[r]]).
 * kth_out[r] (nullable) receives the score of the n-th winner (-inf if n = 0). */
void oracle_indexer_topk(const double *q_rows, const double *k, const double *w_rows,
                         const int32_t *seq_start, const int64_t *row_t, int nrows,
                         int Hi, int Di, int K, int32_t *idx_out, int32_t *len_out,
                         double *kth_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    int64_t t = row_t[r];
    int64_t b = seq_start[t];
    topk_window(q_rows + (size_t)r * Hi * Di, k, w_rows + (size_t)r * Hi, b, t - b + 1, Hi, Di, K,
                idx_out + (size_t)r * K, len_out + r, kth_out ? kth_out + r : NULL);
  }
}

/* The same over explicit windows, the form the context-parallel metadata
 * gives: row r's candidates are the keys [win_start[r], win_start[r] +
 * win_len[r] - 1], none when win_len[r] = 0. */
void oracle_indexer_topk_window(const double *q_rows, const double *k, const double *w_rows,
                                const int32_t *win_start, const int32_t *win_len, int nrows, int Hi, int Di,
                                int K, int32_t *idx_out, int32_t *len_out, double *kth_out) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r)
    topk_window(q_rows + (size_t)r * Hi * Di, k, w_rows + (size_t)r * Hi, win_start[r], win_len[r], Hi, Di, K,
                idx_out + (size_t)r * K, len_out + r, kth_out ? kth_out + r : NULL);
}

/* ------------------------------------------------------------------------ */
/* Slot validity                                                              */
/* [cudnn_dsa] cudnn_sparse_attention: -1 marks an invalid slot; topk_length  */
/* (optional) bounds the valid prefix.  [NoPE-PR] "Change": the kernels mask  */
/* -1 wherever it is.  Reading: a slot j is valid iff j < len (when given)    */
/* and 0 <= idx < T_k.  Duplicate valid indices count once per slot.          */
/* ------------------------------------------------------------------------ */
static int slot_valid(const int32_t *idx_row, const int32_t *len, int64_t r, int j, int Tk) {
  if (len && j >= len[r]) return 0;
  int32_t i = idx_row[j];
  return i >= 0 && i < Tk;
}

/* ------------------------------------------------------------------------ */
/* Absorbed sparse MLA forward                                                */
/* [DSA-blog] "How DSA works" / "Why DSA needs fused kernels": every head of  */
/* a query attends, as an MQA over one shared latent KV, only to that query's */
/* selected rows.  [cudnn_dsa] cudnn_sparse_attention: q [T, H, 576],         */
/* kv_latent [T_k, 1, 576], value = kv[..., :512], explicit softmax_scale,    */
/* output [T, H, 512].  [NoPE-PR] "Change": value is key[..., :512].          */
/* Per (t, h), over the valid slot set J:                                     */
/*   z_j = scale * <q[t,h,:Dqk], kv[idx_j,:Dqk]>                              */
/*   L   = log sum_j exp(z_j)      (natural log; -inf when J is empty)        */
/*   O   = sum_j exp(z_j - L) kv[idx_j, :Dv]   (0 when J is empty)            */
/* Attention sink ([cudnn_dsa] _pad_attention_heads pads a sink [H] together  */
/* with q; the pages print no formula).  Reading: sink[h] is one more logit   */
/* of every row of head h, in the units of z, with no value row:              */
/*   L = log(sum_j exp(z_j) + exp(sink[h])),  O = sum_j exp(z_j - L) kv_j     */
/* so an empty row gets L = sink[h] and O = 0.  sink == NULL: no sink.        */
/* ------------------------------------------------------------------------ */
static void fwd_row(const double *q_r /*[H,Dqk]*/, const double *kv, const int32_t *idx_row,
                    const int32_t *len, int64_t r, int Tk, int H, int Dqk, int Dv, int K,
                    double scale, const double *sink /*[H] or NULL*/, double *o_r /*[H,Dv]*/,
                    double *lse_r /*[H]*/, double *p_r /*[H,K] nullable: softmax weights per slot*/) {
  double *z = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
  for (int h = 0; h < H; ++h) {
    const double *qh = q_r + (size_t)h * Dqk;
    double m = -INFINITY;
    for (int j = 0; j < K; ++j) {
      if (!slot_valid(idx_row, len, r, j, Tk)) { z[j] = -INFINITY; continue; }
      const double *kr = kv + (size_t)idx_row[j] * Dqk;
      double dot = 0.0;
      for (int d = 0; d < Dqk; ++d) dot += qh[d] * kr[d];
      z[j] = scale * dot;
      if (z[j] > m) m = z[j];
    }
    if (sink && sink[h] > m) m = sink[h];
    double *oh = o_r + (size_t)h * Dv;
    for (int v = 0; v < Dv; ++v) oh[v] = 0.0;
    if (m == -INFINITY) {
      lse_r[h] = -INFINITY;
      if (p_r) for (int j = 0; j < K; ++j) p_r[(size_t)h * K + j] = 0.0;
      continue;
    }
    double sum = 0.0;
    for (int j = 0; j < K; ++j) if (z[j] != -INFINITY) sum += exp(z[j] - m);
    if (sink) sum += exp(sink[h] - m);
    double L = m + log(sum);
    lse_r[h] = L;
    for (int j = 0; j < K; ++j) {
      double p = (z[j] == -INFINITY) ? 0.0 : exp(z[j] - L);
      if (p_r) p_r[(size_t)h * K + j] = p;
      if (p == 0.0) continue;
      const double *vr = kv + (size_t)idx_row[j] * Dqk;
      for (int v = 0; v < Dv; ++v) oh[v] += p * vr[v];
    }
  }
  free(z);
}

/* q_rows [nrows, H, Dqk], idx_rows [nrows, K], len_rows [nrows] or NULL,
 * kv [Tk, Dqk].  Outputs out [nrows, H, Dv], lse [nrows, H]. */
void oracle_sparse_mla_fwd(const double *q_rows, const double *kv, const int32_t *idx_rows,
                           const int32_t *len_rows, int nrows, int Tk, int H, int Dqk, int Dv,
                           int K, double scale, const double *sink, double *out, double *lse) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r)
    fwd_row(q_rows + (size_t)r * H * Dqk, kv, idx_rows + (size_t)r * K, len_rows, r, Tk, H,
            Dqk, Dv, K, scale, sink, out + (size_t)r * H * Dv, lse + (size_t)r * H, NULL);
}

/* ------------------------------------------------------------------------ */
/* Absorbed sparse MLA backward (analytic gradient of the forward above)      */
/* [cudnn_dsa] _CudnnSparseAttention.backward: gradients for the query        */
/* [T, H, 576] and the latent KV, from grad_output [T, H, 512].               */
/* With P_j = exp(z_j - L), D = <dO, O>, dP_j = <dO, kv[idx_j,:Dv]>,           */
/* dS_j = P_j (dP_j - D):                                                     */
/*   dq[t,h,:]        = scale * sum_j dS_j kv[idx_j, :Dqk]                    */
/*   dkv[idx_j, :Dqk] += scale * sum_h dS_j q[t,h,:]                          */
/*   dkv[idx_j, :Dv]  += sum_h P_j dO[t,h,:]                                  */
/* O here is the oracle's own fp64 forward output.  [Chunk-PR] "Summary":     */
/* query rows are independent and key gradients sum, so dkv accumulates over  */
/* whatever rows are passed in.  The dkv sum runs over channels in parallel   */
/* with a fixed (row, slot, head) order, so it is deterministic.             */
/* With a sink, P and O are those of the forward above; O is sum_j P_j kv_j  */
/* with P_sink = exp(sink[h] - L) left out, so dO/dsink = -P_sink O and      */
/*   d_sink[h] += -sum_t P_sink[t,h] D[t,h]                                   */
/* (d_sink nullable; added to, like dkv).                                     */
/* dq_mag (nullable) receives scale * sum_j |dS_j| |kv[idx_j, d]| per         */
/* (row, head, channel): the scale of the error that rounding each dS_j to a  */
/* 16-bit float before the dq sum can cause.                                  */
/* ------------------------------------------------------------------------ */
void oracle_sparse_mla_bwd(const double *q_rows, const double *kv, const int32_t *idx_rows,
                           const int32_t *len_rows, int nrows, int Tk, int H, int Dqk, int Dv,
                           int K, double scale, const double *sink /*[H] or NULL*/,
                           const double *dout_rows /*[nrows,H,Dv]*/,
                           double *dq /*[nrows,H,Dqk]*/, double *dkv /*[Tk,Dqk], added to*/,
                           double *d_sink /*[H] or NULL, added to*/,
                           double *dq_mag /*[nrows,H,Dqk] or NULL*/) {
  size_t pk = (size_t)nrows * H * K;
  double *P = (double *)calloc(pk ? pk : 1, sizeof(double));
  double *dS = (double *)calloc(pk ? pk : 1, sizeof(double));
  /* per-row sink gradient terms, summed in row order after the parallel loop */
  double *gs = (sink && d_sink) ? (double *)calloc((size_t)nrows * H + 1, sizeof(double)) : NULL;
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    const double *q_r = q_rows + (size_t)r * H * Dqk;
    const int32_t *idx_row = idx_rows + (size_t)r * K;
    double *o_r = (double *)malloc(sizeof(double) * (size_t)H * Dv);
    double *lse_r = (double *)malloc(sizeof(double) * (size_t)H);
    double *p_r = P + (size_t)r * H * K;
    double *ds_r = dS + (size_t)r * H * K;
    fwd_row(q_r, kv, idx_row, len_rows, r, Tk, H, Dqk, Dv, K, scale, sink, o_r, lse_r, p_r);
    for (int h = 0; h < H; ++h) {
      const double *dO = dout_rows + ((size_t)r * H + h) * Dv;
      double D = 0.0;
      for (int v = 0; v < Dv; ++v) D += dO[v] * o_r[(size_t)h * Dv + v];
      if (gs && lse_r[h] != -INFINITY) gs[(size_t)r * H + h] = -exp(sink[h] - lse_r[h]) * D;
      double *dqh = dq + ((size_t)r * H + h) * Dqk;
      double *mgh = dq_mag ? dq_mag + ((size_t)r * H + h) * Dqk : NULL;
      for (int d = 0; d < Dqk; ++d) dqh[d] = 0.0;
      if (mgh) for (int d = 0; d < Dqk; ++d) mgh[d] = 0.0;
      for (int j = 0; j < K; ++j) {
        double p = p_r[(size_t)h * K + j];
        if (p == 0.0) { ds_r[(size_t)h * K + j] = 0.0; continue; }
        const double *kr = kv + (size_t)idx_row[j] * Dqk;
        double dp = 0.0;
        for (int v = 0; v < Dv; ++v) dp += dO[v] * kr[v];
        double ds = p * (dp - D);
        ds_r[(size_t)h * K + j] = ds;
        for (int d = 0; d < Dqk; ++d) dqh[d] += scale * ds * kr[d];
        if (mgh) for (int d = 0; d < Dqk; ++d) mgh[d] += scale * fabs(ds) * fabs(kr[d]);
      }
    }
    free(o_r);
    free(lse_r);
  }
  if (gs) {
    for (int r = 0; r < nrows; ++r)
      for (int h = 0; h < H; ++h) d_sink[h] += gs[(size_t)r * H + h];
    free(gs);
  }
  /* key gradient: each thread owns a contiguous range of channels and walks the
   * (row, slot, head) triples in a fixed order, so every element sees the same
   * summation order whatever the thread count: per (row, slot) the head terms
   * are summed first (dS term, then P term, head by head), then added to dkv. */
#pragma omp parallel
  {
    int nth = 1, id = 0;
#ifdef _OPENMP
    nth = omp_get_num_threads();
    id = omp_get_thread_num();
#endif
    const int d0 = (int)((int64_t)Dqk * id / nth), d1 = (int)((int64_t)Dqk * (id + 1) / nth);
    double *acc = (double *)malloc(sizeof(double) * (size_t)(d1 > d0 ? d1 - d0 : 1));
    for (int r = 0; r < nrows; ++r) {
      const int32_t *idx_row = idx_rows + (size_t)r * K;
      for (int j = 0; j < K; ++j) {
        if (!slot_valid(idx_row, len_rows, r, j, Tk)) continue;
        for (int d = d0; d < d1; ++d) acc[d - d0] = 0.0;
        for (int h = 0; h < H; ++h) {
          size_t pj = ((size_t)r * H + h) * K + j;
          const double *qh = q_rows + ((size_t)r * H + h) * Dqk;
          const double *doh = dout_rows + ((size_t)r * H + h) * Dv;
          for (int d = d0; d < d1; ++d) {
            acc[d - d0] += scale * dS[pj] * qh[d];
            if (d < Dv) acc[d - d0] += P[pj] * doh[d];
          }
        }
        double *dst = dkv + (size_t)idx_row[j] * Dqk;
        for (int d = d0; d < d1; ++d) dst[d] += acc[d - d0];
      }
    }
    free(acc);
  }
  free(P);
  free(dS);
}

/* ------------------------------------------------------------------------ */
/* Head-averaged attention probability per selected slot                      */
/* [DSA-blog] "How DSA works": the indexer's KL loss aligns its score         */
/* distribution with the main attention's, and "Why DSA needs fused kernels": */
/* the attention-score tensor the KL loss consumes.  Reading: for row t and   */
/* slot j, prob[t,j] = (1/H) sum_h P[t,h,j] with P the sparse-MLA softmax      */
/* weights of the forward above (0 for an invalid slot).                      */
/* ------------------------------------------------------------------------ */
void oracle_attn_slot_prob(const double *q_rows, const double *kv, const int32_t *idx_rows,
                           const int32_t *len_rows, int nrows, int Tk, int H, int Dqk, int Dv, int K,
                           double scale, const double *sink, double *prob /*[nrows,K]*/) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    double *o_r = (double *)malloc(sizeof(double) * (size_t)H * Dv);
    double *lse_r = (double *)malloc(sizeof(double) * (size_t)H);
    double *p_r = (double *)malloc(sizeof(double) * (size_t)H * (K > 0 ? K : 1));
    fwd_row(q_rows + (size_t)r * H * Dqk, kv, idx_rows + (size_t)r * K, len_rows, r, Tk, H, Dqk, Dv, K, scale,
            sink, o_r, lse_r, p_r);
    for (int j = 0; j < K; ++j) {
      double s = 0.0;
      for (int h = 0; h < H; ++h) s += p_r[(size_t)h * K + j];
      prob[(size_t)r * K + j] = s / H;
    }
    free(o_r);
    free(lse_r);
    free(p_r);
  }
}

/* ------------------------------------------------------------------------ */
/* Indexer KL auxiliary loss over the selected slots ("sparse formulation")   */
/* [DSA-blog] "How DSA works" (the indexer emits an auxiliary KL loss that     */
/* aligns its score distribution with the main attention's; its graph is      */
/* independent of the main model's) and "Accelerating ... training results"   */
/* (indexer loss, sparse formulation, coefficient 0.001).  The pages print no */
/* formula.  Reading, per row t over its valid slot set J:                    */
/*   I_j  = score(t, idx_j)            (the indexer score above)              */
/*   q_j  = exp(I_j) / sum_J exp(I)    (the indexer's distribution)           */
/*   p_j  = prob[t,j] / sum_J prob      (the attention's, a constant: no       */
/*                                       gradient reaches the main model)     */
/*   kl[t] = sum_{j in J, p_j > 0} p_j (log p_j - log q_j)                    */
/* and with g_j = coeff (q_j - p_j) = d(coeff kl[t]) / dI_j:                  */
/*   dw[t,h]      = sum_j g_j max(0, s_hj),      s_hj = <q_idx[t,h], k[idx_j]> */
/*   dq_idx[t,h]  = sum_j g_j w[t,h] [s_hj > 0] k[idx_j]                      */
/*   dk[idx_j]   += sum_h g_j w[t,h] [s_hj > 0] q_idx[t,h]                    */
/* (the derivative of max(0, s) is taken as 0 at s = 0).  A row with no valid */
/* slot, or whose probabilities sum to 0, has kl = 0 and no gradient.         */
/* dk is added to (rows accumulate, as query chunks do).                      */
/* ------------------------------------------------------------------------ */
void oracle_indexer_kl(const double *q_rows /*[n,Hi,Di]*/, const double *k /*[Tk,Di]*/,
                       const double *w_rows /*[n,Hi]*/, const int32_t *idx_rows /*[n,K]*/,
                       const int32_t *len_rows, const double *prob_rows /*[n,K]*/, int nrows, int Tk, int Hi,
                       int Di, int K, double coeff, double *kl /*[n]*/, double *dq /*[n,Hi,Di]*/,
                       double *dw /*[n,Hi]*/, double *dk /*[Tk,Di], added to*/) {
  double *gk = (double *)calloc((size_t)nrows * (K > 0 ? K : 1) * Hi, sizeof(double)); /* g_j w_h [s>0] */
#pragma omp parallel for schedule(dynamic, 1)
  for (int r = 0; r < nrows; ++r) {
    const double *qt = q_rows + (size_t)r * Hi * Di, *wt = w_rows + (size_t)r * Hi;
    const int32_t *ir = idx_rows + (size_t)r * K;
    double *dqt = dq + (size_t)r * Hi * Di, *dwt = dw + (size_t)r * Hi;
    for (int x = 0; x < Hi * Di; ++x) dqt[x] = 0.0;
    for (int h = 0; h < Hi; ++h) dwt[h] = 0.0;
    kl[r] = 0.0;
    double *I = (double *)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
    double imax = -INFINITY, psum = 0.0;
    int nvalid = 0;
    for (int j = 0; j < K; ++j) {
      if (!slot_valid(ir, len_rows, r, j, Tk)) continue;
      I[j] = indexer_score(qt, k + (size_t)ir[j] * Di, wt, Hi, Di, NULL);
      if (I[j] > imax) imax = I[j];
      psum += prob_rows[(size_t)r * K + j];
      ++nvalid;
    }
    if (nvalid == 0 || !(psum > 0.0)) {
      free(I);
      continue;
    }
    double z = 0.0;
    for (int j = 0; j < K; ++j)
      if (slot_valid(ir, len_rows, r, j, Tk)) z += exp(I[j] - imax);
    const double logz = imax + log(z);
    double acc = 0.0;
    for (int j = 0; j < K; ++j) {
      if (!slot_valid(ir, len_rows, r, j, Tk)) continue;
      const double logq = I[j] - logz, p = prob_rows[(size_t)r * K + j] / psum;
      if (p > 0.0) acc += p * (log(p) - logq);
      const double g = coeff * (exp(logq) - p);
      const double *kj = k + (size_t)ir[j] * Di;
      for (int h = 0; h < Hi; ++h) {
        double s = 0.0;
        for (int d = 0; d < Di; ++d) s += qt[(size_t)h * Di + d] * kj[d];
        dwt[h] += g * (s > 0.0 ? s : 0.0);
        const double m = (s > 0.0) ? g * wt[h] : 0.0;
        gk[((size_t)r * K + j) * Hi + h] = m;
        for (int d = 0; d < Di; ++d) dqt[(size_t)h * Di + d] += m * kj[d];
      }
    }
    kl[r] = acc;
    free(I);
  }
  /* key gradient: fixed order over (row, slot, head) per channel range, as the MLA backward */
#pragma omp parallel
  {
    int nth = 1, id = 0;
#ifdef _OPENMP
    nth = omp_get_num_threads();
    id = omp_get_thread_num();
#endif
    const int d0 = (int)((int64_t)Di * id / nth), d1 = (int)((int64_t)Di * (id + 1) / nth);
    for (int r = 0; r < nrows; ++r) {
      const int32_t *ir = idx_rows + (size_t)r * K;
      for (int j = 0; j < K; ++j) {
        if (!slot_valid(ir, len_rows, r, j, Tk)) continue;
        double *dst = dk + (size_t)ir[j] * Di;
        for (int h = 0; h < Hi; ++h) {
          const double m = gk[((size_t)r * K + j) * Hi + h];
          if (m == 0.0) continue;
          const double *qh = q_rows + ((size_t)r * Hi + h) * Di;
          for (int d = d0; d < d1; ++d) dst[d] += m * qh[d];
        }
      }
    }
  }
  free(gk);
}

/* ------------------------------------------------------------------------ */
/* k-pool selection (GLM-5.3-Flash).  [NoPE-PR] "Why": the k-pool selection   */
/* appends the query's incomplete tail pool, so the top-k width is            */
/* 2048 + 3 = 2051.  The pages define nothing else; the readings taken:       */
/*  - a pool is P consecutive tokens of one packed sequence, counted from the */
/*    sequence start (P = 4: an incomplete pool holds at most 3 tokens);      */
/*  - a pooled row (index key or kv latent) is the mean of its P token rows,  */
/*    stored in the rows' dtype (bf16, round to nearest even);                */
/*  - query t ranks, by the indexer score against the pooled keys, the        */
/*    complete pools of its sequence that end at or before t, keeps the K     */
/*    best (ties to the lower pool), and appends the tokens of its own        */
/*    incomplete pool (0 .. P-1 of them);                                     */
/*  - attention runs over the rows [pooled rows of every sequence; token      */
/*    rows], pool p at row p and token s at row total_pools + s, so the       */
/*    selection is one ascending index list of width K + P - 1 (-1 suffix);   */
/*  - the key gradient of a token is its own row's plus 1/P of its pool's.    */
/* ------------------------------------------------------------------------ */

/* Per sequence i: pool_cu[i] = complete pools of the sequences before it.    */
/* Per token t of sequence i: pool_start[t] = pool_cu[i] (the sequence's first */
/* pool), n_pools[t] = complete pools ending at or before t, tail_start[t] =   */
/* the first token of t's incomplete pool (t + 1 when there is none).         */
/* Returns the total number of pools, or -1 if cu_seqlens is not a            */
/* non-decreasing cover of [0, T] or P < 1.                                   */
int oracle_kpool_metadata(const int32_t *cu_seqlens, int num_seqs, int T, int P, int32_t *pool_cu,
                          int32_t *pool_start, int32_t *n_pools, int32_t *tail_start) {
  if (P < 1 || num_seqs < 0 || cu_seqlens[0] != 0 || cu_seqlens[num_seqs] != T) return -1;
  int total = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int a = cu_seqlens[i], b = cu_seqlens[i + 1];
    if (b < a) return -1;
    pool_cu[i] = total;
    for (int t = a; t < b; ++t) {
      const int pos = t - a;             /* position of t in its sequence */
      const int np = (pos + 1) / P;      /* pools whose last token is <= t */
      pool_start[t] = total;
      n_pools[t] = np;
      tail_start[t] = a + np * P;        /* == t + 1 when t closes a pool */
    }
    total += (b - a) / P;
  }
  pool_cu[num_seqs] = total;
  return total;
}

/* bf16 with round to nearest even of a double that a float holds exactly or
   nearly (the mean of P bf16 values): through float, then the 16-bit round. */
static double round_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7f800000u) == 0x7f800000u) return x; /* inf / nan: out of contract */
  const uint32_t lsb = (u >> 16) & 1u;
  u = (u + 0x7fffu + lsb) & 0xffff0000u;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Pooled rows: out[pool_cu[i] + p, :] = mean of x[a + P p .. a + P p + P - 1, :] for
   every complete pool p of sequence i (a = cu_seqlens[i]); rounded to bf16 unless
   round_to_bf16 is 0. */
void oracle_kpool_pool(const double *x, int D, const int32_t *cu_seqlens, int num_seqs, int P,
                       int round_to_bf16, double *out) {
  int row = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int a = cu_seqlens[i], n = (cu_seqlens[i + 1] - a) / P;
    for (int p = 0; p < n; ++p, ++row) {
      for (int d = 0; d < D; ++d) {
        double s = 0.0;
        for (int r = 0; r < P; ++r) s += x[(int64_t)(a + p * P + r) * D + d];
        const double m = s / (double)P;
        out[(int64_t)row * D + d] = round_to_bf16 ? round_bf16(m) : m;
      }
    }
  }
}

/* One query row: the pooled selection (pool_idx[0 .. pool_len-1], pools in
   global numbering, ascending) followed by the tail tokens tail_start .. t as
   rows total_pools + s; -1 up to width.  Returns the valid count. */
int oracle_kpool_compose_row(const int32_t *pool_idx, int pool_len, int tail_start, int t, int total_pools,
                             int width, int32_t *out) {
  int n = 0;
  for (int j = 0; j < pool_len; ++j) out[n++] = pool_idx[j];
  for (int s = tail_start; s <= t; ++s) out[n++] = total_pools + s;
  for (int j = n; j < width; ++j) out[j] = -1;
  return n;
}

/* Key gradient of the tokens from the gradient of the attended rows:
   dx[t] = dcat[total_pools + t] + dcat[pool(t)] / P when t lies in a complete
   pool (pool(t) = pool_cu[i] + (t - a) / P), else dcat[total_pools + t]. */
void oracle_kpool_unpool_grad(const double *dcat, int D, const int32_t *cu_seqlens, int num_seqs, int P,
                              int total_pools, double *dx) {
  int pool0 = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int a = cu_seqlens[i], b = cu_seqlens[i + 1], n = (b - a) / P;
    for (int t = a; t < b; ++t) {
      const int p = (t - a) / P;
      for (int d = 0; d < D; ++d) {
        double g = dcat[(int64_t)(total_pools + t) * D + d];
        if (p < n) g += dcat[(int64_t)(pool0 + p) * D + d] / (double)P;
        dx[(int64_t)t * D + d] = g;
      }
    }
    pool0 += n;
  }
}
