/*
 * dsa.h -- C ABI of the GB300 (sm_103a) DeepSeek Sparse Attention hot path.
 *
 * Conventions for every entry point:
 *  - Tensor arguments are caller-owned DEVICE pointers to contiguous row-major
 *    storage (innermost dimension last); host pointers are named *_host.
 *  - bf16 tensors are passed as dsa_bf16_t (the raw 16-bit pattern).
 *  - Calls are asynchronous on the caller's CUDA stream (NULL = legacy default
 *    stream); only dsa_packed_metadata and dsa_read_device_status synchronise.
 *  - The library never allocates device memory.  Scratch comes from the
 *    caller's `workspace` (at least dsa_*_workspace_size() bytes, 256-byte
 *    aligned); its first 4 bytes are the device error word (see
 *    dsa_read_device_status).
 *  - Every call returns a dsa_status_t; argument errors are detected on the
 *    host before anything is launched and leave all outputs untouched.
 *    dsa_last_error_message() describes the most recent failure of the calling
 *    thread.
 *
 * Pages cited (title, then section or API entry):
 *  [DSA-blog]  "Accelerating GLM-5.2 Long-Context Training with cuDNN Fused DSA
 *              Kernels and THD-Packed Context Parallelism using Megatron Bridge"
 *  [NoPE-PR]   SkyRL pull request 2388 (NoPE / unaligned top-k SparseMLA)
 *  [cudnn_dsa] NeMo AutoModel API: glm_moe_dsa.kernels.cudnn_dsa
 *  [Chunk-PR]  SkyRL pull request 2423 (query-chunked sparse attention)
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;
typedef struct CUstream_st* dsa_stream_t; /* same type as cudaStream_t */
typedef uint16_t dsa_bf16_t;              /* bfloat16 bit pattern */

typedef enum {
  DSA_OK = 0,
  DSA_ERR_UNSUPPORTED = 1,      /* no CUDA device, or the device is not sm_103 */
  DSA_ERR_DTYPE = 2,            /* reserved: the ABI fixes every dtype */
  DSA_ERR_INVALID_ARGUMENT = 3, /* null pointer, bad shape, K or scale */
  DSA_ERR_WORKSPACE = 4,        /* workspace missing, too small or misaligned */
  DSA_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed */
  DSA_ERR_DEVICE_INDEX = 6,     /* device saw an index outside [-1, T_k) (slot masked) */
  DSA_ERR_TIMEOUT = 7           /* a bounded device-side wait gave up (CTA exited) */
} dsa_status_t;

/* Text for a status code (static storage). */
const char* dsa_status_string(dsa_status_t status);
/* Message of the calling thread's most recent failed call ("" if none). */
const char* dsa_last_error_message(void);
/* ABI version: 2 (attention sink arguments of the sparse MLA calls). */
int32_t dsa_abi_version(void);

/*
 * dsa_packed_metadata -- THD packing metadata, no context parallelism.
 * Source: [cudnn_dsa] prepare_cudnn_dsa_packed_metadata and
 * CudnnDsaPackedMetadata (starts, causal_lengths, max_seqlen,
 * all_rows_nonempty): per query token t of sequence i,
 *   seq_start[t] = cu_seqlens[i],  causal_len[t] = t - cu_seqlens[i] + 1.
 *  cu_seqlens   device int32 [num_seqs + 1], cu[0] = 0, non-decreasing, cu[num_seqs] = total_tokens
 *  seq_start    device int32 [total_tokens] (out)
 *  causal_len   device int32 [total_tokens] (out)
 *  max_seqlen_host, all_rows_nonempty_host: host int32 scalars (out), may be NULL
 * Like the pages' routine it performs one device-to-host synchronisation (to
 * validate cu_seqlens and return max_seqlen).  Returns
 * DSA_ERR_INVALID_ARGUMENT if cu_seqlens is not a valid cover of [0, T).
 */
dsa_status_t dsa_packed_metadata(const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                 int32_t* seq_start, int32_t* causal_len, int32_t* max_seqlen_host,
                                 int32_t* all_rows_nonempty_host, dsa_stream_t stream);

/*
 * dsa_packed_metadata_cp -- THD packing metadata for rank-local queries and
 * gathered global keys (context parallelism).
 * Source: [cudnn_dsa] prepare_cudnn_dsa_packed_metadata (query_indices,
 * cu_seqlens_padded, padding_mask; per-query global padded-storage starts and
 * real causal lengths) and cudnn_indexer_topk (rank-local index_q, gathered
 * global index_k).  With P = cu_seqlens_padded (or cu_seqlens when NULL) and
 * L_i = cu_seqlens[i+1] - cu_seqlens[i], local row r has global coordinate
 * g = query_indices[r] (r when NULL); when P[i] <= g < P[i+1]:
 *   seq_start[r] = P[i],  causal_len[r] = g - P[i] + 1 if g - P[i] < L_i and
 *   padding_mask[r] == 0, else 0 (a padding row);
 * a row outside every sequence's storage gets seq_start[r] = g, causal_len 0.
 *  cu_seqlens         device int32 [num_seqs + 1], from 0, non-decreasing (real tokens)
 *  cu_seqlens_padded  device int32 [num_seqs + 1] or NULL, from 0, non-decreasing,
 *                     P[i+1] - P[i] >= L_i, P[num_seqs] <= total_key_tokens
 *  query_indices      device int32 [T_q] or NULL (then row r is coordinate r and
 *                     T_q <= total_key_tokens), each in [0, total_key_tokens)
 *  padding_mask       device uint8 [T_q] or NULL; nonzero marks a padding row
 *  seq_start, causal_len  device int32 [T_q] (out)
 *  max_seqlen_host    host int32 (out) = max_i L_i, may be NULL
 *  all_rows_nonempty_host  host int32 (out) = 1 iff T_q > 0 and every
 *                     causal_len > 0, may be NULL
 * Performs one device-to-host synchronisation (to validate the inputs and
 * compute the host scalars) and returns DSA_ERR_INVALID_ARGUMENT when any rule
 * above is broken; the outputs are then untouched.  With no optional input it
 * equals dsa_packed_metadata.
 */
dsa_status_t dsa_packed_metadata_cp(const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, int32_t num_seqs,
                                    int32_t total_key_tokens, const int32_t* query_indices,
                                    const uint8_t* padding_mask, int32_t T_q, int32_t* seq_start,
                                    int32_t* causal_len, int32_t* max_seqlen_host, int32_t* all_rows_nonempty_host,
                                    dsa_stream_t stream);

/*
 * dsa_indexer_topk -- lightning-indexer score fused with per-query causal top-k.
 * Source: [DSA-blog] "How DSA works" (the indexer scores query-key relevance
 * and emits the top-k indices per query); [cudnn_dsa] cudnn_indexer_topk
 * (index_q [T, H_index, 128], index_k [T_k, 128], already-scaled head weights,
 * output int32 global indices, K in [1, 2048]); canonical output form from
 * cudnn_sparse_attention's topk_length (compact ascending prefix).
 *   score(t, s) = sum_h w[t,h] * max(0, <q_idx[t,h,:], k_idx[s,:]>),  s in [seq_start[t], t]
 * For each t the n = min(K, causal_len[t]) highest-scoring keys (ties to the
 * lower index) are written ascending to topk_idx[t, 0:n], then -1 up to K.
 * The [T, T_k] score matrix is never written to memory.
 *  q_idx        device bf16 [T, Hi, Di]; Hi in [1, 64], Di = 128
 *  k_idx        device bf16 [T_k, Di]
 *  head_weights device fp32 [T, Hi] (caller applies any scaling)
 *  seq_start    device int32 [T] from dsa_packed_metadata (window start; the
 *               window end is the token itself, so T_k >= T is required)
 *  topk_idx     device int32 [T, K] (out);  topk_len device int32 [T] (out) or NULL
 *  workspace    >= dsa_indexer_topk_workspace_size() bytes
 */
size_t dsa_indexer_topk_workspace_size(int32_t T, int32_t K);
dsa_status_t dsa_indexer_topk(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx, const float* head_weights,
                              const int32_t* seq_start, int32_t T, int32_t T_k, int32_t Hi, int32_t Di, int32_t K,
                              int32_t* topk_idx, int32_t* topk_len, void* workspace, size_t workspace_bytes,
                              dsa_stream_t stream);

/*
 * dsa_indexer_topk_cp -- the same kernel for rank-local query rows against the
 * gathered global keys (context parallelism).
 * Source: [cudnn_dsa] cudnn_indexer_topk (rank-local index_q [T_q, H_index,
 * 128], gathered global index_k [T_k, 128], query_indices / packed_metadata).
 * Row r's candidates are the keys [seq_start[r], seq_start[r] + causal_len[r]
 * - 1] (none when causal_len[r] = 0), clipped to [0, T_k); otherwise as
 * dsa_indexer_topk: n = min(K, window size) best keys, ascending, -1 suffix.
 *  q_idx        device bf16 [T_q, Hi, Di] (local rows)
 *  k_idx        device bf16 [T_k, Di] (global keys; no relation between T_k and T_q)
 *  head_weights device fp32 [T_q, Hi]
 *  seq_start, causal_len  device int32 [T_q] from dsa_packed_metadata_cp
 *  topk_idx, topk_len, workspace  as dsa_indexer_topk
 * Errors as dsa_indexer_topk (without the T_k >= T rule), plus
 * DSA_ERR_INVALID_ARGUMENT when causal_len is NULL and T_q > 0.
 */
dsa_status_t dsa_indexer_topk_cp(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx, const float* head_weights,
                                 const int32_t* seq_start, const int32_t* causal_len, int32_t T_q, int32_t T_k,
                                 int32_t Hi, int32_t Di, int32_t K, int32_t* topk_idx, int32_t* topk_len,
                                 void* workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * dsa_indexer_topk_with_scores -- diagnostic form of dsa_indexer_topk: the same
 * kernel code and the same results (topk_idx, topk_len), and in addition the
 * fp32 score of every key of the window of rows [score_row0, score_row0 +
 * score_rows), stored at scores[(t - score_row0) * T_k + key] (device fp32
 * [score_rows, T_k], caller-owned; entries outside a row's window are left
 * untouched).  These are exactly the values the selection ranked, so a test
 * can check the selection itself (order by score descending, ties to the
 * lower index) independently of fp32 rounding.  The pages have no
 * counterpart; this entry is for tests and diagnostics.  Errors as for
 * dsa_indexer_topk, plus DSA_ERR_INVALID_ARGUMENT unless 0 <= score_row0,
 * score_row0 + score_rows <= T and scores != NULL when score_rows > 0.
 */
dsa_status_t dsa_indexer_topk_with_scores(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx, const float* head_weights,
                                          const int32_t* seq_start, int32_t T, int32_t T_k, int32_t Hi, int32_t Di,
                                          int32_t K, int32_t* topk_idx, int32_t* topk_len, float* scores,
                                          int32_t score_row0, int32_t score_rows, void* workspace,
                                          size_t workspace_bytes, dsa_stream_t stream);

/*
 * dsa_indexer_topk_scored -- dsa_indexer_topk (causal_len NULL) or
 * dsa_indexer_topk_cp (causal_len given) that also returns, slot for slot, the
 * fp32 score the selection ranked: topk_score[t, j] = score(t, topk_idx[t, j])
 * for j < topk_len[t], -inf after.  Same kernel and same topk_idx / topk_len as
 * those calls; the scores are the ones the kernel kept with each candidate.
 * Their consumer is dsa_indexer_kl, whose loss needs exactly these values
 * (the KL term of [DSA-blog] "How DSA works" compares the indexer's score
 * distribution over the selected slots with the attention's).
 *  topk_score   device fp32 [T, K] (out; required when T > 0)
 *  the rest     as dsa_indexer_topk / dsa_indexer_topk_cp
 * Errors as those calls, plus DSA_ERR_INVALID_ARGUMENT when topk_score is NULL.
 */
dsa_status_t dsa_indexer_topk_scored(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx, const float* head_weights,
                                     const int32_t* seq_start, const int32_t* causal_len, int32_t T, int32_t T_k,
                                     int32_t Hi, int32_t Di, int32_t K, int32_t* topk_idx, int32_t* topk_len,
                                     float* topk_score, void* workspace, size_t workspace_bytes,
                                     dsa_stream_t stream);

/*
 * dsa_indexer_kl -- the indexer's KL auxiliary loss over each row's selected
 * slots, and its gradient.
 * Source: [DSA-blog] "How DSA works" (the indexer emits an auxiliary KL loss
 * that aligns its score distribution with the main attention's; its graph is
 * independent of the main model's) and the training-results section (indexer
 * loss, sparse formulation, coefficient 0.001).  The pages print no formula;
 * reading taken, per row t over its valid slots J (as in the sparse MLA calls):
 *   I_j = score(t, topk_idx[t,j])  (the indexer score of dsa_indexer_topk)
 *   q_j = softmax_J(I),  p_j = attn_prob[t,j] / sum_J attn_prob[t,:]
 *   kl[t] = sum_{j: p_j > 0} p_j (log p_j - log q_j)
 * with g_j = coeff (q_j - p_j), s_hj = <q_idx[t,h], k_idx[idx_j]> and
 * m_hj = g_j w[t,h] [s_hj > 0]:
 *   dw[t,h] = sum_j g_j max(0, s_hj),  dq_idx[t,h,:] = sum_j m_hj k_idx[idx_j,:],
 *   dk_idx_accum[idx_j,:] += sum_h m_hj q_idx[t,h,:].
 * A row with no valid slot, or whose attn_prob sums to 0, gets kl = 0 and no
 * gradient.  The attention side is a constant (no gradient reaches it).
 *  q_idx, k_idx, head_weights  as dsa_indexer_topk (Hi in [1, 64], Di = 128)
 *  topk_idx     device int32 [T, K], K in [1, 4096];  topk_len device int32 [T] or NULL
 *  attn_prob    device fp32 [T, K]: e.g. the attn_prob output of dsa_sparse_mla_bwd
 *  topk_score   device fp32 [T, K] or NULL: the scores I_j of the slots, e.g. the
 *               topk_score output of dsa_indexer_topk_scored for this topk_idx.
 *               Given, they are read instead of formed again (one pass over the
 *               selected keys instead of two); the ReLU masks of the gradient are
 *               formed from the keys as always.  NULL: I_j is formed here.
 *  coeff        the loss coefficient (the pages train with 0.001); the gradients
 *               are those of coeff * sum_t kl[t]
 *  kl           device fp32 [T] (out);  dq_idx device bf16 [T, Hi, Di] (out)
 *  dw           device fp32 [T, Hi] (out)
 *  dk_idx_accum device fp32 [T_k, Di]: zeroed first when accumulate == 0
 *  workspace    >= dsa_indexer_kl_workspace_size() bytes
 * Indices outside [-1, T_k) are masked and reported through the device error
 * word.  Summation order of dk_idx_accum across rows is not deterministic.
 */
size_t dsa_indexer_kl_workspace_size(int32_t T, int32_t K);
dsa_status_t dsa_indexer_kl(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx, const float* head_weights,
                            const int32_t* topk_idx, const int32_t* topk_len, const float* attn_prob,
                            const float* topk_score, int32_t T, int32_t T_k, int32_t Hi, int32_t Di, int32_t K,
                            float coeff, float* kl,
                            dsa_bf16_t* dq_idx, float* dw, float* dk_idx_accum, int32_t accumulate,
                            void* workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * k-pool selection (GLM-5.3-Flash).  Source: [NoPE-PR] "Why" (the k-pool
 * selection appends the query's incomplete tail pool, so the top-k width is
 * 2048 + 3 = 2051) and "Comparing against cuDNN" (the k-pool path makes its own
 * selection instead of the token-level top-k).  The pages define nothing more;
 * readings taken: a pool is P consecutive tokens of one packed sequence counted
 * from its start (P = 4: an incomplete pool holds at most 3 tokens), numbered
 * across the sequences in order; a pooled row is the bf16 mean of its P token
 * rows; query t keeps the K complete pools of its sequence that end at or
 * before t with the best indexer score against the pooled keys, then the tokens
 * of its incomplete pool; attention runs over [pooled kv; token kv] (pool p at
 * row p, token s at row total_pools + s) with the sparse MLA entries unchanged,
 * and a token's key gradient is its row's plus 1/P of its pool's.
 */

/*
 * dsa_kpool_metadata -- pool coordinates of a packed batch.  For sequence i
 * (L_i tokens) and token t of it at position u = t - cu_seqlens[i]:
 *   pool_cu[i] = sum_{j<i} floor(L_j / P),  pool_cu[num_seqs] = total pools,
 *   pool_start[t] = pool_cu[i],  n_pools[t] = floor((u + 1) / P) (complete pools
 *   ending at or before t),  tail_start[t] = cu_seqlens[i] + P n_pools[t] (the
 *   first token of t's incomplete pool; t + 1 when t closes a pool).
 *  cu_seqlens   device int32 [num_seqs + 1], from 0, non-decreasing, ending at total_tokens
 *  pool         P >= 1
 *  pool_cu      device int32 [num_seqs + 1] (out)
 *  pool_start, n_pools, tail_start  device int32 [total_tokens] (out)
 *  total_pools_host  host int32 (out), may be NULL
 * Performs one device-to-host synchronisation to validate cu_seqlens
 * (DSA_ERR_INVALID_ARGUMENT when a rule above is broken; outputs untouched).
 */
dsa_status_t dsa_kpool_metadata(const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens, int32_t pool,
                                int32_t* pool_cu, int32_t* pool_start, int32_t* n_pools, int32_t* tail_start,
                                int32_t* total_pools_host, dsa_stream_t stream);

/*
 * dsa_kpool_pool -- pooled rows: out[pool_cu[i] + p, :] = bf16(sum_{r<P}
 * x[cu_seqlens[i] + P p + r, :] / P) (fp32 sum, round to nearest even) for every
 * complete pool p of every sequence i.  For the index keys (D = 128) and the kv
 * latents (D = 576 or 512).
 *  x            device bf16 [total_tokens, D], D a multiple of 8, 16-byte aligned
 *  cu_seqlens, pool_cu, num_seqs, pool, total_pools  as dsa_kpool_metadata
 *  out          device bf16 [total_pools, D] (out), 16-byte aligned
 */
dsa_status_t dsa_kpool_pool(const dsa_bf16_t* x, int32_t total_tokens, int32_t D, const int32_t* cu_seqlens,
                            const int32_t* pool_cu, int32_t num_seqs, int32_t pool, int32_t total_pools,
                            dsa_bf16_t* out, dsa_stream_t stream);

/*
 * dsa_kpool_topk -- per query row t: the K pools of [pool_start[t],
 * pool_start[t] + n_pools[t] - 1] with the highest indexer score (the score and
 * ranking of dsa_indexer_topk, ties to the lower pool) against the pooled keys,
 * ascending, then the rows total_pools + s for s = tail_start[t] .. t, then -1,
 * in rows of width K + pool - 1; topk_len[t] = the valid count.
 *  q_idx, head_weights  as dsa_indexer_topk (T query rows, Hi in [1, 64], Di = 128)
 *  k_pool       device bf16 [total_pools, Di] (dsa_kpool_pool of the index keys)
 *  pool_start, n_pools, tail_start  device int32 [T] (dsa_kpool_metadata)
 *  K            in [1, 2048] (2048 for GLM-5.3-Flash)
 *  topk_idx     device int32 [T, K + pool - 1] (out);  topk_len device int32 [T] (out) or NULL
 *  workspace    >= dsa_kpool_topk_workspace_size(T, K) bytes; its first word is
 *               the device error word (dsa_read_device_status)
 */
size_t dsa_kpool_topk_workspace_size(int32_t T, int32_t K);
dsa_status_t dsa_kpool_topk(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_pool, const float* head_weights,
                            const int32_t* pool_start, const int32_t* n_pools, const int32_t* tail_start, int32_t T,
                            int32_t total_pools, int32_t Hi, int32_t Di, int32_t K, int32_t pool, int32_t* topk_idx,
                            int32_t* topk_len, void* workspace, size_t workspace_bytes, dsa_stream_t stream);

/*
 * dsa_kpool_unpool_grad -- token key gradient from the gradient of the attended
 * rows (the adjoint of x -> [pooled rows; x], without the bf16 rounding):
 *   dx[t, :] = dcat[total_pools + t, :] + dcat[pool(t), :] / P if t lies in a
 *   complete pool (pool(t) = pool_cu[i] + floor((t - cu_seqlens[i]) / P)),
 *   else dcat[total_pools + t, :].
 *  dcat         device fp32 [total_pools + total_tokens, D] (e.g. the dkv
 *               accumulator of dsa_sparse_mla_bwd over [pooled kv; kv]), D a
 *               multiple of 4, 16-byte aligned
 *  dx           device fp32 [total_tokens, D] (out), 16-byte aligned, not overlapping dcat
 */
dsa_status_t dsa_kpool_unpool_grad(const float* dcat, int32_t total_tokens, int32_t D, const int32_t* cu_seqlens,
                                   const int32_t* pool_cu, int32_t num_seqs, int32_t pool, int32_t total_pools,
                                   float* dx, dsa_stream_t stream);

/*
 * dsa_sparse_mla_fwd -- absorbed sparse MLA forward (MQA over one latent KV).
 * Source: [DSA-blog] "How DSA works" and "Why DSA needs fused kernels";
 * [cudnn_dsa] cudnn_sparse_attention / _CudnnSparseAttention.forward (q
 * [T, H, 576], kv_latent [T_k, 1, 576], int32 indices with -1 invalid, optional
 * topk_length, explicit softmax_scale, output [T, H, 512]); [NoPE-PR] "Change"
 * (value = kv[..., :512], NoPE width 512, unaligned top-k widths).
 * Slot j of row t is valid iff topk_idx[t,j] >= 0 and (topk_len == NULL or
 * j < topk_len[t]); per (t, h):
 *   z_j = softmax_scale * <q[t,h,:], kv[idx_j,:]>,  lse[t,h] = ln sum_j exp(z_j),
 *   out[t,h,:] = sum_j exp(z_j - lse) * kv[idx_j, 0:Dv].
 * A row with no valid slot gets out = 0 and lse = -inf.  Indices >= T_k or
 * < -1 are masked and reported through the device error word.
 * Attention sink ([cudnn_dsa] _pad_attention_heads pads a sink [H] with q;
 * the pages print no formula; reading taken): attn_sink[h] is one more logit
 * of every row of head h, in the units of z, with no value row:
 *   lse[t,h] = ln(sum_j exp(z_j) + exp(attn_sink[h])),  out as above,
 * so a row with no valid slot gets out = 0 and lse = attn_sink[h].  A sink of
 * -inf is no sink; NaN or +inf sinks are outside the contract.
 *  q        device bf16 [T, H, Dqk], Dqk in {512, 576};  kv device bf16 [T_k, Dqk]
 *  topk_idx device int32 [T, K], any K >= 1;  topk_len device int32 [T] or NULL
 *  attn_sink device fp32 [H] or NULL (no sink)
 *  out      device bf16 [T, H, Dv] (out), Dv = 512;  lse device fp32 [T, H] (out)
 *  out_lo   device bf16 [T, H, Dv] (out) or NULL: the rounding residual
 *           bf16(O - out) of the fp32 result O (P.V runs on bf16 hi + lo parts
 *           of P, so O is accurate to about fp32).  Passing it on to the
 *           backward makes D = <dout, O> use that O instead of the rounded out
 *           (library addition; the pages' interface returns out only).
 *  workspace >= dsa_sparse_mla_fwd_workspace_size() bytes
 * Query chunking ([Chunk-PR] "Summary"): rows are independent, so a chunk is a
 * call on row-offset pointers of q/topk_idx/out/lse with the full kv.
 */
size_t dsa_sparse_mla_fwd_workspace_size(int32_t T, int32_t H);
dsa_status_t dsa_sparse_mla_fwd(const dsa_bf16_t* q, const dsa_bf16_t* kv, const int32_t* topk_idx,
                                const int32_t* topk_len, int32_t T, int32_t T_k, int32_t H, int32_t Dqk,
                                int32_t Dv, int32_t K, float softmax_scale, const float* attn_sink, dsa_bf16_t* out,
                                dsa_bf16_t* out_lo, float* lse, void* workspace, size_t workspace_bytes,
                                dsa_stream_t stream);

/*
 * dsa_sparse_mla_bwd -- analytic backward of dsa_sparse_mla_fwd.
 * Source: [cudnn_dsa] _CudnnSparseAttention.backward (gradients for the query
 * [T, H, 576] and the latent KV from grad_output [T, H, 512]); [Chunk-PR]
 * "Summary" (query chunks are independent, key gradients sum).
 * With P_j = exp(z_j - lse), D = <dout, out>, dP_j = <dout, kv[idx_j,:Dv]>,
 * dS_j = P_j (dP_j - D):
 *   dq[t,h,:]         = softmax_scale * sum_j dS_j kv[idx_j, :]
 *   dkv_accum[idx_j,:] += softmax_scale * sum_h dS_j q[t,h,:]
 *   dkv_accum[idx_j,0:Dv] += sum_h P_j dout[t,h,:]
 * and with a sink, P_sink = exp(attn_sink[h] - lse[t,h]):
 *   d_sink[h] += -sum_t P_sink[t,h] D[t,h]
 *  q, kv, topk_idx, topk_len, sizes, softmax_scale, attn_sink: as in the forward call
 *  out, lse       device: the forward's outputs for these rows
 *  out_lo         device bf16 [T, H, Dv]: the forward's residual, or NULL (then D
 *                 is computed from the rounded out)
 *  dout           device bf16 [T, H, Dv]
 *  dq             device bf16 [T, H, Dqk] (out)
 *  dkv_accum      device fp32 [T_k, Dqk]: zeroed first when accumulate == 0,
 *                 added to when accumulate == 1 (query chunks)
 *  d_sink         device fp32 [H] or NULL (needs attn_sink): zeroed first when
 *                 accumulate == 0, added to when accumulate == 1
 *  attn_prob      device fp32 [T, K] (out) or NULL: the head-averaged attention
 *                 probability of every slot, (1/H) sum_h P[t,h,j] (0 for an
 *                 invalid slot), the target distribution of dsa_indexer_kl;
 *                 computed from the P the backward already forms
 *  dkv_bf16       device bf16 [T_k, Dqk] (out, rounded copy of dkv_accum) or NULL
 *  workspace      >= dsa_sparse_mla_bwd_workspace_size(T, H, K) bytes: the
 *                 error word, 256 scratch-slot flags, D (T*H fp32) and the
 *                 scratch slots for the bf16 dS of one row's tiles (256 slots
 *                 x ceil(K/128) x 16 KiB; a CTA claims a free slot and
 *                 releases it on exit).  One workspace serves one call at a
 *                 time: calls whose executions overlap must not share it.
 * Summation order of dkv_accum (and d_sink) across rows is not deterministic
 * (fp32 atomics).
 */
size_t dsa_sparse_mla_bwd_workspace_size(int32_t T, int32_t H, int32_t K);
dsa_status_t dsa_sparse_mla_bwd(const dsa_bf16_t* q, const dsa_bf16_t* kv, const int32_t* topk_idx,
                                const int32_t* topk_len, int32_t T, int32_t T_k, int32_t H, int32_t Dqk,
                                int32_t Dv, int32_t K, float softmax_scale, const float* attn_sink,
                                const dsa_bf16_t* out, const dsa_bf16_t* out_lo, const float* lse,
                                const dsa_bf16_t* dout, dsa_bf16_t* dq, float* dkv_accum, float* d_sink,
                                float* attn_prob, int32_t accumulate, dsa_bf16_t* dkv_bf16, void* workspace,
                                size_t workspace_bytes, dsa_stream_t stream);

/*
 * dsa_sparse_mla_bwd_noalloc -- dsa_sparse_mla_bwd without a caller workspace.
 * The pages have no counterpart: this is a library addition for callers that
 * cannot allocate device memory (runtimes that reserve all device memory in
 * their own pool and forbid other allocations, or plug-ins whose host program
 * owns every allocation) and so cannot supply the workspace.  Arguments,
 * semantics and results are those of dsa_sparse_mla_bwd.
 *  - Scratch is a fixed 84 MiB + 1280 B device array built into the library,
 *    held by every GPU that loads it until the process exits; K must not
 *    exceed dsa_sparse_mla_bwd_noalloc_max_topk() (2176), else
 *    DSA_ERR_WORKSPACE is returned and nothing is launched.  Its D part holds
 *    4 Mi (row, head) pairs: longer calls run in row chunks of
 *    floor(4 Mi / H) rows, one after the other on `stream`, with dkv_accum
 *    and d_sink accumulating over the chunks.
 *  - The call allocates nothing.  The first call on a device (and again after
 *    the device's context is replaced) looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call
 *    before any stream capture.
 *  - Every call uses the same array: calls whose executions overlap on the
 *    GPU race on it and must be ordered by the caller (same stream or events).
 *    Each call clears the array's error word and slot flags; the device error
 *    word is read with dsa_sparse_mla_bwd_noalloc_read_status.
 */
int32_t dsa_sparse_mla_bwd_noalloc_max_topk(void);
dsa_status_t dsa_sparse_mla_bwd_noalloc(const dsa_bf16_t* q, const dsa_bf16_t* kv, const int32_t* topk_idx,
                                        const int32_t* topk_len, int32_t T, int32_t T_k, int32_t H, int32_t Dqk,
                                        int32_t Dv, int32_t K, float softmax_scale, const float* attn_sink,
                                        const dsa_bf16_t* out, const dsa_bf16_t* out_lo, const float* lse,
                                        const dsa_bf16_t* dout, dsa_bf16_t* dq, float* dkv_accum, float* d_sink,
                                        float* attn_prob, int32_t accumulate, dsa_bf16_t* dkv_bf16,
                                        dsa_stream_t stream);
/*
 * dsa_sparse_mla_bwd_noalloc_read_status -- the no-alloc backward's device
 * error word: synchronise `stream`, read and clear the word in the built-in
 * array and store it in *status_host (DSA_OK, DSA_ERR_DEVICE_INDEX or
 * DSA_ERR_TIMEOUT), as dsa_read_device_status does for a workspace.  No
 * counterpart on the pages (library addition).
 */
dsa_status_t dsa_sparse_mla_bwd_noalloc_read_status(dsa_stream_t stream, int32_t* status_host);

/*
 * dsa_set_wait_limit_cycles -- the cycle limit of every bounded device-side
 * wait of the kernels launched after the call (process-wide; the default is
 * 2^31 SM cycles, about one second).  A wait that runs past it records
 * DSA_ERR_TIMEOUT in the device error word and its CTA leaves its work and
 * exits cleanly; 0 gives up at the first wait whose phase has not completed,
 * which lets a test drive every timeout path on purpose.  A negative value
 * restores the default.  Returns the previous limit.  Library addition with
 * no counterpart on the pages.
 */
int64_t dsa_set_wait_limit_cycles(int64_t cycles);

/*
 * dsa_read_device_status -- synchronise `stream`, read and clear the device
 * error word at the start of `workspace`, and store it in *status_host
 * (DSA_OK, DSA_ERR_DEVICE_INDEX or DSA_ERR_TIMEOUT).  Library addition with no
 * counterpart on the pages: it surfaces the bounded-wait and index checks.
 */
dsa_status_t dsa_read_device_status(void* workspace, dsa_stream_t stream, int32_t* status_host);

#ifdef __cplusplus
}
#endif
#endif /* DSA_H_ */
