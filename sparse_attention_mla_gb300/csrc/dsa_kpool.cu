// dsa_kpool.cu -- k-pool selection for GLM-5.3-Flash's DSA layers.
//
// Source: SkyRL PR 2388 "NoPE / unaligned top-k for SparseMLA", section "Why":
// GLM-5.3-Flash's k-pool selection appends the query's incomplete tail pool, so
// the top-k width is 2048 + 3 = 2051 (and section "Comparing against cuDNN": the
// k-pool path does its own selection instead of the token-level top-k).  The
// pages define nothing more; the readings taken here:
//  * a pool is P consecutive tokens of one packed sequence, counted from the
//    sequence start (P = 4: an incomplete pool holds at most 3 tokens), and the
//    pools are numbered across the sequences in order;
//  * a pooled row (index key or kv latent) is the mean of its P token rows,
//    stored in the rows' dtype (bf16, round to nearest even);
//  * query t ranks, with the indexer score against the pooled keys, the complete
//    pools of its sequence that end at or before t, keeps the K best (ties to the
//    lower pool) and appends the tokens of its own incomplete pool;
//  * attention runs over the rows [pooled kv; token kv] (pool p at row p, token
//    s at row total_pools + s), so one ascending index list of width K + P - 1
//    (valid prefix, -1 suffix) feeds the sparse MLA kernels unchanged;
//  * a token's key gradient is its own row's plus 1/P of its pool's (the adjoint
//    of x -> [pooled rows; x]).
//
// The selection itself is the lightning-indexer kernel with per-row key windows
// (the context-parallel entry) run over the pooled keys; this file holds the
// memory-bound pieces around it: the pool coordinates, the pooling, the
// composition of pools and tail into one index row, and the gradient back to the
// tokens.  All of them stream rows with 16-byte accesses.
#include <cuda_bf16.h>

#include <vector>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {
namespace kpool {

// Last i in [0, n) with a[i] <= v, for a non-decreasing a with a[0] <= v.
__device__ __forceinline__ int last_le(const int32_t* __restrict__ a, int n, int v) {
  int lo = 0, hi = n;  // invariant: a[lo] <= v < a[hi] (a[n] taken as +inf)
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (__ldg(a + mid) <= v) lo = mid; else hi = mid;
  }
  return lo;
}

// pool_cu[i] = complete pools of the sequences before i (one thread: the number of
// sequences is small and the scan is sequential by nature).
__global__ void pool_cu_kernel(const int32_t* __restrict__ cu, int nseq, int P, int32_t* __restrict__ pool_cu) {
  int total = 0;
  for (int i = 0; i < nseq; ++i) {
    pool_cu[i] = total;
    total += (__ldg(cu + i + 1) - __ldg(cu + i)) / P;
  }
  pool_cu[nseq] = total;
}

// Per token: the sequence's first pool, the complete pools ending at or before it, and
// the first token of its incomplete pool.
__global__ void token_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ pool_cu, int nseq, int T,
                             int P, int32_t* __restrict__ pool_start, int32_t* __restrict__ n_pools,
                             int32_t* __restrict__ tail_start) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    const int i = last_le(cu, nseq, t);  // skips empty sequences
    const int a = __ldg(cu + i);
    const int np = (t - a + 1) / P;
    pool_start[t] = __ldg(pool_cu + i);
    n_pools[t] = np;
    tail_start[t] = a + np * P;
  }
}

// Pooled rows, one thread per 16-byte unit (8 channels) of a pooled row: the P token
// rows' units are summed in fp32 and divided by P, then rounded to bf16.
__global__ void pool_kernel(const __nv_bfloat16* __restrict__ x, int D, const int32_t* __restrict__ cu,
                            const int32_t* __restrict__ pool_cu, int nseq, int P, int total_pools,
                            __nv_bfloat16* __restrict__ out) {
  const int units = D / 8;
  const long long n = (long long)total_pools * units;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < n; u += (long long)gridDim.x * blockDim.x) {
    const int g = (int)(u / units), c = (int)(u - (long long)g * units);
    const int i = last_le(pool_cu, nseq, g);  // the sequence that holds pool g
    // sequences without a complete pool share pool_cu with the next one: take the last such i
    const int first = __ldg(cu + i) + (g - __ldg(pool_cu + i)) * P;
    float acc[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] = 0.f;
    for (int r = 0; r < P; ++r) {
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(x + (size_t)(first + r) * D) + c);
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h[e]);
        acc[2 * e] += f.x;
        acc[2 * e + 1] += f.y;
      }
    }
    uint4 o;
    __nv_bfloat162* ho = reinterpret_cast<__nv_bfloat162*>(&o);
    const float fp = (float)P;
#pragma unroll
    for (int e = 0; e < 4; ++e) ho[e] = __floats2bfloat162_rn(__fdiv_rn(acc[2 * e], fp), __fdiv_rn(acc[2 * e + 1], fp));
    reinterpret_cast<uint4*>(out + (size_t)g * D)[c] = o;
  }
}

// One warp per query row: the selected pools (already ascending), the tail tokens as
// rows total_pools + s, then -1, into a row of width W; the valid count to len_out.
__global__ void compose_kernel(const int32_t* __restrict__ pidx, const int32_t* __restrict__ plen, int K,
                               const int32_t* __restrict__ tail_start, int T, int total_pools, int W,
                               int32_t* __restrict__ out, int32_t* __restrict__ len_out) {
  const int warps = (gridDim.x * blockDim.x) >> 5;
  const int lane = threadIdx.x & 31;
  for (int t = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; t < T; t += warps) {
    const int np = plen ? __ldg(plen + t) : 0;
    const int ts = __ldg(tail_start + t);
    const int nt = t + 1 - ts;  // tokens of the incomplete pool (0 .. P-1)
    const int32_t* src = pidx + (size_t)t * K;
    int32_t* dst = out + (size_t)t * W;
    for (int j = lane; j < W; j += 32) {
      int v = -1;
      if (j < np) v = __ldg(src + j);
      else if (j < np + nt) v = total_pools + ts + (j - np);
      dst[j] = v;
    }
    if (len_out != nullptr && lane == 0) len_out[t] = np + nt;
  }
}

// Token key gradient, one thread per 4-channel unit: the token's own row plus 1/P of its
// pool's row when the token lies in a complete pool.
__global__ void unpool_kernel(const float* __restrict__ dcat, int T, int D, const int32_t* __restrict__ cu,
                              const int32_t* __restrict__ pool_cu, int nseq, int P, int total_pools,
                              float* __restrict__ dx) {
  const int units = D / 4;
  const long long n = (long long)T * units;
  const float inv = 1.f / (float)P;
  for (long long u = blockIdx.x * (long long)blockDim.x + threadIdx.x; u < n; u += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(u / units), c = (int)(u - (long long)t * units);
    float4 g = __ldg(reinterpret_cast<const float4*>(dcat + (size_t)(total_pools + t) * D) + c);
    const int i = last_le(cu, nseq, t);
    const int a = __ldg(cu + i), p = (t - a) / P;
    if (p < (__ldg(cu + i + 1) - a) / P) {  // t lies in a complete pool
      const float4 q = __ldg(reinterpret_cast<const float4*>(dcat + (size_t)(__ldg(pool_cu + i) + p) * D) + c);
      g.x = fmaf(q.x, inv, g.x);
      g.y = fmaf(q.y, inv, g.y);
      g.z = fmaf(q.z, inv, g.z);
      g.w = fmaf(q.w, inv, g.w);
    }
    reinterpret_cast<float4*>(dx + (size_t)t * D)[c] = g;
  }
}

int grid_for(long long work, int threads) {
  long long b = (work + threads - 1) / threads;
  if (b > 152 * 16) b = 152 * 16;
  return (int)(b < 1 ? 1 : b);
}

}  // namespace kpool
}  // namespace dsa

using namespace dsa;

extern "C" dsa_status_t dsa_kpool_metadata(const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                           int32_t pool, int32_t* pool_cu, int32_t* pool_start, int32_t* n_pools,
                                           int32_t* tail_start, int32_t* total_pools_host, dsa_stream_t stream) {
  const char* who = "dsa_kpool_metadata";
  if (!cu_seqlens || !pool_cu) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: cu_seqlens or pool_cu is NULL", who);
  if (num_seqs < 1) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: num_seqs must be >= 1", who);
  if (total_tokens < 0) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: total_tokens < 0", who);
  if (pool < 1) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: pool must be >= 1 (got %d)", who, pool);
  if (total_tokens > 0 && (!pool_start || !n_pools || !tail_start))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: output pointer is NULL", who);
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::vector<int32_t> cu(num_seqs + 1);
  if ((st = cuda_check(cudaMemcpyAsync(cu.data(), cu_seqlens, sizeof(int32_t) * (num_seqs + 1),
                                       cudaMemcpyDeviceToHost, s),
                       "copying cu_seqlens")))
    return st;
  if ((st = cuda_check(cudaStreamSynchronize(s), "synchronising the stream"))) return st;
  if (cu[0] != 0 || cu[num_seqs] != total_tokens)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: cu_seqlens must run from 0 to total_tokens (%d .. %d, T = %d)", who,
                cu[0], cu[num_seqs], total_tokens);
  int64_t total = 0;
  for (int i = 0; i < num_seqs; ++i) {
    if (cu[i + 1] < cu[i]) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: cu_seqlens decreases at %d", who, i);
    total += (cu[i + 1] - cu[i]) / pool;
  }
  kpool::pool_cu_kernel<<<1, 1, 0, s>>>(cu_seqlens, num_seqs, pool, pool_cu);
  if ((st = cuda_check(cudaGetLastError(), "launching pool_cu_kernel"))) return st;
  if (total_tokens > 0) {
    kpool::token_kernel<<<kpool::grid_for(total_tokens, 256), 256, 0, s>>>(
        cu_seqlens, pool_cu, num_seqs, total_tokens, pool, pool_start, n_pools, tail_start);
    if ((st = cuda_check(cudaGetLastError(), "launching the k-pool token kernel"))) return st;
  }
  if (total_pools_host) *total_pools_host = (int32_t)total;
  return ok();
}

extern "C" dsa_status_t dsa_kpool_pool(const dsa_bf16_t* x, int32_t total_tokens, int32_t D, const int32_t* cu_seqlens,
                                       const int32_t* pool_cu, int32_t num_seqs, int32_t pool, int32_t total_pools,
                                       dsa_bf16_t* out, dsa_stream_t stream) {
  const char* who = "dsa_kpool_pool";
  if (total_tokens < 0 || num_seqs < 1 || pool < 1 || total_pools < 0 || (int64_t)total_pools * pool > total_tokens)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: need T >= 0, num_seqs >= 1, pool >= 1, 0 <= total_pools <= T / pool",
                who);
  if (D < 8 || D % 8 != 0) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: D must be a positive multiple of 8 (got %d)", who, D);
  if (total_pools == 0) {
    dsa_status_t st = check_device();
    return st == DSA_OK ? ok() : st;
  }
  if (!x || !out || !cu_seqlens || !pool_cu) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: null pointer", who);
  if (!aligned16(x) || !aligned16(out)) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: x and out must be 16-byte aligned", who);
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  kpool::pool_kernel<<<kpool::grid_for((long long)total_pools * (D / 8), 256), 256, 0, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(x), D, cu_seqlens, pool_cu, num_seqs, pool, total_pools,
      reinterpret_cast<__nv_bfloat16*>(out));
  if ((st = cuda_check(cudaGetLastError(), "launching the k-pool pooling kernel"))) return st;
  return ok();
}

// Workspace: [the indexer's error word | selected pools int32 [T, K] | their counts int32 [T]].
static size_t align256(size_t b) { return (b + 255) & ~size_t(255); }

extern "C" size_t dsa_kpool_topk_workspace_size(int32_t T, int32_t K) {
  const size_t t = T > 0 ? (size_t)T : 0, k = K > 0 ? (size_t)K : 0;
  return align256(dsa_indexer_topk_workspace_size(T, K)) + align256(t * k * 4) + align256(t * 4);
}

extern "C" dsa_status_t dsa_kpool_topk(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_pool, const float* head_weights,
                                       const int32_t* pool_start, const int32_t* n_pools, const int32_t* tail_start,
                                       int32_t T, int32_t total_pools, int32_t Hi, int32_t Di, int32_t K, int32_t pool,
                                       int32_t* topk_idx, int32_t* topk_len, void* workspace, size_t workspace_bytes,
                                       dsa_stream_t stream) {
  const char* who = "dsa_kpool_topk";
  if (T < 0 || total_pools < 0 || pool < 1)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: need T >= 0, total_pools >= 0 and pool >= 1", who);
  if (K < 1 || K > 2048) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: K must be in [1, 2048] (got %d)", who, K);
  if (Hi < 1 || Hi > 64) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Hi must be in [1, 64] (got %d)", who, Hi);
  if (Di != 128) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Di must be 128 (got %d)", who, Di);
  if (T > 0 && (!tail_start || !topk_idx)) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: null tensor pointer", who);
  if (T > 0 && total_pools > 0 && (!q_idx || !k_pool || !head_weights || !pool_start || !n_pools))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: null tensor pointer", who);
  dsa_status_t st = check_workspace(workspace, workspace_bytes, dsa_kpool_topk_workspace_size(T, K), who);
  if (st != DSA_OK) return st;
  uint8_t* ws = reinterpret_cast<uint8_t*>(workspace);
  const size_t ws_idx = align256(dsa_indexer_topk_workspace_size(T, K));
  int32_t* pidx = reinterpret_cast<int32_t*>(ws + ws_idx);
  int32_t* plen = reinterpret_cast<int32_t*>(ws + ws_idx + align256((size_t)T * K * 4));
  if (total_pools > 0) {
    // the K best complete pools of each row: the indexer over the pooled keys, row t's
    // window being pools [pool_start[t], pool_start[t] + n_pools[t] - 1]
    st = dsa_indexer_topk_cp(q_idx, k_pool, head_weights, pool_start, n_pools, T, total_pools, Hi, Di, K, pidx, plen,
                             workspace, ws_idx, stream);
    if (st != DSA_OK) return st;
  } else {
    if ((st = check_device()) != DSA_OK) return st;
    if ((st = clear_error_word(workspace, reinterpret_cast<cudaStream_t>(stream))) != DSA_OK) return st;
  }
  if (T == 0) return ok();
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int W = K + pool - 1;
  kpool::compose_kernel<<<kpool::grid_for((long long)T * 32, 256), 256, 0, s>>>(
      total_pools > 0 ? pidx : nullptr, total_pools > 0 ? plen : nullptr, K, tail_start, T, total_pools, W, topk_idx,
      topk_len);
  if ((st = cuda_check(cudaGetLastError(), "launching the k-pool compose kernel"))) return st;
  return ok();
}

extern "C" dsa_status_t dsa_kpool_unpool_grad(const float* dcat, int32_t total_tokens, int32_t D,
                                              const int32_t* cu_seqlens, const int32_t* pool_cu, int32_t num_seqs,
                                              int32_t pool, int32_t total_pools, float* dx, dsa_stream_t stream) {
  const char* who = "dsa_kpool_unpool_grad";
  if (total_tokens < 0 || num_seqs < 1 || pool < 1 || total_pools < 0 || (int64_t)total_pools * pool > total_tokens)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: need T >= 0, num_seqs >= 1, pool >= 1, 0 <= total_pools <= T / pool",
                who);
  if (D < 4 || D % 4 != 0) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: D must be a positive multiple of 4 (got %d)", who, D);
  if (total_tokens == 0) {
    dsa_status_t st = check_device();
    return st == DSA_OK ? ok() : st;
  }
  if (!dcat || !dx || !cu_seqlens || !pool_cu) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: null pointer", who);
  if (!aligned16(dcat) || !aligned16(dx)) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: dcat and dx must be 16-byte aligned", who);
  const char* a0 = reinterpret_cast<const char*>(dcat);
  const char* a1 = a0 + ((size_t)total_pools + total_tokens) * D * 4;
  const char* b0 = reinterpret_cast<const char*>(dx);
  const char* b1 = b0 + (size_t)total_tokens * D * 4;
  if (b0 < a1 && a0 < b1) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: dx must not overlap dcat", who);
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  kpool::unpool_kernel<<<kpool::grid_for((long long)total_tokens * (D / 4), 256), 256, 0, s>>>(
      dcat, total_tokens, D, cu_seqlens, pool_cu, num_seqs, pool, total_pools, dx);
  if ((st = cuda_check(cudaGetLastError(), "launching the k-pool gradient kernel"))) return st;
  return ok();
}
