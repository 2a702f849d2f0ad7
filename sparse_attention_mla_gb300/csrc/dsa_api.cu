// dsa_api.cu -- status reporting, device checks, tensor maps, workspace sizes,
// the device error word, and dsa_packed_metadata.
#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "dsa_host.h"
#include "dsa_once.h"

namespace dsa {

static thread_local char g_msg[512] = "";

dsa_status_t fail(dsa_status_t st, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof(g_msg), fmt, ap);
  va_end(ap);
  return st;
}

dsa_status_t ok() {
  g_msg[0] = '\0';
  return DSA_OK;
}

dsa_status_t cuda_check(cudaError_t e, const char* what) {
  if (e == cudaSuccess) return DSA_OK;
  return fail(DSA_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

dsa_status_t check_device() {
  static std::mutex mu;
  static int verdict[64];  // 0 unknown, 1 ok, 2 unsupported
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fail(DSA_ERR_UNSUPPORTED, "no CUDA device available");
  }
  if (dev < 0 || dev >= 64) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (verdict[dev] == 0) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    verdict[dev] = (major == 10 && minor == 3) ? 1 : 2;
    if (verdict[dev] == 2) {
      return fail(DSA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a only", dev,
                  major, minor);
    }
  }
  if (verdict[dev] == 2) return fail(DSA_ERR_UNSUPPORTED, "device %d is not sm_103", dev);
  return DSA_OK;
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
    cudaGetLastError();
  });
  return fn;
}

dsa_status_t make_map_2d_bf16(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                              uint64_t pitch_elems, uint32_t box_cols, uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {pitch_elems * 2};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DSA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return DSA_OK;
}

dsa_status_t check_workspace(const void* ws, size_t bytes, size_t need, const char* who) {
  if (!ws) return fail(DSA_ERR_WORKSPACE, "%s: workspace is NULL (need %zu bytes)", who, need);
  if ((reinterpret_cast<uintptr_t>(ws) & 255u) != 0)
    return fail(DSA_ERR_WORKSPACE, "%s: workspace must be 256-byte aligned", who);
  if (bytes < need) return fail(DSA_ERR_WORKSPACE, "%s: workspace has %zu bytes, needs %zu", who, bytes, need);
  return DSA_OK;
}

dsa_status_t clear_error_word(void* ws, cudaStream_t stream) {
  return cuda_check(cudaMemsetAsync(ws, 0, sizeof(int), stream), "clearing the device error word");
}

static std::atomic<long long> g_wait_limit{1ll << 31};
long long wait_limit_cycles() { return g_wait_limit.load(std::memory_order_relaxed); }

dsa_status_t configure_kernel_smem(const void* func, int bytes, const char* what) {
  static PerDeviceOnce table;
  int dev = 0;
  dsa_status_t st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != DSA_OK) return st;
  table.run(func, dev, [&] {
    st = cuda_check(cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes), what);
    // all of the SM's unified L1 / shared memory as shared memory, so that kernels sized for two
    // CTAs per SM get them
    if (st == DSA_OK)
      st = cuda_check(cudaFuncSetAttribute(func, cudaFuncAttributePreferredSharedMemoryCarveout,
                                           (int)cudaSharedmemCarveoutMaxShared),
                      what);
    return st == DSA_OK;
  });
  return st;
}

// ---------------------------------------------------------------------------
// THD metadata: per token, start of its sequence and causal length.
// ---------------------------------------------------------------------------
__global__ void packed_metadata_kernel(const int32_t* __restrict__ cu, int nseq, int T, int32_t* __restrict__ start,
                                       int32_t* __restrict__ clen) {
  for (int t = blockIdx.x * blockDim.x + threadIdx.x; t < T; t += gridDim.x * blockDim.x) {
    // last i with cu[i] <= t (skips empty sequences, whose cu[i] == cu[i+1])
    int lo = 0, hi = nseq;  // invariant: cu[lo] <= t < cu[hi]
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (__ldg(cu + mid) <= t) lo = mid; else hi = mid;
    }
    int s = __ldg(cu + lo);
    start[t] = s;
    clen[t] = t - s + 1;
  }
}

// Context-parallel form: row r has global padded-storage coordinate g (query_idx[r], or r);
// with P the storage boundaries, the last i with P[i] <= g is its sequence when g < P[nseq].
__global__ void packed_metadata_cp_kernel(const int32_t* __restrict__ cu, const int32_t* __restrict__ P, int nseq,
                                          const int32_t* __restrict__ qidx, const uint8_t* __restrict__ mask, int Tq,
                                          int32_t* __restrict__ start, int32_t* __restrict__ clen) {
  for (int r = blockIdx.x * blockDim.x + threadIdx.x; r < Tq; r += gridDim.x * blockDim.x) {
    const int g = qidx ? __ldg(qidx + r) : r;
    int s = g, len = 0;
    if (g < __ldg(P + nseq)) {
      int lo = 0, hi = nseq;  // invariant: P[lo] <= g < P[hi]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (__ldg(P + mid) <= g) lo = mid; else hi = mid;
      }
      s = __ldg(P + lo);
      const int pos = g - s;
      const bool pad = mask != nullptr && __ldg(mask + r) != 0;
      if (pos < __ldg(cu + lo + 1) - __ldg(cu + lo) && !pad) len = pos + 1;
    }
    start[r] = s;
    clen[r] = len;
  }
}

}  // namespace dsa

using namespace dsa;

extern "C" {

const char* dsa_status_string(dsa_status_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: no sm_103 CUDA device";
    case DSA_ERR_DTYPE: return "DSA_ERR_DTYPE";
    case DSA_ERR_INVALID_ARGUMENT: return "DSA_ERR_INVALID_ARGUMENT";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA";
    case DSA_ERR_DEVICE_INDEX: return "DSA_ERR_DEVICE_INDEX: an index outside [-1, T_k) was masked";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT: a bounded device wait gave up";
  }
  return "unknown dsa_status_t";
}

const char* dsa_last_error_message(void) { return g_msg; }

int32_t dsa_abi_version(void) { return 3; }

int64_t dsa_set_wait_limit_cycles(int64_t cycles) {
  return g_wait_limit.exchange(cycles < 0 ? (1ll << 31) : cycles);
}

dsa_status_t dsa_read_device_status(void* workspace, dsa_stream_t stream, int32_t* status_host) {
  if (!workspace || !status_host) return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_read_device_status: null pointer");
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  int32_t v = 0;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = cuda_check(cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, s), "reading error word")))
    return st;
  if ((st = cuda_check(cudaStreamSynchronize(s), "synchronising the stream"))) return st;
  if ((st = clear_error_word(workspace, s))) return st;
  *status_host = v;
  return ok();
}

dsa_status_t dsa_packed_metadata(const int32_t* cu_seqlens, int32_t num_seqs, int32_t total_tokens,
                                 int32_t* seq_start, int32_t* causal_len, int32_t* max_seqlen_host,
                                 int32_t* all_rows_nonempty_host, dsa_stream_t stream) {
  if (!cu_seqlens) return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_packed_metadata: cu_seqlens is NULL");
  if (num_seqs < 1) return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_packed_metadata: num_seqs must be >= 1");
  if (total_tokens < 0) return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_packed_metadata: total_tokens < 0");
  if (total_tokens > 0 && (!seq_start || !causal_len))
    return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_packed_metadata: output pointer is NULL");
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  std::vector<int32_t> cu(num_seqs + 1);
  if ((st = cuda_check(cudaMemcpyAsync(cu.data(), cu_seqlens, sizeof(int32_t) * (num_seqs + 1),
                                       cudaMemcpyDeviceToHost, s),
                       "copying cu_seqlens")))
    return st;
  if ((st = cuda_check(cudaStreamSynchronize(s), "synchronising the stream"))) return st;
  if (cu[0] != 0) return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_packed_metadata: cu_seqlens[0] = %d, not 0", cu[0]);
  if (cu[num_seqs] != total_tokens)
    return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_packed_metadata: cu_seqlens[%d] = %d != total_tokens %d", num_seqs,
                cu[num_seqs], total_tokens);
  int32_t mx = 0;
  for (int i = 0; i < num_seqs; ++i) {
    if (cu[i + 1] < cu[i])
      return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_packed_metadata: cu_seqlens decreases at %d", i);
    if (cu[i + 1] - cu[i] > mx) mx = cu[i + 1] - cu[i];
  }
  if (total_tokens > 0) {
    int threads = 256;
    int blocks = (total_tokens + threads - 1) / threads;
    if (blocks > 152 * 8) blocks = 152 * 8;
    packed_metadata_kernel<<<blocks, threads, 0, s>>>(cu_seqlens, num_seqs, total_tokens, seq_start, causal_len);
    if ((st = cuda_check(cudaGetLastError(), "launching packed_metadata_kernel"))) return st;
  }
  if (max_seqlen_host) *max_seqlen_host = mx;
  if (all_rows_nonempty_host) *all_rows_nonempty_host = total_tokens > 0 ? 1 : 0;
  return ok();
}

dsa_status_t dsa_packed_metadata_cp(const int32_t* cu_seqlens, const int32_t* cu_seqlens_padded, int32_t num_seqs,
                                    int32_t total_key_tokens, const int32_t* query_indices,
                                    const uint8_t* padding_mask, int32_t T_q, int32_t* seq_start,
                                    int32_t* causal_len, int32_t* max_seqlen_host, int32_t* all_rows_nonempty_host,
                                    dsa_stream_t stream) {
  const char* who = "dsa_packed_metadata_cp";
  if (!cu_seqlens) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: cu_seqlens is NULL", who);
  if (num_seqs < 1) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: num_seqs must be >= 1", who);
  if (T_q < 0 || total_key_tokens < 0) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: T_q and total_key_tokens must be >= 0", who);
  if (!query_indices && T_q > total_key_tokens)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: without query_indices, T_q (%d) must be <= total_key_tokens (%d)", who,
                T_q, total_key_tokens);
  if (T_q > 0 && (!seq_start || !causal_len)) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: output pointer is NULL", who);
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // one device-to-host synchronisation: boundaries, coordinates and mask for validation
  std::vector<int32_t> cu(num_seqs + 1), P(num_seqs + 1), qi(query_indices ? T_q : 0);
  std::vector<uint8_t> pm(padding_mask ? T_q : 0);
  const size_t nb = sizeof(int32_t) * (num_seqs + 1);
  if ((st = cuda_check(cudaMemcpyAsync(cu.data(), cu_seqlens, nb, cudaMemcpyDeviceToHost, s), "copying cu_seqlens")))
    return st;
  if (cu_seqlens_padded &&
      (st = cuda_check(cudaMemcpyAsync(P.data(), cu_seqlens_padded, nb, cudaMemcpyDeviceToHost, s),
                       "copying cu_seqlens_padded")))
    return st;
  if (!qi.empty() && (st = cuda_check(cudaMemcpyAsync(qi.data(), query_indices, sizeof(int32_t) * qi.size(),
                                                      cudaMemcpyDeviceToHost, s),
                                      "copying query_indices")))
    return st;
  if (!pm.empty() &&
      (st = cuda_check(cudaMemcpyAsync(pm.data(), padding_mask, pm.size(), cudaMemcpyDeviceToHost, s),
                       "copying padding_mask")))
    return st;
  if ((st = cuda_check(cudaStreamSynchronize(s), "synchronising the stream"))) return st;
  if (!cu_seqlens_padded) P = cu;
  if (cu[0] != 0 || P[0] != 0)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: cu_seqlens[0] and cu_seqlens_padded[0] must be 0", who);
  if (P[num_seqs] > total_key_tokens)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: the padded storage (%d rows) exceeds total_key_tokens (%d)", who,
                P[num_seqs], total_key_tokens);
  int32_t mx = 0;
  for (int i = 0; i < num_seqs; ++i) {
    const int32_t L = cu[i + 1] - cu[i];
    if (L < 0 || P[i + 1] < P[i])
      return fail(DSA_ERR_INVALID_ARGUMENT, "%s: sequence boundaries decrease at %d", who, i);
    if (L > P[i + 1] - P[i])
      return fail(DSA_ERR_INVALID_ARGUMENT, "%s: sequence %d has %d real tokens but %d storage rows", who, i, L,
                  P[i + 1] - P[i]);
    if (L > mx) mx = L;
  }
  // every coordinate inside the key tokens; a row is nonempty when it is a real, unmasked token
  int nonempty = T_q > 0 ? 1 : 0;
  for (int32_t r = 0; r < T_q; ++r) {
    const int32_t g = qi.empty() ? r : qi[r];
    if (g < 0 || g >= total_key_tokens)
      return fail(DSA_ERR_INVALID_ARGUMENT, "%s: query_indices[%d] = %d outside [0, %d)", who, r, g, total_key_tokens);
    if (!nonempty) continue;
    const int i = (int)(std::upper_bound(P.begin(), P.begin() + num_seqs, g) - P.begin()) - 1;
    if (g >= P[num_seqs] || g - P[i] >= cu[i + 1] - cu[i] || (!pm.empty() && pm[r])) nonempty = 0;
  }
  if (T_q > 0) {
    const int threads = 256;
    int blocks = (T_q + threads - 1) / threads;
    if (blocks > 152 * 8) blocks = 152 * 8;
    packed_metadata_cp_kernel<<<blocks, threads, 0, s>>>(cu_seqlens, cu_seqlens_padded ? cu_seqlens_padded : cu_seqlens,
                                                         num_seqs, query_indices, padding_mask, T_q, seq_start,
                                                         causal_len);
    if ((st = cuda_check(cudaGetLastError(), "launching packed_metadata_cp_kernel"))) return st;
  }
  if (max_seqlen_host) *max_seqlen_host = mx;
  if (all_rows_nonempty_host) *all_rows_nonempty_host = nonempty;
  return ok();
}

}  // extern "C"
