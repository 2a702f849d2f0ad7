// dsa_indexer.cu -- lightning-indexer score fused with per-query causal top-k
// on sm_103a (tcgen05 + TMEM + TMA).
//
//   score(t, s) = sum_h w[t,h] * max(0, <q_idx[t,h,:], k_idx[s,:]>),  s in [seq_start[t], t]
// and for each t the n = min(K, causal length) best keys (score descending,
// ties to the lower index), written ascending with a -1 suffix.  With context
// parallelism the rows are rank-local queries against the gathered global
// keys, and each row's window [seq_start, seq_start + causal_len - 1] comes
// from the context-parallel metadata (empty for padding rows).
// Source: "Accelerating GLM-5.2 Long-Context Training with cuDNN Fused DSA
// Kernels ...", "How DSA works" (the indexer scores query-key relevance and
// emits the top-k per query) and "Why DSA needs fused kernels" (the S x S
// score matrix must stay on chip); NeMo AutoModel
// glm_moe_dsa.kernels.cudnn_indexer_topk (index_q [T, H_index, 128], one
// shared index_k [T_k, 128], pre-scaled fp32 head weights, K in [1, 2048]);
// the canonical ascending/-1 form from cudnn_sparse_attention (topk_length).
//
// Design (sm_103a):
//  * One CTA owns 4 consecutive query tokens.  Their 4 x 64 index heads form
//    the N = 256 side of the MMA; keys are the M = 128 side:
//    D[key, (token, head)] = K_tile . Q^T, fp32 in TMEM, double-buffered
//    (2 x 256 columns).  k_idx tiles arrive by TMA (2 boxes of 64 channels).
//  * 16 epilogue warps, 4 per token (one TMEM lane = one key), apply ReLU and
//    the fp32 head-weighted sum, so scores exist only in registers; each token
//    has its own warp group, named barrier and candidate buffer, so the four
//    tokens' selections run in parallel.
//  * Selection: each token keeps a shared-memory buffer of candidates
//    (score, index) that beat its running threshold.  Candidates are appended
//    in ascending key order (a block-wide scan, not atomics).  A full buffer
//    is compacted by a two-pass (16-bit) radix select on the order-preserving
//    integer image of the score: every candidate at or above the bucket that
//    holds the K-th best is kept, a superset of the final top-K, and the
//    threshold rises to that bucket.  The final selection is an exact
//    four-pass select where ties at the threshold keep the earliest
//    (= lowest-index) entries.  Every compaction is stable, so the buffer
//    stays sorted by index and the output needs no sort; its keep passes take
//    512 candidates per block (4 per thread) with one count scan per block.
#include <climits>
#include <cmath>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {
namespace idx {

constexpr int kEpi = 512;                 // 16 epilogue warps: 4 per query token
constexpr int kThreads = 64 + kEpi;       // + producer warp + MMA warp
constexpr int kTokens = 4;     // query tokens per CTA
constexpr int kHeads = 64;     // index heads (padded)
constexpr int kDi = 128;       // index head dim
constexpr int kTile = 128;     // keys per tile
constexpr int kN = kTokens * kHeads;
constexpr int kMaxK = 2048;

constexpr int OFF_Q = 0;                       // 2 chunks x [256 rows x 128 B]
constexpr int Q_CHUNK = kN * 128;              // 32 KiB
constexpr int OFF_K = OFF_Q + 2 * Q_CHUNK;     // 2 stages x 2 chunks x [128 rows x 128 B]
constexpr int K_CHUNK = kTile * 128;           // 16 KiB
constexpr int K_STAGE = 2 * K_CHUNK;
constexpr int OFF_MISC = OFF_K + 2 * K_STAGE;  // 128 KiB
constexpr int MISC = 6144;
constexpr int OFF_CAND = OFF_MISC + MISC;
constexpr int CAP = 2944;                      // candidates per token
constexpr int TOTAL = OFF_CAND + kTokens * CAP * 8 + 1024;
static_assert(TOTAL <= 232448, "shared memory budget");
static_assert(CAP >= kMaxK + kTile + 128, "candidate buffer must hold K + one tile");

// misc layout
constexpr int M_KF = 0, M_KE = 16, M_DF = 32, M_DE = 48, M_FIN = 64;
constexpr int M_TMEM = 128, M_ABORT = 132;
constexpr int M_W = 256;                // float [4][64]
constexpr int M_WCNT = M_W + 1024;      // int [4 tokens][2 parity][4 warps]
constexpr int M_HIST = M_WCNT + 128;    // int [4 tokens][256]
constexpr int M_SEL = M_HIST + 4096;    // int [4 tokens][4]
static_assert(M_SEL + 64 <= MISC, "misc layout");

__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
// d = a * b + c on two fp32 lanes at once (round to nearest, as fmaf per lane).
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

__device__ __forceinline__ uint32_t ordered(float f) {
  const uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unordered(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Per-token context: 4 warps (128 threads, one per TMEM lane quadrant), one named barrier.
struct Half {
  int bar;     // named barrier id
  int tid;     // 0..127 within the half (ordered by key row)
  int wq;      // warp position 0..3 by key row (lane quadrant)
  int lane;
  int* wcnt;   // [2 parity][4]
  int* hist;   // [256]
  int* sel;    // [4]
};

// Exclusive block scan of a predicate over the 128 threads of a half in
// key-row order; returns (exclusive prefix, total).  Uses wcnt[par].
__device__ __forceinline__ int2 half_scan(const Half& hf, bool pred, int par) {
  const uint32_t ball = __ballot_sync(0xffffffffu, pred);
  if (hf.lane == 0) hf.wcnt[par * 4 + hf.wq] = __popc(ball);
  named_bar(hf.bar, 128);
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int c = hf.wcnt[par * 4 + w];
    before += (w < hf.wq) ? c : 0;
    total += c;
  }
  before += __popc(ball & ((1u << hf.lane) - 1u));
  return make_int2(before, total);
}

// Exclusive block scan of per-thread counts over the 128 threads of a half, in
// thread order; returns (exclusive prefix, total).  Uses wcnt[par].
__device__ __forceinline__ int2 half_scan_count(const Half& hf, int n, int par) {
  int incl = n;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (hf.lane >= o) incl += v;
  }
  if (hf.lane == 31) hf.wcnt[par * 4 + hf.wq] = incl;
  named_bar(hf.bar, 128);
  int before = 0, total = 0;
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    const int c = hf.wcnt[par * 4 + w];
    before += (w < hf.wq) ? c : 0;
    total += c;
  }
  return make_int2(before + incl - n, total);
}

// Exact (passes = 4): keep the best `target` of the cnt candidates (score
// desc, index asc), stably, in place; returns v with "accept iff key > v".
// Approximate (passes = 2): find the key bucket that holds the target-th best
// after two 8-bit digits and keep every candidate at or above that bucket,
// stably: a superset of the best `target` (so the final exact selection is
// unchanged) in half the passes; returns the bucket floor minus one, again
// "accept iff key > v".  *kept_out receives the number kept.
// The digits start just below the candidates' common key prefix (the bits
// where the smallest and the largest key image agree): candidates near a
// running threshold share sign and exponent, so digits taken from the top
// would put nearly all of them into one histogram bin.
__device__ uint32_t compact(const Half& hf, float* cs, int* ci, int cnt, int target, int& parity, int passes,
                            int* kept_out) {
  // common prefix: min and max key image over the candidates
  uint32_t kmin = 0xffffffffu, kmax = 0u;
  for (int e = hf.tid; e < cnt; e += 128) {
    const uint32_t key = ordered(cs[e]);
    kmin = min(kmin, key);
    kmax = max(kmax, key);
  }
  kmin = __reduce_min_sync(0xffffffffu, kmin);
  kmax = __reduce_max_sync(0xffffffffu, kmax);
  if (hf.lane == 0) {
    hf.hist[2 * hf.wq] = (int)kmin;
    hf.hist[2 * hf.wq + 1] = (int)kmax;
  }
  named_bar(hf.bar, 128);
#pragma unroll
  for (int w = 0; w < 4; ++w) {
    kmin = min(kmin, (uint32_t)hf.hist[2 * w]);
    kmax = max(kmax, (uint32_t)hf.hist[2 * w + 1]);
  }
  named_bar(hf.bar, 128);  // hist is cleared next
  const uint32_t diff = kmin ^ kmax;
  int top = diff ? 32 - __clz(diff) : 0;  // bits [top, 32) are common to every candidate
  uint32_t pmask = top >= 32 ? 0u : ~((1u << top) - 1u);
  uint32_t prefix = kmin & pmask;
  // radix select of the target-th largest key image, 8 bits per pass below the resolved bits
  int kk = target;
  for (int pass = 0; pass < passes && top > 0; ++pass) {
    const int shift = top > 8 ? top - 8 : 0;
    const uint32_t dmask = (1u << (top - shift)) - 1u;  // 1..8 bits
    hf.hist[hf.tid] = 0;
    hf.hist[hf.tid + 128] = 0;
    named_bar(hf.bar, 128);
    for (int e = hf.tid; e < cnt; e += 128) {
      const uint32_t key = ordered(cs[e]);
      if ((key & pmask) == prefix) atomicAdd(&hf.hist[(key >> shift) & dmask], 1);
    }
    named_bar(hf.bar, 128);
    if (hf.wq == 0) {
      // lane l owns bins 255-8l .. 248-8l (descending)
      int c[8], s = 0;
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        c[b] = hf.hist[255 - 8 * hf.lane - b];
        s += c[b];
      }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (hf.lane >= o) incl += v;
      }
      int above = incl - s;  // count in bins above this lane's first bin
      if (above < kk && kk <= incl) {
#pragma unroll
        for (int b = 0; b < 8; ++b) {
          if (above < kk && kk <= above + c[b]) {
            hf.sel[0] = 255 - 8 * hf.lane - b;
            hf.sel[1] = above;
          }
          above += c[b];
        }
      }
    }
    named_bar(hf.bar, 128);
    const int d = hf.sel[0];
    kk -= hf.sel[1];
    prefix |= (uint32_t)d << shift;
    pmask |= dmask << shift;
    top = shift;
    named_bar(hf.bar, 128);  // sel is rewritten by the next pass
  }
  if (passes < 4) {
    // keep every key >= prefix (the bucket floor), stably, in place: blocks of 512 candidates,
    // 4 consecutive ones per thread (16-byte loads), one scan and one barrier per block.  Every
    // thread has read its 4 before the barrier, and the block's writes land below its end.
    int kept = 0;
    for (int base = 0; base < cnt; base += 512) {
      const int e0 = base + 4 * hf.tid;
      float sv[4] = {0.f, 0.f, 0.f, 0.f};
      int iv[4] = {0, 0, 0, 0};
      if (e0 + 3 < cnt) {
        const float4 a = *reinterpret_cast<const float4*>(cs + e0);
        const int4 b = *reinterpret_cast<const int4*>(ci + e0);
        sv[0] = a.x, sv[1] = a.y, sv[2] = a.z, sv[3] = a.w;
        iv[0] = b.x, iv[1] = b.y, iv[2] = b.z, iv[3] = b.w;
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (e0 + j < cnt) sv[j] = cs[e0 + j], iv[j] = ci[e0 + j];
      }
      bool keep[4];
      int m = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        keep[j] = (e0 + j < cnt) && ordered(sv[j]) >= prefix;
        m += keep[j];
      }
      const int2 ke = half_scan_count(hf, m, parity);
      parity ^= 1;
      int pos = kept + ke.x;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (keep[j]) {
          cs[pos] = sv[j];
          ci[pos] = iv[j];
          ++pos;
        }
      kept += ke.y;
    }
    named_bar(hf.bar, 128);
    *kept_out = kept;
    return prefix - 1u;  // prefix >= 1: the target-th best has key >= prefix > 0
  }
  const uint32_t v = prefix;  // kk >= 1 ties at v are kept (the earliest ones)
  int kept = 0, ties = 0;
  // blocks of 512 candidates, 4 consecutive ones per thread; per block one scan of the ties at v
  // (earlier ties win) and one of the kept, in candidate order.  Every thread has read its 4
  // before the first barrier, and the block's writes land below its end.
  for (int base = 0; base < cnt; base += 512) {
    const int e0 = base + 4 * hf.tid;
    float sv[4] = {0.f, 0.f, 0.f, 0.f};
    int iv[4] = {0, 0, 0, 0};
    if (e0 + 3 < cnt) {
      const float4 a = *reinterpret_cast<const float4*>(cs + e0);
      const int4 b = *reinterpret_cast<const int4*>(ci + e0);
      sv[0] = a.x, sv[1] = a.y, sv[2] = a.z, sv[3] = a.w;
      iv[0] = b.x, iv[1] = b.y, iv[2] = b.z, iv[3] = b.w;
    } else {
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (e0 + j < cnt) sv[j] = cs[e0 + j], iv[j] = ci[e0 + j];
    }
    uint32_t key[4];
    bool eq[4];
    int neq = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      key[j] = ordered(sv[j]);
      eq[j] = (e0 + j < cnt) && key[j] == v;
      neq += eq[j];
    }
    const int2 te = half_scan_count(hf, neq, parity);
    parity ^= 1;
    int tie_rank = ties + te.x;  // ties at v before this thread's candidates
    bool keep[4];
    int nkeep = 0;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      keep[j] = (e0 + j < cnt) && (key[j] > v || (eq[j] && tie_rank < kk));
      tie_rank += eq[j];
      nkeep += keep[j];
    }
    const int2 ke = half_scan_count(hf, nkeep, parity);
    parity ^= 1;
    int pos = kept + ke.x;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (keep[j]) {
        cs[pos] = sv[j];
        ci[pos] = iv[j];
        ++pos;
      }
    kept += ke.y;
    ties += te.y;
  }
  named_bar(hf.bar, 128);
  *kept_out = kept;
  return v;
}

// kScores: the diagnostic variant that also stores, for rows [score_row0,
// score_row0 + score_rows), the fp32 score of every key of the row's window
// (scores[(t - score_row0) * Tk + key]), i.e. exactly the values it selects from.
template <bool kScores>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_topk_kernel(const __grid_constant__ CUtensorMap k_map, const __nv_bfloat16* __restrict__ q_idx,
                        const float* __restrict__ w, const int32_t* __restrict__ seq_start,
                        const int32_t* __restrict__ causal_len, int T, int Tk, int Hi,
                        int K, int32_t* __restrict__ topk_idx, int32_t* __restrict__ topk_len,
                        float* __restrict__ topk_score, int* __restrict__ err, float* __restrict__ scores,
                        int score_row0, int score_rows, long long wait_limit) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + OFF_Q);
  const uint32_t sK = smem_u32(smem + OFF_K);
  uint8_t* misc = smem + OFF_MISC;
  const uint32_t bar_kf = smem_u32(misc + M_KF), bar_ke = smem_u32(misc + M_KE);
  const uint32_t bar_df = smem_u32(misc + M_DF), bar_de = smem_u32(misc + M_DE);
  const uint32_t bar_fin = smem_u32(misc + M_FIN);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + M_TMEM);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + M_ABORT);
  float* s_w = reinterpret_cast<float*>(misc + M_W);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // heaviest (latest) token blocks first
  const int nblk = (T + kTokens - 1) / kTokens;
  const int t0 = (nblk - 1 - (int)blockIdx.x) * kTokens;
  const int nt = min(kTokens, T - t0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_kf + 8 * s, 1);
      mbar_init(bar_ke + 8 * s, 1);
      mbar_init(bar_df + 8 * s, 1);
      mbar_init(bar_de + 8 * s, kEpi / 32);
    }
    mbar_init(bar_fin, 1);
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  // Key window of token t: [seq_start[t], seq_start[t] + causal_len[t] - 1] when the
  // lengths are given (context-parallel rows, possibly empty), else [seq_start[t], t];
  // clipped to the keys [0, Tk).  Empty: (1, 0).
  auto window = [&](int t, int& a, int& b) {
    a = __ldg(seq_start + t);
    b = causal_len ? a + __ldg(causal_len + t) - 1 : t;
    a = max(a, 0);
    b = min(b, Tk - 1);
    if (b < a) a = 1, b = 0;
  };
  // key-tile range covering every token's window
  int lo = INT_MAX, hi = -1;
  for (int k = 0; k < nt; ++k) {
    int a, b;
    window(t0 + k, a, b);
    if (b >= a) {
      lo = min(lo, a);
      hi = max(hi, b);
    }
  }
  const int kt0 = lo / kTile, kt1 = hi / kTile;
  const int ntiles = (hi >= lo) ? kt1 - kt0 + 1 : 0;

  if (warp >= 2) {
    const int tid = threadIdx.x - 64;
    // Q rows (token k, head h) -> 2 chunks of [256 rows x 128 B], swizzled; padding rows are
    // zero-filled without a read.  All copies are in flight at once (cp.async), one wait.
    const uint64_t pol = l2_evict_first_policy();  // q_idx is read once: evicted first, k_idx stays
    for (int u = tid; u < kN * 16; u += kEpi) {
      const int row = u >> 4, c = (u >> 3) & 1, uc = u & 7;
      const int k = row / kHeads, h = row - k * kHeads;
      const bool ok = k < nt && h < Hi;
      cp_async16_hint(sQ + c * Q_CHUNK + sw128_off(row, uc),
                      q_idx + (ok ? ((size_t)(t0 + k) * Hi + h) * kDi + c * 64 + uc * 8 : 0), ok ? 16u : 0u, pol);
    }
    for (int u = tid; u < kTokens * kHeads; u += kEpi) {
      const int k = u / kHeads, h = u - k * kHeads;
      s_w[u] = (k < nt && h < Hi) ? __ldg(w + (size_t)(t0 + k) * Hi + h) : 0.f;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    fence_proxy_async_smem();
  }
  __syncthreads();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    // ======================= producer: k_idx tiles =======================
    if (lane == 0) {
      int i = 0;
      for (; i < ntiles; ++i) {
        const int s = i & 1;
        if (!mbar_wait(bar_ke + 8 * s, ((i >> 1) & 1) ^ 1, s_abort, err, wait_limit)) break;
        mbar_expect_tx(bar_kf + 8 * s, K_STAGE);
        const int row = (kt0 + i) * kTile;
        tma_load_2d(sK + s * K_STAGE, &k_map, 0, row, bar_kf + 8 * s);
        tma_load_2d(sK + s * K_STAGE + K_CHUNK, &k_map, 64, row, bar_kf + 8 * s);
      }
      if (*s_abort) {
        // tiles i-2 and i-1 may both be in flight (two stages): both land before the CTA exits
        volatile int dummy = 0;
        for (int j = (i >= 2 ? i - 2 : 0); j < i; ++j) mbar_wait(bar_kf + 8 * (j & 1), (j >> 1) & 1, &dummy, err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t kId = idesc_bf16(128, kN, false, false);
      for (int i = 0; i < ntiles; ++i) {
        const int s = i & 1, b = i & 1;
        if (!mbar_wait(bar_kf + 8 * s, (i >> 1) & 1, s_abort, err, wait_limit)) break;
        if (!mbar_wait(bar_de + 8 * b, ((i >> 1) & 1) ^ 1, s_abort, err, wait_limit)) break;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss(tmem + b * kN, sdesc_sw128(sK + s * K_STAGE + c * K_CHUNK + k * 32, 16, 1024),
                   sdesc_sw128(sQ + c * Q_CHUNK + k * 32, 16, 1024), kId, (c | k) != 0);
        mma_commit(bar_ke + 8 * s);
        mma_commit(bar_df + 8 * b);
      }
      mma_commit(bar_fin);
      volatile int dummy = 0;
      mbar_wait(bar_fin, 0, &dummy, err);
    }
    __syncwarp();
  } else {
    // ======================= score epilogue + selection (one 4-warp group per token) =======================
    const int ew = warp - 2;
    const int qd = warp & 3;
    const int k = ew >> 2;  // this group's token
    Half hf;
    hf.bar = 1 + k;
    hf.wq = qd;
    hf.lane = lane;
    hf.tid = qd * 32 + lane;
    hf.wcnt = reinterpret_cast<int*>(misc + M_WCNT) + k * 8;
    hf.hist = reinterpret_cast<int*>(misc + M_HIST) + k * 256;
    hf.sel = reinterpret_cast<int*>(misc + M_SEL) + k * 4;
    float* cs = reinterpret_cast<float*>(smem + OFF_CAND + k * CAP * 8);
    int* ci = reinterpret_cast<int*>(smem + OFF_CAND + k * CAP * 8 + CAP * 4);
    int win_lo = 1, win_hi = 0;  // empty window for an inactive token
    if (k < nt) window(t0 + k, win_lo, win_hi);
    const float* wr = s_w + k * kHeads;
    int cnt = 0;
    uint32_t thr = 0u;
    int parity = 0;
    bool aborted = false;
    for (int i = 0; i < ntiles; ++i) {
      const int b = i & 1;
      const bool got = mbar_wait(bar_df + 8 * b, (i >> 1) & 1, s_abort, err, wait_limit);
      if (named_bar_or(hf.bar, 128, !got)) { aborted = true; break; }
      tc_fence_after();
      uint32_t v[64];
      const uint32_t col = b * kN + k * kHeads;
      tmem_ld32(tmem_addr(tmem + col, qd * 32, 0), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(tmem_addr(tmem + col + 32, qd * 32, 0), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_de + 8 * b);
      const int tile0 = (kt0 + i) * kTile;
      if (tile0 > win_hi || tile0 + kTile <= win_lo) continue;  // whole tile outside this token's window (uniform)
      const int key = tile0 + hf.tid;
      // sum_h w_h * ReLU(s_h) with packed fp32 pairs: two running sums (even / odd heads)
      uint64_t acc2 = 0;
      const float4* wr4 = reinterpret_cast<const float4*>(wr);
#pragma unroll
      for (int h4 = 0; h4 < kHeads / 4; ++h4) {
        const float4 wv = wr4[h4];
        const uint64_t w01 = pack_f32x2(wv.x, wv.y), w23 = pack_f32x2(wv.z, wv.w);
        const uint64_t r01 = pack_f32x2(fmaxf(__uint_as_float(v[4 * h4]), 0.f), fmaxf(__uint_as_float(v[4 * h4 + 1]), 0.f));
        const uint64_t r23 =
            pack_f32x2(fmaxf(__uint_as_float(v[4 * h4 + 2]), 0.f), fmaxf(__uint_as_float(v[4 * h4 + 3]), 0.f));
        acc2 = fma_f32x2(w01, r01, acc2);
        acc2 = fma_f32x2(w23, r23, acc2);
      }
      const float sc = __uint_as_float((uint32_t)acc2) + __uint_as_float((uint32_t)(acc2 >> 32));
      const bool in = key >= win_lo && key <= win_hi;
      if (kScores && in) {
        const int rr = t0 + k - score_row0;
        if (rr >= 0 && rr < score_rows) scores[(size_t)rr * Tk + key] = sc;
      }
      const bool acc = in && ordered(sc) > thr;
      const int2 pos = half_scan(hf, acc, parity);
      parity ^= 1;
      if (acc) {
        cs[cnt + pos.x] = sc;
        ci[cnt + pos.x] = key;
      }
      cnt += pos.y;
      if (cnt > CAP - kTile) {
        named_bar(hf.bar, 128);
        int kept = 0;
        thr = compact(hf, cs, ci, cnt, K, parity, 2, &kept);
        if (kept > CAP - 2 * kTile) thr = compact(hf, cs, ci, kept, K, parity, 4, &kept);  // a crowded bucket
        cnt = kept;
      }
    }
    // ---- final selection and output (ascending, -1 suffix) ----
    if (!aborted) named_bar(hf.bar, 128);
    if (k < nt) {
      const int t = t0 + k;
      const int c = win_hi - win_lo + 1;
      const int n = min(K, c);
      if (!aborted && cnt > n) {
        int kept = 0;
        compact(hf, cs, ci, cnt, n, parity, 4, &kept);
        cnt = n;
      }
      const int have = aborted ? 0 : min(cnt, n);
      int32_t* row = topk_idx + (size_t)t * K;
      for (int j = hf.tid; j < K; j += 128) row[j] = (j < have) ? ci[j] : -1;
      if (topk_score != nullptr) {  // the fp32 scores the selection ranked, slot for slot (-inf after the prefix)
        float* srow = topk_score + (size_t)t * K;
        for (int j = hf.tid; j < K; j += 128) srow[j] = (j < have) ? cs[j] : -INFINITY;
      }
      if (topk_len != nullptr && hf.tid == 0) topk_len[t] = have;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace idx
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_indexer_topk_workspace_size(int32_t T, int32_t K) {
  (void)T;
  (void)K;
  return kErrorWordBytes;
}

namespace dsa {
namespace idx {
template <bool kScores>
static dsa_status_t run(const char* who, const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx, const float* head_weights,
                        const int32_t* seq_start, const int32_t* causal_len, int32_t T, int32_t T_k, int32_t Hi,
                        int32_t Di, int32_t K,
                        int32_t* topk_idx, int32_t* topk_len, float* topk_score, float* scores, int32_t score_row0,
                        int32_t score_rows,
                        void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  if (T < 0 || T_k < 1) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: need T >= 0 and T_k >= 1", who);
  if (!causal_len && T_k < T) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: T_k (%d) must be >= T (%d)", who, T_k, T);
  if (Hi < 1 || Hi > kHeads) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Hi must be in [1, 64] (got %d)", who, Hi);
  if (Di != kDi) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Di must be 128 (got %d)", who, Di);
  if (K < 1 || K > kMaxK) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: K must be in [1, 2048] (got %d)", who, K);
  if (!k_idx) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: k_idx is NULL", who);
  if (T > 0 && (!q_idx || !head_weights || !seq_start || !topk_idx))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: null tensor pointer", who);
  if (!aligned16(k_idx) || (T > 0 && !aligned16(q_idx)))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: q_idx and k_idx must be 16-byte aligned", who);
  if (kScores && (score_rows < 0 || score_row0 < 0 || score_row0 + score_rows > T || (score_rows > 0 && !scores)))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: need 0 <= score_row0, score_row0 + score_rows <= T and scores", who);
  dsa_status_t st = check_workspace(workspace, workspace_bytes, dsa_indexer_topk_workspace_size(T, K), who);
  if (st != DSA_OK) return st;
  if ((st = check_device()) != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = clear_error_word(workspace, s)) != DSA_OK) return st;
  if (T == 0) return ok();
  CUtensorMap map;
  if ((st = make_map_2d_bf16(&map, k_idx, (uint64_t)T_k, (uint64_t)kDi, (uint64_t)kDi, 64, kTile)) != DSA_OK) return st;
  if ((st = configure_kernel_smem(reinterpret_cast<const void*>(indexer_topk_kernel<kScores>), TOTAL,
                                  "configuring indexer_topk_kernel")))
    return st;
  const int nblk = (T + kTokens - 1) / kTokens;
  indexer_topk_kernel<kScores><<<nblk, kThreads, TOTAL, s>>>(
      map, reinterpret_cast<const __nv_bfloat16*>(q_idx), head_weights, seq_start, causal_len, T, T_k, Hi, K, topk_idx,
      topk_len, topk_score, reinterpret_cast<int*>(workspace), scores, score_row0, score_rows, wait_limit_cycles());
  if ((st = cuda_check(cudaGetLastError(), "launching indexer_topk_kernel"))) return st;
  return ok();
}
}  // namespace idx
}  // namespace dsa

extern "C" dsa_status_t dsa_indexer_topk(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx, const float* head_weights,
                                         const int32_t* seq_start, int32_t T, int32_t T_k, int32_t Hi, int32_t Di,
                                         int32_t K, int32_t* topk_idx, int32_t* topk_len, void* workspace,
                                         size_t workspace_bytes, dsa_stream_t stream) {
  return idx::run<false>("dsa_indexer_topk", q_idx, k_idx, head_weights, seq_start, nullptr, T, T_k, Hi, Di, K,
                         topk_idx, topk_len, nullptr, nullptr, 0, 0, workspace, workspace_bytes, stream);
}

extern "C" dsa_status_t dsa_indexer_topk_scored(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx,
                                                const float* head_weights, const int32_t* seq_start,
                                                const int32_t* causal_len, int32_t T, int32_t T_k, int32_t Hi,
                                                int32_t Di, int32_t K, int32_t* topk_idx, int32_t* topk_len,
                                                float* topk_score, void* workspace, size_t workspace_bytes,
                                                dsa_stream_t stream) {
  if (T > 0 && !topk_score) return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_indexer_topk_scored: topk_score is NULL");
  return idx::run<false>("dsa_indexer_topk_scored", q_idx, k_idx, head_weights, seq_start, causal_len, T, T_k, Hi,
                         Di, K, topk_idx, topk_len, topk_score, nullptr, 0, 0, workspace, workspace_bytes, stream);
}

extern "C" dsa_status_t dsa_indexer_topk_cp(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx, const float* head_weights,
                                            const int32_t* seq_start, const int32_t* causal_len, int32_t T_q,
                                            int32_t T_k, int32_t Hi, int32_t Di, int32_t K, int32_t* topk_idx,
                                            int32_t* topk_len, void* workspace, size_t workspace_bytes,
                                            dsa_stream_t stream) {
  if (T_q > 0 && !causal_len) return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_indexer_topk_cp: causal_len is NULL");
  return idx::run<false>("dsa_indexer_topk_cp", q_idx, k_idx, head_weights, seq_start, causal_len, T_q, T_k, Hi, Di,
                         K, topk_idx, topk_len, nullptr, nullptr, 0, 0, workspace, workspace_bytes, stream);
}

extern "C" dsa_status_t dsa_indexer_topk_with_scores(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx,
                                                     const float* head_weights, const int32_t* seq_start, int32_t T,
                                                     int32_t T_k, int32_t Hi, int32_t Di, int32_t K, int32_t* topk_idx,
                                                     int32_t* topk_len, float* scores, int32_t score_row0,
                                                     int32_t score_rows, void* workspace, size_t workspace_bytes,
                                                     dsa_stream_t stream) {
  return idx::run<true>("dsa_indexer_topk_with_scores", q_idx, k_idx, head_weights, seq_start, nullptr, T, T_k, Hi, Di,
                        K, topk_idx, topk_len, nullptr, scores, score_row0, score_rows, workspace, workspace_bytes, stream);
}
