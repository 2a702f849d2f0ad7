// dsa_indexer_kl.cu -- the indexer's KL auxiliary loss over the selected slots
// and its gradient, on sm_103a (tcgen05 + TMEM).
//
// For one query row t over its valid selected slots J (reading of the pages:
// "Accelerating GLM-5.2 Long-Context Training with cuDNN Fused DSA Kernels
// ...", "How DSA works" -- the indexer emits an auxiliary KL loss aligning its
// score distribution with the main attention's, its graph independent of the
// main model's -- and the training-results section -- sparse formulation,
// coefficient 0.001):
//   I_j = sum_h w[t,h] max(0, s_hj),  s_hj = <q_idx[t,h,:], k_idx[idx_j,:]>
//   q_j = softmax_J(I),  p_j = prob[t,j] / sum_J prob   (prob: the attention's
//         head-averaged slot probability, a constant)
//   kl[t] = sum_{j: p_j > 0} p_j (log p_j - log q_j)
// and with g_j = coeff (q_j - p_j) and m_hj = g_j w[t,h] [s_hj > 0]:
//   dw[t,h] = sum_j g_j max(0, s_hj),   dq_idx[t,h,:] = sum_j m_hj k_idx[idx_j,:],
//   dk_idx[idx_j,:] += sum_h m_hj q_idx[t,h,:].
//
// Design (sm_103a): one CTA per query row; 4 worker warps (one TMEM lane
// quadrant each, one slot row per thread), an MMA warp and, in the second
// pass, 4 drain warps.  The selected k_idx rows of a 128-slot tile are
// gathered by cp.async into 128-byte-swizzled shared memory (16 lanes per
// 256-byte row), two tiles deep.  Pass 1: S[slot, head] = K_tile . Q^T
// (M = 128 slots, N = 64 heads) in TMEM, the head-weighted ReLU sum per slot
// and the slot's probability into shared memory; then the row's softmax, KL
// and p normalisation.  Pass 2 gathers and multiplies again and writes
// m'_hj = g_j [s_hj > 0] (bf16 hi + lo parts: two values selected by the ReLU
// mask), with which
//   U^T[dim, head] += K_tile^T . M'   (in TMEM over the tiles), and
//   dK[slot, dim] = M' . Q',  Q' = w_h q_idx[h,:] (bf16 hi + lo, made once),
// and at the end dq_h = w_h U_h and dw_h = <q_h, U_h> (the same sums as
// above, regrouped; the gradients carry about fp32 accuracy).  dK has two
// TMEM buffers: the drain warps reduce one into the fp32 dk_idx accumulator
// (red.global.add.v4.f32, 4 rows x 128 bytes per instruction after a
// transpose through shared memory) while the workers build the next tile's
// M'.  The roles hand over through mbarriers.  A tile's rows are gathered a
// tile ahead, so the workers signal its landing first and issue the next
// tile's gather while S of this one is formed.
//
// When the selection's own scores are given (the indexer keeps each
// candidate's fp32 score), indexer_kl_rows_kernel reads them instead of the
// first pass, with one CTA per SM walking the rows (see there).
#include <cmath>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {
namespace kl {

constexpr int kWorkers = 128;             // warps 0-3
constexpr int kPass1 = kWorkers + 32;     // + the MMA warp (warp 4): the threads of the first pass
constexpr int kThreads = kPass1 + 128;    // + the dK drain warps (warps 5-8)
constexpr int kHeads = 64;                // indexer heads (padded)
constexpr int kDi = 128;                  // indexer head dim
constexpr int kTile = 128;                // slots per tile (MMA M)
constexpr int kMaxK = 4096;

constexpr int Q_CHUNK = kHeads * 128;     // 8 KiB: 64 heads x 64 dims
constexpr int K_CHUNK = kTile * 128;      // 16 KiB: 128 slots x 64 dims
constexpr int K_BUF = 2 * K_CHUNK;        // one gathered tile
constexpr int OFF_Q = 0;
constexpr int OFF_QW = OFF_Q + 2 * Q_CHUNK;         // w_h q_idx[h,:] as bf16 hi (2 chunks), then lo (2 chunks)
constexpr int OFF_K = OFF_QW + 4 * Q_CHUNK;         // two tile buffers
constexpr int OFF_MHI = OFF_K + 2 * K_BUF;
constexpr int OFF_MLO = OFF_MHI + kTile * 128;
constexpr int OFF_FST = OFF_MLO + kTile * 128;      // [4 drain warps][16 rows x 128 B]: dK transposes
constexpr int OFF_I = OFF_FST + 4 * 2048;           // float [kMaxK]: indexer scores (-inf: invalid slot)
constexpr int OFF_P = OFF_I + kMaxK * 4;            // float [kMaxK]: attention slot probabilities
constexpr int OFF_MISC = OFF_P + kMaxK * 4;
constexpr int M_BAR_S = 0, M_BAR_MM = 8, M_BAR_FIN = 16, M_TMEM = 32, M_NEFF = 36, M_ABORT = 40, M_ACTIVE = 44;
// second pass: tile landed, S read, M written, dK buffer b read (two), products into dK buffer b done (two;
// the drain warps wait on these, so that a phase of the buffer they drain cannot be overtaken)
constexpr int M_BAR_LAND = 600, M_BAR_SFREE = 608, M_BAR_M = 616, M_BAR_DKF = 624, M_BAR_MMD = 640;
constexpr int M_STATS = 48;                         // float [3]: logZ, 1/psum, (spare)
constexpr int M_W = 64;                             // float [64]
constexpr int M_DW = M_W + 256;                     // float [64]
constexpr int M_RED = M_DW + 256;                   // float [4]
constexpr int M_KEY = 1024;                         // int [2][128]: the keys of the next two tiles
constexpr int MISC = 2048;
constexpr int TOTAL = OFF_MISC + MISC + 1024;       // + alignment slack
static_assert(TOTAL <= 232448, "shared memory budget");
static_assert(M_RED + 16 <= M_BAR_LAND && M_BAR_MMD + 16 <= M_KEY && M_KEY + 2 * kTile * 4 <= MISC, "misc layout");

// Reduction over the 128 worker threads (named barrier 2); every worker gets the result.
template <bool MAX>
__device__ __forceinline__ float worker_reduce(float v, float* red, int warp, int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const float x = __shfl_xor_sync(0xffffffffu, v, o);
    v = MAX ? fmaxf(v, x) : v + x;
  }
  if (lane == 0) red[warp] = v;
  named_bar(2, kWorkers);
  const float r = MAX ? fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3])) : (red[0] + red[1]) + (red[2] + red[3]);
  named_bar(2, kWorkers);  // red is reused by the next reduction
  return r;
}

// Transposing butterfly: v[0..31] per lane (lane = slot row, index = head) -> lane l returns the sum
// over the warp's 32 rows of head l.
__device__ __forceinline__ float warp_transpose_sum(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      const float send = upper ? v[i] : v[i + o];
      const float keep = upper ? v[i + o] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
  return v[0];
}

__global__ void __launch_bounds__(kThreads, 1)
    indexer_kl_kernel(const __nv_bfloat16* __restrict__ k_idx, const __nv_bfloat16* __restrict__ q_idx,
                      const float* __restrict__ w, const int32_t* __restrict__ topk_idx,
                      const int32_t* __restrict__ topk_len, const float* __restrict__ prob, int Tk, int Hi, int K,
                      float coeff, float* __restrict__ kl_out, __nv_bfloat16* __restrict__ dq_out,
                      float* __restrict__ dw_out, float* __restrict__ dk, int* __restrict__ err,
                      long long wait_limit) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + OFF_Q), sK = smem_u32(smem + OFF_K);
  const uint32_t sMhi = smem_u32(smem + OFF_MHI), sMlo = smem_u32(smem + OFF_MLO);
  float* s_I = reinterpret_cast<float*>(smem + OFF_I);
  float* s_P = reinterpret_cast<float*>(smem + OFF_P);
  uint8_t* misc = smem + OFF_MISC;
  const uint32_t bar_s = smem_u32(misc + M_BAR_S), bar_mm = smem_u32(misc + M_BAR_MM);
  const uint32_t bar_fin = smem_u32(misc + M_BAR_FIN);
  const uint32_t bar_land = smem_u32(misc + M_BAR_LAND), bar_sfree = smem_u32(misc + M_BAR_SFREE);
  const uint32_t bar_m = smem_u32(misc + M_BAR_M), bar_dkf = smem_u32(misc + M_BAR_DKF);
  const uint32_t bar_mmd = smem_u32(misc + M_BAR_MMD);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + M_TMEM);
  int* s_neff = reinterpret_cast<int*>(misc + M_NEFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + M_ABORT);
  int* s_active = reinterpret_cast<int*>(misc + M_ACTIVE);
  float* s_stats = reinterpret_cast<float*>(misc + M_STATS);
  float* s_w = reinterpret_cast<float*>(misc + M_W);
  float* s_dw = reinterpret_cast<float*>(misc + M_DW);
  float* s_red = reinterpret_cast<float*>(misc + M_RED);
  int* s_key = reinterpret_cast<int*>(misc + M_KEY);

  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;  // workers: 0..127, slot row / dim of this thread
  const bool worker = warp < 4;
  const int32_t* idx_row = topk_idx + (size_t)t * K;

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_mm, 1);
    mbar_init(bar_fin, 1);
    mbar_init(bar_land, kWorkers / 32);
    mbar_init(bar_sfree, kWorkers / 32);
    mbar_init(bar_m, kWorkers / 32);
    mbar_init(bar_dkf, 4);
    mbar_init(bar_dkf + 8, 4);
    mbar_init(bar_mmd, 1);
    mbar_init(bar_mmd + 8, 1);
    *s_neff = 0;
    *s_abort = 0;
    *s_active = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  __syncthreads();  // the counters are initialised before any worker adds to them
  if (worker) {
    if (topk_len != nullptr) {
      if (tid == 0) {
        const int n = topk_len[t];
        *s_neff = n < 0 ? 0 : (n > K ? K : n);
      }
    } else {
      int last = 0;
      for (int j = tid; j < K; j += kWorkers)
        if (idx_row[j] >= 0) last = j + 1;
      if (last) atomicMax(s_neff, last);
    }
    // q_idx [64 heads x 128] -> 2 chunks of [64 rows x 128 B], 128B swizzle; padded heads are zero
    const uint64_t pol = l2_evict_first_policy();
    for (int u = tid; u < kHeads * 16; u += kWorkers) {
      const int hh = u >> 4, c = (u >> 3) & 1, uc = u & 7;
      const bool ok = hh < Hi;
      cp_async16_hint(sQ + c * Q_CHUNK + sw128_off(hh, uc),
                      q_idx + (ok ? ((size_t)t * Hi + hh) * kDi + c * 64 + uc * 8 : 0), ok ? 16u : 0u, pol);
    }
    if (tid < kHeads) {
      s_w[tid] = (tid < Hi) ? __ldg(w + (size_t)t * Hi + tid) : 0.f;
      s_dw[tid] = 0.f;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    fence_proxy_async_smem();
  }
  __syncthreads();
  const int n_eff = *s_neff;
  const int ntiles = (n_eff + kTile - 1) / kTile;
  const uint32_t tmem = *s_tmem;
  const uint32_t tS = tmem, tDQ = tmem + 64, tDK = tmem + 128;  // dK: two buffers of 128 columns
  const uint32_t sQW = smem_u32(smem + OFF_QW);
  if (worker) {
    // Q' = w_h q_idx[h,:] as bf16 hi + lo in Q's layout: the B operand of dK = M'.Q' (M' = g [s > 0])
#pragma unroll
    for (int k = 0; k < kHeads * 16 / kWorkers; ++k) {
      const int u = tid + kWorkers * k;  // 16-byte unit: head u >> 4, chunk (u >> 3) & 1, unit u & 7
      const int hh = u >> 4;
      const uint32_t off = ((u >> 3) & 1) * Q_CHUNK + sw128_off(hh, u & 7);
      const uint4 qv = *reinterpret_cast<const uint4*>(smem + OFF_Q + off);
      const float wh = s_w[hh];
      const uint32_t* qe = reinterpret_cast<const uint32_t*>(&qv);
      uint32_t hv[4], lv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qe[e]));
        const float a = wh * qf.x, b = wh * qf.y;
        const __nv_bfloat162 hi = __floats2bfloat162_rn(a, b);
        const float2 hf = __bfloat1622float2(hi);
        hv[e] = *reinterpret_cast<const uint32_t*>(&hi);
        lv[e] = pack_bf16x2(a - hf.x, b - hf.y);
      }
      st_shared_v4(sQW + off, hv[0], hv[1], hv[2], hv[3]);
      st_shared_v4(sQW + 2 * Q_CHUNK + off, lv[0], lv[1], lv[2], lv[3]);
    }
    fence_proxy_async_smem();  // Q' -> visible to the tensor core (first used in the second pass)
  }

  // index of slot j (-1: invalid or beyond the prefix; out-of-range values are reported and masked)
  // A slot's key in two steps: the load (issued a tile ahead of its gather, so that its memory
  // latency hides behind the tile before) and the check (-1: none; bad indices are flagged).
  auto raw_key = [&](int i) -> int {
    const int j = i * kTile + tid;
    return (j < n_eff) ? __ldg(idx_row + j) : -1;
  };
  auto check_key = [&](int raw) -> int {
    if (raw < -1 || raw >= Tk) record_error(err, DSA_ERR_DEVICE_INDEX);
    return (raw >= 0 && raw < Tk) ? raw : -1;
  };
  // Issue the gather of tile i's k_idx rows into buffer i & 1 as one cp.async group: 16 lanes per
  // 256-byte row, so that each instruction covers two contiguous rows; the rows' keys come from the
  // table s_key[i & 1] (written a tile ahead by the thread that owns each row; -1 zero-fills).
  auto gather_rows = [&](int i) {
    const int* keys = s_key + (i & 1) * kTile;
    const uint32_t dst = sK + (uint32_t)(i & 1) * K_BUF;
    const int u = tid & 15;
#pragma unroll
    for (int e = 0; e < kTile / 8; ++e) {
      const int row = (tid >> 4) + 8 * e;
      const int ix = keys[row];
      cp_async16(dst + (u >> 3) * K_CHUNK + sw128_off(row, u & 7), k_idx + (ix >= 0 ? (size_t)ix * kDi : 0) + u * 8,
                 ix >= 0 ? 16u : 0u);
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
  };
  // This thread's keys of tiles i and i + 1 (its own row), the raw index of tile i + 2, and the table
  // entries: the keys of tiles 0 and 1 before the first gather, then that of tile i + 2 at the end of
  // tile i (gather i + 2 follows the tile's last barrier; the table half it reuses was read by gather i).
  int ixa = -1, ixb = -1, rawc = -1;
  auto start_pass = [&]() {
    ixa = check_key(raw_key(0));
    s_key[tid] = ixa;
    ixb = (ntiles > 1) ? check_key(raw_key(1)) : -1;
    s_key[kTile + tid] = ixb;
    rawc = (ntiles > 2) ? raw_key(2) : -1;
    named_bar(2, kWorkers);
    gather_rows(0);
  };
  auto end_tile = [&](int i) {
    const int kc = (i + 2 < ntiles) ? check_key(rawc) : -1;
    if (i + 2 < ntiles) s_key[((i + 2) & 1) * kTile + tid] = kc;
    ixa = ixb;
    ixb = kc;
    rawc = (i + 3 < ntiles) ? raw_key(i + 3) : -1;
  };
  // tile i (its group, and not the one issued after it) has landed and is visible to the tensor core
  auto landed = [&](bool one_more_in_flight) {
    if (one_more_in_flight)
      asm volatile("cp.async.wait_group 1;" ::: "memory");
    else
      asm volatile("cp.async.wait_group 0;" ::: "memory");
    fence_proxy_async_smem();
  };
  constexpr uint32_t kIdS = idesc_bf16(kTile, kHeads, false, false);   // S = K_tile . Q^T
  constexpr uint32_t kIdDQ = idesc_bf16(kDi, kHeads, true, true);      // dQ^T += K_tile^T . M
  constexpr uint32_t kIdDK = idesc_bf16(kTile, kDi, false, true);      // dK = M . Q
  auto issue_s = [&](int i) {
    tc_fence_after();
    const uint32_t kb = sK + (uint32_t)(i & 1) * K_BUF;
#pragma unroll
    for (int c = 0; c < 2; ++c)
#pragma unroll
      for (int k = 0; k < 4; ++k)  // + 16 dims = + 32 bytes per row
        mma_ss_w(tS, sdesc_sw128(kb + c * K_CHUNK, 16, 1024) + (uint64_t)(k * 2),
                 sdesc_sw128(sQ + c * Q_CHUNK, 16, 1024) + (uint64_t)(k * 2), kIdS, (c | k) != 0);
    mma_commit_w(bar_s);
  };

  bool aborted = false;
  uint32_t ph_s = 0;  // phase parity of bar_s, which counts the S products of both passes
  // ---- pass 1: indexer scores of the selected slots, and their attention probabilities ----
  // (each worker loads its slot's probability a tile ahead, stores it for the second pass and keeps
  // running partials of the row's score maximum and probability sum)
  float imax_part = -INFINITY, psum_part = 0.f;
  auto prob_of = [&](int i) -> float {
    const int j = i * kTile + tid;
    return (j < n_eff) ? __ldg(prob + (size_t)t * K + j) : 0.f;
  };
  float p_next = (worker && ntiles > 0) ? prob_of(0) : 0.f;
  if (worker && ntiles > 0) start_pass();
  for (int i = 0; warp <= 4 && i < ntiles; ++i) {  // workers and the MMA warp; the drain warps wait below
    const int ix = ixa;
    if (worker) landed(false);  // tile i, gathered a tile ago (the only copies in flight)
    if (named_bar_or(1, kPass1, false)) { aborted = true; break; }  // the tile has landed
    if (warp == 4) issue_s(i);  // the whole warp, one elected lane issues
    bool ok = true;
    if (worker) {
      // the next tile's rows while S of this one is formed: buffer (i + 1) & 1 was last read by the S
      // product of tile i - 1, which was read before the end-of-tile barrier of tile i - 1
      if (i + 1 < ntiles) gather_rows(i + 1);
      ok = mbar_wait(bar_s, ph_s, s_abort, err, wait_limit);
      if (ok) {
        tc_fence_after();
        uint32_t v[64];
        tmem_ld32(tmem_addr(tS, warp * 32, 0), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tmem_addr(tS, warp * 32, 32), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        float score = 0.f;
#pragma unroll
        for (int h = 0; h < kHeads; ++h) score = fmaf(s_w[h], fmaxf(__uint_as_float(v[h]), 0.f), score);
        const int j = i * kTile + tid;
        if (j < n_eff) {
          const float sc = (ix >= 0) ? score : -INFINITY;
          const float p = (ix >= 0) ? p_next : 0.f;
          s_I[j] = sc;
          s_P[j] = p;
          imax_part = fmaxf(imax_part, sc);
          psum_part += p;
        }
      }
      tc_fence_before();
      end_tile(i);
      p_next = (i + 1 < ntiles) ? prob_of(i + 1) : 0.f;
    }
    ph_s ^= 1;
    if (named_bar_or(1, kPass1, !ok)) { aborted = true; break; }  // S is read: TMEM and the tile are free
  }

  // ---- the row's distributions and its KL value (workers) ----
  if (worker && !aborted) {
    const float imax = worker_reduce<true>(imax_part, s_red, warp, lane);
    const float psum = worker_reduce<false>(psum_part, s_red, warp, lane);
    const bool active = imax > -INFINITY && psum > 0.f;
    float klv = 0.f;
    if (active) {
      float z = 0.f;
      for (int j = tid; j < n_eff; j += kWorkers) z += (s_I[j] > -INFINITY) ? expf(s_I[j] - imax) : 0.f;
      z = worker_reduce<false>(z, s_red, warp, lane);
      const float logz = imax + logf(z), inv_psum = 1.f / psum;
      float acc = 0.f;
      for (int j = tid; j < n_eff; j += kWorkers) {
        const float p = s_P[j] * inv_psum;
        if (s_I[j] > -INFINITY && p > 0.f) acc += p * (logf(p) - (s_I[j] - logz));
      }
      klv = worker_reduce<false>(acc, s_red, warp, lane);
      if (tid == 0) {
        s_stats[0] = logz;
        s_stats[1] = inv_psum;
      }
    }
    if (tid == 0) {
      kl_out[t] = klv;
      *s_active = active ? 1 : 0;
    }
  }
  __syncthreads();  // the statistics are in shared memory for every role, the drain warps included
  const bool active = !aborted && *s_active != 0;
  const float logz = s_stats[0], inv_psum = s_stats[1];

  // ---- pass 2: the gradient, three roles ----
  // workers: gather, S read, m_hj and dw; MMA warp: S, then dQ^T += K_tile^T.M and dK = M.Q into one of
  // two dK buffers; drain warps: dK of the previous product into dk_idx while the workers go on.
  if (worker && active) {
    bool bad = false;  // a wait of this thread gave up (made uniform by the next workers' barrier)
    if (ntiles > 0) start_pass();
    for (int i = 0; i < ntiles; ++i) {
      const int ix = ixa;
      const bool more = i + 1 < ntiles;
      // tile i (gathered a tile ago, the only copies in flight) has landed: S of it may be formed
      // right after the products of tile i - 1, while this warp issues the next gather
      landed(false);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_land);
      // the products of tile i - 1 are done: K buffer (i + 1) & 1 and the M tiles are free
      if (i >= 1 && !bad) bad = !mbar_wait(bar_mm, (i - 1) & 1, s_abort, err, wait_limit);
      // every worker's key table entry for tile i + 1 is written (end of tile i - 1)
      if (named_bar_or(2, kWorkers, bad)) { aborted = true; break; }
      if (more) gather_rows(i + 1);
      const bool ok = mbar_wait(bar_s, ph_s ^ (uint32_t)(i & 1), s_abort, err, wait_limit);
      if (ok) {
        tc_fence_after();
        uint32_t v[64];
        tmem_ld32(tmem_addr(tS, warp * 32, 0), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tmem_addr(tS, warp * 32, 32), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_sfree);  // S is read: the next tile's S may be formed
        const int j = i * kTile + tid;
        float g = 0.f;
        if (j < n_eff && ix >= 0) g = coeff * (expf(s_I[j] - logz) - s_P[j] * inv_psum);
        // m'_h = g [s_h > 0] as bf16 hi + lo, row tid of the two M tiles: two values selected per head by
        // the ReLU mask (w_h enters through Q' for dK and at the end for dq; dw = <q_h, U_h> at the end)
        const __nv_bfloat16 ghi = __float2bfloat16_rn(g);
        const uint32_t gh = __bfloat16_as_ushort(ghi);
        const uint32_t gl = __bfloat16_as_ushort(__float2bfloat16_rn(g - __bfloat162float(ghi)));
        uint32_t mh[32], ml[32];
#pragma unroll
        for (int h = 0; h < kHeads; h += 2) {
          const bool p0 = __uint_as_float(v[h]) > 0.f, p1 = __uint_as_float(v[h + 1]) > 0.f;
          mh[h >> 1] = (p0 ? gh : 0u) | ((p1 ? gh : 0u) << 16);
          ml[h >> 1] = (p0 ? gl : 0u) | ((p1 ? gl : 0u) << 16);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          st_shared_v4(sMhi + sw128_off(tid, u), mh[4 * u], mh[4 * u + 1], mh[4 * u + 2], mh[4 * u + 3]);
          st_shared_v4(sMlo + sw128_off(tid, u), ml[4 * u], ml[4 * u + 1], ml[4 * u + 2], ml[4 * u + 3]);
        }
        fence_proxy_async_smem();  // M' -> visible to the tensor core
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_m);
      end_tile(i);
      bad |= !ok;
    }
    // the last tile's products are done before dQ^T is read
    if (!aborted && !bad && ntiles > 0) bad = !mbar_wait(bar_mm, (ntiles - 1) & 1, s_abort, err, wait_limit);
    aborted = named_bar_or(2, kWorkers, aborted || bad);
  } else if (warp == 4 && active) {
    for (int i = 0; i < ntiles; ++i) {
      if (!warp_all(mbar_wait(bar_land, i & 1, s_abort, err, wait_limit))) { aborted = true; break; }
      if (i >= 1 && !warp_all(mbar_wait(bar_sfree, (i - 1) & 1, s_abort, err, wait_limit))) { aborted = true; break; }
      issue_s(i);
      if (!warp_all(mbar_wait(bar_m, i & 1, s_abort, err, wait_limit))) { aborted = true; break; }
      // dK buffer i & 1 was read by the drain of tile i - 2
      if (i >= 2 && !warp_all(mbar_wait(bar_dkf + 8 * (i & 1), ((i - 2) >> 1) & 1, s_abort, err, wait_limit))) {
        aborted = true;
        break;
      }
      tc_fence_after();
      const uint32_t tdk = tDK + 128 * (uint32_t)(i & 1);
      const uint64_t ka = sdesc_sw128(sK + (uint32_t)(i & 1) * K_BUF, K_CHUNK, 1024);
      const uint64_t mb_hi = sdesc_sw128(sMhi, K_CHUNK, 1024);
      const uint64_t mb_lo = sdesc_sw128(sMlo, K_CHUNK, 1024);
#pragma unroll
      for (int k = 0; k < kTile / 16; ++k) {  // + 16 slots = + 2048 bytes
        mma_ss_w(tDQ, ka + (uint64_t)(k * 128), mb_hi + (uint64_t)(k * 128), kIdDQ, (i > 0 || k > 0) ? 1u : 0u);
        mma_ss_w(tDQ, ka + (uint64_t)(k * 128), mb_lo + (uint64_t)(k * 128), kIdDQ, 1u);
      }
      const uint64_t ma_hi = sdesc_sw128(sMhi, 16, 1024), ma_lo = sdesc_sw128(sMlo, 16, 1024);
      const uint64_t qwh = sdesc_sw128(sQW, Q_CHUNK, 1024), qwl = sdesc_sw128(sQW + 2 * Q_CHUNK, Q_CHUNK, 1024);
#pragma unroll
      for (int k = 0; k < kHeads / 16; ++k) {  // + 16 heads: + 32 bytes along A's rows, + 16 rows of Q'
        // dK = M'_hi Q'_hi + M'_hi Q'_lo + M'_lo Q'_hi (the lo x lo term is below fp32 rounding)
        mma_ss_w(tdk, ma_hi + (uint64_t)(k * 2), qwh + (uint64_t)(k * 128), kIdDK, k > 0 ? 1u : 0u);
        mma_ss_w(tdk, ma_hi + (uint64_t)(k * 2), qwl + (uint64_t)(k * 128), kIdDK, 1u);
        mma_ss_w(tdk, ma_lo + (uint64_t)(k * 2), qwh + (uint64_t)(k * 128), kIdDK, 1u);
      }
      mma_commit_w(bar_mm);
      mma_commit_w(bar_mmd + 8 * (i & 1));
    }
  } else if (warp >= 5 && active) {
    // ======================= dK drain: rows into dk_idx by L2 reductions =======================
    // 32 rows x 32 dims at a time per warp, transposed through the warp's 2 KiB buffer 16 rows at a
    // time, so that each red.global.add.v4.f32 covers 4 rows x 128 bytes
    const int qd = warp & 3;       // TMEM lane quadrant of this warp
    const int r = qd * 32 + lane;  // slot row of the tile
    const uint32_t fst = smem_u32(smem + OFF_FST + (warp - 5) * 2048);
    auto key_of = [&](int i) -> int {  // the row's key (the workers report bad indices)
      const int j = i * kTile + r;
      const int raw = (j < n_eff) ? __ldg(idx_row + j) : -1;
      return (raw >= 0 && raw < Tk) ? raw : -1;
    };
    int key_next = (ntiles > 0) ? key_of(0) : -1;
    for (int i = 0; i < ntiles; ++i) {
      const int key = key_next;
      if (i + 1 < ntiles) key_next = key_of(i + 1);
      if (!mbar_wait(bar_mmd + 8 * (i & 1), (i >> 1) & 1, s_abort, err, wait_limit)) { aborted = true; break; }
      tc_fence_after();
      const uint32_t tdk = tDK + 128 * (uint32_t)(i & 1);
#pragma unroll 1
      for (int b = 0; b < kDi / 32; ++b) {
        uint32_t v[32];
        tmem_ld32(tmem_addr(tdk, qd * 32, 32 * b), v);
        tmem_ld_wait();
        if (b == kDi / 32 - 1) {  // the last load of the buffer: it may be refilled
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_dkf + 8 * (i & 1));
        }
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if ((lane >> 4) == hh) {
            const int rl = lane & 15;
#pragma unroll
            for (int u = 0; u < 8; ++u)
              st_shared_v4(fst + rl * 128 + ((u ^ (rl & 7)) << 4), v[4 * u], v[4 * u + 1], v[4 * u + 2], v[4 * u + 3]);
          }
          __syncwarp();
#pragma unroll
          for (int st = 0; st < 4; ++st) {
            const int rl = 4 * st + (lane >> 3), u = lane & 7;
            const int kr = __shfl_sync(0xffffffffu, key, 16 * hh + rl);
            float4 f;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                         : "r"(fst + rl * 128 + ((u ^ (rl & 7)) << 4))
                         : "memory");
            if (kr >= 0) red_add_v4(dk + (size_t)kr * kDi + 32 * b + 4 * u, f.x, f.y, f.z, f.w);
          }
          __syncwarp();
        }
      }
    }
  }

  // ---- dq_idx (dQ^T in TMEM: lane = dim, column = head) and dw ----
  if (worker) {
    const bool have = active && !aborted && ntiles > 0;
    uint32_t v[64];
    if (have) {
      tc_fence_after();
      tmem_ld32(tmem_addr(tDQ, warp * 32, 0), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
      tmem_ld32(tmem_addr(tDQ, warp * 32, 32), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
      tmem_ld_wait();
    } else {
#pragma unroll
      for (int h = 0; h < kHeads; ++h) v[h] = 0u;
    }
    // TMEM holds U^T (U_h = sum_j g_j [s_jh > 0] k_j): dq_h = w_h U_h, dw_h = <q_h, U_h>
    __nv_bfloat16* dq_row = dq_out + (size_t)t * Hi * kDi + tid;  // dim tid of every head
#pragma unroll 8
    for (int h = 0; h < kHeads; ++h)
      if (h < Hi) dq_row[(size_t)h * kDi] = __float2bfloat16_rn(s_w[h] * __uint_as_float(v[h]));
    const uint8_t* qcol = smem + OFF_Q + (tid >> 6) * Q_CHUNK + (tid & 7) * 2;  // q_idx[., tid]: chunk, lane in unit
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      float d[32];
#pragma unroll
      for (int hh = 0; hh < 32; ++hh) {
        const int h = 32 * half + hh;
        const __nv_bfloat16 qv = *reinterpret_cast<const __nv_bfloat16*>(qcol + sw128_off(h, (tid & 63) >> 3));
        d[hh] = __bfloat162float(qv) * __uint_as_float(v[h]);
      }
      atomicAdd(s_dw + 32 * half + lane, warp_transpose_sum(d, lane));
    }
    named_bar(2, kWorkers);
    if (tid < Hi) dw_out[(size_t)t * Hi + tid] = have ? s_dw[tid] : 0.f;
  }

  if (worker) asm volatile("cp.async.wait_all;" ::: "memory");  // no copy into shared memory outlives the CTA
  if (warp == 4) {
    // every MMA of this CTA completes before the teardown frees TMEM
    mma_commit_w(bar_fin);
    volatile int dummy = 0;
    mbar_wait(bar_fin, 0, &dummy, err);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// Rows kernel: the same loss and gradients when the selection's own scores are given (they are read,
// so there is no first pass).  The gradient pass is bound by the dk_idx reductions; one CTA per row
// would leave the SM without reductions while the row's q_idx, scores and statistics load and while
// its last dK tiles drain.  So one CTA per SM walks the rows blockIdx.x, blockIdx.x + gridDim.x, ...:
// the workers load and reduce the next row while the drain warps still reduce the previous row's last
// tiles.  Each row's tile count reaches the MMA and drain warps through a two-slot row table (bar_row:
// written; bar_rowfree: read by the MMA warp and the 4 drain warps), and every per-tile barrier phase
// follows a tile counter that runs on across rows.
// ---------------------------------------------------------------------------
constexpr int M_BAR_ROW = 656, M_BAR_ROWFREE = 672, M_ROWD = 688;  // row table: 2 x {n_eff, tiles}
static_assert(M_ROWD + 16 <= M_KEY, "misc layout");

__global__ void __launch_bounds__(kThreads, 1)
    indexer_kl_rows_kernel(const __nv_bfloat16* __restrict__ k_idx, const __nv_bfloat16* __restrict__ q_idx,
                           const float* __restrict__ w, const int32_t* __restrict__ topk_idx,
                           const int32_t* __restrict__ topk_len, const float* __restrict__ prob,
                           const float* __restrict__ topk_score, int T, int Tk, int Hi, int K, float coeff,
                           float* __restrict__ kl_out, __nv_bfloat16* __restrict__ dq_out,
                           float* __restrict__ dw_out, float* __restrict__ dk, int* __restrict__ err,
                           long long wait_limit) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + OFF_Q), sK = smem_u32(smem + OFF_K), sQW = smem_u32(smem + OFF_QW);
  const uint32_t sMhi = smem_u32(smem + OFF_MHI), sMlo = smem_u32(smem + OFF_MLO);
  float* s_I = reinterpret_cast<float*>(smem + OFF_I);
  float* s_P = reinterpret_cast<float*>(smem + OFF_P);
  uint8_t* misc = smem + OFF_MISC;
  const uint32_t bar_s = smem_u32(misc + M_BAR_S), bar_mm = smem_u32(misc + M_BAR_MM);
  const uint32_t bar_fin = smem_u32(misc + M_BAR_FIN);
  const uint32_t bar_land = smem_u32(misc + M_BAR_LAND), bar_sfree = smem_u32(misc + M_BAR_SFREE);
  const uint32_t bar_m = smem_u32(misc + M_BAR_M), bar_dkf = smem_u32(misc + M_BAR_DKF);
  const uint32_t bar_mmd = smem_u32(misc + M_BAR_MMD);
  const uint32_t bar_row = smem_u32(misc + M_BAR_ROW), bar_rowfree = smem_u32(misc + M_BAR_ROWFREE);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + M_TMEM);
  int* s_neff = reinterpret_cast<int*>(misc + M_NEFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + M_ABORT);
  float* s_w = reinterpret_cast<float*>(misc + M_W);
  float* s_dw = reinterpret_cast<float*>(misc + M_DW);
  float* s_red = reinterpret_cast<float*>(misc + M_RED);
  int* s_key = reinterpret_cast<int*>(misc + M_KEY);
  volatile int* s_rowd = reinterpret_cast<volatile int*>(misc + M_ROWD);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tid = threadIdx.x;  // workers: 0..127, slot row / dim of this thread
  const bool worker = warp < 4;

  if (tid == 0) {
    mbar_init(bar_s, 1);
    mbar_init(bar_mm, 1);
    mbar_init(bar_fin, 1);
    mbar_init(bar_land, kWorkers / 32);
    mbar_init(bar_sfree, kWorkers / 32);
    mbar_init(bar_m, kWorkers / 32);
    mbar_init(bar_dkf, 4);
    mbar_init(bar_dkf + 8, 4);
    mbar_init(bar_mmd, 1);
    mbar_init(bar_mmd + 8, 1);
    mbar_init(bar_row, 1);
    mbar_init(bar_row + 8, 1);
    mbar_init(bar_rowfree, 5);  // the MMA warp and the 4 drain warps
    mbar_init(bar_rowfree + 8, 5);
    *s_neff = 0;
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  __syncthreads();
  const uint32_t tmem = *s_tmem;
  const uint32_t tS = tmem, tDQ = tmem + 64, tDK = tmem + 128;  // dK: two buffers of 128 columns
  constexpr uint32_t kIdS = idesc_bf16(kTile, kHeads, false, false);   // S = K_tile . Q^T
  constexpr uint32_t kIdDQ = idesc_bf16(kDi, kHeads, true, true);      // dQ^T += K_tile^T . M
  constexpr uint32_t kIdDK = idesc_bf16(kTile, kDi, false, true);      // dK = M . Q
  bool aborted = false;

  if (worker) {
    uint32_t g0 = 0;  // tiles of this CTA before the current row
    int rr = 0;       // rows of this CTA before the current row
    // rows of topk_idx, topk_score and prob start on 16-byte boundaries: vector loads
    const bool vec4 = (K & 3) == 0 &&
                      ((reinterpret_cast<uintptr_t>(topk_idx) | reinterpret_cast<uintptr_t>(topk_score) |
                        reinterpret_cast<uintptr_t>(prob)) & 15) == 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, ++rr) {
      const int32_t* idx_row = topk_idx + (size_t)t * K;
      auto check_key = [&](int raw) -> int {
        if (raw < -1 || raw >= Tk) record_error(err, DSA_ERR_DEVICE_INDEX);
        return (raw >= 0 && raw < Tk) ? raw : -1;
      };
      int n_eff;
      if (topk_len != nullptr) {
        const int n = __ldg(topk_len + t);
        n_eff = n < 0 ? 0 : (n > K ? K : n);
      } else {
        if (tid == 0) *s_neff = 0;
        named_bar(2, kWorkers);
        int last = 0;
        for (int j = tid; j < K; j += kWorkers)
          if (__ldg(idx_row + j) >= 0) last = j + 1;
        if (last) atomicMax(s_neff, last);
        named_bar(2, kWorkers);
        n_eff = *s_neff;
      }
      const int ntiles = (n_eff + kTile - 1) / kTile;
      // q_idx of the row (the previous row's products and dw have finished with Q and Q'); its
      // scores and probabilities load meanwhile
      const uint64_t pol = l2_evict_first_policy();
      for (int u = tid; u < kHeads * 16; u += kWorkers) {
        const int hh = u >> 4, c = (u >> 3) & 1, uc = u & 7;
        const bool ok = hh < Hi;
        cp_async16_hint(sQ + c * Q_CHUNK + sw128_off(hh, uc),
                        q_idx + (ok ? ((size_t)t * Hi + hh) * kDi + c * 64 + uc * 8 : 0), ok ? 16u : 0u, pol);
      }
      if (tid < kHeads) {
        s_w[tid] = (tid < Hi) ? __ldg(w + (size_t)t * Hi + tid) : 0.f;
        s_dw[tid] = 0.f;
      }
      float imax_part = -INFINITY, psum_part = 0.f;
      {
        const float* srow = topk_score + (size_t)t * K;
        const float* prow = prob + (size_t)t * K;
        auto take = [&](int j, int raw, float sc, float p) {
          const int ix = check_key(raw);
          sc = (ix >= 0) ? sc : -INFINITY;
          p = (ix >= 0) ? p : 0.f;
          s_I[j] = sc;
          s_P[j] = p;
          imax_part = fmaxf(imax_part, sc);
          psum_part += p;
        };
        if (vec4) {
          // 16-byte loads, 2048 slots per round trip (4 x 512): these loads wait behind the previous
          // row's reductions, so their number of round trips sets the time of this step
          constexpr int kStride = 4 * kWorkers;
          for (int j0 = 4 * tid; j0 < n_eff; j0 += 4 * kStride) {
            int4 a[4];
            float4 b[4], c[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int j = j0 + kStride * k;
              if (j < n_eff) {
                a[k] = __ldg(reinterpret_cast<const int4*>(idx_row + j));
                b[k] = __ldg(reinterpret_cast<const float4*>(srow + j));
                c[k] = __ldg(reinterpret_cast<const float4*>(prow + j));
              }
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const int j = j0 + kStride * k;
              if (j < n_eff) {
                take(j, a[k].x, b[k].x, c[k].x);
                if (j + 1 < n_eff) take(j + 1, a[k].y, b[k].y, c[k].y);
                if (j + 2 < n_eff) take(j + 2, a[k].z, b[k].z, c[k].z);
                if (j + 3 < n_eff) take(j + 3, a[k].w, b[k].w, c[k].w);
              }
            }
          }
        } else {
#pragma unroll 4
          for (int j = tid; j < n_eff; j += kWorkers) take(j, __ldg(idx_row + j), __ldg(srow + j), __ldg(prow + j));
        }
      }
      asm volatile("cp.async.wait_all;" ::: "memory");
      named_bar(2, kWorkers);  // Q and s_w are in place
      // Q' = w_h q_idx[h,:] as bf16 hi + lo in Q's layout
#pragma unroll
      for (int k = 0; k < kHeads * 16 / kWorkers; ++k) {
        const int u = tid + kWorkers * k;
        const int hh = u >> 4;
        const uint32_t off = ((u >> 3) & 1) * Q_CHUNK + sw128_off(hh, u & 7);
        const uint4 qv = *reinterpret_cast<const uint4*>(smem + OFF_Q + off);
        const float wh = s_w[hh];
        const uint32_t* qe = reinterpret_cast<const uint32_t*>(&qv);
        uint32_t hv[4], lv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 qf = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&qe[e]));
          const float a = wh * qf.x, b = wh * qf.y;
          const __nv_bfloat162 hi = __floats2bfloat162_rn(a, b);
          const float2 hf = __bfloat1622float2(hi);
          hv[e] = *reinterpret_cast<const uint32_t*>(&hi);
          lv[e] = pack_bf16x2(a - hf.x, b - hf.y);
        }
        st_shared_v4(sQW + off, hv[0], hv[1], hv[2], hv[3]);
        st_shared_v4(sQW + 2 * Q_CHUNK + off, lv[0], lv[1], lv[2], lv[3]);
      }
      fence_proxy_async_smem();  // Q and Q' -> visible to the tensor core
      // ---- the row's distributions and its KL value ----
      const float imax = worker_reduce<true>(imax_part, s_red, warp, lane);
      const float psum = worker_reduce<false>(psum_part, s_red, warp, lane);
      const bool active = imax > -INFINITY && psum > 0.f;
      float klv = 0.f, logz = 0.f, inv_psum = 0.f;
      if (active) {
        float z = 0.f;
        for (int j = tid; j < n_eff; j += kWorkers) z += (s_I[j] > -INFINITY) ? expf(s_I[j] - imax) : 0.f;
        z = worker_reduce<false>(z, s_red, warp, lane);
        logz = imax + logf(z);
        inv_psum = 1.f / psum;
        float acc = 0.f;
        for (int j = tid; j < n_eff; j += kWorkers) {
          const float p = s_P[j] * inv_psum;
          if (s_I[j] > -INFINITY && p > 0.f) acc += p * (logf(p) - (s_I[j] - logz));
        }
        klv = worker_reduce<false>(acc, s_red, warp, lane);
      }
      const int nt = active ? ntiles : 0;
      // publish the row to the MMA and drain warps (its table slot was read two rows ago)
      bool bad = false;
      if (tid == 0) {
        kl_out[t] = klv;
        if (rr >= 2) bad = !mbar_wait(bar_rowfree + 8 * (rr & 1), ((rr >> 1) - 1) & 1, s_abort, err, wait_limit);
        if (!bad) {
          s_rowd[2 * (rr & 1)] = n_eff;
          s_rowd[2 * (rr & 1) + 1] = nt;
          mbar_arrive(bar_row + 8 * (rr & 1));
        }
      }
      if (named_bar_or(2, kWorkers, bad)) { aborted = true; break; }

      // ---- the gradient tiles: gather, S read, m_hj; tile g = g0 + i of this CTA ----
      auto raw_key = [&](int i) -> int {
        const int j = i * kTile + tid;
        return (j < n_eff) ? __ldg(idx_row + j) : -1;
      };
      auto gather_rows = [&](uint32_t g) {
        const int* keys = s_key + (g & 1) * kTile;
        const uint32_t dst = sK + (g & 1) * K_BUF;
        const int u = tid & 15;
#pragma unroll
        for (int e = 0; e < kTile / 8; ++e) {
          const int row = (tid >> 4) + 8 * e;
          const int ix = keys[row];
          cp_async16(dst + (u >> 3) * K_CHUNK + sw128_off(row, u & 7),
                     k_idx + (ix >= 0 ? (size_t)ix * kDi : 0) + u * 8, ix >= 0 ? 16u : 0u);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
      };
      if (nt > 0) {
        int ixa = check_key(raw_key(0));
        s_key[(g0 & 1) * kTile + tid] = ixa;
        int ixb = (nt > 1) ? check_key(raw_key(1)) : -1;
        s_key[((g0 + 1) & 1) * kTile + tid] = ixb;
        int rawc = (nt > 2) ? raw_key(2) : -1;
        named_bar(2, kWorkers);
        gather_rows(g0);
        for (int i = 0; i < nt; ++i) {
          const uint32_t g = g0 + i;
          const int ix = ixa;
          const bool more = i + 1 < nt;
          // tile g (gathered a tile ago, the only copies in flight) has landed: S of it may be formed
          // right after the products of tile g - 1, while this warp issues the next gather
          asm volatile("cp.async.wait_group 0;" ::: "memory");
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_land);
          // the products of tile g - 1 are done: K buffer (g + 1) & 1 and the M tiles are free (at a
          // row's first tile the previous row's end already waited for them)
          if (i >= 1 && !bad) bad = !mbar_wait(bar_mm, (g - 1) & 1, s_abort, err, wait_limit);
          if (named_bar_or(2, kWorkers, bad)) { aborted = true; break; }
          if (more) gather_rows(g + 1);
          const bool ok = mbar_wait(bar_s, g & 1, s_abort, err, wait_limit);
          if (ok) {
            tc_fence_after();
            uint32_t v[64];
            tmem_ld32(tmem_addr(tS, warp * 32, 0), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
            tmem_ld32(tmem_addr(tS, warp * 32, 32), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
            tmem_ld_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_sfree);  // S is read: the next tile's S may be formed
            const int j = i * kTile + tid;
            float gj = 0.f;
            if (j < n_eff && ix >= 0) gj = coeff * (expf(s_I[j] - logz) - s_P[j] * inv_psum);
            const __nv_bfloat16 ghi = __float2bfloat16_rn(gj);
            const uint32_t gh = __bfloat16_as_ushort(ghi);
            const uint32_t gl = __bfloat16_as_ushort(__float2bfloat16_rn(gj - __bfloat162float(ghi)));
            uint32_t mh[32], ml[32];
#pragma unroll
            for (int h = 0; h < kHeads; h += 2) {
              const bool p0 = __uint_as_float(v[h]) > 0.f, p1 = __uint_as_float(v[h + 1]) > 0.f;
              mh[h >> 1] = (p0 ? gh : 0u) | ((p1 ? gh : 0u) << 16);
              ml[h >> 1] = (p0 ? gl : 0u) | ((p1 ? gl : 0u) << 16);
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              st_shared_v4(sMhi + sw128_off(tid, u), mh[4 * u], mh[4 * u + 1], mh[4 * u + 2], mh[4 * u + 3]);
              st_shared_v4(sMlo + sw128_off(tid, u), ml[4 * u], ml[4 * u + 1], ml[4 * u + 2], ml[4 * u + 3]);
            }
            fence_proxy_async_smem();  // M' -> visible to the tensor core
          }
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar_m);
          // this thread's key of tile i + 2 into the table half that gather i has read
          const int kc = (i + 2 < nt) ? check_key(rawc) : -1;
          if (i + 2 < nt) s_key[((g + 2) & 1) * kTile + tid] = kc;
          ixa = ixb;
          ixb = kc;
          rawc = (i + 3 < nt) ? raw_key(i + 3) : -1;
          bad |= !ok;
        }
        // the row's last products are done before dQ^T is read
        if (!aborted && !bad) bad = !mbar_wait(bar_mm, (g0 + nt - 1) & 1, s_abort, err, wait_limit);
        aborted = named_bar_or(2, kWorkers, aborted || bad);
        if (aborted) break;
      }
      // ---- dq_idx (dQ^T in TMEM: lane = dim, column = head) and dw ----
      uint32_t v[64];
      if (nt > 0) {
        tc_fence_after();
        tmem_ld32(tmem_addr(tDQ, warp * 32, 0), *reinterpret_cast<uint32_t(*)[32]>(&v[0]));
        tmem_ld32(tmem_addr(tDQ, warp * 32, 32), *reinterpret_cast<uint32_t(*)[32]>(&v[32]));
        tmem_ld_wait();
        tc_fence_before();  // before this warp's arrivals for the next row's first tile
      } else {
#pragma unroll
        for (int h = 0; h < kHeads; ++h) v[h] = 0u;
      }
      __nv_bfloat16* dq_row = dq_out + (size_t)t * Hi * kDi + tid;  // dim tid of every head
#pragma unroll 8
      for (int h = 0; h < kHeads; ++h)
        if (h < Hi) dq_row[(size_t)h * kDi] = __float2bfloat16_rn(s_w[h] * __uint_as_float(v[h]));
      const uint8_t* qcol = smem + OFF_Q + (tid >> 6) * Q_CHUNK + (tid & 7) * 2;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        float d[32];
#pragma unroll
        for (int hh = 0; hh < 32; ++hh) {
          const int h = 32 * half + hh;
          const __nv_bfloat16 qv = *reinterpret_cast<const __nv_bfloat16*>(qcol + sw128_off(h, (tid & 63) >> 3));
          d[hh] = __bfloat162float(qv) * __uint_as_float(v[h]);
        }
        atomicAdd(s_dw + 32 * half + lane, warp_transpose_sum(d, lane));
      }
      named_bar(2, kWorkers);  // every worker is done with Q, s_w and s_dw of this row
      if (tid < Hi) dw_out[(size_t)t * Hi + tid] = (nt > 0) ? s_dw[tid] : 0.f;
      g0 += nt;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy into shared memory outlives the CTA
  } else if (warp == 4) {
    // ======================= MMA warp: S, then dQ^T += K^T.M and dK = M.Q' per tile =======================
    uint32_t g0 = 0;
    int rr = 0;
    for (int t = blockIdx.x; t < T && !aborted; t += gridDim.x, ++rr) {
      if (!warp_all(mbar_wait(bar_row + 8 * (rr & 1), (rr >> 1) & 1, s_abort, err, wait_limit))) {
        aborted = true;
        break;
      }
      const int nt = s_rowd[2 * (rr & 1) + 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_rowfree + 8 * (rr & 1));
      for (int i = 0; i < nt; ++i) {
        const uint32_t g = g0 + i;
        if (!warp_all(mbar_wait(bar_land, g & 1, s_abort, err, wait_limit))) { aborted = true; break; }
        if (g >= 1 && !warp_all(mbar_wait(bar_sfree, (g - 1) & 1, s_abort, err, wait_limit))) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t kb = sK + (g & 1) * K_BUF;
#pragma unroll
        for (int c = 0; c < 2; ++c)
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ss_w(tS, sdesc_sw128(kb + c * K_CHUNK, 16, 1024) + (uint64_t)(k * 2),
                     sdesc_sw128(sQ + c * Q_CHUNK, 16, 1024) + (uint64_t)(k * 2), kIdS, (c | k) != 0);
        mma_commit_w(bar_s);
        if (!warp_all(mbar_wait(bar_m, g & 1, s_abort, err, wait_limit))) { aborted = true; break; }
        // dK buffer g & 1 was read by the drain of tile g - 2
        if (g >= 2 && !warp_all(mbar_wait(bar_dkf + 8 * (g & 1), ((g - 2) >> 1) & 1, s_abort, err, wait_limit))) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t tdk = tDK + 128 * (g & 1);
        const uint64_t ka = sdesc_sw128(kb, K_CHUNK, 1024);
        const uint64_t mb_hi = sdesc_sw128(sMhi, K_CHUNK, 1024);
        const uint64_t mb_lo = sdesc_sw128(sMlo, K_CHUNK, 1024);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k) {
          mma_ss_w(tDQ, ka + (uint64_t)(k * 128), mb_hi + (uint64_t)(k * 128), kIdDQ, (i > 0 || k > 0) ? 1u : 0u);
          mma_ss_w(tDQ, ka + (uint64_t)(k * 128), mb_lo + (uint64_t)(k * 128), kIdDQ, 1u);
        }
        const uint64_t ma_hi = sdesc_sw128(sMhi, 16, 1024), ma_lo = sdesc_sw128(sMlo, 16, 1024);
        const uint64_t qwh = sdesc_sw128(sQW, Q_CHUNK, 1024), qwl = sdesc_sw128(sQW + 2 * Q_CHUNK, Q_CHUNK, 1024);
#pragma unroll
        for (int k = 0; k < kHeads / 16; ++k) {
          mma_ss_w(tdk, ma_hi + (uint64_t)(k * 2), qwh + (uint64_t)(k * 128), kIdDK, k > 0 ? 1u : 0u);
          mma_ss_w(tdk, ma_hi + (uint64_t)(k * 2), qwl + (uint64_t)(k * 128), kIdDK, 1u);
          mma_ss_w(tdk, ma_lo + (uint64_t)(k * 2), qwh + (uint64_t)(k * 128), kIdDK, 1u);
        }
        mma_commit_w(bar_mm);
        mma_commit_w(bar_mmd + 8 * (g & 1));
      }
      g0 += nt;
    }
  } else {
    // ======================= dK drain: rows into dk_idx by L2 reductions =======================
    const int qd = warp & 3;       // TMEM lane quadrant of this warp
    const int r = qd * 32 + lane;  // slot row of the tile
    const uint32_t fst = smem_u32(smem + OFF_FST + (warp - 5) * 2048);
    uint32_t g0 = 0;
    int rr = 0;
    for (int t = blockIdx.x; t < T && !aborted; t += gridDim.x, ++rr) {
      if (!mbar_wait(bar_row + 8 * (rr & 1), (rr >> 1) & 1, s_abort, err, wait_limit)) { aborted = true; break; }
      const int n_eff = s_rowd[2 * (rr & 1)], nt = s_rowd[2 * (rr & 1) + 1];
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_rowfree + 8 * (rr & 1));
      const int32_t* idx_row = topk_idx + (size_t)t * K;
      auto key_of = [&](int i) -> int {  // the row's key (the workers report bad indices)
        const int j = i * kTile + r;
        const int raw = (j < n_eff) ? __ldg(idx_row + j) : -1;
        return (raw >= 0 && raw < Tk) ? raw : -1;
      };
      int key_next = (nt > 0) ? key_of(0) : -1;
      for (int i = 0; i < nt; ++i) {
        const uint32_t g = g0 + i;
        const int key = key_next;
        if (i + 1 < nt) key_next = key_of(i + 1);
        if (!mbar_wait(bar_mmd + 8 * (g & 1), (g >> 1) & 1, s_abort, err, wait_limit)) { aborted = true; break; }
        tc_fence_after();
        const uint32_t tdk = tDK + 128 * (g & 1);
#pragma unroll 1
        for (int b = 0; b < kDi / 32; ++b) {
          uint32_t v[32];
          tmem_ld32(tmem_addr(tdk, qd * 32, 32 * b), v);
          tmem_ld_wait();
          if (b == kDi / 32 - 1) {  // the last load of the buffer: it may be refilled
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_dkf + 8 * (g & 1));
          }
#pragma unroll
          for (int hh = 0; hh < 2; ++hh) {
            if ((lane >> 4) == hh) {
              const int rl = lane & 15;
#pragma unroll
              for (int u = 0; u < 8; ++u)
                st_shared_v4(fst + rl * 128 + ((u ^ (rl & 7)) << 4), v[4 * u], v[4 * u + 1], v[4 * u + 2],
                             v[4 * u + 3]);
            }
            __syncwarp();
#pragma unroll
            for (int st = 0; st < 4; ++st) {
              const int rl = 4 * st + (lane >> 3), u = lane & 7;
              const int kr = __shfl_sync(0xffffffffu, key, 16 * hh + rl);
              float4 f;
              asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                           : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                           : "r"(fst + rl * 128 + ((u ^ (rl & 7)) << 4))
                           : "memory");
              if (kr >= 0) red_add_v4(dk + (size_t)kr * kDi + 32 * b + 4 * u, f.x, f.y, f.z, f.w);
            }
            __syncwarp();
          }
        }
      }
      g0 += nt;
    }
  }

  if (warp == 4) {
    // every MMA of this CTA completes before the teardown frees TMEM
    mma_commit_w(bar_fin);
    volatile int dummy = 0;
    mbar_wait(bar_fin, 0, &dummy, err);
  }
  __syncwarp();
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}


}  // namespace kl
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_indexer_kl_workspace_size(int32_t T, int32_t K) {
  (void)T;
  (void)K;
  return kErrorWordBytes;
}

extern "C" dsa_status_t dsa_indexer_kl(const dsa_bf16_t* q_idx, const dsa_bf16_t* k_idx, const float* head_weights,
                                       const int32_t* topk_idx, const int32_t* topk_len, const float* attn_prob,
                                       const float* topk_score, int32_t T, int32_t T_k, int32_t Hi, int32_t Di, int32_t K, float coeff,
                                       float* kl, dsa_bf16_t* dq_idx, float* dw, float* dk_idx_accum,
                                       int32_t accumulate, void* workspace, size_t workspace_bytes,
                                       dsa_stream_t stream) {
  const char* who = "dsa_indexer_kl";
  if (T < 0 || T_k < 1) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: need T >= 0 and T_k >= 1", who);
  if (Hi < 1 || Hi > kl::kHeads) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Hi must be in [1, 64] (got %d)", who, Hi);
  if (Di != kl::kDi) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Di must be 128 (got %d)", who, Di);
  if (K < 1 || K > kl::kMaxK)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: K must be in [1, %d] (got %d)", who, kl::kMaxK, K);
  if (accumulate != 0 && accumulate != 1) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: accumulate must be 0 or 1", who);
  if (!std::isfinite(coeff)) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: coeff must be finite", who);
  if (!k_idx || !dk_idx_accum) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: k_idx / dk_idx_accum is NULL", who);
  if (T > 0 && (!q_idx || !head_weights || !topk_idx || !attn_prob || !kl || !dq_idx || !dw))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: null tensor pointer", who);
  if (!aligned16(k_idx) || !aligned16(dk_idx_accum) || (T > 0 && !aligned16(q_idx)))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: q_idx, k_idx and dk_idx_accum must be 16-byte aligned", who);
  dsa_status_t st = check_workspace(workspace, workspace_bytes, dsa_indexer_kl_workspace_size(T, K), who);
  if (st != DSA_OK) return st;
  if ((st = check_device()) != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = clear_error_word(workspace, s)) != DSA_OK) return st;
  if (!accumulate && (st = cuda_check(cudaMemsetAsync(dk_idx_accum, 0, (size_t)T_k * Di * sizeof(float), s),
                                      "zeroing dk_idx_accum")))
    return st;
  if (T == 0) return ok();
  if (topk_score != nullptr) {
    // one CTA per SM, each walking its share of the rows
    int dev = 0, nsm = 0;
    if ((st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice")) ||
        (st = cuda_check(cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev), "SM count")))
      return st;
    if ((st = configure_kernel_smem(reinterpret_cast<const void*>(kl::indexer_kl_rows_kernel), kl::TOTAL,
                                    "configuring indexer_kl_rows_kernel")))
      return st;
    const int grid = T < nsm ? T : nsm;
    kl::indexer_kl_rows_kernel<<<grid, kl::kThreads, kl::TOTAL, s>>>(
        reinterpret_cast<const __nv_bfloat16*>(k_idx), reinterpret_cast<const __nv_bfloat16*>(q_idx), head_weights,
        topk_idx, topk_len, attn_prob, topk_score, T, T_k, Hi, K, coeff, kl, reinterpret_cast<__nv_bfloat16*>(dq_idx),
        dw, dk_idx_accum, reinterpret_cast<int*>(workspace), wait_limit_cycles());
    if ((st = cuda_check(cudaGetLastError(), "launching indexer_kl_rows_kernel"))) return st;
    return ok();
  }
  if ((st = configure_kernel_smem(reinterpret_cast<const void*>(kl::indexer_kl_kernel), kl::TOTAL,
                                  "configuring indexer_kl_kernel")))
    return st;
  kl::indexer_kl_kernel<<<T, kl::kThreads, kl::TOTAL, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(k_idx), reinterpret_cast<const __nv_bfloat16*>(q_idx), head_weights,
      topk_idx, topk_len, attn_prob, T_k, Hi, K, coeff, kl, reinterpret_cast<__nv_bfloat16*>(dq_idx), dw,
      dk_idx_accum, reinterpret_cast<int*>(workspace), wait_limit_cycles());
  if ((st = cuda_check(cudaGetLastError(), "launching indexer_kl_kernel"))) return st;
  return ok();
}
