// dsa_fwd.cu -- absorbed sparse MLA forward on sm_103a (tcgen05 + TMEM).
//
// Computes, for one query token t and one group of 64 heads per CTA,
//   z_j = scale <q[t,h,:], kv[idx_j,:]>,  lse = ln sum_j e^{z_j},
//   out[t,h,:] = sum_j e^{z_j - lse} kv[idx_j, 0:512]
// over the token's valid top-k slots.  Source: "Accelerating GLM-5.2
// Long-Context Training with cuDNN Fused DSA Kernels ...", sections "How DSA
// works" (every head of a query attends only to that query's selected rows)
// and "Why DSA needs fused kernels" (absorbed MLA: an MQA over one shared
// latent, so the gathered rows are shared by all heads); NeMo AutoModel
// glm_moe_dsa.kernels.cudnn_dsa, cudnn_sparse_attention (shapes, -1 slots,
// topk_length, explicit softmax_scale); SkyRL PR 2388, "Change" (value =
// kv[..., :512], NoPE width 512).
//
// Design (sm_103a):
//  * The selected kv rows of a 128-slot tile are gathered ONCE into shared
//    memory (128-byte swizzled, 9 chunks of 64 channels) and used by all 64
//    heads of the CTA.  The gather is 16-byte cp.async issued by the 256
//    softmax threads (many requests in flight; a per-chunk mbarrier counts the
//    landings), so the tensor core starts on chunk 0 while later chunks land.
//  * Scores are computed transposed, S^T[key, head] = KV_tile . Q^T: the
//    tensor-core M axis is the 128 keys of the tile and N = 64 heads
//    (M = 128 is the full-rate tcgen05 shape; the heads are the shared
//    operand).  Output is accumulated transposed too, O^T[ch, head] +=
//    V^T . P^T, as four M = 128 channel tiles.
//  * P is split into bf16 hi + lo parts and P.V runs on both, so O is accurate
//    to about fp32 and the backward's D = <dO, O> matches the exact softmax:
//    with P in bf16 alone (the operand precision of the pages' kernels) D is
//    off by about 2^-8 of its terms, and dq / dkv miss the 2e-2 max-abs target
//    on unit-scale inputs.  For channel tiles 0..2 the two parts sit side by
//    side on the MMA's N axis (N = 128, hi and lo accumulated in separate TMEM
//    columns and added at the end): one MMA reads each V^T tile once, and N =
//    128 runs at the full rate where N = 64 runs at two thirds of it.  TMEM
//    (512 columns: S^T 64, O^T 3 x 128 + 64) leaves tile 3 at N = 64, hi and lo
//    one after the other into the same columns.
//  * P.V runs key rows 0..63 first, then rows 64..127, and signals after the
//    first half: the next tile's rows 0..63 of every value chunk are
//    gathered while the tensor core works on rows 64..127.  Rows 64..127 go
//    channel pair by channel pair, each pair signalled once read, so the next
//    tile's rows 64..127 of a pair are gathered while later pairs run.
//  * Online softmax with the running max per head; a rescale of O^T happens
//    only when some score exceeds the running max by more than 2^8 (lazy
//    rescale), otherwise P uses the stale max.
//  * P^T is written into the shared-memory slot of the tile's RoPE channels
//    (no longer needed once S^T is done) and an 8 KiB slot before it, which
//    keeps the working set (Q 72 KiB + tile 144 KiB + 8 KiB) inside one SM's
//    shared memory.  For each 64-key half the hi and lo blocks of the N = 128
//    operand are 8 KiB apart: keys 0..63 hold hi in rows 0..63 of the P slot
//    and lo in rows 64..127; keys 64..127 hold hi in the slot before, and their
//    lo goes into the P slot's rows 0..63 once the first key half of P.V has
//    read them, while the tensor core runs P_hi of rows 64..127 of tile 3.
//  * An attention sink (optional, one logit per head: NeMo AutoModel
//    glm_moe_dsa.kernels.cudnn_dsa, _pad_attention_heads) starts the running
//    max of its head and adds its own term to the denominator at the end; it
//    has no value row.
//  * The epilogue stages O (and, on request, the bf16 residual O - bf16(O))
//    through shared memory for coalesced 16-byte stores.
//
// Warp roles: warp 0 issues MMAs (the whole warp runs the issuing loop, one elected
// lane issues each instruction) and owns TMEM; warps 1..8 run
// the gather, the softmax and the epilogue.
#include <cmath>
#include <type_traits>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {
namespace fwd {

constexpr int kThreads = 288;
constexpr int kWorkers = 256;
constexpr int kTile = 128;   // top-k slots per tile (MMA M)
constexpr int kHeads = 64;   // heads per CTA (MMA N)
constexpr int kDv = 512;
constexpr float kRescaleThreshold = 8.0f;  // log2 units

template <int DQK>
struct Smem {
  static constexpr int NCH = DQK / 64;          // 64-channel chunks (9 or 8)
  static constexpr int Q_CHUNK = kHeads * 128;  // one chunk of Q: 64 heads x 128 B
  static constexpr int KV_CHUNK = kTile * 128;  // one chunk of the tile: 128 keys x 128 B
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = OFF_Q + NCH * Q_CHUNK;  // value chunks 0..7
  // P^T, one 64-key half at a time, as an MN-major operand of N = 128 ([hi | lo] column blocks
  // 8 KiB apart).  The P slot is the RoPE chunk when there is one (free once S^T is done), else a
  // slot of its own; its rows 0..63 hold P_hi and rows 64..127 P_lo of keys 0..63.  The 8 KiB
  // slot just before it holds P_hi of keys 64..127, whose P_lo goes into the P slot's rows 0..63
  // once keys 0..63 have been multiplied.
  static constexpr int OFF_PHI2 = OFF_KV + 8 * KV_CHUNK;
  static constexpr int OFF_P = OFF_PHI2 + KV_CHUNK / 2;
  static constexpr int OFF_MISC = OFF_P + KV_CHUNK;
  static constexpr int MISC = 2048;
  static constexpr int TOTAL = OFF_MISC + MISC + 1024;  // + alignment slack
  static_assert(TOTAL <= 232448, "shared memory budget");
};

// misc layout (bytes)
constexpr int M_BAR_KV = 0;    // [9] chunk landed
constexpr int M_BAR_PV = 80;   // P.V of the tile done
constexpr int M_BAR_PVP = 88;  // [3]: key rows 0..63 of channel pair m read (pair 3: M_BAR_PVH)
constexpr int M_BAR_S = 112, M_BAR_P = 120, M_BAR_FIN = 128, M_BAR_PLO = 136, M_BAR_PVH = 144;
constexpr int M_BAR_PVM = 152;  // [3]: key rows 64..127 of channel pair m (chunks 2m, 2m+1) read
constexpr int M_TMEM = 192, M_NEFF = 196, M_ABORT = 200;
constexpr int M_RED = 256;             // float [4][64]
constexpr int M_STAT = M_RED + 1024;   // float [64]: running max per head
constexpr int M_LSUM = M_STAT + 256;   // float [64]: softmax denominator per head
constexpr int M_MMIN = M_LSUM + 256;   // float [2]: smallest running max of each head half

// Element-wise fp32 on two lanes at once (add / fma / sub .f32x2, round to nearest as the scalar ops).
__device__ __forceinline__ float2 f32x2_add(float2 a, float2 b) {
  uint64_t r;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(r)
      : "l"((uint64_t)__float_as_uint(a.x) | ((uint64_t)__float_as_uint(a.y) << 32)),
        "l"((uint64_t)__float_as_uint(b.x) | ((uint64_t)__float_as_uint(b.y) << 32)));
  return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}
__device__ __forceinline__ float2 f32x2_fma(float2 a, float2 b, float2 c) {
  uint64_t r;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(r)
      : "l"((uint64_t)__float_as_uint(a.x) | ((uint64_t)__float_as_uint(a.y) << 32)),
        "l"((uint64_t)__float_as_uint(b.x) | ((uint64_t)__float_as_uint(b.y) << 32)),
        "l"((uint64_t)__float_as_uint(c.x) | ((uint64_t)__float_as_uint(c.y) << 32)));
  return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}
__device__ __forceinline__ float2 f32x2_sub(float2 a, float2 b) {
  uint64_t r;
  asm("sub.rn.f32x2 %0, %1, %2;"
      : "=l"(r)
      : "l"((uint64_t)__float_as_uint(a.x) | ((uint64_t)__float_as_uint(a.y) << 32)),
        "l"((uint64_t)__float_as_uint(b.x) | ((uint64_t)__float_as_uint(b.y) << 32)));
  return make_float2(__uint_as_float((uint32_t)r), __uint_as_float((uint32_t)(r >> 32)));
}

// Transposing butterfly: v[0..31] per lane (lane = key, index = head) ->
// lane l returns the reduction over the warp's 32 keys of head l.
template <bool MAX>
__device__ __forceinline__ float warp_transpose_reduce(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      float send = upper ? v[i] : v[i + o];
      float keep = upper ? v[i + o] : v[i];
      float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// Gather channels [64c, 64c+64) of the tile's rows into chunk slot c.  Thread
// `tid` copies 16-byte unit (tid & 7) of rows r_e = (tid >> 3) + 32 e.  Rows
// whose slot is invalid or beyond the valid prefix are zero-filled (no global
// read), so every row of the tile is finite and P = 0 times it stays 0.
template <int DQK>
__device__ __forceinline__ void gather_chunk(uint32_t dst_chunk, const __nv_bfloat16* __restrict__ kv, int c, int tid,
                                             const int (&rix)[4], uint32_t bar) {
  const int uc = tid & 7;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const int r = (tid >> 3) + 32 * e;
    const bool ok = rix[e] >= 0;
    const __nv_bfloat16* src = kv + (ok ? (size_t)rix[e] * DQK + c * 64 + uc * 8 : 0);
    cp_async16(dst_chunk + sw128_off(r, uc), src, ok ? 16u : 0u);
  }
  cp_async_arrive(bar);
}

// Rows 0..63 (half 0) or 64..127 (half 1) of the same copy, without the arrive.
template <int DQK>
__device__ __forceinline__ void gather_half(uint32_t dst_chunk, const __nv_bfloat16* __restrict__ kv, int c, int tid,
                                            const int (&rix)[4], int half) {
  const int uc = tid & 7;
#pragma unroll
  for (int e = 2 * half; e < 2 * half + 2; ++e) {
    const int r = (tid >> 3) + 32 * e;
    const bool ok = rix[e] >= 0;
    const __nv_bfloat16* src = kv + (ok ? (size_t)rix[e] * DQK + c * 64 + uc * 8 : 0);
    cp_async16(dst_chunk + sw128_off(r, uc), src, ok ? 16u : 0u);
  }
}

template <int DQK>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_fwd_kernel(const __nv_bfloat16* __restrict__ kv, const __nv_bfloat16* __restrict__ q,
                          const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ topk_len, int T, int Tk,
                          int H, int K, float sl2e, const float* __restrict__ sink, __nv_bfloat16* __restrict__ out,
                          __nv_bfloat16* __restrict__ out_lo, float* __restrict__ lse, int* __restrict__ err,
                          long long wait_limit) {
  using L = Smem<DQK>;
  constexpr int NCH = L::NCH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + L::OFF_Q);
  const uint32_t sKV = smem_u32(smem + L::OFF_KV);
  const uint32_t sP = smem_u32(smem + L::OFF_P);
  const uint32_t sPhi2 = smem_u32(smem + L::OFF_PHI2);
  // chunk slot c of the tile: value chunks 0..7, the RoPE chunk in the P slot
  auto chunk_addr = [&](int c) -> uint32_t { return c < 8 ? sKV + c * L::KV_CHUNK : sP; };
  uint8_t* misc = smem + L::OFF_MISC;
  const uint32_t bar_kv = smem_u32(misc + M_BAR_KV), bar_pv = smem_u32(misc + M_BAR_PV);
  const uint32_t bar_s = smem_u32(misc + M_BAR_S), bar_p = smem_u32(misc + M_BAR_P);
  const uint32_t bar_fin = smem_u32(misc + M_BAR_FIN);
  const uint32_t bar_plo = smem_u32(misc + M_BAR_PLO), bar_pvh = smem_u32(misc + M_BAR_PVH);
  const uint32_t bar_pvm = smem_u32(misc + M_BAR_PVM);
  const uint32_t bar_pvp = smem_u32(misc + M_BAR_PVP);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + M_TMEM);
  int* s_neff = reinterpret_cast<int*>(misc + M_NEFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + M_ABORT);
  float* s_red = reinterpret_cast<float*>(misc + M_RED);
  float* s_stat = reinterpret_cast<float*>(misc + M_STAT);
  float* s_lsum = reinterpret_cast<float*>(misc + M_LSUM);
  float* s_mmin = reinterpret_cast<float*>(misc + M_MMIN);

  const int t = blockIdx.x;
  const int hg = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* idx_row = topk_idx + (size_t)t * K;

  if (threadIdx.x == 0) {
    for (int c = 0; c < NCH; ++c) mbar_init(bar_kv + 8 * c, kWorkers);
    mbar_init(bar_pv, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 8);
    mbar_init(bar_pvh, 1);
    for (int m = 0; m < 3; ++m) mbar_init(bar_pvm + 8 * m, 1);
    for (int m = 0; m < 3; ++m) mbar_init(bar_pvp + 8 * m, 1);
    mbar_init(bar_plo, 4);  // the warps of key rows 64..127 (lane quadrants 2, 3)
    mbar_init(bar_fin, 1);
    *s_neff = 0;
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  __syncthreads();

  const int tid = threadIdx.x - 32;  // worker id 0..255 (negative for warp 0)
  // ---- valid prefix length and Q staging (workers) ----
  if (warp >= 1) {
    if (topk_len != nullptr) {
      if (tid == 0) {
        int n = topk_len[t];
        *s_neff = n < 0 ? 0 : (n > K ? K : n);
      }
    } else {
      int last = 0;
      for (int j = tid; j < K; j += kWorkers)
        if (idx_row[j] >= 0) last = j + 1;
      if (last) atomicMax(s_neff, last);
    }
    if (tid < kHeads) {  // running max per head (log2 units), from the sink logit when there is one
      const int h = hg * kHeads + tid;
      s_stat[tid] = (sink != nullptr && h < H) ? __ldg(sink + h) * 1.4426950408889634f : -INFINITY;
    }
    // Q [64 heads, DQK] -> NCH chunks of [64 rows x 128 B], 128B swizzle; heads >= H are zero.
    constexpr int UNITS = kHeads * NCH * 8;
    const uint64_t pol = l2_evict_first_policy();  // q is read once: evicted first, the kv rows stay
    for (int u = tid; u < UNITS; u += kWorkers) {
      const int hh = u / (NCH * 8);
      const int rem = u - hh * (NCH * 8);
      const int c = rem >> 3, uc = rem & 7;
      const int h = hg * kHeads + hh;
      const bool ok = h < H;  // padded heads are zero-filled without a read
      cp_async16_hint(sQ + c * L::Q_CHUNK + sw128_off(hh, uc),
                      q + (ok ? ((size_t)t * H + h) * DQK + c * 64 + uc * 8 : 0), ok ? 16u : 0u, pol);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // all copies in flight at once, one wait
    fence_proxy_async_smem();
  }
  __syncthreads();
  const int n_eff = *s_neff;
  const int ntiles = (n_eff + kTile - 1) / kTile;
  const uint32_t tmem = *s_tmem;
  const uint32_t tS = tmem;        // S^T: 128 lanes x 64 columns
  // O^T: channel tiles 0..2 as [hi | lo] (128 columns each), channel tile 3 with hi and lo
  // accumulated together (64 columns): 64 + 3 x 128 + 64 = 512 columns
  const uint32_t tO = tmem + 64;
  const uint32_t tO3 = tO + 3 * 128;

  if (warp == 0) {
    // ======================= MMA issuer (the whole warp, one elected lane issues) =======================
    {
      constexpr uint32_t kIdS = idesc_bf16(128, kHeads, false, false);  // A = KV (K-major), B = Q (K-major)
      constexpr uint32_t kIdPV = idesc_bf16(128, kHeads, true, true);   // A = V^T (MN-major), B = P^T (MN-major)
      constexpr uint32_t kIdPV2 = idesc_bf16(128, 2 * kHeads, true, true);  // B = [P_hi | P_lo]^T, N = 128
      for (int i = 0; i < ntiles; ++i) {
        bool stop = false;
        // one burst per group of landed chunks: wait for the next chunk, then take every
        // later chunk that has landed too (fewer fences and waits between MMAs)
        const uint64_t b00 = sdesc_sw128(sQ, 16, 1024);
        for (int c = 0; c < NCH && !stop;) {
          if (!warp_all(mbar_wait(bar_kv + 8 * c, i & 1, s_abort, err, wait_limit))) { stop = true; break; }
          int ce = c + 1;
          while (ce < NCH && warp_all(mbar_test(bar_kv + 8 * ce, i & 1))) ++ce;
          fence_proxy_async_smem();  // cp.async landings -> visible to the tensor core
          tc_fence_after();
          for (; c < ce; ++c) {
            const uint64_t a0 = sdesc_sw128(chunk_addr(c), 16, 1024), b0 = b00 + (uint64_t)((c * L::Q_CHUNK) >> 4);
#pragma unroll
            for (int k = 0; k < 4; ++k)  // + 16 channels = + 32 bytes per row
              mma_ss_w(tS, a0 + (uint64_t)(k * 2), b0 + (uint64_t)(k * 2), kIdS, (c | k) != 0);
          }
        }
        if (stop) break;
        mma_commit_w(bar_s);
        // O^T += V^T [P_hi | P_lo]^T, key rows 0..63 first, so that rows 0..63 of every chunk slot
        // are free while rows 64..127 are multiplied.  Channel tiles 0..2 take hi and lo in one MMA
        // (N = 128, separate accumulators); tile 3 takes them one after the other (N = 64 each).
        if (!warp_all(mbar_wait(bar_p, i & 1, s_abort, err, wait_limit))) break;
        tc_fence_after();
        constexpr uint64_t kLo = (L::KV_CHUNK / 2) >> 4;    // descriptor step from the hi to the lo block
        const uint64_t pa = sdesc_sw128(sP, L::KV_CHUNK / 2, 1024);     // keys 0..63
        const uint64_t pb = sdesc_sw128(sPhi2, L::KV_CHUNK / 2, 1024);  // keys 64..127
        const uint64_t va0 = sdesc_sw128(sKV, L::KV_CHUNK, 1024);
        constexpr uint64_t kPair = (2 * L::KV_CHUNK) >> 4;  // descriptor step between channel pairs
        constexpr int kHalf = kTile / 32;                   // 16-key steps per 64-key half
#pragma unroll
        for (int m = 0; m < 3; ++m) {
#pragma unroll
          for (int k = 0; k < kHalf; ++k)  // + 16 key rows = + 2048 bytes
            mma_ss_w(tO + m * 128, va0 + m * kPair + (uint64_t)(k * 128), pa + (uint64_t)(k * 128), kIdPV2,
                     (i > 0 || k > 0) ? 1u : 0u);
          mma_commit_w(bar_pvp + 8 * m);  // rows 0..63 of channel pair m are read
        }
#pragma unroll
        for (int k = 0; k < kHalf; ++k)
          mma_ss_w(tO3, va0 + 3 * kPair + (uint64_t)(k * 128), pa + (uint64_t)(k * 128), kIdPV,
                   (i > 0 || k > 0) ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < kHalf; ++k)
          mma_ss_w(tO3, va0 + 3 * kPair + (uint64_t)(k * 128), pa + kLo + (uint64_t)(k * 128), kIdPV, 1u);
        mma_commit_w(bar_pvh);  // rows 0..63 of the chunk slots (and the P slot) are read
        // Key rows 64..127 channel pair by channel pair, with a commit after each pair, so that the
        // next tile's rows 64..127 of a pair are gathered while later pairs are multiplied.  P_hi of
        // tile 3 first: the tensor core works on it while the workers move P_lo of rows 64..127 into
        // the P slot's rows 0..63.
#pragma unroll
        for (int k = 0; k < kHalf; ++k)
          mma_ss_w(tO3, va0 + 3 * kPair + (uint64_t)((kHalf + k) * 128), pb + (uint64_t)(k * 128), kIdPV, 1u);
        if (!warp_all(mbar_wait(bar_plo, i & 1, s_abort, err, wait_limit))) break;
        tc_fence_after();
#pragma unroll
        for (int m = 0; m < 3; ++m) {
#pragma unroll
          for (int k = 0; k < kHalf; ++k)
            mma_ss_w(tO + m * 128, va0 + m * kPair + (uint64_t)((kHalf + k) * 128), pb + (uint64_t)(k * 128), kIdPV2,
                     1u);
          mma_commit_w(bar_pvm + 8 * m);
        }
#pragma unroll
        for (int k = 0; k < kHalf; ++k)
          mma_ss_w(tO3, va0 + 3 * kPair + (uint64_t)((kHalf + k) * 128), pb + kLo + (uint64_t)(k * 128), kIdPV, 1u);
        mma_commit_w(bar_pv);  // P.V of this tile is complete
      }
      // every MMA of this CTA completes before the teardown frees TMEM
      mma_commit_w(bar_fin);
      volatile int dummy = 0;
      mbar_wait(bar_fin, 0, &dummy, err);
    }
    __syncwarp();
  } else {
    // ======================= gather + softmax + epilogue =======================
    const int wk = warp - 1;          // 0..7
    const int qd = warp & 3;          // TMEM lane quadrant this warp may access
    const int ch = wk >> 2;           // head half: heads ch*32 .. ch*32+31
    const int r = qd * 32 + lane;     // key row of the tile / channel row of an O^T tile
    const int bar_id = 1 + ch;        // named barrier of the 128 threads of this half
    // Row indices this thread gathers for tile i, in two steps: the raw loads (issued a tile
    // ahead, so that their memory latency hides behind the softmax and P.V of the tile before)
    // and the check that turns them into row numbers, -1 = zero-fill (invalid or beyond the prefix).
    auto load_raw = [&](int i, int (&raw)[4]) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = i * kTile + (tid >> 3) + 32 * e;
        raw[e] = (j < n_eff) ? __ldg(idx_row + j) : -1;
      }
    };
    auto check_rows = [&](const int (&raw)[4], int (&rix)[4]) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int ix = raw[e];
        rix[e] = (ix >= 0 && ix < Tk) ? ix : -1;
        if (ix < -1 || ix >= Tk) record_error(err, DSA_ERR_DEVICE_INDEX);
      }
    };
    int nraw[4];  // raw indices of the next tile
    if (ntiles > 0) {
      int rix[4];
      load_raw(0, nraw);
      check_rows(nraw, rix);
      for (int c = 0; c < NCH; ++c) gather_chunk<DQK>(chunk_addr(c), kv, c, tid, rix, bar_kv + 8 * c);
    }
    // running max per head lives in s_stat (identical for all threads of a half)
    const float* m_run = s_stat + ch * 32;
    float l_part[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) l_part[h] = 0.f;
    bool aborted = false;
    for (int i = 0; i < ntiles; ++i) {
      // this key row's index and the next tile's gather rows do not depend on the MMA: their
      // loads overlap the wait (and, for the gather rows, this whole tile)
      const int j = i * kTile + r;
      const int ixw = (j < n_eff) ? __ldg(idx_row + j) : -1;
      const bool more = i + 1 < ntiles;
      if (more) load_raw(i + 1, nraw);
      const bool got = mbar_wait(bar_s, i & 1, s_abort, err, wait_limit);
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tmem_addr(tS, qd * 32, ch * 32), sv);  // (after a failed wait a stale value is harmless)
      tmem_ld_wait();
      const bool valid = ixw >= 0 && ixw < Tk;
      bool mine = (i == 0);  // the first tile always sets the running max
      if (!mine) {
        // Does any score of this key exceed its head's running max by the threshold?  First against
        // the smallest running max of the half (this key's largest score, one compare), per head only
        // when that test fails.
        float smax = __uint_as_float(sv[0]);
#pragma unroll
        for (int h = 1; h < 32; ++h) smax = fmaxf(smax, __uint_as_float(sv[h]));
        mine = valid && smax * sl2e > s_mmin[ch] + kRescaleThreshold;
        if (mine) {
          mine = false;
#pragma unroll
          for (int h4 = 0; h4 < 8; ++h4) {  // running max as 16-byte loads (4 heads)
            const float4 m4 = reinterpret_cast<const float4*>(m_run)[h4];
            mine |= (__uint_as_float(sv[4 * h4]) * sl2e > m4.x + kRescaleThreshold) |
                    (__uint_as_float(sv[4 * h4 + 1]) * sl2e > m4.y + kRescaleThreshold) |
                    (__uint_as_float(sv[4 * h4 + 2]) * sl2e > m4.z + kRescaleThreshold) |
                    (__uint_as_float(sv[4 * h4 + 3]) * sl2e > m4.w + kRescaleThreshold);
          }
        }
      }
      // one barrier of the half per tile in the common case; a rescale, the first tile or an abort takes a
      // second one to tell them apart (every thread of the half leaves together, or none does)
      bool need = false;
      if (named_bar_or(bar_id, 128, mine || !got)) {
        if (named_bar_or(bar_id, 128, !got)) { aborted = true; break; }
        need = true;
      }
      if (need) {
        float v[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) v[h] = valid ? __uint_as_float(sv[h]) * sl2e : -INFINITY;
        const float wmax = warp_transpose_reduce<true>(v, lane);
        s_red[qd * 64 + ch * 32 + lane] = wmax;
        named_bar(bar_id, 128);
        const float bm = fmaxf(fmaxf(s_red[ch * 32 + lane], s_red[64 + ch * 32 + lane]),
                               fmaxf(s_red[128 + ch * 32 + lane], s_red[192 + ch * 32 + lane]));
        const float mn = fmaxf(s_stat[ch * 32 + lane], bm);
        // old max (mo) of every head of this half, then publish the new one
        float alpha[32];
        bool any = false;
        const float mo_lane = s_stat[ch * 32 + lane];
        named_bar(bar_id, 128);
        if (qd == 0) {
          s_stat[ch * 32 + lane] = mn;
          float mm = mn;
#pragma unroll
          for (int o = 16; o >= 1; o >>= 1) mm = fminf(mm, __shfl_xor_sync(0xffffffffu, mm, o));
          if (lane == 0) s_mmin[ch] = mm;
        }
        named_bar(bar_id, 128);
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const float mo = __shfl_sync(0xffffffffu, mo_lane, h);
          const float mnew = m_run[h];
          alpha[h] = (mo == -INFINITY) ? 0.f : exp2f(mo - mnew);
          any |= (i > 0) && (alpha[h] != 1.f);
          l_part[h] *= alpha[h];
        }
        if (any) {
          // O^T is complete for the previous tile: bar_s of this tile was
          // committed after those MMAs by the same thread.
#pragma unroll 1
          for (int g = 0; g < 7; ++g) {  // hi and lo of channel tiles 0..2, then tile 3
            uint32_t ov[32];
            const uint32_t ta = tmem_addr(g < 6 ? tO + (g >> 1) * 128 + (g & 1) * 64 : tO3, qd * 32, ch * 32);
            tmem_ld32(ta, ov);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
            tmem_st32(ta, ov);
          }
          tmem_st_wait();
        }
      }
      uint32_t pk[16], pl[16];
      // exponent argument s * scale * log2(e) - m in one rounding; an invalid slot gets -inf (P = +0)
      const float shift = valid ? 0.f : -INFINITY;
#pragma unroll
      for (int h = 0; h < 32; h += 2) {
        const float4 m4 = reinterpret_cast<const float4*>(m_run)[h >> 2];
        const float ma = (h & 2) ? m4.z : m4.x, mb = (h & 2) ? m4.w : m4.y;
        const float mu0 = (ma == -INFINITY) ? 0.f : ma;  // a head with no valid slot yet (all its slots masked)
        const float mu1 = (mb == -INFINITY) ? 0.f : mb;
        const float2 nmu = f32x2_sub(make_float2(shift, shift), make_float2(mu0, mu1));
        const float2 e = f32x2_fma(make_float2(__uint_as_float(sv[h]), __uint_as_float(sv[h + 1])),
                                   make_float2(sl2e, sl2e), nmu);
        const float2 pp = make_float2(exp2f(e.x), exp2f(e.y));
        const float2 ls = f32x2_add(make_float2(l_part[h], l_part[h + 1]), pp);
        l_part[h] = ls.x;
        l_part[h + 1] = ls.y;
        const __nv_bfloat162 hi = __floats2bfloat162_rn(pp.x, pp.y);
        const float2 lo = f32x2_sub(pp, __bfloat1622float2(hi));
        pk[h >> 1] = *reinterpret_cast<const uint32_t*>(&hi);
        pl[h >> 1] = pack_bf16x2(lo.x, lo.y);
      }
      // P^T row: 64 heads x bf16 = 128 B; this half owns units ch*4 .. ch*4+3.  Keys 0..63: hi in
      // the P slot's row r, lo in row r + 64; keys 64..127: hi in row r - 64 of the slot before it.
      const uint32_t hi_row = (qd < 2) ? sP + (uint32_t)r * 128u : sPhi2 + (uint32_t)(r - 64) * 128u;
#pragma unroll
      for (int uu = 0; uu < 4; ++uu)
        st_shared_v4(hi_row + (((ch * 4 + uu) ^ (r & 7)) << 4), pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2],
                     pk[4 * uu + 3]);
      if (qd < 2) {
#pragma unroll
        for (int uu = 0; uu < 4; ++uu)
          st_shared_v4(sP + sw128_off(r + 64, ch * 4 + uu), pl[4 * uu], pl[4 * uu + 1], pl[4 * uu + 2], pl[4 * uu + 3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p);
      // Rows 0..63 of channel pair m are free once the first key half of the pair is multiplied: the
      // next tile's rows 0..63 of the pair are gathered then.  Once the last pair's are (bar_pvh), the
      // lo part of key rows 64..127 goes into the P slot's rows 0..63.
      int rix[4];
      if (more) check_rows(nraw, rix);
      {
        bool okh = true, plo_done = false;
#pragma unroll 1
        for (int m = 0; m < kDv / 128; ++m) {
          okh = okh && mbar_wait(m < 3 ? bar_pvp + 8 * m : bar_pvh, i & 1, s_abort, err, wait_limit);
          // the P_lo move is on the tensor core's path: done as soon as the whole first half is read,
          // tested between the gathers of the pairs (the gathers run behind the MMAs)
          if (qd >= 2 && !plo_done && (m == 3 || (okh && warp_all(mbar_test(bar_pvh, i & 1))))) {
            if (okh) {
#pragma unroll
              for (int uu = 0; uu < 4; ++uu)
                st_shared_v4(sP + sw128_off(r - 64, ch * 4 + uu), pl[4 * uu], pl[4 * uu + 1], pl[4 * uu + 2],
                             pl[4 * uu + 3]);
              fence_proxy_async_smem();
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_plo);
            plo_done = true;
          }
          if (more && okh) {
            gather_half<DQK>(sKV + (2 * m) * L::KV_CHUNK, kv, 2 * m, tid, rix, 0);
            gather_half<DQK>(sKV + (2 * m + 1) * L::KV_CHUNK, kv, 2 * m + 1, tid, rix, 0);
          }
        }
        if (named_bar_or(bar_id, 128, !okh)) { aborted = true; break; }
      }
      if (more) {
        // rows 64..127 of channel pair m once P.V has read them, and the RoPE chunk (which
        // holds P) once P.V is complete
        for (int m = 0; m < kDv / 128 && !aborted; ++m) {
          if (!mbar_wait(m < 3 ? bar_pvm + 8 * m : bar_pv, i & 1, s_abort, err, wait_limit)) {
            aborted = true;
            break;
          }
#pragma unroll
          for (int c = 2 * m; c < 2 * m + 2; ++c) {
            gather_half<DQK>(sKV + c * L::KV_CHUNK, kv, c, tid, rix, 1);
            cp_async_arrive(bar_kv + 8 * c);  // covers this thread's copies of both halves
          }
        }
        if (!aborted && NCH == 9) gather_chunk<DQK>(sP, kv, 8, tid, rix, bar_kv + 8 * 8);
        if (named_bar_or(bar_id, 128, aborted)) { aborted = true; break; }
      }
    }
    if (!aborted && ntiles > 0) {
      const bool got = mbar_wait(bar_pv, (ntiles - 1) & 1, s_abort, err, wait_limit);
      aborted = named_bar_or(bar_id, 128, !got);
      tc_fence_after();
    }
    // after an abort some gathers may still be landing: none may land once the epilogue reuses the tile
    asm volatile("cp.async.wait_all;" ::: "memory");
    // ---- epilogue: l per head, lse, out = O^T / l ----
    const float lsum = warp_transpose_reduce<false>(l_part, lane);
    named_bar(bar_id, 128);  // everyone is done reading s_red / s_stat of the loop
    s_red[qd * 64 + ch * 32 + lane] = lsum;
    named_bar(bar_id, 128);
    const float mh = s_stat[ch * 32 + lane];
    const int hl = hg * kHeads + ch * 32 + lane;
    // the sink's own term, relative to the final running max (which started at the sink)
    const float s2 = (sink != nullptr && hl < H) ? __ldg(sink + hl) * 1.4426950408889634f : -INFINITY;
    const float lsink = (s2 > -INFINITY) ? exp2f(s2 - mh) : 0.f;  // a -inf sink is no sink
    const float lt = s_red[ch * 32 + lane] + s_red[64 + ch * 32 + lane] + s_red[128 + ch * 32 + lane] +
                     s_red[192 + ch * 32 + lane] + lsink;
    if (qd == 0 && hl < H) lse[(size_t)t * H + hl] = (lt > 0.f) ? (mh * 0.69314718055994531f + logf(lt)) : -INFINITY;
    if (qd == 0) s_lsum[ch * 32 + lane] = lt;
    named_bar(bar_id, 128);
    float inv[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) {
      const float l = s_lsum[ch * 32 + h];
      inv[h] = (l > 0.f) ? 1.f / l : 0.f;
    }
    // stage out (and its residual) as [64 heads][512] bf16 in the free tile region
    uint8_t* stage = smem + L::OFF_KV;
    uint8_t* stage_lo = stage + kHeads * kDv * 2;
#pragma unroll 1
    for (int mt = 0; mt < kDv / 128; ++mt) {
      uint32_t ov[32];
      if (ntiles > 0 && !aborted) {
        if (mt < 3) {  // O = hi + lo
          uint32_t ol[32];
          tmem_ld32(tmem_addr(tO + mt * 128, qd * 32, ch * 32), ov);
          tmem_ld32(tmem_addr(tO + mt * 128 + 64, qd * 32, ch * 32), ol);
          tmem_ld_wait();
#pragma unroll
          for (int h = 0; h < 32; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) + __uint_as_float(ol[h]));
        } else {
          tmem_ld32(tmem_addr(tO3, qd * 32, ch * 32), ov);
          tmem_ld_wait();
        }
      } else {
#pragma unroll
        for (int h = 0; h < 32; ++h) ov[h] = 0u;
      }
      const int c = mt * 128 + qd * 32 + lane;
#pragma unroll
      for (int h = 0; h < 32; ++h) {
        const float o = __uint_as_float(ov[h]) * inv[h];
        const __nv_bfloat16 hi = __float2bfloat16_rn(o);
        reinterpret_cast<__nv_bfloat16*>(stage)[(ch * 32 + h) * kDv + c] = hi;
        if (out_lo) reinterpret_cast<__nv_bfloat16*>(stage_lo)[(ch * 32 + h) * kDv + c] =
            __float2bfloat16_rn(o - __bfloat162float(hi));
      }
    }
    named_bar(3, kWorkers);
    const int hcount = min(kHeads, H - hg * kHeads);
    const size_t gbase = ((size_t)t * H + hg * kHeads) * kDv;
    const uint64_t pol = l2_evict_first_policy();  // out and out_lo are written once
    for (int u = tid; u < hcount * (kDv / 8); u += kWorkers) {
      stg16_hint(reinterpret_cast<uint4*>(out + gbase) + u, reinterpret_cast<const uint4*>(stage)[u], pol);
      if (out_lo) stg16_hint(reinterpret_cast<uint4*>(out_lo + gbase) + u, reinterpret_cast<const uint4*>(stage_lo)[u], pol);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

constexpr int kTileF = 64;  // top-k slots per tile of the few-heads kernel (S^T's MMA M)

// misc offsets of the few-heads kernel (bytes), after its barriers:
constexpr int F_RED = 256;    // float [4 quadrants][NH]: per-quadrant maxima and sums
constexpr int F_STAT = 768;   // float [NH]: running max per head (log2 units)
constexpr int F_LSUM = 1024;  // float [NH]: softmax denominator per head

// P element (row n of the [hi | lo] operand, key r < 64) in the K-major 128B-swizzled layout:
// row n of 128 bytes, 16-byte unit r / 8 swizzled with the row.
template <int NH>
__device__ __forceinline__ uint32_t p_off(int n, int r) {
  return (uint32_t)(n * 128 + ((((r >> 3) ^ (n & 7))) << 4) + (r & 7) * 2);
}

// Transposing butterfly over N values (N a power of two <= 32): v[0..N-1] per lane (lane = key,
// index = head) -> lane l returns the reduction over the warp's 32 keys of head l % N.
template <int N, bool MAX>
__device__ __forceinline__ float warp_transpose_reduce_n(float (&v)[N], int lane) {
#pragma unroll
  for (int o = 16; o >= N; o >>= 1) {
#pragma unroll
    for (int i = 0; i < N; ++i) {
      const float x = __shfl_xor_sync(0xffffffffu, v[i], o);
      v[i] = MAX ? fmaxf(v[i], x) : v[i] + x;
    }
  }
#pragma unroll
  for (int o = N / 2; o >= 1; o >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < o; ++i) {
      float send = upper ? v[i] : v[i + o];
      float keep = upper ? v[i + o] : v[i];
      float recv = __shfl_xor_sync(0xffffffffu, send, o);
      v[i] = MAX ? fmaxf(keep, recv) : keep + recv;
    }
  }
  return v[0];
}

// 16 TMEM lanes x 64 bits, 4 times (the 16x64b shape): thread t of the warp gets lane base + (t >> 2) +
// 8 (t & 1) and the columns c + 2j + ((t >> 1) & 1), j = 0..3, of the address (lane base, c).
__device__ __forceinline__ void tmem_ld16x64b_x4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.16x64b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld16x64b_x2(uint32_t taddr, uint32_t (&r)[2]) {  // columns c + (t >> 1) & 1, + 2
  asm volatile("tcgen05.ld.sync.aligned.16x64b.x2.b32 {%0, %1}, [%2];" : "=r"(r[0]), "=r"(r[1]) : "r"(taddr));
}
template <int N>
__device__ __forceinline__ void tmem_ld16x64b(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 4) tmem_ld16x64b_x4(taddr, r);
  else tmem_ld16x64b_x2(taddr, r);
}
// 32 lanes x 32 bits, 4 columns (32x32b.x4): thread i gets lane base + i, columns c .. c + 3
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, uint32_t (&r)[4]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const uint32_t (&r)[4]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(r[0]), "r"(r[1]),
               "r"(r[2]), "r"(r[3])
               : "memory");
}
// NHH consecutive columns of the warp's 32 lanes (NHH = 4, 8 or 16)
template <int N>
__device__ __forceinline__ void tmem_ld_n(uint32_t taddr, uint32_t (&r)[N]) {
  if constexpr (N == 4) tmem_ld4(taddr, r);
  else if constexpr (N == 8) tmem_ld8(taddr, r);
  else tmem_ld16(taddr, r);
}
template <int N>
__device__ __forceinline__ void tmem_st_n(uint32_t taddr, const uint32_t (&r)[N]) {
  if constexpr (N == 4) tmem_st4(taddr, r);
  else if constexpr (N == 8) tmem_st8(taddr, r);
  else tmem_st16(taddr, r);
}

// ---------------------------------------------------------------------------
// Few heads (H <= 16): the same computation with NH = 16 heads per CTA on the
// MMA's N side instead of 64 (so that H = 8 does not multiply 56 zero heads)
// and 64-key tiles.  With so few heads the tensor core has little to do per
// key, and the tile is bound by its MMA instructions (48 small ones per 64
// keys), by shared-memory traffic and by the gathers, not by the arithmetic.
// So one CTA per SM holds a ring of R tiles (R = 3 at width 512, 2 at 576),
// filled by four gather warps (a slot is refilled once P.V of the tile it held
// is done), and three warps issue the MMAs: two form S^T of a tile from half
// the channel chunks each, into two TMEM partials that the softmax adds, and
// one forms P.V.  S^T is double-buffered in TMEM and runs up to two tiles
// ahead of the softmax; P is double-buffered in shared memory.  A rescale of O
// at tile i waits for P.V(i - 1) explicitly.
//  * S^T of a tile is an M = 64 MMA: key row 16q + i lands in TMEM lane 32q + i
//    (i < 16) of lane quadrant q.  The softmax reads it with the 16x64b shape,
//    which spreads those 16 lanes over all 32 threads of the warp (two threads
//    per key, alternate columns): each thread takes one key and 4 heads.
//  * P^T is split into bf16 hi + lo, both halves side by side in one K-major
//    operand of 2 NH rows ([hi heads | lo heads], 64 keys along K), so one P.V
//    MMA (N = 2 NH, M = 128 channels) forms O_hi and O_lo together; the
//    epilogue adds them.
// Warps: 0 and 14 issue S^T, 1-8 run the softmax and the epilogue, 9-12 gather,
// 13 issues P.V.
// ---------------------------------------------------------------------------
constexpr int kRingGather = 128;                       // gather threads (warps 9-12)
constexpr int kRingRows = kTileF / (kRingGather / 8); // rows of a tile per gather thread
constexpr int kRingThreads = 32 + kWorkers + kRingGather + 64;  // + the P.V issuer (warp 13), S^T issuer 2 (14)

template <int DQK, int NH>
struct SmemRing {
  static constexpr int NCH = DQK / 64;
  static constexpr int R = (DQK == 512) ? 3 : 2;        // tiles in the ring
  static constexpr int Q_CHUNK = NH * 128;
  static constexpr int KV_CHUNK = kTileF * 128;
  static constexpr int SLOT = NCH * KV_CHUNK;
  static constexpr int P_BLOCK = 2 * NH * 128;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_KV = (NCH * Q_CHUNK + 1023) / 1024 * 1024;
  static constexpr int OFF_P = OFF_KV + R * SLOT;        // two P buffers
  static constexpr int OFF_MISC = OFF_P + 2 * P_BLOCK;
  static constexpr int MISC = 2048;
  static constexpr int TOTAL = OFF_MISC + MISC + 1024;  // + alignment slack
  static_assert(TOTAL <= 232448, "shared memory budget");
  static_assert(2 * NH * kDv * 2 <= SLOT, "output staging fits in slot 0");
  static_assert(NH <= 16, "TMEM layout: S^T partials of 16 columns");
};
// misc layout (bytes): barriers, then the statistics at the offsets above
constexpr int RB_KV = 0, RB_PV = 32, RB_S = 64, RB_P = 80, RB_FIN = 96;  // [R], [R], [2], [2], [3]
constexpr int RM_TMEM = 128, RM_NEFF = 132, RM_ABORT = 136;
static_assert(RB_FIN + 24 <= RM_TMEM && RM_ABORT + 4 <= F_RED, "ring misc layout");

template <int DQK, int NH>
__global__ void __launch_bounds__(kRingThreads, 1)
    sparse_mla_fwd_ring_kernel(const __nv_bfloat16* __restrict__ kv, const __nv_bfloat16* __restrict__ q,
                               const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ topk_len, int T,
                               int Tk, int H, int K, float sl2e, const float* __restrict__ sink,
                               __nv_bfloat16* __restrict__ out, __nv_bfloat16* __restrict__ out_lo,
                               float* __restrict__ lse, int* __restrict__ err, long long wait_limit) {
  using L = SmemRing<DQK, NH>;
  constexpr int NCH = L::NCH, R = L::R;
  constexpr int NHH = NH / 2;  // heads per softmax thread
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + L::OFF_Q);
  const uint32_t sKV = smem_u32(smem + L::OFF_KV);
  const uint32_t sP = smem_u32(smem + L::OFF_P);
  uint8_t* misc = smem + L::OFF_MISC;
  const uint32_t bar_kv = smem_u32(misc + RB_KV), bar_pv = smem_u32(misc + RB_PV);
  const uint32_t bar_s = smem_u32(misc + RB_S), bar_p = smem_u32(misc + RB_P);
  const uint32_t bar_fin = smem_u32(misc + RB_FIN);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + RM_TMEM);
  int* s_neff = reinterpret_cast<int*>(misc + RM_NEFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + RM_ABORT);
  float* s_red = reinterpret_cast<float*>(misc + F_RED);
  float* s_stat = reinterpret_cast<float*>(misc + F_STAT);
  float* s_lsum = reinterpret_cast<float*>(misc + F_LSUM);

  const int t = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const bool worker = warp >= 1 && warp <= 8;
  const int32_t* idx_row = topk_idx + (size_t)t * K;

  if (threadIdx.x == 0) {
    for (int s = 0; s < R; ++s) {
      mbar_init(bar_kv + 8 * s, kRingGather);
      mbar_init(bar_pv + 8 * s, 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar_s + 8 * b, 2);  // both S^T partials
      mbar_init(bar_p + 8 * b, 8);
    }
    for (int f = 0; f < 3; ++f) mbar_init(bar_fin + 8 * f, 1);
    *s_neff = 0;
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(s_tmem), 256);
    tmem_relinquish();
  }
  __syncthreads();

  const int tid = threadIdx.x - 32;  // worker id 0..255
  // ---- valid prefix length and Q staging (workers) ----
  if (worker) {
    if (topk_len != nullptr) {
      if (tid == 0) {
        int n = topk_len[t];
        *s_neff = n < 0 ? 0 : (n > K ? K : n);
      }
    } else {
      int last = 0;
      for (int j = tid; j < K; j += kWorkers)
        if (idx_row[j] >= 0) last = j + 1;
      if (last) atomicMax(s_neff, last);
    }
    if (tid < NH) {  // running max per head (log2 units), from the sink logit when there is one
      s_stat[tid] = (sink != nullptr && tid < H) ? __ldg(sink + tid) * 1.4426950408889634f : -INFINITY;
    }
    constexpr int UNITS = NH * NCH * 8;
    const uint64_t pol = l2_evict_first_policy();
    for (int u = tid; u < UNITS; u += kWorkers) {
      const int hh = u / (NCH * 8);
      const int rem = u - hh * (NCH * 8);
      const int c = rem >> 3, uc = rem & 7;
      const bool ok = hh < H;
      cp_async16_hint(sQ + c * L::Q_CHUNK + sw128_off(hh, uc),
                      q + (ok ? ((size_t)t * H + hh) * DQK + c * 64 + uc * 8 : 0), ok ? 16u : 0u, pol);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    fence_proxy_async_smem();
  }
  __syncthreads();
  const int n_eff = *s_neff;
  const int ntiles = (n_eff + kTileF - 1) / kTileF;
  const uint32_t tmem = *s_tmem;
  const uint32_t tS = tmem;       // S^T buffer b, partial p (channel chunks) at column 32 b + 16 p
  const uint32_t tO = tmem + 64;  // [O_hi^T | O_lo^T]: 4 channel tiles x 2 NH columns

  if (warp == 0 || warp == 14) {
    // ============ S^T issuers (the whole warp, one elected lane issues), half the channel chunks each ============
    constexpr uint32_t kIdS = idesc_bf16(kTileF, NH, false, false);  // A = KV (K-major), B = Q (K-major)
    constexpr int NCH_A = (NCH + 1) / 2;
    const int part = (warp == 0) ? 0 : 1;
    const int c0 = part ? NCH_A : 0, c1 = part ? NCH : NCH_A;
    for (int i = 0; i < ntiles; ++i) {
      const int sl = i % R;
      // S^T buffer i & 1 was last read by the softmax of tile i - 2, which then published P(i - 2)
      if (i >= 2 && !warp_all(mbar_wait(bar_p + 8 * (i & 1), ((i - 2) >> 1) & 1, s_abort, err, wait_limit))) break;
      if (!warp_all(mbar_wait(bar_kv + 8 * sl, (i / R) & 1, s_abort, err, wait_limit))) break;
      fence_proxy_async_smem();
      tc_fence_after();
      const uint32_t tSb = tS + 32 * (i & 1) + 16 * part;
      const uint64_t b00 = sdesc_sw128(sQ, 16, 1024);
#pragma unroll 1
      for (int c = c0; c < c1; ++c) {
        const uint64_t a0 = sdesc_sw128(sKV + sl * L::SLOT + c * L::KV_CHUNK, 16, 1024);
        const uint64_t b0 = b00 + (uint64_t)((c * L::Q_CHUNK) >> 4);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss_w(tSb, a0 + (uint64_t)(k * 2), b0 + (uint64_t)(k * 2), kIdS, (c != c0 || k != 0) ? 1u : 0u);
      }
      mma_commit_w(bar_s + 8 * (i & 1));
    }
    mma_commit_w(bar_fin + 8 * (1 + part));
    volatile int dummy = 0;
    mbar_wait(bar_fin + 8 * (1 + part), 0, &dummy, err);
    __syncwarp();
  } else if (warp == 13) {
    // ======================= P.V issuer: O^T += V^T [P_hi | P_lo] per tile =======================
    constexpr uint32_t kIdPV = idesc_bf16(128, 2 * NH, true, false);  // A = V^T (MN-major), B = [P_hi|P_lo]
    for (int i = 0; i < ntiles; ++i) {
      if (!warp_all(mbar_wait(bar_p + 8 * (i & 1), (i >> 1) & 1, s_abort, err, wait_limit))) break;
      tc_fence_after();
      const uint64_t va0 = sdesc_sw128(sKV + (i % R) * L::SLOT, L::KV_CHUNK, 1024);
      const uint64_t pb0 = sdesc_sw128(sP + (i & 1) * L::P_BLOCK, 16, 1024);
      constexpr uint64_t kPair = (2 * L::KV_CHUNK) >> 4;  // descriptor step between channel pairs
#pragma unroll
      for (int m = 0; m < kDv / 128; ++m)
#pragma unroll
        for (int k = 0; k < kTileF / 16; ++k)
          mma_ss_w(tO + m * 2 * NH, va0 + m * kPair + (uint64_t)(k * 128), pb0 + (uint64_t)(k * 2), kIdPV,
                   (i > 0 || k > 0) ? 1u : 0u);
      mma_commit_w(bar_pv + 8 * (i % R));  // the slot and P buffer i & 1 are free
    }
    mma_commit_w(bar_fin);
    volatile int dummy = 0;
    mbar_wait(bar_fin, 0, &dummy, err);
    __syncwarp();
  } else if (!worker) {
    // ======================= gather warps (9-12): the ring's slots, a tile at a time =======================
    const int gt = threadIdx.x - 32 - kWorkers;  // 0..kRingGather-1
    const int uc = gt & 7;
    constexpr int kRowStep = kRingGather / 8;
    auto load_raw = [&](int i, int (&raw)[kRingRows]) {
#pragma unroll
      for (int e = 0; e < kRingRows; ++e) {
        const int j = i * kTileF + (gt >> 3) + kRowStep * e;
        raw[e] = (j < n_eff) ? __ldg(idx_row + j) : -1;
      }
    };
    int raw[kRingRows];
#pragma unroll
    for (int e = 0; e < kRingRows; ++e) raw[e] = -1;
    if (ntiles > 0) load_raw(0, raw);
    for (int i = 0; i < ntiles; ++i) {
      const int sl = i % R;
      int rix[kRingRows];
#pragma unroll
      for (int e = 0; e < kRingRows; ++e) {
        rix[e] = (raw[e] >= 0 && raw[e] < Tk) ? raw[e] : -1;
        if (raw[e] < -1 || raw[e] >= Tk) record_error(err, DSA_ERR_DEVICE_INDEX);
      }
      if (i + 1 < ntiles) load_raw(i + 1, raw);
      // the slot's previous tile (i - R) has been multiplied: P.V done (its S^T came before)
      if (i >= R && !mbar_wait(bar_pv + 8 * sl, ((i - R) / R) & 1, s_abort, err, wait_limit)) break;
      const uint32_t dst = sKV + sl * L::SLOT;
#pragma unroll
      for (int c = 0; c < NCH; ++c)
#pragma unroll
        for (int e = 0; e < kRingRows; ++e) {
          const int r = (gt >> 3) + kRowStep * e;
          const bool ok = rix[e] >= 0;
          cp_async16(dst + c * L::KV_CHUNK + sw128_off(r, uc), kv + (ok ? (size_t)rix[e] * DQK + c * 64 + uc * 8 : 0),
                     ok ? 16u : 0u);
        }
      cp_async_arrive(bar_kv + 8 * sl);
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else {
    // ======================= softmax + epilogue =======================
    const int wk = warp - 1;       // 0..7
    const int qd = warp & 3;       // TMEM lane quadrant this warp may access
    const int ch = wk >> 2;        // head half: heads ch*NHH .. ch*NHH+NHH-1
    // S^T's 16 keys of the quadrant over all 32 threads (16x64b loads): this thread's key row and its
    // NQ heads ch*NHH + par + 2j
    constexpr int NQ = NHH / 2;
    const int par = (lane >> 1) & 1;
    const int r = qd * 16 + (lane >> 2) + 8 * (lane & 1);  // key row of the tile
    const int bar_id = 1 + ch;     // named barrier of the 128 threads of this half
    float l_part[NQ];
#pragma unroll
    for (int j = 0; j < NQ; ++j) l_part[j] = 0.f;
    // per-head reduction over the warp's 16 keys: the lanes of one column parity hold the same heads
    auto reduce_keys = [&](float v, bool is_max) -> float {
#pragma unroll
      for (int o = 1; o <= 16; o <<= 1) {
        if (o == 2) continue;
        const float x = __shfl_xor_sync(0xffffffffu, v, o);
        v = is_max ? fmaxf(v, x) : v + x;
      }
      return v;
    };
    bool aborted = false;
    int ixw_next = (ntiles > 0 && r < n_eff) ? __ldg(idx_row + r) : -1;
    for (int i = 0; i < ntiles; ++i) {
      const int ixw = ixw_next;
      {
        const int jn = (i + 1) * kTileF + r;
        ixw_next = (i + 1 < ntiles && jn < n_eff) ? __ldg(idx_row + jn) : -1;
      }
      const bool got = mbar_wait(bar_s + 8 * (i & 1), (i >> 1) & 1, s_abort, err, wait_limit);
      // P buffer i & 1 was last read by P.V(i - 2), long done: waited here, so that the one barrier below
      // also covers it
      const bool okp = (i < 2) || mbar_wait(bar_pv + 8 * ((i - 2) % R), ((i - 2) / R) & 1, s_abort, err, wait_limit);
      const bool bad = !got || !okp;  // (TMEM is still read below: a stale value is harmless, the tile is dropped)
      tc_fence_after();
      uint32_t sv[NQ], sw[NQ];  // the two partial sums of S^T
      tmem_ld16x64b<NQ>(tmem_addr(tS + 32 * (i & 1) + ch * NHH, qd * 32, 0), sv);
      tmem_ld16x64b<NQ>(tmem_addr(tS + 32 * (i & 1) + 16 + ch * NHH, qd * 32, 0), sw);
      tmem_ld_wait();
      const bool valid = ixw >= 0 && ixw < Tk;
      float z[NQ];
#pragma unroll
      for (int j = 0; j < NQ; ++j) z[j] = valid ? (__uint_as_float(sv[j]) + __uint_as_float(sw[j])) * sl2e : -INFINITY;
      bool mine = (i == 0);  // the first tile always sets the running max
      if (!mine) {
#pragma unroll
        for (int j = 0; j < NQ; ++j) mine |= z[j] > s_stat[ch * NHH + par + 2 * j] + kRescaleThreshold;
      }
      // one barrier of the half per tile in the common case; a rescale, the first tile or an abort takes a
      // second one to tell them apart (every thread of the half leaves together, or none does)
      bool need = false;
      if (named_bar_or(bar_id, 128, mine || bad)) {
        if (named_bar_or(bar_id, 128, bad)) { aborted = true; break; }
        need = true;
      }
      if (need) {
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
          const float wmax = reduce_keys(z[j], true);
          if ((lane & ~2) == 0) s_red[qd * NH + ch * NHH + par + 2 * j] = wmax;
        }
        named_bar(bar_id, 128);
        // old and new running max of every head of the half (all of them: O is rescaled per head below)
        float mo[NHH], mn[NHH], alpha[NHH];
        bool any = false;
#pragma unroll
        for (int h = 0; h < NHH; ++h) {
          const int hh = ch * NHH + h;
          const float bm = fmaxf(fmaxf(s_red[hh], s_red[NH + hh]), fmaxf(s_red[2 * NH + hh], s_red[3 * NH + hh]));
          mo[h] = s_stat[hh];
          mn[h] = fmaxf(mo[h], bm);
          alpha[h] = (mo[h] == -INFINITY) ? 0.f : exp2f(mo[h] - mn[h]);
          any |= (i > 0) && (alpha[h] != 1.f);
        }
        named_bar(bar_id, 128);
        if (qd == 0 && lane == 0) {
#pragma unroll
          for (int h = 0; h < NHH; ++h) s_stat[ch * NHH + h] = mn[h];
        }
#pragma unroll
        for (int j = 0; j < NQ; ++j) l_part[j] *= par ? alpha[2 * j + 1] : alpha[2 * j];
        bool okw = true;
        if (any) {
          // O holds the products through tile i - 1 once P.V(i - 1) is done
          okw = mbar_wait(bar_pv + 8 * ((i - 1) % R), ((i - 1) / R) & 1, s_abort, err, wait_limit);
          if (okw) {
            tc_fence_after();
#pragma unroll 1
            for (int mt = 0; mt < kDv / 128; ++mt) {
#pragma unroll
              for (int part = 0; part < 2; ++part) {
                const uint32_t ta = tmem_addr(tO + mt * 2 * NH + part * NH + ch * NHH, qd * 32, 0);
                uint32_t ov[NHH];
                tmem_ld_n<NHH>(ta, ov);
                tmem_ld_wait();
#pragma unroll
                for (int h = 0; h < NHH; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
                tmem_st_n<NHH>(ta, ov);
              }
            }
            tmem_st_wait();
          }
        }
        // (also orders the s_stat update before every thread's reads below)
        if (named_bar_or(bar_id, 128, !okw)) { aborted = true; break; }
      }
      const uint32_t sPb = sP + (i & 1) * L::P_BLOCK;
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        const int n = ch * NHH + par + 2 * j;
        const float mh = s_stat[n];
        const float mu = (mh == -INFINITY) ? 0.f : mh;
        const float pv = exp2f(z[j] - mu);
        l_part[j] += pv;
        const __nv_bfloat16 hi = __float2bfloat16_rn(pv);
        const __nv_bfloat16 lo = __float2bfloat16_rn(pv - __bfloat162float(hi));
        st_shared_u16(sPb + p_off<NH>(n, r), __bfloat16_as_ushort(hi));
        st_shared_u16(sPb + p_off<NH>(NH + n, r), __bfloat16_as_ushort(lo));
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p + 8 * (i & 1));
    }
    if (!aborted && ntiles > 0) {
      const bool got = mbar_wait(bar_pv + 8 * ((ntiles - 1) % R), ((ntiles - 1) / R) & 1, s_abort, err, wait_limit);
      aborted = named_bar_or(bar_id, 128, !got);
      tc_fence_after();
    }
    // ---- epilogue: l per head, lse, out = (O_hi + O_lo)^T / l ----
    named_bar(bar_id, 128);  // everyone is done reading s_red / s_stat of the loop
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      const float lsum = reduce_keys(l_part[j], false);
      if ((lane & ~2) == 0) s_red[qd * NH + ch * NHH + par + 2 * j] = lsum;
    }
    named_bar(bar_id, 128);
    if (qd == 0 && lane < NHH) {
      const int hh = ch * NHH + lane;
      const float mh = s_stat[hh];
      const float s2 = (sink != nullptr && hh < H) ? __ldg(sink + hh) * 1.4426950408889634f : -INFINITY;
      const float lsink = (s2 > -INFINITY) ? exp2f(s2 - mh) : 0.f;
      const float lt = s_red[hh] + s_red[NH + hh] + s_red[2 * NH + hh] + s_red[3 * NH + hh] + lsink;
      if (hh < H) lse[(size_t)t * H + hh] = (lt > 0.f) ? (mh * 0.69314718055994531f + logf(lt)) : -INFINITY;
      s_lsum[hh] = lt;
    }
    named_bar(bar_id, 128);
    float inv[NHH];
#pragma unroll
    for (int h = 0; h < NHH; ++h) {
      const float l = s_lsum[ch * NHH + h];
      inv[h] = (l > 0.f) ? 1.f / l : 0.f;
    }
    // staging in slot 0 of the ring: every product is done, and no gather is in flight (every tile's
    // copies landed before its S^T)
    uint8_t* stage = smem + L::OFF_KV;
    uint8_t* stage_lo = stage + NH * kDv * 2;
#pragma unroll 1
    for (int mt = 0; mt < kDv / 128; ++mt) {
      uint32_t oh[NHH], ol[NHH];
      if (ntiles > 0 && !aborted) {
        const uint32_t ta = tmem_addr(tO + mt * 2 * NH + ch * NHH, qd * 32, 0);
        tmem_ld_n<NHH>(ta, oh);
        tmem_ld_n<NHH>(ta + NH, ol);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int h = 0; h < NHH; ++h) oh[h] = ol[h] = 0u;
      }
      const int c = mt * 128 + qd * 32 + lane;
#pragma unroll
      for (int h = 0; h < NHH; ++h) {
        const float o = (__uint_as_float(oh[h]) + __uint_as_float(ol[h])) * inv[h];
        const __nv_bfloat16 hi = __float2bfloat16_rn(o);
        reinterpret_cast<__nv_bfloat16*>(stage)[(ch * NHH + h) * kDv + c] = hi;
        if (out_lo) reinterpret_cast<__nv_bfloat16*>(stage_lo)[(ch * NHH + h) * kDv + c] =
            __float2bfloat16_rn(o - __bfloat162float(hi));
      }
    }
    named_bar(3, kWorkers);
    const int hcount = min(NH, H);
    const size_t gbase = (size_t)t * H * kDv;
    const uint64_t pol = l2_evict_first_policy();
    for (int u = tid; u < hcount * (kDv / 8); u += kWorkers) {
      stg16_hint(reinterpret_cast<uint4*>(out + gbase) + u, reinterpret_cast<const uint4*>(stage)[u], pol);
      if (out_lo) stg16_hint(reinterpret_cast<uint4*>(out_lo + gbase) + u, reinterpret_cast<const uint4*>(stage_lo)[u], pol);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int DQK>
dsa_status_t launch(const void* kv, const void* q, const int32_t* idx, const int32_t* len, int T, int Tk, int H,
                    int K, float scale, const float* sink, void* out, void* out_lo, float* lse, int* err,
                    cudaStream_t s) {
  const float sl2e = scale * 1.4426950408889634f;
  if (H <= 16) {  // few heads: 8 or 16 per CTA on the MMA's N side, one CTA per SM
    auto ring = [&](auto nh) -> dsa_status_t {
      constexpr int NH = decltype(nh)::value;
      using F = SmemRing<DQK, NH>;
      dsa_status_t st = configure_kernel_smem(reinterpret_cast<const void*>(sparse_mla_fwd_ring_kernel<DQK, NH>),
                                              F::TOTAL, "configuring sparse_mla_fwd_ring_kernel");
      if (st != DSA_OK) return st;
      sparse_mla_fwd_ring_kernel<DQK, NH><<<dim3(T, 1), kRingThreads, F::TOTAL, s>>>(
          reinterpret_cast<const __nv_bfloat16*>(kv), reinterpret_cast<const __nv_bfloat16*>(q), idx, len, T, Tk, H,
          K, sl2e, sink, reinterpret_cast<__nv_bfloat16*>(out), reinterpret_cast<__nv_bfloat16*>(out_lo), lse, err,
          wait_limit_cycles());
      return cuda_check(cudaGetLastError(), "launching sparse_mla_fwd_ring_kernel");
    };
    return H <= 8 ? ring(std::integral_constant<int, 8>{}) : ring(std::integral_constant<int, 16>{});
  }
  using L = Smem<DQK>;
  dsa_status_t st = configure_kernel_smem(reinterpret_cast<const void*>(sparse_mla_fwd_kernel<DQK>), L::TOTAL,
                                          "configuring sparse_mla_fwd_kernel");
  if (st != DSA_OK) return st;
  dim3 grid(T, (H + kHeads - 1) / kHeads);
  sparse_mla_fwd_kernel<DQK><<<grid, kThreads, L::TOTAL, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(kv), reinterpret_cast<const __nv_bfloat16*>(q), idx, len, T, Tk, H, K,
      sl2e, sink, reinterpret_cast<__nv_bfloat16*>(out), reinterpret_cast<__nv_bfloat16*>(out_lo), lse, err,
      wait_limit_cycles());
  return cuda_check(cudaGetLastError(), "launching sparse_mla_fwd_kernel");
}

}  // namespace fwd
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_sparse_mla_fwd_workspace_size(int32_t T, int32_t H) {
  (void)T;
  (void)H;
  return kErrorWordBytes;
}

extern "C" dsa_status_t dsa_sparse_mla_fwd(const dsa_bf16_t* q, const dsa_bf16_t* kv, const int32_t* topk_idx,
                                           const int32_t* topk_len, int32_t T, int32_t T_k, int32_t H, int32_t Dqk,
                                           int32_t Dv, int32_t K, float softmax_scale, const float* attn_sink,
                                           dsa_bf16_t* out, dsa_bf16_t* out_lo, float* lse, void* workspace,
                                           size_t workspace_bytes, dsa_stream_t stream) {
  const char* who = "dsa_sparse_mla_fwd";
  if (T < 0 || T_k < 1 || H < 1 || K < 1)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: need T >= 0, T_k >= 1, H >= 1, K >= 1 (got %d, %d, %d, %d)", who, T,
                T_k, H, K);
  if (Dqk != 576 && Dqk != 512) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Dqk must be 576 or 512 (got %d)", who, Dqk);
  if (Dv != 512) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Dv must be 512 (got %d)", who, Dv);
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: softmax_scale must be finite and > 0", who);
  if (T > 0 && (!q || !kv || !topk_idx || !out || !lse))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: null tensor pointer", who);
  if (!kv) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: kv is NULL", who);
  if (T > 0 && (!aligned16(q) || !aligned16(kv) || !aligned16(out) || (out_lo && !aligned16(out_lo))))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: q, kv, out and out_lo must be 16-byte aligned", who);
  dsa_status_t st = check_workspace(workspace, workspace_bytes, dsa_sparse_mla_fwd_workspace_size(T, H), who);
  if (st != DSA_OK) return st;
  if ((st = check_device()) != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = clear_error_word(workspace, s)) != DSA_OK) return st;
  if (T == 0) return ok();
  int* err = reinterpret_cast<int*>(workspace);
  st = (Dqk == 576) ? fwd::launch<576>(kv, q, topk_idx, topk_len, T, T_k, H, K, softmax_scale, attn_sink, out, out_lo,
                                      lse, err, s)
                    : fwd::launch<512>(kv, q, topk_idx, topk_len, T, T_k, H, K, softmax_scale, attn_sink, out, out_lo,
                                      lse, err, s);
  return st == DSA_OK ? ok() : st;
}
