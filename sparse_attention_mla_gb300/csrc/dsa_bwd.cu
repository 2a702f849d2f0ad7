// dsa_bwd.cu -- absorbed sparse MLA backward on sm_103a (tcgen05 + TMEM).
//
// For one query token t and a group of 64 heads per CTA, with P_j =
// exp(z_j - lse), D = <dO, O>, dP_j = <dO, kv[idx_j, :512]>, dS_j = P_j(dP_j - D):
//   dq[t,h,:]          = scale sum_j dS_j kv[idx_j, :]
//   dkv[idx_j, :]     += scale sum_h dS_j q[t,h,:]
//   dkv[idx_j, :512]  += sum_h P_j dO[t,h,:]
// Source: NeMo AutoModel glm_moe_dsa.kernels.cudnn_dsa,
// _CudnnSparseAttention.backward (query gradient [T, H, 576] and latent-KV
// gradient from grad_output [T, H, 512]); SkyRL PR 2423, "Summary" (query
// rows independent, key gradients sum); the forward it differentiates is
// described in "Accelerating GLM-5.2 Long-Context Training with cuDNN Fused
// DSA Kernels ...", "How DSA works".
//
// Design (sm_103a):
//  * P is recomputed from the saved lse (no running max).  D comes from a
//    small kernel; when the forward's bf16 residual of O is given, D uses the
//    unrounded O, so that sum_j dS_j = 0 holds to fp32 accuracy.
//  * All MMAs have M = 128: S^T = KV Q^T and dP^T = V dO^T (keys on M, N = 64
//    heads), dQ^T += KV^T dS^T (channels on M), dKV = dS^T Q + P^T dO (keys on
//    M, 32-channel groups).
//  * Q [64 x Dqk] and dO [64 x 512] stay in shared memory for the token; the
//    gathered tile streams twice through a 2-slot ring of 128-channel pairs
//    (once for S^T / dP^T, once for dQ^T).  The gather is 16-byte cp.async
//    issued by the 256 worker threads.
//  * dS (x scale) and P are split into bf16 hi + lo parts so that dkv is
//    accurate to about fp32 even for keys shared by many rows.  dS hi sits in
//    shared memory (B operand of dQ^T, A operand of dS^T Q); dS lo, P hi and
//    P lo are written into TMEM over the thread's own S^T / dP^T columns and
//    are A operands of the dKV products.
//  * dKV of a tile is produced 64 channels at a time into one TMEM staging
//    buffer and flushed by the workers with red.global.add.v4.f32 on the
//    gathered rows of the fp32 accumulator (reductions in L2).  While the
//    tensor core works on dKV, the workers have already issued the gather of
//    the next tile's first channel pairs.
//
// Warp roles (4 warpgroups): warp 0 issues MMAs (one thread) and owns TMEM;
// warpgroups 1-2 gather, run the softmax backward and write dq; warpgroup 3
// copies each dKV group out of TMEM, releases it and issues the L2
// reductions, so that the reductions overlap everything else.
#include <cmath>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {
namespace bwd {

constexpr int kThreads = 512;  // 4 warpgroups: MMA / math / math / flush
constexpr int kMath = 256;    // math threads (warpgroups 1 and 2)
constexpr int kTile = 128;
constexpr int kHeads = 64;
constexpr int kDv = 512;
constexpr int kGroup = 64;  // dKV channels per staging group (one 64-channel chunk)

template <int DQK>
struct Smem {
  static constexpr int NCH = DQK / 64;         // channel chunks of kv / q
  static constexpr int NP = (NCH + 1) / 2;     // channel pairs (128 channels)
  static constexpr int NG = DQK / kGroup;      // dKV groups
  static constexpr int Q_CHUNK = kHeads * 128; // 8 KiB
  static constexpr int KV_CHUNK = kTile * 128; // 16 KiB
  static constexpr int SLOT = 2 * KV_CHUNK;    // ring slot: one pair
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_DO = OFF_Q + NCH * Q_CHUNK;
  static constexpr int OFF_RING = OFF_DO + 8 * Q_CHUNK;
  static constexpr int OFF_DS = OFF_RING + 2 * SLOT;
  static constexpr int OFF_MISC = OFF_DS + KV_CHUNK;
  static constexpr int MISC = 1024;
  static constexpr int OFF_FST = OFF_MISC + MISC;  // flush transpose buffers: 4 warps x 32 rows x 64 B
  static constexpr int TOTAL = OFF_FST + 4 * 2048 + 1024;
  static_assert(TOTAL <= 232448, "shared memory budget");
  static_assert(2 * SLOT + KV_CHUNK >= kHeads * DQK * 2, "dq staging fits ring + dS");
};

// misc layout
constexpr int M_FULL = 0, M_EMPTY = 16, M_SDP = 32, M_DS = 40, M_STF = 48, M_STE = 64, M_DQ = 80, M_KVD = 88,
              M_FIN = 96;
constexpr int M_TMEM = 128, M_NEFF = 132, M_ABORT = 136;
constexpr int M_LSE = 256, M_DL = 512;  // float [64] each

// TMEM columns: dQ^T (5 x 64), S^T, dP^T, dKV staging (64)
constexpr uint32_t C_DQ = 0, C_S = 320, C_DP = 384, C_STG = 448;

// D[t,h] = <dO[t,h,:], O[t,h,:] (+ O_lo[t,h,:])> in fp32; one warp per (t, h).
__global__ void bwd_delta_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ out_lo,
                                 const __nv_bfloat16* __restrict__ dout, float* __restrict__ delta, long long rows) {
  const long long w = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (w >= rows) return;
  const uint4* o = reinterpret_cast<const uint4*>(out + w * kDv);
  const uint4* ol = out_lo ? reinterpret_cast<const uint4*>(out_lo + w * kDv) : nullptr;
  const uint4* d = reinterpret_cast<const uint4*>(dout + w * kDv);
  float acc = 0.f;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    uint4 a = __ldg(o + lane + 32 * k), b = __ldg(d + lane + 32 * k);
    uint4 c = ol ? __ldg(ol + lane + 32 * k) : make_uint4(0, 0, 0, 0);
    const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* b2 = reinterpret_cast<const __nv_bfloat162*>(&b);
    const __nv_bfloat162* c2 = reinterpret_cast<const __nv_bfloat162*>(&c);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float2 fa = __bfloat1622float2(a2[e]), fb = __bfloat1622float2(b2[e]), fc = __bfloat1622float2(c2[e]);
      acc = fmaf(fa.x + fc.x, fb.x, acc);
      acc = fmaf(fa.y + fc.y, fb.y, acc);
    }
  }
#pragma unroll
  for (int o2 = 16; o2 >= 1; o2 >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o2);
  if (lane == 0) delta[w] = acc;
}

__global__ void f32_to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, long long n4) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (long long)gridDim.x * blockDim.x) {
    float4 v = reinterpret_cast<const float4*>(src)[i];
    __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
    uint2 o;
    o.x = *reinterpret_cast<uint32_t*>(&lo);
    o.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(dst)[i] = o;
  }
}

// Gather channel pair p of the tile into a ring slot (see the forward's
// gather: 16-byte units, zero-fill for invalid / beyond-prefix rows).
template <int DQK>
__device__ __forceinline__ void gather_pair(uint32_t slot, const __nv_bfloat16* __restrict__ kv, int p, int tid,
                                            const int (&rix)[4], uint32_t bar) {
  constexpr int NCH = DQK / 64;
  const int uc = tid & 7;
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int c = 2 * p + cc;
    if (c >= NCH) break;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int r = (tid >> 3) + 32 * e;
      const bool ok = rix[e] >= 0;
      const __nv_bfloat16* src = kv + (ok ? (size_t)rix[e] * DQK + c * 64 + uc * 8 : 0);
      cp_async16(slot + cc * (kTile * 128) + sw128_off(r, uc), src, ok ? 16u : 0u);
    }
  }
  cp_async_arrive(bar);
}

template <int DQK>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_bwd_kernel(const __nv_bfloat16* __restrict__ kv, const __nv_bfloat16* __restrict__ q,
                          const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ topk_len,
                          const float* __restrict__ lse, const float* __restrict__ delta,
                          const __nv_bfloat16* __restrict__ dout, int T, int Tk, int H, int K, float scale,
                          __nv_bfloat16* __restrict__ dq, float* __restrict__ dkv, int* __restrict__ err) {
  using L = Smem<DQK>;
  constexpr int NCH = L::NCH;
  constexpr int NP = L::NP;
  constexpr int NG = L::NG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + L::OFF_Q);
  const uint32_t sDO = smem_u32(smem + L::OFF_DO);
  const uint32_t sRing = smem_u32(smem + L::OFF_RING);
  const uint32_t sDS = smem_u32(smem + L::OFF_DS);
  uint8_t* misc = smem + L::OFF_MISC;
  const uint32_t bar_full = smem_u32(misc + M_FULL), bar_empty = smem_u32(misc + M_EMPTY);
  const uint32_t bar_sdp = smem_u32(misc + M_SDP), bar_ds = smem_u32(misc + M_DS);
  const uint32_t bar_stf = smem_u32(misc + M_STF), bar_ste = smem_u32(misc + M_STE);
  const uint32_t bar_dq = smem_u32(misc + M_DQ), bar_kvd = smem_u32(misc + M_KVD), bar_fin = smem_u32(misc + M_FIN);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + M_TMEM);
  int* s_neff = reinterpret_cast<int*>(misc + M_NEFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + M_ABORT);
  float* s_lse2 = reinterpret_cast<float*>(misc + M_LSE);
  float* s_dl = reinterpret_cast<float*>(misc + M_DL);

  const int t = blockIdx.x;
  const int hg = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* idx_row = topk_idx + (size_t)t * K;
  const bool is_math = warp >= 4 && warp < 12;   // warpgroups 1, 2
  const bool is_flush = warp >= 12;              // warpgroup 3
  const int tid = threadIdx.x - 128;             // math thread id 0..255

  if (threadIdx.x == 0) {
    for (int s = 0; s < 2; ++s) {
      mbar_init(bar_full + 8 * s, kMath);
      mbar_init(bar_empty + 8 * s, 1);
    }
    mbar_init(bar_stf, 1);
    mbar_init(bar_ste, 4);
    mbar_init(bar_sdp, 1);
    mbar_init(bar_ds, 8);
    mbar_init(bar_dq, 1);
    mbar_init(bar_kvd, 1);
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

  if (is_math) {
    if (topk_len != nullptr) {
      if (tid == 0) {
        int n = topk_len[t];
        *s_neff = n < 0 ? 0 : (n > K ? K : n);
      }
    } else {
      int last = 0;
      for (int j = tid; j < K; j += kMath)
        if (idx_row[j] >= 0) last = j + 1;
      if (last) atomicMax(s_neff, last);
    }
    // Q [64 x DQK] and dO [64 x 512] -> 128B-swizzled chunks (rows = heads); heads >= H are zero.
    for (int u = tid; u < kHeads * NCH * 8; u += kMath) {
      const int hh = u / (NCH * 8), rem = u - hh * (NCH * 8), c = rem >> 3, uc = rem & 7;
      const int h = hg * kHeads + hh;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (h < H) v = __ldg(reinterpret_cast<const uint4*>(q + ((size_t)t * H + h) * DQK + c * 64 + uc * 8));
      st_shared_v4(sQ + c * L::Q_CHUNK + sw128_off(hh, uc), v.x, v.y, v.z, v.w);
    }
    for (int u = tid; u < kHeads * 8 * 8; u += kMath) {
      const int hh = u >> 6, rem = u & 63, c = rem >> 3, uc = rem & 7;
      const int h = hg * kHeads + hh;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (h < H) v = __ldg(reinterpret_cast<const uint4*>(dout + ((size_t)t * H + h) * kDv + c * 64 + uc * 8));
      st_shared_v4(sDO + c * L::Q_CHUNK + sw128_off(hh, uc), v.x, v.y, v.z, v.w);
    }
    // per-head lse (log2 units) and D, shared by every key row
    if (tid < kHeads) {
      const int hh = hg * kHeads + tid;
      s_lse2[tid] = (hh < H) ? lse[(size_t)t * H + hh] * 1.4426950408889634f : INFINITY;  // padded heads: P = 0
      s_dl[tid] = (hh < H) ? delta[(size_t)t * H + hh] : 0.f;
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  const int n_eff = *s_neff;
  const int ntiles = (n_eff + kTile - 1) / kTile;
  const uint32_t tmem = *s_tmem;

  if (warp < 4) {
    if (warp == 0 && lane == 0) {
      // ======================= MMA issuer =======================
      constexpr uint32_t kIdKK = idesc_bf16(128, 64, false, false);      // S^T, dP^T
      constexpr uint32_t kIdMM = idesc_bf16(128, 64, true, true);        // dQ^T
      constexpr uint32_t kIdKM = idesc_bf16(128, kGroup, false, true);   // dKV: A (smem/TMEM) x B MN-major
      int L_cnt = 0, G = 0;
      bool stop = false;
      for (int i = 0; i < ntiles && !stop; ++i) {
        if (i > 0) {  // the previous tile's dKV reads its A operands from the S^T / dP^T columns
          if (!mbar_wait(bar_kvd, (i - 1) & 1, s_abort, err)) break;
        }
        // ---- pass A: S^T = KV Q^T, dP^T = V dO^T ----
        for (int p = 0; p < NP; ++p, ++L_cnt) {
          const int slot = L_cnt & 1;
          if (!mbar_wait(bar_full + 8 * slot, (L_cnt >> 1) & 1, s_abort, err)) { stop = true; break; }
          fence_proxy_async_smem();
          tc_fence_after();
          for (int cc = 0; cc < 2; ++cc) {
            const int c = 2 * p + cc;
            if (c >= NCH) break;
            const uint32_t a0 = sRing + slot * L::SLOT + cc * L::KV_CHUNK;
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_ss(tmem + C_S, sdesc_sw128(a0 + k * 32, 16, 1024), sdesc_sw128(sQ + c * L::Q_CHUNK + k * 32, 16, 1024),
                     kIdKK, (c | k) != 0);
            if (c < 8) {
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_ss(tmem + C_DP, sdesc_sw128(a0 + k * 32, 16, 1024),
                       sdesc_sw128(sDO + c * L::Q_CHUNK + k * 32, 16, 1024), kIdKK, (c | k) != 0);
            }
          }
          mma_commit(bar_empty + 8 * slot);
        }
        if (stop) break;
        mma_commit(bar_sdp);
        if (!mbar_wait(bar_ds, i & 1, s_abort, err)) break;
        tc_fence_after();
        // ---- pass B: dQ^T[pair p] += KV^T dS^T ----
        for (int p = 0; p < NP; ++p, ++L_cnt) {
          const int slot = L_cnt & 1;
          if (!mbar_wait(bar_full + 8 * slot, (L_cnt >> 1) & 1, s_abort, err)) { stop = true; break; }
          fence_proxy_async_smem();
          tc_fence_after();
          const uint32_t a0 = sRing + slot * L::SLOT;
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k)
            mma_ss(tmem + C_DQ + p * 64, sdesc_sw128(a0 + k * 2048, L::KV_CHUNK, 1024),
                   sdesc_sw128(sDS + k * 2048, L::KV_CHUNK, 1024), kIdMM, (i > 0 || k > 0) ? 1u : 0u);
          mma_commit(bar_empty + 8 * slot);
        }
        if (stop) break;
        // ---- dKV = (dS_hi + dS_lo)^T Q + (P_hi + P_lo)^T dO, one 64-channel chunk at a time ----
        for (int g = 0; g < NG; ++g, ++G) {
          if (!mbar_wait(bar_ste, (G & 1) ^ 1, s_abort, err)) { stop = true; break; }
          tc_fence_after();
          const uint32_t d = tmem + C_STG;
          const uint32_t qb = sQ + g * L::Q_CHUNK;
          const uint32_t ob = sDO + g * L::Q_CHUNK;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint32_t acol = (k >> 1) * 32 + (k & 1) * 8;  // heads 16k..16k+15 of a thread-half region
            const uint64_t bq = sdesc_sw128(qb + k * 2048, 16, 1024);
            mma_ss(d, sdesc_sw128(sDS + k * 32, 16, 1024), bq, kIdKM, k > 0);  // dS hi (shared memory)
            mma_ts(d, tmem + C_S + acol, bq, kIdKM, 1u);                      // dS lo
            if (g < 8) {
              const uint64_t bo = sdesc_sw128(ob + k * 2048, 16, 1024);
              mma_ts(d, tmem + C_DP + acol, bo, kIdKM, 1u);                   // P hi
              mma_ts(d, tmem + C_DP + 16 + acol, bo, kIdKM, 1u);              // P lo
            }
          }
          mma_commit(bar_stf);
        }
        mma_commit(bar_kvd);
      }
      mma_commit(bar_dq);
      mma_commit(bar_fin);
      volatile int dummy = 0;
      mbar_wait(bar_fin, 0, &dummy, err);
    }
    __syncwarp();
  } else if (is_flush) {
    // ======================= dKV flush: TMEM staging -> registers -> L2 reductions =======================
    const int qd = warp & 3;
    const int r = qd * 32 + lane;  // key row of the tile
    const uint32_t fst = smem_u32(smem + L::OFF_FST + qd * 2048);
    int G = 0;
    for (int i = 0; i < ntiles; ++i) {
      const int j = i * kTile + r;
      int ix = -1;
      if (j < n_eff) ix = __ldg(idx_row + j);
      const bool valid = ix >= 0 && ix < Tk;
      bool stop = false;
      for (int g = 0; g < NG; ++g, ++G) {
        if (!mbar_wait(bar_stf, G & 1, s_abort, err)) { stop = true; break; }
        tc_fence_after();
        uint32_t v[4][16];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) tmem_ld16(tmem_addr(tmem + C_STG + 16 * qq, qd * 32, 0), v[qq]);
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_ste);  // staging free: the next group's MMAs may start
        // Transpose 16 channels at a time through this warp's 2 KB buffer so that 4
        // lanes cover one row's 64 contiguous bytes: each reduction instruction then
        // touches 8 rows x 64 B instead of 32 rows x 16 B.
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
#pragma unroll
          for (int k = 0; k < 4; ++k)
            st_shared_v4(fst + lane * 64 + ((k ^ ((lane >> 1) & 3)) << 4), v[qq][4 * k], v[qq][4 * k + 1],
                         v[qq][4 * k + 2], v[qq][4 * k + 3]);
          __syncwarp();
#pragma unroll
          for (int st = 0; st < 4; ++st) {
            const int rl = 8 * st + (lane >> 2), u = lane & 3;
            const int ixr = __shfl_sync(0xffffffffu, valid ? ix : -1, rl);
            float4 f;
            asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                         : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                         : "r"(fst + rl * 64 + ((u ^ ((rl >> 1) & 3)) << 4))
                         : "memory");
            if (ixr >= 0) red_add_v4(dkv + (size_t)ixr * DQK + g * kGroup + 16 * qq + 4 * u, f.x, f.y, f.z, f.w);
          }
          __syncwarp();
        }
      }
      if (stop) break;
    }
  } else {
    // ======================= math warps: gather, softmax backward, dq epilogue =======================
    const int mw = warp - 4;          // 0..7
    const int qd = warp & 3;
    const int ch = mw >> 2;           // heads ch*32 .. ch*32+31
    const int r = qd * 32 + lane;     // key row of the tile
    const int bar_id = 1 + ch;
    const float sl2e = scale * 1.4426950408889634f;
    const float* lse2 = s_lse2 + ch * 32;
    const float* dl = s_dl + ch * 32;
    auto load_rows = [&](int i, int (&rix)[4]) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = i * kTile + (tid >> 3) + 32 * e;
        int v = -1;
        if (j < n_eff) {
          const int ix = __ldg(idx_row + j);
          v = (ix >= 0 && ix < Tk) ? ix : -1;
          if (ix < -1 || ix >= Tk) record_error(err, DSA_ERR_DEVICE_INDEX);
        }
        rix[e] = v;
      }
    };
    int L_cnt = 0;
    bool aborted = false;
    auto gather_pairs = [&](const int (&rix)[4], int p0, int p1) {
      for (int p = p0; p < p1; ++p, ++L_cnt) {
        const int slot = L_cnt & 1;
        if (!mbar_wait(bar_empty + 8 * slot, ((L_cnt >> 1) & 1) ^ 1, s_abort, err)) return false;
        gather_pair<DQK>(sRing + slot * L::SLOT, kv, p, tid, rix, bar_full + 8 * slot);
      }
      return true;
    };
    int rix[4], rix_next[4];
    if (ntiles > 0) {
      load_rows(0, rix);
      aborted = named_bar_or(bar_id, 128, !gather_pairs(rix, 0, NP));
    }
    for (int i = 0; i < ntiles && !aborted; ++i) {
      const bool got = mbar_wait(bar_sdp, i & 1, s_abort, err);
      if (named_bar_or(bar_id, 128, !got)) { aborted = true; break; }
      tc_fence_after();
      uint32_t sv[32], dv[32];
      tmem_ld32(tmem_addr(tmem + C_S + ch * 32, qd * 32, 0), sv);
      tmem_ld32(tmem_addr(tmem + C_DP + ch * 32, qd * 32, 0), dv);
      tmem_ld_wait();
      const int j = i * kTile + r;
      int ix = -1;
      if (j < n_eff) ix = __ldg(idx_row + j);
      const bool valid = ix >= 0 && ix < Tk;
      uint32_t ph[16], pl[16], sh[16], sl[16];
#pragma unroll
      for (int h = 0; h < 32; h += 2) {
        float p0 = 0.f, p1 = 0.f, s0 = 0.f, s1 = 0.f;
        if (valid) {
          p0 = exp2f(__uint_as_float(sv[h]) * sl2e - lse2[h]);
          p1 = exp2f(__uint_as_float(sv[h + 1]) * sl2e - lse2[h + 1]);
          s0 = scale * p0 * (__uint_as_float(dv[h]) - dl[h]);
          s1 = scale * p1 * (__uint_as_float(dv[h + 1]) - dl[h + 1]);
        }
        const __nv_bfloat162 phi = __floats2bfloat162_rn(p0, p1);
        const __nv_bfloat162 shi = __floats2bfloat162_rn(s0, s1);
        const float2 phf = __bfloat1622float2(phi), shf = __bfloat1622float2(shi);
        ph[h >> 1] = *reinterpret_cast<const uint32_t*>(&phi);
        sh[h >> 1] = *reinterpret_cast<const uint32_t*>(&shi);
        pl[h >> 1] = pack_bf16x2(p0 - phf.x, p1 - phf.y);
        sl[h >> 1] = pack_bf16x2(s0 - shf.x, s1 - shf.y);
      }
#pragma unroll
      for (int uu = 0; uu < 4; ++uu)
        st_shared_v4(sDS + sw128_off(r, ch * 4 + uu), sh[4 * uu], sh[4 * uu + 1], sh[4 * uu + 2], sh[4 * uu + 3]);
      // TMEM A operands of the dKV products, over this thread's own S^T / dP^T columns
      tmem_st16(tmem_addr(tmem + C_S + ch * 32, qd * 32, 0), sl);
      tmem_st16(tmem_addr(tmem + C_DP + ch * 32, qd * 32, 0), ph);
      tmem_st16(tmem_addr(tmem + C_DP + ch * 32 + 16, qd * 32, 0), pl);
      tmem_st_wait();
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_ds);
      bool ok = gather_pairs(rix, 0, NP);                 // pass B data
      if (ok && i + 1 < ntiles) {                         // the next tile's pass A data
        load_rows(i + 1, rix_next);
        ok = gather_pairs(rix_next, 0, NP);
#pragma unroll
        for (int e = 0; e < 4; ++e) rix[e] = rix_next[e];
      }
      aborted = named_bar_or(bar_id, 128, !ok);
    }
    // ---- dq epilogue: dQ^T (lanes = channels) -> staged [64 heads][DQK] bf16 -> coalesced stores ----
    bool have = false;
    if (!aborted && ntiles > 0) {
      const bool got = mbar_wait(bar_dq, 0, s_abort, err);
      have = !named_bar_or(bar_id, 128, !got);
      tc_fence_after();
    }
    named_bar(3, kMath);  // both halves are done with the ring before it becomes the staging area
    __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem + L::OFF_RING);
#pragma unroll 1
    for (int p = 0; p < NP; ++p) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(tmem_addr(tmem + C_DQ + p * 64 + ch * 32, qd * 32, 0), v);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int h = 0; h < 32; ++h) v[h] = 0u;
      }
      const int c = p * 128 + qd * 32 + lane;
      if (c < DQK) {
#pragma unroll
        for (int h = 0; h < 32; ++h) stage[(ch * 32 + h) * DQK + c] = __float2bfloat16_rn(__uint_as_float(v[h]));
      }
    }
    named_bar(3, kMath);
    const int hcount = min(kHeads, H - hg * kHeads);
    uint4* dst = reinterpret_cast<uint4*>(dq + ((size_t)t * H + hg * kHeads) * DQK);
    for (int u = tid; u < hcount * (DQK / 8); u += kMath) dst[u] = reinterpret_cast<const uint4*>(stage)[u];
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK>
dsa_status_t launch(const void* kv, const void* q, const int32_t* idx, const int32_t* len, const float* lse,
                    const float* delta, const void* dout, int T, int Tk, int H, int K, float scale, void* dq,
                    float* dkv, int* err, cudaStream_t s) {
  using L = Smem<DQK>;
  static bool configured = false;
  if (!configured) {
    dsa_status_t st = cuda_check(cudaFuncSetAttribute(sparse_mla_bwd_kernel<DQK>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL),
                                 "configuring sparse_mla_bwd_kernel");
    if (st != DSA_OK) return st;
    configured = true;
  }
  dim3 grid(T, (H + kHeads - 1) / kHeads);
  sparse_mla_bwd_kernel<DQK><<<grid, kThreads, L::TOTAL, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(kv), reinterpret_cast<const __nv_bfloat16*>(q), idx, len, lse, delta,
      reinterpret_cast<const __nv_bfloat16*>(dout), T, Tk, H, K, scale, reinterpret_cast<__nv_bfloat16*>(dq), dkv,
      err);
  return cuda_check(cudaGetLastError(), "launching sparse_mla_bwd_kernel");
}

}  // namespace bwd
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_sparse_mla_bwd_workspace_size(int32_t T, int32_t H) {
  const size_t delta = (size_t)(T > 0 ? T : 0) * (size_t)(H > 0 ? H : 0) * sizeof(float);
  return kErrorWordBytes + ((delta + 255) & ~size_t(255));
}

extern "C" dsa_status_t dsa_sparse_mla_bwd(const dsa_bf16_t* q, const dsa_bf16_t* kv, const int32_t* topk_idx,
                                           const int32_t* topk_len, int32_t T, int32_t T_k, int32_t H, int32_t Dqk,
                                           int32_t Dv, int32_t K, float softmax_scale, const dsa_bf16_t* out,
                                           const dsa_bf16_t* out_lo, const float* lse, const dsa_bf16_t* dout,
                                           dsa_bf16_t* dq, float* dkv_accum, int32_t accumulate, dsa_bf16_t* dkv_bf16,
                                           void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  const char* who = "dsa_sparse_mla_bwd";
  if (T < 0 || T_k < 1 || H < 1 || K < 1)
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: need T >= 0, T_k >= 1, H >= 1, K >= 1 (got %d, %d, %d, %d)", who, T,
                T_k, H, K);
  if (Dqk != 576 && Dqk != 512) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Dqk must be 576 or 512 (got %d)", who, Dqk);
  if (Dv != 512) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: Dv must be 512 (got %d)", who, Dv);
  if (accumulate != 0 && accumulate != 1) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: accumulate must be 0 or 1", who);
  if (!std::isfinite(softmax_scale) || !(softmax_scale > 0.f))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: softmax_scale must be finite and > 0", who);
  if (!kv || !dkv_accum) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: kv / dkv_accum is NULL", who);
  if (T > 0 && (!q || !topk_idx || !out || !lse || !dout || !dq))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: null tensor pointer", who);
  if (!aligned16(kv) || !aligned16(dkv_accum) ||
      (T > 0 && (!aligned16(q) || !aligned16(out) || !aligned16(dout) || !aligned16(dq) ||
                 (out_lo && !aligned16(out_lo)))))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: q, kv, out, out_lo, dout, dq and dkv_accum must be 16-byte aligned",
                who);
  if (dkv_bf16 && (reinterpret_cast<uintptr_t>(dkv_bf16) & 7u))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: dkv_bf16 must be 8-byte aligned", who);
  dsa_status_t st = check_workspace(workspace, workspace_bytes, dsa_sparse_mla_bwd_workspace_size(T, H), who);
  if (st != DSA_OK) return st;
  if ((st = check_device()) != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = clear_error_word(workspace, s)) != DSA_OK) return st;
  if (!accumulate &&
      (st = cuda_check(cudaMemsetAsync(dkv_accum, 0, (size_t)T_k * Dqk * sizeof(float), s), "zeroing dkv_accum")))
    return st;
  int* err = reinterpret_cast<int*>(workspace);
  float* delta = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) + kErrorWordBytes);
  if (T > 0) {
    const long long rows = (long long)T * H;
    bwd::bwd_delta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(
        reinterpret_cast<const __nv_bfloat16*>(out), reinterpret_cast<const __nv_bfloat16*>(out_lo),
        reinterpret_cast<const __nv_bfloat16*>(dout), delta, rows);
    if ((st = cuda_check(cudaGetLastError(), "launching bwd_delta_kernel"))) return st;
    st = (Dqk == 576) ? bwd::launch<576>(kv, q, topk_idx, topk_len, lse, delta, dout, T, T_k, H, K, softmax_scale, dq,
                                         dkv_accum, err, s)
                      : bwd::launch<512>(kv, q, topk_idx, topk_len, lse, delta, dout, T, T_k, H, K, softmax_scale, dq,
                                         dkv_accum, err, s);
    if (st != DSA_OK) return st;
  }
  if (dkv_bf16) {
    const long long n4 = (long long)T_k * Dqk / 4;
    bwd::f32_to_bf16_kernel<<<152 * 4, 256, 0, s>>>(dkv_accum, reinterpret_cast<__nv_bfloat16*>(dkv_bf16), n4);
    if ((st = cuda_check(cudaGetLastError(), "launching f32_to_bf16_kernel"))) return st;
  }
  return ok();
}

// ---------------------------------------------------------------------------
// dsa_sparse_mla_bwd_noalloc: the backward for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc: runtimes that reserve all device memory
// up front in their own pool and forbid any other allocation, or plug-ins
// loaded into a host program that owns every allocation.  They cannot provide
// the workspace dsa_sparse_mla_bwd needs (the device error word and the
// per-(row, head) D array).  This entry point takes its scratch from the
// file-scope device array below instead, so it allocates nothing.
//
// The array is a fixed 16 MiB + 256 B that every GPU which loads this library
// holds until the process exits.  Its name is only a host-side stand-in for
// the device array, so the host looks up the array's real device address with
// cudaGetSymbolAddress, once per device, on the first call made with that
// device current; that first call should therefore come before any stream
// capture.  All calls share the one array: two calls whose executions overlap
// on the GPU race on it, so callers must order them (one stream, or events).
// Each call clears the error word it uses and overwrites the D array it
// reads, so stale contents from an earlier call do not leak into the result.
// ---------------------------------------------------------------------------
#include <mutex>

namespace dsa {
namespace bwd {
constexpr size_t kNoAllocDeltaBytes = size_t(16) << 20;  // D for up to 4 Mi (row, head) pairs
constexpr size_t kNoAllocScratchBytes = kErrorWordBytes + kNoAllocDeltaBytes;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device (looked up once per device).
static dsa_status_t noalloc_scratch(void** ptr) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = 0;
  dsa_status_t st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != DSA_OK) return st;
  if (dev < 0 || dev >= 64) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if ((st = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(scratch)")) != DSA_OK)
      return st;
    addr[dev] = p;
  }
  *ptr = addr[dev];
  return DSA_OK;
}
}  // namespace bwd
}  // namespace dsa

extern "C" size_t dsa_sparse_mla_bwd_noalloc_max_rows(void) { return bwd::kNoAllocDeltaBytes / sizeof(float); }

extern "C" dsa_status_t dsa_sparse_mla_bwd_noalloc(const dsa_bf16_t* q, const dsa_bf16_t* kv, const int32_t* topk_idx,
                                                   const int32_t* topk_len, int32_t T, int32_t T_k, int32_t H,
                                                   int32_t Dqk, int32_t Dv, int32_t K, float softmax_scale,
                                                   const dsa_bf16_t* out, const dsa_bf16_t* out_lo, const float* lse,
                                                   const dsa_bf16_t* dout, dsa_bf16_t* dq, float* dkv_accum,
                                                   int32_t accumulate, dsa_bf16_t* dkv_bf16, dsa_stream_t stream) {
  const size_t need = dsa_sparse_mla_bwd_workspace_size(T, H);
  if (need > bwd::kNoAllocScratchBytes)
    return fail(DSA_ERR_WORKSPACE,
                "dsa_sparse_mla_bwd_noalloc: T*H = %lld rows x heads exceeds the built-in scratch limit of %zu "
                "(use dsa_sparse_mla_bwd with a caller workspace, or split the rows into chunks)",
                (long long)T * H, dsa_sparse_mla_bwd_noalloc_max_rows());
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  void* scratch = nullptr;
  if ((st = bwd::noalloc_scratch(&scratch)) != DSA_OK) return st;
  return dsa_sparse_mla_bwd(q, kv, topk_idx, topk_len, T, T_k, H, Dqk, Dv, K, softmax_scale, out, out_lo, lse, dout,
                            dq, dkv_accum, accumulate, dkv_bf16, scratch, bwd::kNoAllocScratchBytes, stream);
}
