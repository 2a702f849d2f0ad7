// dsa_fwd.cu -- absorbed sparse MLA forward on sm_103a (tcgen05 + TMEM + TMA).
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
//    memory with TMA tile::gather4 (4 rows x 64 channels per instruction,
//    128-byte swizzle) and used by all 64 heads of the CTA.
//  * Scores are computed transposed, S^T[key, head] = KV_tile . Q^T, so the
//    tensor-core M axis is the 128 keys of the tile and N = 64 heads
//    (M = 128 is the full-rate tcgen05 shape; the 64 heads are the shared
//    operand).  Output is accumulated transposed too, O^T[ch, head] +=
//    V^T . P^T, as four M = 128 channel tiles.  TMEM holds S^T (64 columns)
//    and O^T (256 columns); the 576-wide O of 64 heads would not fit TMEM in
//    the heads-on-M orientation.
//  * Online softmax with the running max per head; a rescale of O^T happens
//    only when some score exceeds the running max by more than 2^8 (lazy
//    rescale), otherwise P uses the stale max.
//  * P^T (bf16) is written into the shared-memory slot of the tile's RoPE
//    channels (no longer needed once S^T is done), which keeps the whole
//    working set (Q 72 KiB + tile 144 KiB) inside one SM's shared memory.
//
// Warp roles: warp 0 gathers (TMA), warp 1 issues MMAs (one thread) and owns
// TMEM, warps 2..9 run the softmax and the epilogue.
#include <cmath>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {
namespace fwd {

constexpr int kThreads = 320;
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
  static constexpr int OFF_KV = OFF_Q + NCH * Q_CHUNK;
  // P^T lives in the RoPE chunk when there is one, else in its own slot.
  static constexpr int OFF_P = (DQK == 576) ? OFF_KV + 8 * KV_CHUNK : OFF_KV + NCH * KV_CHUNK;
  static constexpr int OFF_MISC = (DQK == 576) ? OFF_KV + NCH * KV_CHUNK : OFF_P + KV_CHUNK;
  static constexpr int MISC = 2048;
  static constexpr int TOTAL = OFF_MISC + MISC + 1024;  // + alignment slack
};

// misc layout (bytes)
constexpr int M_BAR_KV = 0, M_BAR_S = 8, M_BAR_P = 16, M_BAR_O = 24, M_BAR_FIN = 32;
constexpr int M_TMEM = 64, M_NEFF = 68, M_ABORT = 72;
constexpr int M_RED = 128;         // float [4][64]
constexpr int M_STAT = 128 + 1024; // float [64]: running max per head
constexpr int M_LSUM = M_STAT + 256;  // float [64]: softmax denominator per head

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

template <int DQK>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_fwd_kernel(const __grid_constant__ CUtensorMap kv_map, const __nv_bfloat16* __restrict__ q,
                          const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ topk_len, int T, int Tk,
                          int H, int K, float sl2e, __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                          int* __restrict__ err) {
  using L = Smem<DQK>;
  constexpr int NCH = L::NCH;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQ = smem_u32(smem + L::OFF_Q);
  const uint32_t sKV = smem_u32(smem + L::OFF_KV);
  const uint32_t sP = smem_u32(smem + L::OFF_P);
  uint8_t* misc = smem + L::OFF_MISC;
  const uint32_t bar_kv = smem_u32(misc + M_BAR_KV), bar_s = smem_u32(misc + M_BAR_S);
  const uint32_t bar_p = smem_u32(misc + M_BAR_P), bar_o = smem_u32(misc + M_BAR_O);
  const uint32_t bar_fin = smem_u32(misc + M_BAR_FIN);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + M_TMEM);
  int* s_neff = reinterpret_cast<int*>(misc + M_NEFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + M_ABORT);
  float* s_red = reinterpret_cast<float*>(misc + M_RED);
  float* s_stat = reinterpret_cast<float*>(misc + M_STAT);
  float* s_lsum = reinterpret_cast<float*>(misc + M_LSUM);

  const int t = blockIdx.x;
  const int hg = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* idx_row = topk_idx + (size_t)t * K;

  if (threadIdx.x == 0) {
    mbar_init(bar_kv, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_p, 8);
    mbar_init(bar_o, 1);
    mbar_init(bar_fin, 1);
    *s_neff = 0;
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  __syncthreads();

  // ---- valid prefix length and Q staging (softmax warps) ----
  if (warp >= 2) {
    const int tid = threadIdx.x - 64;  // 0..255
    if (topk_len != nullptr) {
      if (tid == 0) {
        int n = topk_len[t];
        *s_neff = n < 0 ? 0 : (n > K ? K : n);
      }
    } else {
      int last = 0;
      for (int j = tid; j < K; j += 256)
        if (idx_row[j] >= 0) last = j + 1;
      if (last) atomicMax(s_neff, last);
    }
    if (tid < kHeads) s_stat[tid] = -INFINITY;  // running max per head (log2 units)
    // Q [64 heads, DQK] -> NCH chunks of [64 rows x 128 B], 128B swizzle; heads >= H are zero.
    constexpr int UNITS = kHeads * NCH * 8;
    for (int u = tid; u < UNITS; u += 256) {
      const int hh = u / (NCH * 8);
      const int rem = u - hh * (NCH * 8);
      const int c = rem >> 3, uc = rem & 7;
      const int h = hg * kHeads + hh;
      uint4 v = make_uint4(0, 0, 0, 0);
      if (h < H) v = __ldg(reinterpret_cast<const uint4*>(q + ((size_t)t * H + h) * DQK + c * 64 + uc * 8));
      st_shared_v4(sQ + c * L::Q_CHUNK + sw128_off(hh, uc), v.x, v.y, v.z, v.w);
    }
    fence_proxy_async_smem();
  }
  __syncthreads();
  const int n_eff = *s_neff;
  const int ntiles = (n_eff + kTile - 1) / kTile;
  // A single partial tile leaves rows it never gathers: make them finite (zero)
  // so that P = 0 times V stays 0.  Later tiles only hold stale gathered rows.
  if (ntiles == 1 && warp >= 2) {
    const int tid = threadIdx.x - 64;
    const int r0 = ((n_eff + 3) >> 2) << 2;
    const int units = (kTile - r0) * 8;
    for (int c = 0; c < NCH; ++c)
      for (int u = tid; u < units; u += 256)
        st_shared_v4(sKV + c * L::KV_CHUNK + (r0 + (u >> 3)) * 128 + ((u & 7) << 4), 0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  __syncthreads();
  const uint32_t tmem = *s_tmem;
  const uint32_t tS = tmem;        // S^T: 128 lanes x 64 columns
  const uint32_t tO = tmem + 64;   // O^T: 4 channel tiles x 64 columns

  if (warp == 0) {
    // ======================= producer: TMA gather =======================
    int issued = 0;
    for (int i = 0; i < ntiles; ++i) {
      if (i > 0 && !mbar_wait(bar_o, (i - 1) & 1, s_abort, err)) break;
      const int base = i * kTile;
      const int rem = n_eff - base;
      const int ngroups = min(32, (rem + 3) >> 2);
      if (lane == 0) mbar_expect_tx(bar_kv, (uint32_t)(ngroups * 4 * DQK * 2));
      __syncwarp();
      if (lane < ngroups) {
        int r[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const int j = base + 4 * lane + e;
          int ix = -1;
          if (j < n_eff) ix = __ldg(idx_row + j);
          if (ix < -1 || ix >= Tk) record_error(err, DSA_ERR_DEVICE_INDEX);
          r[e] = (ix >= 0 && ix < Tk) ? ix : 0;
        }
        const uint32_t dst = sKV + (4 * lane) * 128;
#pragma unroll 1
        for (int c = 0; c < NCH; ++c)
          tma_gather4(dst + c * L::KV_CHUNK, &kv_map, c * 64, r[0], r[1], r[2], r[3], bar_kv);
      }
      issued = i + 1;
    }
    // On abort, wait (bounded) for our own copies still in flight.
    if (*s_abort && issued > 0 && lane == 0) {
      volatile int dummy = 0;
      mbar_wait(bar_kv, (issued - 1) & 1, &dummy, err);
    }
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    if (lane == 0) {
      constexpr uint32_t kIdS = idesc_bf16(128, kHeads, false, false);  // A = KV (K-major), B = Q (K-major)
      constexpr uint32_t kIdPV = idesc_bf16(128, kHeads, true, true);   // A = V^T (MN-major), B = P^T (MN-major)
      for (int i = 0; i < ntiles; ++i) {
        if (!mbar_wait(bar_kv, i & 1, s_abort, err)) break;
        tc_fence_after();
#pragma unroll 1
        for (int c = 0; c < NCH; ++c) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint64_t a = sdesc_sw128(sKV + c * L::KV_CHUNK + k * 32, 16, 1024);
            const uint64_t b = sdesc_sw128(sQ + c * L::Q_CHUNK + k * 32, 16, 1024);
            mma_ss(tS, a, b, kIdS, (c | k) != 0);
          }
        }
        mma_commit(bar_s);
        if (!mbar_wait(bar_p, i & 1, s_abort, err)) break;
        tc_fence_after();
#pragma unroll 1
        for (int m = 0; m < kDv / 128; ++m) {
#pragma unroll
          for (int k = 0; k < kTile / 16; ++k) {
            const uint64_t a = sdesc_sw128(sKV + (2 * m) * L::KV_CHUNK + k * 2048, L::KV_CHUNK, 1024);
            const uint64_t b = sdesc_sw128(sP + k * 2048, L::KV_CHUNK, 1024);
            mma_ss(tO + m * kHeads, a, b, kIdPV, (i > 0 || k > 0) ? 1u : 0u);
          }
        }
        mma_commit(bar_o);
      }
      // every MMA of this CTA completes before the teardown frees TMEM
      mma_commit(bar_fin);
      volatile int dummy = 0;
      mbar_wait(bar_fin, 0, &dummy, err);
    }
    __syncwarp();
  } else {
    // ======================= softmax + epilogue =======================
    const int sw = warp - 2;          // 0..7
    const int qd = warp & 3;          // TMEM lane quadrant this warp may access
    const int ch = sw >> 2;           // head half: heads ch*32 .. ch*32+31
    const int r = qd * 32 + lane;     // key row of the tile / channel row of an O^T tile
    const int bar_id = 1 + ch;        // named barrier of the 128 threads of this half
    float m_run[32], l_part[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) {
      m_run[h] = -INFINITY;
      l_part[h] = 0.f;
    }
    bool aborted = false;
    for (int i = 0; i < ntiles; ++i) {
      const bool got = mbar_wait(bar_s, i & 1, s_abort, err);
      // every thread of the half leaves together, or none does (named barriers follow)
      if (named_bar_or(bar_id, 128, !got)) { aborted = true; break; }
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tmem_addr(tS, qd * 32, ch * 32), sv);
      tmem_ld_wait();
      const int j = i * kTile + r;
      bool valid = false;
      if (j < n_eff) {
        const int ix = __ldg(idx_row + j);
        valid = ix >= 0 && ix < Tk;
      }
      float z[32];
#pragma unroll
      for (int h = 0; h < 32; ++h) z[h] = valid ? __uint_as_float(sv[h]) * sl2e : -INFINITY;
      bool need = (i == 0);
      if (!need) {
        bool mine = false;
#pragma unroll
        for (int h = 0; h < 32; ++h) mine |= z[h] > m_run[h] + kRescaleThreshold;
        need = named_bar_or(bar_id, 128, mine);
      }
      if (need) {
        float v[32];
#pragma unroll
        for (int h = 0; h < 32; ++h) v[h] = z[h];
        const float wmax = warp_transpose_reduce<true>(v, lane);
        s_red[qd * 64 + ch * 32 + lane] = wmax;
        named_bar(bar_id, 128);
        const float bm = fmaxf(fmaxf(s_red[ch * 32 + lane], s_red[64 + ch * 32 + lane]),
                               fmaxf(s_red[128 + ch * 32 + lane], s_red[192 + ch * 32 + lane]));
        const float mn = fmaxf(s_stat[ch * 32 + lane], bm);
        named_bar(bar_id, 128);
        if (qd == 0) s_stat[ch * 32 + lane] = mn;
        named_bar(bar_id, 128);
        float alpha[32];
        bool any = false;
#pragma unroll
        for (int h = 0; h < 32; ++h) {
          const float mnew = s_stat[ch * 32 + h];
          alpha[h] = (m_run[h] == -INFINITY) ? 0.f : exp2f(m_run[h] - mnew);
          any |= (i > 0) && (alpha[h] != 1.f);
          l_part[h] *= alpha[h];
          m_run[h] = mnew;
        }
        if (any) {
          // O^T is complete for the previous tile: bar_s of this tile was
          // committed after those MMAs by the same thread.
#pragma unroll 1
          for (int mt = 0; mt < kDv / 128; ++mt) {
            uint32_t ov[32];
            const uint32_t ta = tmem_addr(tO + mt * kHeads, qd * 32, ch * 32);
            tmem_ld32(ta, ov);
            tmem_ld_wait();
#pragma unroll
            for (int h = 0; h < 32; ++h) ov[h] = __float_as_uint(__uint_as_float(ov[h]) * alpha[h]);
            tmem_st32(ta, ov);
          }
          tmem_st_wait();
        }
      }
      uint32_t pk[16];
#pragma unroll
      for (int h = 0; h < 32; h += 2) {
        const float mu0 = (m_run[h] == -INFINITY) ? 0.f : m_run[h];
        const float mu1 = (m_run[h + 1] == -INFINITY) ? 0.f : m_run[h + 1];
        const float p0 = (z[h] == -INFINITY) ? 0.f : exp2f(z[h] - mu0);
        const float p1 = (z[h + 1] == -INFINITY) ? 0.f : exp2f(z[h + 1] - mu1);
        l_part[h] += p0;
        l_part[h + 1] += p1;
        pk[h >> 1] = pack_bf16x2(p0, p1);
      }
      // P^T row r: 64 heads x bf16 = 128 B; this half owns units ch*4 .. ch*4+3.
#pragma unroll
      for (int uu = 0; uu < 4; ++uu)
        st_shared_v4(sP + sw128_off(r, ch * 4 + uu), pk[4 * uu], pk[4 * uu + 1], pk[4 * uu + 2], pk[4 * uu + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p);
    }
    if (!aborted && ntiles > 0) {
      const bool got = mbar_wait(bar_o, (ntiles - 1) & 1, s_abort, err);
      aborted = named_bar_or(bar_id, 128, !got);
      tc_fence_after();
    }
    // ---- epilogue: l per head, lse, out = O^T / l ----
    const float lsum = warp_transpose_reduce<false>(l_part, lane);
    named_bar(bar_id, 128);  // everyone is done reading s_red / s_stat of the loop
    s_red[qd * 64 + ch * 32 + lane] = lsum;
    named_bar(bar_id, 128);
    const float lt = s_red[ch * 32 + lane] + s_red[64 + ch * 32 + lane] + s_red[128 + ch * 32 + lane] +
                     s_red[192 + ch * 32 + lane];
    const float mh = s_stat[ch * 32 + lane];
    const int hl = hg * kHeads + ch * 32 + lane;
    if (qd == 0 && hl < H) lse[(size_t)t * H + hl] = (lt > 0.f) ? (mh * 0.69314718055994531f + logf(lt)) : -INFINITY;
    named_bar(bar_id, 128);
    if (qd == 0) s_lsum[ch * 32 + lane] = lt;
    named_bar(bar_id, 128);
    float inv[32];
#pragma unroll
    for (int h = 0; h < 32; ++h) {
      const float l = s_lsum[ch * 32 + h];
      inv[h] = (l > 0.f) ? 1.f / l : 0.f;
    }
    const int hbase = hg * kHeads + ch * 32;
    const int hcount = min(32, H - hbase);
#pragma unroll 1
    for (int mt = 0; mt < kDv / 128; ++mt) {
      uint32_t ov[32];
      if (ntiles > 0 && !aborted) {
        tmem_ld32(tmem_addr(tO + mt * kHeads, qd * 32, ch * 32), ov);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int h = 0; h < 32; ++h) ov[h] = 0u;
      }
      const int c = mt * 128 + qd * 32 + lane;
      __nv_bfloat16* op = out + ((size_t)t * H + hbase) * kDv + c;
#pragma unroll
      for (int h = 0; h < 32; ++h)
        if (h < hcount) op[(size_t)h * kDv] = __float2bfloat16_rn(__uint_as_float(ov[h]) * inv[h]);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int DQK>
dsa_status_t launch(const CUtensorMap& map, const void* q, const int32_t* idx, const int32_t* len, int T, int Tk,
                    int H, int K, float scale, void* out, float* lse, int* err, cudaStream_t s) {
  using L = Smem<DQK>;
  static bool configured = false;
  if (!configured) {
    dsa_status_t st = cuda_check(cudaFuncSetAttribute(sparse_mla_fwd_kernel<DQK>,
                                                      cudaFuncAttributeMaxDynamicSharedMemorySize, L::TOTAL),
                                 "configuring sparse_mla_fwd_kernel");
    if (st != DSA_OK) return st;
    configured = true;
  }
  dim3 grid(T, (H + kHeads - 1) / kHeads);
  const float sl2e = scale * 1.4426950408889634f;
  sparse_mla_fwd_kernel<DQK><<<grid, kThreads, L::TOTAL, s>>>(
      map, reinterpret_cast<const __nv_bfloat16*>(q), idx, len, T, Tk, H, K, sl2e,
      reinterpret_cast<__nv_bfloat16*>(out), lse, err);
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
                                           int32_t Dv, int32_t K, float softmax_scale, dsa_bf16_t* out, float* lse,
                                           void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
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
  if (T > 0 && (!aligned16(q) || !aligned16(kv)))
    return fail(DSA_ERR_INVALID_ARGUMENT, "%s: q and kv must be 16-byte aligned", who);
  dsa_status_t st = check_workspace(workspace, workspace_bytes, dsa_sparse_mla_fwd_workspace_size(T, H), who);
  if (st != DSA_OK) return st;
  if ((st = check_device()) != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = clear_error_word(workspace, s)) != DSA_OK) return st;
  if (T == 0) return ok();
  CUtensorMap map;
  if ((st = make_map_2d_bf16(&map, kv, (uint64_t)T_k, (uint64_t)Dqk, (uint64_t)Dqk, 64, 1)) != DSA_OK) return st;
  int* err = reinterpret_cast<int*>(workspace);
  st = (Dqk == 576) ? fwd::launch<576>(map, q, topk_idx, topk_len, T, T_k, H, K, softmax_scale, out, lse, err, s)
                    : fwd::launch<512>(map, q, topk_idx, topk_len, T, T_k, H, K, softmax_scale, out, lse, err, s);
  return st == DSA_OK ? ok() : st;
}
