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
// Design (sm_103a).  The key gradient is scattered into an fp32 accumulator
// with L2 reductions (red.global.add), one 2304-byte row per selected key and
// token; those reductions bound the kernel, so everything else is arranged
// to keep them running back to back:
//  * P is recomputed from the saved lse (no running max; an attention sink of
//    the forward is inside lse, so P needs nothing more).  D = <dO, O> comes
//    from a small kernel that streams O and dO at full memory bandwidth
//    before the main kernel starts (every CTA then finds D ready); when the
//    forward's bf16 residual of O is given, D uses O + residual, so that
//    sum_j dS_j = 0 holds to fp32 accuracy.  With a sink, the same kernel
//    adds the sink gradient -exp(sink - lse) D of each (token, head) to d_sink.
//  * Main loop, per 128-slot tile: [S^T | dP^T] = KV [Q | dO]^T (keys on the
//    MMA M axis; Q and dO chunks side by side give N = 128) into one of TWO
//    TMEM buffers; the softmax backward turns them, in place, into dS (x
//    scale) and P, each split into bf16 hi + lo parts (dkv accurate to about
//    fp32 even for keys shared by many rows); dKV = dS^T Q + P^T dO is then
//    formed 128 channels at a time (N = 128) with all four A operands read
//    from TMEM, into one of TWO TMEM staging slots.  The slots are drained
//    into L2 reductions by the flush warps and the math warps (64 channels
//    each, read out of TMEM and released at once, then transposed so that
//    every reduction instruction covers 4 rows x 128 bytes).  With two S/dP
//    buffers and two staging slots, the next tile's S^T / dP^T and softmax
//    run while the reductions of this tile are still in flight.
//  * dq needs dS for every tile of the token but the main loop has no TMEM
//    left for its accumulator, so dS hi of each tile is also written to a
//    scratch slot in global memory (L2-resident) and dQ^T = KV^T dS^T is
//    formed in an end phase per token, when Q and dO are dead and their
//    shared memory becomes a deep gather ring.  A CTA claims its scratch slot
//    from a table of slot flags in the workspace (compare-and-swap, starting
//    at the SM id as a hint) and frees it when it exits, so two CTAs never
//    share a slot whatever SMs they run on.
//  * The gathered rows stream through shared memory in 64-channel chunks
//    (128-byte swizzle) loaded by 16-byte cp.async (zero-fill for invalid or
//    beyond-prefix rows).
//  * One warp issues every MMA (one elected lane per instruction, the
//    whole warp running the issuing loop).  It polls its inputs (ring chunks landed,
//    dS ready, staging slot free, buffer free) and issues whichever unit of
//    work is ready, dKV groups first, so that the tensor core follows the
//    reductions instead of a fixed program order.
//
// Warp roles: warp 0 issues MMAs and owns TMEM; warps 1-3 gather (with warps
// 4-11 in the end phase); warps 4-11 run the softmax backward, drain their
// share of the dKV groups and write dq; warps 12-15 drain the rest of the dKV
// groups.
#include <cmath>

#include "dsa_device.cuh"
#include "dsa_host.h"

namespace dsa {
namespace bwd {

constexpr int kThreads = 512;
constexpr int kGather = 96;    // warps 1-3
constexpr int kMath = 256;     // warps 4-11
constexpr int kTile = 128;     // top-k slots per tile (MMA M)
constexpr int kHeads = 64;     // heads per CTA (MMA N)
constexpr int kDv = 512;
constexpr int kGroup = 128;    // dKV channels per staging slot (MMA N)
constexpr int kRing = 4;       // main-loop ring: 16 KiB chunk slots
constexpr int kERing = 6;      // end-phase ring: 32 KiB slots (a dS tile or a 128-channel pair)
constexpr int kStage = 2;      // dKV staging slots
constexpr int kMaxSlots = 256;                    // dS scratch slots (more than the resident CTAs)
constexpr long long kHintRetryCycles = 8192;      // retries of the SM's own slot before scanning
constexpr int kDsTileBytes = kTile * kHeads * 2;  // bf16 dS of one tile: 16 KiB
constexpr int kUnits = kTile * 8;                 // 16-byte units of one 64-channel chunk

template <int DQK>
struct Smem {
  static constexpr int NCH = DQK / 64;          // channel chunks of kv / q
  static constexpr int NP = (NCH + 1) / 2;      // channel pairs (128 channels)
  static constexpr int NG = (DQK + kGroup - 1) / kGroup;  // dKV groups (the last may be 64 channels)
  static constexpr int Q_CHUNK = kHeads * 128;  // 8 KiB: 64 heads x 64 channels
  static constexpr int QDO = 2 * Q_CHUNK;       // chunk c of Q followed by chunk c of dO
  static constexpr int KV_CHUNK = kTile * 128;  // 16 KiB
  static constexpr int ESLOT = 2 * KV_CHUNK;    // end-phase slot
  // Q and dO, chunk-interleaved: [Q_0 dO_0][Q_1 dO_1]...[Q_7 dO_7][Q_8].  One K-major
  // operand of N = 128 rows then covers the 64 heads of Q_c and of dO_c, so that a
  // single MMA forms S^T and dP^T; two consecutive chunks of Q (or of dO) form an
  // MN-major operand of N = 128 channels with LBO = QDO.
  static constexpr int OFF_QDO = 0;
  static constexpr int OFF_RING = OFF_QDO + 8 * QDO + (NCH - 8) * Q_CHUNK;
  static constexpr int OFF_FST = OFF_RING + kRing * KV_CHUNK;  // flush transposes: 12 warps x 16 rows x 128 B
  static constexpr int OFF_MISC = OFF_FST + 12 * 2048;
  static constexpr int MISC = 1024;
  static constexpr int TOTAL = OFF_MISC + MISC + 1024;  // + alignment slack
  static constexpr int OFF_ERING = 0;                   // end phase: over Q, dO and the main ring
  static_assert(TOTAL <= 232448, "shared memory budget");
  static_assert(kERing * ESLOT <= OFF_FST, "end-phase ring fits below the flush buffers");
  static_assert(kHeads * DQK * 2 <= OFF_FST, "dq staging fits below the flush buffers");
};

// misc layout: mbarriers (8 bytes each), then scalars and per-head vectors
constexpr int B_FULL = 0, B_EMPTY = 5, B_EFULL = 10, B_EEMPTY = 16, B_SDP = 22, B_DS = 24, B_KVD = 26, B_STF = 28,
              B_STE = 32, B_DSDONE = 36, B_ENDGO = 37, B_DQ = 38, B_FIN = 39, B_COUNT = 40;
constexpr int M_TMEM = 384, M_NEFF = 388, M_ABORT = 392, M_SLOT = 396;
constexpr int M_LSE = 512, M_DL = 768;  // float [64] each
static_assert(B_COUNT * 8 <= M_TMEM, "barriers fit");

// TMEM columns.  Main loop: buffer b holds S^T at 128b and dP^T at 128b + 64;
// staging slot s at 256 + 128s.  End phase: dQ^T channel tile p at 64p.
constexpr uint32_t C_BUF = 128, C_STG = 256;
static_assert(C_STG + kStage * kGroup <= 512, "TMEM budget");

// D[t,h] = <dO[t,h,:], O[t,h,:] (+ O_lo[t,h,:])> in fp32; one warp per (t, h).  With a sink,
// d_sink[h] += -exp(sink[h] - lse[t,h]) D[t,h] (nothing for an empty row, lse = -inf).
__global__ void bwd_delta_kernel(const __nv_bfloat16* __restrict__ out, const __nv_bfloat16* __restrict__ out_lo,
                                 const __nv_bfloat16* __restrict__ dout, float* __restrict__ delta, long long rows,
                                 const float* __restrict__ lse, const float* __restrict__ sink,
                                 float* __restrict__ d_sink, int H) {
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
  if (lane == 0) {
    delta[w] = acc;
    if (d_sink != nullptr) {
      const int h = (int)(w % H);
      const float l = __ldg(lse + w), sk = __ldg(sink + h);
      if (sk > -INFINITY && l > -INFINITY) atomicAdd(d_sink + h, -expf(sk - l) * acc);
    }
  }
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

// Drain 64 staged dKV channels of this warp's 32 key rows into L2 reductions.
// v holds the warp's TMEM load (lane = key row, 64 consecutive channels); the
// rows are transposed through the warp's 2 KB buffer, 16 rows x 32 channels at
// a time, so that 8 lanes cover one row's 128 contiguous bytes and each
// reduction instruction touches 4 rows x 128 B.  ix: this lane's key (-1 = skip).
template <int DQK>
__device__ __forceinline__ void reduce_rows64(const uint32_t (&v)[4][16], uint32_t fst, int lane, int ix,
                                              float* dst_col) {
#pragma unroll
  for (int bc = 0; bc < 2; ++bc) {
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      if ((lane >> 4) == hh) {
        const int rl = lane & 15;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const uint32_t(&w)[16] = v[2 * bc + (u >> 2)];
          st_shared_v4(fst + rl * 128 + ((u ^ (rl & 7)) << 4), w[4 * (u & 3)], w[4 * (u & 3) + 1], w[4 * (u & 3) + 2],
                       w[4 * (u & 3) + 3]);
        }
      }
      __syncwarp();
#pragma unroll
      for (int st = 0; st < 4; ++st) {
        const int rl = 4 * st + (lane >> 3), u = lane & 7;
        const int ixr = __shfl_sync(0xffffffffu, ix, 16 * hh + rl);
        float4 f;
        asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                     : "=f"(f.x), "=f"(f.y), "=f"(f.z), "=f"(f.w)
                     : "r"(fst + rl * 128 + ((u ^ (rl & 7)) << 4))
                     : "memory");
        if (ixr >= 0) red_add_v4(dst_col + (size_t)ixr * DQK + 32 * bc + 4 * u, f.x, f.y, f.z, f.w);
      }
      __syncwarp();
    }
  }
}

// Drain warps of a quadrant: the flush warp (role 0) and the two math warps
// (roles 1, 2 = head halves).  The flush warp drains the first half (64
// channels) of every dKV group; the second halves alternate between the math
// warps, which also run the softmax on the critical path.  (When the upper
// head half is all padding its math warp runs no softmax; giving it more of
// the second halves was measured slower than the alternation.)
__device__ __forceinline__ int drain_role(int g, int hf) { return hf == 0 ? 0 : 1 + (g & 1); }

// One thread's share of gathering a tile's rows, 64 channels at a time, with
// NT threads: per unit (row, 16-byte column) the source pointer of channel 0
// and the swizzled destination offset are computed once per tile, so that a
// chunk costs one cp.async per unit.  Invalid or beyond-prefix rows are
// zero-filled (src-size 0; the pointer stays inside kv and is not read).
template <int DQK, int NT>
struct TileGather {
  static constexpr int KU = (kUnits + NT - 1) / NT;
  const __nv_bfloat16* src[KU];
  uint32_t dst[KU];
  uint32_t okm;
  int raw[KU];  // indices of the tile loaded by load(), not yet checked
  // Issue the index loads of tile i.  Nothing uses the values until resolve(), so a caller
  // that loads the next tile before gathering the current one hides their memory latency.
  __device__ __forceinline__ void load(const int32_t* __restrict__ idx_row, int i, int n_eff, int et) {
#pragma unroll
    for (int k = 0; k < KU; ++k) {
      const int u = et + NT * k;
      const int j = i * kTile + (u >> 3);
      raw[k] = (u < kUnits && j < n_eff) ? __ldg(idx_row + j) : -1;
    }
  }
  // Source rows and destinations of the loaded tile; bad indices are flagged and zero-filled.
  __device__ __forceinline__ void resolve(const __nv_bfloat16* __restrict__ kv, int Tk, int et, int* err) {
    okm = 0;
#pragma unroll
    for (int k = 0; k < KU; ++k) {
      const int u = et + NT * k;
      const int ix = raw[k];
      const int v = (ix >= 0 && ix < Tk) ? ix : -1;
      if (ix < -1 || ix >= Tk) record_error(err, DSA_ERR_DEVICE_INDEX);
      src[k] = kv + (v >= 0 ? (size_t)v * DQK : 0) + (u & 7) * 8;
      dst[k] = sw128_off((u >> 3) & (kTile - 1), u & 7);
      okm |= (v >= 0 ? 1u : 0u) << k;
    }
  }
  __device__ __forceinline__ void chunk(uint32_t base, int c, int et) const {
#pragma unroll
    for (int k = 0; k < KU; ++k)
      if (et + NT * k < kUnits) cp_async16(base + dst[k], src[k] + c * 64, ((okm >> k) & 1u) ? 16u : 0u);
  }
};

template <int DQK>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_bwd_kernel(const __nv_bfloat16* __restrict__ kv, const __nv_bfloat16* __restrict__ q,
                          const int32_t* __restrict__ topk_idx, const int32_t* __restrict__ topk_len,
                          const float* __restrict__ lse, const float* __restrict__ delta,
                          const __nv_bfloat16* __restrict__ dout, int T, int Tk, int H, int K, float scale,
                          __nv_bfloat16* __restrict__ dq, float* __restrict__ dkv, float* __restrict__ attn_prob,
                          float inv_heads,
                          int* __restrict__ slot_flags, uint8_t* __restrict__ ds_scratch, int tiles_per_slot,
                          int* __restrict__ err, long long wait_limit) {
  using L = Smem<DQK>;
  constexpr int NCH = L::NCH;
  constexpr int NP = L::NP;
  constexpr int NG = L::NG;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sQDO = smem_u32(smem + L::OFF_QDO);
  const uint32_t sRing = smem_u32(smem + L::OFF_RING);
  const uint32_t sERing = smem_u32(smem + L::OFF_ERING);
  uint8_t* misc = smem + L::OFF_MISC;
  const uint32_t bars = smem_u32(misc);
  auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(misc + M_TMEM);
  int* s_neff = reinterpret_cast<int*>(misc + M_NEFF);
  volatile int* s_abort = reinterpret_cast<volatile int*>(misc + M_ABORT);
  int* s_slot = reinterpret_cast<int*>(misc + M_SLOT);
  float* s_lse2 = reinterpret_cast<float*>(misc + M_LSE);
  float* s_dl = reinterpret_cast<float*>(misc + M_DL);

  const int t = blockIdx.x;
  const int hg = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int32_t* idx_row = topk_idx + (size_t)t * K;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kRing; ++i) {
      mbar_init(bar(B_FULL + i), kGather);
      mbar_init(bar(B_EMPTY + i), 1);
    }
    for (int i = 0; i < kERing; ++i) {
      mbar_init(bar(B_EFULL + i), kGather + kMath);  // the math warps join the end-phase gathers
      mbar_init(bar(B_EEMPTY + i), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(B_SDP + b), 1);
      mbar_init(bar(B_DS + b), kMath / 32);
      mbar_init(bar(B_KVD + b), 1);
    }
    for (int s = 0; s < kStage; ++s) {
      mbar_init(bar(B_STF + s), 1);
      mbar_init(bar(B_STE + s), kMath / 32 + 4);  // every drain warp (8 math + 4 flush) releases every use
    }
    mbar_init(bar(B_DSDONE), kMath);
    mbar_init(bar(B_ENDGO), 1);
    mbar_init(bar(B_DQ), 1);
    mbar_init(bar(B_FIN), 1);
    *s_neff = 0;
    *s_abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(s_tmem), 512);
    tmem_relinquish();
  }
  if (threadIdx.x == 32) {
    // claim a free dS scratch slot by compare-and-swap over the slot flags.  The SM id is a hint
    // (slots are owned by CTAs, not SMs): the CTA that ran here before frees that slot as it
    // exits, and its release may still be on its way to L2, so the hint is retried for a short
    // while before the other slots are scanned; reusing it keeps the scratch footprint at one
    // slot per SM in L2.  Gives up (DSA_ERR_TIMEOUT) after the wait limit.
    const int hint = (int)(sm_id() % (uint32_t)kMaxSlots);
    int slot = -1;
    const long long c0 = clock64();
    while (slot < 0 && clock64() - c0 < kHintRetryCycles)
      if (atomicCAS(slot_flags + hint, 0, 1) == 0) slot = hint;
    for (int k = 1; slot < 0; ++k) {
      const int sl = (hint + k) % kMaxSlots;
      if (atomicCAS(slot_flags + sl, 0, 1) == 0) {
        slot = sl;
      } else if (k >= kMaxSlots && clock64() - c0 > wait_limit) {
        record_error(err, DSA_ERR_TIMEOUT);
        break;
      }
    }
    __threadfence();  // the previous owner's scratch accesses precede this CTA's
    *s_slot = slot;
  }
  __syncthreads();

  const bool is_gather = warp >= 1 && warp < 4;
  const bool is_math = warp >= 4 && warp < 12;
  const bool is_flush = warp >= 12;
  if (is_math) {
    const int tid = threadIdx.x - 128;
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
    // Read once per CTA: evicted from L2 first (the scratch, dkv and kv rows stay)
    const uint64_t pol = l2_evict_first_policy();
    for (int u = tid; u < kHeads * NCH * 8; u += kMath) {
      const int hh = u / (NCH * 8), rem = u - hh * (NCH * 8), c = rem >> 3, uc = rem & 7;
      const int h = hg * kHeads + hh;
      const bool ok = h < H;  // padded heads are zero-filled without a read
      cp_async16_hint(sQDO + c * L::QDO + sw128_off(hh, uc),
                      q + (ok ? ((size_t)t * H + h) * DQK + c * 64 + uc * 8 : 0), ok ? 16u : 0u, pol);
    }
    for (int u = tid; u < kHeads * 8 * 8; u += kMath) {
      const int hh = u >> 6, rem = u & 63, c = rem >> 3, uc = rem & 7;
      const int h = hg * kHeads + hh;
      const bool ok = h < H;
      cp_async16_hint(sQDO + c * L::QDO + L::Q_CHUNK + sw128_off(hh, uc),
                      dout + (ok ? ((size_t)t * H + h) * kDv + c * 64 + uc * 8 : 0), ok ? 16u : 0u, pol);
    }
    // per-head lse (log2 units) and D, shared by every key row
    if (tid < kHeads) {
      const int hh = hg * kHeads + tid;
      s_lse2[tid] = (hh < H) ? lse[(size_t)t * H + hh] * 1.4426950408889634f : INFINITY;  // padded heads: P = 0
      s_dl[tid] = (hh < H) ? delta[(size_t)t * H + hh] : 0.f;
    }
    asm volatile("cp.async.wait_all;" ::: "memory");  // all copies in flight at once, one wait
    fence_proxy_async_smem();
  }
  __syncthreads();
  int ntiles = (*s_neff + kTile - 1) / kTile;
  const int n_eff = *s_neff;
  const uint32_t tmem = *s_tmem;
  // this CTA's dS scratch slot (none: the claim timed out, and the CTA computes nothing)
  const int slot = *s_slot;
  if (slot < 0 || ntiles > tiles_per_slot) {
    if (threadIdx.x == 0 && slot >= 0) record_error(err, DSA_ERR_UNSUPPORTED);
    ntiles = 0;
  }
  uint8_t* ds_slot = ds_scratch + (size_t)(slot < 0 ? 0 : slot) * tiles_per_slot * kDsTileBytes;

  // End-phase gathers, shared by the gather and the math warps (et = 0..351):
  // per tile the swizzled dS image from the scratch, then the channel pairs.
  auto end_gathers = [&](int et) {
    constexpr int NT = kGather + kMath;
    if (!mbar_wait(bar(B_ENDGO), 0, s_abort, err, wait_limit) || !mbar_wait(bar(B_DSDONE), 0, s_abort, err, wait_limit)) return;
    TileGather<DQK, NT> tg;
    int Le = 0;
    tg.load(idx_row, 0, n_eff, et);
    for (int i = 0; i < ntiles; ++i) {
      int slot = Le % kERing;
      if (Le >= kERing && !mbar_wait(bar(B_EEMPTY + slot), ((Le / kERing) - 1) & 1, s_abort, err, wait_limit)) return;
      const uint8_t* src = ds_slot + (size_t)i * kDsTileBytes;
      for (int u = et; u < kDsTileBytes / 16; u += NT) cp_async16(sERing + slot * L::ESLOT + 16 * u, src + 16 * u, 16u);
      cp_async_arrive(bar(B_EFULL + slot));
      ++Le;
      tg.resolve(kv, Tk, et, err);
      if (i + 1 < ntiles) tg.load(idx_row, i + 1, n_eff, et);  // the next tile's indices, a tile ahead
      for (int p = 0; p < NP; ++p, ++Le) {
        slot = Le % kERing;
        if (Le >= kERing && !mbar_wait(bar(B_EEMPTY + slot), ((Le / kERing) - 1) & 1, s_abort, err, wait_limit)) return;
        tg.chunk(sERing + slot * L::ESLOT, 2 * p, et);
        if (2 * p + 1 < NCH) tg.chunk(sERing + slot * L::ESLOT + L::KV_CHUNK, 2 * p + 1, et);
        cp_async_arrive(bar(B_EFULL + slot));
      }
    }
  };

  // A drain warp's part of staged dKV group G (group g of its tile): wait for it (every drain warp
  // waits for every group, in order, so that each slot barrier is read phase by phase), load the
  // half this warp owns if any, release the slot, then reduce it into dkv.
  const bool pad_hi = hg * kHeads + 32 >= H;  // heads 32..63 of this CTA are all padding
  auto drain_group = [&](int G, int g, int role, int ix, uint32_t fst) -> bool {
    const int s = G & (kStage - 1);
    if (!mbar_wait(bar(B_STF + s), (G / kStage) & 1, s_abort, err, wait_limit)) return false;
    const int halves = (g * kGroup + kGroup <= DQK) ? 2 : 1;
    int mine = -1;  // the half this warp owns, if any (drain_role gives a warp at most one per group)
    for (int hf = 0; hf < halves; ++hf)
      if (drain_role(g, hf) == role) mine = hf;
    if (mine >= 0) {
      tc_fence_after();
      uint32_t v[4][16];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq)
        tmem_ld16(tmem_addr(tmem + C_STG + kGroup * s + 64 * mine + 16 * qq, (warp & 3) * 32, 0), v[qq]);
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_STE + s));  // the slot may be refilled
      reduce_rows64<DQK>(v, fst, lane, ix, dkv + g * kGroup + 64 * mine);
    } else {
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_STE + s));
    }
    return true;
  };

  if (warp == 0) {
    {
      // ============ MMA issuer (the whole warp runs it; one elected lane issues each instruction) ============
      constexpr uint32_t kIdSP = idesc_bf16(128, 128, false, false);  // [S^T | dP^T] = KV [Q | dO]^T
      constexpr uint32_t kIdS = idesc_bf16(128, 64, false, false);    // S^T only (RoPE chunk)
      constexpr uint32_t kIdMM = idesc_bf16(128, 64, true, true);     // dQ^T
      constexpr uint32_t kIdKM = idesc_bf16(128, 128, false, true);   // dKV, 128 channels: A (TMEM) x B MN-major
      constexpr uint32_t kIdKM64 = idesc_bf16(128, 64, false, true);  // dKV, last 64 channels
      int ia = 0, ca = 0, La = 0;  // S^T / dP^T stream: next (tile, chunk), ring item
      int id = 0, gd = 0, G = 0;   // dKV stream: next (tile, group), staging item
      bool ds_seen = false, buf_seen = false, idle = false, stop = false;
      long long idle_t0 = 0;
      while (id < ntiles) {
        bool progressed = false;
        // ---- dKV group gd of tile id: needs dS/P of tile id in TMEM and a free staging slot ----
        if (id < ia) {
          if (!ds_seen) ds_seen = warp_all(mbar_test(bar(B_DS + (id & 1)), (id >> 1) & 1));
          const int s = G & (kStage - 1), n = G / kStage;
          if (ds_seen && (n == 0 || warp_all(mbar_test(bar(B_STE + s), (n - 1) & 1)))) {
            tc_fence_after();
            const uint32_t bS = tmem + C_BUF * (id & 1), bP = bS + 64;
            const uint32_t d = tmem + C_STG + kGroup * s;
            const uint32_t qb = sQDO + 2 * gd * L::QDO;  // chunks 2gd, 2gd+1 of Q (and of dO at + Q_CHUNK)
            if (gd * kGroup + kGroup <= DQK) {
              const uint64_t bq0 = sdesc_sw128(qb, L::QDO, 1024), bo0 = sdesc_sw128(qb + L::Q_CHUNK, L::QDO, 1024);
              const bool with_p = gd * kGroup + kGroup <= kDv;
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint32_t acol = (k >> 1) * 32 + (k & 1) * 8;  // heads 16k..16k+15 in a thread-half region
                const uint64_t bq = bq0 + (uint64_t)(k * 128), bo = bo0 + (uint64_t)(k * 128);  // + 16 head rows
                mma_ts_w(d, bS + 16 + acol, bq, kIdKM, k > 0);  // dS hi
                mma_ts_w(d, bS + acol, bq, kIdKM, 1u);          // dS lo
                if (with_p) {
                  mma_ts_w(d, bP + acol, bo, kIdKM, 1u);        // P hi
                  mma_ts_w(d, bP + 16 + acol, bo, kIdKM, 1u);   // P lo
                }
              }
            } else {  // the RoPE channels 512..575: dS terms only
              const uint64_t bq0 = sdesc_sw128(qb, 16, 1024);
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const uint32_t acol = (k >> 1) * 32 + (k & 1) * 8;
                const uint64_t bq = bq0 + (uint64_t)(k * 128);
                mma_ts_w(d, bS + 16 + acol, bq, kIdKM64, k > 0);
                mma_ts_w(d, bS + acol, bq, kIdKM64, 1u);
              }
            }
            mma_commit_w(bar(B_STF + s));
            ++G;
            progressed = true;
            if (++gd == NG) {
              mma_commit_w(bar(B_KVD + (id & 1)));  // buffer id & 1 may be overwritten once this lands
              gd = 0;
              ++id;
              ds_seen = false;
            }
          }
        }
        // ---- chunk ca of tile ia: S^T (+ dP^T) into buffer ia & 1 ----
        if (ia < ntiles) {
          if (!buf_seen) buf_seen = (ia < 2) || warp_all(mbar_test(bar(B_KVD + (ia & 1)), ((ia - 2) >> 1) & 1));
          const int slot = La % kRing;
          if (buf_seen && warp_all(mbar_test(bar(B_FULL + slot), (La / kRing) & 1))) {
            fence_proxy_async_smem();  // cp.async landings -> visible to the tensor core
            tc_fence_after();
            const uint32_t bS = tmem + C_BUF * (ia & 1);
            const uint64_t a0 = sdesc_sw128(sRing + slot * L::KV_CHUNK, 16, 1024);
            const uint64_t b0 = sdesc_sw128(sQDO + ca * L::QDO, 16, 1024);  // rows: 64 heads of Q_c, then of dO_c
            const uint32_t idn = (ca < 8) ? kIdSP : kIdS;
#pragma unroll
            for (int k = 0; k < 4; ++k)  // + 16 channels = + 32 bytes per row
              mma_ss_w(bS, a0 + (uint64_t)(k * 2), b0 + (uint64_t)(k * 2), idn, (ca | k) != 0);
            mma_commit_w(bar(B_EMPTY + slot));
            ++La;
            progressed = true;
            if (++ca == NCH) {
              mma_commit_w(bar(B_SDP + (ia & 1)));
              ca = 0;
              ++ia;
              buf_seen = false;
            }
          }
        }
        if (progressed) {
          idle = false;
          continue;
        }
        __nanosleep(32);  // leave the issue slots to the math and flush warps of this sub-partition
        if (!idle) {
          idle = true;
          idle_t0 = clock64();
        } else if (__any_sync(0xffffffffu, *s_abort != 0)) {
          stop = true;
          break;
        } else if (__any_sync(0xffffffffu, clock64() - idle_t0 > wait_limit)) {
          *s_abort = 1;
          record_error(err, DSA_ERR_TIMEOUT);
          stop = true;
          break;
        }
      }
      // ---- end phase: dQ^T[pair p] += KV^T dS^T over every tile of the token ----
      if (!stop && ntiles > 0) {
        // every dKV MMA has landed: Q, dO, the main ring and the S/dP buffers are dead
        stop = !warp_all(mbar_wait(bar(B_KVD + ((ntiles - 1) & 1)), ((ntiles - 1) >> 1) & 1, s_abort, err, wait_limit));
        if (!stop && lane == 0) mbar_arrive(bar(B_ENDGO));
        // the rope tile of dQ^T overlaps staging slot 0: wait for its last drain
        bool rope_free = (NP * 64 <= (int)C_STG);
        const int uses0 = (G + kStage - 1) / kStage;
        int Le = 0;
        for (int i = 0; i < ntiles && !stop; ++i) {
          const int sds = Le % kERing;
          if (!warp_all(mbar_wait(bar(B_EFULL + sds), (Le / kERing) & 1, s_abort, err, wait_limit))) { stop = true; break; }
          const uint32_t dsb = sERing + sds * L::ESLOT;
          ++Le;
          for (int p = 0; p < NP; ++p, ++Le) {
            const int sl = Le % kERing;
            if (!warp_all(mbar_wait(bar(B_EFULL + sl), (Le / kERing) & 1, s_abort, err, wait_limit))) { stop = true; break; }
            if (p * 64 + 64 > (int)C_STG && !rope_free) {
              if (uses0 > 0 && !warp_all(mbar_wait(bar(B_STE), (uses0 - 1) & 1, s_abort, err, wait_limit))) { stop = true; break; }
              rope_free = true;
            }
            fence_proxy_async_smem();
            tc_fence_after();
            const uint64_t a0 = sdesc_sw128(sERing + sl * L::ESLOT, L::KV_CHUNK, 1024);
            const uint64_t b0 = sdesc_sw128(dsb, L::KV_CHUNK, 1024);
#pragma unroll
            for (int k = 0; k < kTile / 16; ++k)  // + 16 key rows = + 2048 bytes
              mma_ss_w(tmem + 64 * p, a0 + (uint64_t)(k * 128), b0 + (uint64_t)(k * 128), kIdMM, (i > 0 || k > 0) ? 1u : 0u);
            mma_commit_w(bar(B_EEMPTY + sl));
          }
          if (stop) break;
          mma_commit_w(bar(B_EEMPTY + sds));
        }
      }
      if (stop) *s_abort = 1;
      mma_commit_w(bar(B_DQ));
      // every MMA of this CTA completes before the teardown frees TMEM
      mma_commit_w(bar(B_FIN));
      volatile int dummy = 0;
      mbar_wait(bar(B_FIN), 0, &dummy, err);
    }
    __syncwarp();
  } else if (is_gather) {
    // ======================= gathers (cp.async, 16-byte units) =======================
    const int gt = threadIdx.x - 32;  // 0..95
    TileGather<DQK, kGather> tg;
    bool aborted = false;
    int La = 0;
    if (ntiles > 0) tg.load(idx_row, 0, n_eff, gt);
    for (int i = 0; i < ntiles && !aborted; ++i) {
      tg.resolve(kv, Tk, gt, err);
      if (i + 1 < ntiles) tg.load(idx_row, i + 1, n_eff, gt);  // the next tile's indices, a tile ahead
      for (int c = 0; c < NCH; ++c, ++La) {
        const int slot = La % kRing;
        if (La >= kRing && !mbar_wait(bar(B_EMPTY + slot), ((La / kRing) - 1) & 1, s_abort, err, wait_limit)) {
          aborted = true;
          break;
        }
        tg.chunk(sRing + slot * L::KV_CHUNK, c, gt);
        cp_async_arrive(bar(B_FULL + slot));
      }
    }
    // the end phase overwrites Q, dO and the main ring, and reads the dS scratch
    if (!aborted && ntiles > 0) end_gathers(gt);
    // no copy may still be landing in this CTA's shared memory when it exits
    asm volatile("cp.async.wait_all;" ::: "memory");
  } else if (is_flush) {
    // ======================= dKV flush: its share of every staged group -> L2 reductions =======================
    const int qd = warp & 3;
    const int r = qd * 32 + lane;  // key row of the tile
    const uint32_t fst = smem_u32(smem + L::OFF_FST + qd * 2048);
    for (int i = 0; i < ntiles; ++i) {
      const int j = i * kTile + r;
      int ix = -1;
      if (j < n_eff) ix = __ldg(idx_row + j);
      if (!(ix >= 0 && ix < Tk)) ix = -1;
      bool stop = false;
      for (int g = 0; g < NG; ++g)
        if (!drain_group(i * NG + g, g, 0, ix, fst)) { stop = true; break; }
      if (stop) break;
    }
  } else {
    // ======================= math warps: softmax backward, dS scratch, dq epilogue =======================
    const int mw = warp - 4;  // 0..7
    const int qd = warp & 3;
    const int ch = mw >> 2;        // heads ch*32 .. ch*32+31
    const int r = qd * 32 + lane;  // key row of the tile
    const float sl2e = scale * 1.4426950408889634f;
    const float* lse2 = s_lse2 + ch * 32;
    const float* dl = s_dl + ch * 32;
    const uint32_t fst_m = smem_u32(smem + L::OFF_FST + (4 + mw) * 2048);  // this warp's transpose buffer
    const bool pad_half = ch == 1 && pad_hi;  // every head of this half is padding
    bool aborted = false;
    for (int i = 0; i < ntiles; ++i) {
      const int b = i & 1;
      // this key row's index does not depend on the MMA: its load overlaps the wait
      const int j = i * kTile + r;
      const int ix = (j < n_eff) ? __ldg(idx_row + j) : -1;
      if (!mbar_wait(bar(B_SDP + b), (i >> 1) & 1, s_abort, err, wait_limit)) { aborted = true; break; }
      tc_fence_after();
      const uint32_t tS = tmem_addr(tmem + C_BUF * b + ch * 32, qd * 32, 0);
      const uint32_t tP = tS + 64;
      const bool valid = ix >= 0 && ix < Tk;
      if (pad_half) {
        // heads of zero q and dO rows only: S^T and dP^T are exact zeros, whose fp32 bits are also the
        // bf16 hi + lo zeros the dKV products read, and dq of these heads is not stored
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_DS + b));
        const int kix = valid ? ix : -1;
        for (int g = 0; g < NG && !aborted; ++g)
          if (!drain_group(i * NG + g, g, 1 + ch, kix, fst_m)) aborted = true;
        if (aborted) break;
        continue;
      }
      uint32_t sv[32], dv[32];
      tmem_ld32(tS, sv);
      tmem_ld32(tP, dv);
      tmem_ld_wait();
      uint32_t ph[16], pl[16], sh[16], sl[16];
      float psum = 0.f;  // this half's sum of P over its 32 heads (the slot probability, on request)
#pragma unroll
      for (int h = 0; h < 32; h += 2) {
        float p0 = 0.f, p1 = 0.f, s0 = 0.f, s1 = 0.f;
        if (valid) {
          // per-head lse and D as 16-byte loads (4 heads), picked apart per pair
          const float4 L4 = reinterpret_cast<const float4*>(lse2)[h >> 2];
          const float4 D4 = reinterpret_cast<const float4*>(dl)[h >> 2];
          const float l0 = (h & 2) ? L4.z : L4.x, l1 = (h & 2) ? L4.w : L4.y;
          const float d0 = (h & 2) ? D4.z : D4.x, d1 = (h & 2) ? D4.w : D4.y;
          p0 = exp2f(__uint_as_float(sv[h]) * sl2e - l0);
          p1 = exp2f(__uint_as_float(sv[h + 1]) * sl2e - l1);
          s0 = scale * p0 * (__uint_as_float(dv[h]) - d0);
          s1 = scale * p1 * (__uint_as_float(dv[h + 1]) - d1);
          psum += p0 + p1;
        }
        const __nv_bfloat162 phi = __floats2bfloat162_rn(p0, p1);
        const __nv_bfloat162 shi = __floats2bfloat162_rn(s0, s1);
        const float2 phf = __bfloat1622float2(phi), shf = __bfloat1622float2(shi);
        ph[h >> 1] = *reinterpret_cast<const uint32_t*>(&phi);
        sh[h >> 1] = *reinterpret_cast<const uint32_t*>(&shi);
        pl[h >> 1] = pack_bf16x2(p0 - phf.x, p1 - phf.y);
        sl[h >> 1] = pack_bf16x2(s0 - shf.x, s1 - shf.y);
      }
      // A operands of the dKV products, in place over this thread's S^T / dP^T columns
      tmem_st16(tS, sl);
      tmem_st16(tS + 16, sh);
      tmem_st16(tP, ph);
      tmem_st16(tP + 16, pl);
      // dS hi of the tile in the swizzled [128 keys][64 heads] layout the end phase feeds to the tensor core
      uint4* img = reinterpret_cast<uint4*>(ds_slot + (size_t)i * kDsTileBytes);
#pragma unroll
      for (int uu = 0; uu < 4; ++uu)
        img[sw128_off(r, ch * 4 + uu) >> 4] = make_uint4(sh[4 * uu], sh[4 * uu + 1], sh[4 * uu + 2], sh[4 * uu + 3]);
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(B_DS + b));
      // head-averaged attention probability of this slot (each half of each head group adds its part)
      if (attn_prob != nullptr && valid) atomicAdd(attn_prob + (size_t)t * K + j, psum * inv_heads);
      // ---- this warp's share of the tile's staged dKV groups (role 1 + ch) ----
      const int kix = valid ? ix : -1;
      for (int g = 0; g < NG && !aborted; ++g)
        if (!drain_group(i * NG + g, g, 1 + ch, kix, fst_m)) aborted = true;
      if (aborted) break;
    }
    mbar_arrive(bar(B_DSDONE));  // this thread's dS scratch stores precede the end-phase gathers
    if (!aborted && ntiles > 0) end_gathers(threadIdx.x - 32);
    asm volatile("cp.async.wait_all;" ::: "memory");
    // ---- dq epilogue: dQ^T (lanes = channels) -> staged [64 heads][DQK] bf16 -> coalesced stores ----
    const int bar_id = 1 + ch;
    // every thread of the half joins the barrier, whether or not its warp left the loop early
    // (`aborted` is per warp here: the drains fail warp by warp)
    bool ok = !aborted && ntiles > 0;
    if (ok) ok = mbar_wait(bar(B_DQ), 0, s_abort, err, wait_limit);
    const bool have = !named_bar_or(bar_id, 128, !ok);
    if (have) tc_fence_after();
    named_bar(3, kMath);  // both halves have left the loop before the staging area is written
    __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(smem + L::OFF_ERING);
#pragma unroll 1
    for (int p = 0; p < NP; ++p) {
      uint32_t v[32];
      if (have) {
        tmem_ld32(tmem_addr(tmem + 64 * p + ch * 32, qd * 32, 0), v);
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
    const uint64_t pol = l2_evict_first_policy();  // dq is written once
    for (int u = threadIdx.x - 128; u < hcount * (DQK / 8); u += kMath)
      stg16_hint(dst + u, reinterpret_cast<const uint4*>(stage)[u], pol);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 32) {
    const int held = *s_slot;
    if (held >= 0) {
      __threadfence();  // every access of this CTA to the slot precedes its release
      atomicExch(slot_flags + held, 0);
    }
  }
}

template <int DQK>
dsa_status_t launch(const void* kv, const void* q, const int32_t* idx, const int32_t* len, const float* lse,
                    const float* delta, const void* dout, int T, int Tk, int H, int K, float scale, void* dq,
                    float* dkv, float* attn_prob, int* slot_flags, uint8_t* ds_scratch, int* err, cudaStream_t s) {
  using L = Smem<DQK>;
  dsa_status_t st = configure_kernel_smem(reinterpret_cast<const void*>(sparse_mla_bwd_kernel<DQK>), L::TOTAL,
                                          "configuring sparse_mla_bwd_kernel");
  if (st != DSA_OK) return st;
  dim3 grid(T, (H + kHeads - 1) / kHeads);
  sparse_mla_bwd_kernel<DQK><<<grid, kThreads, L::TOTAL, s>>>(
      reinterpret_cast<const __nv_bfloat16*>(kv), reinterpret_cast<const __nv_bfloat16*>(q), idx, len, lse, delta,
      reinterpret_cast<const __nv_bfloat16*>(dout), T, Tk, H, K, scale, reinterpret_cast<__nv_bfloat16*>(dq), dkv,
      attn_prob, 1.f / (float)H, slot_flags, ds_scratch, (K + kTile - 1) / kTile, err, wait_limit_cycles());
  return cuda_check(cudaGetLastError(), "launching sparse_mla_bwd_kernel");
}

// Workspace layout: [error word, 256 B][slot flags: kMaxSlots int32][D: T*H fp32]
//                   [dS scratch: kMaxSlots x ceil(K/128) x 16 KiB]
constexpr size_t kFlagBytes = kMaxSlots * sizeof(int);
constexpr size_t kHeadBytes = kErrorWordBytes + kFlagBytes;  // cleared at every call
static size_t delta_bytes(int32_t T, int32_t H) {
  const size_t d = (size_t)(T > 0 ? T : 0) * (size_t)(H > 0 ? H : 0) * sizeof(float);
  return (d + 255) & ~size_t(255);
}
static size_t scratch_bytes(int32_t K) {
  const size_t tiles = (size_t)((K > 0 ? K : 1) + kTile - 1) / kTile;
  return (size_t)kMaxSlots * tiles * kDsTileBytes;
}

}  // namespace bwd
}  // namespace dsa

using namespace dsa;

extern "C" size_t dsa_sparse_mla_bwd_workspace_size(int32_t T, int32_t H, int32_t K) {
  return bwd::kHeadBytes + bwd::delta_bytes(T, H) + bwd::scratch_bytes(K);
}

namespace dsa {
namespace bwd {
// The backward proper, on a scratch region of `workspace_bytes` bytes laid out as above.  A call
// split into row chunks passes first = false after its first chunk (the device error word keeps
// what earlier chunks recorded) and last = false before its last one (dkv is rounded to bf16 once).
static dsa_status_t run(const char* who, const dsa_bf16_t* q, const dsa_bf16_t* kv, const int32_t* topk_idx,
                        const int32_t* topk_len, int32_t T, int32_t T_k, int32_t H, int32_t Dqk, int32_t Dv,
                        int32_t K, float softmax_scale, const float* attn_sink, const dsa_bf16_t* out,
                        const dsa_bf16_t* out_lo, const float* lse, const dsa_bf16_t* dout, dsa_bf16_t* dq,
                        float* dkv_accum, float* d_sink, float* attn_prob, int32_t accumulate, dsa_bf16_t* dkv_bf16,
                        void* workspace, size_t workspace_bytes, dsa_stream_t stream, bool first = true,
                        bool last = true) {
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
  if (d_sink && !attn_sink) return fail(DSA_ERR_INVALID_ARGUMENT, "%s: d_sink needs attn_sink", who);
  dsa_status_t st = check_workspace(workspace, workspace_bytes, kHeadBytes + delta_bytes(T, H) + scratch_bytes(K), who);
  if (st != DSA_OK) return st;
  if ((st = check_device()) != DSA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // the error word (on a call's first chunk) and every slot flag start at zero
  uint8_t* clear_from = reinterpret_cast<uint8_t*>(workspace) + (first ? 0 : kErrorWordBytes);
  if ((st = cuda_check(cudaMemsetAsync(clear_from, 0, first ? kHeadBytes : kFlagBytes, s),
                       "clearing the error word and slot flags")))
    return st;
  if (!accumulate &&
      (st = cuda_check(cudaMemsetAsync(dkv_accum, 0, (size_t)T_k * Dqk * sizeof(float), s), "zeroing dkv_accum")))
    return st;
  if (!accumulate && d_sink &&
      (st = cuda_check(cudaMemsetAsync(d_sink, 0, (size_t)H * sizeof(float), s), "zeroing d_sink")))
    return st;
  if (attn_prob && T > 0 &&
      (st = cuda_check(cudaMemsetAsync(attn_prob, 0, (size_t)T * K * sizeof(float), s), "zeroing attn_prob")))
    return st;
  int* err = reinterpret_cast<int*>(workspace);
  int* flags = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(workspace) + kErrorWordBytes);
  float* delta = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(workspace) + kHeadBytes);
  uint8_t* ds_scratch = reinterpret_cast<uint8_t*>(workspace) + kHeadBytes + delta_bytes(T, H);
  if (T > 0) {
    const long long rows = (long long)T * H;
    bwd_delta_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(
        reinterpret_cast<const __nv_bfloat16*>(out), reinterpret_cast<const __nv_bfloat16*>(out_lo),
        reinterpret_cast<const __nv_bfloat16*>(dout), delta, rows, lse, attn_sink, d_sink, H);
    if ((st = cuda_check(cudaGetLastError(), "launching bwd_delta_kernel"))) return st;
    st = (Dqk == 576) ? launch<576>(kv, q, topk_idx, topk_len, lse, delta, dout, T, T_k, H, K, softmax_scale, dq,
                                    dkv_accum, attn_prob, flags, ds_scratch, err, s)
                      : launch<512>(kv, q, topk_idx, topk_len, lse, delta, dout, T, T_k, H, K, softmax_scale, dq,
                                    dkv_accum, attn_prob, flags, ds_scratch, err, s);
    if (st != DSA_OK) return st;
  }
  if (dkv_bf16 && last) {
    const long long n4 = (long long)T_k * Dqk / 4;
    f32_to_bf16_kernel<<<152 * 4, 256, 0, s>>>(dkv_accum, reinterpret_cast<__nv_bfloat16*>(dkv_bf16), n4);
    if ((st = cuda_check(cudaGetLastError(), "launching f32_to_bf16_kernel"))) return st;
  }
  return ok();
}
}  // namespace bwd
}  // namespace dsa

extern "C" dsa_status_t dsa_sparse_mla_bwd(const dsa_bf16_t* q, const dsa_bf16_t* kv, const int32_t* topk_idx,
                                           const int32_t* topk_len, int32_t T, int32_t T_k, int32_t H, int32_t Dqk,
                                           int32_t Dv, int32_t K, float softmax_scale, const float* attn_sink,
                                           const dsa_bf16_t* out, const dsa_bf16_t* out_lo, const float* lse,
                                           const dsa_bf16_t* dout, dsa_bf16_t* dq, float* dkv_accum, float* d_sink,
                                           float* attn_prob, int32_t accumulate, dsa_bf16_t* dkv_bf16,
                                           void* workspace, size_t workspace_bytes, dsa_stream_t stream) {
  return bwd::run("dsa_sparse_mla_bwd", q, kv, topk_idx, topk_len, T, T_k, H, Dqk, Dv, K, softmax_scale, attn_sink,
                  out, out_lo, lse, dout, dq, dkv_accum, d_sink, attn_prob, accumulate, dkv_bf16, workspace,
                  workspace_bytes, stream);
}

// ---------------------------------------------------------------------------
// dsa_sparse_mla_bwd_noalloc: the backward for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc: runtimes that reserve all device memory
// up front in their own pool and forbid any other allocation, or plug-ins
// loaded into a host program that owns every allocation.  They cannot provide
// the workspace dsa_sparse_mla_bwd needs (the device error word, the scratch
// slot flags and the dS scratch).  This entry point takes its scratch from the
// file-scope device array below instead, so it allocates nothing.
//
// The array is a fixed 84 MiB + 1280 B (error word, slot flags, D for 4 Mi
// (row, head) pairs, dS scratch for top-k up to 2176) that every GPU which
// loads this library holds until the process exits.  Query rows beyond what
// its D part holds are processed in chunks (rows are independent and key
// gradients sum, so dkv and d_sink accumulate over the chunks).  Its name is only a host-side stand-in for the device array,
// so the host looks up the array's real device address with
// cudaGetSymbolAddress, once per device and CUDA context, on the first call
// made there; that first call should therefore come before any stream capture.
// All calls share the one array: two calls whose executions overlap on the GPU
// race on it, so callers must order them (one stream, or events).  Each call
// clears the error word and the slot flags it uses, and its dS scratch is
// written before it is read, so stale contents from an earlier call do not
// leak into the result.  dsa_sparse_mla_bwd_noalloc_read_status reads the
// array's error word, as dsa_read_device_status does for a workspace.
// ---------------------------------------------------------------------------
#include <algorithm>
#include <climits>
#include <mutex>

namespace dsa {
namespace bwd {
constexpr int kNoAllocMaxTopk = 17 * kTile;                   // dS scratch for up to 17 tiles per row
constexpr size_t kNoAllocDeltaBytes = size_t(16) << 20;        // D for up to 4 Mi (row, head) pairs per chunk
constexpr size_t kNoAllocScratchBytes =
    kHeadBytes + kNoAllocDeltaBytes + (size_t)kMaxSlots * (kNoAllocMaxTopk / kTile) * kDsTileBytes;
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

typedef int (*CtxGetCurrentFn)(void** ctx);
typedef int (*CtxGetIdFn)(void* ctx, unsigned long long* id);

// Id of the calling thread's current CUDA context (0 if the driver cannot say).
static unsigned long long current_context_id() {
  static CtxGetCurrentFn get_ctx = nullptr;
  static CtxGetIdFn get_id = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_ctx = reinterpret_cast<CtxGetCurrentFn>(p);
    if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      get_id = reinterpret_cast<CtxGetIdFn>(p);
    cudaGetLastError();
  });
  void* ctx = nullptr;
  unsigned long long id = 0;
  if (get_ctx && get_id && get_ctx(&ctx) == 0 && ctx && get_id(ctx, &id) == 0) return id;
  return 0;
}

// Device address of g_noalloc_scratch in the current device's context.  It is looked up once per
// (device, context): a reset of the device's primary context reloads the module, and the array may
// then sit elsewhere, so a new context id means a new lookup.  (A thread with no context bound yet
// reads id 0 and looks the address up again; the lookup binds the context.)
static dsa_status_t noalloc_scratch(void** ptr) {
  static std::mutex mu;
  static void* addr[64] = {};
  static unsigned long long ctx_of[64] = {};
  int dev = 0;
  dsa_status_t st = cuda_check(cudaGetDevice(&dev), "cudaGetDevice");
  if (st != DSA_OK) return st;
  if (dev < 0 || dev >= 64) return fail(DSA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
  const unsigned long long ctx = current_context_id();
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev] || ctx == 0 || ctx != ctx_of[dev]) {
    void* p = nullptr;
    if ((st = cuda_check(cudaGetSymbolAddress(&p, g_noalloc_scratch), "cudaGetSymbolAddress(scratch)")) != DSA_OK)
      return st;
    addr[dev] = p;
    ctx_of[dev] = current_context_id();
  }
  *ptr = addr[dev];
  return DSA_OK;
}
}  // namespace bwd
}  // namespace dsa

extern "C" int32_t dsa_sparse_mla_bwd_noalloc_max_topk(void) { return bwd::kNoAllocMaxTopk; }

extern "C" dsa_status_t dsa_sparse_mla_bwd_noalloc(const dsa_bf16_t* q, const dsa_bf16_t* kv, const int32_t* topk_idx,
                                                   const int32_t* topk_len, int32_t T, int32_t T_k, int32_t H,
                                                   int32_t Dqk, int32_t Dv, int32_t K, float softmax_scale,
                                                   const float* attn_sink, const dsa_bf16_t* out,
                                                   const dsa_bf16_t* out_lo, const float* lse, const dsa_bf16_t* dout,
                                                   dsa_bf16_t* dq, float* dkv_accum, float* d_sink, float* attn_prob,
                                                   int32_t accumulate, dsa_bf16_t* dkv_bf16, dsa_stream_t stream) {
  if (K > bwd::kNoAllocMaxTopk)
    return fail(DSA_ERR_WORKSPACE,
                "dsa_sparse_mla_bwd_noalloc: top-k K = %d exceeds the built-in scratch limit of %d (use "
                "dsa_sparse_mla_bwd with a caller workspace)",
                K, bwd::kNoAllocMaxTopk);
  const size_t max_pairs = bwd::kNoAllocDeltaBytes / sizeof(float);
  if (H < 1 || (size_t)H > max_pairs)
    return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_sparse_mla_bwd_noalloc: H must be in [1, %zu] (got %d)", max_pairs, H);
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  void* scratch = nullptr;
  if ((st = bwd::noalloc_scratch(&scratch)) != DSA_OK) return st;
  const char* who = "dsa_sparse_mla_bwd_noalloc";
  // rows in chunks whose D fits the array (one chunk for T * H <= 4 Mi)
  const int32_t per = (int32_t)std::min<size_t>(max_pairs / (size_t)H, (size_t)INT32_MAX);
  if (T <= 0)
    return bwd::run(who, q, kv, topk_idx, topk_len, T, T_k, H, Dqk, Dv, K, softmax_scale, attn_sink, out, out_lo, lse,
                    dout, dq, dkv_accum, d_sink, attn_prob, accumulate, dkv_bf16, scratch, bwd::kNoAllocScratchBytes,
                    stream);
  for (int32_t r0 = 0; r0 < T; r0 += per) {
    const int32_t n = std::min(per, T - r0);
    const size_t rh = (size_t)r0 * H;
    st = bwd::run(who, q ? q + rh * Dqk : q, kv, topk_idx ? topk_idx + (size_t)r0 * K : topk_idx,
                  topk_len ? topk_len + r0 : nullptr, n, T_k, H, Dqk, Dv, K, softmax_scale, attn_sink,
                  out ? out + rh * Dv : out, out_lo ? out_lo + rh * Dv : nullptr, lse ? lse + rh : lse,
                  dout ? dout + rh * Dv : dout, dq ? dq + rh * Dqk : dq, dkv_accum, d_sink,
                  attn_prob ? attn_prob + (size_t)r0 * K : nullptr, (r0 > 0) ? 1 : accumulate, dkv_bf16, scratch, bwd::kNoAllocScratchBytes, stream, r0 == 0,
                  r0 + n >= T);
    if (st != DSA_OK) return st;
  }
  return ok();
}

extern "C" dsa_status_t dsa_sparse_mla_bwd_noalloc_read_status(dsa_stream_t stream, int32_t* status_host) {
  if (!status_host) return fail(DSA_ERR_INVALID_ARGUMENT, "dsa_sparse_mla_bwd_noalloc_read_status: null pointer");
  dsa_status_t st = check_device();
  if (st != DSA_OK) return st;
  void* scratch = nullptr;
  if ((st = bwd::noalloc_scratch(&scratch)) != DSA_OK) return st;
  return dsa_read_device_status(scratch, stream, status_host);
}
