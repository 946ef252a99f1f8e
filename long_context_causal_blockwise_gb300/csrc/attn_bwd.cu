// Backward kernels: gradients of exact attention by recomputation
// ("EasyContext核心技术解析：序列并行与Flash Attention的完美结合", §2 "Flash
// Attention优化": the backward recomputes the probabilities tile by tile from
// the stored row statistics instead of keeping the score matrix).
//
// With P_ij = exp(scale q_i.k_j - LSE_i), dP_ij = dO_i.v_j and
// dS_ij = P_ij (dP_ij - Delta_i):
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
//
// Two passes, each deterministic (no atomics):
//   dK/dV pass: one CTA per 128-key tile, looping over query tiles.
//     S^T = K Q_i^T and dP^T = V dO_i^T land in TMEM with one key per lane, so
//     the per-query statistics (LSE_i, Delta_i) are columns, staged in shared
//     memory. P^T and dS^T (bf16) overwrite S^T and dP^T in TMEM and feed
//     dV += P^T dO_i and dK += dS^T Q_i directly from TMEM.
//   dQ pass: one CTA per 128-query tile, looping over key tiles.
//     S = Q K_j^T and dP = dO V_j^T with one query per lane; dS (bf16)
//     overwrites S in TMEM and feeds dQ += dS K_j.
//
// Warps: 0-3 compute (thread = TMEM lane = tile row), 4 TMA producer,
// 5 MMA issuer and TMEM owner.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "lcb_attn.h"
#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kT = 128;  // rows per tile (both query and key tiles)
constexpr int kD = 128;
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = kT * kD * 2;  // 32 KB
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr int kStages = 2;
constexpr float kLog2e = 1.4426950408889634f;

// Fixed operands (2 tiles), a ring of kStages x 2 tiles, stats, barriers.
constexpr uint32_t kSmFixed = 0;
constexpr uint32_t kSmRing = 2 * kTileBytes;
constexpr uint32_t kSmStats = kSmRing + kStages * 2 * kTileBytes;  // 2 buffers x (lse2[128], delta[128]) fp32
constexpr uint32_t kSmBar = kSmStats + 2 * 2 * kT * 4;

struct Bars {
  uint64_t fixed_full;
  uint64_t ring_full[kStages];
  uint64_t ring_empty[kStages];
  uint64_t s_full;
  uint64_t p_full;
  uint64_t acc_full;
  uint64_t mma_done;
  uint64_t stats_full[2];  // dK/dV pass: the 128 compute threads staged a tile's LSE/Delta
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t kSmemBytes = kSmBar + sizeof(Bars) + 1024;

struct Params {
  const float* lse;
  const float* delta;
  long long l_hs, l_bs;
  void* g0;  // dK (dK/dV pass) or dQ (dQ pass)
  void* g1;  // dV (dK/dV pass)
  long long g_rs, g_bs;
  int B, H, Sq, Sk, causal, grad_mode;
  float scale, scale_log2;
  DevStatus st;
};

__device__ bool drain_wait(uint64_t* bar, uint32_t parity, unsigned long long limit) {
  const unsigned long long t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit) return false;
  }
  return true;
}

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

__device__ __forceinline__ void init_bars(Bars* bars) {
  mbar_init(&bars->fixed_full, 1);
  for (int s = 0; s < kStages; ++s) {
    mbar_init(&bars->ring_full[s], 1);
    mbar_init(&bars->ring_empty[s], 1);
  }
  mbar_init(&bars->s_full, 1);
  mbar_init(&bars->p_full, kT);
  mbar_init(&bars->acc_full, 1);
  mbar_init(&bars->mma_done, 1);
  mbar_init(&bars->stats_full[0], kT);
  mbar_init(&bars->stats_full[1], kT);
  bars->abort = 0;
  fence_mbar_init();
}

// Loads two fixed tiles once and then a ring of tile pairs; row_of(it) gives
// the tile row of ring item `it`.
__device__ void producer(uint8_t* smem, Bars* bars, const CUtensorMap* f0, const CUtensorMap* f1, int f_row,
                         const CUtensorMap* r0, const CUtensorMap* r1, int first_row_tile, int n, int h, int b,
                         const Params& p, uint32_t where) {
  volatile int* abort_flag = &bars->abort;
  const int x0 = h * kD;
  const uint64_t pol = l2_policy_evict_last();
  mbar_arrive_expect_tx(&bars->fixed_full, 2 * kTileBytes);
  for (int half = 0; half < 2; ++half) {
    tma_load_3d(smem + kSmFixed + half * kHalfBytes, f0, &bars->fixed_full, x0 + half * 64, f_row, b);
    tma_load_3d(smem + kSmFixed + kTileBytes + half * kHalfBytes, f1, &bars->fixed_full, x0 + half * 64, f_row, b);
  }
  int it = 0;
  bool ok = true;
  for (; it < n; ++it) {
    const int s = it % kStages;
    const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
    if (!mbar_wait(&bars->ring_empty[s], ph ^ 1u, abort_flag, p.st, where | (1u << 16))) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(&bars->ring_full[s], 2 * kTileBytes);
    const int row = (first_row_tile + it) * kT;
    uint8_t* dst = smem + kSmRing + s * 2 * kTileBytes;
    for (int half = 0; half < 2; ++half) {
      tma_load_3d_hint(dst + half * kHalfBytes, r0, &bars->ring_full[s], x0 + half * 64, row, b, pol);
      tma_load_3d_hint(dst + kTileBytes + half * kHalfBytes, r1, &bars->ring_full[s], x0 + half * 64, row, b, pol);
    }
  }
  if (!ok) {
    drain_wait(&bars->fixed_full, 0, p.st.limit);
    for (int k = std::max(0, it - kStages); k < it; ++k)
      drain_wait(&bars->ring_full[k % kStages], static_cast<uint32_t>(k / kStages) & 1u, p.st.limit);
  }
}

// 8 MMAs of K = 16 over a 128-deep contraction, both operands K-major SW128 tiles.
__device__ __forceinline__ void mma_tile_ss(uint32_t d, uint32_t a_base, uint32_t b_base, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
    mma_ss(d, sdesc_sw128(a_base + off, 16, 1024), sdesc_sw128(b_base + off, 16, 1024), idesc, kk > 0);
  }
}

// A (128 x 128 bf16) from TMEM columns a_col.., B an MN-major SW128 tile [K rows][N = 128].
__device__ __forceinline__ void mma_tile_ts(uint32_t d, uint32_t a_tmem, uint32_t b_base, uint32_t idesc,
                                            bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kT / 16; ++kk) {
    mma_ts(d, a_tmem + kk * 8, sdesc_sw128(b_base + kk * 2048, kHalfBytes, 1024), idesc, (accumulate || kk > 0));
  }
}

// Stores one 32-column chunk of a gradient row (fp32 accumulator values x mul).
__device__ __forceinline__ void store_grad_chunk(void* base, long long off, const uint32_t (&a)[32], float mul,
                                                 int mode) {
  if (mode == LCB_GRAD_BF16) {
    __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(base) + off;
#pragma unroll
    for (int i = 0; i < 32; i += 8) {
      uint4 v;
      v.x = pack_bf16x2(__uint_as_float(a[i]) * mul, __uint_as_float(a[i + 1]) * mul);
      v.y = pack_bf16x2(__uint_as_float(a[i + 2]) * mul, __uint_as_float(a[i + 3]) * mul);
      v.z = pack_bf16x2(__uint_as_float(a[i + 4]) * mul, __uint_as_float(a[i + 5]) * mul);
      v.w = pack_bf16x2(__uint_as_float(a[i + 6]) * mul, __uint_as_float(a[i + 7]) * mul);
      *reinterpret_cast<uint4*>(dst + i) = v;
    }
  } else {
    float* dst = static_cast<float*>(base) + off;
#pragma unroll
    for (int i = 0; i < 32; i += 4) {
      float4 v = make_float4(__uint_as_float(a[i]) * mul, __uint_as_float(a[i + 1]) * mul,
                             __uint_as_float(a[i + 2]) * mul, __uint_as_float(a[i + 3]) * mul);
      if (mode == LCB_GRAD_F32_ACCUM) {
        const float4 o = *reinterpret_cast<const float4*>(dst + i);
        v.x += o.x;
        v.y += o.y;
        v.z += o.z;
        v.w += o.w;
      }
      *reinterpret_cast<float4*>(dst + i) = v;
    }
  }
}

__device__ __forceinline__ void store_zero_row(void* base, long long off, int mode) {
  if (mode == LCB_GRAD_F32_ACCUM) return;
  if (mode == LCB_GRAD_BF16) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
    for (int i = 0; i < kD / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
  } else {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
    for (int i = 0; i < kD / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Natural-log LSE of a query row -> base-2, with hidden/empty rows mapped to +inf (P = 0).
__device__ __forceinline__ float lse2_of(const Params& p, int b, int h, int q) {
  if (q >= p.Sq) return INFINITY;
  const float l = __ldg(p.lse + b * p.l_bs + h * p.l_hs + q);
  return (l == -INFINITY) ? INFINITY : l * kLog2e;
}

// ============================================================== dK / dV pass
// TMEM: S^T [0,128) (P^T bf16 in [0,64)), dP^T [128,256) (dS^T in [128,192)),
// dV [256,384), dK [384,512). Fixed tiles: K, V. Ring: (Q_i, dO_i).
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                         const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kSmBar);
  volatile int* abort_flag = &bars->abort;
  float* stats = reinterpret_cast<float*>(smem + kSmStats);
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  constexpr uint32_t kWhere = 2u << 24;

  // Work item: key tile kt of (b, h); causal work shrinks with kt, so low kt first.
  const int nk = (p.Sk + kT - 1) / kT;
  const int nq = (p.Sq + kT - 1) / kT;
  const int BH = p.B * p.H;
  const int bh = blockIdx.x % BH;
  const int kt = static_cast<int>(blockIdx.x / BH);
  const int b = bh / p.H, h = bh % p.H;
  const int i0 = p.causal ? kt : 0;
  const int n = std::max(0, nq - i0);
  (void)nk;

  if (threadIdx.x == 0) init_bars(bars);
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0 && n > 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 4) {
    if (lane == 0 && n > 0) producer(smem, bars, &tm_k, &tm_v, kt * kT, &tm_q, &tm_do, i0, n, h, b, p, kWhere);
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0 && n > 0) {
      const uint32_t id_ss = idesc_bf16(kT, kT, false, false);
      const uint32_t id_ts = idesc_bf16(kT, kD, false, true);
      const uint32_t sK = sbase + kSmFixed, sV = sbase + kSmFixed + kTileBytes;
      bool ok = mbar_wait(&bars->fixed_full, 0, abort_flag, p.st, kWhere | (2u << 16));
      for (int it = 0; it < n && ok; ++it) {
        const int s = it % kStages;
        ok = mbar_wait(&bars->ring_full[s], static_cast<uint32_t>(it / kStages) & 1u, abort_flag, p.st,
                       kWhere | (3u << 16));
        if (!ok) break;
        tc_fence_after();
        const uint32_t sQ = sbase + kSmRing + s * 2 * kTileBytes, sdO = sQ + kTileBytes;
        mma_tile_ss(tbase + 0, sK, sQ, id_ss);     // S^T  = K Q^T
        mma_tile_ss(tbase + 128, sV, sdO, id_ss);  // dP^T = V dO^T
        tc_commit(&bars->s_full);
        ok = mbar_wait(&bars->p_full, static_cast<uint32_t>(it) & 1u, abort_flag, p.st, kWhere | (4u << 16));
        if (!ok) break;
        tc_fence_after();
        mma_tile_ts(tbase + 256, tbase + 0, sdO, id_ts, it > 0);   // dV += P^T dO
        mma_tile_ts(tbase + 384, tbase + 128, sQ, id_ts, it > 0);  // dK += dS^T Q
        tc_commit(&bars->ring_empty[s]);
      }
      if (ok) tc_commit(&bars->acc_full);
      tc_commit(&bars->mma_done);
      drain_wait(&bars->mma_done, 0, p.st.limit);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- compute
    const int row = threadIdx.x;  // key row within the tile, TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int j = kt * kT + row;
    const float c = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      const int i = i0 + it;
      float* buf = stats + (it & 1) * 2 * kT;
      {
        const int q = i * kT + row;
        buf[row] = lse2_of(p, b, h, q);
        buf[kT + row] = (q < p.Sq) ? __ldg(p.delta + b * p.l_bs + h * p.l_hs + q) : 0.f;
      }
      mbar_arrive(&bars->stats_full[it & 1]);
      ok = warp_all(mbar_wait(&bars->stats_full[it & 1], static_cast<uint32_t>(it >> 1) & 1u, abort_flag, p.st,
                              kWhere | (7u << 16)));
      if (!ok) break;
      ok = warp_all(mbar_wait(&bars->s_full, static_cast<uint32_t>(it) & 1u, abort_flag, p.st, kWhere | (5u << 16)));
      if (!ok) break;
      tc_fence_after();
      const bool diag = p.causal && (i == kt);
      const int qbase = i * kT;
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t s[32], dp[32];
        tmem_ld_x32(tbase + lane_off + ch * 32, s);
        tmem_ld_x32(tbase + lane_off + 128 + ch * 32, dp);
        uint32_t pk[16], dk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const int col = ch * 32 + e;
          const float4 l2 = *reinterpret_cast<const float4*>(buf + (col & ~3));
          const float4 dl = *reinterpret_cast<const float4*>(buf + kT + (col & ~3));
          const float l2a = (e & 2) ? l2.z : l2.x, l2b = (e & 2) ? l2.w : l2.y;
          const float dla = (e & 2) ? dl.z : dl.x, dlb = (e & 2) ? dl.w : dl.y;
          float p0 = ex2_approx(fmaf(__uint_as_float(s[e]), c, -l2a));
          float p1 = ex2_approx(fmaf(__uint_as_float(s[e + 1]), c, -l2b));
          if (diag) {
            if (qbase + col < j) p0 = 0.f;
            if (qbase + col + 1 < j) p1 = 0.f;
          }
          const float d0 = p0 * (__uint_as_float(dp[e]) - dla);
          const float d1 = p1 * (__uint_as_float(dp[e + 1]) - dlb);
          pk[e >> 1] = pack_bf16x2(p0, p1);
          dk[e >> 1] = pack_bf16x2(d0, d1);
        }
        tmem_st_x16(tbase + lane_off + ch * 16, pk);
        tmem_st_x16(tbase + lane_off + 128 + ch * 16, dk);
      }
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    const bool valid = j < p.Sk;
    const long long off = b * p.g_bs + static_cast<long long>(j) * p.g_rs + h * kD;
    if (n == 0) {
      if (valid) {
        store_zero_row(p.g0, off, p.grad_mode);
        store_zero_row(p.g1, off, p.grad_mode);
      }
    } else if (ok) {
      ok = warp_all(mbar_wait(&bars->acc_full, 0, abort_flag, p.st, kWhere | (6u << 16)));
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t a[32];
          tmem_ld_x32(tbase + lane_off + 256 + ch * 32, a);
          if (valid) store_grad_chunk(p.g1, off + ch * 32, a, 1.f, p.grad_mode);
          tmem_ld_x32(tbase + lane_off + 384 + ch * 32, a);
          if (valid) store_grad_chunk(p.g0, off + ch * 32, a, p.scale, p.grad_mode);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ============================================================== dQ pass
// TMEM: S [0,128) (dS bf16 in [0,64)), dP [128,256), dQ [256,384).
// Fixed tiles: Q, dO. Ring: (K_j, V_j).
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_do,
                       const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kSmBar);
  volatile int* abort_flag = &bars->abort;
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  constexpr uint32_t kWhere = 3u << 24;

  // Work item: query tile qt of (b, h); causal work grows with qt, so high qt first.
  const int nq = (p.Sq + kT - 1) / kT;
  const int nk = (p.Sk + kT - 1) / kT;
  const int BH = p.B * p.H;
  const int bh = blockIdx.x % BH;
  const int qt = nq - 1 - static_cast<int>(blockIdx.x / BH);
  const int b = bh / p.H, h = bh % p.H;
  const int n = p.causal ? std::min(nk, qt + 1) : nk;

  if (threadIdx.x == 0) init_bars(bars);
  if (warp == 5) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0 && n > 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 4) {
    if (lane == 0 && n > 0) producer(smem, bars, &tm_q, &tm_do, qt * kT, &tm_k, &tm_v, 0, n, h, b, p, kWhere);
    __syncwarp();
  } else if (warp == 5) {
    if (lane == 0 && n > 0) {
      const uint32_t id_ss = idesc_bf16(kT, kT, false, false);
      const uint32_t id_ts = idesc_bf16(kT, kD, false, true);
      const uint32_t sQ = sbase + kSmFixed, sdO = sbase + kSmFixed + kTileBytes;
      bool ok = mbar_wait(&bars->fixed_full, 0, abort_flag, p.st, kWhere | (2u << 16));
      for (int it = 0; it < n && ok; ++it) {
        const int s = it % kStages;
        ok = mbar_wait(&bars->ring_full[s], static_cast<uint32_t>(it / kStages) & 1u, abort_flag, p.st,
                       kWhere | (3u << 16));
        if (!ok) break;
        tc_fence_after();
        const uint32_t sK = sbase + kSmRing + s * 2 * kTileBytes, sV = sK + kTileBytes;
        mma_tile_ss(tbase + 0, sQ, sK, id_ss);     // S  = Q K^T
        mma_tile_ss(tbase + 128, sdO, sV, id_ss);  // dP = dO V^T
        tc_commit(&bars->s_full);
        ok = mbar_wait(&bars->p_full, static_cast<uint32_t>(it) & 1u, abort_flag, p.st, kWhere | (4u << 16));
        if (!ok) break;
        tc_fence_after();
        mma_tile_ts(tbase + 256, tbase + 0, sK, id_ts, it > 0);  // dQ += dS K
        tc_commit(&bars->ring_empty[s]);
      }
      if (ok) tc_commit(&bars->acc_full);
      tc_commit(&bars->mma_done);
      drain_wait(&bars->mma_done, 0, p.st.limit);
    }
    __syncwarp();
  } else {
    const int row = threadIdx.x;
    const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;
    const int qi = qt * kT + row;
    const float c = p.scale_log2;
    const float l2 = lse2_of(p, b, h, qi);
    const float dl = (qi < p.Sq) ? __ldg(p.delta + b * p.l_bs + h * p.l_hs + qi) : 0.f;
    const int q_first = qt * kT;
    bool ok = true;
    for (int it = 0; it < n; ++it) {
      ok = warp_all(mbar_wait(&bars->s_full, static_cast<uint32_t>(it) & 1u, abort_flag, p.st, kWhere | (5u << 16)));
      if (!ok) break;
      tc_fence_after();
      const int kbase = it * kT;
      const bool need_mask = (p.causal && kbase + kT - 1 > q_first) || (kbase + kT > p.Sk);
      const int lim = p.causal ? std::min(qi + 1, p.Sk) : p.Sk;  // keys < lim are visible
#pragma unroll 1
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t s[32], dp[32];
        tmem_ld_x32(tbase + lane_off + ch * 32, s);
        tmem_ld_x32(tbase + lane_off + 128 + ch * 32, dp);
        uint32_t ds[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float p0 = ex2_approx(fmaf(__uint_as_float(s[e]), c, -l2));
          float p1 = ex2_approx(fmaf(__uint_as_float(s[e + 1]), c, -l2));
          if (need_mask) {
            const int key = kbase + ch * 32 + e;
            if (key >= lim) p0 = 0.f;
            if (key + 1 >= lim) p1 = 0.f;
          }
          ds[e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - dl), p1 * (__uint_as_float(dp[e + 1]) - dl));
        }
        tmem_st_x16(tbase + lane_off + ch * 16, ds);
      }
      tc_fence_before();
      mbar_arrive(&bars->p_full);
    }
    const bool valid = qi < p.Sq;
    const long long off = b * p.g_bs + static_cast<long long>(qi) * p.g_rs + h * kD;
    if (n == 0) {
      if (valid) store_zero_row(p.g0, off, p.grad_mode);
    } else if (ok) {
      ok = warp_all(mbar_wait(&bars->acc_full, 0, abort_flag, p.st, kWhere | (6u << 16)));
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t a[32];
          tmem_ld_x32(tbase + lane_off + 256 + ch * 32, a);
          if (valid) store_grad_chunk(p.g0, off + ch * 32, a, p.scale, p.grad_mode);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

int make_maps(const BwdLaunch& a, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tdo) {
  int rc;
  const int HD = a.H * kD;
  // An empty side is never loaded (the kernel's loop count is 0): its maps stay zeroed.
  memset(tq, 0, sizeof(CUtensorMap));
  memset(tdo, 0, sizeof(CUtensorMap));
  memset(tk, 0, sizeof(CUtensorMap));
  memset(tv, 0, sizeof(CUtensorMap));
  if (a.Sq > 0) {
    if ((rc = make_tma_map_bf16(tq, a.q, a.B, a.Sq, HD, kT)) != 0) return rc;
    if ((rc = make_tma_map_bf16(tdo, a.dO, a.B, a.Sq, HD, kT)) != 0) return rc;
  }
  if (a.Sk > 0) {
    if ((rc = make_tma_map_bf16(tk, a.k, a.B, a.Sk, HD, kT)) != 0) return rc;
    if ((rc = make_tma_map_bf16(tv, a.v, a.B, a.Sk, HD, kT)) != 0) return rc;
  }
  return 0;
}

Params base_params(const BwdLaunch& a) {
  Params p;
  p.lse = a.lse;
  p.delta = a.delta;
  p.l_hs = a.lse_head_stride;
  p.l_bs = a.lse_batch_stride;
  p.B = a.B;
  p.H = a.H;
  p.Sq = a.Sq;
  p.Sk = a.Sk;
  p.causal = a.causal;
  p.grad_mode = a.grad_mode;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.st = a.st;
  return p;
}

}  // namespace

int launch_attn_bwd_dkdv(const BwdLaunch& a, cudaStream_t stream) {
  if (a.Sk == 0) return 0;
  CUtensorMap tq, tk, tv, tdo;
  int rc = make_maps(a, &tq, &tk, &tv, &tdo);
  if (rc != 0) return rc;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return -4;
    attr = true;
  }
  Params p = base_params(a);
  p.g0 = a.dk;
  p.g1 = a.dv;
  p.g_rs = a.dkv_row_stride;
  p.g_bs = a.dkv_batch_stride;
  const long long grid = static_cast<long long>((a.Sk + kT - 1) / kT) * a.B * a.H;
  if (grid > 0x7fffffffLL) return -1;
  attn_bwd_dkdv_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_attn_bwd_dq(const BwdLaunch& a, cudaStream_t stream) {
  if (a.Sq == 0) return 0;
  CUtensorMap tq, tk, tv, tdo;
  int rc = make_maps(a, &tq, &tk, &tv, &tdo);
  if (rc != 0) return rc;
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(attn_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes) !=
        cudaSuccess)
      return -4;
    attr = true;
  }
  Params p = base_params(a);
  p.g0 = a.dq;
  p.g1 = nullptr;
  p.g_rs = a.dq_row_stride;
  p.g_bs = a.dq_batch_stride;
  const long long grid = static_cast<long long>((a.Sq + kT - 1) / kT) * a.B * a.H;
  if (grid > 0x7fffffffLL) return -1;
  attn_bwd_dq_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tq, tk, tv, tdo, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace lcb
