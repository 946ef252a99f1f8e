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
//     S^T = K Q^T and dP^T = V dO^T land in TMEM with one key per lane, so the
//     per-query statistics (LSE, Delta) are columns, staged in shared memory.
//     P^T and dS^T (bf16) overwrite S^T and dP^T in TMEM and feed
//     dV += P^T dO and dK += dS^T Q directly from TMEM.
//   dQ pass: one CTA per 128-query tile, looping over key tiles.
//     S = Q K^T and dP = dO V^T with one query per lane; dS (bf16) overwrites
//     S in TMEM and feeds dQ += dS K.
//
// Each streamed 128-row tile is handled as two 64-row halves with their own
// TMEM buffers and barriers: while the compute warps turn half h of one tile
// into P/dS, the tensor core multiplies the other half, so elementwise work
// and MMA overlap. Streamed operands arrive as 64-row half tiles in a 4-slot
// ring, so a slot is refilled one full tile ahead of its use.
//
// Warps: 0-3 and 4-7 are two compute warpgroups, warpgroup h owning half h
// (thread = TMEM lane = tile row); warp 8 is the TMA producer, warp 9 the MMA
// issuer and TMEM owner.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "lcb_attn.h"
#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kT = 128;  // rows per tile (both query and key tiles)
constexpr int kHalf = 64;
constexpr int kD = 128;
constexpr int kThreads = 320;  // 8 compute warps (2 warpgroups), producer, MMA issuer
constexpr uint32_t kTileBytes = kT * kD * 2;      // 32 KB: two 16 KB boxes of 128 rows x 64 columns
constexpr uint32_t kTileColHalf = kTileBytes / 2;  // column-half stride inside a full tile
constexpr uint32_t kHtBytes = kHalf * kD * 2;      // 16 KB half tile: two 8 KB boxes of 64 rows x 64 columns
constexpr uint32_t kHtColHalf = kHtBytes / 2;      // column-half stride inside a half tile
constexpr int kStages = 4;                         // ring slots, each (half tile A, half tile B) = 32 KB
constexpr float kLog2e = 1.4426950408889634f;

// Fixed operands (2 full tiles), the ring, per-query stats, barriers.
constexpr uint32_t kSmFixed = 0;
constexpr uint32_t kSmRing = 2 * kTileBytes;
constexpr uint32_t kSmStats = kSmRing + kStages * 2 * kHtBytes;  // [warpgroup][parity] x (lse2[64], delta[64]) fp32
constexpr uint32_t kSmBar = kSmStats + 2 * 2 * kT * 4;

struct Bars {
  uint64_t fixed_full;
  uint64_t ring_full[kStages];
  uint64_t ring_empty[kStages];
  uint64_t s_full[2];      // per half: S (and dP) accumulated in TMEM
  uint64_t p_full[2];      // per half: P / dS written back to TMEM
  uint64_t acc_full;
  uint64_t mma_done;
  uint64_t stats_full[2][2];  // dK/dV pass: [warpgroup][parity], that warpgroup staged its LSE/Delta half
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
  for (int h = 0; h < 2; ++h) {
    mbar_init(&bars->s_full[h], 1);
    mbar_init(&bars->p_full[h], kT);
    mbar_init(&bars->stats_full[h][0], kT);
    mbar_init(&bars->stats_full[h][1], kT);
  }
  mbar_init(&bars->acc_full, 1);
  mbar_init(&bars->mma_done, 1);
  bars->abort = 0;
  fence_mbar_init();
}

// Loads two fixed full tiles (rows f_row..f_row+127 of f0 and f1) once, then
// ring items m = 0 .. 2n-1: the half tile of rows (first_tile + m/2)*128 +
// (m%2)*64 of r0 and of r1.
__device__ void producer(uint8_t* smem, Bars* bars, const CUtensorMap* f0, const CUtensorMap* f1, int f_row,
                         const CUtensorMap* r0, const CUtensorMap* r1, int first_tile, int n, int h, int b,
                         const Params& p, uint32_t where) {
  volatile int* abort_flag = &bars->abort;
  const int x0 = h * kD;
  const uint64_t pol = l2_policy_evict_last();
  mbar_arrive_expect_tx(&bars->fixed_full, 2 * kTileBytes);
  for (int c = 0; c < 2; ++c) {
    tma_load_3d(smem + kSmFixed + c * kTileColHalf, f0, &bars->fixed_full, x0 + c * 64, f_row, b);
    tma_load_3d(smem + kSmFixed + kTileBytes + c * kTileColHalf, f1, &bars->fixed_full, x0 + c * 64, f_row, b);
  }
  const int items = 2 * n;
  int m = 0;
  bool ok = true;
  for (; m < items; ++m) {
    const int s = m % kStages;
    const uint32_t ph = static_cast<uint32_t>(m / kStages) & 1u;
    if (!mbar_wait(&bars->ring_empty[s], ph ^ 1u, abort_flag, p.st, where | (1u << 16))) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(&bars->ring_full[s], 2 * kHtBytes);
    const int row = (first_tile + (m >> 1)) * kT + (m & 1) * kHalf;
    uint8_t* dst = smem + kSmRing + s * 2 * kHtBytes;
    for (int c = 0; c < 2; ++c) {
      tma_load_3d_hint(dst + c * kHtColHalf, r0, &bars->ring_full[s], x0 + c * 64, row, b, pol);
      tma_load_3d_hint(dst + kHtBytes + c * kHtColHalf, r1, &bars->ring_full[s], x0 + c * 64, row, b, pol);
    }
  }
  if (!ok) {
    drain_wait(&bars->fixed_full, 0, p.st.limit);
    for (int k = std::max(0, m - kStages); k < m; ++k)
      drain_wait(&bars->ring_full[k % kStages], static_cast<uint32_t>(k / kStages) & 1u, p.st.limit);
  }
}

// D (128 x 64) = A (full tile, K-major) x B^T (half tile of 64 rows, K-major), contraction over D = 128.
__device__ __forceinline__ void mma_full_x_half(uint32_t d, uint32_t a_base, uint32_t b_base, uint32_t idesc) {
#pragma unroll
  for (int kk = 0; kk < kD / 16; ++kk) {
    const uint32_t a_off = (kk >> 2) * kTileColHalf + (kk & 3) * 32;
    const uint32_t b_off = (kk >> 2) * kHtColHalf + (kk & 3) * 32;
    mma_ss(d, sdesc_sw128(a_base + a_off, 16, 1024), sdesc_sw128(b_base + b_off, 16, 1024), idesc, kk > 0);
  }
}

// D (128 x 128) (+)= A (TMEM, 128 x 64 bf16 in 32 columns) x B (half tile [64 rows = K][128 = N], MN-major).
__device__ __forceinline__ void mma_tmem_x_half(uint32_t d, uint32_t a_tmem, uint32_t b_base, uint32_t idesc,
                                                bool accumulate) {
#pragma unroll
  for (int kk = 0; kk < kHalf / 16; ++kk) {
    mma_ts(d, a_tmem + kk * 8, sdesc_sw128(b_base + kk * 2048, kHtColHalf, 1024), idesc, (accumulate || kk > 0));
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

__device__ __forceinline__ void store_zero_half_row(void* base, long long off, int mode) {
  if (mode == LCB_GRAD_F32_ACCUM) return;
  if (mode == LCB_GRAD_BF16) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
#pragma unroll
    for (int i = 0; i < kHalf / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
  } else {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
#pragma unroll
    for (int i = 0; i < kHalf / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Natural-log LSE of a query row -> base-2, with hidden/empty rows mapped to +inf (P = 0).
__device__ __forceinline__ float lse2_of(const Params& p, int b, int h, int q) {
  if (q >= p.Sq) return INFINITY;
  const float l = __ldg(p.lse + b * p.l_bs + h * p.l_hs + q);
  return (l == -INFINITY) ? INFINITY : l * kLog2e;
}

// ============================================================== dK / dV pass
// TMEM, per half h of the query tile: S^T_h [128h, 128h+64) (P^T_h bf16 in its
// first 32 columns), dP^T_h [128h+64, 128h+128) (dS^T_h in its first 32).
// dV [256,384), dK [384,512). Fixed tiles: K, V. Ring items: (Q half, dO half).
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
  const int nq = (p.Sq + kT - 1) / kT;
  const int BH = p.B * p.H;
  const int bh = blockIdx.x % BH;
  const int kt = static_cast<int>(blockIdx.x / BH);
  const int b = bh / p.H, h = bh % p.H;
  const int i0 = p.causal ? kt : 0;
  const int n = std::max(0, nq - i0);

  if (threadIdx.x == 0) init_bars(bars);
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0 && n > 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 8) {
    if (lane == 0 && n > 0) producer(smem, bars, &tm_k, &tm_v, kt * kT, &tm_q, &tm_do, i0, n, h, b, p, kWhere);
    __syncwarp();
  } else if (warp == 9) {
    if (lane == 0 && n > 0) {
      const uint32_t id_s = idesc_bf16(kT, kHalf, false, false);  // 128 x 64 score half
      const uint32_t id_g = idesc_bf16(kT, kD, false, true);      // 128 x 128 gradient update
      const uint32_t sK = sbase + kSmFixed, sV = sbase + kSmFixed + kTileBytes;
      auto item_q = [&](int m) { return sbase + kSmRing + (m % kStages) * 2 * kHtBytes; };
      auto issue_scores = [&](int hh, int m) {  // S^T_h = K Q_h^T, dP^T_h = V dO_h^T
        mma_full_x_half(tbase + 128 * hh, sK, item_q(m), id_s);
        mma_full_x_half(tbase + 128 * hh + 64, sV, item_q(m) + kHtBytes, id_s);
      };
      auto wait_item = [&](int m) {
        const bool r = mbar_wait(&bars->ring_full[m % kStages], static_cast<uint32_t>(m / kStages) & 1u, abort_flag,
                                 p.st, kWhere | (3u << 16));
        tc_fence_after();
        return r;
      };
      bool ok = mbar_wait(&bars->fixed_full, 0, abort_flag, p.st, kWhere | (2u << 16));
      for (int hh = 0; hh < 2 && ok; ++hh) {
        ok = wait_item(hh);
        if (!ok) break;
        issue_scores(hh, hh);
        tc_commit(&bars->s_full[hh]);
      }
      for (int it = 0; it < n && ok; ++it) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (!ok) continue;
          const int m = 2 * it + hh;
          ok = mbar_wait(&bars->p_full[hh], static_cast<uint32_t>(it) & 1u, abort_flag, p.st, kWhere | (4u << 16));
          if (!ok) continue;
          tc_fence_after();
          const bool acc = it > 0 || hh > 0;
          mma_tmem_x_half(tbase + 256, tbase + 128 * hh, item_q(m) + kHtBytes, id_g, acc);  // dV += P^T_h dO_h
          mma_tmem_x_half(tbase + 384, tbase + 128 * hh + 64, item_q(m), id_g, acc);        // dK += dS^T_h Q_h
          tc_commit(&bars->ring_empty[m % kStages]);
          if (it + 1 < n) {
            ok = wait_item(m + 2);
            if (!ok) continue;
            issue_scores(hh, m + 2);
            tc_commit(&bars->s_full[hh]);
          }
        }
      }
      if (ok) tc_commit(&bars->acc_full);
      tc_commit(&bars->mma_done);
      drain_wait(&bars->mma_done, 0, p.st.limit);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- compute
    const int hh = warp >> 2;          // this warpgroup's half of every query tile
    const int row = threadIdx.x & 127;  // key row within the tile, TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + 128 * hh;
    const int j = kt * kT + row;
    const float c = p.scale_log2;
    bool ok = true;
    for (int it = 0; it < n && ok; ++it) {
      const int i = i0 + it;
      const int qh = i * kT + hh * kHalf;  // first query of this half
      float* buf = stats + (hh * 2 + (it & 1)) * 2 * kHalf;
      if (row < kHalf) {
        buf[row] = lse2_of(p, b, h, qh + row);
        buf[kHalf + row] = (qh + row < p.Sq) ? __ldg(p.delta + b * p.l_bs + h * p.l_hs + qh + row) : 0.f;
      }
      mbar_arrive(&bars->stats_full[hh][it & 1]);
      ok = warp_all(mbar_wait(&bars->stats_full[hh][it & 1], static_cast<uint32_t>(it >> 1) & 1u, abort_flag, p.st,
                              kWhere | (7u << 16)));
      if (ok) {
        ok = warp_all(
            mbar_wait(&bars->s_full[hh], static_cast<uint32_t>(it) & 1u, abort_flag, p.st, kWhere | (5u << 16)));
      }
      if (!ok) break;
      tc_fence_after();
      const bool diag = p.causal && (i == kt);
#pragma unroll 1
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t s[32], dp[32];
        tmem_ld2_x32(tS + ch * 32, tS + 64 + ch * 32, s, dp);
        uint32_t pk[16], dk[16];
        const int cb = ch * 32;  // query column within the half
#pragma unroll
        for (int e = 0; e < 32; e += 4) {
          const float4 l2 = *reinterpret_cast<const float4*>(buf + cb + e);
          const float4 dl = *reinterpret_cast<const float4*>(buf + kHalf + cb + e);
          float p0 = ex2_approx(fmaf(__uint_as_float(s[e]), c, -l2.x));
          float p1 = ex2_approx(fmaf(__uint_as_float(s[e + 1]), c, -l2.y));
          float p2 = ex2_approx(fmaf(__uint_as_float(s[e + 2]), c, -l2.z));
          float p3 = ex2_approx(fmaf(__uint_as_float(s[e + 3]), c, -l2.w));
          if (diag) {
            const int q0 = qh + cb + e;
            if (q0 < j) p0 = 0.f;
            if (q0 + 1 < j) p1 = 0.f;
            if (q0 + 2 < j) p2 = 0.f;
            if (q0 + 3 < j) p3 = 0.f;
          }
          pk[e >> 1] = pack_bf16x2(p0, p1);
          pk[(e >> 1) + 1] = pack_bf16x2(p2, p3);
          dk[e >> 1] = pack_bf16x2(p0 * (__uint_as_float(dp[e]) - dl.x), p1 * (__uint_as_float(dp[e + 1]) - dl.y));
          dk[(e >> 1) + 1] =
              pack_bf16x2(p2 * (__uint_as_float(dp[e + 2]) - dl.z), p3 * (__uint_as_float(dp[e + 3]) - dl.w));
        }
        tmem_st_x16_nowait(tS + ch * 16, pk);
        tmem_st_x16_nowait(tS + 64 + ch * 16, dk);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[hh]);
    }
    // Epilogue: warpgroup 0 writes dV, warpgroup 1 writes dK (scaled).
    const bool valid = j < p.Sk;
    const long long off = b * p.g_bs + static_cast<long long>(j) * p.g_rs + h * kD;
    void* gdst = hh == 0 ? p.g1 : p.g0;
    const float mul = hh == 0 ? 1.f : p.scale;
    if (n == 0) {
      if (valid) store_zero_row(gdst, off, p.grad_mode);
    } else if (ok) {
      ok = warp_all(mbar_wait(&bars->acc_full, 0, abort_flag, p.st, kWhere | (6u << 16)));
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < 4; ++ch) {
          uint32_t a[32];
          tmem_ld_x32(tbase + lane_off + 256 + 128 * hh + ch * 32, a);
          if (valid) store_grad_chunk(gdst, off + ch * 32, a, mul, p.grad_mode);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ============================================================== dQ pass
// TMEM, per half h of the key tile: S_h [128h, 128h+64) (dS_h bf16 in its
// first 32 columns), dP_h [128h+64, 128h+128); dQ [256,384).
// Fixed tiles: Q, dO. Ring items: (K half, V half).
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
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0 && n > 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
    tma_prefetch_desc(&tm_do);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 8) {
    if (lane == 0 && n > 0) producer(smem, bars, &tm_q, &tm_do, qt * kT, &tm_k, &tm_v, 0, n, h, b, p, kWhere);
    __syncwarp();
  } else if (warp == 9) {
    if (lane == 0 && n > 0) {
      const uint32_t id_s = idesc_bf16(kT, kHalf, false, false);
      const uint32_t id_g = idesc_bf16(kT, kD, false, true);
      const uint32_t sQ = sbase + kSmFixed, sdO = sbase + kSmFixed + kTileBytes;
      auto item_k = [&](int m) { return sbase + kSmRing + (m % kStages) * 2 * kHtBytes; };
      auto issue_scores = [&](int hh, int m) {  // S_h = Q K_h^T, dP_h = dO V_h^T
        mma_full_x_half(tbase + 128 * hh, sQ, item_k(m), id_s);
        mma_full_x_half(tbase + 128 * hh + 64, sdO, item_k(m) + kHtBytes, id_s);
      };
      auto wait_item = [&](int m) {
        const bool r = mbar_wait(&bars->ring_full[m % kStages], static_cast<uint32_t>(m / kStages) & 1u, abort_flag,
                                 p.st, kWhere | (3u << 16));
        tc_fence_after();
        return r;
      };
      bool ok = mbar_wait(&bars->fixed_full, 0, abort_flag, p.st, kWhere | (2u << 16));
      for (int hh = 0; hh < 2 && ok; ++hh) {
        ok = wait_item(hh);
        if (!ok) break;
        issue_scores(hh, hh);
        tc_commit(&bars->s_full[hh]);
      }
      for (int it = 0; it < n && ok; ++it) {
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          if (!ok) continue;
          const int m = 2 * it + hh;
          ok = mbar_wait(&bars->p_full[hh], static_cast<uint32_t>(it) & 1u, abort_flag, p.st, kWhere | (4u << 16));
          if (!ok) continue;
          tc_fence_after();
          mma_tmem_x_half(tbase + 256, tbase + 128 * hh, item_k(m), id_g, it > 0 || hh > 0);  // dQ += dS_h K_h
          tc_commit(&bars->ring_empty[m % kStages]);
          if (it + 1 < n) {
            ok = wait_item(m + 2);
            if (!ok) continue;
            issue_scores(hh, m + 2);
            tc_commit(&bars->s_full[hh]);
          }
        }
      }
      if (ok) tc_commit(&bars->acc_full);
      tc_commit(&bars->mma_done);
      drain_wait(&bars->mma_done, 0, p.st.limit);
    }
    __syncwarp();
  } else {
    const int hh = warp >> 2;  // this warpgroup's half of every key tile
    const int row = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + lane_off + 128 * hh;
    const int qi = qt * kT + row;
    const float c = p.scale_log2;
    const float l2 = lse2_of(p, b, h, qi);
    const float dl = (qi < p.Sq) ? __ldg(p.delta + b * p.l_bs + h * p.l_hs + qi) : 0.f;
    const int q_first = qt * kT;
    const int lim = p.causal ? std::min(qi + 1, p.Sk) : p.Sk;  // keys < lim are visible
    bool ok = true;
    for (int it = 0; it < n && ok; ++it) {
      ok = warp_all(
          mbar_wait(&bars->s_full[hh], static_cast<uint32_t>(it) & 1u, abort_flag, p.st, kWhere | (5u << 16)));
      if (!ok) break;
      tc_fence_after();
      const int kbase = it * kT + hh * kHalf;
      const bool need_mask = (p.causal && kbase + kHalf - 1 > q_first) || (kbase + kHalf > p.Sk);
#pragma unroll 1
      for (int ch = 0; ch < 2; ++ch) {
        uint32_t s[32], dp[32];
        tmem_ld2_x32(tS + ch * 32, tS + 64 + ch * 32, s, dp);
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
        tmem_st_x16_nowait(tS + ch * 16, ds);
      }
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->p_full[hh]);
    }
    // Epilogue: warpgroup h writes dQ columns [64h, 64h + 64).
    const bool valid = qi < p.Sq;
    const long long off = b * p.g_bs + static_cast<long long>(qi) * p.g_rs + h * kD + hh * kHalf;
    if (n == 0) {
      if (valid) store_zero_half_row(p.g0, off, p.grad_mode);
    } else if (ok) {
      ok = warp_all(mbar_wait(&bars->acc_full, 0, abort_flag, p.st, kWhere | (6u << 16)));
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t a[32];
          tmem_ld_x32(tbase + lane_off + 256 + hh * kHalf + ch * 32, a);
          if (valid) store_grad_chunk(p.g0, off + ch * 32, a, p.scale, p.grad_mode);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// Maps for one pass: the fixed operands use 128-row boxes, the streamed ones 64-row boxes.
// An empty side is never loaded (the loop count is 0): its maps stay zeroed.
int make_maps(const BwdLaunch& a, bool dkdv, CUtensorMap* tq, CUtensorMap* tk, CUtensorMap* tv, CUtensorMap* tdo) {
  int rc;
  const int HD = a.H * kD;
  memset(tq, 0, sizeof(CUtensorMap));
  memset(tdo, 0, sizeof(CUtensorMap));
  memset(tk, 0, sizeof(CUtensorMap));
  memset(tv, 0, sizeof(CUtensorMap));
  const int q_box = dkdv ? kHalf : kT;
  const int k_box = dkdv ? kT : kHalf;
  if (a.Sq > 0) {
    if ((rc = make_tma_map_bf16(tq, a.q, a.B, a.Sq, HD, q_box)) != 0) return rc;
    if ((rc = make_tma_map_bf16(tdo, a.dO, a.B, a.Sq, HD, q_box)) != 0) return rc;
  }
  if (a.Sk > 0) {
    if ((rc = make_tma_map_bf16(tk, a.k, a.B, a.Sk, HD, k_box)) != 0) return rc;
    if ((rc = make_tma_map_bf16(tv, a.v, a.B, a.Sk, HD, k_box)) != 0) return rc;
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
  int rc = make_maps(a, true, &tq, &tk, &tv, &tdo);
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
  int rc = make_maps(a, false, &tq, &tk, &tv, &tdo);
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
