// Backward kernels: gradients of exact attention by recomputation
// ("EasyContext核心技术解析：序列并行与Flash Attention的完美结合", §2 "Flash
// Attention优化": the backward recomputes the probabilities tile by tile from
// the stored row statistics instead of keeping the score matrix).
//
// With P_ij = exp(scale q_i.k_j - LSE_i), dP_ij = dO_i.v_j and
// dS_ij = P_ij (dP_ij - Delta_i):
//   dV_j = sum_i P_ij dO_i,  dK_j = scale sum_i dS_ij q_i,  dQ_i = scale sum_j dS_ij k_j.
//
// Two forms:
//   one pass (attn_bwd's): one CTA per 128-key tile, looping over 128-query
//     tiles, forming dK, dV and every query tile's dQ partial; the partials
//     are added into a tiled fp32 accumulator in L2, half by bulk
//     asynchronous reductions from shared memory, half by vector reductions
//     from registers (five MMAs per tile pair; dQ's summation order is not
//     fixed);
//   two passes, each deterministic (no reductions across CTAs):
//     dK/dV pass: one CTA per 128-key tile, looping over 128-query tiles;
//     dQ pass:    one CTA per 128-query tile, looping over 128-key tiles
//     (seven MMAs per tile pair: dQ's pass recomputes S and dP).
//
// Every MMA is M=128 x N=128 x K=16: on this part a tcgen05.mma instruction
// with N <= 128 costs about the same time whatever N is, so the work is issued
// as few, full-width instructions. To keep the tensor core busy while the
// compute warps turn scores into probabilities, a score buffer in TMEM is
// released as soon as its values are in registers, and dS (the A operand of
// dK or dQ) goes to shared memory in the 128-byte-swizzled K-major layout. The
// next tile's score products then run during the elementwise work.
//
// Warps: 0-15 are four compute warpgroups (thread = TMEM lane = row of the
// CTA's fixed tile); warpgroup x owns columns [32x, 32x+32) of each score
// tile. Warp 16 is the TMA producer, warp 17 the MMA issuer and TMEM owner,
// and in the one-pass kernel warp 18 adds the staged dQ blocks into global
// memory.
#include <cuda_bf16.h>

#include <algorithm>
#include <cstring>

#include "lcb_attn.h"
#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kT = 128;  // rows of every tile
constexpr int kD = 128;
constexpr int kThreads = 576;                    // 16 compute warps, producer, MMA issuer
constexpr int kCompute = 512;                    // compute threads
constexpr int kProducerWarp = 16;
constexpr int kMmaWarp = 17;
constexpr uint32_t kTileBytes = kT * kD * 2;     // 32 KB: two 16 KB boxes of 128 rows x 64 columns
constexpr uint32_t kColHalf = kTileBytes / 2;    // column-half stride of a tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxStages = 3;

struct Bars {
  uint64_t fixed_full;  // the CTA's fixed operands are in place
  uint64_t ring_full[kMaxStages];  // dK/dV pass: the Q ring; dQ pass: the (K, V) ring
  uint64_t ring_empty[kMaxStages];
  uint64_t do_full[2];  // dK/dV pass: the dO ring
  uint64_t do_empty[2];
  uint64_t s_full;    // S (S^T) computed
  uint64_t dp_full;   // dP (dP^T) computed
  uint64_t s_free;    // dQ pass: S and dP loaded by every compute thread
  uint64_t dp_free;   // dK/dV pass: dP^T loaded by every compute thread
  uint64_t p_full;    // dS written to shared memory (dK/dV pass: dS^T)
  uint64_t pt_full;   // dK/dV pass: P^T written to TMEM
  uint64_t ds_free;   // the MMA that read dS from shared memory completed
  uint64_t acc_full;
  uint64_t dq_full;   // fused pass: the dQ partial of one query tile is in TMEM
  uint64_t dq_free;   // fused pass: it was loaded by every compute thread
  uint64_t stg_full[2];  // fused pass: warpgroup x's (x = 0, 1) dQ block is staged
  uint64_t stg_free[2];  // fused pass: warpgroup x's staged block was read by the reducer
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};

// Fused pass: one block of the launch, query rows [q_off, q_off + q_len)
// against key rows [k_off, k_off + k_len); its CTAs start at cta0.
struct BwdTaskP {
  int q_off, q_len, k_off, k_len, causal, cta0;
};

struct Params {
  const float* lse;
  const float* delta;
  long long l_hs, l_bs;
  const __nv_bfloat16* f0;  // dQ pass: Q and dO, written into TMEM as A operands
  const __nv_bfloat16* f1;
  long long f_rs, f_bs;
  void* g0;  // dK (dK/dV and fused passes) or dQ (dQ pass)
  void* g1;  // dV (dK/dV and fused passes)
  long long g_rs, g_bs;
  float* dq_acc;  // fused pass: tiled fp32 dQ accumulator, added into
  long long dq_hs, dq_bs;  // its head and batch strides (floats)
  int n_tasks;             // fused pass: blocks of the launch (rows into the shared tensors)
  BwdTaskP task[kMaxBwdTasks];
  int B, H, Sq, Sk, causal, grad_mode;
  float scale, scale_log2;
  DevStatus st;
};


__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void init_bars(Bars* bars, int stages, uint32_t fixed_count) {
  mbar_init(&bars->fixed_full, fixed_count);
  for (int s = 0; s < stages; ++s) {
    mbar_init(&bars->ring_full[s], 1);
    mbar_init(&bars->ring_empty[s], 1);
  }
  mbar_init(&bars->s_full, 1);
  mbar_init(&bars->dp_full, 1);
  mbar_init(&bars->s_free, kCompute);
  mbar_init(&bars->dp_free, kCompute);
  mbar_init(&bars->p_full, kCompute);
  mbar_init(&bars->pt_full, kCompute);
  mbar_init(&bars->ds_free, 1);
  mbar_init(&bars->acc_full, 1);
  mbar_init(&bars->dq_full, 1);
  mbar_init(&bars->dq_free, kCompute);
  mbar_init(&bars->mma_done, 1);
  for (int s = 0; s < 2; ++s) {
    mbar_init(&bars->do_full[s], 1);
    mbar_init(&bars->do_empty[s], 1);
  }
  bars->abort = 0;
  fence_mbar_init();
}

// Loads one 128-row tile (two 64-column boxes) of `map` at row `row`.
__device__ __forceinline__ void load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar, int x0, int row, int b,
                                          uint64_t pol) {
  tma_load_3d_hint(dst, map, bar, x0, row, b, pol);
  tma_load_3d_hint(dst + kColHalf, map, bar, x0 + 64, row, b, pol);
}

// Streams tiles i = 0 .. n-1 (rows (first_tile + i) * 128) of r0 and r1 into
// ring slot i % kStages laid out [r0 tile][r1 tile].
template <int kStages>
__device__ void stream_tiles(uint8_t* ring, Bars* bars, const CUtensorMap* r0, const CUtensorMap* r1, int first_tile,
                             int n, int h, int b, const Params& p, uint32_t where) {
  volatile int* abort_flag = &bars->abort;
  const int x0 = h * kD;
  const uint64_t pol = l2_policy_evict_last();
  int i = 0;
  bool ok = true;
  for (; i < n; ++i) {
    const int s = i % kStages;
    const uint32_t ph = static_cast<uint32_t>(i / kStages) & 1u;
    if (!mbar_wait(&bars->ring_empty[s], ph ^ 1u, abort_flag, p.st, where | (1u << 16))) {
      ok = false;
      break;
    }
    mbar_arrive_expect_tx(&bars->ring_full[s], 2 * kTileBytes);
    uint8_t* dst = ring + s * 2 * kTileBytes;
    const int row = (first_tile + i) * kT;
    load_tile(dst, r0, &bars->ring_full[s], x0, row, b, pol);
    load_tile(dst + kTileBytes, r1, &bars->ring_full[s], x0, row, b, pol);
  }
  if (!ok) {
    for (int k = std::max(0, i - kStages); k < i; ++k)
      drain_wait(&bars->ring_full[k % kStages], static_cast<uint32_t>(k / kStages) & 1u, p.st.limit);
  }
}

// Each thread copies row `row` (D = 128 bf16) of a fixed operand into TMEM as
// A-operand columns (bf16 pairs, lane = row); rows past `rows` are zero.
__device__ __forceinline__ void fixed_to_tmem(const __nv_bfloat16* base, long long rs, long long bs, int b, int h,
                                              int row, int rows, uint32_t taddr) {
  uint32_t w[64];
  if (row < rows) {
    const uint4* src = reinterpret_cast<const uint4*>(base + b * bs + static_cast<long long>(row) * rs + h * kD);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const uint4 u = __ldg(src + i);
      w[4 * i] = u.x;
      w[4 * i + 1] = u.y;
      w[4 * i + 2] = u.z;
      w[4 * i + 3] = u.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 64; ++i) w[i] = 0u;
  }
  tmem_st_x64_nowait(taddr, w);
}

// D = A x B^T over K = 128, A and B 128-row K-major tiles in shared memory.
__device__ __forceinline__ void mma_ss_tile(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc, bool accumulate) {
  const uint64_t da = sdesc_sw128(a, 16, 1024), db = sdesc_sw128(b, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk >> 2) * kColHalf + (kk & 3) * 32;
    mma_ss(d, sdesc_advance(da, off), sdesc_advance(db, off), idesc, (accumulate || kk > 0));
  }
}

// D = A x B^T over K = 128, A in TMEM (64 columns of bf16 pairs), B a K-major tile.
__device__ __forceinline__ void mma_ts_tile(uint32_t d, uint32_t a_tmem, uint32_t b, uint32_t idesc) {
  const uint64_t db = sdesc_sw128(b, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t off = (kk >> 2) * kColHalf + (kk & 3) * 32;
    mma_ts(d, a_tmem + kk * 8, sdesc_advance(db, off), idesc, kk > 0);
  }
}

// D (+)= A x B over K = 128, A a K-major tile in shared memory, B an MN-major tile [K rows][N = 128].
__device__ __forceinline__ void mma_ss_tile_mn(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc, bool accumulate) {
  const uint64_t da = sdesc_sw128(a, 16, 1024), db = sdesc_sw128(b, kColHalf, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    const uint32_t a_off = (kk >> 2) * kColHalf + (kk & 3) * 32;
    mma_ss(d, sdesc_advance(da, a_off), sdesc_advance(db, kk * 2048), idesc,
           (accumulate || kk > 0));
  }
}

// D = A x B over K = 128, A and B MN-major tiles [K rows][M or N = 128] (A^T and B as stored).
__device__ __forceinline__ void mma_ss_tile_mnmn(uint32_t d, uint32_t a, uint32_t b, uint32_t idesc) {
  const uint64_t da = sdesc_sw128(a, kColHalf, 1024), db = sdesc_sw128(b, kColHalf, 1024);
#pragma unroll
  for (int kk = 0; kk < 8; ++kk) {
    mma_ss(d, sdesc_advance(da, kk * 2048), sdesc_advance(db, kk * 2048), idesc,
           kk > 0);
  }
}

// Writes 32 bf16 values (16 packed words) as columns [32q, 32q+32) of row `r`
// of a 128 x 128 K-major tile with 128-byte swizzle (the layout TMA produces).
__device__ __forceinline__ void st_tile_quarter_row(uint8_t* tile, int r, int q, const uint32_t (&w)[16]) {
  uint8_t* rowp = tile + (q >> 1) * kColHalf + r * 128;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const int ch = 4 * (q & 1) + c;
    *reinterpret_cast<uint4*>(rowp + ((ch ^ (r & 7)) << 4)) =
        make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
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
        // Added in L2, fire and forget: the epilogue does not wait for the old value, which in a ring
        // step's fp32 accumulator is rarely in L2. One CTA owns these rows in a launch, so the sum is
        // the plain fp32 add (subnormal sums flush to zero, as the atomic add does).
        asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + i), "f"(v.x), "f"(v.y), "f"(v.z),
                     "f"(v.w)
                     : "memory");
      } else {
        *reinterpret_cast<float4*>(dst + i) = v;
      }
    }
  }
}

// Zeroes `cols` values of a gradient row (overwrite modes only).
__device__ __forceinline__ void store_zero(void* base, long long off, int cols, int mode) {
  if (mode == LCB_GRAD_F32_ACCUM) return;
  if (mode == LCB_GRAD_BF16) {
    uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + off);
    for (int i = 0; i < cols / 8; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
  } else {
    float4* dst = reinterpret_cast<float4*>(static_cast<float*>(base) + off);
    for (int i = 0; i < cols / 4; ++i) dst[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Natural-log LSE of a query row -> base-2, with hidden/empty rows mapped to +inf (P = 0).
__device__ __forceinline__ float lse2_of(const Params& p, int b, int h, int q) {
  if (q >= p.Sq) return INFINITY;
  const float l = __ldg(p.lse + b * p.l_bs + h * p.l_hs + q);
  return (l == -INFINITY) ? INFINITY : l * kLog2e;
}

__device__ __forceinline__ uint32_t start(Bars* bars, int stages, uint32_t fixed_count, int warp) {
  if (threadIdx.x == 0) init_bars(bars, stages, fixed_count);
  if (warp == kMmaWarp) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  return bars->tmem_base;
}

__device__ __forceinline__ void teardown(uint32_t tbase, int warp) {
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

// ============================================================== dK / dV pass
// Shared memory: K, V (fixed, TMA), a 2-slot Q ring, a 2-slot dO ring, dS^T.
// TMEM: S^T [0,128) (P^T bf16: queries [32x, 32x+32) packed at columns
// [32x, 32x+16)), dP^T [128,256), dV [256,384), dK [384,512).
// MMA order per query tile i: dP^T(i+1) as soon as dP^T(i) is loaded; then,
// once P^T(i)/dS^T(i) exist: dV += P^T dO_i (frees dO_i), S^T(i+1),
// dK += dS^T Q_i (frees Q_i).
constexpr int kKvStages = 2;
constexpr uint32_t kKvSmK = 0;
constexpr uint32_t kKvSmV = kTileBytes;
constexpr uint32_t kKvSmQ = 2 * kTileBytes;
constexpr uint32_t kKvSmDo = kKvSmQ + kKvStages * kTileBytes;
constexpr uint32_t kKvSmDs = kKvSmDo + kKvStages * kTileBytes;
constexpr uint32_t kKvSmBar = kKvSmDs + kTileBytes;
constexpr uint32_t kKvSmem = kKvSmBar + sizeof(Bars) + 1024;

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                         const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                         const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kKvSmBar);
  volatile int* abort_flag = &bars->abort;
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  constexpr uint32_t kWhere = 2u << 24;

  // Work item: key tile kt of (b, h). Head-major order: the CTAs running at once
  // belong to one or two heads, so the query tiles they all stream stay in L2;
  // within a head, causal work shrinks with kt, so low kt first.
  const int nq = (p.Sq + kT - 1) / kT;
  const int nkt = (p.Sk + kT - 1) / kT;
  const int bh = static_cast<int>(blockIdx.x / nkt);
  const int kt = static_cast<int>(blockIdx.x % nkt);
  const int b = bh / p.H, h = bh % p.H;
  const int i0 = p.causal ? kt : 0;
  const int n = std::max(0, nq - i0);  // query tiles

  const uint32_t tbase = start(bars, kKvStages, 1, warp);
  const uint32_t tS = tbase, tDP = tbase + 128, tDV = tbase + 256, tDK = tbase + 384;

  if (warp == kProducerWarp) {
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      const int x0 = h * kD;
      const uint64_t pol = l2_policy_evict_last();
      mbar_arrive_expect_tx(&bars->fixed_full, 2 * kTileBytes);
      load_tile(smem + kKvSmK, &tm_k, &bars->fixed_full, x0, kt * kT, b, pol);
      load_tile(smem + kKvSmV, &tm_v, &bars->fixed_full, x0, kt * kT, b, pol);
      // dO_i then Q_i, each into its own 2-slot ring.
      int i = 0;
      bool ok = true;
      for (; i < n && ok; ++i) {
        const int s = i % kKvStages;
        const uint32_t ph = static_cast<uint32_t>(i / kKvStages) & 1u;
        const int row = (i0 + i) * kT;
        ok = mbar_wait(&bars->do_empty[s], ph ^ 1u, abort_flag, p.st, kWhere | (1u << 16));
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->do_full[s], kTileBytes);
        load_tile(smem + kKvSmDo + s * kTileBytes, &tm_do, &bars->do_full[s], x0, row, b, pol);
        ok = mbar_wait(&bars->ring_empty[s], ph ^ 1u, abort_flag, p.st, kWhere | (1u << 16));
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->ring_full[s], kTileBytes);
        load_tile(smem + kKvSmQ + s * kTileBytes, &tm_q, &bars->ring_full[s], x0, row, b, pol);
      }
      if (!ok) {
        drain_wait(&bars->fixed_full, 0, p.st.limit);
        for (int k2 = std::max(0, i - kKvStages); k2 <= i && k2 < n; ++k2) {
          const uint32_t ph2 = static_cast<uint32_t>(k2 / kKvStages) & 1u;
          drain_wait(&bars->do_full[k2 % kKvStages], ph2, p.st.limit);
          drain_wait(&bars->ring_full[k2 % kKvStages], ph2, p.st.limit);
        }
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && n > 0) {
      const uint32_t id_s = idesc_bf16(kT, kT, false, false);  // scores: both operands K-major
      const uint32_t id_g = idesc_bf16(kT, kD, false, true);   // gradients: B MN-major
      const uint32_t sK = sbase + kKvSmK, sV = sbase + kKvSmV, sDs = sbase + kKvSmDs;
      auto q_slot = [&](int i) { return sbase + kKvSmQ + (i % kKvStages) * kTileBytes; };
      auto do_slot = [&](int i) { return sbase + kKvSmDo + (i % kKvStages) * kTileBytes; };
      auto wait_q = [&](int i) {
        const bool r = mbar_wait(&bars->ring_full[i % kKvStages], static_cast<uint32_t>(i / kKvStages) & 1u,
                                 abort_flag, p.st, kWhere | (3u << 16));
        tc_fence_after();
        return r;
      };
      auto wait_do = [&](int i) {
        const bool r = mbar_wait(&bars->do_full[i % kKvStages], static_cast<uint32_t>(i / kKvStages) & 1u,
                                 abort_flag, p.st, kWhere | (12u << 16));
        tc_fence_after();
        return r;
      };
      bool ok = mbar_wait(&bars->fixed_full, 0, abort_flag, p.st, kWhere | (2u << 16));
      if (ok) ok = wait_do(0);
      if (ok) {
        mma_ss_tile(tDP, sV, do_slot(0), id_s, false);  // dP^T(0) = V dO_0^T
        tc_commit(&bars->dp_full);
      }
      if (ok) ok = wait_q(0);
      if (ok) {
        mma_ss_tile(tS, sK, q_slot(0), id_s, false);  // S^T(0) = K Q_0^T
        tc_commit(&bars->s_full);
      }
      for (int i = 0; i < n && ok; ++i) {
        const uint32_t ph = static_cast<uint32_t>(i) & 1u;
        if (i + 1 < n) {
          ok = wait_do(i + 1);
          if (ok) ok = mbar_wait(&bars->dp_free, ph, abort_flag, p.st, kWhere | (8u << 16));
          if (!ok) break;
          tc_fence_after();
          mma_ss_tile(tDP, sV, do_slot(i + 1), id_s, false);  // dP^T(i+1)
          tc_commit(&bars->dp_full);
        }
        ok = mbar_wait(&bars->pt_full, ph, abort_flag, p.st, kWhere | (4u << 16));
        if (!ok) break;
        tc_fence_after();
        const uint64_t ddo = sdesc_sw128(do_slot(i), kColHalf, 1024);
        // dV += P^T(i) dO_i; P^T K-step kk (queries 16kk..16kk+15) sits at columns 32(kk/2) + 8(kk%2)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a = tS + 32 * (kk >> 1) + 8 * (kk & 1);
          mma_ts(tDV, a, sdesc_advance(ddo, kk * 2048), id_g, (i > 0 || kk > 0));
        }
        tc_commit(&bars->do_empty[i % kKvStages]);
        if (i + 1 < n) {
          ok = wait_q(i + 1);
          if (!ok) break;
          mma_ss_tile(tS, sK, q_slot(i + 1), id_s, false);  // S^T(i+1), after dV read P^T(i)
          tc_commit(&bars->s_full);
        }
        ok = mbar_wait(&bars->p_full, ph, abort_flag, p.st, kWhere | (13u << 16));
        if (!ok) break;
        tc_fence_after();
        mma_ss_tile_mn(tDK, sDs, q_slot(i), id_g, i > 0);  // dK += dS^T(i) Q_i
        tc_commit(&bars->ds_free);
        tc_commit(&bars->ring_empty[i % kKvStages]);
      }
      if (ok) tc_commit(&bars->acc_full);
      tc_commit(&bars->mma_done);
      drain_wait(&bars->mma_done, 0, p.st.limit);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- compute
    const int x = warp >> 2;            // this warpgroup's query columns [32x, 32x + 32)
    const int row = threadIdx.x & 127;  // key row within the tile, TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint8_t* ds_tile = smem + kKvSmDs;
    const int j = kt * kT + row;
    const float c = p.scale_log2;
    // Lane l holds the statistics of query 32x + l of a tile (loaded a tile
    // ahead): -LSE * log2(e) (-inf for a hidden or empty row) and
    // -scale * Delta; every thread reads all 32 through warp shuffles. The
    // arithmetic is the one-pass kernel's, so dK and dV match it bit for bit.
    // The raw values are loaded a whole step before their use; a query row
    // past the block reads as LSE = -inf, Delta = 0.
    float rl = 0.f, rd = 0.f;  // raw LSE and Delta of the next tile
    auto fetch_stats = [&](int i) {
      const int q = (i0 + i) * kT + 32 * x + lane;
      rl = q < p.Sq ? __ldg(p.lse + b * p.l_bs + h * p.l_hs + q) : -INFINITY;
      rd = q < p.Sq ? __ldg(p.delta + b * p.l_bs + h * p.l_hs + q) : 0.f;
    };
    if (n > 0) fetch_stats(0);
    bool ok = true;
    for (int i = 0; i < n && ok; ++i) {
      const uint32_t ph = static_cast<uint32_t>(i) & 1u;
      const int it = i0 + i;            // query tile
      const int qx = it * kT + 32 * x;  // first query of this warpgroup's columns
      const float l2v = (rl == -INFINITY) ? -INFINITY : -rl * kLog2e;  // fetched a step ago
      const float dlv = -p.scale * rd;
      if (i + 1 < n) fetch_stats(i + 1);
      ok = warp_all(mbar_wait(&bars->s_full, ph, abort_flag, p.st, kWhere | (5u << 16)));
      if (ok) ok = warp_all(mbar_wait(&bars->dp_full, ph, abort_flag, p.st, kWhere | (6u << 16)));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[32], dp[32];
      tmem_ld2_x32(tS + lane_off + 32 * x, tDP + lane_off + 32 * x, s, dp);
      tc_fence_before();
      mbar_arrive(&bars->dp_free);  // dP^T(i) is in registers: its TMEM may take dP^T(i+1)
      const bool diag = p.causal && (it == kt);
      // Phase 1: P^T, into this warpgroup's own S^T columns (already read by it).
      float pv[32];
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const float m0 = __shfl_sync(0xffffffffu, l2v, e);
        const float m1 = __shfl_sync(0xffffffffu, l2v, e + 1);
        float x0, x1;
        ffma2(x0, x1, __uint_as_float(s[e]), __uint_as_float(s[e + 1]), c, c, m0, m1);
        pv[e] = ex2_approx(x0);
        pv[e + 1] = ex2_approx(x1);
      }
      if (diag) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (qx + e < j) pv[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(pv[e], pv[e + 1]);
      tmem_st_x16_nowait(tS + lane_off + 32 * x, pk);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(&bars->pt_full);  // dV(i) and S^T(i+1) may go
      // Phase 2: dS'^T = P^T (scale dP^T - scale Delta), into shared memory for dK.
      uint32_t dk[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const float d0 = __shfl_sync(0xffffffffu, dlv, e);
        const float d1 = __shfl_sync(0xffffffffu, dlv, e + 1);
        float t0, t1, u0, u1;
        ffma2(t0, t1, __uint_as_float(dp[e]), __uint_as_float(dp[e + 1]), p.scale, p.scale, d0, d1);
        fmul2(u0, u1, pv[e], pv[e + 1], t0, t1);
        dk[e >> 1] = pack_bf16x2(u0, u1);
      }
      if (i > 0) {
        ok = warp_all(mbar_wait(&bars->ds_free, ph ^ 1u, abort_flag, p.st, kWhere | (9u << 16)));
        if (!ok) break;
      }
      st_tile_quarter_row(ds_tile, row, x, dk);
      fence_proxy_async_smem();
      mbar_arrive(&bars->p_full);
    }
    // Epilogue: warpgroups 0/1 write dV columns [0,64)/[64,128), 2/3 write dK (scaled).
    const bool valid = j < p.Sk;
    const int half = x & 1;
    const long long off = b * p.g_bs + static_cast<long long>(j) * p.g_rs + h * kD + 64 * half;
    void* gdst = x < 2 ? p.g1 : p.g0;
    const float mul = 1.f;  // dK is already scaled through dS'
    const uint32_t tacc = (x < 2 ? tDV : tDK) + lane_off + 64 * half;
    if (n == 0) {
      if (valid) store_zero(gdst, off, 64, p.grad_mode);
    } else if (ok) {
      ok = warp_all(mbar_wait(&bars->acc_full, 0, abort_flag, p.st, kWhere | (10u << 16)));
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t a[32];
          tmem_ld_x32(tacc + ch * 32, a);
          if (valid) store_grad_chunk(gdst, off + ch * 32, a, mul, p.grad_mode);
        }
      }
    }
  }
  teardown(tbase, warp);
}

// ============================================================== fused pass
// One pass over the same (key tile, query tile) pairs as the dK/dV pass that
// also forms dQ: per pair, dQ_i += scale dS_i K_j is one more MMA (A = dS read
// MN-major from the dS^T tile, B = K read MN-major). Five MMAs per pair
// instead of the seven of the two passes (dQ's S and dP are not recomputed).
// The 128 x 128 fp32 partial of each pair is added into a tiled fp32 dQ
// accumulator in L2; its summation order is not fixed. Two paths share the
// work, because each alone stalls: warpgroups 0 and 1 stage their 128 x 32
// blocks (columns 0-63) in a shared-memory slot each, which the reducer warp
// adds with one bulk asynchronous reduction per block; warpgroups 2 and 3 add
// columns 64-127 straight from registers with red.global.add.v4.f32, each
// warp instruction covering 512 contiguous bytes. With all four blocks staged
// through two slots, warpgroups 2 and 3 waited about 1500 clocks per tile for
// the bulk engine to finish reading warpgroups 0 and 1's blocks; with all four
// blocks as register reductions, L2 took longer to absorb them.
//
// Accumulator layout (floats): the tile of query rows [128t, 128t + 128) of
// (b, h) is at dq + b * tile_bs + h * tile_hs + t * 16384. Columns 0-63 are
// two blocks of 4096 (block x = columns [32x, 32x + 32) at x * 4096): row r
// of block x holds its 8 four-float chunks c at chunk position c ^ (r & 7)
// (128 B per row). Columns 64-127 are chunk-major from float 8192 on: the
// four floats of chunk c (columns 64 + 4c .. 64 + 4c + 3) of row r at
// 8192 + (c * 128 + r) * 4.
//
// TMEM as in the dK/dV pass; the dQ partial of query tile i reuses the dP^T
// columns once dP^T(i) is in registers. Shared memory: K, V, a 2-slot Q ring,
// ONE dO slot (dO(i+1) loads while dS(i) is formed), dS^T, and two 16 KB
// staging slots for dQ blocks (slot x for warpgroup x = 0, 1).
// Warps 0-15 compute, 16 TMA producer, 17 MMA issuer, 18 dQ reducer.
// MMA order per query tile i: dV += P^T dO_i, S^T(i+1), dQ(i),
// dK += dS^T Q_i, then dP^T(i+1) once dQ(i) has been read out. The compute
// warps form dS^T(i), then P^T(i+1) while dQ(i) and dK(i) run, then read
// out dQ(i) and add it into the accumulator.
constexpr int kFuThreads = 608;
constexpr int kFuReduceWarp = 18;
constexpr uint32_t kDqBlock = 128 * 32 * 4;  // one staged dQ block: 128 rows x 32 columns fp32
constexpr uint32_t kFuSmK = 0;
constexpr uint32_t kFuSmV = kTileBytes;
constexpr uint32_t kFuSmQ = 2 * kTileBytes;
constexpr uint32_t kFuSmDo = kFuSmQ + kKvStages * kTileBytes;
constexpr uint32_t kFuSmDs = kFuSmDo + kTileBytes;
constexpr uint32_t kFuSmStg = kFuSmDs + kTileBytes;
constexpr uint32_t kFuSmBar = kFuSmStg + 2 * kDqBlock;
constexpr uint32_t kFuSmStats = kFuSmBar + ((sizeof(Bars) + 15) & ~15u);  // per-warpgroup row statistics, 1 KB
constexpr uint32_t kFuSmem = kFuSmStats + 1024 + 1024;

__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;" ::"l"(gdst), "r"(ssrc),
               "r"(bytes)
               : "memory");
}
// Adds four floats at gaddr (16-byte aligned) in L2, fire and forget.
__device__ __forceinline__ void red_add_v4(float* gaddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(gaddr), "f"(__uint_as_float(a)),
               "f"(__uint_as_float(b)), "f"(__uint_as_float(c)), "f"(__uint_as_float(d))
               : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__global__ void __launch_bounds__(kFuThreads, 1)
    attn_bwd_fused_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                          const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_do,
                          const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kFuSmBar);
  volatile int* abort_flag = &bars->abort;
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  constexpr uint32_t kWhere = 4u << 24;

  // Work item: the task owning this CTA (tasks come longest rows first), then
  // key tile kt of (b, h) in it, in the dK/dV pass's order (head-major, long
  // rows first). Row indices below are task-local; q_off / k_off place them
  // in the shared tensors.
  int ti = 0;
  while (ti + 1 < p.n_tasks && static_cast<int>(blockIdx.x) >= p.task[ti + 1].cta0) ++ti;
  const int Sq = p.task[ti].q_len, Sk = p.task[ti].k_len, causal = p.task[ti].causal;
  const int q_off = p.task[ti].q_off, k_off = p.task[ti].k_off;
  const int local = static_cast<int>(blockIdx.x) - p.task[ti].cta0;
  const int nq = (Sq + kT - 1) / kT;
  const int nkt = (Sk + kT - 1) / kT;
  const int bh = local / nkt;
  const int kt = local % nkt;
  const int b = bh / p.H, h = bh % p.H;
  const int i0 = causal ? kt : 0;
  const int n = std::max(0, nq - i0);  // query tiles

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(&bars->stg_full[x], 128);
      mbar_init(&bars->stg_free[x], 1);
    }
  }
  const uint32_t tbase = start(bars, kKvStages, 1, warp);  // its barrier fence covers the inits above
  const uint32_t tS = tbase, tDP = tbase + 128, tDV = tbase + 256, tDK = tbase + 384;
  const uint32_t tDQ = tDP;

  if (warp == kProducerWarp) {
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_do);
      const int x0 = h * kD;
      const uint64_t pol = l2_policy_evict_last();
      mbar_arrive_expect_tx(&bars->fixed_full, 2 * kTileBytes);
      load_tile(smem + kFuSmK, &tm_k, &bars->fixed_full, x0, k_off + kt * kT, b, pol);
      load_tile(smem + kFuSmV, &tm_v, &bars->fixed_full, x0, k_off + kt * kT, b, pol);
      int i = 0;
      bool ok = true;
      for (; i < n && ok; ++i) {
        const int s = i % kKvStages;
        const uint32_t ph = static_cast<uint32_t>(i / kKvStages) & 1u;
        const uint32_t dph = static_cast<uint32_t>(i) & 1u;  // one dO slot
        const int row = q_off + (i0 + i) * kT;
        ok = mbar_wait(&bars->ring_empty[s], ph ^ 1u, abort_flag, p.st, kWhere | (1u << 16));
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->ring_full[s], kTileBytes);
        load_tile(smem + kFuSmQ + s * kTileBytes, &tm_q, &bars->ring_full[s], x0, row, b, pol);
        ok = mbar_wait(&bars->do_empty[0], dph ^ 1u, abort_flag, p.st, kWhere | (11u << 16));
        if (!ok) break;
        mbar_arrive_expect_tx(&bars->do_full[0], kTileBytes);
        load_tile(smem + kFuSmDo, &tm_do, &bars->do_full[0], x0, row, b, pol);
      }
      if (!ok) {
        drain_wait(&bars->fixed_full, 0, p.st.limit);
        for (int k2 = std::max(0, i - kKvStages); k2 <= i && k2 < n; ++k2)
          drain_wait(&bars->ring_full[k2 % kKvStages], static_cast<uint32_t>(k2 / kKvStages) & 1u, p.st.limit);
        for (int k2 = std::max(0, i - 1); k2 <= i && k2 < n; ++k2)
          drain_wait(&bars->do_full[0], static_cast<uint32_t>(k2) & 1u, p.st.limit);
      }
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && n > 0) {
      const uint32_t id_s = idesc_bf16(kT, kT, false, false);  // scores: both operands K-major
      const uint32_t id_g = idesc_bf16(kT, kD, false, true);   // dK, dV: B MN-major
      const uint32_t id_q = idesc_bf16(kT, kD, true, true);    // dQ: A (dS) and B (K) MN-major
      const uint32_t sK = sbase + kFuSmK, sV = sbase + kFuSmV, sDs = sbase + kFuSmDs, sDo = sbase + kFuSmDo;
      auto q_slot = [&](int i) { return sbase + kFuSmQ + (i % kKvStages) * kTileBytes; };
      auto wait_q = [&](int i) {
        const bool r = mbar_wait(&bars->ring_full[i % kKvStages], static_cast<uint32_t>(i / kKvStages) & 1u,
                                 abort_flag, p.st, kWhere | (3u << 16));
        tc_fence_after();
        return r;
      };
      auto wait_do = [&](int i) {
        const bool r = mbar_wait(&bars->do_full[0], static_cast<uint32_t>(i) & 1u, abort_flag, p.st,
                                 kWhere | (12u << 16));
        tc_fence_after();
        return r;
      };
      bool ok = mbar_wait(&bars->fixed_full, 0, abort_flag, p.st, kWhere | (2u << 16));
      if (ok) ok = wait_q(0);
      if (ok) {
        mma_ss_tile(tS, sK, q_slot(0), id_s, false);  // S^T(0) = K Q_0^T
        tc_commit(&bars->s_full);
      }
      if (ok) ok = wait_do(0);
      if (ok) {
        mma_ss_tile(tDP, sV, sDo, id_s, false);  // dP^T(0) = V dO_0^T
        tc_commit(&bars->dp_full);
      }
      for (int i = 0; i < n && ok; ++i) {
        const uint32_t ph = static_cast<uint32_t>(i) & 1u;
        ok = mbar_wait(&bars->pt_full, ph, abort_flag, p.st, kWhere | (4u << 16));
        if (!ok) break;
        tc_fence_after();
        const uint64_t ddo = sdesc_sw128(sDo, kColHalf, 1024);
        // dV += P^T(i) dO_i; P^T K-step kk (queries 16kk..16kk+15) sits at columns 32(kk/2) + 8(kk%2)
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint32_t a = tS + 32 * (kk >> 1) + 8 * (kk & 1);
          mma_ts(tDV, a, sdesc_advance(ddo, kk * 2048), id_g, (i > 0 || kk > 0));
        }
        tc_commit(&bars->do_empty[0]);  // the dO slot may take dO(i+1)
        if (i + 1 < n) {
          ok = wait_q(i + 1);
          if (!ok) break;
          mma_ss_tile(tS, sK, q_slot(i + 1), id_s, false);  // S^T(i+1), after dV read P^T(i)
          tc_commit(&bars->s_full);
        }
        // dS^T(i) is in shared memory; every compute thread loaded dP^T(i) before arriving
        ok = mbar_wait(&bars->p_full, ph, abort_flag, p.st, kWhere | (13u << 16));
        if (!ok) break;
        tc_fence_after();
        mma_ss_tile_mnmn(tDQ, sDs, sK, id_q);  // dQ(i) = dS(i) K
        tc_commit(&bars->dq_full);
        mma_ss_tile_mn(tDK, sDs, q_slot(i), id_g, i > 0);  // dK += dS^T(i) Q_i
        tc_commit(&bars->ds_free);
        tc_commit(&bars->ring_empty[i % kKvStages]);
        if (i + 1 < n) {
          ok = wait_do(i + 1);
          if (ok) ok = mbar_wait(&bars->dq_free, ph, abort_flag, p.st, kWhere | (8u << 16));
          if (!ok) break;
          tc_fence_after();
          mma_ss_tile(tDP, sV, sDo, id_s, false);  // dP^T(i+1), over the read dQ(i)
          tc_commit(&bars->dp_full);
        }
      }
      if (ok) tc_commit(&bars->acc_full);
      tc_commit(&bars->mma_done);
      drain_wait(&bars->mma_done, 0, p.st.limit);
    }
    __syncwarp();
  } else if (warp == kFuReduceWarp) {
    // Adds the two staged 16 KB dQ blocks of each tile (columns 0-63) into the
    // accumulator and frees each slot once read; both reductions are issued
    // before the first read is waited for, so the two reads overlap.
    if (lane == 0 && n > 0) {
      bool ok = true;
      for (int i = 0; i < n && ok; ++i) {
        const uint32_t ph = static_cast<uint32_t>(i) & 1u;
        float* tile =
            p.dq_acc + b * p.dq_bs + h * p.dq_hs + static_cast<long long>(q_off / kT + i0 + i) * (kT * kD);
        {  // blocks 0 and 1 (columns 0-63), each in a slot of its own
          ok = mbar_wait(&bars->stg_full[0], ph, abort_flag, p.st, kWhere | (14u << 16));
          if (!ok) break;
          bulk_reduce_add_f32(tile, sbase + kFuSmStg, kDqBlock);
          bulk_commit();
          ok = mbar_wait(&bars->stg_full[1], ph, abort_flag, p.st, kWhere | (14u << 16));
          if (!ok) break;
          bulk_reduce_add_f32(tile + kDqBlock / 4, sbase + kFuSmStg + kDqBlock, kDqBlock);
          bulk_commit();
          bulk_wait_read<1>();
          mbar_arrive(&bars->stg_free[0]);
          bulk_wait_read<0>();
          mbar_arrive(&bars->stg_free[1]);
        }
      }
      bulk_wait_all();  // every reduction issued has completed
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- compute
    const int x = warp >> 2;            // this warpgroup's query columns [32x, 32x + 32)
    const int row = threadIdx.x & 127;  // key row of S^T/dP^T/dV/dK, query row of dQ: the TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint8_t* ds_tile = smem + kFuSmDs;
    uint8_t* stg_row = smem + kFuSmStg + (x & 1) * kDqBlock + row * 128;  // used by warpgroups 0 and 1
    // This warpgroup's 32 query statistics of the current tile, published by
    // every warp of the group (same values) and read back as broadcast float4s:
    // -LSE * log2(e) for phase 1, -scale * Delta for phase 2. Each array is
    // rewritten only after a barrier that every reader of its previous values
    // has passed (s_full(s) needs all of phase 1 of tile s-1 done; dp_full(i)
    // needs dq_free(i-1), which follows phase 2 of tile i-1 in every warp).
    float* l2s = reinterpret_cast<float*>(smem + kFuSmStats) + 32 * x;
    float* sds = reinterpret_cast<float*>(smem + kFuSmStats) + 128 + 32 * x;
    const int j = kt * kT + row;
    const bool key_ok = j < Sk;  // rows past the block's keys (zero-filled or another block's): P must be 0
    const float c = p.scale_log2;
    // Lane l holds the statistics of query 32x + l of a tile: -LSE * log2(e)
    // (-inf for a hidden or empty row: P = 0) and -scale * Delta. The raw
    // values are loaded a whole step before their use, so no warp waits on
    // the loads; a query row past the block reads as LSE = -inf, Delta = 0.
    float rl = 0.f, rd = 0.f;  // raw LSE and Delta of the next tile
    auto fetch_stats = [&](int i) {
      const int q = (i0 + i) * kT + 32 * x + lane;
      const long long si = b * p.l_bs + h * p.l_hs + q_off + q;
      rl = q < Sq ? __ldg(p.lse + si) : -INFINITY;
      rd = q < Sq ? __ldg(p.delta + si) : 0.f;
    };
    if (n > 0) fetch_stats(0);
    bool ok = true;
    // Step s runs phase 2 of query tile s-1, phase 1 of tile s, then phase 3
    // of tile s-1: P^T(s) is computed while the tensor pipe runs dQ(s-1) and
    // dK(s-1), so the next dV and S^T can be issued as soon as dP^T(s) is.
    // dS carries the softmax scale (dS' = scale * P (dP - Delta)), so dQ and
    // dK come out of the MMAs scaled and are stored without a multiply.
    // Pairs of values go through the packed f32x2 instructions.
    float pv[32];      // P^T of the tile between its phases 1 and 2
    float sd = 0.f;    // -scale * Delta of that tile
    const float scl = p.scale;
    for (int s = 0; s <= n && ok; ++s) {
      if (s > 0) {
        // Phase 2: dS'^T = P^T (scale dP^T - scale Delta), into shared memory for dK and dQ.
        const int i = s - 1;
        const uint32_t ph = static_cast<uint32_t>(i) & 1u;
        ok = warp_all(mbar_wait(&bars->dp_full, ph, abort_flag, p.st, kWhere | (6u << 16)));
        if (!ok) break;
        tc_fence_after();
        sds[lane] = sd;
        __syncwarp();
        uint32_t dk[16];
        {
          uint32_t dp[32];
          tmem_ld_x32(tDP + lane_off + 32 * x, dp);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 d = *reinterpret_cast<const float4*>(sds + e);
            float t0, t1, u0, u1;
            ffma2(t0, t1, __uint_as_float(dp[e]), __uint_as_float(dp[e + 1]), scl, scl, d.x, d.y);
            fmul2(u0, u1, pv[e], pv[e + 1], t0, t1);
            dk[e >> 1] = pack_bf16x2(u0, u1);
            ffma2(t0, t1, __uint_as_float(dp[e + 2]), __uint_as_float(dp[e + 3]), scl, scl, d.z, d.w);
            fmul2(u0, u1, pv[e + 2], pv[e + 3], t0, t1);
            dk[(e >> 1) + 1] = pack_bf16x2(u0, u1);
          }
        }
        if (i > 0) {
          ok = warp_all(mbar_wait(&bars->ds_free, ph ^ 1u, abort_flag, p.st, kWhere | (9u << 16)));
          if (!ok) break;
        }
        st_tile_quarter_row(ds_tile, row, x, dk);
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&bars->p_full);  // also: dP^T(i) is in registers, its columns may take dQ(i)
      }
      if (s < n) {
        // Phase 1: P^T(s), into this warpgroup's own S^T columns (already read by it).
        const int it = i0 + s;            // query tile
        const int qx = it * kT + 32 * x;  // first query of this warpgroup's columns
        const float l2v = (rl == -INFINITY) ? -INFINITY : -rl * kLog2e;  // fetched a step ago
        sd = -p.scale * rd;
        if (s + 1 < n) fetch_stats(s + 1);
        ok = warp_all(mbar_wait(&bars->s_full, static_cast<uint32_t>(s) & 1u, abort_flag, p.st, kWhere | (5u << 16)));
        if (!ok) break;
        tc_fence_after();
        l2s[lane] = l2v;
        __syncwarp();
        // Only the diagonal tile and a ragged last key tile need a per-element mask.
        const bool masked = __any_sync(0xffffffffu, (causal && it == kt) || !key_ok);
        {
          uint32_t sv[32];
          tmem_ld_x32(tS + lane_off + 32 * x, sv);
#pragma unroll
          for (int e = 0; e < 32; e += 4) {
            const float4 m = *reinterpret_cast<const float4*>(l2s + e);
            float x0, x1;
            ffma2(x0, x1, __uint_as_float(sv[e]), __uint_as_float(sv[e + 1]), c, c, m.x, m.y);
            pv[e] = ex2_approx(x0);
            pv[e + 1] = ex2_approx(x1);
            ffma2(x0, x1, __uint_as_float(sv[e + 2]), __uint_as_float(sv[e + 3]), c, c, m.z, m.w);
            pv[e + 2] = ex2_approx(x0);
            pv[e + 3] = ex2_approx(x1);
          }
          if (masked) {
            const bool diag = causal && (it == kt);
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if ((diag && qx + e < j) || !key_ok) pv[e] = 0.f;
          }
        }
        {
          uint32_t pk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) pk[e >> 1] = pack_bf16x2(pv[e], pv[e + 1]);
          tmem_st_x16_nowait(tS + lane_off + 32 * x, pk);
          tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive(&bars->pt_full);  // dV(s) and S^T(s+1) may go
      }
      if (s > 0) {
        // Phase 3: row `row` of dQ(i) (TMEM lane = query row), columns [32x, 32x + 32), staged for the reducer.
        const int i = s - 1;
        const uint32_t ph = static_cast<uint32_t>(i) & 1u;
        ok = warp_all(mbar_wait(&bars->dq_full, ph, abort_flag, p.st, kWhere | (7u << 16)));
        if (!ok) break;
        tc_fence_after();
        uint32_t g[32];
        tmem_ld_x32(tDQ + lane_off + 32 * x, g);
        tc_fence_before();
        mbar_arrive(&bars->dq_free);
        float* tile = p.dq_acc + b * p.dq_bs + h * p.dq_hs + static_cast<long long>(q_off / kT + i0 + i) * (kT * kD);
        if (x < 2) {
          // columns [32x, 32x + 32): staged in slot x (free once its block of tile i-1 was read), bulk-reduced
          if (i > 0)
            ok = warp_all(mbar_wait(&bars->stg_free[x], ph ^ 1u, abort_flag, p.st, kWhere | (15u << 16)));
          if (!ok) break;
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            *reinterpret_cast<uint4*>(stg_row + ((ch ^ (row & 7)) << 4)) =
                make_uint4(g[4 * ch], g[4 * ch + 1], g[4 * ch + 2], g[4 * ch + 3]);
          fence_proxy_async_smem();
          mbar_arrive(&bars->stg_full[x]);
        } else {
          // columns [64, 128): chunk-major half, four floats of chunk c (columns 64 + 4c..) of row r at
          // 8192 + (c * 128 + r) * 4: one warp's reduction covers 512 contiguous bytes
#pragma unroll
          for (int ch = 0; ch < 8; ++ch)
            red_add_v4(tile + 8192 + ((8 * (x - 2) + ch) * 128 + row) * 4, g[4 * ch], g[4 * ch + 1], g[4 * ch + 2],
                       g[4 * ch + 3]);
        }
      }
    }
    // Epilogue: warpgroups 0/1 write dV columns [0,64)/[64,128), 2/3 write dK (already scaled through dS').
    const bool valid = j < Sk;
    const int half = x & 1;
    const long long off = b * p.g_bs + static_cast<long long>(k_off + j) * p.g_rs + h * kD + 64 * half;
    void* gdst = x < 2 ? p.g1 : p.g0;
    const float mul = 1.f;
    const uint32_t tacc = (x < 2 ? tDV : tDK) + lane_off + 64 * half;
    if (n == 0) {
      if (valid) store_zero(gdst, off, 64, p.grad_mode);
    } else if (ok) {
      ok = warp_all(mbar_wait(&bars->acc_full, 0, abort_flag, p.st, kWhere | (10u << 16)));
      if (ok) {
        tc_fence_after();
#pragma unroll 1
        for (int ch = 0; ch < 2; ++ch) {
          uint32_t a[32];
          tmem_ld_x32(tacc + ch * 32, a);
          if (valid) store_grad_chunk(gdst, off + ch * 32, a, mul, p.grad_mode);
        }
      }
    }
  }
  teardown(tbase, warp);
}

// Tiled fp32 dQ accumulator (the fused pass's layout) -> bf16 [B, S, H, D].
// One thread per 4 consecutive values of a row.
__global__ void __launch_bounds__(256) dq_untile_kernel(const float* __restrict__ acc, long long tile_hs,
                                                        long long tile_bs, __nv_bfloat16* __restrict__ dq,
                                                        long long rs, long long bs, int B, int H, int S) {
  const long long n = static_cast<long long>(B) * S * H * (kD / 4);
  for (long long w = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; w < n;
       w += static_cast<long long>(gridDim.x) * blockDim.x) {
    const int c4 = static_cast<int>(w % (kD / 4));  // four-float chunk of the row, 0..31
    const long long rest = w / (kD / 4);
    const int h = static_cast<int>(rest % H);
    const long long bs_ = rest / H;
    const int s = static_cast<int>(bs_ % S);
    const int b = static_cast<int>(bs_ / S);
    const int r = s & (kT - 1), x = c4 >> 3, ch = c4 & 7;
    const float* tl = acc + b * tile_bs + h * tile_hs + static_cast<long long>(s / kT) * (kT * kD);
    const float4 v = __ldg(reinterpret_cast<const float4*>(
        x < 2 ? tl + x * 4096 + r * 32 + ((ch ^ (r & 7)) << 2) : tl + 8192 + ((c4 - 16) * 128 + r) * 4));
    uint2 u;
    u.x = pack_bf16x2(v.x, v.y);
    u.y = pack_bf16x2(v.z, v.w);
    *reinterpret_cast<uint2*>(dq + b * bs + static_cast<long long>(s) * rs + h * kD + c4 * 4) = u;
  }
}

// ============================================================== dQ pass
// TMEM: Q [0,64) and dO [64,128) as A operands, S [128,256), dP [256,384),
// dQ [384,512). Shared memory: a 3-slot ring of (K_j, V_j), dS.
// MMA order per key tile j: S(j), dP(j) once S(j-1)/dP(j-1) are loaded;
// then dQ += dS(j-1) K_{j-1}.
constexpr int kQStages = 3;
constexpr uint32_t kQSmRing = 0;
constexpr uint32_t kQSmDs = kQStages * 2 * kTileBytes;
constexpr uint32_t kQSmBar = kQSmDs + kTileBytes;
constexpr uint32_t kQSmem = kQSmBar + sizeof(Bars) + 1024;

__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                       const Params p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kQSmBar);
  volatile int* abort_flag = &bars->abort;
  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());
  constexpr uint32_t kWhere = 3u << 24;

  // Work item: query tile qt of (b, h). Head-major order (the key tiles every
  // running CTA streams stay in L2); within a head, causal work grows with qt,
  // so high qt first.
  const int nq = (p.Sq + kT - 1) / kT;
  const int nk = (p.Sk + kT - 1) / kT;
  const int bh = static_cast<int>(blockIdx.x / nq);
  const int qt = nq - 1 - static_cast<int>(blockIdx.x % nq);
  const int b = bh / p.H, h = bh % p.H;
  const int n = p.causal ? std::min(nk, qt + 1) : nk;  // key tiles

  const uint32_t tbase = start(bars, kQStages, 256, warp);
  const uint32_t tQ = tbase, tdO = tbase + 64, tS = tbase + 128, tDP = tbase + 256, tDQ = tbase + 384;

  if (warp < 8 && n > 0) {
    // Q (warps 0-3) and dO (warps 4-7) into TMEM, one row per thread.
    const int wg = warp >> 2;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    fixed_to_tmem(wg == 0 ? p.f0 : p.f1, p.f_rs, p.f_bs, b, h, qt * kT + (threadIdx.x & 127), p.Sq,
                  (wg == 0 ? tQ : tdO) + lane_off);
    tmem_wait_st();
    tc_fence_before();
    mbar_arrive(&bars->fixed_full);
  }

  if (warp == kProducerWarp) {
    if (lane == 0 && n > 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      stream_tiles<kQStages>(smem + kQSmRing, bars, &tm_k, &tm_v, 0, n, h, b, p, kWhere);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0 && n > 0) {
      const uint32_t id_s = idesc_bf16(kT, kT, false, false);
      const uint32_t id_g = idesc_bf16(kT, kD, false, true);
      const uint32_t sDs = sbase + kQSmDs;
      auto slot = [&](int j) { return sbase + kQSmRing + (j % kQStages) * 2 * kTileBytes; };
      bool ok = mbar_wait(&bars->fixed_full, 0, abort_flag, p.st, kWhere | (2u << 16));
      for (int j = 0; j <= n && ok; ++j) {
        if (j < n) {
          ok = mbar_wait(&bars->ring_full[j % kQStages], static_cast<uint32_t>(j / kQStages) & 1u, abort_flag, p.st,
                         kWhere | (3u << 16));
          if (ok && j > 0)
            ok = mbar_wait(&bars->s_free, static_cast<uint32_t>(j - 1) & 1u, abort_flag, p.st, kWhere | (8u << 16));
          if (!ok) break;
          tc_fence_after();
          mma_ts_tile(tS, tQ, slot(j), id_s);                // S(j)  = Q K_j^T
          mma_ts_tile(tDP, tdO, slot(j) + kTileBytes, id_s);  // dP(j) = dO V_j^T
          tc_commit(&bars->s_full);
        }
        if (j > 0) {
          ok = mbar_wait(&bars->p_full, static_cast<uint32_t>(j - 1) & 1u, abort_flag, p.st, kWhere | (4u << 16));
          if (!ok) break;
          tc_fence_after();
          mma_ss_tile_mn(tDQ, sDs, slot(j - 1), id_g, j > 1);  // dQ += dS(j-1) K_{j-1}
          tc_commit(&bars->ds_free);
          tc_commit(&bars->ring_empty[(j - 1) % kQStages]);
        }
      }
      if (ok) tc_commit(&bars->acc_full);
      tc_commit(&bars->mma_done);
      drain_wait(&bars->mma_done, 0, p.st.limit);
    }
    __syncwarp();
  } else {
    const int x = warp >> 2;  // this warpgroup's key columns [32x, 32x + 32)
    const int row = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    uint8_t* ds_tile = smem + kQSmDs;
    const int qi = qt * kT + row;
    const float c = p.scale_log2;
    const float nl2 = -lse2_of(p, b, h, qi);
    const float nsd = (qi < p.Sq) ? -p.scale * __ldg(p.delta + b * p.l_bs + h * p.l_hs + qi) : 0.f;
    const int q_first = qt * kT;
    const int lim = p.causal ? std::min(qi + 1, p.Sk) : p.Sk;  // keys < lim are visible
    bool ok = true;
    for (int j = 0; j < n && ok; ++j) {
      const uint32_t ph = static_cast<uint32_t>(j) & 1u;
      ok = warp_all(mbar_wait(&bars->s_full, ph, abort_flag, p.st, kWhere | (5u << 16)));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[32], dp[32];
      tmem_ld2_x32(tS + lane_off + 32 * x, tDP + lane_off + 32 * x, s, dp);
      tc_fence_before();
      mbar_arrive(&bars->s_free);  // S(j), dP(j) are in registers: their TMEM may take S(j+1), dP(j+1)
      const int kbase = j * kT + 32 * x;
      const bool need_mask = (p.causal && kbase + 31 > q_first) || (kbase + 32 > p.Sk);
      // dS' = P (scale dP - scale Delta): dQ comes out of the MMA scaled
      uint32_t ds[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float x0, x1, t0, t1, u0, u1;
        ffma2(x0, x1, __uint_as_float(s[e]), __uint_as_float(s[e + 1]), c, c, nl2, nl2);
        float p0 = ex2_approx(x0);
        float p1 = ex2_approx(x1);
        if (need_mask) {
          if (kbase + e >= lim) p0 = 0.f;
          if (kbase + e + 1 >= lim) p1 = 0.f;
        }
        ffma2(t0, t1, __uint_as_float(dp[e]), __uint_as_float(dp[e + 1]), p.scale, p.scale, nsd, nsd);
        fmul2(u0, u1, p0, p1, t0, t1);
        ds[e >> 1] = pack_bf16x2(u0, u1);
      }
      if (j > 0) {
        ok = warp_all(mbar_wait(&bars->ds_free, ph ^ 1u, abort_flag, p.st, kWhere | (9u << 16)));
        if (!ok) break;
      }
      st_tile_quarter_row(ds_tile, row, x, ds);
      fence_proxy_async_smem();
      mbar_arrive(&bars->p_full);
    }
    // Epilogue: warpgroup x writes dQ columns [32x, 32x + 32).
    const bool valid = qi < p.Sq;
    const long long off = b * p.g_bs + static_cast<long long>(qi) * p.g_rs + h * kD + x * 32;
    if (n == 0) {
      if (valid) store_zero(p.g0, off, 32, p.grad_mode);
    } else if (ok) {
      ok = warp_all(mbar_wait(&bars->acc_full, 0, abort_flag, p.st, kWhere | (10u << 16)));
      if (ok) {
        tc_fence_after();
        uint32_t a[32];
        tmem_ld_x32(tDQ + lane_off + x * 32, a);
        if (valid) store_grad_chunk(p.g0, off, a, 1.f, p.grad_mode);  // scaled through dS'
      }
    }
  }
  teardown(tbase, warp);
}

Params base_params(const BwdLaunch& a) {
  Params p;
  p.lse = a.lse;
  p.delta = a.delta;
  p.l_hs = a.lse_head_stride;
  p.l_bs = a.lse_batch_stride;
  p.f0 = nullptr;
  p.f1 = nullptr;
  p.f_rs = 0;
  p.f_bs = 0;
  p.dq_acc = nullptr;
  p.dq_hs = 0;
  p.dq_bs = 0;
  p.n_tasks = 0;
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
  // An empty query side is never loaded (the kernel's loop count is 0): its maps stay zeroed.
  CUtensorMap tk, tv, tq, tdo;
  memset(&tq, 0, sizeof(tq));
  memset(&tdo, 0, sizeof(tdo));
  int rc;
  if ((rc = make_tma_map_bf16(&tk, a.k, a.B, a.Sk, a.H * kD, kT)) != 0) return rc;
  if ((rc = make_tma_map_bf16(&tv, a.v, a.B, a.Sk, a.H * kD, kT)) != 0) return rc;
  if (a.Sq > 0) {
    if ((rc = make_tma_map_bf16(&tq, a.q, a.B, a.Sq, a.H * kD, kT)) != 0) return rc;
    if ((rc = make_tma_map_bf16(&tdo, a.dO, a.B, a.Sq, a.H * kD, kT)) != 0) return rc;
  }
  static DeviceOnce smem_set;
  if ((rc = set_smem_limit_once(smem_set, reinterpret_cast<const void*>(attn_bwd_dkdv_kernel), kKvSmem)) != 0) return rc;
  Params p = base_params(a);
  p.g0 = a.dk;
  p.g1 = a.dv;
  p.g_rs = a.dkv_row_stride;
  p.g_bs = a.dkv_batch_stride;
  const long long grid = static_cast<long long>((a.Sk + kT - 1) / kT) * a.B * a.H;
  if (grid > 0x7fffffffLL) return -1;
  attn_bwd_dkdv_kernel<<<static_cast<unsigned>(grid), kThreads, kKvSmem, stream>>>(tk, tv, tq, tdo, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_attn_bwd_fused(const BwdLaunch& a, const BwdTask* tasks, int n_tasks, int q_rows, int k_rows,
                          cudaStream_t stream) {
  if (n_tasks < 1 || n_tasks > kMaxBwdTasks) return -1;
  if (k_rows == 0 || q_rows == 0) return 0;
  CUtensorMap tk, tv, tq, tdo;
  int rc;
  if ((rc = make_tma_map_bf16(&tk, a.k, a.B, k_rows, a.H * kD, kT)) != 0) return rc;
  if ((rc = make_tma_map_bf16(&tv, a.v, a.B, k_rows, a.H * kD, kT)) != 0) return rc;
  if ((rc = make_tma_map_bf16(&tq, a.q, a.B, q_rows, a.H * kD, kT)) != 0) return rc;
  if ((rc = make_tma_map_bf16(&tdo, a.dO, a.B, q_rows, a.H * kD, kT)) != 0) return rc;
  static DeviceOnce smem_set;
  if ((rc = set_smem_limit_once(smem_set, reinterpret_cast<const void*>(attn_bwd_fused_kernel), kFuSmem)) != 0) return rc;
  Params p = base_params(a);
  p.g0 = a.dk;
  p.g1 = a.dv;
  p.g_rs = a.dkv_row_stride;
  p.g_bs = a.dkv_batch_stride;
  p.dq_acc = static_cast<float*>(a.dq);
  p.dq_hs = a.dq_row_stride;    // tile head stride
  p.dq_bs = a.dq_batch_stride;  // tile batch stride
  long long grid = 0;
  p.n_tasks = 0;
  for (int i = 0; i < n_tasks; ++i) {
    const BwdTask& t = tasks[i];
    if (t.q_len == 0 || t.k_len == 0) continue;  // handled by the caller
    p.task[p.n_tasks++] = {t.q_off, t.q_len, t.k_off, t.k_len, t.causal, static_cast<int>(grid)};
    grid += static_cast<long long>((t.k_len + kT - 1) / kT) * a.B * a.H;
    if (grid > 0x7fffffffLL) return -1;
  }
  if (grid == 0) return 0;
  attn_bwd_fused_kernel<<<static_cast<unsigned>(grid), kFuThreads, kFuSmem, stream>>>(tk, tv, tq, tdo, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

// The same conversion for 16-byte aligned rows: one thread per 8 consecutive
// values of a row (two four-float chunks, one 16-byte store); a CTA of 256
// threads covers 16 rows of one tile; CTA index ((b * H + h) * ntiles + t) * 8
// + group. Index arithmetic in 32 bits except the final offsets.
__global__ void __launch_bounds__(256) dq_untile16_kernel(const float* __restrict__ acc, long long tile_hs,
                                                          long long tile_bs, __nv_bfloat16* __restrict__ dq,
                                                          long long rs, long long bs, int H, int S, int ntiles) {
  const int tile_lin = static_cast<int>(blockIdx.x >> 3);
  const int t = tile_lin % ntiles;
  const int bh = tile_lin / ntiles;
  const int h = bh % H, b = bh / H;
  const int r = static_cast<int>(blockIdx.x & 7) * 16 + static_cast<int>(threadIdx.x >> 4);  // row in the tile
  const int s = t * kT + r;
  if (s >= S) return;
  const int k16 = threadIdx.x & 15;  // columns [8 k16, 8 k16 + 8): block k16 / 4, chunks 2 (k16 % 4) and + 1
  const int c0 = (k16 & 3) * 2;
  const float* tl = acc + b * tile_bs + h * tile_hs + static_cast<long long>(t) * (kT * kD);
  float4 v0, v1;
  if (k16 < 8) {
    const float* row = tl + (k16 >> 2) * 4096 + r * 32;
    v0 = __ldg(reinterpret_cast<const float4*>(row + ((c0 ^ (r & 7)) << 2)));
    v1 = __ldg(reinterpret_cast<const float4*>(row + (((c0 + 1) ^ (r & 7)) << 2)));
  } else {
    v0 = __ldg(reinterpret_cast<const float4*>(tl + 8192 + ((2 * k16 - 16) * 128 + r) * 4));
    v1 = __ldg(reinterpret_cast<const float4*>(tl + 8192 + ((2 * k16 - 15) * 128 + r) * 4));
  }
  uint4 u;
  u.x = pack_bf16x2(v0.x, v0.y);
  u.y = pack_bf16x2(v0.z, v0.w);
  u.z = pack_bf16x2(v1.x, v1.y);
  u.w = pack_bf16x2(v1.z, v1.w);
  *reinterpret_cast<uint4*>(dq + b * bs + static_cast<long long>(s) * rs + h * kD + k16 * 8) = u;
}

int launch_dq_untile(const float* acc, long long tile_hs, long long tile_bs, void* dq, long long rs, long long bs,
                     int B, int H, int S, cudaStream_t stream) {
  const long long n = static_cast<long long>(B) * S * H * (kD / 4);
  if (n == 0) return 0;
  const long long ntiles = (S + kT - 1) / kT;
  const long long grid16 = static_cast<long long>(B) * H * ntiles * 8;
  if ((reinterpret_cast<uintptr_t>(dq) & 15u) == 0 && rs % 8 == 0 && bs % 8 == 0 && grid16 < (1LL << 31)) {
    dq_untile16_kernel<<<static_cast<unsigned>(grid16), 256, 0, stream>>>(
        acc, tile_hs, tile_bs, static_cast<__nv_bfloat16*>(dq), rs, bs, H, S, static_cast<int>(ntiles));
  } else {
    const long long blocks = std::min<long long>((n + 255) / 256, 152LL * 16);
    dq_untile_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
        acc, tile_hs, tile_bs, static_cast<__nv_bfloat16*>(dq), rs, bs, B, H, S);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_attn_bwd_dq(const BwdLaunch& a, cudaStream_t stream) {
  if (a.Sq == 0) return 0;
  CUtensorMap tk, tv;
  memset(&tk, 0, sizeof(tk));
  memset(&tv, 0, sizeof(tv));
  int rc;
  if (a.Sk > 0) {
    if ((rc = make_tma_map_bf16(&tk, a.k, a.B, a.Sk, a.H * kD, kT)) != 0) return rc;
    if ((rc = make_tma_map_bf16(&tv, a.v, a.B, a.Sk, a.H * kD, kT)) != 0) return rc;
  }
  static DeviceOnce smem_set;
  if ((rc = set_smem_limit_once(smem_set, reinterpret_cast<const void*>(attn_bwd_dq_kernel), kQSmem)) != 0) return rc;
  Params p = base_params(a);
  p.f0 = static_cast<const __nv_bfloat16*>(a.q.ptr);
  p.f1 = static_cast<const __nv_bfloat16*>(a.dO.ptr);
  p.f_rs = a.q.row_stride;
  p.f_bs = a.q.batch_stride;
  p.g0 = a.dq;
  p.g1 = nullptr;
  p.g_rs = a.dq_row_stride;
  p.g_bs = a.dq_batch_stride;
  const long long grid = static_cast<long long>((a.Sq + kT - 1) / kT) * a.B * a.H;
  if (grid > 0x7fffffffLL) return -1;
  attn_bwd_dq_kernel<<<static_cast<unsigned>(grid), kThreads, kQSmem, stream>>>(tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace lcb
