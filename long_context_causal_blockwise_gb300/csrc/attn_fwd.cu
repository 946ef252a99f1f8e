// Forward kernel: exact softmax attention computed blockwise with an online
// softmax ("EasyContext核心技术解析：序列并行与Flash Attention的完美结合",
// §2 "Flash Attention优化": tiles of Q, K, V, no stored score matrix).
//
// One CTA owns 256 query rows of one (batch, head) in one task: two 128-row Q
// tiles that ping-pong, so the tensor core works on one tile while the softmax
// warps work on the other. A launch may carry several tasks (blocks of query
// rows against blocks of key rows of the same tensors, as the steps of a ring
// have), laid side by side in one grid; a CTA finds its task by its index.
//
//   warp 8      TMA producer: Q tiles once, then K_j, V_j into a 4-slot ring
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM,
//               O_t += P_t V_j with P_t read from TMEM; owns the TMEM allocation
//   warps 0-3   softmax for Q tile 0 (thread = query row = TMEM lane)
//   warps 4-7   softmax for Q tile 1
//
// TMEM (512 columns x 128 lanes, fp32): S_0 [0,128), S_1 [128,256),
// O_0 [256,384), O_1 [384,512). P_t (bf16 pairs) overwrites the first 64
// columns of S_t; the MMA pipe executes one thread's tcgen05.mma in issue
// order, so the next S_t = Q_t K^T is issued after the PV that reads P_t.
//
// Online softmax in base 2: m is the running reference maximum of
// scale*log2(e)*s, l the running sum of 2^(x - m). m is only raised (and O, l
// rescaled by 2^(m_old - m_new)) when the new row maximum exceeds m by more
// than 8, so P stays <= 256 and most tiles skip the rescale; O / l is exact for
// any reference maximum.
#include <cuda_bf16.h>

#include <algorithm>

#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kBM = 128;           // query rows per tile (MMA M)
constexpr int kBN = 128;           // keys per tile
constexpr int kD = 128;            // head dim
constexpr int kStages = 4;         // K/V ring slots
constexpr int kThreads = 320;      // 10 warps
constexpr uint32_t kTileBytes = kBN * kD * 2;   // 32 KB, two 16 KB halves of 64 columns
constexpr uint32_t kHalfBytes = kTileBytes / 2;
constexpr uint32_t kSmQ = 0;                    // Q_0, Q_1
constexpr uint32_t kSmKV = 2 * kTileBytes;      // ring
constexpr uint32_t kSmBar = kSmKV + kStages * kTileBytes;
constexpr float kRescaleThreshold = 8.0f;       // log2 units
constexpr int kHeadGroup = 4;                   // (b, h) pairs whose query blocks interleave in the CTA order

struct Bars {
  uint64_t q_full;
  uint64_t kv_full[kStages];
  uint64_t kv_empty[kStages];
  uint64_t s_full[2];
  uint64_t p_full[2];
  uint64_t o_full[2];
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort;
};
constexpr uint32_t kSmemBytes = kSmBar + sizeof(Bars) + 1024;  // + alignment slack

// One block of the launch: query rows [q_off, q_off + q_len) against key rows
// [k_off, k_off + k_len) of the shared tensors; its CTAs start at cta0.
struct Task {
  int q_off, q_len, k_off, k_len, causal, o_mode;  // o_mode: 0 bf16 out, 1 fp32 out, 2 merge into fp32 (O, LSE)
  int cta0;
};

struct Params {
  void* o;
  float* lse;
  long long o_rs, o_bs, l_hs, l_bs;
  int B, H, n_tasks;
  float scale_log2;
  DevStatus st;
  Task task[kMaxFwdTasks];
};

// Barrier ids for timeout reports (bits 16-23 of the where word), kernel id 1.
constexpr uint32_t kWhere = 1u << 24;

__device__ __forceinline__ void tile_counts(int Sq, int Sk, int causal, int q0, int& n0, int& n1) {
  const int nk = (Sk + kBN - 1) / kBN;
  int n[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int r0 = q0 + t * kBM;
    if (r0 >= Sq) {
      n[t] = 0;
    } else if (causal) {
      n[t] = min(nk, r0 / kBN + 1);
    } else {
      n[t] = nk;
    }
  }
  n0 = n[0];
  n1 = n[1];
}

__device__ __forceinline__ bool warp_all(bool ok) { return __all_sync(0xffffffffu, ok); }


__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const Params p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  Bars* bars = reinterpret_cast<Bars*>(smem + kSmBar);
  volatile int* abort_flag = &bars->abort;

  const int warp = static_cast<int>(warp_id());
  const int lane = static_cast<int>(lane_id());

  // Work item: the task owning this CTA, then query block qblk of (b, h) in it.
  // Tasks come heaviest first. Within a task, (b, h) pairs go in groups of
  // kHeadGroup: a group's CTAs come heaviest (latest) query block first with
  // its heads interleaved. The running CTAs then stream the K/V tiles of a few
  // heads only (they stay in L2), and the light blocks of every group finish
  // the grid rather than one head's light blocks after the others' heavy ones.
  // Row indices below are task-local; q_off / k_off place them in the shared
  // tensors.
  int ti = 0;
  while (ti + 1 < p.n_tasks && static_cast<int>(blockIdx.x) >= p.task[ti + 1].cta0) ++ti;
  const int Sq = p.task[ti].q_len, Sk = p.task[ti].k_len, causal = p.task[ti].causal;
  const int q_off = p.task[ti].q_off, k_off = p.task[ti].k_off, o_mode = p.task[ti].o_mode;
  const int local = static_cast<int>(blockIdx.x) - p.task[ti].cta0;
  const int nq = (Sq + 2 * kBM - 1) / (2 * kBM);
  const int group = local / (nq * kHeadGroup);
  const int g0 = group * kHeadGroup;                     // first (b, h) of the group
  const int gsz = min(kHeadGroup, p.B * p.H - g0);       // the last group may be smaller
  const int within = local - group * nq * kHeadGroup;    // [0, nq * gsz)
  const int bh = g0 + within % gsz;
  const int qblk = nq - 1 - within / gsz;
  const int b = bh / p.H;
  const int h = bh % p.H;
  const int q0 = qblk * 2 * kBM;
  int n_t0, n_t1;
  tile_counts(Sq, Sk, causal, q0, n_t0, n_t1);
  const int n_max = max(n_t0, n_t1);

  if (threadIdx.x == 0) {
    mbar_init(&bars->q_full, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&bars->kv_full[s], 1);
      mbar_init(&bars->kv_empty[s], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&bars->s_full[t], 1);
      mbar_init(&bars->p_full[t], 128);
      mbar_init(&bars->o_full[t], 1);
    }
    mbar_init(&bars->mma_done, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  if (warp == 9) {
    tmem_alloc(&bars->tmem_base, 512);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = bars->tmem_base;

  if (warp == 8) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      const int x0 = h * kD;
      const uint32_t q_bytes = (n_t1 > 0 ? 2u : 1u) * kTileBytes;
      mbar_arrive_expect_tx(&bars->q_full, q_bytes);
      for (int t = 0; t < 2; ++t) {
        if ((t ? n_t1 : n_t0) == 0) continue;
        for (int half = 0; half < 2; ++half)
          tma_load_3d(smem + kSmQ + t * kTileBytes + half * kHalfBytes, &tm_q, &bars->q_full, x0 + half * 64,
                      q_off + q0 + t * kBM, b);
      }
      int it = 0;
      bool ok = true;
      for (int j = 0; j < n_max && ok; ++j) {
        for (int kv = 0; kv < 2; ++kv, ++it) {
          const int slot = it % kStages;
          const uint32_t ph = static_cast<uint32_t>(it / kStages) & 1u;
          if (!mbar_wait(&bars->kv_empty[slot], ph ^ 1u, abort_flag, p.st, kWhere | (1u << 16))) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(&bars->kv_full[slot], kTileBytes);
          const CUtensorMap* map = kv == 0 ? &tm_k : &tm_v;
          for (int half = 0; half < 2; ++half)
            tma_load_3d_hint(smem + kSmKV + slot * kTileBytes + half * kHalfBytes, map, &bars->kv_full[slot],
                             x0 + half * 64, k_off + j * kBN, b, pol);
        }
      }
      if (!ok) {
        // Let every copy already issued land before the CTA can exit.
        drain_wait(&bars->q_full, 0, p.st.limit);
        for (int k = max(0, it - kStages); k < it; ++k)
          drain_wait(&bars->kv_full[k % kStages], static_cast<uint32_t>(k / kStages) & 1u, p.st.limit);
      }
    }
    __syncwarp();
  } else if (warp == 9) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc_qk = idesc_bf16(kBM, kBN, false, false);
      const uint32_t idesc_pv = idesc_bf16(kBM, kD, false, true);
      auto issue_qk = [&](int t, int slot) {
        const uint64_t qa = sdesc_sw128(sbase + kSmQ + t * kTileBytes, 16, 1024);
        const uint64_t kb = sdesc_sw128(sbase + kSmKV + slot * kTileBytes, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kD / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
          mma_ss(tbase + t * 128, sdesc_advance(qa, off), sdesc_advance(kb, off), idesc_qk, kk > 0);
        }
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        const uint64_t vb = sdesc_sw128(sbase + kSmKV + slot * kTileBytes, kHalfBytes, 1024);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          mma_ts(tbase + 256 + t * 128, tbase + t * 128 + kk * 8, sdesc_advance(vb, kk * 2048), idesc_pv,
                 (acc || kk > 0));
        }
      };
      bool ok = mbar_wait(&bars->q_full, 0, abort_flag, p.st, kWhere | (2u << 16));
      if (ok) ok = mbar_wait(&bars->kv_full[0], 0, abort_flag, p.st, kWhere | (3u << 16));
      if (ok) {
        tc_fence_after();
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if ((t ? n_t1 : n_t0) > 0) {
            issue_qk(t, 0);
            tc_commit(&bars->s_full[t]);
          }
        }
        tc_commit(&bars->kv_empty[0]);
      }
      for (int j = 0; j < n_max && ok; ++j) {
        const int itV = 2 * j + 1, itK = 2 * j + 2;
        const int sV = itV % kStages, sK = itK % kStages;
        ok = mbar_wait(&bars->kv_full[sV], static_cast<uint32_t>(itV / kStages) & 1u, abort_flag, p.st,
                       kWhere | (3u << 16));
        if (!ok) break;
        tc_fence_after();
        bool k_ready = false;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          const int nt = t ? n_t1 : n_t0;
          if (!ok || j >= nt) continue;
          ok = mbar_wait(&bars->p_full[t], static_cast<uint32_t>(j) & 1u, abort_flag, p.st, kWhere | (4u << 16));
          if (!ok) continue;
          tc_fence_after();
          issue_pv(t, sV, j > 0);
          if (j + 1 < nt) {
            if (!k_ready) {
              ok = mbar_wait(&bars->kv_full[sK], static_cast<uint32_t>(itK / kStages) & 1u, abort_flag, p.st,
                             kWhere | (3u << 16));
              if (!ok) continue;
              tc_fence_after();
              k_ready = true;
            }
            issue_qk(t, sK);
            tc_commit(&bars->s_full[t]);
          } else {
            tc_commit(&bars->o_full[t]);
          }
        }
        if (!ok) break;
        tc_commit(&bars->kv_empty[sV]);
        if (j + 1 < n_max) tc_commit(&bars->kv_empty[sK]);
      }
      // Every MMA issued must finish before TMEM is released.
      tc_commit(&bars->mma_done);
      drain_wait(&bars->mma_done, 0, p.st.limit);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax
    const int t = warp >> 2;
    const int row = threadIdx.x & 127;
    const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const uint32_t tS = tbase + t * 128 + lane_off;
    const uint32_t tO = tbase + 256 + t * 128 + lane_off;
    const int qi = q0 + t * kBM + row;
    const int my_n = t ? n_t1 : n_t0;
    const float c = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < my_n; ++j) {
      ok = warp_all(mbar_wait(&bars->s_full[t], static_cast<uint32_t>(j) & 1u, abort_flag, p.st,
                              kWhere | (5u << 16)));
      if (!ok) break;
      tc_fence_after();
      uint32_t s[128];
      tmem_ld_x128(tS, s);
      const int kbase = j * kBN;
      const bool need_mask = (causal && kbase + kBN - 1 > q0 + t * kBM) || (kbase + kBN > Sk);
      if (need_mask) {
        const int lim = causal ? min(qi + 1, Sk) : Sk;  // keys < lim are visible (task-local)
#pragma unroll
        for (int cc = 0; cc < 128; ++cc)
          if (kbase + cc >= lim) s[cc] = __float_as_uint(-INFINITY);
      }
      // Row maximum: four chains of three-input maxima (64 instructions for 128 values).
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int cc = 0; cc < 128; cc += 8)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          m4[k] = fmax3(m4[k], __uint_as_float(s[cc + 2 * k]), __uint_as_float(s[cc + 2 * k + 1]));
      const float mx = fmax3(m4[0], m4[1], fmaxf(m4[2], m4[3]));
      const float m_new = fmaxf(m, mx * c);
      if (j == 0) {
        m = m_new;
      } else {
        const bool resc = m_new > m + kRescaleThreshold;
        if (__any_sync(0xffffffffu, resc)) {
          const float alpha = resc ? ex2_approx(m - m_new) : 1.0f;
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            uint32_t o[32];
            tmem_ld_x32(tO + ch * 32, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
            tmem_st_x32(tO + ch * 32, o);
          }
          if (resc) {
            l *= alpha;
            m = m_new;
          }
        }
      }
      const float neg_m = (m == -INFINITY) ? 0.f : -m;
      // p = 2^(c s - m) for pairs of values (packed f32x2 FMA and sums). P goes
      // back to TMEM in two 32-column halves, each stored as soon as it is
      // formed (one 64-column store at the end measured 3% slower).
      float sa0 = 0.f, sa1 = 0.f, sb0 = 0.f, sb1 = 0.f;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int e = 64 * hf + 2 * i;
          float x0, x1;
          ffma2(x0, x1, __uint_as_float(s[e]), __uint_as_float(s[e + 1]), c, c, neg_m, neg_m);
          const float p0 = ex2_approx(x0);
          const float p1 = ex2_approx(x1);
          if (i & 1)
            fadd2(sb0, sb1, sb0, sb1, p0, p1);
          else
            fadd2(sa0, sa1, sa0, sa1, p0, p1);
          pk[i] = pack_bf16x2(p0, p1);
        }
        tmem_st_x32(tS + 32 * hf, pk);
      }
      l += (sa0 + sb0) + (sa1 + sb1);
      tc_fence_before();
      mbar_arrive(&bars->p_full[t]);
    }
    if (ok && my_n > 0) {
      ok = warp_all(mbar_wait(&bars->o_full[t], 0, abort_flag, p.st, kWhere | (6u << 16)));
    }
    if (ok && my_n > 0) {
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      const bool valid = qi < Sq;
      const long long orow = static_cast<long long>(q_off + qi);  // row in the shared output tensors
      const long long lidx = b * p.l_bs + h * p.l_hs + orow;
      const float lse_blk = l > 0.f ? (m + __log2f(l)) * 0.69314718055994531f : -INFINITY;
      // Merge mode (a fused ring step): O_acc <- (w_acc O_acc + w_blk O_blk) / (w_acc + w_blk)
      // with w_x = exp(LSE_x - max); here O_blk = O_tmem / l, so its weight absorbs 1/l.
      float c_acc = 0.f, c_blk = inv_l, lse_out = lse_blk;
      if (o_mode == 2 && valid) {
        const float la = p.lse[lidx];
        const float mx = fmaxf(la, lse_blk);
        if (mx == -INFINITY) {
          c_blk = 0.f;
          lse_out = -INFINITY;
        } else {
          const float wa = __expf(la - mx), wb = __expf(lse_blk - mx);
          const float inv = 1.f / (wa + wb);
          c_acc = wa * inv;
          c_blk = wb * inv * inv_l;
          lse_out = mx + __logf(wa + wb);
        }
      }
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t o[32];
        tmem_ld_x32(tO + ch * 32, o);
        if (valid) {
          if (o_mode == 2) {
            float* dst = static_cast<float*>(p.o) + b * p.o_bs + orow * p.o_rs + h * kD + ch * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              // an accumulator row with no keys yet (weight 0) is not read: its O may be unset
              const float4 a = c_acc != 0.f ? *reinterpret_cast<const float4*>(dst + i) : make_float4(0.f, 0.f, 0.f, 0.f);
              float4 v = make_float4(c_acc * a.x + c_blk * __uint_as_float(o[i]),
                                     c_acc * a.y + c_blk * __uint_as_float(o[i + 1]),
                                     c_acc * a.z + c_blk * __uint_as_float(o[i + 2]),
                                     c_acc * a.w + c_blk * __uint_as_float(o[i + 3]));
              *reinterpret_cast<float4*>(dst + i) = v;
            }
          } else if (o_mode == 1) {
            float* dst = static_cast<float*>(p.o) + b * p.o_bs + orow * p.o_rs + h * kD + ch * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 4) {
              float4 v = make_float4(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l,
                                     __uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
              *reinterpret_cast<float4*>(dst + i) = v;
            }
          } else {
            __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(p.o) + b * p.o_bs + orow * p.o_rs + h * kD + ch * 32;
#pragma unroll
            for (int i = 0; i < 32; i += 8) {
              uint4 v;
              v.x = pack_bf16x2(__uint_as_float(o[i]) * inv_l, __uint_as_float(o[i + 1]) * inv_l);
              v.y = pack_bf16x2(__uint_as_float(o[i + 2]) * inv_l, __uint_as_float(o[i + 3]) * inv_l);
              v.z = pack_bf16x2(__uint_as_float(o[i + 4]) * inv_l, __uint_as_float(o[i + 5]) * inv_l);
              v.w = pack_bf16x2(__uint_as_float(o[i + 6]) * inv_l, __uint_as_float(o[i + 7]) * inv_l);
              *reinterpret_cast<uint4*>(dst + i) = v;
            }
          }
        }
      }
      if (valid) p.lse[lidx] = lse_out;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tbase, 512);
  }
}

__global__ void fill_empty_kernel(void* o, int o_f32, long long o_rs, long long o_bs, float* lse, long long l_hs,
                                  long long l_bs, int B, int H, int rows) {
  const long long n = static_cast<long long>(B) * rows * H;
  for (long long w = blockIdx.x * (blockDim.x / 32) + threadIdx.x / 32; w < n;
       w += static_cast<long long>(gridDim.x) * (blockDim.x / 32)) {
    const int h = static_cast<int>(w % H);
    const int r = static_cast<int>((w / H) % rows);
    const int b = static_cast<int>(w / (static_cast<long long>(H) * rows));
    const long long off = b * o_bs + static_cast<long long>(r) * o_rs + h * kD;
    const int ln = threadIdx.x & 31;
    if (o_f32) {
      reinterpret_cast<float4*>(static_cast<float*>(o) + off)[ln] = make_float4(0.f, 0.f, 0.f, 0.f);
    } else {
      reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(o) + off)[ln] = make_uint2(0u, 0u);
    }
    if (ln == 0) lse[b * l_bs + h * l_hs + r] = -INFINITY;
  }
}

}  // namespace

int launch_attn_fwd(const FwdLaunch& a, cudaStream_t stream) {
  if (a.n_tasks < 1 || a.n_tasks > kMaxFwdTasks) return -1;
  CUtensorMap tq, tk, tv;
  int rc;
  if ((rc = make_tma_map_bf16(&tq, a.q, a.B, a.q_rows, a.H * kD, kBM)) != 0) return rc;
  if ((rc = make_tma_map_bf16(&tk, a.k, a.B, a.k_rows, a.H * kD, kBN)) != 0) return rc;
  if ((rc = make_tma_map_bf16(&tv, a.v, a.B, a.k_rows, a.H * kD, kBN)) != 0) return rc;
  static DeviceOnce smem_set;
  if ((rc = set_smem_limit_once(smem_set, reinterpret_cast<const void*>(attn_fwd_kernel), kSmemBytes)) != 0)
    return rc;
  Params p;
  p.o = a.o;
  p.lse = a.lse;
  p.o_rs = a.o_row_stride;
  p.o_bs = a.o_batch_stride;
  p.l_hs = a.lse_head_stride;
  p.l_bs = a.lse_batch_stride;
  p.B = a.B;
  p.H = a.H;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.st = a.st;
  long long grid = 0;
  p.n_tasks = a.n_tasks;
  for (int i = 0; i < a.n_tasks; ++i) {
    const FwdTask& t = a.tasks[i];
    p.task[i] = {t.q_off, t.q_len, t.k_off, t.k_len, t.causal, t.o_mode, static_cast<int>(grid)};
    grid += static_cast<long long>((t.q_len + 2 * kBM - 1) / (2 * kBM)) * a.B * a.H;
    if (grid > 0x7fffffffLL) return -1;
  }
  if (grid == 0) return 0;
  attn_fwd_kernel<<<static_cast<unsigned>(grid), kThreads, kSmemBytes, stream>>>(tq, tk, tv, p);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_fill_empty(void* o, int o_f32, long long o_row_stride, long long o_batch_stride, float* lse,
                      long long lse_head_stride, long long lse_batch_stride, int B, int H, int rows,
                      cudaStream_t stream) {
  const long long warps = static_cast<long long>(B) * rows * H;
  const int blocks = static_cast<int>(std::min<long long>((warps + 7) / 8, 152LL * 16));
  if (blocks <= 0) return 0;
  fill_empty_kernel<<<blocks, 256, 0, stream>>>(o, o_f32, o_row_stride, o_batch_stride, lse, lse_head_stride,
                                                lse_batch_stride, B, H, rows);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace lcb
