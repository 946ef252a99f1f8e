// Cross-entropy loss head with an in-place backward: the loss kernel the
// long-context training script takes from Flash Attention
// ("EasyContext内存优化秘籍DeepSpeed Zero3卸载策略详解", §进阶优化与其他技术结合:
// CrossEntropyLoss(inplace_backward=True)).
//
// Per token row i of V logits x, label y_i, upstream gradient g_i:
//   LSE_i = ln sum_j exp(x_ij),  loss_i = LSE_i - x_{i,y_i},
//   dx_ij = g_i (exp(x_ij - LSE_i) - [j == y_i])   (written over x),
// ignore_index rows: loss 0, gradient 0.
//
// One row at a time per CTA, staged whole in shared memory: one bulk async
// copy brings the row in (an mbarrier with a bounded wait), the CTA reduces
// max and sum of exp2 from shared memory (one read), turns the row into its
// gradient in place in shared memory (bf16) and one bulk async copy writes
// it back over the logits. HBM sees each logit read once and, with the
// backward, written once. Rows whose address or length is not a multiple of
// 16 bytes are staged with plain loads and stores instead.
// CTAs are persistent (three per SM, 64 KB rows at V = 32000), so one CTA's
// copies overlap another's arithmetic.
#include <cuda_bf16.h>

#include <algorithm>

#include "lcb_attn.h"
#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kCeThreads = 512;
constexpr int kCeWarps = kCeThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

struct CeBars {
  uint64_t full;
  int abort;
  float red_m[kCeWarps];
  float red_s[kCeWarps];
  float m, s, x_lab;
};

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(dst)),
               "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void bulk_s2g(void* dst, const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
               "r"(bytes)
               : "memory");
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// (m, s) with m a running maximum of logits and s = sum exp(x - m); merging
// two such pairs. Differences of bf16 logits are exact in fp32, so exp(x - m)
// keeps full relative accuracy even for logits of large magnitude.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = s * ex2_approx((m - M) * kLog2e) + s2 * ex2_approx((m2 - M) * kLog2e);
  m = M;
}

__global__ void __launch_bounds__(kCeThreads) ce_kernel(__nv_bfloat16* logits, const long long* labels, float* loss,
                                                        float* lse_io, const float* dloss, int N, int V,
                                                        long long rs, int ignore_index, int mode, int bulk,
                                                        DevStatus st) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((128u - (smem_u32(smem_raw) & 127u)) & 127u);
  CeBars* bars = reinterpret_cast<CeBars*>(smem);
  __nv_bfloat16* row_s = reinterpret_cast<__nv_bfloat16*>(smem + 128 * ((sizeof(CeBars) + 127) / 128));
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const uint32_t row_bytes = static_cast<uint32_t>(V) * 2u;
  const int units = V / 8;  // 16-byte units; the tail (V % 8 values) is handled one by one
  constexpr uint32_t kWhere = 5u << 24;
  if (t == 0) {
    mbar_init(&bars->full, 1);
    bars->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  uint32_t phase = 0;
  bool ok = true;
  for (long long r = blockIdx.x; r < N && ok; r += gridDim.x, phase ^= 1u) {
    __nv_bfloat16* gx = logits + r * rs;
    // ---- stage the row
    if (bulk) {
      if (t == 0) {
        bulk_wait_read_all();  // the previous row's store has left shared memory
        mbar_arrive_expect_tx(&bars->full, row_bytes);
        bulk_g2s(row_s, gx, row_bytes, &bars->full);
      }
      ok = mbar_wait(&bars->full, phase, &bars->abort, st, kWhere | (1u << 16));
      ok = __syncthreads_and(ok);
      if (!ok) break;
    } else {
      for (int j = t; j < V; j += kCeThreads) row_s[j] = gx[j];
      __syncthreads();
    }
    const long long lab = labels[r];
    const bool keep = lab != ignore_index;
    const bool lab_ok = lab >= 0 && lab < V;
    // ---- row maximum and sum of exp(x - max), or the given LSE
    // p_j = exp(x_j - shift) * inv: shift = max and inv = 1 / sum, or shift = LSE and inv = 1
    float shift, inv;
    if (mode == LCB_CE_BWD) {
      shift = lse_io[r];
      inv = 1.f;
    } else {
      float m = -INFINITY, s = 0.f;
      for (int u = t; u < units; u += kCeThreads) {
        const uint4 w = reinterpret_cast<const uint4*>(row_s)[u];
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
        float y[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          y[2 * e] = bf16lo_to_f32(ww[e]);
          y[2 * e + 1] = bf16hi_to_f32(ww[e]);
        }
        float mu = y[0];
#pragma unroll
        for (int e = 1; e < 8; ++e) mu = fmaxf(mu, y[e]);
        if (mu == -INFINITY) continue;  // eight -inf logits add nothing
        float su = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) su += ex2_approx((y[e] - mu) * kLog2e);
        merge_ms(m, s, mu, su);
      }
      for (int j = units * 8 + t; j < V; j += kCeThreads) merge_ms(m, s, __bfloat162float(row_s[j]), 1.f);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
        merge_ms(m, s, m2, s2);
      }
      if (lane == 0) {
        bars->red_m[warp] = m;
        bars->red_s[warp] = s;
      }
      __syncthreads();
      if (warp == 0) {
        m = lane < kCeWarps ? bars->red_m[lane] : -INFINITY;
        s = lane < kCeWarps ? bars->red_s[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
          merge_ms(m, s, m2, s2);
        }
        if (lane == 0) {
          bars->m = m;
          bars->s = s;
          bars->x_lab = (keep && lab_ok) ? __bfloat162float(row_s[lab]) : 0.f;
        }
      }
      __syncthreads();
      shift = bars->m;
      inv = 1.f / bars->s;
      if (t == 0) {
        const float ln_s = __log2f(bars->s) * kLn2;
        lse_io[r] = bars->m + ln_s;
        // loss = (max - x_label) + ln sum: the difference of two bf16 logits is exact
        if (loss) loss[r] = !keep ? 0.f : (lab_ok ? (bars->m - bars->x_lab) + ln_s : __int_as_float(0x7fc00000));
      }
    }
    if (mode == LCB_CE_FWD) continue;
    // ---- gradient over the staged row, then back to global memory
    const float g = keep ? (dloss ? dloss[r] : 1.f) : 0.f;
    const int lab_i = (keep && lab_ok) ? static_cast<int>(lab) : -1;
    for (int u = t; u < units; u += kCeThreads) {
      uint4 w = reinterpret_cast<const uint4*>(row_s)[u];
      uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int j = 8 * u + 2 * e;
        const float p0 = ex2_approx((bf16lo_to_f32(ww[e]) - shift) * kLog2e) * inv;
        const float p1 = ex2_approx((bf16hi_to_f32(ww[e]) - shift) * kLog2e) * inv;
        ww[e] = pack_bf16x2(g * (p0 - (j == lab_i ? 1.f : 0.f)), g * (p1 - (j + 1 == lab_i ? 1.f : 0.f)));
      }
      reinterpret_cast<uint4*>(row_s)[u] = make_uint4(ww[0], ww[1], ww[2], ww[3]);
    }
    for (int j = units * 8 + t; j < V; j += kCeThreads) {
      const float p = ex2_approx((__bfloat162float(row_s[j]) - shift) * kLog2e) * inv;
      row_s[j] = __float2bfloat16_rn(g * (p - (j == lab_i ? 1.f : 0.f)));
    }
    if (bulk) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncthreads();
      if (t == 0) bulk_s2g(gx, row_s, row_bytes);
    } else {
      __syncthreads();
      for (int j = t; j < V; j += kCeThreads) gx[j] = row_s[j];
      __syncthreads();  // the next row overwrites the staging buffer
    }
  }
  if (t == 0) {
    if (!ok && bulk) drain_wait(&bars->full, phase, st.limit);  // a row copy still in flight lands first
    bulk_wait_all();
  }
}

}  // namespace

int launch_cross_entropy(void* logits, const long long* labels, float* loss, float* lse, const float* dloss, int N,
                         int V, long long row_stride, int ignore_index, int mode, DevStatus st, cudaStream_t stream) {
  const int bars = 128 * static_cast<int>((sizeof(CeBars) + 127) / 128);
  const size_t smem = 128 + bars + ((static_cast<size_t>(V) * 2 + 15) & ~static_cast<size_t>(15));
  if (smem > 232448) return LCB_ERR_UNSUPPORTED;
  static size_t attr = 0;
  if (smem > attr) {
    if (cudaFuncSetAttribute(ce_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return -4;
    attr = smem;
  }
  const int bulk = ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0) && (V % 8 == 0) && (row_stride % 8 == 0);
  const int per_sm = std::max(1, std::min(4, static_cast<int>(232448 / (smem + 1024))));
  const long long grid = std::min<long long>(N, 152LL * per_sm);
  ce_kernel<<<static_cast<unsigned>(grid), kCeThreads, smem, stream>>>(static_cast<__nv_bfloat16*>(logits), labels,
                                                                        loss, lse, dloss, N, V, row_stride,
                                                                        ignore_index, mode, bulk, st);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace lcb
