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
// One CTA per row at a time (persistent over rows), the row streamed through
// registers: every thread keeps four 16-byte loads in flight, reduces its
// share of the row to (max, sum of exp) in batches of 32 logits (one exp per
// logit), the CTA merges the threads' pairs; the gradient pass reads the row
// again and writes it in place. Many rows are in flight per SM, so HBM
// latency is covered without staging rows in shared memory. With the forward
// and backward in one call the second read of a row comes soon after the
// first: the launch keeps the rows in flight within L2 (about 40 MB), so HBM
// still sees each logit read once and written once. Rows whose address or
// length is not a multiple of 16 bytes are read one logit at a time.
#include <cuda_bf16.h>

#include <algorithm>

#include "lcb_attn.h"
#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kBatch = 4;  // 16-byte loads in flight per thread
constexpr int kSms = 152;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

// (m, s) with m a running maximum of logits and s = sum exp(x - m); merging
// two such pairs. Differences of bf16 logits are exact in fp32, so exp(x - m)
// keeps full relative accuracy even for logits of large magnitude.
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
  const float M = fmaxf(m, m2);
  if (M == -INFINITY) return;
  s = s * ex2_approx((m - M) * kLog2e) + s2 * ex2_approx((m2 - M) * kLog2e);
  m = M;
}

// Folds 8 * n logits (n 16-byte units of bf16 pairs) into (m, s): the batch
// maximum first, then one exp per logit against the updated running maximum.
template <int n>
__device__ __forceinline__ void fold_units(float& m, float& s, const uint4* w) {
  float bm = -INFINITY;
#pragma unroll
  for (int i = 0; i < n; ++i) {
    const uint32_t ww[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) bm = fmaxf(bm, fmaxf(bf16lo_to_f32(ww[e]), bf16hi_to_f32(ww[e])));
  }
  if (bm == -INFINITY) return;  // -inf logits add nothing
  if (bm > m) {
    s = (m == -INFINITY) ? 0.f : s * ex2_approx((m - bm) * kLog2e);
    m = bm;
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < n; ++i) {
    const uint32_t ww[4] = {w[i].x, w[i].y, w[i].z, w[i].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      acc += ex2_approx((bf16lo_to_f32(ww[e]) - m) * kLog2e);
      acc += ex2_approx((bf16hi_to_f32(ww[e]) - m) * kLog2e);
    }
  }
  s += acc;
}

// Gradient of logits 8u .. 8u + 7: q * exp(x - shift) with q = g / sum (or g
// with a given LSE); the label's logit, if among them, gets g * (p - 1).
__device__ __forceinline__ uint4 grad_unit(uint4 w, int u, float shift, float inv, float q, float g, int lab_i) {
  uint32_t ww[4] = {w.x, w.y, w.z, w.w};
  if (lab_i < 8 * u || lab_i >= 8 * u + 8) {
#pragma unroll
    for (int e = 0; e < 4; ++e)
      ww[e] = pack_bf16x2(ex2_approx((bf16lo_to_f32(ww[e]) - shift) * kLog2e) * q,
                          ex2_approx((bf16hi_to_f32(ww[e]) - shift) * kLog2e) * q);
  } else {
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int j = 8 * u + 2 * e;
      const float p0 = ex2_approx((bf16lo_to_f32(ww[e]) - shift) * kLog2e) * inv;
      const float p1 = ex2_approx((bf16hi_to_f32(ww[e]) - shift) * kLog2e) * inv;
      ww[e] = pack_bf16x2(g * (p0 - (j == lab_i ? 1.f : 0.f)), g * (p1 - (j + 1 == lab_i ? 1.f : 0.f)));
    }
  }
  return make_uint4(ww[0], ww[1], ww[2], ww[3]);
}

template <int kThreads>
__global__ void __launch_bounds__(kThreads) ce_kernel(__nv_bfloat16* logits, const long long* labels, float* loss,
                                                      float* lse_io, const float* dloss, int N, int V, long long rs,
                                                      int ignore_index, int mode, int vec) {
  constexpr int kWarps = kThreads / 32;
  __shared__ float red_m[kWarps], red_s[kWarps];
  __shared__ float row_m, row_s;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int units = vec ? V / 8 : 0;  // 16-byte units; the rest is read one logit at a time
  for (long long r = blockIdx.x; r < N; r += gridDim.x) {
    __nv_bfloat16* gx = logits + r * rs;
    const long long lab = labels[r];
    const bool keep = lab != ignore_index;
    const bool lab_ok = lab >= 0 && lab < V;
    // p_j = exp(x_j - shift) * inv: shift = max and inv = 1 / sum, or shift = the given LSE and inv = 1
    float shift, inv;
    if (mode == LCB_CE_BWD) {
      shift = lse_io[r];
      inv = 1.f;
    } else {
      float m = -INFINITY, s = 0.f;
      const uint4* g4 = reinterpret_cast<const uint4*>(gx);
      int u = t;
      for (; u + (kBatch - 1) * kThreads < units; u += kBatch * kThreads) {
        uint4 w[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) w[i] = g4[u + i * kThreads];
        fold_units<kBatch>(m, s, w);
      }
      for (; u < units; u += kThreads) fold_units<1>(m, s, g4 + u);
      for (int j = units * 8 + t; j < V; j += kThreads) merge_ms(m, s, __bfloat162float(gx[j]), 1.f);
      // the label logit is read before the barriers below, ahead of any gradient write
      const float x_lab = (t == 0 && keep && lab_ok) ? __bfloat162float(gx[lab]) : 0.f;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
        merge_ms(m, s, m2, s2);
      }
      if (lane == 0) {
        red_m[warp] = m;
        red_s[warp] = s;
      }
      __syncthreads();
      if (warp == 0) {
        m = lane < kWarps ? red_m[lane] : -INFINITY;
        s = lane < kWarps ? red_s[lane] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float m2 = __shfl_xor_sync(0xffffffffu, m, o), s2 = __shfl_xor_sync(0xffffffffu, s, o);
          merge_ms(m, s, m2, s2);
        }
        if (lane == 0) {
          row_m = m;
          row_s = s;
        }
      }
      __syncthreads();  // also: the next row's partials go to red_* only after warp 0 read these
      m = row_m;
      s = row_s;
      shift = m;
      inv = 1.f / s;
      if (t == 0) {
        const float ln_s = __log2f(s) * kLn2;
        lse_io[r] = m + ln_s;
        // loss = (max - x_label) + ln sum: the difference of two bf16 logits is exact
        if (loss) loss[r] = !keep ? 0.f : (lab_ok ? (m - x_lab) + ln_s : __int_as_float(0x7fc00000));
      }
    }
    if (mode == LCB_CE_FWD) continue;
    // ---- gradient, written over the row
    const float g = keep ? (dloss ? dloss[r] : 1.f) : 0.f;
    const float q = g * inv;
    const int lab_i = (keep && lab_ok) ? static_cast<int>(lab) : -1;  // -1: no one-hot term
    uint4* g4 = reinterpret_cast<uint4*>(gx);
    int u = t;
    for (; u + (kBatch - 1) * kThreads < units; u += kBatch * kThreads) {
      uint4 w[kBatch];
#pragma unroll
      for (int i = 0; i < kBatch; ++i) w[i] = g4[u + i * kThreads];
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        g4[u + i * kThreads] = grad_unit(w[i], u + i * kThreads, shift, inv, q, g, lab_i);
    }
    for (; u < units; u += kThreads) g4[u] = grad_unit(g4[u], u, shift, inv, q, g, lab_i);
    for (int j = units * 8 + t; j < V; j += kThreads) {
      const float p = ex2_approx((__bfloat162float(gx[j]) - shift) * kLog2e) * inv;
      gx[j] = __float2bfloat16_rn(g * (p - (j == lab_i ? 1.f : 0.f)));
    }
  }
}

}  // namespace

int launch_cross_entropy(void* logits, const long long* labels, float* loss, float* lse, const float* dloss, int N,
                         int V, long long row_stride, int ignore_index, int mode, cudaStream_t stream) {
  __nv_bfloat16* x = static_cast<__nv_bfloat16*>(logits);
  const int vec = ((reinterpret_cast<uintptr_t>(logits) & 15u) == 0) && (V % 8 == 0) && (row_stride % 8 == 0);
  // 256-thread CTAs, five per SM (the most its 44 registers a thread allow):
  // 760 rows in flight, the row-end reductions of one CTA covered by the
  // loads of four others. With forward and backward in one call a row is read
  // twice, so the rows in flight must stay within L2 (64 MB of it) for the
  // second read: above that, four CTAs per SM (608 rows, V up to about 55000),
  // then one 1024-thread CTA per SM (152 rows). The shape depends on V alone,
  // and the order in which a row is reduced only on the CTA size, so every
  // mode gives the same loss and LSE bits.
  const long long row_bytes = 2LL * V;
  if (4LL * kSms * row_bytes > (64LL << 20)) {
    const long long grid = std::min<long long>(N, kSms);
    ce_kernel<1024><<<static_cast<unsigned>(grid), 1024, 0, stream>>>(x, labels, loss, lse, dloss, N, V, row_stride,
                                                                      ignore_index, mode, vec);
  } else {
    const long long per_sm = (5LL * kSms * row_bytes > (64LL << 20)) ? 4 : 5;
    const long long grid = std::min<long long>(N, per_sm * kSms);
    ce_kernel<256><<<static_cast<unsigned>(grid), 256, 0, stream>>>(x, labels, loss, lse, dloss, N, V, row_stride,
                                                                    ignore_index, mode, vec);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace lcb
