// Bandwidth-bound kernels around the attention tiles:
//  * LSE merge of two partial results over disjoint key sets, the step that
//    composes ring attention ("EasyContext核心技术解析：序列并行与Flash
//    Attention的完美结合", §1 "序列并行技术");
//  * the backward preprocess Delta_i = dO_i . O_i;
//  * row gather/scatter into and out of zigzag order ("EasyContext代码解析200行
//    核心训练脚本实现原理", §训练循环核心逻辑, per-rank sequence pieces);
//  * the bounded-wait self test.
//
// Each (batch, row, head) vector of D = 128 values is handled by one warp:
// a lane owns 4 consecutive values, so a warp reads 256 B of bf16 or 512 B of
// fp32 contiguously. Grids are a multiple of the SM count and stride over the
// vectors.
#include <cuda_bf16.h>

#include <algorithm>
#include <type_traits>

#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kD = 128;
constexpr int kSMs = 152;

__device__ __forceinline__ float4 load_bf16x4(const __nv_bfloat16* p) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p));
  return make_float4(bf16lo_to_f32(u.x), bf16hi_to_f32(u.x), bf16lo_to_f32(u.y), bf16hi_to_f32(u.y));
}

// The same merge with one warp per token row over all heads, four heads'
// loads in flight per lane (16 bytes of the fp32 accumulator and 8 or 16
// bytes of the block result each), four CTAs resident per SM; the row's base addresses are formed once,
// the block's dtype and the bf16 copy out are template parameters. Per element
// the arithmetic is lse_merge_kernel's.
template <bool kObF32, bool kOut>
__global__ void __launch_bounds__(256, 4) lse_merge_rows_kernel(float* __restrict__ o_acc, float* __restrict__ lse_acc,
                                                                const void* __restrict__ o_b,
                                                                const float* __restrict__ lse_b, __nv_bfloat16* o_out,
                                                                int B, int H, int rows, long long o_rs, long long o_bs,
                                                                long long ob_rs, long long ob_bs, long long l_hs,
                                                                long long l_bs, long long lb_hs, long long lb_bs) {
  constexpr int G = 4;  // eight heads with two CTAs per SM: 0.78 of HBM, four with four: 0.83
  using BT = typename std::conditional<kObF32, float, __nv_bfloat16>::type;
  const long long n = static_cast<long long>(B) * rows;
  const int ln = threadIdx.x & 31;
  const long long wstep = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < n; w += wstep) {
    const int r = static_cast<int>(w % rows);
    const int b = static_cast<int>(w / rows);
    // per-row bases, advanced by one group of heads per iteration: the heads
    // of a group sit at fixed offsets (p * 128 values) from them
    float* pa = o_acc + b * o_bs + static_cast<long long>(r) * o_rs + ln * 4;
    const BT* pb = static_cast<const BT*>(o_b) + b * ob_bs + static_cast<long long>(r) * ob_rs + ln * 4;
    __nv_bfloat16* po = kOut ? o_out + b * o_bs + static_cast<long long>(r) * o_rs + ln * 4 : nullptr;
    float* pla = lse_acc + b * l_bs + r;
    const float* plb = lse_b + b * lb_bs + r;
    for (int h0 = 0; h0 < H; h0 += G, pa += G * kD, pb += G * kD, po += kOut ? G * kD : 0) {
      float4 oa[G], ob[G];
      float la[G], lb[G];
      {
        const float* qa = pla;
        const float* qb = plb;
#pragma unroll
        for (int p = 0; p < G; ++p, qa += l_hs, qb += lb_hs) {
          if (h0 + p >= H) continue;
          oa[p] = *reinterpret_cast<const float4*>(pa + p * kD);
          if constexpr (kObF32) {
            ob[p] = __ldg(reinterpret_cast<const float4*>(pb + p * kD));
          } else {
            ob[p] = load_bf16x4(pb + p * kD);
          }
          la[p] = *qa;
          lb[p] = __ldg(qb);
        }
      }
      __syncwarp();  // every lane has read the group's LSE before lane 0 overwrites it
#pragma unroll
      for (int p = 0; p < G; ++p, pla += l_hs, plb += lb_hs) {
        if (h0 + p >= H) continue;
        const float m = fmaxf(la[p], lb[p]);
        float4 out;
        float lse;
        if (m == -INFINITY) {
          out = make_float4(0.f, 0.f, 0.f, 0.f);
          lse = -INFINITY;
        } else {
          const float wa = __expf(la[p] - m);  // exp(-inf) = 0 for an empty side
          const float wb = __expf(lb[p] - m);
          const float den = wa + wb;
          const float inv = 1.f / den;
          const float ca = wa * inv, cb = wb * inv;
          out = make_float4(ca * oa[p].x + cb * ob[p].x, ca * oa[p].y + cb * ob[p].y, ca * oa[p].z + cb * ob[p].z,
                            ca * oa[p].w + cb * ob[p].w);
          lse = m + __logf(den);
        }
        *reinterpret_cast<float4*>(pa + p * kD) = out;
        if constexpr (kOut) {
          uint2 u;
          u.x = pack_bf16x2(out.x, out.y);
          u.y = pack_bf16x2(out.z, out.w);
          *reinterpret_cast<uint2*>(po + p * kD) = u;
        }
        if (ln == 0) *pla = lse;
      }
    }
  }
}

__global__ void __launch_bounds__(256) lse_merge_kernel(float* __restrict__ o_acc, float* __restrict__ lse_acc,
                                                        const void* __restrict__ o_b, int o_b_f32,
                                                        const float* __restrict__ lse_b, __nv_bfloat16* o_out,
                                                        int B, int H, int rows, long long o_rs, long long o_bs,
                                                        long long ob_rs, long long ob_bs, long long l_hs,
                                                        long long l_bs, long long lb_hs, long long lb_bs) {
  const long long n = static_cast<long long>(B) * rows * H;
  const int ln = threadIdx.x & 31;
  const long long wstep = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < n; w += wstep) {
    const int h = static_cast<int>(w % H);
    const long long br = w / H;
    const int r = static_cast<int>(br % rows);
    const int b = static_cast<int>(br / rows);
    const long long off = b * o_bs + static_cast<long long>(r) * o_rs + h * kD + ln * 4;
    const long long boff = b * ob_bs + static_cast<long long>(r) * ob_rs + h * kD + ln * 4;
    const long long loff = b * l_bs + h * l_hs + r;
    const float la = lse_acc[loff];
    const float lb = __ldg(lse_b + b * lb_bs + h * lb_hs + r);
    const float m = fmaxf(la, lb);
    float4 oa = *reinterpret_cast<const float4*>(o_acc + off);
    float4 ob = o_b_f32 ? __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(o_b) + boff))
                        : load_bf16x4(static_cast<const __nv_bfloat16*>(o_b) + boff);
    float4 out;
    float lse;
    if (m == -INFINITY) {
      out = make_float4(0.f, 0.f, 0.f, 0.f);
      lse = -INFINITY;
    } else {
      const float wa = __expf(la - m);  // exp(-inf) = 0 for an empty side
      const float wb = __expf(lb - m);
      const float den = wa + wb;
      const float inv = 1.f / den;
      const float ca = wa * inv, cb = wb * inv;
      out = make_float4(ca * oa.x + cb * ob.x, ca * oa.y + cb * ob.y, ca * oa.z + cb * ob.z, ca * oa.w + cb * ob.w);
      lse = m + __logf(den);
    }
    *reinterpret_cast<float4*>(o_acc + off) = out;
    if (o_out) {
      uint2 u;
      u.x = pack_bf16x2(out.x, out.y);
      u.y = pack_bf16x2(out.z, out.w);
      *reinterpret_cast<uint2*>(o_out + off) = u;
    }
    __syncwarp();
    if (ln == 0) lse_acc[loff] = lse;
  }
}

// Delta for one token row per warp, all heads: the row's H * 256 bytes of O and
// of dO are read 512 contiguous bytes per instruction (16 bytes a lane, two
// heads per warp-wide load, four such loads in flight), and each half-warp
// reduces one head's dot product. Rows must start on 16 bytes and H be even.
__global__ void __launch_bounds__(256) bwd_preprocess_rows_kernel(const uint4* __restrict__ o,
                                                                  const uint4* __restrict__ dO, long long rs16,
                                                                  long long bs16, float* __restrict__ delta,
                                                                  long long d_hs, long long d_bs, int B, int H, int S) {
  const long long rows = static_cast<long long>(B) * S;
  const int ln = threadIdx.x & 31;
  const int half = ln >> 4;  // which head of the pair this lane's 16 bytes belong to
  const long long wstep = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows;
       w += wstep) {
    const int s = static_cast<int>(w % S);
    const int b = static_cast<int>(w / S);
    const long long row = b * bs16 + static_cast<long long>(s) * rs16;
    for (int h0 = 0; h0 < H; h0 += 8) {
      float acc[4];
#pragma unroll
      for (int p = 0; p < 4; ++p) {
        const int hp = h0 + 2 * p;  // heads hp, hp + 1
        acc[p] = 0.f;
        if (hp < H) {
          const uint4 x = __ldg(o + row + hp * (kD / 8) + ln);
          const uint4 y = __ldg(dO + row + hp * (kD / 8) + ln);
          const uint32_t xs[4] = {x.x, x.y, x.z, x.w}, ys[4] = {y.x, y.y, y.z, y.w};
#pragma unroll
          for (int e = 0; e < 4; ++e)
            acc[p] += bf16lo_to_f32(xs[e]) * bf16lo_to_f32(ys[e]) + bf16hi_to_f32(xs[e]) * bf16hi_to_f32(ys[e]);
        }
      }
#pragma unroll
      for (int p = 0; p < 4; ++p) {
#pragma unroll
        for (int k = 8; k > 0; k >>= 1) acc[p] += __shfl_xor_sync(0xffffffffu, acc[p], k);
        const int h = h0 + 2 * p + half;
        if ((ln & 15) == 0 && h < H) delta[b * d_bs + h * d_hs + s] = acc[p];
      }
    }
  }
}

__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ dO, long long rs,
                                                             long long bs, float* __restrict__ delta, long long d_hs,
                                                             long long d_bs, int B, int H, int S) {
  const long long n = static_cast<long long>(B) * S * H;
  const int ln = threadIdx.x & 31;
  const long long wstep = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < n; w += wstep) {
    const int h = static_cast<int>(w % H);
    const long long bs_ = w / H;
    const int s = static_cast<int>(bs_ % S);
    const int b = static_cast<int>(bs_ / S);
    const long long off = b * bs + static_cast<long long>(s) * rs + h * kD + ln * 4;
    const float4 x = load_bf16x4(o + off);
    const float4 y = load_bf16x4(dO + off);
    float acc = x.x * y.x + x.y * y.y + x.z * y.z + x.w * y.w;
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, k);
    if (ln == 0) delta[b * d_bs + h * d_hs + s] = acc;
  }
}

__global__ void __launch_bounds__(256) permute_rows_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                           const int* __restrict__ perm, int rows, long long vecs,
                                                           int scatter) {
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const long long from = scatter ? r : __ldg(perm + r);
    const long long to = scatter ? __ldg(perm + r) : r;
    const uint4* s = src + from * vecs;
    uint4* d = dst + to * vecs;
    for (long long i = threadIdx.x; i < vecs; i += blockDim.x) d[i] = __ldg(s + i);
  }
}

// Waits on a barrier that nothing completes; must end by its own time limit.
__global__ void wait_selftest_kernel(DevStatus st) {
  __shared__ uint64_t bar;
  __shared__ volatile int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  mbar_wait(&bar, 0, &abort_flag, st, 0xffu << 24);
  __syncthreads();
}

__global__ void __launch_bounds__(256) cast_f32_bf16_kernel(const float4* __restrict__ src, uint2* __restrict__ dst,
                                                            long long n4) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 x = __ldg(src + i);
    dst[i] = make_uint2(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w));
  }
}

__global__ void cast_tail_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst, long long from,
                                 long long n) {
  const long long i = from + threadIdx.x;
  if (i < n) dst[i] = __float2bfloat16_rn(src[i]);
}

int grid_for(long long warps) {
  const long long blocks = (warps + 7) / 8;
  return static_cast<int>(std::max<long long>(1, std::min<long long>(blocks, kSMs * 16LL)));
}

}  // namespace

int launch_lse_merge(float* o_acc, float* lse_acc, const void* o_b, int o_b_f32, const float* lse_b, void* o_out_bf16,
                     int B, int H, int rows, long long o_row_stride, long long o_batch_stride,
                     long long ob_row_stride, long long ob_batch_stride, long long lse_head_stride,
                     long long lse_batch_stride, long long lseb_head_stride, long long lseb_batch_stride,
                     cudaStream_t stream) {
  const long long warps = static_cast<long long>(B) * rows * H;
  if (warps == 0) return 0;
  if (H >= 4) {
    // a warp per token row (four CTAs of 8 warps resident per SM at 64
    // registers a thread), four heads' loads of every warp in flight
    const long long row_warps = static_cast<long long>(B) * rows;
    const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>((row_warps + 7) / 8, kSMs * 16LL)));
    auto* out = static_cast<__nv_bfloat16*>(o_out_bf16);
    auto kernel = o_b_f32 ? (out ? lse_merge_rows_kernel<true, true> : lse_merge_rows_kernel<true, false>)
                          : (out ? lse_merge_rows_kernel<false, true> : lse_merge_rows_kernel<false, false>);
    kernel<<<grid, 256, 0, stream>>>(o_acc, lse_acc, o_b, lse_b, out, B, H, rows, o_row_stride, o_batch_stride,
                                     ob_row_stride, ob_batch_stride, lse_head_stride, lse_batch_stride,
                                     lseb_head_stride, lseb_batch_stride);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
  }
  lse_merge_kernel<<<grid_for(warps), 256, 0, stream>>>(o_acc, lse_acc, o_b, o_b_f32, lse_b,
                                                        static_cast<__nv_bfloat16*>(o_out_bf16), B, H, rows,
                                                        o_row_stride, o_batch_stride, ob_row_stride,
                                                        ob_batch_stride, lse_head_stride, lse_batch_stride,
                                                        lseb_head_stride, lseb_batch_stride);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_bwd_preprocess(const void* o, const void* dO, long long row_stride, long long batch_stride, float* delta,
                          long long d_head_stride, long long d_batch_stride, int B, int H, int S, cudaStream_t stream) {
  const long long warps = static_cast<long long>(B) * S * H;
  if (warps == 0) return 0;
  const bool rows16 = ((reinterpret_cast<uintptr_t>(o) | reinterpret_cast<uintptr_t>(dO)) & 15u) == 0 &&
                      row_stride % 8 == 0 && batch_stride % 8 == 0 && H % 2 == 0;
  if (rows16) {
    bwd_preprocess_rows_kernel<<<grid_for(static_cast<long long>(B) * S), 256, 0, stream>>>(
        static_cast<const uint4*>(o), static_cast<const uint4*>(dO), row_stride / 8, batch_stride / 8, delta,
        d_head_stride, d_batch_stride, B, H, S);
    return cudaGetLastError() == cudaSuccess ? 0 : -4;
  }
  bwd_preprocess_kernel<<<grid_for(warps), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(o), static_cast<const __nv_bfloat16*>(dO), row_stride, batch_stride, delta,
      d_head_stride, d_batch_stride, B, H, S);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_permute_rows(const void* src, void* dst, const int* perm, int rows, long long row_bytes, int scatter,
                        cudaStream_t stream) {
  if (rows == 0) return 0;
  const int blocks = std::min(rows, kSMs * 8);
  permute_rows_kernel<<<blocks, 256, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), perm, rows,
                                                  row_bytes / 16, scatter);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_cast_f32_bf16(const float* src, void* dst, long long n, cudaStream_t stream) {
  const long long n4 = n / 4;
  if (n4 > 0) {
    const int blocks = static_cast<int>(std::max<long long>(1, std::min<long long>((n4 + 255) / 256, kSMs * 16LL)));
    cast_f32_bf16_kernel<<<blocks, 256, 0, stream>>>(reinterpret_cast<const float4*>(src), static_cast<uint2*>(dst),
                                                     n4);
  }
  if (n4 * 4 < n) {
    cast_tail_kernel<<<1, 32, 0, stream>>>(src, static_cast<__nv_bfloat16*>(dst), n4 * 4, n);
  }
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

int launch_wait_selftest(DevStatus st, cudaStream_t stream) {
  wait_selftest_kernel<<<1, 32, 0, stream>>>(st);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace lcb
