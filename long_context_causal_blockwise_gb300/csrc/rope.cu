// Rotary position embedding with a raised base, applied once to Q and K
// before attention (and, inverted, to dQ and dK after it): the long-context
// recipe raises the rotary base theta ("EasyContext核心技术解析：序列并行与
// Flash Attention的完美结合" §3 "RoPE扩展技术"; --rope-theta 1000000 on
// "EasyContext内存优化秘籍DeepSpeed Zero3卸载策略详解" §训练脚本配置).
//
// Pair k of a head couples features k and k + 64 and turns by
// a = (pos0 + s) * f_k, f_k = theta^(-2k/128). The product and its reduction
// modulo 2 pi run in fp64 (an fp32 angle at position 5e5 would be off by
// about 0.03 rad); sin and cos of the reduced angle, and the rotation, in fp32
// (the angle's fp32 rounding corrected to first order).
//
// One warp per token row (b, s): lane l owns pairs 2l and 2l + 1, computes
// their two angles once and rotates them in every head, reading and writing
// 4 bytes from each half of each head (a warp moves 128 contiguous bytes per
// half-head). The kernel is bound by HBM: every element is read and written
// once; in place is allowed. A call may be in place, so the compiler cannot
// move one head's loads above the previous head's stores; the loads of eight
// heads are therefore issued together before their stores (one head at a
// time held about 256 bytes per warp in flight and reached 0.84 of the copy
// bandwidth, eight reach 0.98).
#include <cuda_bf16.h>

#include <algorithm>

#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kD = 128;

// cos and sin of a reduced fp64 angle a = hi + lo with hi = (float)a: sincosf
// of hi, then one first-order step for lo (|lo| < 4e-7), which removes the
// error of rounding the angle to fp32.
__device__ __forceinline__ void turn(double a, float& c, float& s) {
  const float hi = static_cast<float>(a);
  const float lo = static_cast<float>(a - static_cast<double>(hi));
  float sh, ch;
  sincosf(hi, &sh, &ch);
  c = fmaf(-lo, sh, ch);
  s = fmaf(lo, ch, sh);
}

__global__ void __launch_bounds__(256) rope_kernel(const __nv_bfloat16* x, __nv_bfloat16* y, int B, int S, int H,
                                                   long long rs, long long bs, long long pos0, float sign,
                                                   RopeFreqs fr) {
  const long long rows = static_cast<long long>(B) * S;
  const int lane = threadIdx.x & 31;
  const long long wstep = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  for (long long w = static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); w < rows;
       w += wstep) {
    const int s = static_cast<int>(w % S);
    const int b = static_cast<int>(w / S);
    const double pos = static_cast<double>(pos0 + s);
    float c0, s0, c1, s1;
    turn(fmod(pos * fr.f[2 * lane], kTwoPi), c0, s0);
    turn(fmod(pos * fr.f[2 * lane + 1], kTwoPi), c1, s1);
    s0 *= sign;
    s1 *= sign;
    const long long row = b * bs + static_cast<long long>(s) * rs;
    int h = 0;
    for (; h + 8 <= H; h += 8) {  // eight heads' loads in flight before their stores
      uint32_t a[8], cc[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const long long lo = row + (h + u) * kD + 2 * lane;
        a[u] = *reinterpret_cast<const uint32_t*>(x + lo);
        cc[u] = *reinterpret_cast<const uint32_t*>(x + lo + kD / 2);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const long long lo = row + (h + u) * kD + 2 * lane;
        const float a0 = bf16lo_to_f32(a[u]), a1 = bf16hi_to_f32(a[u]);
        const float c0v = bf16lo_to_f32(cc[u]), c1v = bf16hi_to_f32(cc[u]);
        *reinterpret_cast<uint32_t*>(y + lo) = pack_bf16x2(a0 * c0 - c0v * s0, a1 * c1 - c1v * s1);
        *reinterpret_cast<uint32_t*>(y + lo + kD / 2) = pack_bf16x2(c0v * c0 + a0 * s0, c1v * c1 + a1 * s1);
      }
    }
    for (; h < H; ++h) {
      const long long lo = row + h * kD + 2 * lane;
      const uint32_t a = *reinterpret_cast<const uint32_t*>(x + lo);
      const uint32_t c = *reinterpret_cast<const uint32_t*>(x + lo + kD / 2);
      const float a0 = bf16lo_to_f32(a), a1 = bf16hi_to_f32(a);
      const float c0v = bf16lo_to_f32(c), c1v = bf16hi_to_f32(c);
      *reinterpret_cast<uint32_t*>(y + lo) = pack_bf16x2(a0 * c0 - c0v * s0, a1 * c1 - c1v * s1);
      *reinterpret_cast<uint32_t*>(y + lo + kD / 2) = pack_bf16x2(c0v * c0 + a0 * s0, c1v * c1 + a1 * s1);
    }
  }
}

}  // namespace

int launch_rope(const void* x, void* y, int B, int S, int H, long long row_stride, long long batch_stride,
                long long pos0, int inverse, const RopeFreqs& fr, cudaStream_t stream) {
  const long long warps = static_cast<long long>(B) * S;
  if (warps == 0) return 0;
  const long long blocks = std::min<long long>((warps + 7) / 8, 152LL * 16);
  rope_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(x), static_cast<__nv_bfloat16*>(y), B, S, H, row_stride, batch_stride, pos0,
      inverse ? -1.f : 1.f, fr);
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace lcb
