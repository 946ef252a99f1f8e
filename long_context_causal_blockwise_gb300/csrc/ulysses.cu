// Ulysses sequence parallelism emulated on one device: the all-to-all that
// turns P sequence pieces into P head groups and back
// ("EasyContext核心技术解析：序列并行与Flash Attention的完美结合", §1
// "序列并行技术": Ulysses注意力; "EasyContext未来展望：从1M到10M上下文的技术路线图",
// §关键技术突破点: Deepspeed Ulysses).
//
// Rank r of P holds sequence rows [r S/P, (r+1) S/P) of all H heads; after
// the all-to-all rank j holds every row of heads [j H/P, (j+1) H/P). With all
// ranks on one device the sequence layout is the ordinary [B, S, H, D]
// tensor, and the head layout is [P, B, S, H/P, D]: rank j's part is a
// [B, S, H/P, D] tensor, and the P parts together are one [P*B, S, H/P, D]
// batch, so a single attention launch serves every rank.
//
// A pure copy, bound by HBM: each element is read once and written once.
// Seen as 16-byte vectors, a row of the sequence layout is P blocks of bv
// vectors (one per head group), and the kernel moves block j of row r to
// position r of group j. Threads walk the head layout linearly, so one side is
// fully contiguous and the other is contiguous over runs of bv vectors
// ((H/P) * D * elem_bytes bytes, 1 KB for 4 bf16 heads).
#include <cuda_runtime.h>

#include <algorithm>

#include "lcb_attn.h"
#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;  // vectors in flight per thread

// dir 0: sequence layout -> head layout; dir 1: the inverse.
template <int kDir>
__global__ void __launch_bounds__(kThreads) ulysses_a2a_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst,
                                                               unsigned rows, unsigned bv, unsigned P) {
  const unsigned j = blockIdx.y;       // head group (receiving rank for dir 0)
  const unsigned n = rows * bv;        // vectors of one group: fits 32 bits (checked by the host)
  const unsigned stride = gridDim.x * kThreads;
  const size_t group_base = static_cast<size_t>(j) * n;
  for (unsigned i0 = blockIdx.x * kThreads + threadIdx.x; i0 < n; i0 += kUnroll * stride) {
    uint4 v[kUnroll];
    size_t dst_at[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const unsigned i = i0 + u * stride;
      if (i < n) {
        const unsigned row = i / bv, w = i - row * bv;
        const size_t head_at = group_base + i;
        const size_t seq_at = (static_cast<size_t>(row) * P + j) * bv + w;
        v[u] = __ldg(src + (kDir == 0 ? seq_at : head_at));
        dst_at[u] = kDir == 0 ? head_at : seq_at;
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (i0 + u * stride < n) dst[dst_at[u]] = v[u];
    }
  }
}

}  // namespace

int launch_ulysses_a2a(const void* src, void* dst, long long rows, long long bv, int P, int dir,
                       cudaStream_t stream) {
  const long long n = rows * bv;
  if (n == 0) return 0;
  if (n >= (1LL << 31) || P > 65535) return -1;
  const long long want = (static_cast<long long>(152) * 8 + P - 1) / P;  // about 8 CTAs per SM over the groups
  const unsigned gx = static_cast<unsigned>(std::max(1LL, std::min(want, (n + kThreads - 1) / kThreads)));
  const dim3 grid(gx, static_cast<unsigned>(P));
  if (dir == 0)
    ulysses_a2a_kernel<0><<<grid, kThreads, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                        static_cast<unsigned>(rows), static_cast<unsigned>(bv),
                                                        static_cast<unsigned>(P));
  else
    ulysses_a2a_kernel<1><<<grid, kThreads, 0, stream>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst),
                                                        static_cast<unsigned>(rows), static_cast<unsigned>(bv),
                                                        static_cast<unsigned>(P));
  return cudaGetLastError() == cudaSuccess ? 0 : -4;
}

}  // namespace lcb
