// attn_bwd_noalloc: the attention backward for callers that cannot allocate
// device memory.
//
// attn_bwd needs a scratch buffer for Delta (one fp32 per query row and head),
// which the caller normally passes as a workspace. Some callers cannot
// produce one. Examples: a host framework whose memory manager owns all
// device memory and hands this library only the tensors it computes on; a
// service that fixes its memory plan at start-up and forbids allocation
// afterwards; code that must not call cudaMalloc because that call can
// synchronise the device in the middle of an asynchronous pipeline. For them
// this entry point keeps the scratch in a fixed array in device global
// memory, compiled into the library. The array is reserved on a device when
// this file's module is loaded into that device's context: with CUDA's lazy
// module loading (the default) that happens during the first call of this
// entry point on the device, and the array is then held until the process
// exits or the context is reset.
//
// The entry point runs the same kernels as attn_bwd_ex: Delta preprocess, then
// the dK/dV and dQ passes, with Delta read from the array.
#include <cuda_runtime.h>

#include "lcb_attn.h"

namespace {

// Up to this many (batch, head, row) Delta values: 2^21 fp32 = 8 MiB.
constexpr long long kNoAllocMaxRows = 1LL << 21;

static __device__ __align__(256) float g_noalloc_delta[kNoAllocMaxRows];

// Device address of the array in the current device's context. The host-side
// name of the array is not a device address. The address is looked up on
// every call, not cached: after cudaDeviceReset the module is loaded again and
// the array may sit elsewhere. Once the module is loaded the lookup allocates
// nothing; the first lookup on a device loads it.
int scratch_ptr(float** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_delta) != cudaSuccess || p == nullptr) return LCB_ERR_CUDA;
  *out = static_cast<float*>(p);
  return LCB_OK;
}

}  // namespace

extern "C" long long attn_bwd_noalloc_max_rows(void) { return kNoAllocMaxRows; }

extern "C" int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                                const void* dO, void* dq, void* dk, void* dv, int B, int H, int S, int D, int causal,
                                float scale, void* stream) {
  if (B < 1 || H < 1 || S < 0) return LCB_ERR_ARG;
  if (static_cast<long long>(B) * H * S > kNoAllocMaxRows) return LCB_ERR_SCRATCH;
  if (S == 0) return LCB_OK;
  float* delta = nullptr;
  int rc = scratch_ptr(&delta);
  if (rc != LCB_OK) return rc;
  // Delta is written in full by the preprocess before the passes read it, so
  // nothing left in the array by an earlier call is ever read.
  const long long rs = static_cast<long long>(H) * D;
  const long long bs = rs * S;
  rc = attn_bwd_preprocess(o, dO, delta, B, H, S, D, rs, bs, S, static_cast<long long>(H) * S, stream);
  if (rc != LCB_OK) return rc;
  return attn_bwd_ex(q, k, v, lse, delta, dO, dq, dk, dv, B, H, S, S, D, causal, scale, rs, bs, rs, bs, S,
                     static_cast<long long>(H) * S, LCB_GRAD_BF16, rs, bs, rs, bs, stream);
}
