// C ABI of libattn.so: argument validation, TMA descriptor set-up, status
// handling and the host-side zigzag schedule. Every compute entry point
// enqueues kernels of this library on the caller's stream; there is no other
// backend and no CPU fallback.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "lcb_attn.h"
#include "lcb_internal.h"

namespace lcb {
namespace {

constexpr int kHeadDim = 128;

__device__ uint32_t g_status_words[4];


unsigned long long env_wait_limit() {
  const char* s = std::getenv("LCB_WAIT_LIMIT_NS");
  if (s && *s) {
    const unsigned long long v = std::strtoull(s, nullptr, 10);
    if (v > 0) return v;
  }
  return 2000000000ULL;
}

std::atomic<unsigned long long> g_wait_limit{env_wait_limit()};

bool checked_mode() {
  static const bool on = [] {
    const char* s = std::getenv("LCB_CHECKED");
    return s && s[0] == '1';
  }();
  return on;
}

// Device address of the status word in the current device's context. Looked
// up on every call rather than cached: a context torn down by
// cudaDeviceReset and created again may place the word elsewhere.
int status_words(uint32_t** out) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_status_words) != cudaSuccess || p == nullptr) return LCB_ERR_CUDA;
  *out = static_cast<uint32_t*>(p);
  return LCB_OK;
}

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

template <class Fn>
Fn driver_fn(const char* name) {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<Fn>(p);
}

int dev_status(DevStatus* st) {
  uint32_t* w = nullptr;
  const int rc = status_words(&w);
  if (rc != LCB_OK) return rc;
  st->words = w;
  st->limit = g_wait_limit.load();
  return LCB_OK;
}

// Reads and clears the status word (synchronous).
int take_status(uint32_t* bits, uint32_t* where) {
  uint32_t w[4] = {0, 0, 0, 0};
  if (cudaMemcpyFromSymbol(w, g_status_words, sizeof(w)) != cudaSuccess) return LCB_ERR_CUDA;
  if (w[0] != 0) {
    const uint32_t z[4] = {0, 0, 0, 0};
    if (cudaMemcpyToSymbol(g_status_words, z, sizeof(z)) != cudaSuccess) return LCB_ERR_CUDA;
  }
  *bits = w[0];
  if (where) *where = w[1];
  return LCB_OK;
}

int finish(int rc, cudaStream_t stream) {
  if (rc != LCB_OK) return rc;
  if (!checked_mode()) return LCB_OK;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return LCB_ERR_CUDA;
  uint32_t bits = 0;
  if ((rc = take_status(&bits, nullptr)) != LCB_OK) return rc;
  return (bits & DEV_TIMEOUT) ? LCB_ERR_TIMEOUT : LCB_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool stride_ok(long long s) { return s >= 0 && (s % 8) == 0 && s < (1LL << 38); }

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(p);
  }();
  return fn;
}

}  // namespace

int make_tma_map_bf16(CUtensorMap* map, const RowView& v, int B, int rows, int HD, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return LCB_ERR_CUDA;
  const long long bstride = (B == 1) ? static_cast<long long>(rows) * v.row_stride : v.batch_stride;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(HD), static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(B)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(v.row_stride) * 2, static_cast<cuuint64_t>(bstride) * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v.ptr), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? LCB_OK : LCB_ERR_ARG;
}

unsigned long long current_context_id() {
  static const CtxGetCurrentFn get_cur = driver_fn<CtxGetCurrentFn>("cuCtxGetCurrent");
  static const CtxGetIdFn get_id = driver_fn<CtxGetIdFn>("cuCtxGetId");
  if (!get_cur || !get_id) return 0;
  CUcontext ctx = nullptr;
  unsigned long long id = 0;
  if (get_cur(&ctx) != CUDA_SUCCESS || ctx == nullptr || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
  return id;
}

int set_smem_limit_once(DeviceOnce& once, const void* kernel, int bytes) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return LCB_ERR_CUDA;
  return once.run(
      dev, current_context_id(),
      [&] {
        return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess
                   ? LCB_OK
                   : LCB_ERR_CUDA;
      },
      LCB_ERR_CUDA);
}

}  // namespace lcb

using namespace lcb;

extern "C" {

const char* attn_status_string(int status) {
  switch (status) {
    case LCB_OK: return "ok";
    case LCB_ERR_ARG: return "invalid argument";
    case LCB_ERR_UNSUPPORTED: return "unsupported configuration";
    case LCB_ERR_SCHEDULE: return "invalid zigzag schedule size";
    case LCB_ERR_CUDA: return "CUDA error";
    case LCB_ERR_TIMEOUT: return "device bounded wait expired";
    case LCB_ERR_SCRATCH: return "problem larger than the fixed scratch of attn_bwd_noalloc (B*H*S > 2^21)";
    default: return "unknown status";
  }
}

int lcb_version(void) { return 100; }

unsigned long long lcb_set_wait_limit_ns(unsigned long long ns) {
  if (ns == 0) ns = 1;
  return g_wait_limit.exchange(ns);
}

int lcb_take_device_status(unsigned int* where) {
  uint32_t bits = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return LCB_ERR_CUDA;
  const int rc = take_status(&bits, where);
  return rc != LCB_OK ? rc : static_cast<int>(bits);
}

// Checks the tensors shared by the tasks of a forward launch and fills `a`.
static int prep_fwd(FwdLaunch* a, const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                    int q_rows, int k_rows, int D, float scale, long long q_row_stride, long long q_batch_stride,
                    long long kv_row_stride, long long kv_batch_stride, long long o_row_stride,
                    long long o_batch_stride, long long lse_head_stride, long long lse_batch_stride) {
  if (B < 1 || H < 1 || q_rows < 0 || k_rows < 0) return LCB_ERR_ARG;
  if (D != kHeadDim) return LCB_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) return LCB_ERR_ARG;
  const long long HD = static_cast<long long>(H) * kHeadDim;
  if (q_rows > 0) {
    if (!o || !lse || !aligned16(o)) return LCB_ERR_ARG;
    if (!stride_ok(o_row_stride) || !stride_ok(o_batch_stride) || HD > o_row_stride) return LCB_ERR_ARG;
    if (lse_head_stride < 0 || lse_batch_stride < 0) return LCB_ERR_ARG;
  }
  if (q_rows > 0 && k_rows > 0) {
    if (!q || !k || !v || !aligned16(q) || !aligned16(k) || !aligned16(v)) return LCB_ERR_ARG;
    if (!stride_ok(q_row_stride) || !stride_ok(q_batch_stride) || !stride_ok(kv_row_stride) ||
        !stride_ok(kv_batch_stride))
      return LCB_ERR_ARG;
    if (HD > q_row_stride || HD > kv_row_stride) return LCB_ERR_ARG;
  }
  a->q = {q, q_row_stride, q_batch_stride};
  a->k = {k, kv_row_stride, kv_batch_stride};
  a->v = {v, kv_row_stride, kv_batch_stride};
  a->o = o;
  a->lse = lse;
  a->o_row_stride = o_row_stride;
  a->o_batch_stride = o_batch_stride;
  a->lse_head_stride = lse_head_stride;
  a->lse_batch_stride = lse_batch_stride;
  a->B = B;
  a->H = H;
  a->q_rows = q_rows;
  a->k_rows = k_rows;
  a->n_tasks = 0;
  a->scale = scale;
  return LCB_OK;
}

static int out_mode(int o_dtype) {
  return o_dtype == LCB_OUT_F32_MERGE ? 2 : (o_dtype == LCB_DTYPE_F32 ? 1 : (o_dtype == LCB_DTYPE_BF16 ? 0 : -1));
}

// Enqueues the tasks of `a` (already checked): rows of tasks without keys are
// filled with O = 0, LSE = -inf (or left alone in merge mode); the rest run as
// one launch, heaviest per-CTA work first.
static int run_fwd(FwdLaunch& a, const FwdTask* tasks, int n, cudaStream_t st) {
  FwdTask order[kMaxFwdTasks];
  int m = 0;
  for (int i = 0; i < n; ++i) {
    const FwdTask& t = tasks[i];
    if (t.q_len == 0) continue;
    if (t.k_len == 0) {
      if (t.o_mode == 2) continue;  // an empty block leaves the accumulator unchanged
      const size_t esz = t.o_mode == 1 ? 4 : 2;
      void* o_rows = static_cast<char*>(a.o) + static_cast<long long>(t.q_off) * a.o_row_stride * esz;
      const int rc = launch_fill_empty(o_rows, t.o_mode == 1, a.o_row_stride, a.o_batch_stride, a.lse + t.q_off,
                                       a.lse_head_stride, a.lse_batch_stride, a.B, a.H, t.q_len, st);
      if (rc != LCB_OK) return rc;
      continue;
    }
    order[m++] = t;
  }
  if (m == 0) return LCB_OK;
  const int rc = dev_status(&a.st);
  if (rc != LCB_OK) return rc;
  auto weight = [](const FwdTask& t) { return t.causal ? t.q_len : t.k_len; };  // key tiles of the longest CTA
  std::stable_sort(order, order + m, [&](const FwdTask& x, const FwdTask& y) { return weight(x) > weight(y); });
  for (int i = 0; i < m; ++i) a.tasks[i] = order[i];
  a.n_tasks = m;
  return launch_attn_fwd(a, st);
}

int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq, int Sk,
                int D, int causal, float scale, long long q_row_stride, long long q_batch_stride,
                long long kv_row_stride, long long kv_batch_stride, long long o_row_stride,
                long long o_batch_stride, int o_dtype, long long lse_head_stride, long long lse_batch_stride,
                void* stream) {
  if (causal != 0 && causal != 1) return LCB_ERR_ARG;
  if (causal && Sq != Sk) return LCB_ERR_UNSUPPORTED;
  const int mode = out_mode(o_dtype);
  if (mode < 0) return LCB_ERR_UNSUPPORTED;
  FwdLaunch a;
  int rc = prep_fwd(&a, q, k, v, o, lse, B, H, Sq, Sk, D, scale, q_row_stride, q_batch_stride, kv_row_stride,
                    kv_batch_stride, o_row_stride, o_batch_stride, lse_head_stride, lse_batch_stride);
  if (rc != LCB_OK) return rc;
  if (Sq == 0) return LCB_OK;
  const FwdTask t = {0, Sq, 0, Sk, causal, mode};
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(run_fwd(a, &t, 1, st), st);
}

int attn_fwd_group(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int q_rows,
                   int k_rows, int D, float scale, long long q_row_stride, long long q_batch_stride,
                   long long kv_row_stride, long long kv_batch_stride, long long o_row_stride,
                   long long o_batch_stride, long long lse_head_stride, long long lse_batch_stride,
                   const lcb_fwd_task* tasks, int n_tasks, void* stream) {
  if (n_tasks < 0 || n_tasks > kMaxFwdTasks || (n_tasks > 0 && !tasks)) return LCB_ERR_ARG;
  FwdLaunch a;
  int rc = prep_fwd(&a, q, k, v, o, lse, B, H, q_rows, k_rows, D, scale, q_row_stride, q_batch_stride,
                    kv_row_stride, kv_batch_stride, o_row_stride, o_batch_stride, lse_head_stride, lse_batch_stride);
  if (rc != LCB_OK) return rc;
  FwdTask t[kMaxFwdTasks];
  int bf16_out = -1;  // all tasks write one output tensor: bf16, or fp32 (stored or merged)
  for (int i = 0; i < n_tasks; ++i) {
    const lcb_fwd_task& x = tasks[i];
    const int mode = out_mode(x.o_dtype);
    if (mode < 0) return LCB_ERR_UNSUPPORTED;
    if (bf16_out >= 0 && bf16_out != (mode == 0)) return LCB_ERR_ARG;
    bf16_out = mode == 0;
    if (x.causal != 0 && x.causal != 1) return LCB_ERR_ARG;
    if (x.causal && x.q_len != x.k_len) return LCB_ERR_UNSUPPORTED;
    if (x.q_off < 0 || x.q_len < 0 || x.k_off < 0 || x.k_len < 0) return LCB_ERR_ARG;
    if (static_cast<long long>(x.q_off) + x.q_len > q_rows || static_cast<long long>(x.k_off) + x.k_len > k_rows)
      return LCB_ERR_ARG;
    for (int j = 0; j < i; ++j) {  // query ranges must not overlap: each task owns its output rows
      const lcb_fwd_task& y = tasks[j];
      if (x.q_len > 0 && y.q_len > 0 && x.q_off < y.q_off + y.q_len && y.q_off < x.q_off + x.q_len)
        return LCB_ERR_ARG;
    }
    t[i] = {x.q_off, x.q_len, x.k_off, x.k_len, x.causal, mode};
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(run_fwd(a, t, n_tasks, st), st);
}

int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int S, int D,
             int causal, float scale, void* stream) {
  const long long rs = static_cast<long long>(H) * D;
  const long long bs = rs * S;
  return attn_fwd_ex(q, k, v, o, lse, B, H, S, S, D, causal, scale, rs, bs, rs, bs, rs, bs, LCB_DTYPE_BF16, S,
                     static_cast<long long>(H) * S, stream);
}

// Workspace of attn_bwd: Delta [B, H, S] fp32, then the fused pass's tiled
// fp32 dQ accumulator (B * H * ceil(S / 128) tiles of 128 x 128), each at a
// 256-byte boundary.
static size_t delta_bytes(int B, int H, int S) {
  const size_t n = static_cast<size_t>(B) * H * S * sizeof(float);
  return (n + 255) & ~static_cast<size_t>(255);
}
static long long dq_tiles(int S) { return (S + 127) / 128; }
constexpr long long kDqTileFloats = 128LL * 128;

size_t attn_bwd_workspace_bytes(int B, int H, int S, int D) {
  if (B < 1 || H < 1 || S < 0 || D != kHeadDim) return 0;
  return delta_bytes(B, H, S) + static_cast<size_t>(B) * H * dq_tiles(S) * kDqTileFloats * sizeof(float);
}

int attn_bwd_preprocess(const void* o, const void* dO, float* delta, int B, int H, int S, int D,
                        long long row_stride, long long batch_stride, long long delta_head_stride,
                        long long delta_batch_stride, void* stream) {
  if (B < 1 || H < 1 || S < 0) return LCB_ERR_ARG;
  if (D != kHeadDim) return LCB_ERR_UNSUPPORTED;
  if (S == 0) return LCB_OK;
  if (!o || !dO || !delta || (reinterpret_cast<uintptr_t>(o) & 7u) || (reinterpret_cast<uintptr_t>(dO) & 7u))
    return LCB_ERR_ARG;
  if (row_stride < static_cast<long long>(H) * D || (row_stride % 4) || batch_stride < 0 || (batch_stride % 4))
    return LCB_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_bwd_preprocess(o, dO, row_stride, batch_stride, delta, delta_head_stride, delta_batch_stride, B,
                                      H, S, st),
                st);
}

// Validates the arguments shared by the block-backward entry points and fills `a`.
static int prep_bwd(BwdLaunch* a, const void* q, const void* k, const void* v, const float* lse, const float* delta,
                    const void* dO, void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, int causal,
                    float scale, long long q_row_stride, long long q_batch_stride, long long kv_row_stride,
                    long long kv_batch_stride, long long lse_head_stride, long long lse_batch_stride, int grad_mode,
                    long long dq_row_stride, long long dq_batch_stride, long long dkv_row_stride,
                    long long dkv_batch_stride) {
  if (B < 1 || H < 1 || Sq < 0 || Sk < 0) return LCB_ERR_ARG;
  if (D != kHeadDim) return LCB_ERR_UNSUPPORTED;
  if (causal != 0 && causal != 1) return LCB_ERR_ARG;
  if (causal && Sq != Sk) return LCB_ERR_UNSUPPORTED;
  if (grad_mode != LCB_GRAD_BF16 && grad_mode != LCB_GRAD_F32_ACCUM && grad_mode != LCB_GRAD_F32_STORE)
    return LCB_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !std::isfinite(scale)) return LCB_ERR_ARG;
  // Operands of an empty side (Sq == 0: q, dO, lse, delta, dq; Sk == 0: k, v, dk, dv) may be NULL.
  if (Sq > 0 && (!q || !lse || !delta || !dO || !dq)) return LCB_ERR_ARG;
  if (Sk > 0 && (!k || !v || !dk || !dv)) return LCB_ERR_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dO) || !aligned16(dq) || !aligned16(dk) ||
      !aligned16(dv))
    return LCB_ERR_ARG;
  if (!stride_ok(q_row_stride) || !stride_ok(q_batch_stride) || !stride_ok(kv_row_stride) ||
      !stride_ok(kv_batch_stride) || !stride_ok(dq_row_stride) || !stride_ok(dq_batch_stride) ||
      !stride_ok(dkv_row_stride) || !stride_ok(dkv_batch_stride))
    return LCB_ERR_ARG;
  const long long HD = static_cast<long long>(H) * kHeadDim;
  if (HD > q_row_stride || HD > kv_row_stride || HD > dq_row_stride || HD > dkv_row_stride) return LCB_ERR_ARG;
  if (lse_head_stride < 0 || lse_batch_stride < 0) return LCB_ERR_ARG;
  a->q = {q, q_row_stride, q_batch_stride};
  a->dO = {dO, q_row_stride, q_batch_stride};
  a->k = {k, kv_row_stride, kv_batch_stride};
  a->v = {v, kv_row_stride, kv_batch_stride};
  a->lse = lse;
  a->delta = delta;
  a->lse_head_stride = lse_head_stride;
  a->lse_batch_stride = lse_batch_stride;
  a->dq = dq;
  a->dk = dk;
  a->dv = dv;
  a->dq_row_stride = dq_row_stride;
  a->dq_batch_stride = dq_batch_stride;
  a->dkv_row_stride = dkv_row_stride;
  a->dkv_batch_stride = dkv_batch_stride;
  a->B = B;
  a->H = H;
  a->Sq = Sq;
  a->Sk = Sk;
  a->causal = causal;
  a->grad_mode = grad_mode;
  a->scale = scale;
  return dev_status(&a->st);
}

#define LCB_BWD_EX_ARGS                                                                                           \
  q, k, v, lse, delta, dO, dq, dk, dv, B, H, Sq, Sk, D, causal, scale, q_row_stride, q_batch_stride, kv_row_stride, \
      kv_batch_stride, lse_head_stride, lse_batch_stride, grad_mode, dq_row_stride, dq_batch_stride, dkv_row_stride,   \
      dkv_batch_stride

int attn_bwd_dkdv_ex(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                     const void* dO, void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, int causal,
                     float scale, long long q_row_stride, long long q_batch_stride, long long kv_row_stride,
                     long long kv_batch_stride, long long lse_head_stride, long long lse_batch_stride,
                     int grad_mode, long long dq_row_stride, long long dq_batch_stride, long long dkv_row_stride,
                     long long dkv_batch_stride, void* stream) {
  BwdLaunch a;
  int rc = prep_bwd(&a, LCB_BWD_EX_ARGS);
  if (rc != LCB_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_attn_bwd_dkdv(a, st), st);
}

int attn_bwd_dq_ex(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, int causal,
                   float scale, long long q_row_stride, long long q_batch_stride, long long kv_row_stride,
                   long long kv_batch_stride, long long lse_head_stride, long long lse_batch_stride, int grad_mode,
                   long long dq_row_stride, long long dq_batch_stride, long long dkv_row_stride,
                   long long dkv_batch_stride, void* stream) {
  BwdLaunch a;
  int rc = prep_bwd(&a, LCB_BWD_EX_ARGS);
  if (rc != LCB_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_attn_bwd_dq(a, st), st);
}

int attn_bwd_fused_ex(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                      const void* dO, float* dq_tiles, void* dk, void* dv, int B, int H, int Sq, int Sk, int D,
                      int causal, float scale, long long q_row_stride, long long q_batch_stride,
                      long long kv_row_stride, long long kv_batch_stride, long long lse_head_stride,
                      long long lse_batch_stride, int grad_mode, long long dq_tile_head_stride,
                      long long dq_tile_batch_stride, long long dkv_row_stride, long long dkv_batch_stride,
                      void* stream) {
  const lcb_bwd_task t = {0, Sq, 0, Sk, causal};
  return attn_bwd_fused_group(q, k, v, lse, delta, dO, dq_tiles, dk, dv, B, H, Sq, Sk, D, scale, q_row_stride,
                              q_batch_stride, kv_row_stride, kv_batch_stride, lse_head_stride, lse_batch_stride,
                              grad_mode, dq_tile_head_stride, dq_tile_batch_stride, dkv_row_stride,
                              dkv_batch_stride, &t, 1, stream);
}

int attn_bwd_fused_group(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                         const void* dO, float* dq_tiles, void* dk, void* dv, int B, int H, int q_rows, int k_rows,
                         int D, float scale, long long q_row_stride, long long q_batch_stride,
                         long long kv_row_stride, long long kv_batch_stride, long long lse_head_stride,
                         long long lse_batch_stride, int grad_mode, long long dq_tile_head_stride,
                         long long dq_tile_batch_stride, long long dkv_row_stride, long long dkv_batch_stride,
                         const lcb_bwd_task* tasks, int n_tasks, void* stream) {
  if (n_tasks < 0 || n_tasks > kMaxBwdTasks || (n_tasks > 0 && !tasks)) return LCB_ERR_ARG;
  // The accumulator is checked here; prep_bwd sees row strides that always pass.
  if (dq_tile_head_stride < 0 || dq_tile_batch_stride < 0 || (dq_tile_head_stride % 4) ||
      (dq_tile_batch_stride % 4))
    return LCB_ERR_ARG;
  void* dq = dq_tiles;
  const int Sq = q_rows, Sk = k_rows, causal = 0;  // shared tensors; causality is per task
  const long long HD = static_cast<long long>(H) * kHeadDim;
  const long long dq_row_stride = HD, dq_batch_stride = HD * Sq;
  if (q_rows < 0 || k_rows < 0) return LCB_ERR_ARG;
  for (int i = 0; i < n_tasks; ++i) {
    const lcb_bwd_task& x = tasks[i];
    if (x.causal != 0 && x.causal != 1) return LCB_ERR_ARG;
    if (x.causal && x.q_len != x.k_len) return LCB_ERR_UNSUPPORTED;
    if (x.q_off < 0 || x.q_len < 0 || x.k_off < 0 || x.k_len < 0 || (x.q_off % 128)) return LCB_ERR_ARG;
    if (static_cast<long long>(x.q_off) + x.q_len > q_rows || static_cast<long long>(x.k_off) + x.k_len > k_rows)
      return LCB_ERR_ARG;
    for (int j = 0; j < i; ++j) {  // key ranges must not overlap: each task owns its dK/dV rows
      const lcb_bwd_task& y = tasks[j];
      if (x.k_len > 0 && y.k_len > 0 && x.k_off < y.k_off + y.k_len && y.k_off < x.k_off + x.k_len)
        return LCB_ERR_ARG;
    }
  }
  BwdLaunch a;
  int rc = prep_bwd(&a, LCB_BWD_EX_ARGS);
  if (rc != LCB_OK) return rc;
  a.dq_row_stride = dq_tile_head_stride;
  a.dq_batch_stride = dq_tile_batch_stride;
  BwdTask order[kMaxBwdTasks];
  int m = 0;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  for (int i = 0; i < n_tasks; ++i) {
    const lcb_bwd_task& x = tasks[i];
    if (x.k_len == 0) continue;
    if (x.q_len == 0) {  // no queries: dK = dV = 0 (overwrite modes), nothing added to dQ
      if (grad_mode == LCB_GRAD_F32_ACCUM) continue;
      const size_t esz = grad_mode == LCB_GRAD_BF16 ? 2 : 4;
      for (int g = 0; g < 2; ++g) {
        char* base = static_cast<char*>(g ? dv : dk) + static_cast<long long>(x.k_off) * dkv_row_stride * esz;
        for (int b = 0; b < B; ++b) {
          if (cudaMemset2DAsync(base + b * dkv_batch_stride * esz, dkv_row_stride * esz, 0, HD * esz, x.k_len, st) !=
              cudaSuccess)
            return LCB_ERR_CUDA;
        }
      }
      continue;
    }
    order[m++] = {x.q_off, x.q_len, x.k_off, x.k_len, x.causal};
  }
  if (m == 0) return finish(LCB_OK, st);
  auto weight = [](const BwdTask& t) { return t.q_len; };  // query tiles of the longest CTA
  std::stable_sort(order, order + m, [&](const BwdTask& x, const BwdTask& y) { return weight(x) > weight(y); });
  return finish(launch_attn_bwd_fused(a, order, m, q_rows, k_rows, st), st);
}

int lcb_dq_tiles_zero(float* dq_tiles, long long n_floats, void* stream) {
  if (n_floats < 0) return LCB_ERR_ARG;
  if (n_floats == 0) return LCB_OK;
  if (!dq_tiles || !aligned16(dq_tiles)) return LCB_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(dq_tiles, 0, static_cast<size_t>(n_floats) * sizeof(float), st) != cudaSuccess)
    return LCB_ERR_CUDA;
  return finish(LCB_OK, st);
}

int lcb_dq_untile(const float* dq_tiles, long long tile_head_stride, long long tile_batch_stride, void* dq,
                  long long row_stride, long long batch_stride, int B, int H, int S, void* stream) {
  if (B < 1 || H < 1 || S < 0) return LCB_ERR_ARG;
  if (S == 0) return LCB_OK;
  if (!dq_tiles || !dq || !aligned16(dq_tiles) || (reinterpret_cast<uintptr_t>(dq) & 7u)) return LCB_ERR_ARG;
  if (tile_head_stride < 0 || tile_batch_stride < 0 || (tile_head_stride % 4) || (tile_batch_stride % 4))
    return LCB_ERR_ARG;
  if (row_stride < static_cast<long long>(H) * kHeadDim || (row_stride % 4) || batch_stride < 0 ||
      (batch_stride % 4))
    return LCB_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_dq_untile(dq_tiles, tile_head_stride, tile_batch_stride, dq, row_stride, batch_stride, B, H,
                                 S, st),
                st);
}

int attn_bwd_ex(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                const void* dO, void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, int causal,
                float scale, long long q_row_stride, long long q_batch_stride, long long kv_row_stride,
                long long kv_batch_stride, long long lse_head_stride, long long lse_batch_stride, int grad_mode,
                long long dq_row_stride, long long dq_batch_stride, long long dkv_row_stride,
                long long dkv_batch_stride, void* stream) {
  BwdLaunch a;
  int rc = prep_bwd(&a, LCB_BWD_EX_ARGS);
  if (rc != LCB_OK) return rc;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((rc = launch_attn_bwd_dkdv(a, st)) != LCB_OK) return rc;
  if ((rc = launch_attn_bwd_dq(a, st)) != LCB_OK) return rc;
  return finish(LCB_OK, st);
}

int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
             void* dq, void* dk, void* dv, int B, int H, int S, int D, int causal, float scale, void* workspace,
             size_t ws_bytes, void* stream) {
  if (B < 1 || H < 1 || S < 0) return LCB_ERR_ARG;
  if (D != kHeadDim) return LCB_ERR_UNSUPPORTED;
  if (S == 0) return LCB_OK;
  if (!workspace || !aligned16(workspace) || ws_bytes < attn_bwd_workspace_bytes(B, H, S, D)) return LCB_ERR_ARG;
  if (!dq || !aligned16(dq)) return LCB_ERR_ARG;
  const long long rs = static_cast<long long>(H) * D;
  const long long bs = rs * S;
  float* delta = static_cast<float*>(workspace);
  float* dq_acc = reinterpret_cast<float*>(static_cast<char*>(workspace) + delta_bytes(B, H, S));
  const long long tile_hs = dq_tiles(S) * kDqTileFloats, tile_bs = tile_hs * H;
  int rc = attn_bwd_preprocess(o, dO, delta, B, H, S, D, rs, bs, S, static_cast<long long>(H) * S, stream);
  if (rc != LCB_OK) return rc;
  if ((rc = lcb_dq_tiles_zero(dq_acc, tile_bs * B, stream)) != LCB_OK) return rc;
  rc = attn_bwd_fused_ex(q, k, v, lse, delta, dO, dq_acc, dk, dv, B, H, S, S, D, causal, scale, rs, bs, rs, bs, S,
                         static_cast<long long>(H) * S, LCB_GRAD_BF16, tile_hs, tile_bs, rs, bs, stream);
  if (rc != LCB_OK) return rc;
  return lcb_dq_untile(dq_acc, tile_hs, tile_bs, dq, rs, bs, B, H, S, stream);
}

int attn_lse_merge(float* o_acc, float* lse_acc, const void* o_b, const float* lse_b, int o_b_dtype,
                   void* o_out_bf16, int B, int H, int rows, int D, long long o_row_stride, long long o_batch_stride,
                   long long ob_row_stride, long long ob_batch_stride, long long lse_head_stride,
                   long long lse_batch_stride, long long lseb_head_stride, long long lseb_batch_stride,
                   void* stream) {
  if (B < 1 || H < 1 || rows < 0) return LCB_ERR_ARG;
  if (D != kHeadDim) return LCB_ERR_UNSUPPORTED;
  if (o_b_dtype != LCB_DTYPE_BF16 && o_b_dtype != LCB_DTYPE_F32) return LCB_ERR_UNSUPPORTED;
  if (rows == 0) return LCB_OK;
  if (!o_acc || !lse_acc || !o_b || !lse_b || !aligned16(o_acc) || !aligned16(o_b)) return LCB_ERR_ARG;
  if (o_out_bf16 && !aligned16(o_out_bf16)) return LCB_ERR_ARG;
  const long long HD = static_cast<long long>(H) * D;
  if (!stride_ok(o_row_stride) || !stride_ok(o_batch_stride) || o_row_stride < HD) return LCB_ERR_ARG;
  if (!stride_ok(ob_row_stride) || !stride_ok(ob_batch_stride) || ob_row_stride < HD) return LCB_ERR_ARG;
  if (lse_head_stride < 0 || lse_batch_stride < 0 || lseb_head_stride < 0 || lseb_batch_stride < 0)
    return LCB_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_lse_merge(o_acc, lse_acc, o_b, o_b_dtype == LCB_DTYPE_F32, lse_b, o_out_bf16, B, H, rows,
                                 o_row_stride, o_batch_stride, ob_row_stride, ob_batch_stride, lse_head_stride,
                                 lse_batch_stride, lseb_head_stride, lseb_batch_stride, st),
                st);
}

int zigzag_schedule(int S, int P, int* perm, lcb_task* tasks) {
  if (P < 1 || S < 2 * P || S % (2 * P) != 0) return LCB_ERR_SCHEDULE;
  const int c = S / (2 * P);
  if (perm) {
    for (int r = 0; r < P; ++r) {
      const int early = r, late = 2 * P - 1 - r;
      for (int t = 0; t < c; ++t) {
        perm[r * 2 * c + t] = early * c + t;
        perm[r * 2 * c + c + t] = late * c + t;
      }
    }
  }
  if (tasks) {
    for (int r = 0; r < P; ++r) {
      for (int s = 0; s < P; ++s) {
        const int src = ((r - s) % P + P) % P;
        lcb_task t;
        t.rank = r;
        t.step = s;
        t.src = src;
        if (s == 0) {
          t.kind = LCB_TASK_DIAG;
          t.q_off = r * 2 * c;
          t.q_len = 2 * c;
          t.k_off = r * 2 * c;
          t.k_len = 2 * c;
          t.causal = 1;
        } else if (src < r) {
          t.kind = LCB_TASK_LOWER;
          t.q_off = r * 2 * c;
          t.q_len = 2 * c;
          t.k_off = src * 2 * c;
          t.k_len = c;
          t.causal = 0;
        } else {
          t.kind = LCB_TASK_UPPER;
          t.q_off = r * 2 * c + c;
          t.q_len = c;
          t.k_off = src * 2 * c;
          t.k_len = 2 * c;
          t.causal = 0;
        }
        tasks[r * P + s] = t;
      }
    }
  }
  return LCB_OK;
}

int ring_schedule(int S, int P, int* perm, lcb_task* tasks) {
  if (P < 1 || S < P || S % P != 0) return LCB_ERR_SCHEDULE;
  const int n = S / P;
  if (perm) {
    for (int i = 0; i < S; ++i) perm[i] = i;
  }
  if (tasks) {
    for (int r = 0; r < P; ++r) {
      for (int s = 0; s < P; ++s) {
        const int src = ((r - s) % P + P) % P;
        lcb_task t;
        t.rank = r;
        t.step = s;
        t.src = src;
        t.q_off = r * n;
        t.k_off = src * n;
        if (s == 0) {
          t.kind = LCB_TASK_DIAG;
          t.q_len = n;
          t.k_len = n;
          t.causal = 1;
        } else if (src < r) {
          t.kind = LCB_TASK_FULL;
          t.q_len = n;
          t.k_len = n;
          t.causal = 0;
        } else {  // every key of a later rank follows every local query
          t.kind = LCB_TASK_NONE;
          t.q_len = 0;
          t.k_len = 0;
          t.causal = 0;
        }
        tasks[r * P + s] = t;
      }
    }
  }
  return LCB_OK;
}

static int permute_common(const void* src, void* dst, const int* perm, int rows, long long row_bytes, int scatter,
                          void* stream) {
  if (rows < 0 || row_bytes <= 0 || (row_bytes % 16)) return LCB_ERR_ARG;
  if (rows == 0) return LCB_OK;
  if (!src || !dst || !perm || src == dst || !aligned16(src) || !aligned16(dst)) return LCB_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_permute_rows(src, dst, perm, rows, row_bytes, scatter, st), st);
}

int lcb_permute_rows(const void* src, void* dst, const int* perm, int rows, long long row_bytes, void* stream) {
  return permute_common(src, dst, perm, rows, row_bytes, 0, stream);
}

int lcb_scatter_rows(const void* src, void* dst, const int* perm, int rows, long long row_bytes, void* stream) {
  return permute_common(src, dst, perm, rows, row_bytes, 1, stream);
}

int lcb_ulysses_all_to_all(const void* src, void* dst, int B, int S, int H, int D, int P, int elem_bytes,
                           int direction, void* stream) {
  if (B < 1 || H < 1 || S < 0 || D < 1 || P < 1) return LCB_ERR_ARG;
  if (H % P != 0 || S % P != 0) return LCB_ERR_ARG;
  if (elem_bytes != 2 && elem_bytes != 4) return LCB_ERR_UNSUPPORTED;
  if (direction != LCB_ULYSSES_SEQ_TO_HEAD && direction != LCB_ULYSSES_HEAD_TO_SEQ) return LCB_ERR_ARG;
  const long long block_bytes = static_cast<long long>(H / P) * D * elem_bytes;
  if (block_bytes % 16 != 0) return LCB_ERR_ARG;
  if (S == 0) return LCB_OK;
  if (!src || !dst || src == dst || !aligned16(src) || !aligned16(dst)) return LCB_ERR_ARG;
  const long long rows = static_cast<long long>(B) * S;
  const long long bv = block_bytes / 16;
  const long long total = rows * bv * P;  // vectors in the tensor
  const char* s0 = static_cast<const char*>(src);
  const char* d0 = static_cast<const char*>(dst);
  if (s0 < d0 + total * 16 && d0 < s0 + total * 16) return LCB_ERR_ARG;  // overlapping buffers
  if (rows * bv >= (1LL << 31)) return LCB_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_ulysses_a2a(src, dst, rows, bv, P, direction, st), st);
}

int lcb_cast_f32_bf16(const float* src, void* dst, long long n, void* stream) {
  if (n < 0) return LCB_ERR_ARG;
  if (n == 0) return LCB_OK;
  if (!src || !dst || !aligned16(src) || !aligned16(dst)) return LCB_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_cast_f32_bf16(src, dst, n, st), st);
}

int lcb_cross_entropy(void* logits, const long long* labels, float* loss, float* lse, const float* dloss, int N,
                      int V, long long row_stride, int ignore_index, int mode, void* stream) {
  if (N < 0 || V < 1 || row_stride < V) return LCB_ERR_ARG;
  if (mode != LCB_CE_FWD && mode != LCB_CE_FWD_BWD && mode != LCB_CE_BWD) return LCB_ERR_UNSUPPORTED;
  if (N == 0) return LCB_OK;
  if (!logits || !labels || !lse || (reinterpret_cast<uintptr_t>(logits) & 1u)) return LCB_ERR_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_cross_entropy(logits, labels, loss, lse, dloss, N, V, row_stride, ignore_index, mode, st), st);
}

int lcb_rope(const void* x, void* y, int B, int S, int H, int D, double theta, long long pos0, int inverse,
             long long row_stride, long long batch_stride, void* stream) {
  if (B < 1 || H < 1 || S < 0) return LCB_ERR_ARG;
  if (D != kHeadDim) return LCB_ERR_UNSUPPORTED;
  if (!(theta > 0.0) || !std::isfinite(theta) || (inverse != 0 && inverse != 1)) return LCB_ERR_ARG;
  if (pos0 < 0 || pos0 + S > (1LL << 40)) return LCB_ERR_ARG;
  if (S == 0) return LCB_OK;
  if (!x || !y || (reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u)) return LCB_ERR_ARG;
  if (row_stride < static_cast<long long>(H) * D || (row_stride % 2) || batch_stride < 0 || (batch_stride % 2))
    return LCB_ERR_ARG;
  RopeFreqs fr;
  for (int k = 0; k < D / 2; ++k) fr.f[k] = std::pow(theta, -2.0 * k / D);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  return finish(launch_rope(x, y, B, S, H, row_stride, batch_stride, pos0, inverse, fr, st), st);
}

int lcb_selftest_bounded_wait(void* stream) {
  DevStatus st;
  int rc = dev_status(&st);
  if (rc != LCB_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if ((rc = launch_wait_selftest(st, s)) != LCB_OK) return rc;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LCB_ERR_CUDA;
  uint32_t bits = 0;
  if ((rc = take_status(&bits, nullptr)) != LCB_OK) return rc;
  return (bits & DEV_TIMEOUT) ? LCB_ERR_TIMEOUT : LCB_OK;
}

}  // extern "C"
