// Host-side plumbing shared by the C-ABI layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "device_once.h"

namespace lcb {

// A [B, rows, H, D] bf16/fp32 view: element (b, s, h, d) lives at
// base + b * batch_stride + s * row_stride + h * D + d (strides in elements).
struct RowView {
  const void* ptr;
  long long row_stride;
  long long batch_stride;
};

// Builds a 3-D TMA map over a bf16 [B, rows, H*D] view with a box of
// 64 (inner, 128 bytes) x box_rows x 1 and 128-byte swizzle.
// Returns 0 on success, a negative LCB status on failure.
int make_tma_map_bf16(CUtensorMap* map, const RowView& v, int B, int rows, int HD, int box_rows);

// Id of the calling thread's current CUDA context (unique within the process),
// or 0 when there is none or the driver cannot tell.
unsigned long long current_context_id();

// Raises `kernel`'s dynamic shared-memory limit to `bytes` in the current
// device's context, the first time it is asked for that context (function
// attributes belong to a device context). Returns 0, or LCB_ERR_CUDA.
int set_smem_limit_once(DeviceOnce& once, const void* kernel, int bytes);

// One block of a forward launch (rows relative to the shared tensors).
struct FwdTask {
  int q_off, q_len, k_off, k_len, causal, o_mode;  // o_mode: 0 bf16, 1 fp32, 2 merge into fp32 (O, LSE)
};
constexpr int kMaxFwdTasks = 16;

// q/o/lse views hold q_rows rows, k/v views k_rows; every task has k_len > 0,
// tasks are ordered heaviest first and their query ranges do not overlap.
struct FwdLaunch {
  RowView q, k, v;
  void* o;
  float* lse;
  long long o_row_stride, o_batch_stride;
  long long lse_head_stride, lse_batch_stride;
  int B, H, q_rows, k_rows;
  int n_tasks;
  FwdTask tasks[kMaxFwdTasks];
  float scale;
  DevStatus st;
};
int launch_attn_fwd(const FwdLaunch& a, cudaStream_t stream);

struct BwdLaunch {
  RowView q, k, v, dO;
  const float* lse;
  const float* delta;
  long long lse_head_stride, lse_batch_stride;  // also used for delta
  void* dq;
  void* dk;
  void* dv;
  long long dq_row_stride, dq_batch_stride;    // in elements of the gradient dtype
  long long dkv_row_stride, dkv_batch_stride;
  int B, H, Sq, Sk, causal, grad_mode;  // LCB_GRAD_*
  float scale;
  DevStatus st;
};
int launch_attn_bwd_dkdv(const BwdLaunch& a, cudaStream_t stream);
int launch_attn_bwd_dq(const BwdLaunch& a, cudaStream_t stream);
// One block of a one-pass backward launch (rows relative to the shared tensors;
// q_off a multiple of 128, the dQ accumulator's tile height).
struct BwdTask {
  int q_off, q_len, k_off, k_len, causal;
};
constexpr int kMaxBwdTasks = 16;
// One pass over the tasks in one launch (blocks without queries or keys are
// skipped): dK/dV as a.grad_mode says; dQ is added into the tiled fp32
// accumulator a.dq (a.dq_row_stride / a.dq_batch_stride carry its tile head /
// batch strides in floats). The q/dO views hold q_rows rows, k/v/dk/dv k_rows;
// tasks are ordered longest rows first and their key ranges do not overlap.
int launch_attn_bwd_fused(const BwdLaunch& a, const BwdTask* tasks, int n_tasks, int q_rows, int k_rows,
                          cudaStream_t stream);
// Tiled fp32 dQ accumulator -> bf16 [B, S, H, D] rows (strides in elements).
int launch_dq_untile(const float* acc, long long tile_hs, long long tile_bs, void* dq, long long rs, long long bs,
                     int B, int H, int S, cudaStream_t stream);

int launch_bwd_preprocess(const void* o, const void* dO, long long row_stride, long long batch_stride, float* delta,
                          long long d_head_stride, long long d_batch_stride, int B, int H, int S, cudaStream_t stream);

int launch_lse_merge(float* o_acc, float* lse_acc, const void* o_b, int o_b_f32, const float* lse_b, void* o_out_bf16,
                     int B, int H, int rows, long long o_row_stride, long long o_batch_stride,
                     long long ob_row_stride, long long ob_batch_stride, long long lse_head_stride,
                     long long lse_batch_stride, long long lseb_head_stride, long long lseb_batch_stride,
                     cudaStream_t stream);

int launch_permute_rows(const void* src, void* dst, const int* perm, int rows, long long row_bytes, int scatter,
                        cudaStream_t stream);

int launch_fill_empty(void* o, int o_f32, long long o_row_stride, long long o_batch_stride, float* lse,
                      long long lse_head_stride, long long lse_batch_stride, int B, int H, int rows,
                      cudaStream_t stream);

int launch_wait_selftest(DevStatus st, cudaStream_t stream);

// Ulysses all-to-all over 16-byte vectors: rows = B * S rows of P blocks of bv
// vectors; dir 0 sequence -> head layout, 1 head -> sequence layout.
int launch_ulysses_a2a(const void* src, void* dst, long long rows, long long bv, int P, int dir,
                       cudaStream_t stream);

int launch_cast_f32_bf16(const float* src, void* dst, long long n, cudaStream_t stream);

// Cross-entropy over rows of bf16 logits streamed through registers (mode LCB_CE_*).
int launch_cross_entropy(void* logits, const long long* labels, float* loss, float* lse, const float* dloss, int N,
                         int V, long long row_stride, int ignore_index, int mode, cudaStream_t stream);

// RoPE frequencies f_k = theta^(-2k/128), k < 64, computed on the host in fp64.
struct RopeFreqs {
  double f[64];
};
// y = RoPE(x) (inverse: the transpose) on bf16 [B, S, H, 128] views sharing strides.
int launch_rope(const void* x, void* y, int B, int S, int H, long long row_stride, long long batch_stride,
                long long pos0, int inverse, const RopeFreqs& fr, cudaStream_t stream);

}  // namespace lcb
