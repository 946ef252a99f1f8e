/*
 * lcb_attn.h — C ABI of the blockwise causal attention library (libattn.so).
 *
 * Exact softmax attention, forward and backward, computed tile by tile with an
 * online softmax on GB300 (sm_103a) tensor cores, plus the two pieces that
 * ring and zigzag-ring sequence parallelism add on top of it: merging partial
 * results by log-sum-exp and the zigzag split/schedule.
 *
 * Sources (web pages on EasyContext, cited by title and section):
 *  [FA]  "EasyContext核心技术解析：序列并行与Flash Attention的完美结合",
 *        §2 "Flash Attention优化": exact attention computed in blocks with
 *        recomputation, never storing the full score matrix; the block
 *        forward/backward entry points of Flash Attention.
 *  [SP]  same page, §1 "序列并行技术": ring attention over sequence shards.
 *  [ZZ]  "EasyContext代码解析200行核心训练脚本实现原理", §模型并行策略解析
 *        (zigzag_ring_attn) and §训练循环核心逻辑 (prepare_seq_parallel_inputs
 *        splits each sequence into rank-local pieces).
 *  [FULL] "EasyContext：用最少资源扩展大模型至百万Token": full attention.
 *  [ZO]  "EasyContext内存优化秘籍DeepSpeed Zero3卸载策略详解",
 *        §进阶优化与其他技术结合 (the fused cross-entropy loss with an
 *        in-place backward; the raised RoPE base) and §训练脚本配置
 *        (--rope-theta 1000000).
 *
 * Beyond attention: the rotary position embedding with a raised base that
 * long-context training puts on Q and K ([FA] §3 "RoPE扩展技术", [ZO]) and
 * the cross-entropy loss head ([ZO]).
 *
 * Conventions shared by every entry point
 *  - Tensors Q, K, V, O, dO, dQ, dK, dV are [B, S, H, D] (token-major, heads
 *    interleaved in a row), bf16 unless stated; D must be 128. LSE and Delta
 *    are fp32 [B, H, S].
 *  - LSE is the natural log of sum_j exp(scale * q . k_j) over visible keys
 *    (scale included); -inf for a row with no visible key.
 *  - causal: key j is visible to query i iff j <= i (requires Sq == Sk).
 *  - All tensor pointers are DEVICE pointers owned by the caller; the library
 *    keeps no pointer after a call returns and allocates nothing.
 *  - stream is a cudaStream_t (NULL = legacy default stream). Every compute
 *    call only enqueues work and returns; results are ready when the stream
 *    reaches that point.
 *  - Device pointers of the attention calls must be 16-byte aligned and
 *    strides multiples of 8 elements (16 bytes), as required by the
 *    tensor-memory-access (TMA) unit; lcb_rope and lcb_cross_entropy state
 *    their own, weaker rules.
 *  - Return value: LCB_OK or a negative LCB_ERR_* code; nothing is launched on
 *    an argument error. With the environment variable LCB_CHECKED=1 every call
 *    synchronises its stream and reports LCB_ERR_TIMEOUT if a kernel's
 *    bounded wait expired (the kernel then returned early, outputs undefined).
 */
#ifndef LCB_ATTN_H
#define LCB_ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LCB_OK 0
#define LCB_ERR_ARG (-1)         /* null pointer, bad size, misaligned pointer or stride */
#define LCB_ERR_UNSUPPORTED (-2) /* D != 128, causal with Sq != Sk, unknown dtype */
#define LCB_ERR_SCHEDULE (-3)    /* zigzag: P < 1 or S not a positive multiple of 2P */
#define LCB_ERR_CUDA (-4)        /* a CUDA runtime/driver call or launch failed */
#define LCB_ERR_TIMEOUT (-5)     /* checked mode: a device-side bounded wait expired */
#define LCB_ERR_SCRATCH (-6)     /* attn_bwd_noalloc: B*H*S exceeds its fixed scratch */

#define LCB_DTYPE_BF16 0
#define LCB_DTYPE_F32 1
/* attn_fwd_ex output mode: fold the block's (O, LSE) into an fp32 ring
 * accumulator held in o and lse (a fused ring step). */
#define LCB_OUT_F32_MERGE 2

/* How attn_bwd_ex writes dq/dk/dv. */
#define LCB_GRAD_BF16 0      /* bf16, overwritten */
#define LCB_GRAD_F32_ACCUM 1 /* fp32, the block's contribution is added */
#define LCB_GRAD_F32_STORE 2 /* fp32, overwritten */

#define LCB_TASK_DIAG 0
#define LCB_TASK_LOWER 1
#define LCB_TASK_UPPER 2
#define LCB_TASK_FULL 3 /* ring_schedule: all local queries x all of src's keys */
#define LCB_TASK_NONE 4 /* ring_schedule: src's keys follow every local query; no work */

/* One attention task of the zigzag ring: rank `rank` at ring step `step`
 * attends its queries [q_off, q_off+q_len) to the keys/values it holds from
 * rank `src`, [k_off, k_off+k_len); offsets are rows in zigzag order. */
typedef struct lcb_task {
  int32_t rank, step, src, kind;
  int32_t q_off, q_len, k_off, k_len;
  int32_t causal;
} lcb_task;

/* One block of attn_fwd_group: query rows [q_off, q_off + q_len) against key
 * rows [k_off, k_off + k_len) of the shared tensors; o_dtype as attn_fwd_ex's. */
typedef struct lcb_fwd_task {
  int32_t q_off, q_len, k_off, k_len;
  int32_t causal, o_dtype;
} lcb_fwd_task;

/* One block of attn_bwd_fused_group: query rows [q_off, q_off + q_len)
 * (q_off a multiple of 128) against key rows [k_off, k_off + k_len). */
typedef struct lcb_bwd_task {
  int32_t q_off, q_len, k_off, k_len;
  int32_t causal;
} lcb_bwd_task;

/* Human-readable name of a status code (static string, never NULL). */
const char* attn_status_string(int status);

/* Library version, major * 10000 + minor * 100 + patch. */
int lcb_version(void);

/*
 * attn_fwd — causal (or full) attention forward, [FA] §2, [FULL].
 *   O_i = sum_j softmax_j(scale * q_i . k_j) v_j,  LSE_i as above.
 * q, k, v: [B,S,H,D] bf16 (in); o: [B,S,H,D] bf16 (out); lse: [B,H,S] fp32
 * (out). Contiguous layouts. S may be any positive size (ragged tails are
 * masked); causal is 0 or 1; scale > 0 (normally 1/sqrt(D)).
 */
int attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int S, int D,
             int causal, float scale, void* stream);

/*
 * attn_fwd_ex — forward on strided views, for ring steps ([SP], [ZZ]).
 * Queries have Sq rows, keys/values Sk rows (Sq != Sk only when causal == 0).
 * Strides are in elements: row stride between consecutive tokens, batch stride
 * between batches; q and o share nothing but shape. o_dtype selects bf16 or
 * fp32 output, or LCB_OUT_F32_MERGE: o (fp32) and lse already hold a partial
 * result over other keys, and this block's result is merged into them in the
 * kernel's epilogue exactly as attn_lse_merge would (a fused ring step, [SP]).
 * lse strides: between heads and between batches.
 * Sk == 0 writes O = 0 and LSE = -inf (merge mode: leaves o, lse unchanged).
 */
int attn_fwd_ex(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int Sq, int Sk,
                int D, int causal, float scale, long long q_row_stride, long long q_batch_stride,
                long long kv_row_stride, long long kv_batch_stride, long long o_row_stride,
                long long o_batch_stride, int o_dtype, long long lse_head_stride, long long lse_batch_stride,
                void* stream);

/*
 * attn_fwd_group — several attn_fwd_ex blocks over the same tensors in ONE
 * launch: the tasks of a ring step, [SP] / [ZZ], run side by side so that the
 * grid fills whole waves of the GPU instead of one partial wave per block.
 * q, k, v, o, lse as attn_fwd_ex's, holding q_rows query/output rows and
 * k_rows key rows; strides likewise. tasks: HOST array of n_tasks <= 16.
 * Each task is an attn_fwd_ex block on its row ranges (causal needs
 * q_len == k_len, in task-local indices); query ranges of different tasks
 * must not overlap (LCB_ERR_ARG); all tasks write bf16, or all write fp32
 * (LCB_DTYPE_F32 or LCB_OUT_F32_MERGE, mixed freely). k_len == 0 behaves as
 * in attn_fwd_ex. The library orders the tasks itself (longest CTAs first).
 */
int attn_fwd_group(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int q_rows,
                   int k_rows, int D, float scale, long long q_row_stride, long long q_batch_stride,
                   long long kv_row_stride, long long kv_batch_stride, long long o_row_stride,
                   long long o_batch_stride, long long lse_head_stride, long long lse_batch_stride,
                   const lcb_fwd_task* tasks, int n_tasks, void* stream);

/* Bytes of device workspace attn_bwd needs: Delta (fp32 [B,H,S]) and the
 * fused pass's tiled fp32 dQ accumulator (B*H*ceil(S/128) tiles of 128x128);
 * 0 for D != 128. */
size_t attn_bwd_workspace_bytes(int B, int H, int S, int D);

/*
 * attn_bwd — backward of attn_fwd with recomputation, [FA] §2 ("重新计算").
 * Inputs q, k, v, o, dO bf16 [B,S,H,D] and lse fp32 [B,H,S] as returned by
 * attn_fwd; outputs dq, dk, dv bf16 [B,S,H,D] (overwritten). Runs the
 * Delta = rowsum(dO * O) preprocess, zeroes the tiled fp32 dQ accumulator in
 * the workspace, runs the fused pass (attn_bwd_fused_ex) and converts dQ to
 * bf16 (lcb_dq_untile).
 * dQ's fp32 summation order is not fixed (the partials of many CTAs are added
 * into the accumulator by asynchronous bulk reductions in L2), so repeated
 * calls may differ in the last bits of dq; dk and dv are deterministic.
 * workspace: device memory of at least attn_bwd_workspace_bytes(), 16-byte
 * aligned, owned by the caller, contents ignored.
 */
int attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
             void* dq, void* dk, void* dv, int B, int H, int S, int D, int causal, float scale, void* workspace,
             size_t ws_bytes, void* stream);

/*
 * attn_bwd_preprocess — Delta_i = sum_d dO_id * O_id in fp32 (the per-row
 * term of dS = P * (dP - Delta)). o, dO bf16 [B,S,H,D] views with the given
 * row/batch strides (elements); delta fp32 with head/batch strides.
 */
int attn_bwd_preprocess(const void* o, const void* dO, float* delta, int B, int H, int S, int D,
                        long long row_stride, long long batch_stride, long long delta_head_stride,
                        long long delta_batch_stride, void* stream);

/*
 * attn_bwd_ex — backward of one block of keys with the row statistics given,
 * for ring steps ([SP], [ZZ]): P_ij = exp(scale q_i.k_j - LSE_i),
 * dS_ij = P_ij (dO_i.v_j - Delta_i). lse and delta ([B,H,Sq] with the given
 * strides) are the statistics over ALL keys of the full problem, so gradients
 * of disjoint key blocks add up to the monolithic gradient.
 * grad_mode LCB_GRAD_BF16: dq/dk/dv are bf16 and overwritten.
 * grad_mode LCB_GRAD_F32_ACCUM: dq/dk/dv are fp32 and the block's
 *   contribution is ADDED to them, each element by one fp32 atomic addition
 *   in L2 (subnormal sums flush to zero): the kernel does not wait for the
 *   old values, and contributions of calls on different streams to the same
 *   rows add up too, in no fixed order.
 * grad_mode LCB_GRAD_F32_STORE: dq/dk/dv are fp32 and overwritten.
 * Gradient strides: dq uses dq_row/batch strides, dk and dv share dkv strides
 * (elements of the gradient dtype).
 */
int attn_bwd_ex(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                const void* dO, void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, int causal,
                float scale, long long q_row_stride, long long q_batch_stride, long long kv_row_stride,
                long long kv_batch_stride, long long lse_head_stride, long long lse_batch_stride, int grad_mode,
                long long dq_row_stride, long long dq_batch_stride, long long dkv_row_stride,
                long long dkv_batch_stride, void* stream);

/*
 * attn_bwd_fused_ex — attn_bwd_ex's gradients in ONE pass over the (key tile,
 * query tile) pairs, [FA] §2: each CTA owns 128 keys, keeps dK and dV in
 * TMEM, and adds every query tile's partial dQ = scale * dS K into a TILED
 * fp32 accumulator by reductions in L2 (bulk asynchronous reductions for
 * columns 0-63, vector reductions for 64-127). Five tensor-core products per
 * tile pair instead of the two passes' seven (dQ's S and dP are not
 * recomputed). dQ's summation order is not fixed.
 * dq_tiles: fp32, the tile holding this call's query rows [128t, 128t+128) of
 *   (b, h) starts at dq_tiles + b*dq_tile_batch_stride + h*dq_tile_head_stride
 *   + t*16384 (floats; 16-byte aligned; strides multiples of 4). Inside a
 *   tile, columns 0-63 are two blocks: block x = 0, 1 (columns [32x, 32x+32))
 *   at x*4096, row r of the block at r*32, and its four-float chunk c
 *   (columns 32x+4c..) at chunk position c ^ (r & 7); columns 64-127 are
 *   chunk-major: the four floats of chunk c (columns 64+4c..64+4c+3) of row r
 *   at 8192 + (c*128 + r)*4. ALWAYS added into: zero it for a fresh gradient;
 *   lcb_dq_untile converts it to bf16 rows. A ring whose query blocks start
 *   at multiples of 128 rows accumulates all its steps into one such buffer.
 * grad_mode applies to dk and dv only (LCB_GRAD_BF16: bf16 overwritten;
 *   LCB_GRAD_F32_ACCUM / _STORE: fp32 added into / overwritten).
 * Other arguments and errors as attn_bwd_ex.
 */
int attn_bwd_fused_ex(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                      const void* dO, float* dq_tiles, void* dk, void* dv, int B, int H, int Sq, int Sk, int D,
                      int causal, float scale, long long q_row_stride, long long q_batch_stride,
                      long long kv_row_stride, long long kv_batch_stride, long long lse_head_stride,
                      long long lse_batch_stride, int grad_mode, long long dq_tile_head_stride,
                      long long dq_tile_batch_stride, long long dkv_row_stride, long long dkv_batch_stride,
                      void* stream);

/*
 * attn_bwd_fused_group — several attn_bwd_fused_ex blocks over the same
 * tensors in ONE launch (the tasks of a ring step, [SP] / [ZZ]). q, dO, lse,
 * delta and the dQ accumulator cover q_rows query rows, k, v, dk, dv k_rows
 * key rows; strides and grad_mode as attn_bwd_fused_ex's. tasks: HOST array
 * of n_tasks <= 16; q_off must be a multiple of 128 (a task adds into the
 * accumulator's tiles from q_off / 128 on); key ranges of different tasks
 * must not overlap (each owns its dK/dV rows; LCB_ERR_ARG), query ranges may.
 * A task without queries zeroes its dK/dV rows in the overwrite modes.
 * The library orders the tasks itself (longest rows first).
 */
int attn_bwd_fused_group(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                         const void* dO, float* dq_tiles, void* dk, void* dv, int B, int H, int q_rows, int k_rows,
                         int D, float scale, long long q_row_stride, long long q_batch_stride,
                         long long kv_row_stride, long long kv_batch_stride, long long lse_head_stride,
                         long long lse_batch_stride, int grad_mode, long long dq_tile_head_stride,
                         long long dq_tile_batch_stride, long long dkv_row_stride, long long dkv_batch_stride,
                         const lcb_bwd_task* tasks, int n_tasks, void* stream);

/* lcb_dq_tiles_zero — zeroes n_floats of a tiled dQ accumulator (an async
 * memset on `stream`; dq_tiles 16-byte aligned). */
int lcb_dq_tiles_zero(float* dq_tiles, long long n_floats, void* stream);

/*
 * lcb_dq_untile — the tiled fp32 dQ accumulator of attn_bwd_fused_ex (tile
 * strides as there) to bf16 rows of a [B, S, H, D] view (row/batch strides in
 * elements, dq 8-byte aligned): dq[b, s, h, :] = tile rows as stored.
 */
int lcb_dq_untile(const float* dq_tiles, long long tile_head_stride, long long tile_batch_stride, void* dq,
                  long long row_stride, long long batch_stride, int B, int H, int S, void* stream);

/*
 * attn_bwd_dkdv_ex / attn_bwd_dq_ex — the two passes of attn_bwd_ex on their
 * own, same arguments and semantics: the first writes only dk and dv (dq is
 * not touched), the second only dq (dk, dv not touched). Given Delta, the two
 * passes are independent and may run on different streams.
 */
int attn_bwd_dkdv_ex(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                     const void* dO, void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, int causal,
                     float scale, long long q_row_stride, long long q_batch_stride, long long kv_row_stride,
                     long long kv_batch_stride, long long lse_head_stride, long long lse_batch_stride,
                     int grad_mode, long long dq_row_stride, long long dq_batch_stride, long long dkv_row_stride,
                     long long dkv_batch_stride, void* stream);
int attn_bwd_dq_ex(const void* q, const void* k, const void* v, const float* lse, const float* delta,
                   const void* dO, void* dq, void* dk, void* dv, int B, int H, int Sq, int Sk, int D, int causal,
                   float scale, long long q_row_stride, long long q_batch_stride, long long kv_row_stride,
                   long long kv_batch_stride, long long lse_head_stride, long long lse_batch_stride, int grad_mode,
                   long long dq_row_stride, long long dq_batch_stride, long long dkv_row_stride,
                   long long dkv_batch_stride, void* stream);

/*
 * attn_lse_merge — fold a partial result into an accumulator, [SP]:
 *   m = max(L_acc, L_b), w_x = exp(L_x - m),
 *   L_acc <- m + ln(w_acc + w_b),  O_acc <- (w_acc O_acc + w_b O_b)/(w_acc + w_b)
 * Both sides -inf gives L = -inf, O = 0. o_acc (fp32) and o_b (bf16 or fp32
 * per o_b_dtype) are [B, rows, H, D] views, each with its own row/batch
 * strides (elements); lse_acc and lse_b are fp32 [B, H, rows] views with
 * their own head/batch strides. If o_out_bf16 is not NULL the merged O is
 * also written there as bf16 with o_acc's strides, which ends a ring without
 * a separate cast. In-place on (o_acc, lse_acc); o_b and lse_b are read only.
 */
int attn_lse_merge(float* o_acc, float* lse_acc, const void* o_b, const float* lse_b, int o_b_dtype,
                   void* o_out_bf16, int B, int H, int rows, int D, long long o_row_stride, long long o_batch_stride,
                   long long ob_row_stride, long long ob_batch_stride, long long lse_head_stride,
                   long long lse_batch_stride, long long lseb_head_stride, long long lseb_batch_stride,
                   void* stream);

/*
 * zigzag_schedule — the zigzag split and ring task table, [ZZ]. HOST memory.
 * c = S / (2P); rank r holds chunks r and 2P-1-r (in that order); perm[t]
 * (t < S) is the natural token index at zigzag position t. tasks[r*P + s]
 * (P*P entries) is rank r's task at ring step s, src = (r - s) mod P:
 * DIAG (s = 0): local x local, causal; LOWER (src < r): 2c local queries x
 * src's first chunk; UPPER (src > r): local second chunk x src's 2c keys.
 * Either output pointer may be NULL. Returns LCB_ERR_SCHEDULE on bad S, P.
 */
int zigzag_schedule(int S, int P, int* perm, lcb_task* tasks);

/*
 * ring_schedule — the plain (contiguous) ring that the zigzag split improves
 * on ([SP] §1: ring attention over sequence shards). Rank r of P holds rows
 * [r S/P, (r+1) S/P); perm (S ints, may be NULL) is the identity. tasks
 * (P*P entries, may be NULL) at [r*P + s], as zigzag_schedule's: at step s
 * rank r holds the keys of src = (r - s) mod P; s = 0 DIAG (causal, local x
 * local), src < r FULL (local queries x src's keys, non-causal), src > r NONE
 * (q_len = k_len = 0: src's keys all follow every local query). Rank r does
 * one causal block and r full blocks: the work grows with r, which the zigzag
 * split evens out. Host-only. LCB_ERR_SCHEDULE unless P >= 1 and S is a
 * positive multiple of P.
 */
int ring_schedule(int S, int P, int* perm, lcb_task* tasks);

/* lcb_cross_entropy modes. */
#define LCB_CE_FWD 0     /* loss and LSE; logits read only */
#define LCB_CE_FWD_BWD 1 /* loss and LSE, and the gradient written over the logits: one read, one write */
#define LCB_CE_BWD 2     /* the gradient over the logits from a given LSE (a previous LCB_CE_FWD) */

/*
 * lcb_cross_entropy — the cross-entropy loss head with an in-place backward,
 * [ZO] §进阶优化与其他技术结合 (Flash Attention's fused CrossEntropyLoss with
 * inplace_backward=True). Per row i of logits x (bf16 [N, V], row stride in
 * elements, 2-byte aligned) with label y_i (int64 [N], DEVICE):
 *   lse[i]  = ln sum_j exp(x_ij)                       (fp32 [N], DEVICE)
 *   loss[i] = lse[i] - x_{i,y_i}                       (fp32 [N], DEVICE; NULL: not written)
 *   x_ij   <- dloss[i] * (exp(x_ij - lse[i]) - [j == y_i])   (bf16, in place)
 * dloss: fp32 [N] DEVICE, NULL meaning 1 for every row. A row whose label is
 * ignore_index gets loss 0 and a zero gradient; a label outside [0, V)
 * otherwise gives loss NaN (and no one-hot term). Any V >= 1: rows are
 * streamed through registers, many in flight per SM; with LCB_CE_FWD_BWD the
 * gradient pass reads each row a second time, from L2 (HBM: one read, and
 * one write with the gradient).
 */
int lcb_cross_entropy(void* logits, const long long* labels, float* loss, float* lse, const float* dloss, int N,
                      int V, long long row_stride, int ignore_index, int mode, void* stream);

/*
 * lcb_rope — rotary position embedding with a raised base, [FA] §3
 * ("RoPE扩展技术"): y = RoPE(x) on bf16 [B, S, H, D=128] views (x and y share
 * row/batch strides in elements; 4-byte aligned; x == y allowed). Pair k
 * couples features k and k + 64 and turns by (pos0 + s) * theta^(-2k/128) at
 * token s; inverse = 1 turns the other way (the transpose: it maps dQ, dK of
 * the rotated tensors back to the unrotated ones). Angles are reduced in
 * fp64, rotated in fp32, rounded to bf16 once.
 */
int lcb_rope(const void* x, void* y, int B, int S, int H, int D, double theta, long long pos0, int inverse,
             long long row_stride, long long batch_stride, void* stream);

/*
 * lcb_permute_rows — row gather/scatter on the device, used to move a
 * [B=1, S, H, D] tensor into zigzag order and back, [ZZ].
 * scatter == 0: dst[t] = src[perm[t]];  scatter == 1: dst[perm[t]] = src[t].
 * perm: DEVICE int32 [rows]; row_bytes a multiple of 16; src != dst.
 */
int lcb_permute_rows(const void* src, void* dst, const int* perm, int rows, long long row_bytes, void* stream);
int lcb_scatter_rows(const void* src, void* dst, const int* perm, int rows, long long row_bytes, void* stream);

/* lcb_cast_f32_bf16 — dst[i] = bf16(src[i]) (round to nearest even) for
 * i < n; ends a ring whose accumulators are fp32. Both 16-byte aligned. */
int lcb_cast_f32_bf16(const float* src, void* dst, long long n, void* stream);

/* Bounded-wait limit of all kernels, nanoseconds (default 2e9, or the
 * environment variable LCB_WAIT_LIMIT_NS). Returns the previous value. */
unsigned long long lcb_set_wait_limit_ns(unsigned long long ns);

/*
 * lcb_selftest_bounded_wait — launches a one-CTA kernel that waits on a
 * barrier nothing ever completes, with the current wait limit, synchronises
 * the stream and returns the outcome: LCB_ERR_TIMEOUT when the wait expired
 * and the kernel returned cleanly (the expected result), LCB_OK if it did not
 * expire, LCB_ERR_CUDA on a CUDA failure. Clears the status word afterwards.
 */
int lcb_selftest_bounded_wait(void* stream);

/* Reads and clears the device status word of the current device (a
 * synchronising call): 0, or a bitmask with 1 = a bounded wait expired. */
int lcb_take_device_status(unsigned int* where);

/*
 * lcb_ulysses_all_to_all — the all-to-all of Ulysses sequence parallelism for
 * P ranks emulated on one device ([SP] §1: Ulysses注意力, based on DeepSpeed;
 * [ZZ] §模型并行策略解析: ulysses_attn). Rank r of P holds sequence rows
 * [r S/P, (r+1) S/P) of all heads; rank j after the exchange holds every row
 * of heads [j H/P, (j+1) H/P).
 * Layouts (contiguous, elements of elem_bytes bytes, 2 = bf16 or 4 = fp32):
 *   sequence layout: [B, S, H, D], the P ranks' pieces one after another;
 *   head layout:     [P, B, S, H/P, D], rank j's part at element offset
 *                    j * B * S * (H/P) * D. Taken together the parts are one
 *                    [P*B, S, H/P, D] tensor: a single attention call with
 *                    batch P*B and H/P heads computes every rank's heads.
 * direction LCB_ULYSSES_SEQ_TO_HEAD: head[j][b][s][hh] = seq[b][s][j*H/P+hh];
 * direction LCB_ULYSSES_HEAD_TO_SEQ: the inverse.
 * A copy (no arithmetic). Requires P | H, P | S, (H/P)*D*elem_bytes a multiple
 * of 16 bytes, src and dst 16-byte aligned and not overlapping (no in-place),
 * B*S*(H/P)*D*elem_bytes/16 < 2^31; LCB_ERR_ARG otherwise.
 */
#define LCB_ULYSSES_SEQ_TO_HEAD 0
#define LCB_ULYSSES_HEAD_TO_SEQ 1
int lcb_ulysses_all_to_all(const void* src, void* dst, int B, int S, int H, int D, int P, int elem_bytes,
                           int direction, void* stream);

/*
 * attn_bwd_noalloc — attn_bwd for callers that cannot allocate device memory.
 * The source pages have no counterpart of this call; it exists for callers
 * that cannot hand the library a workspace, because their memory manager
 * owns all device memory and gives out only the tensors they compute on,
 * because their memory plan is fixed at start-up, or because they must not
 * call cudaMalloc, which can synchronise the device mid-pipeline.
 * Same arguments and results as attn_bwd minus the workspace. The Delta
 * scratch lives in a fixed 8 MiB array in device memory inside the library.
 *  - Limit: B * H * S <= attn_bwd_noalloc_max_rows() (2^21); larger problems
 *    return LCB_ERR_SCRATCH and launch nothing.
 *  - First call on a device: CUDA loads modules lazily by default, so the
 *    first call on each device (in each context, after a cudaDeviceReset too)
 *    loads the library's module there, which reserves the 8 MiB array and may
 *    synchronise the device. Make that first call outside any stream capture.
 *    The array then stays reserved until the process exits or the context is
 *    reset.
 *  - No allocation after that: later calls make no cudaMalloc/cudaFree or
 *    other allocating call; each looks up the array's device address, which
 *    allocates nothing once the module is loaded.
 *  - Sharing: the array exists once per device. Every call on one device uses
 *    it and it keeps the previous call's contents; the call writes all the
 *    Delta values it reads before reading them, so nothing needs clearing.
 *    Calls that overlap on the GPU of the same device (issued on different
 *    streams without ordering) race on the array; calls ordered on one stream
 *    are safe, and calls on different devices each use their own copy.
 */
int attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse, const void* dO,
                     void* dq, void* dk, void* dv, int B, int H, int S, int D, int causal, float scale,
                     void* stream);

/* Largest B * H * S accepted by attn_bwd_noalloc. */
long long attn_bwd_noalloc_max_rows(void);

#ifdef __cplusplus
}
#endif

#endif /* LCB_ATTN_H */
