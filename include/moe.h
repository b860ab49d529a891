/*
 * moe.h -- C ABI of libmoe.so: the forward pass of one sparse
 * Mixture-of-Experts (MoE) layer on one NVIDIA B300 (sm_103a).
 *
 * The layer, per token t with hidden state x[t] (row of x[T,d]):
 *   1. router logits   l[e] = x[t] . W_g[:,e] + b[e]          (e < N)
 *   2. top-k           the k largest logits, descending, equal logits ->
 *                      lower expert id; NaN ranks below every number
 *   3. gate weights    w_j = softmax over the k selected logits
 *   4. dispatch        tokens regrouped by expert, stable by token index,
 *                      optionally capped at C rows per expert
 *   5. expert FFN      SwiGLU: o = (SiLU(x W_gate[e]) * (x W_up[e])) W_down[e]
 *   6. combine         y[t] = sum over kept slots j of w_j * o_j
 *                      (+ the always-on shared expert's output, weight 1)
 *
 * Sources, by page title and section:
 *   steps 1-3: "MoE 分片：混合專家模型的平行化策略", section 動態 token 路由,
 *              steps 2 and 6; "MoE 推理：激活参数 vs 总参数与专家路由",
 *              sections 深入原理 and 代码; "大模型MoE混合专家架构原理与
 *              DeepSeek-V4工程实践解析", section MoE核心机制.
 *   step 4:    "MoE稀疏激活原理与工程实践", 3.1 (token-level batching: regroup
 *              a batch's tokens by target expert id) and 2.2 (expert capacity).
 *   step 5:    "MoE 分片", section 什麼是 MoE 模型 (an expert is two linear
 *              maps with an activation between) and step 4; the SwiGLU form
 *              (gate, up, SiLU, down) is this library's reading.
 *   step 6:    "MoE 分片", step 6; "MoE 架构科普", section 专家粒度 (shared
 *              experts every token passes through).
 *
 * Conventions for every entry point:
 *   - All pointers to tensors are DEVICE pointers unless the name says host.
 *     Every tensor is row-major and contiguous; base addresses are 16-byte
 *     aligned; d and f (and fs) are multiples of 8.  The caller owns every
 *     buffer, including the workspace; the library allocates no device memory
 *     and keeps no per-call state.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Every call only enqueues work on it; none synchronises the host, and
 *     none reads device results back to the host.
 *   - Argument errors are found on the host and returned synchronously with
 *     nothing enqueued.  A failed kernel launch returns MOE_ERR_CUDA.
 *   - Errors found on the device (bad expert ids, NaN logits, a bounded wait
 *     that gave up) are OR-ed as MOE_DEV_* bits into *device_status when that
 *     pointer is non-NULL; the affected rows are skipped.  The caller reads it
 *     after synchronising.  No kernel traps, asserts or waits without bound.
 *   - moe_last_error() gives a one-line description of the last failure on
 *     the calling host thread.
 */
#ifndef MOE_H_
#define MOE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1, /* a size, pointer or alignment the call rejects   */
  MOE_ERR_UNSUPPORTED = 2, /* valid, but outside what the kernels implement   */
  MOE_ERR_WORKSPACE = 3,   /* workspace NULL or smaller than *_workspace_size */
  MOE_ERR_CUDA = 4,        /* a CUDA runtime call or kernel launch failed     */
  MOE_ERR_DEVICE = 5       /* no usable CUDA device / wrong architecture      */
} moe_status_t;

typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

/* Bits OR-ed into *device_status by the kernels. */
#define MOE_DEV_BAD_EXPERT_ID 0x1 /* an expert id outside [0,N) reached moe_permute */
#define MOE_DEV_NAN_LOGIT 0x2     /* a router logit was NaN (ranked last)           */
#define MOE_DEV_TIMEOUT 0x4       /* a bounded on-chip wait gave up; output invalid */
#define MOE_DEV_BAD_TILE 0x8      /* grouped-GEMM tile outside the expert layout     */
#define MOE_DEV_BAD_COUNTS 0x10   /* expert-parallel counts do not add up to the rows */
#define MOE_DEV_BAD_ROW 0x20      /* an output-row index outside the output rows      */

const char *moe_status_string(moe_status_t s);
const char *moe_last_error(void);
/* Library version, e.g. "moe63 1.0 sm_103a". */
const char *moe_version(void);
/* Kernel launches this process has enqueued through the library so far
 * (all entry points, all threads); for counting launches per call. */
uint64_t moe_launch_counter(void);

/* Capacity in rows per expert for a capacity factor: ceil(cf * T * k / N),
 * computed in double precision; 0 (no limit) when cf <= 0.  Capacity reading:
 * "MoE稀疏激活原理与工程实践", 2.2 -- the page caps each expert's queue but
 * gives no formula; C = factor x the even-split load is this library's. */
int moe_capacity(float capacity_factor, int T, int k, int N);

/* ---------------------------------------------------------------------------
 * Step 1-3: router GEMM, top-k and softmax over the selected k.
 *   x [T,d] (dtype), W_g [d,N] (dtype), bias [N] fp32 or NULL.
 *   logits [T,N] fp32 output, or NULL to skip writing it.
 *   topk_idx [T,k] int32, topk_w [T,k] fp32 outputs (slot order = rank order).
 * Requires 1 <= k <= N <= 256, k <= 32, T >= 0, d >= 8, d % 8 == 0.
 * fp32 accumulation; the softmax is exp(l_j - l_0) / sum_j' exp(l_j' - l_0).
 * ------------------------------------------------------------------------- */
moe_status_t moe_router_topk(const void *x, const void *W_g, const float *bias,
                             moe_dtype_t dtype, int T, int d, int N, int k,
                             float *logits, int32_t *topk_idx, float *topk_w,
                             int32_t *device_status, void *stream);

/* ---------------------------------------------------------------------------
 * Step 4: dispatch.  Regroups the T*k assignments by expert, stable by token
 * index, and gathers the token rows.
 *   topk_idx [T,k] int32; topk_w [T,k] fp32 or NULL (then row_scale unused).
 *   capacity: rows kept per expert (0 = no limit); an assignment is kept iff
 *   its 0-based rank among its expert's assignments, by token index, is below
 *   the capacity.
 * Outputs (device):
 *   counts [N]      assignments routed to each expert, before capacity
 *   offsets [N+1]   exclusive prefix sum of KEPT rows; offsets[N] = kept total A
 *   perm_token [T*k] token of row p (p < A)
 *   row_scale [T*k] gate weight of row p, or NULL
 *   inv_pos [T,k]   row p of assignment (t,j), -1 if dropped
 *   x_perm [T*k,d]  x[perm_token[p]] for p < A (dtype), or NULL to skip
 *   dropped         scalar int32: assignments dropped, or NULL
 * An expert id outside [0,N) sets MOE_DEV_BAD_EXPERT_ID and that assignment
 * is treated as dropped.  Workspace: moe_permute_workspace_size(T, N, k).
 * ------------------------------------------------------------------------- */
size_t moe_permute_workspace_size(int T, int N, int k);
moe_status_t moe_permute(const int32_t *topk_idx, const float *topk_w,
                         const void *x, moe_dtype_t dtype, int T, int d, int N,
                         int k, int capacity, int32_t *counts, int32_t *offsets,
                         int32_t *perm_token, float *row_scale,
                         int32_t *inv_pos, void *x_perm, int32_t *dropped,
                         int32_t *device_status, void *workspace,
                         size_t workspace_bytes, void *stream);

/* moe_permute without a workspace argument, for callers that cannot allocate
 * device memory where they dispatch tokens (e.g. an operator inside a host
 * framework that receives only its input and output buffers and may not
 * allocate while the model runs).  It has no counterpart in the source pages:
 * it is an interface convenience of this library.  Same arguments, outputs
 * and errors as moe_permute; the scratch comes from a fixed array inside the
 * library (256 KB, held on every GPU that loads it until the process exits):
 *   - requires ceil(T/256) * N <= 65536, else MOE_ERR_UNSUPPORTED with a
 *     message (e.g. T <= 65536 tokens for N = 256 experts);
 *   - allocates nothing; the first call on each device looks up the array's
 *     device address (with that device current), so make that first call
 *     before any stream capture.  The address is kept for later calls, which
 *     assumes the device's context is not reset (cudaDeviceReset) while the
 *     library stays loaded;
 *   - every call shares the one array: calls that overlap on the GPU race;
 *     order them on one stream.  Nothing in it needs clearing between calls. */
moe_status_t moe_permute_noalloc(const int32_t *topk_idx, const float *topk_w,
                                 const void *x, moe_dtype_t dtype, int T, int d,
                                 int N, int k, int capacity, int32_t *counts,
                                 int32_t *offsets, int32_t *perm_token,
                                 float *row_scale, int32_t *inv_pos,
                                 void *x_perm, int32_t *dropped,
                                 int32_t *device_status, void *stream);

/* ---------------------------------------------------------------------------
 * Step 4b: dispatch with capacity overflow RE-ROUTED to the next-best expert.
 * Source: "MoE稀疏激活原理与工程实践", 2.2 (专家容量的硬约束: a token whose
 * selected expert already holds its capacity goes to its next-best expert).
 *   cand_idx [T,k+R] int32: each token's experts by rank (moe_router_topk
 *     with k+R); cand_w [T,k+R] fp32: the router's softmax over those k+R.
 *   First pass: each expert keeps its first `capacity` assignments by token
 *   index (as moe_permute).  Then R rounds: every slot still without an
 *   expert proposes its token's next untried candidate (ranks k, k+1, ...,
 *   taken in slot order, used up whether granted or not); each expert grants
 *   its remaining room to the round's proposals in (token, slot) order.  A
 *   slot unplaced after R rounds is dropped.
 *   final_idx [T,k] out: each slot's expert, -1 if dropped.
 *   final_w [T,k] out: softmax over the token's final experts' logits (the
 *     k+R softmax renormalised over them; a dropped slot keeps its first
 *     choice in the denominator and contributes nothing).
 *   demand [N] out (may be NULL): first-choice assignments per expert before
 *     the capacity (the router's selection frequency).
 *   counts, offsets, perm_token, row_scale, inv_pos, x_perm, dropped: as
 *     moe_permute, over the final selection (counts = placed per expert).
 *   rerouted: scalar out (may be NULL), slots placed in rounds >= 1.
 *   capacity >= 1, 0 <= R, k + R <= N <= 1024.  Deterministic.
 *   Workspace: moe_permute_reroute_workspace_size(T, N, k, R).
 * ------------------------------------------------------------------------- */
size_t moe_permute_reroute_workspace_size(int T, int N, int k, int R);
moe_status_t moe_permute_reroute(const int32_t *cand_idx, const float *cand_w,
                                 const void *x, moe_dtype_t dtype, int T, int d,
                                 int N, int k, int R, int capacity,
                                 int32_t *final_idx, float *final_w,
                                 int32_t *demand, int32_t *counts,
                                 int32_t *offsets, int32_t *perm_token,
                                 float *row_scale, int32_t *inv_pos,
                                 void *x_perm, int32_t *dropped,
                                 int32_t *rerouted, int32_t *device_status,
                                 void *workspace, size_t workspace_bytes,
                                 void *stream);

/* ---------------------------------------------------------------------------
 * Step 5: grouped expert FFN (SwiGLU) over permuted rows.
 *   x_perm [A_max,d] (dtype): rows of expert e are offsets[e]..offsets[e+1]-1.
 *   offsets [N+1] device int32 (from moe_permute); offsets[N] <= A_max.
 *   row_scale [A_max] fp32 or NULL: each output row is multiplied by it.
 *   W_gate, W_up [N,d,f]; W_down [N,f,d] (dtype).
 *   y_perm [A_max,d] (dtype) output: row_scale[p] * SwiGLU_e(x_perm[p]).
 * bf16 runs on tcgen05 tensor cores (fp32 accumulation in tensor memory; the
 * hidden activation h is rounded to bf16 between the two GEMMs); fp32 runs
 * on the CUDA cores in fp32.  Workspace: moe_expert_ffn_workspace_size().
 * ------------------------------------------------------------------------- */
size_t moe_expert_ffn_workspace_size(int A_max, int d, int f, int N,
                                     moe_dtype_t dtype);
moe_status_t moe_expert_ffn(const void *x_perm, const int32_t *offsets,
                            const float *row_scale, int A_max, int d, int f,
                            int N, moe_dtype_t dtype, const void *W_gate,
                            const void *W_up, const void *W_down, void *y_perm,
                            int32_t *device_status, void *workspace,
                            size_t workspace_bytes, void *stream);

/* The same FFN storing each output row at a caller-given row: y[out_row[p]]
 * = row_scale[p] * SwiGLU_e(x_perm[p]) for every p < offsets[N].  out_row
 * [A_max] device int32, indices into y [rows_out, d] (dtype); an index
 * outside [0, rows_out) stores nothing and sets MOE_DEV_BAD_ROW in
 * device_status.  Rows of y no p maps to are left as they are.  The
 * expert-parallel layer passes moe_ep_regroup's `dest`, so the outputs land
 * in received order without a moe_ep_return copy.  Same workspace as
 * moe_expert_ffn; argument errors as there, plus NULL out_row or rows_out < 0
 * (MOE_ERR_INVALID_ARG). */
moe_status_t moe_expert_ffn_to_rows(const void *x_perm, const int32_t *offsets,
                                    const float *row_scale, const int32_t *out_row,
                                    int A_max, int d, int f, int N, moe_dtype_t dtype,
                                    const void *W_gate, const void *W_up,
                                    const void *W_down, void *y, int rows_out,
                                    int32_t *device_status, void *workspace,
                                    size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Low-precision expert weights: FP8 E4M3 with absmax scales.
 * Source: "大模型MoE混合专家架构原理与DeepSeek-V4工程实践解析", section
 * MoE模型推理部署与显存优化实战 (decoding is bound by the bytes of weights
 * read; storing them in fewer bits is the remedy); "MoE稀疏激活原理与工程实践",
 * 4.3.  Format: OCP E4M3 (largest finite 448).  A vector v is stored as
 * E4M3(v * (448 / amax|v|)) (nearest even, saturating) and the fp32 scale
 * amax / 448 (an all-zero vector: scale 1).
 *
 * moe_quantize_weights_e4m3: weights W [N,d,f] bf16 read as [N, K=d, M=f]
 *   (gate/up: K = model dim; W_down [N,f,d]: pass (d=f, f=d)), one scale per
 *   output column m over K: Wq [N,f,d] codes (channel-major, so the GEMM
 *   reads it K-major), scale [N,f].  d % 16 == 0.  An offline step.
 * moe_quantize_rows_e4m3: rows x [R,C] bf16, one scale per row: q [R,C],
 *   scale [R].  C % 16 == 0.
 * moe_expert_ffn_fp8: moe_expert_ffn with E4M3 gate/up: xq_perm [A_max,d]
 *   codes of the permuted token rows (row p = the codes of token
 *   perm_token[p] from moe_quantize_rows_e4m3; moe_forward writes them while
 *   it dispatches),
 *   row p's scale = x_scale[perm_token[p]] (x_scale [T] per token);
 *   g = (xq . Wq_gate[e][j]) * x_scale * wscale_gate[e][j], u likewise,
 *   h = SiLU(g) * u rounded to bf16, y_perm = row_scale * (h W_down) as in
 *   moe_expert_ffn.  With Wq_down ([N,d,f] codes, wscale_down [N,d]; W_down
 *   may be NULL) the down projection is E4M3 too: h is kept in fp32 and each
 *   kept row quantised from those values like x (one scale per row,
 *   f % 16 == 0), and y_perm[p][m] = row_scale[p] * (hq . Wq_down[e][m]) *
 *   h_scale[p] * wscale_down[e][m].  Workspace:
 *   moe_expert_ffn_fp8_workspace_size.
 * ------------------------------------------------------------------------- */
size_t moe_expert_ffn_fp8_workspace_size(int A_max, int d, int f, int N,
                                         int fp8_down);
moe_status_t moe_quantize_weights_e4m3(const void *W, int N, int d, int f,
                                       uint8_t *Wq, float *scale, void *stream);
moe_status_t moe_quantize_rows_e4m3(const void *x, int R, int C, uint8_t *q,
                                    float *scale, void *stream);
moe_status_t moe_expert_ffn_fp8(const uint8_t *xq_perm, const float *x_scale,
                                const int32_t *perm_token,
                                const int32_t *offsets, const float *row_scale,
                                int A_max, int d, int f, int N,
                                const uint8_t *Wq_gate, const float *wscale_gate,
                                const uint8_t *Wq_up, const float *wscale_up,
                                const void *W_down, const uint8_t *Wq_down,
                                const float *wscale_down, void *y_perm,
                                int32_t *device_status, void *workspace,
                                size_t workspace_bytes, void *stream);

/* ---------------------------------------------------------------------------
 * Step 6: combine.  y[t] = sum_{j<k, inv_pos[t,j] >= 0} y_perm[inv_pos[t,j]]
 *                          (+ shared_y[t]), summed in fp32 in that order.
 *   y_perm [*,d] and shared_y [T,d] (NULL = none) in y_perm_dtype;
 *   y [T,d] in y_dtype (fp32 or bf16, rounded once at the end).
 * ------------------------------------------------------------------------- */
moe_status_t moe_combine(const void *y_perm, moe_dtype_t y_perm_dtype,
                         const int32_t *inv_pos, int T, int k, int d,
                         const void *shared_y, void *y, moe_dtype_t y_dtype,
                         void *stream);

/* ---------------------------------------------------------------------------
 * The whole layer in one call: steps 1-6 plus the optional shared expert.
 * Optional outputs may be NULL (then workspace holds them).
 *   Sizes: T >= 1 and 1 <= k <= N; d, f and fs multiples of 8 (d of 16 with
 *   E4M3 gate/up, f of 16 with an E4M3 down projection); T*k < 2^31; every
 *   tensor 16-byte aligned; re-routing needs a capacity and k + rounds <= N.
 *   Otherwise MOE_ERR_INVALID_ARG (moe_forward_workspace_size returns 0).
 *   N > 256, or k (+ reroute_rounds) > 32: MOE_ERR_UNSUPPORTED.
 * ------------------------------------------------------------------------- */
typedef struct moe_forward_args {
  int T, d, f, N, k;
  moe_dtype_t dtype;          /* x and every weight                          */
  const void *x;              /* [T,d]                                       */
  const void *W_g;            /* [d,N]                                       */
  const float *router_bias;   /* [N] fp32, or NULL                           */
  const void *W_gate;         /* [N,d,f]                                     */
  const void *W_up;           /* [N,d,f]                                     */
  const void *W_down;         /* [N,f,d]                                     */
  int fs;                     /* shared-expert hidden dim, 0 = no shared     */
  const void *Ws_gate;        /* [d,fs]                                      */
  const void *Ws_up;          /* [d,fs]                                      */
  const void *Ws_down;        /* [fs,d]                                      */
  float capacity_factor;      /* <= 0: no capacity limit                     */
  void *y;                    /* [T,d] output                                */
  moe_dtype_t y_dtype;        /* MOE_F32 (default) or MOE_BF16               */
  float *logits;              /* [T,N] optional output                       */
  int32_t *topk_idx;          /* [T,k] optional output                       */
  float *topk_w;              /* [T,k] optional output                       */
  int32_t *counts;            /* [N]   optional output                       */
  int32_t *offsets;           /* [N+1] optional output                       */
  int32_t *inv_pos;           /* [T,k] optional output                       */
  int32_t *dropped;           /* scalar optional output                      */
  int32_t *device_status;     /* scalar, OR-ed MOE_DEV_* bits, optional      */
  int reroute_rounds;         /* 0: overflow dropped; R > 0 (with a capacity):
                                 overflow re-routed in R rounds, see
                                 moe_permute_reroute; topk_idx/topk_w then
                                 hold the final selection (-1 = dropped)     */
  int32_t *rerouted;          /* scalar optional output: slots re-routed     */
  /* FP8 gate/up (optional, bf16 layers): when set, the routed experts'
   * gate/up projections run in E4M3 from these (W_gate/W_up may be NULL);
   * x is quantised per token row on the fly; W_down stays bf16.  See
   * moe_quantize_weights_e4m3.                                             */
  const uint8_t *Wq_gate;     /* [N,f,d] E4M3 codes                          */
  const float *wscale_gate;   /* [N,f] channel scales                        */
  const uint8_t *Wq_up;       /* [N,f,d]                                     */
  const float *wscale_up;     /* [N,f]                                       */
  const uint8_t *Wq_down;     /* optional with the above: E4M3 down projection
                                 [N,d,f] (W_down may then be NULL); h is
                                 quantised per row before it               */
  const float *wscale_down;   /* [N,d]                                       */
  /* Timing hooks (optional, NULL = none): two cudaEvent_t (as void*) that
   * moe_forward records on its stream right before the routed experts' first
   * grouped-GEMM launch and right after their last one, so a caller can time
   * the expert FFN inside the same step it times the layer.  Recording them
   * orders the FFN's first launch after the dispatch's completion (no early
   * launch across the event), which costs a few microseconds per step.     */
  void *ffn_event_begin;
  void *ffn_event_end;
} moe_forward_args;

size_t moe_forward_workspace_size(const moe_forward_args *args);
moe_status_t moe_forward(const moe_forward_args *args, void *workspace,
                         size_t workspace_bytes, void *stream);

/* The same call with x read from, and y written to, HOST memory: enqueues
 * the host->device copy of x_host into args->x, the layer, and the
 * device->host copy of args->y into y_host on `stream`.  args->x and args->y
 * are the device staging buffers.  Pinned host memory makes the copies
 * asynchronous; the caller synchronises the stream before reading y_host. */
moe_status_t moe_forward_host_io(const moe_forward_args *args,
                                 const void *x_host, void *y_host,
                                 void *workspace, size_t workspace_bytes,
                                 void *stream);

/* The host-buffer call with the copies overlapped with the layer: the T
 * tokens run as `chunks` consecutive batches on `stream` (with three or more,
 * the first and the last half the size of the others: their copy in and copy
 * out are what no compute hides); every chunk's x
 * rows go host->device on h2d_stream (all issued at once, each batch waits
 * for its own), and each batch's y rows go back on d2h_stream as soon as it
 * is done; `stream` then waits for the last copy.  Each token's output row
 * depends on that token alone, so y equals moe_forward_host_io's -- except
 * under a capacity limit or re-routing, whose drops depend on the whole
 * batch: there chunks is taken as 1.  chunks <= 0: moe_forward_overlap_chunks
 * (as many as keep each batch's tensor work at least four times the time
 * to stream its weights again, at most one per 2048 tokens, 16 in all).  The
 * call returns y only: the routing outputs of args must be NULL.  Three
 * distinct streams; workspace: moe_forward_workspace_size(args).  Pinned
 * host memory makes the copies asynchronous.  The first call on a host thread
 * and device creates the CUDA events it orders the streams with and keeps
 * them for later calls (make that first call outside any stream capture). */
int moe_forward_overlap_chunks(const moe_forward_args *args);
moe_status_t moe_forward_host_io_overlapped(const moe_forward_args *args,
                                            const void *x_host, void *y_host,
                                            void *workspace,
                                            size_t workspace_bytes, int chunks,
                                            void *stream, void *h2d_stream,
                                            void *d2h_stream);

/* ---------------------------------------------------------------------------
 * Expert parallelism: the device steps around the two all-to-all exchanges.
 * Source: "MoE 分片：混合專家模型的平行化策略", sections 專家平行化詳解 (the N
 * experts split over G GPUs) and 動態 token 路由 steps 3-5 (rows go to the
 * GPU holding their expert, are computed there and come back);
 * "MoE稀疏激活原理与工程实践", 2.2 (one all-to-all per routing step).
 *
 * Rank r holds experts [r*Ne, (r+1)*Ne), N = G*Ne.  Its moe_permute over all
 * N experts orders its rows by expert, so the rows for rank q are the
 * contiguous range x_perm[offsets[q*Ne] : offsets[(q+1)*Ne]) and need no
 * packing.  The caller exchanges, with its own collective library, each
 * rank's kept counts per expert and then those row ranges (and their
 * row_scale values); rank r then holds, from each source s in turn, the rows
 * of each of its experts e: block (s, e), recv_counts[s*Ne + e] rows.
 *
 * moe_ep_regroup: moves block (s, e) to expert e's range, after the blocks of
 *   sources 0..s-1 (stable), so the grouped GEMM sees each expert's rows
 *   together:
 *   recv_counts [G*Ne] device int32; x_recv [R,d] (dtype) and row_scale_recv
 *   [R] fp32 (or NULL) in received order, R = sum of recv_counts.
 *   Outputs: x_local [R,d], row_scale_local [R] (if row_scale_recv),
 *   offsets_local [Ne+1] (moe_expert_ffn's offsets over the local experts),
 *   dest [R] int32: where received row i went; src [R] int32 or NULL: the
 *   inverse, src[dest[i]] = i (moe_expert_ffn_to_rows's out_row, so the
 *   outputs land in received order directly).  If the counts do not add up
 *   to R nothing is copied and MOE_DEV_BAD_COUNTS is set.
 * moe_ep_return: y_back[i] = y_local[dest[i]], the expert outputs put back in
 *   received order, ready for the return exchange; afterwards the source
 *   rank's rows are in its own x_perm order and moe_combine finishes the layer.
 * Requirements: 1 <= G, 1 <= Ne, G*Ne <= 4096, d*sizeof(dtype) % 16 == 0,
 * 16-byte aligned rows.  No workspace; asynchronous on `stream`.
 * ------------------------------------------------------------------------- */
moe_status_t moe_ep_regroup(const int32_t *recv_counts, int G, int Ne,
                            const void *x_recv, const float *row_scale_recv,
                            int R, int d, moe_dtype_t dtype, void *x_local,
                            float *row_scale_local, int32_t *offsets_local,
                            int32_t *dest, int32_t *src,
                            int32_t *device_status, void *stream);
moe_status_t moe_ep_return(const void *y_local, const int32_t *dest, int R,
                           int d, moe_dtype_t dtype, void *y_back,
                           void *stream);

/* ---------------------------------------------------------------------------
 * Routing diagnostics (forward only): how evenly the router spreads the load.
 * Source: "MoE稀疏激活原理与工程实践", 4.2 路由质量诊断 (selection frequency of
 * each expert, entropy of that distribution in bits against log2 N, the three
 * most chosen experts and their share, the largest single share, std/mean of
 * the frequencies); "大模型MoE混合专家架构原理与DeepSeek-V4工程实践解析"
 * (balance statistic N * sum_i f_i * p_i, p_i the mean routing probability).
 *   counts [N] device int32: assignments per expert before any capacity
 *     (moe_permute's or moe_forward's `counts`); f_i = counts_i / sum(counts).
 *   logits [T,N] device fp32 or NULL (moe_router_topk's `logits`): p_i is the
 *     mean over the T tokens of the softmax over all N logits.  NULL: no p_i,
 *     balance = NaN.
 *   stats: device pointer to one moe_routing_stats_t (output).
 *   freq [N], prob_mean [N]: device fp32 outputs, each may be NULL
 *     (prob_mean is not written when logits is NULL).
 * Conventions: entropy takes 0 log 0 = 0; std is the population std; the
 * three most chosen go by count, equal counts -> lower id, -1 past N; with no
 * assignments every statistic is 0.  Deterministic (fixed reduction order),
 * fp32.  Workspace: moe_routing_stats_workspace_size(T, N) bytes (0 when
 * logits is NULL).  Argument errors return synchronously; N <= 1024.
 * ------------------------------------------------------------------------- */
typedef struct {
  float entropy_bits;         /* -sum f_i log2 f_i                           */
  float entropy_max_bits;     /* log2 N (an even load)                       */
  float top3_share;           /* f of the three most chosen experts          */
  float max_share;            /* largest f_i                                 */
  float freq_cv;              /* std(f) / mean(f)                            */
  float balance;              /* N * sum f_i p_i; NaN without logits         */
  int32_t top3[3];            /* ids of the three most chosen (-1 past N)    */
  int32_t assignments;        /* sum of counts                               */
} moe_routing_stats_t;

size_t moe_routing_stats_workspace_size(int T, int N);
moe_status_t moe_routing_stats(const float *logits, const int32_t *counts, int T,
                               int N, moe_routing_stats_t *stats, float *freq,
                               float *prob_mean, void *workspace,
                               size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H_ */
