// Internal declarations shared by the CUDA translation units of libmoe.so.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// Records a one-line description of the last failure (thread-local).
void set_error(const char *fmt, ...);
// Counts one enqueued kernel launch (read by moe_launch_counter()).
void count_launch();

#define MOE_CUDA_TRY(expr)                                                     \
  do {                                                                         \
    cudaError_t err_ = (expr);                                                 \
    if (err_ != cudaSuccess) {                                                 \
      ::moe::set_error("%s: %s (%s:%d)", #expr, cudaGetErrorString(err_),      \
                       __FILE__, __LINE__);                                    \
      return MOE_ERR_CUDA;                                                     \
    }                                                                          \
  } while (0)

#define MOE_LAUNCH_CHECK()                                                     \
  do {                                                                         \
    ::moe::count_launch();                                                     \
    cudaError_t err_ = cudaGetLastError();                                     \
    if (err_ != cudaSuccess) {                                                 \
      ::moe::set_error("kernel launch: %s (%s:%d)", cudaGetErrorString(err_),  \
                       __FILE__, __LINE__);                                    \
      return MOE_ERR_CUDA;                                                     \
    }                                                                          \
  } while (0)

// ---- element helpers --------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }
template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

// Loads 8 consecutive elements (16 B for bf16, 32 B for fp32) as fp32.
__device__ __forceinline__ void load8(const __nv_bfloat16 *p, float (&v)[8]) {
  uint4 q = *reinterpret_cast<const uint4 *>(p);
  const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    v[2 * i] = f.x;
    v[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float *p, float (&v)[8]) {
  float4 a = *reinterpret_cast<const float4 *>(p);
  float4 b = *reinterpret_cast<const float4 *>(p + 4);
  v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
  v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Programmatic dependent launch.  A kernel launched with launch_pdl may start
// while the previous kernel on its stream is still running; pdl_begin() lets
// the next kernel start launching (it waits in its own pdl_begin) and then
// waits until the previous kernel has finished and its writes are visible.
// Every kernel of the layer calls it before touching global memory (without
// the launch attribute both are no-ops), so kernel i finishing implies every
// earlier kernel has finished.
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_begin() {
  pdl_trigger();
  pdl_wait();
}

__device__ __forceinline__ void report(int32_t *status, int32_t bits) {
  if (status) atomicOr(status, bits);
}

// Launches `kernel` with programmatic stream serialisation (see pdl_begin).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- launchers (each returns MOE_OK or an error; never synchronises) --------
moe_status_t launch_router_topk(const void *x, const void *W_g, const float *bias,
                                moe_dtype_t dtype, int T, int d, int N, int k,
                                float *logits, int32_t *topk_idx, float *topk_w,
                                int32_t *device_status, cudaStream_t stream);

size_t permute_workspace_bytes(int T, int N, int k);
// Launch attributes and occupancy answers are per device; a process may drive
// several GPUs, so the launchers remember them per device index.
constexpr int kMaxDevicesCached = 64;
inline int current_device() {
  int d = 0;
  cudaGetDevice(&d);
  return d;
}

moe_status_t launch_permute(const int32_t *topk_idx, const float *topk_w, const void *x,
                            moe_dtype_t dtype, int T, int d, int N, int k, int capacity,
                            int32_t *counts, int32_t *offsets, int32_t *perm_token,
                            float *row_scale, int32_t *inv_pos, void *x_perm,
                            int32_t *dropped, int32_t *device_status, void *workspace,
                            cudaStream_t stream,
                            bool neg_one_drops = false);

// Copies each token's row of x to the positions inv_pos gives its slots
// (-1: dropped), in token order; nothing when x_perm is null.  Rows of
// row_bytes bytes (a multiple of 16).
moe_status_t launch_copy_rows(const void *x, moe_dtype_t dtype, const int32_t *inv_pos, int T,
                              int d, int k, void *x_perm, cudaStream_t stream);
moe_status_t launch_copy_row_bytes(const void *x, size_t row_bytes, const int32_t *inv_pos,
                                   int T, int k, void *x_perm, cudaStream_t stream);

// FP8 E4M3 with absmax scales: rows of x [R, C] bf16 (fp32 with f32_in) ->
// codes [R, C] + [R] scales; gate/up weights W [N, d, f] bf16 -> codes
// [N, f, d] + [N, f].
moe_status_t launch_quantize_rows_e4m3(const void *x, int R, int C, uint8_t *q, float *scale,
                                       cudaStream_t stream, const int32_t *rows_valid = nullptr,
                                       bool f32_in = false);
moe_status_t launch_quantize_weights_e4m3(const void *W, int N, int d, int f, uint8_t *q,
                                          float *scale, cudaStream_t stream);
// The dispatch row copy with the rows quantised on the way (codes of token t
// to every kept slot's permuted row; scale[t] as quantize_rows).
moe_status_t launch_copy_rows_e4m3(const void *x, const int32_t *inv_pos, int T, int d, int k,
                                   uint8_t *x_perm, float *scale, cudaStream_t stream);
// Expert FFN with E4M3 gate/up and, when Wq_down is given, E4M3 down (see
// ffn_tc.cu).  Workspace: ffn_fp8_workspace_bytes.
size_t ffn_fp8_workspace_bytes(int A_max, int f, bool fp8_down);
moe_status_t launch_ffn_tc_fp8(const void *xq_perm, const float *x_scale,
                               const int32_t *perm_token, const int32_t *offsets,
                               const float *row_scale, int A_max, int d, int f, int N,
                               int capacity, const void *Wq_gate, const float *sw_gate,
                               const void *Wq_up, const float *sw_up, const void *W_down,
                               const void *Wq_down, const float *sw_down, void *workspace,
                               void *y_perm, int32_t *device_status, cudaStream_t stream);

size_t ffn_workspace_bytes(int A_max, int d, int f, int N, moe_dtype_t dtype);
// capacity: rows per expert the dispatch kept at most (0 = unknown/none); a
// tiling hint only.
// out_row (nullable): output row p goes to y_perm row out_row[p] (< rows_out).
moe_status_t launch_expert_ffn(const void *x_perm, const int32_t *offsets,
                               const float *row_scale, int A_max, int d, int f, int N,
                               int capacity, moe_dtype_t dtype, const void *W_gate,
                               const void *W_up, const void *W_down, void *y_perm,
                               int32_t *device_status, void *workspace, cudaStream_t stream,
                               const int32_t *out_row = nullptr, int rows_out = 0);

size_t reroute_workspace_bytes(int T, int N, int k);
moe_status_t launch_permute_reroute(const int32_t *cand, const float *cand_w, const void *x,
                                    moe_dtype_t dtype, int T, int d, int N, int k, int R,
                                    int capacity, int32_t *final_idx, float *final_w,
                                    int32_t *demand, int32_t *counts, int32_t *offsets,
                                    int32_t *perm_token, float *row_scale, int32_t *inv_pos,
                                    void *x_perm, int32_t *dropped, int32_t *rerouted,
                                    int32_t *device_status, void *workspace,
                                    cudaStream_t stream);
size_t routing_stats_workspace_bytes(int T, int N);
moe_status_t launch_routing_stats(const float *logits, const int32_t *counts, int T, int N,
                                  moe_routing_stats_t *stats, float *freq, float *prob_mean,
                                  void *workspace, cudaStream_t stream);
moe_status_t launch_combine(const void *y_perm, moe_dtype_t y_perm_dtype,
                            const int32_t *inv_pos, int T, int k, int d,
                            const void *shared_y, void *y, moe_dtype_t y_dtype,
                            cudaStream_t stream);

// fp32 SIMT grouped SwiGLU FFN (any dtype; the fp32 layer's path).
moe_status_t launch_ffn_simt(const void *x_perm, const int32_t *offsets,
                             const float *row_scale, int A_max, int d, int f, int N,
                             moe_dtype_t dtype, const void *W_gate, const void *W_up,
                             const void *W_down, void *h, void *y_perm,
                             int32_t *device_status, cudaStream_t stream,
                             const int32_t *out_row = nullptr, int rows_out = 0);

// bf16 tcgen05 router (returns MOE_ERR_UNSUPPORTED when N does not suit it).
moe_status_t launch_router_tc(const void *x, const void *W_g, const float *bias, int T, int d,
                              int N, int k, float *logits, int32_t *topk_idx, float *topk_w,
                              int32_t *device_status, cudaStream_t stream);

// bf16 tcgen05 grouped SwiGLU FFN (the bf16 layer's path).
// out_row (nullable): output row p goes to y_perm row out_row[p], checked
// against rows_out (MOE_DEV_BAD_ROW).
moe_status_t launch_ffn_tc(const void *x_perm, const int32_t *offsets, const float *row_scale,
                           int A_max, int d, int f, int N, int capacity, const void *W_gate,
                           const void *W_up, const void *W_down, void *h, void *y_perm,
                           int32_t *device_status, cudaStream_t stream,
                           const int32_t *out_row = nullptr, int rows_out = 0);

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Expert parallelism (ep.cu): regroup received rows by local expert, and put
// the expert outputs back in received order.
int ep_max_blocks();
moe_status_t launch_ep_regroup(const int32_t *recv_counts, int G, int Ne, const void *x_recv,
                               const float *row_scale_recv, int R, size_t row_bytes,
                               void *x_local, float *row_scale_local, int32_t *offsets_local,
                               int32_t *dest, int32_t *src_row, int32_t *device_status,
                               cudaStream_t stream);
moe_status_t launch_ep_return(const void *y_local, const int32_t *dest, int R, size_t row_bytes,
                              void *y_back, cudaStream_t stream);

}  // namespace moe
