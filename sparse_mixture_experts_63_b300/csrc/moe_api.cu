// libmoe.so entry points: argument checks, workspace layout and launch order.
// Every compute step runs in the kernels of the other translation units; this
// file only validates, carves the caller's workspace and enqueues launches.
#include <math.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include <atomic>

#include "moe_internal.cuh"

namespace moe {

static thread_local char g_err[512] = "";
static std::atomic<uint64_t> g_launches{0};

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

void set_error(const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof g_err, fmt, ap);
  va_end(ap);
}

namespace {

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline size_t esize(moe_dtype_t t) { return t == MOE_BF16 ? 2 : 4; }
inline bool dtype_ok(moe_dtype_t t) { return t == MOE_F32 || t == MOE_BF16; }

#define CHECK_ARG(cond, ...)              \
  do {                                    \
    if (!(cond)) {                        \
      ::moe::set_error(__VA_ARGS__);      \
      return MOE_ERR_INVALID_ARG;         \
    }                                     \
  } while (0)

// The kernels are built for sm_103a only.
moe_status_t check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    set_error("no CUDA device");
    return MOE_ERR_DEVICE;
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) {
    set_error("device %d is sm_%d%d; libmoe is built for sm_103a (B300) only", dev, major,
              minor);
    return MOE_ERR_DEVICE;
  }
  return MOE_OK;
}

// Sub-allocator over the caller's workspace (256-byte aligned slices).
struct Carve {
  char *base;
  size_t used = 0;
  explicit Carve(void *b) : base(static_cast<char *>(b)) {}
  template <typename T>
  T *take(size_t count) {
    size_t off = used;
    used = align_up(used + count * sizeof(T), 256);
    return base ? reinterpret_cast<T *>(base + off) : nullptr;
  }
  void *take_bytes(size_t bytes) {
    size_t off = used;
    used = align_up(used + bytes, 256);
    return base ? base + off : nullptr;
  }
};

__global__ void set_shared_offsets(int32_t *off, int T) {
  pdl_begin();
  off[0] = 0;
  off[1] = T;
}

long routed_rows_max(int T, int N, int k, int capacity) {
  long a = (long)T * k;
  if (capacity > 0 && (long)N * capacity < a) a = (long)N * capacity;
  return a;
}

struct ForwardLayout {
  int32_t *topk_idx, *counts, *offsets, *inv_pos, *perm_token, *dropped, *sh_offsets;
  float *topk_w, *row_scale;
  void *x_perm, *y_perm, *ffn_ws, *perm_ws, *ys, *sh_ffn_ws;
  float *xs;         // [T] token scales (FP8 gate/up only)
  int32_t *cand;     // [T, k+R] router candidates (re-routing only)
  float *cand_w;     // [T, k+R]
  void *rr_ws;       // re-routing workspace
  size_t bytes;
};

ForwardLayout layout_forward(const moe_forward_args *a, void *ws) {
  ForwardLayout L{};
  Carve c(ws);
  const int cap = moe_capacity(a->capacity_factor, a->T, a->k, a->N);
  const long A_max = routed_rows_max(a->T, a->N, a->k, cap);
  const size_t tk = (size_t)a->T * a->k;
  const size_t es = esize(a->dtype);
  L.topk_idx = a->topk_idx ? a->topk_idx : c.take<int32_t>(tk);
  L.topk_w = a->topk_w ? a->topk_w : c.take<float>(tk);
  L.counts = a->counts ? a->counts : c.take<int32_t>(a->N);
  L.offsets = a->offsets ? a->offsets : c.take<int32_t>(a->N + 1);
  L.inv_pos = a->inv_pos ? a->inv_pos : c.take<int32_t>(tk);
  L.dropped = a->dropped ? a->dropped : c.take<int32_t>(1);
  L.perm_token = c.take<int32_t>(tk);
  L.row_scale = c.take<float>(tk);
  L.x_perm = c.take_bytes((size_t)A_max * a->d * es);   // E4M3 rows use the first half
  if (a->Wq_gate) {
    L.xs = c.take<float>(a->T);
  }
  L.y_perm = c.take_bytes((size_t)A_max * a->d * es);
  L.ffn_ws = c.take_bytes(a->Wq_gate ? ffn_fp8_workspace_bytes((int)A_max, a->f, a->Wq_down != nullptr)
                                     : ffn_workspace_bytes((int)A_max, a->d, a->f, a->N, a->dtype));
  L.perm_ws = c.take_bytes(permute_workspace_bytes(a->T, a->N, a->k));
  if (a->reroute_rounds > 0) {
    const size_t tkr = (size_t)a->T * (a->k + a->reroute_rounds);
    L.cand = c.take<int32_t>(tkr);
    L.cand_w = c.take<float>(tkr);
    L.rr_ws = c.take_bytes(reroute_workspace_bytes(a->T, a->N, a->k));
  }
  if (a->fs > 0) {
    L.sh_offsets = c.take<int32_t>(2);
    L.ys = c.take_bytes((size_t)a->T * a->d * es);
    L.sh_ffn_ws = c.take_bytes(ffn_workspace_bytes(a->T, a->d, a->fs, 1, a->dtype));
  }
  L.bytes = c.used;
  return L;
}

moe_status_t validate_router(const void *x, const void *W_g, moe_dtype_t dtype, int T, int d,
                             int N, int k, const int32_t *topk_idx, const float *topk_w) {
  CHECK_ARG(dtype_ok(dtype), "dtype %d is not MOE_F32 or MOE_BF16", (int)dtype);
  CHECK_ARG(T >= 0 && d >= 8 && N >= 1, "bad sizes T=%d d=%d N=%d", T, d, N);
  CHECK_ARG(k >= 1 && k <= N, "k=%d must satisfy 1 <= k <= N=%d", k, N);
  CHECK_ARG(d % 8 == 0, "d=%d must be a multiple of 8", d);
  if (N > 256 || k > 32) {
    set_error("router supports N <= 256 and k <= 32 (got N=%d k=%d)", N, k);
    return MOE_ERR_UNSUPPORTED;
  }
  CHECK_ARG(T == 0 || (x && W_g && topk_idx && topk_w), "required pointer is NULL");
  CHECK_ARG(aligned16(x), "x must be 16-byte aligned");
  return MOE_OK;
}

moe_status_t validate_ffn(const void *x_perm, const int32_t *offsets, int A_max, int d, int f,
                          int N, moe_dtype_t dtype, const void *Wg, const void *Wu,
                          const void *Wd, const void *y_perm) {
  CHECK_ARG(dtype_ok(dtype), "dtype %d is not MOE_F32 or MOE_BF16", (int)dtype);
  CHECK_ARG(A_max >= 0 && d >= 8 && f >= 8 && N >= 1, "bad sizes A_max=%d d=%d f=%d N=%d",
            A_max, d, f, N);
  CHECK_ARG(d % 8 == 0 && f % 8 == 0, "d=%d and f=%d must be multiples of 8", d, f);
  CHECK_ARG(offsets && Wg && Wu && Wd, "required pointer is NULL");
  CHECK_ARG(A_max == 0 || (x_perm && y_perm), "x_perm / y_perm is NULL");
  CHECK_ARG(aligned16(x_perm) && aligned16(y_perm) && aligned16(Wg) && aligned16(Wu) &&
                aligned16(Wd),
            "tensors must be 16-byte aligned");
  return MOE_OK;
}

constexpr int kMaxChunks = 16;

// Chunks for the overlapped host-buffer call: as many as keep each chunk's
// tensor work at least four times its weight streaming (every chunk reads every
// touched expert's weights again), at most one per 2048 tokens and 16 in all;
// estimated with 274 FLOP per byte (dense bf16 rate over copy bandwidth).  On
// the prefill layer that is 3 chunks, measured best among 1-16.
int auto_chunks(const moe_forward_args *a) {
  const double kFlopPerByte = 274.0;
  const double rows = (double)a->T * a->k;
  const double flop = 6.0 * rows * a->d * a->f + 6.0 * (double)a->T * a->d * a->fs;
  const double touched = rows < a->N ? rows : a->N;
  const double bytes = esize(a->dtype) * (3.0 * a->d * a->f * touched + 3.0 * (double)a->d * a->fs);
  int n = (int)(flop / (4.0 * bytes * kFlopPerByte));
  const int by_tokens = a->T / 2048;
  if (n > by_tokens) n = by_tokens;
  if (n > kMaxChunks) n = kMaxChunks;
  return n < 1 ? 1 : n;
}

// Events of the overlapped call (2 per chunk + 2), made once per thread and
// device.
moe_status_t chunk_events(cudaEvent_t **out) {
  constexpr int kEv = 2 * kMaxChunks + 2;
  thread_local cudaEvent_t ev[kMaxDevicesCached][kEv];
  thread_local bool made[kMaxDevicesCached];
  const int dev = current_device();
  if (dev < 0 || dev >= kMaxDevicesCached) {
    set_error("device index %d above %d", dev, kMaxDevicesCached);
    return MOE_ERR_UNSUPPORTED;
  }
  if (!made[dev]) {
    for (int i = 0; i < kEv; ++i)
      MOE_CUDA_TRY(cudaEventCreateWithFlags(&ev[dev][i], cudaEventDisableTiming));
    made[dev] = true;
  }
  *out = ev[dev];
  return MOE_OK;
}

}  // namespace

size_t ffn_workspace_bytes(int A_max, int d, int f, int N, moe_dtype_t dtype) {
  (void)d;
  (void)N;
  // h [A_max, f] in the layer dtype.
  return align_up((size_t)A_max * f * esize(dtype), 256);
}

moe_status_t launch_expert_ffn(const void *x_perm, const int32_t *offsets, const float *row_scale,
                               int A_max, int d, int f, int N, int capacity, moe_dtype_t dtype,
                               const void *W_gate, const void *W_up, const void *W_down,
                               void *y_perm, int32_t *device_status, void *workspace,
                               cudaStream_t stream, const int32_t *out_row, int rows_out) {
  void *h = workspace;
  if (dtype == MOE_BF16)
    return launch_ffn_tc(x_perm, offsets, row_scale, A_max, d, f, N, capacity, W_gate, W_up,
                         W_down, h, y_perm, device_status, stream, out_row, rows_out);
  return launch_ffn_simt(x_perm, offsets, row_scale, A_max, d, f, N, dtype, W_gate, W_up,
                         W_down, h, y_perm, device_status, stream, out_row, rows_out);
}

}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_DEVICE: return "unsupported or missing device";
  }
  return "unknown status";
}

const char *moe_last_error(void) { return g_err; }

const char *moe_version(void) { return "moe63 1.0 sm_103a"; }

uint64_t moe_launch_counter(void) { return g_launches.load(std::memory_order_relaxed); }

int moe_capacity(float capacity_factor, int T, int k, int N) {
  if (!(capacity_factor > 0.f) || N < 1) return 0;
  return (int)ceil((double)capacity_factor * (double)T * (double)k / (double)N);
}

moe_status_t moe_router_topk(const void *x, const void *W_g, const float *bias,
                             moe_dtype_t dtype, int T, int d, int N, int k, float *logits,
                             int32_t *topk_idx, float *topk_w, int32_t *device_status,
                             void *stream) {
  moe_status_t s = validate_router(x, W_g, dtype, T, d, N, k, topk_idx, topk_w);
  if (s != MOE_OK) return s;
  if ((s = check_device()) != MOE_OK) return s;
  return launch_router_topk(x, W_g, bias, dtype, T, d, N, k, logits, topk_idx, topk_w,
                            device_status, static_cast<cudaStream_t>(stream));
}

size_t moe_permute_workspace_size(int T, int N, int k) {
  if (T < 0 || N < 1 || k < 1) return 0;
  return permute_workspace_bytes(T, N, k);
}

moe_status_t moe_permute(const int32_t *topk_idx, const float *topk_w, const void *x,
                         moe_dtype_t dtype, int T, int d, int N, int k, int capacity,
                         int32_t *counts, int32_t *offsets, int32_t *perm_token,
                         float *row_scale, int32_t *inv_pos, void *x_perm, int32_t *dropped,
                         int32_t *device_status, void *workspace, size_t workspace_bytes,
                         void *stream) {
  CHECK_ARG(dtype_ok(dtype), "dtype %d is not MOE_F32 or MOE_BF16", (int)dtype);
  CHECK_ARG(T >= 0 && N >= 1 && k >= 1 && k <= N && capacity >= 0,
            "bad sizes T=%d N=%d k=%d capacity=%d", T, N, k, capacity);
  CHECK_ARG(counts && offsets && perm_token && inv_pos && (T == 0 || topk_idx),
            "required pointer is NULL");
  CHECK_ARG(!row_scale || topk_w, "row_scale needs topk_w");
  if (x_perm) {
    CHECK_ARG(x && d >= 8 && d % 8 == 0, "x_perm needs x and d %% 8 == 0 (d=%d)", d);
    CHECK_ARG(aligned16(x) && aligned16(x_perm), "x / x_perm must be 16-byte aligned");
  }
  if (N > 1024) {
    set_error("moe_permute supports N <= 1024");
    return MOE_ERR_UNSUPPORTED;
  }
  size_t need = permute_workspace_bytes(T, N, k);
  if (need > 0 && (!workspace || workspace_bytes < need)) {
    set_error("moe_permute: workspace %zu bytes, needs %zu", workspace_bytes, need);
    return MOE_ERR_WORKSPACE;
  }
  moe_status_t s = check_device();
  if (s != MOE_OK) return s;
  return launch_permute(topk_idx, topk_w, x, dtype, T, d, N, k, capacity, counts, offsets,
                        perm_token, row_scale, inv_pos, x_perm, dropped, device_status,
                        workspace, static_cast<cudaStream_t>(stream));
}

size_t moe_expert_ffn_workspace_size(int A_max, int d, int f, int N, moe_dtype_t dtype) {
  if (A_max < 0 || d < 1 || f < 1 || N < 1 || !dtype_ok(dtype)) return 0;
  return ffn_workspace_bytes(A_max, d, f, N, dtype);
}

moe_status_t moe_expert_ffn(const void *x_perm, const int32_t *offsets, const float *row_scale,
                            int A_max, int d, int f, int N, moe_dtype_t dtype,
                            const void *W_gate, const void *W_up, const void *W_down,
                            void *y_perm, int32_t *device_status, void *workspace,
                            size_t workspace_bytes, void *stream) {
  moe_status_t s = validate_ffn(x_perm, offsets, A_max, d, f, N, dtype, W_gate, W_up, W_down,
                                y_perm);
  if (s != MOE_OK) return s;
  size_t need = ffn_workspace_bytes(A_max, d, f, N, dtype);
  if (need > 0 && (!workspace || workspace_bytes < need)) {
    set_error("moe_expert_ffn: workspace %zu bytes, needs %zu", workspace_bytes, need);
    return MOE_ERR_WORKSPACE;
  }
  if ((s = check_device()) != MOE_OK) return s;
  return launch_expert_ffn(x_perm, offsets, row_scale, A_max, d, f, N, 0, dtype, W_gate, W_up,
                           W_down, y_perm, device_status, workspace,
                           static_cast<cudaStream_t>(stream));
}

moe_status_t moe_expert_ffn_to_rows(const void *x_perm, const int32_t *offsets,
                                    const float *row_scale, const int32_t *out_row, int A_max,
                                    int d, int f, int N, moe_dtype_t dtype, const void *W_gate,
                                    const void *W_up, const void *W_down, void *y, int rows_out,
                                    int32_t *device_status, void *workspace,
                                    size_t workspace_bytes, void *stream) {
  moe_status_t s = validate_ffn(x_perm, offsets, A_max, d, f, N, dtype, W_gate, W_up, W_down,
                                y);
  if (s != MOE_OK) return s;
  CHECK_ARG(rows_out >= 0, "rows_out=%d must be >= 0", rows_out);
  CHECK_ARG(A_max == 0 || out_row, "out_row is NULL");
  size_t need = ffn_workspace_bytes(A_max, d, f, N, dtype);
  if (need > 0 && (!workspace || workspace_bytes < need)) {
    set_error("moe_expert_ffn_to_rows: workspace %zu bytes, needs %zu", workspace_bytes, need);
    return MOE_ERR_WORKSPACE;
  }
  if ((s = check_device()) != MOE_OK) return s;
  return launch_expert_ffn(x_perm, offsets, row_scale, A_max, d, f, N, 0, dtype, W_gate, W_up,
                           W_down, y, device_status, workspace,
                           static_cast<cudaStream_t>(stream), out_row, rows_out);
}

moe_status_t moe_quantize_weights_e4m3(const void *W, int N, int d, int f, uint8_t *Wq,
                                       float *scale, void *stream) {
  CHECK_ARG(N >= 1 && d >= 16 && f >= 1 && d % 16 == 0, "bad sizes N=%d d=%d f=%d (d %% 16 == 0)",
            N, d, f);
  CHECK_ARG(W && Wq && scale, "required pointer is NULL");
  CHECK_ARG(aligned16(Wq), "Wq must be 16-byte aligned");
  moe_status_t s = check_device();
  if (s != MOE_OK) return s;
  return launch_quantize_weights_e4m3(W, N, d, f, Wq, scale, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_quantize_rows_e4m3(const void *x, int R, int C, uint8_t *q, float *scale,
                                    void *stream) {
  CHECK_ARG(R >= 0 && C >= 16 && C % 16 == 0, "bad sizes R=%d C=%d (C %% 16 == 0)", R, C);
  CHECK_ARG(R == 0 || (x && q && scale), "required pointer is NULL");
  CHECK_ARG(aligned16(x) && aligned16(q), "x and q must be 16-byte aligned");
  moe_status_t s = check_device();
  if (s != MOE_OK) return s;
  return launch_quantize_rows_e4m3(x, R, C, q, scale, static_cast<cudaStream_t>(stream));
}

size_t moe_expert_ffn_fp8_workspace_size(int A_max, int d, int f, int N, int fp8_down) {
  if (A_max < 0 || d < 1 || f < 1 || N < 1) return 0;
  return ffn_fp8_workspace_bytes(A_max, f, fp8_down != 0);
}

moe_status_t moe_expert_ffn_fp8(const uint8_t *xq_perm, const float *x_scale,
                                const int32_t *perm_token, const int32_t *offsets,
                                const float *row_scale, int A_max, int d, int f, int N,
                                const uint8_t *Wq_gate, const float *wscale_gate,
                                const uint8_t *Wq_up, const float *wscale_up,
                                const void *W_down, const uint8_t *Wq_down,
                                const float *wscale_down, void *y_perm,
                                int32_t *device_status, void *workspace,
                                size_t workspace_bytes, void *stream) {
  CHECK_ARG(A_max >= 0 && d >= 16 && f >= 16 && N >= 1, "bad sizes A_max=%d d=%d f=%d N=%d",
            A_max, d, f, N);
  CHECK_ARG(d % 16 == 0 && f % 8 == 0, "d=%d must be a multiple of 16 and f=%d of 8", d, f);
  CHECK_ARG(!Wq_down || f % 16 == 0, "an E4M3 down projection needs f %% 16 == 0 (f=%d)", f);
  CHECK_ARG(offsets && Wq_gate && Wq_up && wscale_gate && wscale_up,
            "required pointer is NULL");
  CHECK_ARG(Wq_down ? wscale_down != nullptr : W_down != nullptr,
            "the down projection needs W_down, or Wq_down with wscale_down");
  CHECK_ARG(A_max == 0 || (xq_perm && x_scale && perm_token && y_perm),
            "required pointer is NULL");
  CHECK_ARG(aligned16(xq_perm) && aligned16(y_perm) && aligned16(Wq_gate) && aligned16(Wq_up) &&
                aligned16(W_down) && aligned16(Wq_down),
            "tensors must be 16-byte aligned");
  size_t need = ffn_fp8_workspace_bytes(A_max, f, Wq_down != nullptr);
  if (need > 0 && (!workspace || workspace_bytes < need)) {
    set_error("moe_expert_ffn_fp8: workspace %zu bytes, needs %zu", workspace_bytes, need);
    return MOE_ERR_WORKSPACE;
  }
  moe_status_t s = check_device();
  if (s != MOE_OK) return s;
  return launch_ffn_tc_fp8(xq_perm, x_scale, perm_token, offsets, row_scale, A_max, d, f, N, 0,
                           Wq_gate, wscale_gate, Wq_up, wscale_up, W_down, Wq_down, wscale_down,
                           workspace, y_perm, device_status, static_cast<cudaStream_t>(stream));
}

size_t moe_permute_reroute_workspace_size(int T, int N, int k, int R) {
  if (T < 0 || N < 1 || k < 1 || R < 0) return 0;
  return reroute_workspace_bytes(T, N, k);
}

moe_status_t moe_permute_reroute(const int32_t *cand_idx, const float *cand_w, const void *x,
                                 moe_dtype_t dtype, int T, int d, int N, int k, int R,
                                 int capacity, int32_t *final_idx, float *final_w,
                                 int32_t *demand, int32_t *counts, int32_t *offsets,
                                 int32_t *perm_token, float *row_scale, int32_t *inv_pos,
                                 void *x_perm, int32_t *dropped, int32_t *rerouted,
                                 int32_t *device_status, void *workspace,
                                 size_t workspace_bytes, void *stream) {
  CHECK_ARG(dtype_ok(dtype), "dtype %d is not MOE_F32 or MOE_BF16", (int)dtype);
  CHECK_ARG(T >= 0 && N >= 1 && k >= 1 && R >= 0 && k + R <= N && capacity >= 1,
            "bad sizes T=%d N=%d k=%d R=%d capacity=%d (need k+R <= N, capacity >= 1)", T, N,
            k, R, capacity);
  CHECK_ARG(counts && offsets && perm_token && inv_pos && final_idx && final_w &&
                (T == 0 || (cand_idx && cand_w)),
            "required pointer is NULL");
  if (x_perm) {
    CHECK_ARG(x && d >= 8 && d % 8 == 0, "x_perm needs x and d %% 8 == 0 (d=%d)", d);
    CHECK_ARG(aligned16(x) && aligned16(x_perm), "x / x_perm must be 16-byte aligned");
  }
  if (N > 1024) {
    set_error("moe_permute_reroute supports N <= 1024");
    return MOE_ERR_UNSUPPORTED;
  }
  const size_t need = reroute_workspace_bytes(T, N, k);
  if (!workspace || workspace_bytes < need) {
    set_error("moe_permute_reroute: workspace %zu bytes, needs %zu", workspace_bytes, need);
    return MOE_ERR_WORKSPACE;
  }
  moe_status_t s = check_device();
  if (s != MOE_OK) return s;
  return launch_permute_reroute(cand_idx, cand_w, x, dtype, T, d, N, k, R, capacity, final_idx,
                                final_w, demand, counts, offsets, perm_token, row_scale,
                                inv_pos, x_perm, dropped, rerouted, device_status, workspace,
                                static_cast<cudaStream_t>(stream));
}

size_t moe_routing_stats_workspace_size(int T, int N) {
  if (T < 0 || N < 1) return 0;
  return routing_stats_workspace_bytes(T, N);
}

moe_status_t moe_routing_stats(const float *logits, const int32_t *counts, int T, int N,
                               moe_routing_stats_t *stats, float *freq, float *prob_mean,
                               void *workspace, size_t workspace_bytes, void *stream) {
  CHECK_ARG(T >= 0 && N >= 1 && N <= 1024, "bad sizes T=%d N=%d (N <= 1024)", T, N);
  CHECK_ARG(counts && stats, "counts and stats are required");
  if (logits && T > 0) {
    const size_t need = routing_stats_workspace_bytes(T, N);
    if (!workspace || workspace_bytes < need) {
      set_error("moe_routing_stats: workspace %zu bytes, needs %zu", workspace_bytes, need);
      return MOE_ERR_WORKSPACE;
    }
  }
  moe_status_t s = check_device();
  if (s != MOE_OK) return s;
  return launch_routing_stats(logits, counts, T, N, stats, freq, prob_mean, workspace,
                              static_cast<cudaStream_t>(stream));
}

moe_status_t moe_combine(const void *y_perm, moe_dtype_t y_perm_dtype, const int32_t *inv_pos,
                         int T, int k, int d, const void *shared_y, void *y, moe_dtype_t y_dtype,
                         void *stream) {
  CHECK_ARG(dtype_ok(y_perm_dtype) && dtype_ok(y_dtype), "bad dtype");
  CHECK_ARG(T >= 0 && k >= 1 && d >= 8 && d % 8 == 0, "bad sizes T=%d k=%d d=%d", T, k, d);
  CHECK_ARG(T == 0 || (y_perm && inv_pos && y), "required pointer is NULL");
  CHECK_ARG(aligned16(y_perm) && aligned16(shared_y) && aligned16(y),
            "tensors must be 16-byte aligned");
  moe_status_t s = check_device();
  if (s != MOE_OK) return s;
  return launch_combine(y_perm, y_perm_dtype, inv_pos, T, k, d, shared_y, y, y_dtype,
                        static_cast<cudaStream_t>(stream));
}

moe_status_t moe_ep_regroup(const int32_t *recv_counts, int G, int Ne, const void *x_recv,
                            const float *row_scale_recv, int R, int d, moe_dtype_t dtype,
                            void *x_local, float *row_scale_local, int32_t *offsets_local,
                            int32_t *dest, int32_t *src, int32_t *device_status, void *stream) {
  CHECK_ARG(dtype_ok(dtype), "bad dtype");
  CHECK_ARG(G >= 1 && Ne >= 1 && R >= 0 && d >= 1, "bad sizes G=%d Ne=%d R=%d d=%d", G, Ne, R, d);
  if ((long)G * Ne > ep_max_blocks()) {
    set_error("moe_ep_regroup: G*Ne = %ld exceeds %d", (long)G * Ne, ep_max_blocks());
    return MOE_ERR_UNSUPPORTED;
  }
  CHECK_ARG(((size_t)d * esize(dtype)) % 16 == 0, "rows must be a multiple of 16 bytes (d=%d)", d);
  CHECK_ARG(recv_counts && offsets_local && (R == 0 || (x_recv && x_local && dest)),
            "required pointer is NULL");
  CHECK_ARG(!row_scale_recv || row_scale_local || R == 0, "row_scale_local is NULL");
  CHECK_ARG(aligned16(x_recv) && aligned16(x_local), "tensors must be 16-byte aligned");
  moe_status_t s = check_device();
  if (s != MOE_OK) return s;
  return launch_ep_regroup(recv_counts, G, Ne, x_recv, row_scale_recv, R,
                           (size_t)d * esize(dtype), x_local, row_scale_local, offsets_local,
                           dest, src, device_status, static_cast<cudaStream_t>(stream));
}

moe_status_t moe_ep_return(const void *y_local, const int32_t *dest, int R, int d,
                           moe_dtype_t dtype, void *y_back, void *stream) {
  CHECK_ARG(dtype_ok(dtype), "bad dtype");
  CHECK_ARG(R >= 0 && d >= 1, "bad sizes R=%d d=%d", R, d);
  CHECK_ARG(((size_t)d * esize(dtype)) % 16 == 0, "rows must be a multiple of 16 bytes (d=%d)", d);
  CHECK_ARG(R == 0 || (y_local && dest && y_back), "required pointer is NULL");
  CHECK_ARG(aligned16(y_local) && aligned16(y_back), "tensors must be 16-byte aligned");
  moe_status_t s = check_device();
  if (s != MOE_OK) return s;
  return launch_ep_return(y_local, dest, R, (size_t)d * esize(dtype), y_back,
                          static_cast<cudaStream_t>(stream));
}

static moe_status_t validate_forward(const moe_forward_args *a) {
  CHECK_ARG(a, "args is NULL");
  CHECK_ARG(dtype_ok(a->dtype) && dtype_ok(a->y_dtype), "bad dtype");
  CHECK_ARG(a->T >= 1 && a->d >= 8 && a->f >= 8 && a->N >= 1, "bad sizes T=%d d=%d f=%d N=%d",
            a->T, a->d, a->f, a->N);
  CHECK_ARG(a->k >= 1 && a->k <= a->N, "k=%d must satisfy 1 <= k <= N=%d", a->k, a->N);
  CHECK_ARG(a->d % 8 == 0 && a->f % 8 == 0, "d=%d and f=%d must be multiples of 8", a->d, a->f);
  CHECK_ARG(a->fs >= 0 && a->fs % 8 == 0, "fs=%d must be a non-negative multiple of 8", a->fs);
  const bool fp8 = a->Wq_gate || a->Wq_up || a->wscale_gate || a->wscale_up;
  CHECK_ARG(a->x && a->W_g && (fp8 || (a->W_gate && a->W_up)) && (a->W_down || a->Wq_down) &&
                a->y,
            "required pointer is NULL");
  CHECK_ARG(!a->Wq_down || (fp8 && a->wscale_down && a->f % 16 == 0 && aligned16(a->Wq_down)),
            "an E4M3 down projection needs the E4M3 gate/up, wscale_down and f %% 16 == 0");
  if (fp8) {
    CHECK_ARG(a->Wq_gate && a->Wq_up && a->wscale_gate && a->wscale_up,
              "FP8 gate/up needs Wq_gate, Wq_up, wscale_gate and wscale_up");
    CHECK_ARG(a->dtype == MOE_BF16, "FP8 gate/up needs a bf16 layer");
    CHECK_ARG(a->d % 16 == 0, "FP8 gate/up needs d %% 16 == 0 (d=%d)", a->d);
    CHECK_ARG(aligned16(a->Wq_gate) && aligned16(a->Wq_up), "tensors must be 16-byte aligned");
  }
  CHECK_ARG(a->fs == 0 || (a->Ws_gate && a->Ws_up && a->Ws_down), "shared weights are NULL");
  CHECK_ARG(aligned16(a->x) && aligned16(a->y) && aligned16(a->W_gate) && aligned16(a->W_up) &&
                aligned16(a->W_down) && aligned16(a->Ws_gate) && aligned16(a->Ws_up) &&
                aligned16(a->Ws_down),
            "tensors must be 16-byte aligned");
  CHECK_ARG((long)a->T * a->k < (1L << 31) - 1, "T*k too large");
  if (a->N > 256 || a->k > 32) {
    set_error("N <= 256 and k <= 32 are supported (got N=%d k=%d)", a->N, a->k);
    return MOE_ERR_UNSUPPORTED;
  }
  CHECK_ARG(a->reroute_rounds >= 0, "reroute_rounds=%d must be >= 0", a->reroute_rounds);
  if (a->reroute_rounds > 0) {
    CHECK_ARG(a->capacity_factor > 0, "re-routing needs a capacity (capacity_factor > 0)");
    CHECK_ARG(a->k + a->reroute_rounds <= a->N, "k + reroute_rounds = %d exceeds N = %d",
              a->k + a->reroute_rounds, a->N);
    if (a->k + a->reroute_rounds > 32) {
      set_error("k + reroute_rounds <= 32 is supported (got %d)", a->k + a->reroute_rounds);
      return MOE_ERR_UNSUPPORTED;
    }
  }
  return MOE_OK;
}

size_t moe_forward_workspace_size(const moe_forward_args *args) {
  if (validate_forward(args) != MOE_OK) return 0;
  return layout_forward(args, nullptr).bytes;
}

moe_status_t moe_forward(const moe_forward_args *a, void *workspace, size_t workspace_bytes,
                         void *stream_) {
  moe_status_t s = validate_forward(a);
  if (s != MOE_OK) return s;
  ForwardLayout need = layout_forward(a, nullptr);
  if (!workspace || workspace_bytes < need.bytes) {
    set_error("moe_forward: workspace %zu bytes, needs %zu", workspace_bytes, need.bytes);
    return MOE_ERR_WORKSPACE;
  }
  if (!aligned16(workspace)) {
    set_error("workspace must be 16-byte aligned");
    return MOE_ERR_INVALID_ARG;
  }
  if ((s = check_device()) != MOE_OK) return s;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  ForwardLayout L = layout_forward(a, workspace);
  const int cap = moe_capacity(a->capacity_factor, a->T, a->k, a->N);
  const int A_max = (int)routed_rows_max(a->T, a->N, a->k, cap);
  const bool fp8 = a->Wq_gate != nullptr;
  void *x_perm = fp8 ? nullptr : L.x_perm;   // FP8: the rows are quantised as they are copied

  if (a->reroute_rounds > 0) {
    // the router ranks k+R candidates; the dispatch re-routes overflow to them
    const int kr = a->k + a->reroute_rounds;
    s = launch_router_topk(a->x, a->W_g, a->router_bias, a->dtype, a->T, a->d, a->N, kr,
                           a->logits, L.cand, L.cand_w, a->device_status, stream);
    if (s != MOE_OK) return s;
    s = launch_permute_reroute(L.cand, L.cand_w, a->x, a->dtype, a->T, a->d, a->N, a->k,
                               a->reroute_rounds, cap, L.topk_idx, L.topk_w, nullptr, L.counts,
                               L.offsets, L.perm_token, L.row_scale, L.inv_pos, x_perm,
                               L.dropped, a->rerouted, a->device_status, L.rr_ws, stream);
    if (s != MOE_OK) return s;
  } else {
    s = launch_router_topk(a->x, a->W_g, a->router_bias, a->dtype, a->T, a->d, a->N, a->k,
                           a->logits, L.topk_idx, L.topk_w, a->device_status, stream);
    if (s != MOE_OK) return s;
    s = launch_permute(L.topk_idx, L.topk_w, a->x, a->dtype, a->T, a->d, a->N, a->k, cap,
                       L.counts, L.offsets, L.perm_token, L.row_scale, L.inv_pos, x_perm,
                       L.dropped, a->device_status, L.perm_ws, stream);
    if (s != MOE_OK) return s;
    if (a->rerouted) MOE_CUDA_TRY(cudaMemsetAsync(a->rerouted, 0, sizeof(int32_t), stream));
  }
  if (fp8) {
    // E4M3 gate/up: the dispatched rows are the quantised token rows
    s = launch_copy_rows_e4m3(a->x, L.inv_pos, a->T, a->d, a->k,
                              static_cast<uint8_t *>(L.x_perm), L.xs, stream);
    if (s != MOE_OK) return s;
  }
  if (a->ffn_event_begin)
    MOE_CUDA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(a->ffn_event_begin), stream));
  if (fp8) {
    s = launch_ffn_tc_fp8(L.x_perm, L.xs, L.perm_token, L.offsets, L.row_scale, A_max, a->d,
                          a->f, a->N, cap, a->Wq_gate, a->wscale_gate, a->Wq_up, a->wscale_up,
                          a->W_down, a->Wq_down, a->wscale_down, L.ffn_ws, L.y_perm,
                          a->device_status, stream);
  } else {
    s = launch_expert_ffn(L.x_perm, L.offsets, L.row_scale, A_max, a->d, a->f, a->N, cap,
                          a->dtype, a->W_gate, a->W_up, a->W_down, L.y_perm, a->device_status,
                          L.ffn_ws, stream);
  }
  if (s != MOE_OK) return s;
  if (a->ffn_event_end)
    MOE_CUDA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(a->ffn_event_end), stream));
  if (a->fs > 0) {
    MOE_CUDA_TRY(launch_pdl(set_shared_offsets, dim3(1), dim3(1), 0, stream, L.sh_offsets, a->T));
    MOE_LAUNCH_CHECK();
    s = launch_expert_ffn(a->x, L.sh_offsets, nullptr, a->T, a->d, a->fs, 1, 0, a->dtype,
                          a->Ws_gate, a->Ws_up, a->Ws_down, L.ys, a->device_status,
                          L.sh_ffn_ws, stream);
    if (s != MOE_OK) return s;
  }
  return launch_combine(L.y_perm, a->dtype, L.inv_pos, a->T, a->k, a->d,
                        a->fs > 0 ? L.ys : nullptr, a->y, a->y_dtype, stream);
}

moe_status_t moe_forward_host_io(const moe_forward_args *a, const void *x_host, void *y_host,
                                 void *workspace, size_t workspace_bytes, void *stream_) {
  moe_status_t s = validate_forward(a);
  if (s != MOE_OK) return s;
  CHECK_ARG(x_host && y_host, "host buffers are NULL");
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  const size_t xb = (size_t)a->T * a->d * esize(a->dtype);
  const size_t yb = (size_t)a->T * a->d * esize(a->y_dtype);
  MOE_CUDA_TRY(cudaMemcpyAsync(const_cast<void *>(a->x), x_host, xb, cudaMemcpyHostToDevice,
                               stream));
  s = moe_forward(a, workspace, workspace_bytes, stream_);
  if (s != MOE_OK) return s;
  MOE_CUDA_TRY(cudaMemcpyAsync(y_host, a->y, yb, cudaMemcpyDeviceToHost, stream));
  return MOE_OK;
}

int moe_forward_overlap_chunks(const moe_forward_args *a) {
  if (validate_forward(a) != MOE_OK) return 0;
  return auto_chunks(a);
}

moe_status_t moe_forward_host_io_overlapped(const moe_forward_args *a, const void *x_host,
                                            void *y_host, void *workspace,
                                            size_t workspace_bytes, int chunks, void *stream_,
                                            void *h2d_stream_, void *d2h_stream_) {
  moe_status_t s = validate_forward(a);
  if (s != MOE_OK) return s;
  CHECK_ARG(x_host && y_host, "host buffers are NULL");
  CHECK_ARG(h2d_stream_ && d2h_stream_ && h2d_stream_ != stream_ && d2h_stream_ != stream_ &&
                h2d_stream_ != d2h_stream_,
            "three distinct streams are needed");
  CHECK_ARG(!a->logits && !a->topk_idx && !a->topk_w && !a->counts && !a->offsets &&
                !a->inv_pos && !a->dropped && !a->rerouted,
            "the overlapped call returns y only: routing outputs must be NULL");
  ForwardLayout need = layout_forward(a, nullptr);
  if (!workspace || workspace_bytes < need.bytes) {
    set_error("moe_forward_host_io_overlapped: workspace %zu bytes, needs %zu",
              workspace_bytes, need.bytes);
    return MOE_ERR_WORKSPACE;
  }
  if ((s = check_device()) != MOE_OK) return s;
  int n = chunks > 0 ? chunks : auto_chunks(a);
  if (a->capacity_factor > 0 || a->reroute_rounds > 0) n = 1;   // drops depend on the batch
  if (n > kMaxChunks) n = kMaxChunks;
  if (n > a->T) n = a->T;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_);
  cudaStream_t h2d = static_cast<cudaStream_t>(h2d_stream_);
  cudaStream_t d2h = static_cast<cudaStream_t>(d2h_stream_);
  cudaEvent_t *ev = nullptr;
  if ((s = chunk_events(&ev)) != MOE_OK) return s;   // [0] start, [1..n] h2d, [n+1..2n] layer
  const size_t xr = (size_t)a->d * esize(a->dtype), yr = (size_t)a->d * esize(a->y_dtype);
  // Chunk c covers tokens [start[c], start[c+1]).  With three or more chunks
  // the first and the last are half the size of the others: the first one's
  // copy in and the last one's copy out are the parts no compute hides.
  int start[kMaxChunks + 1];
  {
    const double wsum = n >= 3 ? (double)(n - 1) : (double)n;   // 0.5 + (n-2) + 0.5
    double acc = 0.0;
    start[0] = 0;
    for (int c = 0; c < n; ++c) {
      acc += (n >= 3 && (c == 0 || c == n - 1)) ? 0.5 : 1.0;
      start[c + 1] = c + 1 == n ? a->T : (int)((double)a->T * acc / wsum + 0.5);
    }
    bool empty = false;
    for (int c = 0; c < n; ++c) empty = empty || start[c + 1] <= start[c];
    if (empty) {                               // tiny batches: equal chunks, none empty
      const int Tc = (a->T + n - 1) / n;
      n = (a->T + Tc - 1) / Tc;
      for (int c = 0; c <= n; ++c) start[c] = c * Tc < a->T ? c * Tc : a->T;
    }
  }
  // the copies start after the caller's earlier work on `stream`
  MOE_CUDA_TRY(cudaEventRecord(ev[0], stream));
  MOE_CUDA_TRY(cudaStreamWaitEvent(h2d, ev[0], 0));
  MOE_CUDA_TRY(cudaStreamWaitEvent(d2h, ev[0], 0));
  for (int c = 0; c < n; ++c) {
    const size_t t0 = (size_t)start[c], tc = (size_t)(start[c + 1] - start[c]);
    MOE_CUDA_TRY(cudaMemcpyAsync(static_cast<char *>(const_cast<void *>(a->x)) + t0 * xr,
                                 static_cast<const char *>(x_host) + t0 * xr, tc * xr,
                                 cudaMemcpyHostToDevice, h2d));
    MOE_CUDA_TRY(cudaEventRecord(ev[1 + c], h2d));
  }
  for (int c = 0; c < n; ++c) {
    const size_t t0 = (size_t)start[c], tc = (size_t)(start[c + 1] - start[c]);
    moe_forward_args ac = *a;
    ac.T = (int)tc;
    ac.x = static_cast<const char *>(a->x) + t0 * xr;
    ac.y = static_cast<char *>(a->y) + t0 * yr;
    ac.ffn_event_begin = ac.ffn_event_end = nullptr;   // one layer call spans several chunks
    MOE_CUDA_TRY(cudaStreamWaitEvent(stream, ev[1 + c], 0));
    s = moe_forward(&ac, workspace, workspace_bytes, stream_);
    if (s != MOE_OK) return s;
    MOE_CUDA_TRY(cudaEventRecord(ev[1 + n + c], stream));
    MOE_CUDA_TRY(cudaStreamWaitEvent(d2h, ev[1 + n + c], 0));
    MOE_CUDA_TRY(cudaMemcpyAsync(static_cast<char *>(y_host) + t0 * yr,
                                 static_cast<const char *>(ac.y), tc * yr, cudaMemcpyDeviceToHost,
                                 d2h));
  }
  // `stream` covers the whole call: it waits for the last copy back
  MOE_CUDA_TRY(cudaEventRecord(ev[2 * n + 1], d2h));
  MOE_CUDA_TRY(cudaStreamWaitEvent(stream, ev[2 * n + 1], 0));
  return MOE_OK;
}

}  // extern "C"
