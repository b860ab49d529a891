// Router: logits = x W_g (+ b), top-k by (logit desc, expert id asc), softmax
// over the k selected logits.
//
// Source: "MoE 分片：混合專家模型的平行化策略", section 動態 token 路由, step 2
// (the router scores all N experts, keeps the top-k) and step 6 (the k outputs
// are combined with the router's normalised scores, e.g. 0.6 / 0.4);
// "MoE 推理：激活参数 vs 总参数与专家路由", section 深入原理 (a linear layer
// gives N gate logits; top-k softmax gives the weights).
//
// Two kernels:
//   * router_small_n: N <= 32.  One warp per token; W_g staged once per CTA in
//     shared memory; each lane accumulates all N dot products over its slice of
//     d with 16-byte loads of x, then a butterfly reduction.  Used for the
//     8-expert layers (x read once: HBM-bound).
//   * router_tiled:   N <= 256.  A CTA computes a 32-token x N tile with a
//     register micro-tile on the CUDA cores (fp32 FFMA), then one warp per
//     token runs the top-k.
// Both finish with the same warp-wide top-k/softmax (warp_topk_softmax).
#include <float.h>
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kWarp = 32;

// Ranking key: NaN ranks below every number (treated as -inf).
__device__ __forceinline__ float rank_key(float v) { return isnan(v) ? -INFINITY : v; }

// Does candidate (va, ia) rank before (vb, ib)?  Larger key first, then lower id.
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  float ka = rank_key(va), kb = rank_key(vb);
  if (ka != kb) return ka > kb;
  return ia < ib;
}

// Each lane offers up to C candidates (logit v[c], expert id e[c], e < 0 = none).
// Writes topk_idx/topk_w for one token.  Returns true if a NaN was seen.
template <int C>
__device__ __forceinline__ bool warp_topk_softmax(float (&v)[C], int (&e)[C], int k, int lane,
                                                  int32_t *out_idx, float *out_w) {
  bool nan_seen = false;
#pragma unroll
  for (int c = 0; c < C; ++c) nan_seen |= (e[c] >= 0 && isnan(v[c]));
  float my_v = 0.f;
  int my_i = -1;
  for (int j = 0; j < k; ++j) {
    // Best candidate of this lane.
    float bv = -INFINITY;
    int bi = INT_MAX;
#pragma unroll
    for (int c = 0; c < C; ++c)
      if (e[c] >= 0 && ranks_before(v[c], e[c], bv, bi)) { bv = v[c]; bi = e[c]; }
    // Warp-wide best.
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, off);
      int oi = __shfl_xor_sync(0xffffffffu, bi, off);
      if (ranks_before(ov, oi, bv, bi)) { bv = ov; bi = oi; }
    }
    // Slot j is recorded by lane j; the owner drops the winner from its list.
    if (lane == j) { my_v = bv; my_i = bi; }
#pragma unroll
    for (int c = 0; c < C; ++c)
      if (e[c] == bi) e[c] = -1;
  }
  float v0 = __shfl_sync(0xffffffffu, my_v, 0);
  float ex = (lane < k) ? expf(my_v - v0) : 0.f;
  float s = ex;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (lane < k) {
    out_idx[lane] = my_i;
    out_w[lane] = ex / s;
  }
  return nan_seen;
}

// ---------------------------------------------------------------------------
// N <= NP <= 32: one warp per token.
// ---------------------------------------------------------------------------
template <typename T, int NP>
__global__ void __launch_bounds__(256) router_small_n(const T *__restrict__ x,
                                                      const T *__restrict__ Wg,
                                                      const float *__restrict__ bias, int Tn,
                                                      int d, int N, int k, float *logits,
                                                      int32_t *topk_idx, float *topk_w,
                                                      int32_t *status) {
  pdl_begin();
  extern __shared__ __align__(16) unsigned char smem_raw[];
  T *ws = reinterpret_cast<T *>(smem_raw);  // [d][NP], zero-padded experts
  if (N == NP && (reinterpret_cast<uintptr_t>(Wg) & 15) == 0) {
    // no padding: a straight copy in 16-byte vectors, several in flight
    const uint4 *src = reinterpret_cast<const uint4 *>(Wg);
    uint4 *dst = reinterpret_cast<uint4 *>(ws);
    const int n16 = (int)((size_t)d * NP * sizeof(T) / 16);
#pragma unroll 4
    for (int i = threadIdx.x; i < n16; i += blockDim.x) dst[i] = __ldg(src + i);
  } else {
    for (int i = threadIdx.x; i < d * NP; i += blockDim.x) {
      int r = i / NP, c = i % NP;
      ws[i] = c < N ? Wg[(size_t)r * N + c] : from_f32<T>(0.f);
    }
  }
  __syncthreads();
  const int lane = threadIdx.x % kWarp;
  const int warps = blockDim.x / kWarp;
  bool nan_seen = false;
  for (int t = blockIdx.x * warps + threadIdx.x / kWarp; t < Tn; t += gridDim.x * warps) {
    const T *xr = x + (size_t)t * d;
    float acc[NP];
#pragma unroll
    for (int c = 0; c < NP; ++c) acc[c] = 0.f;
    // four 16-byte loads of x in flight per lane before the math (one at a
    // time, a decode-sized batch waited on DRAM latency 16 times per token)
    constexpr int kX = 4;
    for (int i0 = lane * 8; i0 < d; i0 += kWarp * 8 * kX) {
      float xv[kX][8];
#pragma unroll
      for (int q = 0; q < kX; ++q) {
        const int ii = i0 + q * kWarp * 8;
        if (ii < d) {
          load8(xr + ii, xv[q]);
        } else {
#pragma unroll
          for (int u = 0; u < 8; ++u) xv[q][u] = 0.f;
        }
      }
#pragma unroll
      for (int q = 0; q < kX; ++q) {
        const int ii = i0 + q * kWarp * 8;
        if (ii >= d) break;
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const T *wr = ws + (size_t)(ii + u) * NP;
#pragma unroll
          for (int c = 0; c < NP; c += 8) {
            float wv[8];
            load8(wr + c, wv);
#pragma unroll
            for (int r = 0; r < 8; ++r) acc[c + r] = fmaf(xv[q][u], wv[r], acc[c + r]);
          }
        }
      }
    }
#pragma unroll
    for (int c = 0; c < NP; ++c) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], off);
    }
    // Lane c holds expert c's logit.
    float v[1];
    int e[1];
    float mine = 0.f;
#pragma unroll
    for (int c = 0; c < NP; ++c)
      if (lane == c) mine = acc[c];
    e[0] = lane < N ? lane : -1;
    if (bias && lane < N) mine += bias[lane];
    v[0] = mine;
    if (logits && lane < N) logits[(size_t)t * N + lane] = mine;
    nan_seen |= warp_topk_softmax<1>(v, e, k, lane, topk_idx + (size_t)t * k,
                                     topk_w + (size_t)t * k);
  }
  if (nan_seen) report(status, MOE_DEV_NAN_LOGIT);
}

// ---------------------------------------------------------------------------
// Decode-sized batches (T <= 512, N <= 32): one CTA of kDecWarps warps per
// token, the warps splitting d; W_g is read from L2 (it is small and every
// token's CTA reads it), x once.  Lane partials are summed over the warp, the
// warps' sums in warp order in shared memory, then warp 0 ranks.  Each lane
// keeps all its 16-byte loads of a step in flight, so a token waits on memory
// a few times, not once per step of d.
// ---------------------------------------------------------------------------
constexpr int kDecWarps = 4;

template <typename T, int NP>
__global__ void __launch_bounds__(kDecWarps * 32) router_decode(
    const T *__restrict__ x, const T *__restrict__ Wg, const float *__restrict__ bias, int Tn,
    int d, int N, int k, float *logits, int32_t *topk_idx, float *topk_w, int32_t *status) {
  pdl_begin();
  __shared__ float part[kDecWarps][NP];
  const int t = blockIdx.x;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const T *xr = x + (size_t)t * d;
  float acc[NP];
#pragma unroll
  for (int c = 0; c < NP; ++c) acc[c] = 0.f;
  const bool vec = (N == NP) && ((reinterpret_cast<uintptr_t>(Wg) & 15) == 0);
  // lane (warp w) takes 8 consecutive columns of d at i0 = 8 * (w * 32 + lane) + step
#pragma unroll 4
  for (int i0 = 8 * (warp * 32 + lane); i0 < d; i0 += 8 * 32 * kDecWarps) {
    float xv[8];
    load8(xr + i0, xv);
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const T *wr = Wg + (size_t)(i0 + u) * N;
      if (vec) {
#pragma unroll
        for (int c = 0; c < NP; c += 8) {
          float wv[8];
          load8(wr + c, wv);
#pragma unroll
          for (int q = 0; q < 8; ++q) acc[c + q] = fmaf(xv[u], wv[q], acc[c + q]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < NP; ++c)
          if (c < N) acc[c] = fmaf(xv[u], to_f32(wr[c]), acc[c]);
      }
    }
  }
#pragma unroll
  for (int c = 0; c < NP; ++c) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc[c] += __shfl_xor_sync(0xffffffffu, acc[c], off);
  }
  if (lane == 0) {
#pragma unroll
    for (int c = 0; c < NP; ++c) part[warp][c] = acc[c];
  }
  __syncthreads();
  if (warp != 0) return;
  float mine = 0.f;
  if (lane < N) {
    for (int w = 0; w < kDecWarps; ++w) mine += part[w][lane];
    if (bias) mine += bias[lane];
    if (logits) logits[(size_t)t * N + lane] = mine;
  }
  float v[1] = {mine};
  int e[1] = {lane < N ? lane : -1};
  const bool nan_seen = warp_topk_softmax<1>(v, e, k, lane, topk_idx + (size_t)t * k,
                                             topk_w + (size_t)t * k);
  if (nan_seen) report(status, MOE_DEV_NAN_LOGIT);
}

// ---------------------------------------------------------------------------
// N <= NP <= 256: 32-token x NP tile per CTA, fp32 FFMA micro-tiles.
// Thread (ty, tx), ty < 8, tx < 32: tokens ty + 8i (i < 4), experts tx + 32j.
// ---------------------------------------------------------------------------
constexpr int kTM = 32;  // tokens per CTA
constexpr int kKC = 32;  // d-chunk staged in shared memory

template <typename T, int NP>
__global__ void __launch_bounds__(256) router_tiled(const T *__restrict__ x,
                                                    const T *__restrict__ Wg,
                                                    const float *__restrict__ bias, int Tn, int d,
                                                    int N, int k, float *logits,
                                                    int32_t *topk_idx, float *topk_w,
                                                    int32_t *status) {
  pdl_begin();
  constexpr int EJ = NP / kWarp;  // experts per thread
  __shared__ float xs[kTM][kKC + 1];
  __shared__ __align__(16) float wsm[kKC * NP];  // [kKC][NP]; reused as logits [kTM][NP]
  const int tx = threadIdx.x % kWarp, ty = threadIdx.x / kWarp;
  const int t0 = blockIdx.x * kTM;
  float acc[4][EJ];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EJ; ++j) acc[i][j] = 0.f;

  for (int k0 = 0; k0 < d; k0 += kKC) {
    for (int q = threadIdx.x; q < kTM * kKC; q += blockDim.x) {
      int r = q / kKC, c = q % kKC;
      int t = t0 + r;
      xs[r][c] = (t < Tn && k0 + c < d) ? to_f32(x[(size_t)t * d + k0 + c]) : 0.f;
    }
    for (int q = threadIdx.x; q < kKC * NP; q += blockDim.x) {
      int r = q / NP, c = q % NP;
      wsm[q] = (c < N && k0 + r < d) ? to_f32(Wg[(size_t)(k0 + r) * N + c]) : 0.f;
    }
    __syncthreads();
    // Blocked summation: each 32-element chunk is summed into a fresh partial
    // that is then added to the total, so the rounding error grows with the
    // number of chunks (d/32) rather than with d.
    float part[4][EJ];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < EJ; ++j) part[i][j] = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < kKC; ++kk) {
      float a[4], b[EJ];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[ty + 8 * i][kk];
#pragma unroll
      for (int j = 0; j < EJ; ++j) b[j] = wsm[kk * NP + tx + kWarp * j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < EJ; ++j) part[i][j] = fmaf(a[i], b[j], part[i][j]);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < EJ; ++j) acc[i][j] += part[i][j];
    __syncthreads();
  }
  // Stage logits [kTM][NP] in shared memory (NP <= kKC * NP / kTM holds since kKC == kTM).
  float *ls = wsm;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
      int e = tx + kWarp * j;
      float b = (bias && e < N) ? bias[e] : 0.f;
      ls[(ty + 8 * i) * NP + e] = acc[i][j] + b;
    }
  __syncthreads();
  bool nan_seen = false;
  for (int r = ty; r < kTM; r += 8) {
    int t = t0 + r;
    if (t >= Tn) break;
    float v[EJ];
    int e[EJ];
#pragma unroll
    for (int j = 0; j < EJ; ++j) {
      int ex = tx + kWarp * j;
      v[j] = ls[r * NP + ex];
      e[j] = ex < N ? ex : -1;
      if (logits && ex < N) logits[(size_t)t * N + ex] = v[j];
    }
    nan_seen |= warp_topk_softmax<EJ>(v, e, k, tx, topk_idx + (size_t)t * k,
                                      topk_w + (size_t)t * k);
  }
  if (nan_seen) report(status, MOE_DEV_NAN_LOGIT);
}

template <typename T>
moe_status_t launch_typed(const void *x, const void *W_g, const float *bias, int T_, int d,
                          int N, int k, float *logits, int32_t *topk_idx, float *topk_w,
                          int32_t *status, cudaStream_t stream) {
  const T *xp = static_cast<const T *>(x);
  const T *wp = static_cast<const T *>(W_g);
  if (T_ == 0) return MOE_OK;
  if (T_ <= 512 && N <= 32 && d % 8 == 0) {
    if (N <= 8)
      MOE_CUDA_TRY(launch_pdl(router_decode<T, 8>, dim3(T_), dim3(kDecWarps * 32), 0, stream, xp,
          wp, bias, T_, d, N, k, logits, topk_idx, topk_w, status));
    else if (N <= 16)
      MOE_CUDA_TRY(launch_pdl(router_decode<T, 16>, dim3(T_), dim3(kDecWarps * 32), 0, stream, xp,
          wp, bias, T_, d, N, k, logits, topk_idx, topk_w, status));
    else
      MOE_CUDA_TRY(launch_pdl(router_decode<T, 32>, dim3(T_), dim3(kDecWarps * 32), 0, stream, xp,
          wp, bias, T_, d, N, k, logits, topk_idx, topk_w, status));
    MOE_LAUNCH_CHECK();
    return MOE_OK;
  }
  if (N <= 32) {
    int NP = N <= 8 ? 8 : (N <= 16 ? 16 : 32);
    size_t smem = (size_t)d * NP * sizeof(T);
    if (smem <= 200 * 1024) {
      int warps = 8;
      int grid = (T_ + warps - 1) / warps;
      if (grid > 148 * 8) grid = 148 * 8;
      // the shared-memory opt-in is set once per kernel variant (a driver
      // call on every launch cost more than the kernel at decode sizes)
      static bool smem_set[kMaxDevicesCached][3] = {};
      const int dev = current_device();
      bool *done = dev < kMaxDevicesCached ? smem_set[dev] : nullptr;
      if (NP == 8) {
        if (!done || !done[0]) {
          MOE_CUDA_TRY(cudaFuncSetAttribute(router_small_n<T, 8>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
          if (done) done[0] = true;
        }
        MOE_CUDA_TRY(launch_pdl(router_small_n<T, 8>, dim3(grid), dim3(256), smem, stream, xp, wp,
            bias, T_, d, N, k, logits, topk_idx, topk_w, status));
      } else if (NP == 16) {
        if (!done || !done[1]) {
          MOE_CUDA_TRY(cudaFuncSetAttribute(router_small_n<T, 16>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
          if (done) done[1] = true;
        }
        MOE_CUDA_TRY(launch_pdl(router_small_n<T, 16>, dim3(grid), dim3(256), smem, stream, xp, wp,
            bias, T_, d, N, k, logits, topk_idx, topk_w, status));
      } else {
        if (!done || !done[2]) {
          MOE_CUDA_TRY(cudaFuncSetAttribute(router_small_n<T, 32>,
                                            cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024));
          if (done) done[2] = true;
        }
        MOE_CUDA_TRY(launch_pdl(router_small_n<T, 32>, dim3(grid), dim3(256), smem, stream, xp, wp,
            bias, T_, d, N, k, logits, topk_idx, topk_w, status));
      }
      MOE_LAUNCH_CHECK();
      return MOE_OK;
    }
  }
  int grid = (T_ + kTM - 1) / kTM;
  if (N <= 32)
    MOE_CUDA_TRY(launch_pdl(router_tiled<T, 32>, dim3(grid), dim3(256), 0, stream, xp, wp, bias, T_,
        d, N, k, logits, topk_idx, topk_w, status));
  else if (N <= 64)
    MOE_CUDA_TRY(launch_pdl(router_tiled<T, 64>, dim3(grid), dim3(256), 0, stream, xp, wp, bias, T_,
        d, N, k, logits, topk_idx, topk_w, status));
  else if (N <= 128)
    MOE_CUDA_TRY(launch_pdl(router_tiled<T, 128>, dim3(grid), dim3(256), 0, stream, xp, wp, bias,
        T_, d, N, k, logits, topk_idx, topk_w, status));
  else
    MOE_CUDA_TRY(launch_pdl(router_tiled<T, 256>, dim3(grid), dim3(256), 0, stream, xp, wp, bias,
        T_, d, N, k, logits, topk_idx, topk_w, status));
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace

moe_status_t launch_router_topk(const void *x, const void *W_g, const float *bias,
                                moe_dtype_t dtype, int T, int d, int N, int k, float *logits,
                                int32_t *topk_idx, float *topk_w, int32_t *device_status,
                                cudaStream_t stream) {
  // Tensor cores when the expert count suits them (N % 8 == 0, N <= 256) and
  // the batch fills more than a few 128-token tiles; a decode-sized batch
  // (T <= 512) with few experts (N <= 32) takes the CUDA-core kernel, which
  // gives every token its own warp instead of one latency-bound tile.
  const bool small_batch = T <= 512 && N <= 32;
  if (dtype == MOE_BF16 && !small_batch) {
    moe_status_t s = launch_router_tc(x, W_g, bias, T, d, N, k, logits, topk_idx, topk_w,
                                      device_status, stream);
    if (s != MOE_ERR_UNSUPPORTED) return s;
  }
  if (dtype == MOE_BF16)
    return launch_typed<__nv_bfloat16>(x, W_g, bias, T, d, N, k, logits, topk_idx, topk_w,
                                       device_status, stream);
  return launch_typed<float>(x, W_g, bias, T, d, N, k, logits, topk_idx, topk_w,
                             device_status, stream);
}

}  // namespace moe
