// FP8 E4M3 expert weights and token rows, calibration-free absmax scales.
//
// Source: "大模型MoE混合专家架构原理与DeepSeek-V4工程实践解析", section
// MoE模型推理部署与显存优化实战 (inference is bound by memory bandwidth; the
// remedy named third is storing the weights in fewer bits, with FP8 used for
// the cached activations); "MoE稀疏激活原理与工程实践", 4.3 (16-bit weights
// compressed to fewer bits to shrink memory).
//
// Reading (the pages name the idea, not a format): OCP FP8 E4M3 (bias 7, 3
// mantissa bits, largest finite 448, no infinities).  A vector v -- one row
// of x (or of h) over its length, or one output channel of a weight matrix
// over its reduction dim -- is
// stored as q = E4M3(v * (448 / amax|v|)) (round to nearest even, saturated)
// and one fp32 scale amax / 448; both factors are formed in fp32 (an all-zero
// vector takes scale 1).  Weights W [N, K, M] (K the reduction dim) are
// written channel-major, [N, M, K], so the FP8 GEMM reads both operands
// K-major: gate/up [N, d, f] -> [N, f, d], down [N, f, d] -> [N, d, f].
#include <cuda_fp8.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint8_t to_e4m3(float v) {
  return (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}

// G threads per row (G a power of two, 32..256; 256 / G rows per CTA,
// grid-stride over row batches); C % 8 == 0, 16-byte rows of bf16 or fp32
// values.  With rows_valid, rows from *rows_valid on are left alone.
template <typename TIn>
__global__ void __launch_bounds__(256) quantize_rows_e4m3(const TIn *__restrict__ x,
                                                          int R, int C, int G,
                                                          uint8_t *__restrict__ q,
                                                          float *__restrict__ scale,
                                                          const int32_t *__restrict__ rows_valid) {
  pdl_begin();
  __shared__ float red[8];                     // one per warp
  const int lg = threadIdx.x % G;              // thread within the row's group
  const int grp = threadIdx.x / G;
  const int rpc = blockDim.x / G;              // rows per CTA
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nv = C / 8;
  if (rows_valid) R = min(R, *rows_valid);
  for (long b = blockIdx.x; b * rpc < R; b += gridDim.x) {
    const long r = b * rpc + grp;
    const bool active = r < R;
    const TIn *row = x + (size_t)(active ? r : 0) * C;
    float am = 0.f;
    if (active)
      for (int v = lg; v < nv; v += G) {
        float f[8];
        load8(row + 8 * v, f);
#pragma unroll
        for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if (G > 32) {                              // combine the group's warps
      if (lane == 0) red[warp] = am;
      __syncthreads();
      const int w0 = (grp * G) / 32;
      am = 0.f;
      for (int w = 0; w < G / 32; ++w) am = fmaxf(am, red[w0 + w]);
      __syncthreads();
    }
    const float inv = am > 0.f ? 448.0f / am : 1.0f;
    if (active && lg == 0) scale[r] = am > 0.f ? am / 448.0f : 1.0f;
    if (active) {
      uint2 *out = reinterpret_cast<uint2 *>(q + (size_t)r * C);
      for (int v = lg; v < nv; v += G) {
        float f[8];
        load8(row + 8 * v, f);
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i / 4] |= (uint32_t)to_e4m3(f[i] * inv) << (8 * (i % 4));
        out[v] = make_uint2(w[0], w[1]);
      }
    }
  }
}

// The dispatch row copy of an FP8 layer: G threads per token (as in
// quantize_rows_e4m3: 256 / G tokens per CTA, grid-stride) quantise the
// token's row as quantize_rows_e4m3 does (scale to scale[t]) and write its
// codes to the permuted row of each kept slot (inv_pos; -1 = dropped).  The
// row is read twice (absmax, then codes; the second read hits L1/L2).
// d % 16 == 0, k <= 32.
__global__ void __launch_bounds__(256) copy_rows_e4m3(const __nv_bfloat16 *__restrict__ x,
                                                      const int32_t *__restrict__ inv_pos, int T,
                                                      int d, int k, int G,
                                                      uint8_t *__restrict__ x_perm,
                                                      float *__restrict__ scale) {
  pdl_begin();
  __shared__ float red[8];                     // one per warp
  __shared__ int32_t pos_s[8][32];             // kept positions of each token of the CTA
  const int lg = threadIdx.x % G;
  const int grp = threadIdx.x / G;
  const int rpc = blockDim.x / G;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int nv = d / 8;
  for (long b = blockIdx.x; b * rpc < T; b += gridDim.x) {
    const long t = b * rpc + grp;
    const bool active = t < T;
    const uint4 *row = reinterpret_cast<const uint4 *>(x + (size_t)(active ? t : 0) * d);
    if (active && lg < k) pos_s[grp][lg] = inv_pos[(size_t)t * k + lg];
    float am = 0.f;
    if (active)
      for (int v = lg; v < nv; v += G) {
        float f[8];
        load8(reinterpret_cast<const __nv_bfloat16 *>(row + v), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) am = fmaxf(am, fabsf(f[i]));
      }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    if (lane == 0) red[warp] = am;
    __syncthreads();
    am = 0.f;
    for (int w = 0; w < (G + 31) / 32; ++w) am = fmaxf(am, red[(grp * G) / 32 + w]);
    const float inv = am > 0.f ? 448.0f / am : 1.0f;
    if (active && lg == 0) scale[t] = am > 0.f ? am / 448.0f : 1.0f;
    if (active)
      for (int v = lg; v < nv; v += G) {
        float f[8];
        load8(reinterpret_cast<const __nv_bfloat16 *>(row + v), f);
        uint32_t w[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 8; ++i) w[i / 4] |= (uint32_t)to_e4m3(f[i] * inv) << (8 * (i % 4));
        const uint2 code = make_uint2(w[0], w[1]);
        for (int j = 0; j < k; ++j) {
          const int pos = pos_s[grp][j];
          if (pos >= 0) reinterpret_cast<uint2 *>(x_perm + (size_t)pos * d)[v] = code;
        }
      }
    __syncthreads();   // red and pos_s are rewritten by the next batch
  }
}

// W [N, d, f] viewed as [N, K = d, M = f].  Block (32 output channels, expert
// e): the channels' absmax over d, then the codes in tiles of 128 d,
// transposed through shared memory so each channel's 128 bytes leave as eight
// 16-byte stores.  d % 16 == 0.
constexpr int kQCols = 32;
constexpr int kQRows = 128;
__global__ void __launch_bounds__(256) quantize_weights_e4m3(
    const __nv_bfloat16 *__restrict__ W, int d, int f, uint8_t *__restrict__ q,
    float *__restrict__ scale) {
  __shared__ float red[8][kQCols];
  __shared__ float inv_s[kQCols];
  __shared__ __align__(16) uint8_t tile[kQCols][kQRows + 16];
  const int e = blockIdx.y, f0 = blockIdx.x * kQCols;
  const int c = threadIdx.x % kQCols, rg = threadIdx.x / kQCols;   // 8 row groups
  const __nv_bfloat16 *We = W + (size_t)e * d * f;
  const bool col_ok = f0 + c < f;
  float am = 0.f;
  if (col_ok)
    for (int i = rg; i < d; i += 8) am = fmaxf(am, fabsf(__bfloat162float(We[(size_t)i * f + f0 + c])));
  red[rg][c] = am;
  __syncthreads();
  if (rg == 0) {
    float a = 0.f;
    for (int g = 0; g < 8; ++g) a = fmaxf(a, red[g][c]);
    inv_s[c] = a > 0.f ? 448.0f / a : 1.0f;
    if (col_ok) scale[(size_t)e * f + f0 + c] = a > 0.f ? a / 448.0f : 1.0f;
  }
  __syncthreads();
  const int wc = threadIdx.x / 8, wch = threadIdx.x % 8;   // writer: channel, 16-B chunk
  for (int d0 = 0; d0 < d; d0 += kQRows) {
    if (col_ok) {
      const float inv = inv_s[c];
      for (int j = rg; j < kQRows && d0 + j < d; j += 8)
        tile[c][j] = to_e4m3(__bfloat162float(We[(size_t)(d0 + j) * f + f0 + c]) * inv);
    }
    __syncthreads();
    if (f0 + wc < f && d0 + wch * 16 < d)
      *reinterpret_cast<uint4 *>(q + ((size_t)e * f + f0 + wc) * d + d0 + wch * 16) =
          *reinterpret_cast<const uint4 *>(&tile[wc][wch * 16]);
    __syncthreads();
  }
}

}  // namespace

moe_status_t launch_quantize_rows_e4m3(const void *x, int R, int C, uint8_t *q, float *scale,
                                       cudaStream_t stream, const int32_t *rows_valid,
                                       bool f32_in) {
  if (R == 0) return MOE_OK;
  // threads per row: enough for a few 16-byte vectors each, 32..256
  const int nv = C / 8;
  int G = 32;
  while (G < 256 && G * 4 < nv) G *= 2;
  const long rpc = 256 / G;
  long grid = ((long)R + rpc - 1) / rpc;
  if (grid > 148L * 8) grid = 148L * 8;
  if (f32_in)
    MOE_CUDA_TRY(launch_pdl(quantize_rows_e4m3<float>, dim3((int)grid), dim3(256), 0, stream,
                            static_cast<const float *>(x), R, C, G, q, scale, rows_valid));
  else
    MOE_CUDA_TRY(launch_pdl(quantize_rows_e4m3<__nv_bfloat16>, dim3((int)grid), dim3(256), 0,
                            stream, static_cast<const __nv_bfloat16 *>(x), R, C, G, q, scale,
                            rows_valid));
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

moe_status_t launch_copy_rows_e4m3(const void *x, const int32_t *inv_pos, int T, int d, int k,
                                   uint8_t *x_perm, float *scale, cudaStream_t stream) {
  if (T == 0) return MOE_OK;
  const int nv = d / 8;                         // threads per token as in the row quantiser
  int G = 32;
  while (G < 256 && G * 4 < nv) G *= 2;
  const long rpc = 256 / G;
  long grid = ((long)T + rpc - 1) / rpc;
  if (grid > 148L * 8) grid = 148L * 8;
  MOE_CUDA_TRY(launch_pdl(copy_rows_e4m3, dim3((int)grid), dim3(256), 0, stream,
                          static_cast<const __nv_bfloat16 *>(x), inv_pos, T, d, k, G, x_perm,
                          scale));
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

moe_status_t launch_quantize_weights_e4m3(const void *W, int N, int d, int f, uint8_t *q,
                                          float *scale, cudaStream_t stream) {
  dim3 grid((f + kQCols - 1) / kQCols, N);
  quantize_weights_e4m3<<<grid, 256, 0, stream>>>(static_cast<const __nv_bfloat16 *>(W), d, f,
                                                  q, scale);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
