// Grouped SwiGLU expert FFN on the CUDA cores (fp32 FFMA) -- the path for
// fp32 layers.
//
// Source: "MoE 分片：混合專家模型的平行化策略", section 什麼是 MoE 模型 (an
// expert is two linear maps with an activation between) and section 動態 token
// 路由 step 4 (each expert runs on the tokens routed to it).  SwiGLU reading:
//   h = SiLU(x W_gate[e]) * (x W_up[e]),  SiLU(z) = z / (1 + exp(-z))
//   y_perm = row_scale * (h W_down[e])
//
// Two launches of one tiled kernel: gate/up (two accumulators, SwiGLU in the
// epilogue) then down (row scale in the epilogue).  A CTA computes a 32-row x
// 64-column tile of one expert; the tile -> (expert, row block) map is read
// from the device offsets, so the host never reads the routing back.
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kBM = 32, kBN = 64, kKC = 32;

// Finds the expert owning row-tile `tile` (tiles of kBM rows, per expert).
// Returns -1 if the tile lies past the last expert's last tile.
__device__ int find_expert_tile(const int32_t *offsets, int N, int tile, int &row0, int &row1) {
  __shared__ int s_e, s_r0, s_r1;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int before = 0;  // tiles of experts already passed
    int found = -1, r0 = 0, r1 = 0;
    for (int e0 = 0; e0 < N && found < 0; e0 += 32) {
      int e = e0 + lane;
      int n = 0, lo = 0, hi = 0;
      if (e < N) {
        lo = offsets[e];
        hi = offsets[e + 1];
        n = (hi - lo + kBM - 1) / kBM;
      }
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      int excl = before + incl - n;
      bool mine = (e < N) && tile >= excl && tile < excl + n;
      unsigned m = __ballot_sync(0xffffffffu, mine);
      if (m) {
        int src = __ffs(m) - 1;
        int t_excl = __shfl_sync(0xffffffffu, excl, src);
        int t_lo = __shfl_sync(0xffffffffu, lo, src);
        int t_hi = __shfl_sync(0xffffffffu, hi, src);
        found = e0 + src;
        r0 = t_lo + (tile - t_excl) * kBM;
        r1 = min(t_hi, r0 + kBM);
      }
      before += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) { s_e = found; s_r0 = r0; s_r1 = r1; }
  }
  __syncthreads();
  row0 = s_r0;
  row1 = s_r1;
  return s_e;
}

// DUAL: out = SiLU(A B0) * (A B1); else out = row_scale * (A B0), row p
// stored at out_row[p] when out_row is set (an index outside [0, rows_out)
// stores nothing and sets MOE_DEV_BAD_ROW).
template <typename T, bool DUAL>
__global__ void __launch_bounds__(256) grouped_gemm_simt(const T *__restrict__ A,
                                                         const int32_t *__restrict__ offsets,
                                                         int N, int K, int Ncols,
                                                         const T *__restrict__ B0,
                                                         const T *__restrict__ B1,
                                                         const float *__restrict__ row_scale,
                                                         T *__restrict__ out,
                                                         const int32_t *__restrict__ out_row,
                                                         int rows_out, int32_t *status) {
  __shared__ float as[kBM][kKC + 1];
  __shared__ float b0s[kKC][kBN];
  __shared__ float b1s[DUAL ? kKC : 1][kBN];
  int row0, row1;
  const int e = find_expert_tile(offsets, N, blockIdx.x, row0, row1);
  if (e < 0) return;
  const int n0 = blockIdx.y * kBN;
  const T *Be0 = B0 + (size_t)e * K * Ncols;
  const T *Be1 = DUAL ? B1 + (size_t)e * K * Ncols : nullptr;
  const int tx = threadIdx.x % 32, ty = threadIdx.x / 32;
  float acc0[4][2], acc1[4][2];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 2; ++j) acc0[i][j] = acc1[i][j] = 0.f;

  for (int k0 = 0; k0 < K; k0 += kKC) {
    for (int q = threadIdx.x; q < kBM * kKC; q += blockDim.x) {
      int r = q / kKC, c = q % kKC;
      int p = row0 + r;
      as[r][c] = (p < row1 && k0 + c < K) ? to_f32(A[(size_t)p * K + k0 + c]) : 0.f;
    }
    for (int q = threadIdx.x; q < kKC * kBN; q += blockDim.x) {
      int r = q / kBN, c = q % kBN;
      bool ok = (k0 + r < K) && (n0 + c < Ncols);
      b0s[r][c] = ok ? to_f32(Be0[(size_t)(k0 + r) * Ncols + n0 + c]) : 0.f;
      if (DUAL) b1s[r][c] = ok ? to_f32(Be1[(size_t)(k0 + r) * Ncols + n0 + c]) : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < kKC; ++kk) {
      float a[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = as[ty + 8 * i][kk];
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        float b0 = b0s[kk][tx + 32 * j];
        float b1 = DUAL ? b1s[kk][tx + 32 * j] : 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          acc0[i][j] = fmaf(a[i], b0, acc0[i][j]);
          if (DUAL) acc1[i][j] = fmaf(a[i], b1, acc1[i][j]);
        }
      }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    int p = row0 + ty + 8 * i;
    if (p >= row1) continue;
    size_t orow = (size_t)p;
    if (!DUAL && out_row) {
      const int o = out_row[p];
      if (o < 0 || o >= rows_out) {
        report(status, MOE_DEV_BAD_ROW);
        continue;
      }
      orow = (size_t)o;
    }
    float s = (!DUAL && row_scale) ? row_scale[p] : 1.f;
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      int c = n0 + tx + 32 * j;
      if (c >= Ncols) continue;
      float v;
      if (DUAL) {
        float g = acc0[i][j];
        v = g / (1.f + expf(-g)) * acc1[i][j];
      } else {
        v = acc0[i][j] * s;
      }
      out[orow * Ncols + c] = from_f32<T>(v);
    }
  }
}

template <typename T>
moe_status_t launch_simt_typed(const void *x_perm, const int32_t *offsets, const float *row_scale,
                               int A_max, int d, int f, int N, const void *W_gate,
                               const void *W_up, const void *W_down, void *h, void *y_perm,
                               const int32_t *out_row, int rows_out, int32_t *status,
                               cudaStream_t stream) {
  if (A_max == 0) return MOE_OK;
  // Upper bound on row tiles: each expert adds at most one partial tile.
  const int max_tiles = (A_max + kBM - 1) / kBM + N;
  dim3 g1(max_tiles, (f + kBN - 1) / kBN);
  grouped_gemm_simt<T, true><<<g1, 256, 0, stream>>>(
      static_cast<const T *>(x_perm), offsets, N, d, f, static_cast<const T *>(W_gate),
      static_cast<const T *>(W_up), nullptr, static_cast<T *>(h), nullptr, 0, status);
  MOE_LAUNCH_CHECK();
  dim3 g2(max_tiles, (d + kBN - 1) / kBN);
  grouped_gemm_simt<T, false><<<g2, 256, 0, stream>>>(
      static_cast<const T *>(h), offsets, N, f, d, static_cast<const T *>(W_down), nullptr,
      row_scale, static_cast<T *>(y_perm), out_row, rows_out, status);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace

moe_status_t launch_ffn_simt(const void *x_perm, const int32_t *offsets, const float *row_scale,
                             int A_max, int d, int f, int N, moe_dtype_t dtype,
                             const void *W_gate, const void *W_up, const void *W_down, void *h,
                             void *y_perm, int32_t *device_status, cudaStream_t stream,
                             const int32_t *out_row, int rows_out) {
  if (dtype == MOE_BF16)
    return launch_simt_typed<__nv_bfloat16>(x_perm, offsets, row_scale, A_max, d, f, N, W_gate,
                                            W_up, W_down, h, y_perm, out_row, rows_out,
                                            device_status, stream);
  return launch_simt_typed<float>(x_perm, offsets, row_scale, A_max, d, f, N, W_gate, W_up,
                                  W_down, h, y_perm, out_row, rows_out, device_status, stream);
}

}  // namespace moe
