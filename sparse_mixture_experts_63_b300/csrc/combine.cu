// Combine: y[t] = sum_{j<k, kept} y_perm[inv_pos[t,j]] (+ shared_y[t]).
//
// Source: "MoE 分片：混合專家模型的平行化策略", section 動態 token 路由, step 6
// (the k expert outputs are combined with the router's weights, back on the
// token's own position); "MoE 架构科普", section 专家粒度 (the shared expert
// every token passes through).  The gate weight is already applied to each
// y_perm row by the down-projection epilogue, so this is a plain gather-sum,
// in fp32, slots in ascending order, then the shared output: deterministic.
//
// HBM-bound: one thread per 8 output elements, 16-byte loads of bf16 rows
// (32-byte of fp32), coalesced along d.  A thread reads the token's slot
// positions for up to KB slots at once and issues all of their row loads
// before adding any: KB loads in flight per thread instead of one at a time
// behind its position load (the sums are taken in the same slot order).
#include "moe_internal.cuh"

namespace moe {
namespace {

// 8 consecutive elements of a row, as loaded (bf16: 16 bytes; fp32: 32 bytes)
template <typename TI> struct Raw8;
template <> struct Raw8<__nv_bfloat16> {
  uint4 q;
  __device__ __forceinline__ void load(const __nv_bfloat16 *p) {
    q = *reinterpret_cast<const uint4 *>(p);
  }
  __device__ __forceinline__ void add_to(float (&acc)[8]) const {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&q);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(h[i]);
      acc[2 * i] += f.x;
      acc[2 * i + 1] += f.y;
    }
  }
};
template <> struct Raw8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float *p) {
    a = *reinterpret_cast<const float4 *>(p);
    b = *reinterpret_cast<const float4 *>(p + 4);
  }
  __device__ __forceinline__ void add_to(float (&acc)[8]) const {
    acc[0] += a.x; acc[1] += a.y; acc[2] += a.z; acc[3] += a.w;
    acc[4] += b.x; acc[5] += b.y; acc[6] += b.z; acc[7] += b.w;
  }
};

template <typename TI, typename TO, int KB>
__global__ void __launch_bounds__(256) combine_kernel(const TI *__restrict__ y_perm,
                                                      const int32_t *__restrict__ inv_pos, int T,
                                                      int k, int d, const TI *__restrict__ shared,
                                                      TO *__restrict__ y) {
  pdl_begin();
  const int groups = d / 8;
  const long total = (long)T * groups;
  for (long g = (long)blockIdx.x * blockDim.x + threadIdx.x; g < total;
       g += (long)gridDim.x * blockDim.x) {
    const int t = (int)(g / groups);
    const int c = (int)(g % groups) * 8;
    float acc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] = 0.f;
    for (int j0 = 0; j0 < k; j0 += KB) {
      int pos[KB];
#pragma unroll
      for (int j = 0; j < KB; ++j)
        pos[j] = j0 + j < k ? __ldg(inv_pos + (size_t)t * k + j0 + j) : -1;
      Raw8<TI> r[KB];
#pragma unroll
      for (int j = 0; j < KB; ++j)
        if (pos[j] >= 0) r[j].load(y_perm + (size_t)pos[j] * d + c);
#pragma unroll
      for (int j = 0; j < KB; ++j)   // slot order, dropped slots skipped
        if (pos[j] >= 0) r[j].add_to(acc);
    }
    if (shared) {
      Raw8<TI> r;
      r.load(shared + (size_t)t * d + c);
      r.add_to(acc);
    }
    TO *dst = y + (size_t)t * d + c;
    if constexpr (sizeof(TO) == 4) {
      float4 *o = reinterpret_cast<float4 *>(dst);
      o[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
      o[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    } else {
      __nv_bfloat162 q[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) q[i] = __floats2bfloat162_rn(acc[2 * i], acc[2 * i + 1]);
      *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<uint4 *>(q);
    }
  }
}

template <typename TI, typename TO>
moe_status_t launch_typed(const void *y_perm, const int32_t *inv_pos, int T, int k, int d,
                          const void *shared_y, void *y, cudaStream_t stream) {
  long total = (long)T * (d / 8);
  if (total == 0) return MOE_OK;
  long grid = (total + 255) / 256;
  if (grid > 148L * 32) grid = 148L * 32;
  // slots batched 2, 4 or 8 at a time (larger k in batches of 8)
  auto fn = k <= 2 ? combine_kernel<TI, TO, 2> : k <= 4 ? combine_kernel<TI, TO, 4>
                                                        : combine_kernel<TI, TO, 8>;
  MOE_CUDA_TRY(launch_pdl(fn, dim3((int)grid), dim3(256), 0, stream,
      static_cast<const TI *>(y_perm), inv_pos, T, k, d, static_cast<const TI *>(shared_y),
      static_cast<TO *>(y)));
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace

moe_status_t launch_combine(const void *y_perm, moe_dtype_t y_perm_dtype, const int32_t *inv_pos,
                            int T, int k, int d, const void *shared_y, void *y,
                            moe_dtype_t y_dtype, cudaStream_t stream) {
  if (y_perm_dtype == MOE_BF16) {
    if (y_dtype == MOE_BF16)
      return launch_typed<__nv_bfloat16, __nv_bfloat16>(y_perm, inv_pos, T, k, d, shared_y, y,
                                                        stream);
    return launch_typed<__nv_bfloat16, float>(y_perm, inv_pos, T, k, d, shared_y, y, stream);
  }
  if (y_dtype == MOE_BF16)
    return launch_typed<float, __nv_bfloat16>(y_perm, inv_pos, T, k, d, shared_y, y, stream);
  return launch_typed<float, float>(y_perm, inv_pos, T, k, d, shared_y, y, stream);
}

}  // namespace moe
