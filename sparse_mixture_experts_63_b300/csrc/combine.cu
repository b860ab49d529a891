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
// (32-byte of fp32), coalesced along d.
#include "moe_internal.cuh"

namespace moe {
namespace {

template <typename TI, typename TO>
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
    for (int j = 0; j < k; ++j) {
      const int p = __ldg(inv_pos + (size_t)t * k + j);
      if (p < 0) continue;
      float v[8];
      load8(y_perm + (size_t)p * d + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
    }
    if (shared) {
      float v[8];
      load8(shared + (size_t)t * d + c, v);
#pragma unroll
      for (int i = 0; i < 8; ++i) acc[i] += v[i];
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
  MOE_CUDA_TRY(launch_pdl(combine_kernel<TI, TO>, dim3((int)grid), dim3(256), 0, stream,
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
