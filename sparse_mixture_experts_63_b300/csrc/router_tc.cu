// Router on the tensor cores (bf16 layers): logits = x W_g + b with tcgen05,
// then top-k and the softmax over the k selected logits in the epilogue.
//
// Source: "MoE 分片：混合專家模型的平行化策略", section 動態 token 路由, step 2
// (the router scores every expert and keeps the top-k) and step 6 (weights
// normalised over the selected experts, e.g. 0.6 / 0.4); "MoE 推理：激活参数
// vs 总参数与专家路由", section 深入原理 (a linear layer gives N gate logits;
// top-k softmax gives the weights).
//
// Layout: tokens are the MMA M operand (128 rows of x, K-major) and the
// experts the N operand (W_g [d, N] read MN-major, N padded to a multiple of
// 16, at most 256), so TMEM lane t holds token t's whole logit row and each
// epilogue thread ranks its own token with a register top-k list -- no
// logits round trip through memory and no cross-thread merge.
// Ranking: logit descending, equal logits -> lower expert id, NaN lowest.
//
// Precision: the tensor core's fp32 accumulator loses about half an ulp per
// accumulation step in one direction, so a long K (d = 4096..7168) alone
// would put the gate weights ~2e-5 off.  K is therefore split over kParts
// partial accumulators (contiguous K ranges), summed in fp32 in a fixed order
// by the epilogue: 8x fewer steps per accumulator.  TMEM holds kParts x 64
// columns, so experts are processed in passes of up to 64 (x re-read from L2).
//
// CTA = 6 warps (TMA producer, MMA issuer, 4 epilogue warps), persistent over
// 128-token tiles, 4-stage mbarrier pipeline.
#include <cuda.h>
#include <math.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;                      // tokens per tile
constexpr int kBK = 64;
constexpr int kStages = 6;
constexpr int kMaxNE = 256;                   // experts (MMA N) limit
constexpr int kXBytes = kBM * kBK * 2;        // 16 KB
constexpr int kWChunk = 64 * kBK * 2;         // 8 KB: 64 experts x 64 k
constexpr int kStageBytes = kXBytes + kWChunk;      // 24 KB
constexpr int kThreads = 192;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kMaxK = 32;
constexpr int kParts = 8;                     // partial accumulators over K
constexpr int kGroup = 64;                    // experts per pass (TMEM: kParts * 64 = 512)

struct RParams {
  int T, d, N, k;
  int ng;                    // experts per pass (multiple of 16, <= 64)
  int passes;                // ceil(N / ng)
  const float *bias;
  float *logits;             // nullable
  int32_t *topk_idx;
  float *topk_w;
  int32_t *status;
};

__device__ __forceinline__ float rank_key(float v) { return isnan(v) ? -INFINITY : v; }
__device__ __forceinline__ bool ranks_before(float va, int ia, float vb, int ib) {
  float ka = rank_key(va), kb = rank_key(vb);
  if (ka != kb) return ka > kb;
  return ia < ib;
}

template <int KMAX>
__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, const RParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kStages], empty[kStages], acc_full[2], acc_empty[2], drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag_s, epi_ok_s;
  volatile int *abort_flag = &abort_flag_s;
  volatile int *epi_ok = &epi_ok_s;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], 4);
    }
    tc::mbar_init(&drain, 1);
    abort_flag_s = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tmX);
    tc::tma_prefetch_desc(&tmW);
  }
  if (warp == 1) {
    tc::tmem_alloc(&tmem_slot, 512);
    tc::tmem_relinquish();
  }
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = tmem_slot;
  const int tiles = (p.T + kBM - 1) / kBM;
  const int kblocks = (p.d + kBK - 1) / kBK;

  if (warp == 0) {
    // ---- TMA producer: lane 0 runs a tight loop (stage/phase counters)
    if (lane == 0) {
      const uint64_t pol_x = tc::policy_evict_last();   // re-read by every pass
      const uint64_t pol_w = tc::policy_evict_last();
      const uint32_t bytes = kXBytes + kWChunk;
      int s = 0;
      uint32_t ph = 0, issued = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int ps = 0; ps < p.passes && ok; ++ps) {
          for (int kb = 0; kb < kblocks; ++kb) {
            if (!tc::mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, kTimeoutNs)) {
              ok = false;
              break;
            }
            unsigned char *st = smem + s * kStageBytes;
            tc::mbar_arrive_expect_tx(&full[s], bytes);
            tc::tma_load_2d(st, &tmX, &full[s], kb * kBK, t * kBM, pol_x);
            tc::tma_load_2d(st + kXBytes, &tmW, &full[s], ps * p.ng, kb * kBK, pol_w);
            ++issued;
            if (++s == kStages) { s = 0; ph ^= 1; }
          }
        }
      }
      if (!ok) {
        const uint32_t first = issued >= kStages ? issued - kStages : 0;
        for (uint32_t q = first; q < issued; ++q) {
          volatile int dummy = 0;
          tc::mbar_wait_bounded(&full[q % kStages], (q / kStages) & 1, &dummy, kTimeoutNs / 4);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer: lane 0 runs a tight loop.  K block kb accumulates into
    // partial `part`, which advances every ceil-spaced boundary bound[part].
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(kBM, p.ng, /*a_mn=*/0, /*b_mn=*/1);
      const int parts = kblocks < kParts ? kblocks : kParts;
      const uint32_t stage0 = tc::smem_u32(smem);
      const uint64_t a_desc0 = tc::sdesc_sw128(stage0, 16, 1024);              // x, K-major
      const uint64_t b_desc0 = tc::sdesc_sw128(stage0 + kXBytes, kWChunk, 1024); // W, MN-major
      int s = 0;
      uint32_t ph = 0, round = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < tiles && ok; t += gridDim.x) {
        for (int ps = 0; ps < p.passes; ++ps, ++round) {
          if (!tc::mbar_wait_bounded(&acc_empty[0], (round & 1) ^ 1, abort_flag, kTimeoutNs)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          int part = 0;
          int next_bound = (kblocks + parts - 1) / parts;   // first kb of partial 1
          for (int kb = 0; kb < kblocks; ++kb) {
            if (!tc::mbar_wait_bounded(&full[s], ph, abort_flag, kTimeoutNs)) {
              ok = false;
              break;
            }
            tc::tc_fence_after();
            bool first = (kb == 0);
            if (kb == next_bound) {
              ++part;
              next_bound = ((part + 1) * kblocks + parts - 1) / parts;
              first = true;
            }
            const uint32_t d_tmem = tmem_base + part * kGroup;
            const uint64_t off = (uint64_t)((s * kStageBytes) >> 4);
            const uint64_t ad = a_desc0 + off, bd = b_desc0 + off;
            // x K-major: +32 B per 16 k (+2); W MN-major: +2048 B per 16 k (+128)
            tc::mma_f16(d_tmem, ad, bd, idesc, first ? 0u : 1u);
            tc::mma_f16(d_tmem, ad + 2, bd + 128, idesc, 1u);
            tc::mma_f16(d_tmem, ad + 4, bd + 256, idesc, 1u);
            tc::mma_f16(d_tmem, ad + 6, bd + 384, idesc, 1u);
            tc::mma_commit(&empty[s]);
            if (++s == kStages) { s = 0; ph ^= 1; }
          }
          if (!ok) break;
          tc::mma_commit(&acc_full[0]);
        }
      }
      tc::mma_commit(&drain);
      volatile int dummy = 0;
      tc::mbar_wait_bounded(&drain, 0, &dummy, kTimeoutNs);
    }
    __syncwarp();
  } else {
    // epilogue: thread = token row (TMEM lane)
    const int lane_grp = warp % 4;
    const int etid = threadIdx.x - 64;
    const int row_in_tile = lane_grp * 32 + lane;
    bool nan_seen = false;
    const int parts = kblocks < kParts ? kblocks : kParts;
    uint32_t round = 0;
    bool go = true;
    for (int t = blockIdx.x; t < tiles && go; t += gridDim.x) {
      const int tok = t * kBM + row_in_tile;
      float bv[KMAX];
      int bi[KMAX];
#pragma unroll
      for (int j = 0; j < KMAX; ++j) { bv[j] = -INFINITY; bi[j] = INT_MAX; }
      for (int ps = 0; ps < p.passes; ++ps, ++round) {
        if (etid == 0)
          *epi_ok = tc::mbar_wait_bounded(&acc_full[0], round & 1, abort_flag, kTimeoutNs) ? 1
                                                                                           : 0;
        tc::named_bar(1, 128);
        go = *epi_ok != 0;
        tc::named_bar(1, 128);
        if (!go) break;
        tc::tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(lane_grp * 32) << 16);
        const int e0 = ps * p.ng;
        const int ncol = min(p.ng, p.N - e0);
        for (int c0 = 0; c0 < ncol; c0 += 32) {
          float v32[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) v32[c] = 0.f;
          for (int q = 0; q < parts; ++q) {
            uint32_t r[32];
            tc::tmem_ld_32x32b_x32(taddr + q * kGroup + c0, r);
            tc::tmem_ld_wait();
#pragma unroll
            for (int c = 0; c < 32; ++c) v32[c] += __uint_as_float(r[c]);
          }
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            if (c0 + c >= ncol) break;
            const int e = e0 + c0 + c;
            float v = v32[c];
            if (p.bias) v += __ldg(p.bias + e);
            nan_seen |= isnan(v);
            if (p.logits && tok < p.T) p.logits[(size_t)tok * p.N + e] = v;
            // insert (v, e) into the sorted list of the best k (a candidate
            // that ranks below all of them moves nothing)
            float cv = v;
            int ci = e;
#pragma unroll
            for (int j = 0; j < KMAX; ++j) {
              if (j < p.k && ranks_before(cv, ci, bv[j], bi[j])) {
                const float tv = bv[j];
                const int ti = bi[j];
                bv[j] = cv;
                bi[j] = ci;
                cv = tv;
                ci = ti;
              }
            }
          }
        }
        tc::tc_fence_before();
        if (lane == 0) tc::mbar_arrive(&acc_empty[0]);
      }
      if (go && tok < p.T) {
        float s = 0.f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < p.k) s += expf(bv[j] - bv[0]);
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < p.k) {
            p.topk_idx[(size_t)tok * p.k + j] = bi[j];
            p.topk_w[(size_t)tok * p.k + j] = expf(bv[j] - bv[0]) / s;
          }
      }
    }
    if (nan_seen) report(p.status, MOE_DEV_NAN_LOGIT);
  }

  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) report(p.status, MOE_DEV_TIMEOUT);
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, 512);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *q = nullptr;
    cudaDriverEntryPointQueryResult r;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000, cudaEnableDefault,
                                         &r) == cudaSuccess &&
        r == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(q);
  }
  return fn;
}

bool encode2d(CUtensorMap *m, const void *base, uint64_t inner, uint64_t outer, uint32_t box_in,
              uint32_t box_out) {
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * 2};
  cuuint32_t box[2] = {box_in, box_out};
  cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Returns MOE_ERR_UNSUPPORTED when the shape does not suit the tensor-core
// router (the caller then uses the CUDA-core one).
moe_status_t launch_router_tc(const void *x, const void *W_g, const float *bias, int T, int d,
                              int N, int k, float *logits, int32_t *topk_idx, float *topk_w,
                              int32_t *device_status, cudaStream_t stream) {
  if (N > kMaxNE || N % 8 != 0 || k > kMaxK || !encode_fn()) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  CUtensorMap tx, tw;
  if (!encode2d(&tx, x, d, T, kBK, kBM) || !encode2d(&tw, W_g, N, d, 64, kBK))
    return MOE_ERR_UNSUPPORTED;
  const int ng = N < kGroup ? ((N + 15) & ~15) : kGroup;
  RParams p{T, d, N, k, ng, (N + ng - 1) / ng, bias, logits, topk_idx, topk_w, device_status};
  const int smem = kStages * kStageBytes + 1024;
  int dev = 0, sms = 148;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int tiles = (T + kBM - 1) / kBM;
  const int grid = tiles < sms ? tiles : sms;
  if (k <= 2) {
    static bool attr2 = false;
    if (!attr2) {
      MOE_CUDA_TRY(cudaFuncSetAttribute(router_tc_kernel<2>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
      attr2 = true;
    }
    router_tc_kernel<2><<<grid, kThreads, smem, stream>>>(tx, tw, p);
  } else if (k <= 8) {
    static bool attr8 = false;
    if (!attr8) {
      MOE_CUDA_TRY(cudaFuncSetAttribute(router_tc_kernel<8>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
      attr8 = true;
    }
    router_tc_kernel<8><<<grid, kThreads, smem, stream>>>(tx, tw, p);
  } else {
    static bool attr32 = false;
    if (!attr32) {
      MOE_CUDA_TRY(cudaFuncSetAttribute(router_tc_kernel<32>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
      attr32 = true;
    }
    router_tc_kernel<32><<<grid, kThreads, smem, stream>>>(tx, tw, p);
  }
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
