// Router on the tensor cores (bf16 layers): logits = x W_g + b with tcgen05,
// then top-k and the softmax over the k selected logits in the epilogue.
//
// Source: "MoE 分片：混合專家模型的平行化策略", section 動態 token 路由, step 2
// (the router scores every expert and keeps the top-k) and step 6 (weights
// normalised over the selected experts, e.g. 0.6 / 0.4); "MoE 推理：激活参数
// vs 总参数与专家路由", section 深入原理 (a linear layer gives N gate logits;
// top-k softmax gives the weights).
//
// Layout: tokens are the MMA M operand (128 rows of x, K-major) and experts
// the N operand (W_g [d, N] read MN-major), so TMEM lane t holds token t's
// logits and each epilogue thread ranks its own token with a register top-k
// list.  Ranking: logit descending, equal logits -> lower expert id, NaN lowest.
//
// Work split: one 128-token tile per cluster, one group of at most 128 experts
// per CTA of the cluster (N = 256 -> 2 CTAs, <= 128 -> 1), so T = 8192 tokens
// and 256 experts run as 128 CTAs, one wave on 148 SMs.  Each CTA
// ranks its group; the cluster's first CTA merges the groups' candidate lists
// through distributed shared memory (the comparator is a total order, so the
// merge gives exactly the global top-k), applies the softmax and writes.
//
// Precision: the tensor core's fp32 accumulator loses about half an ulp per
// accumulation step in one direction, so a long K (d = 4096..7168) alone
// would put the gate weights ~2e-5 off.  K is split over kParts partial
// accumulators (contiguous K ranges), summed in fp32 in a fixed order by the
// epilogue: 4x fewer steps per accumulator (TMEM: kParts x 128 columns).
//
// CTA = 6 warps: TMA producer, MMA issuer, 4 epilogue warps; 6-8 stage
// mbarrier pipeline; every wait bounded (2 s) with a clean drain on timeout.
#include <cuda.h>
#include <math.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;                      // tokens per tile
constexpr int kBK = 64;
constexpr int kMaxStages = 8;
constexpr int kMaxNE = 256;                   // experts limit
constexpr int kXBytes = kBM * kBK * 2;        // 16 KB
constexpr int kWChunk = 64 * kBK * 2;         // 8 KB: 64 experts x 64 k
constexpr int kStageRegion = 192 * 1024;      // 6 x 32 KB (128 experts) or 8 x 24 KB (<= 64)
constexpr int kThreads = 192;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kMaxK = 32;
constexpr int kParts = 4;                     // partial accumulators over K
constexpr int kGroup = 128;                   // experts per CTA (TMEM: kParts * 128 = 512)
constexpr int kCandOffset = kStageRegion;     // candidate lists after the stages

struct RParams {
  int T, d, N, k;
  int ng;                    // experts per CTA (multiple of 16, <= 128)
  int group_ctas;            // CTAs per cluster = ceil(N / ng)
  int wchunks;               // 64-expert W boxes per stage = ceil(ng / 64)
  int stages;                // pipeline stages
  int stage_bytes;           // kXBytes + wchunks * kWChunk
  const float *bias;
  float *logits;             // nullable
  int32_t *topk_idx;
  float *topk_w;
  int32_t *status;
};

__device__ __forceinline__ float rank_key(float v) { return isnan(v) ? -INFINITY : v; }

__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ int ld_cluster_s32(uint32_t addr) {
  int v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Inserts (v, e) into the sorted list of the best k; a candidate that ranks
// below all of them moves nothing.  Branch-free: every slot compares against
// the candidate at once (the list is sorted, so the slots it beats are a
// suffix), then each slot of that suffix takes the candidate or its
// predecessor -- no chain of dependent compare-and-swaps.
template <int KMAX>
__device__ __forceinline__ void insert_sorted(float (&bv)[KMAX], int (&bi)[KMAX], int k, float v,
                                              int e) {
  const float kv = rank_key(v);
  bool gt[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    const float kj = rank_key(bv[j]);
    // rank order: larger key first (NaN lowest), equal keys by lower index;
    // written without branches
    gt[j] = (j < k) & ((kv > kj) | ((kv == kj) & (e < bi[j])));
  }
#pragma unroll
  for (int j = KMAX - 1; j > 0; --j) {
    const float nv = gt[j - 1] ? bv[j - 1] : v;
    const int ni = gt[j - 1] ? bi[j - 1] : e;
    bv[j] = gt[j] ? nv : bv[j];
    bi[j] = gt[j] ? ni : bi[j];
  }
  bv[0] = gt[0] ? v : bv[0];
  bi[0] = gt[0] ? e : bi[0];
}

template <int KMAX>
__global__ void __launch_bounds__(kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap tmX,
                     const __grid_constant__ CUtensorMap tmW, const RParams p) {
  pdl_begin();
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  __shared__ uint64_t full[kMaxStages], empty[kMaxStages], acc_full, drain;
  __shared__ uint32_t tmem_slot;
  __shared__ int abort_flag_s, epi_ok_s;
  volatile int *abort_flag = &abort_flag_s;
  volatile int *epi_ok = &epi_ok_s;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int rank = p.group_ctas > 1 ? (int)tc::cluster_ctarank() : 0;
  const int tile = p.group_ctas > 1 ? (int)tc::cluster_id_x() : (int)blockIdx.x;
  const int e0 = rank * p.ng;                           // this CTA's expert group
  const int ncol = min(p.ng, p.N - e0);
  float *cand_v = reinterpret_cast<float *>(smem + kCandOffset);        // [KMAX][128]
  int *cand_i = reinterpret_cast<int *>(smem + kCandOffset + KMAX * kBM * 4);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    tc::mbar_init(&acc_full, 1);
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
  const int kblocks = (p.d + kBK - 1) / kBK;
  const int parts = kblocks < kParts ? kblocks : kParts;
  float bv[KMAX];
  int bi[KMAX];
#pragma unroll
  for (int j = 0; j < KMAX; ++j) { bv[j] = -INFINITY; bi[j] = INT_MAX; }
  bool nan_seen = false;
  bool have_list = false;

  if (warp == 0) {
    // ---- TMA producer: lane 0 runs a tight loop (stage/phase counters)
    if (lane == 0) {
      const uint64_t pol_x = tc::policy_evict_normal();
      const uint64_t pol_w = tc::policy_evict_last();
      int s = 0;
      uint32_t ph = 0, issued = 0;
      bool ok = true;
      for (int kb = 0; kb < kblocks; ++kb) {
        if (!tc::mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, kTimeoutNs)) {
          ok = false;
          break;
        }
        unsigned char *st = smem + s * p.stage_bytes;
        tc::mbar_arrive_expect_tx(&full[s], (uint32_t)p.stage_bytes);
        tc::tma_load_2d(st, &tmX, &full[s], kb * kBK, tile * kBM, pol_x);
        tc::tma_load_2d(st + kXBytes, &tmW, &full[s], e0, kb * kBK, pol_w);
        if (p.wchunks > 1)
          tc::tma_load_2d(st + kXBytes + kWChunk, &tmW, &full[s], e0 + 64, kb * kBK, pol_w);
        ++issued;
        if (++s == p.stages) { s = 0; ph ^= 1; }
      }
      if (!ok) {
        const uint32_t ns = (uint32_t)p.stages;
        const uint32_t first = issued >= ns ? issued - ns : 0;
        for (uint32_t q = first; q < issued; ++q) {
          volatile int dummy = 0;
          tc::mbar_wait_bounded(&full[q % ns], (q / ns) & 1, &dummy, kTimeoutNs / 4);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer: lane 0 runs a tight loop.  K block kb accumulates into
    // partial `part`, which advances at the ceil-spaced boundaries.
    if (lane == 0) {
      const uint32_t idesc = tc::idesc_bf16(kBM, p.ng, /*a_mn=*/0, /*b_mn=*/1);
      const uint32_t stage0 = tc::smem_u32(smem);
      const uint64_t a_desc0 = tc::sdesc_sw128(stage0, 16, 1024);               // x, K-major
      const uint64_t b_desc0 = tc::sdesc_sw128(stage0 + kXBytes, kWChunk, 1024); // W, MN-major
      int s = 0;
      uint32_t ph = 0;
      int part = 0;
      int next_bound = (kblocks + parts - 1) / parts;   // first kb of partial 1
      bool ok = true;
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
        const uint64_t off = (uint64_t)((s * p.stage_bytes) >> 4);
        const uint64_t ad = a_desc0 + off, bd = b_desc0 + off;
        // x K-major: +32 B per 16 k (+2); W MN-major: +2048 B per 16 k (+128)
        tc::mma_f16(d_tmem, ad, bd, idesc, first ? 0u : 1u);
        tc::mma_f16(d_tmem, ad + 2, bd + 128, idesc, 1u);
        tc::mma_f16(d_tmem, ad + 4, bd + 256, idesc, 1u);
        tc::mma_f16(d_tmem, ad + 6, bd + 384, idesc, 1u);
        tc::mma_commit(&empty[s]);
        if (++s == p.stages) { s = 0; ph ^= 1; }
      }
      if (ok) tc::mma_commit(&acc_full);
      tc::mma_commit(&drain);
      volatile int dummy = 0;
      tc::mbar_wait_bounded(&drain, 0, &dummy, kTimeoutNs);
    }
    __syncwarp();
  } else {
    // ---- epilogue: thread = token row (TMEM lane)
    const int lane_grp = warp % 4;
    const int etid = threadIdx.x - 64;
    const int row = lane_grp * 32 + lane;
    const int tok = tile * kBM + row;
    if (etid == 0)
      *epi_ok = tc::mbar_wait_bounded(&acc_full, 0, abort_flag, kTimeoutNs) ? 1 : 0;
    tc::named_bar(1, 128);
    const bool go = *epi_ok != 0;
    if (go) {
      tc::tc_fence_after();
      const uint32_t taddr = tmem_base + ((uint32_t)(lane_grp * 32) << 16);
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
          insert_sorted<KMAX>(bv, bi, p.k, v, e);
        }
      }
      have_list = true;
      if (p.group_ctas > 1) {
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (j < p.k) {
            cand_v[j * kBM + row] = bv[j];
            cand_i[j * kBM + row] = bi[j];
          }
      }
    }
    if (nan_seen) report(p.status, MOE_DEV_NAN_LOGIT);
  }

  __syncthreads();
  if (p.group_ctas > 1) tc::cluster_sync();   // every group's list is in place
  if (warp >= 2 && rank == 0 && have_list) {
    const int row = (warp % 4) * 32 + lane;
    const int tok = tile * kBM + row;
    for (int q = 1; q < p.group_ctas; ++q) {
      const uint32_t rv = tc::mapa_shared(cand_v, (uint32_t)q);
      const uint32_t ri = tc::mapa_shared(cand_i, (uint32_t)q);
      for (int j = 0; j < p.k; ++j) {
        const float v = ld_cluster_f32(rv + (uint32_t)((j * kBM + row) * 4));
        const int e = ld_cluster_s32(ri + (uint32_t)((j * kBM + row) * 4));
        insert_sorted<KMAX>(bv, bi, p.k, v, e);
      }
    }
    if (tok < p.T) {
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
  if (p.group_ctas > 1) tc::cluster_sync();   // peers keep their lists until read
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

template <int KMAX>
moe_status_t launch_k(const CUtensorMap &tx, const CUtensorMap &tw, const RParams &p, int tiles,
                      cudaStream_t stream) {
  constexpr int smem = kStageRegion + 2 * KMAX * kBM * 4 + 1024;   // stages + candidate lists
  static bool attr[kMaxDevicesCached] = {};
  const int dev = current_device();
  if (dev >= kMaxDevicesCached || !attr[dev]) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(router_tc_kernel<KMAX>,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, smem));
    if (dev < kMaxDevicesCached) attr[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_begin
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = p.group_ctas;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(tiles * p.group_ctas);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attrs;
  cfg.numAttrs = p.group_ctas > 1 ? 2 : 1;
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, router_tc_kernel<KMAX>, tx, tw, p));
  MOE_LAUNCH_CHECK();
  return MOE_OK;
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
  const int groups = (N + ng - 1) / ng;
  const int wchunks = (ng + 63) / 64;
  const int stage_bytes = kXBytes + wchunks * kWChunk;
  int stages = kStageRegion / stage_bytes;
  if (stages > kMaxStages) stages = kMaxStages;
  RParams p{T, d, N, k, ng, groups, wchunks, stages, stage_bytes, bias, logits, topk_idx,
            topk_w, device_status};
  const int tiles = (T + kBM - 1) / kBM;
  if (k <= 2) return launch_k<2>(tx, tw, p, tiles, stream);
  if (k <= 8) return launch_k<8>(tx, tw, p, tiles, stream);
  return launch_k<32>(tx, tw, p, tiles, stream);
}

}  // namespace moe
