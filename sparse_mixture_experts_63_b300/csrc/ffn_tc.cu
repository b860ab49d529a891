// Grouped SwiGLU expert FFN on the 5th-generation tensor cores (tcgen05).
//
// Source: "MoE 分片：混合專家模型的平行化策略", section 什麼是 MoE 模型 (an
// expert is two linear maps with an activation between) and section 動態 token
// 路由 step 4 (each expert runs on the tokens routed to it);
// "MoE稀疏激活原理与工程实践", 3.1 (tokens regrouped by expert so each expert
// runs once per batch -- here one persistent launch covers every expert).
// SwiGLU reading: h = SiLU(x W_gate) * (x W_up), y_perm = row_scale * (h W_down).
//
// Formulation ("swap AB"): the weights are the 128-row M operand and the
// expert's tokens the N operand, so a tile's N is that expert's row count
// rounded up to 16 (no padding of small experts to 128 rows):
//   GEMM1  D[128 x n] = [W_gate[:, f0:f0+64] | W_up[:, f0:f0+64]]^T x x_perm^T
//          lanes 0-63 hold gate, lanes 64-127 up for the same 64 hidden units;
//          the epilogue writes h = SiLU(gate) * up (bf16) for those tokens.
//   GEMM2  D[128 x n] = W_down[:, m0:m0+128]^T x h^T
//          the epilogue writes y_perm = row_scale * D (bf16).
// A (weights) is read MN-major straight from W[N, K, M] by 3-D TMA boxes of
// 64(M) x 64(K) with 128-byte swizzle; B (token rows, K contiguous) is read
// K-major by 2-D boxes of 64(K) x {32,64,128,256}(rows).
//
// CTA = 6 warps, persistent (one CTA per SM):
//   warp 0      TMA producer (one lane)
//   warp 1      tensor-memory allocator + MMA issuer (one lane)
//   warps 2..5  epilogue (tcgen05.ld of their 32 lanes, math, coalesced stores)
// Pipelines: kStages shared-memory stages (full/empty mbarriers) and two
// 256-column TMEM accumulators (acc_full/acc_empty), so the epilogue of one
// tile overlaps the MMAs of the next.  Every wait is bounded (2 s): on timeout
// the CTA sets MOE_DEV_TIMEOUT, drains what it issued and exits cleanly.
#include <cuda.h>
#include <math.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;          // MMA M (weight rows per tile)
constexpr int kBK = 64;           // K per pipeline stage (128 B of bf16)
constexpr int kMaxBN = 256;       // MMA N limit (tokens per tile)
constexpr int kStages = 4;
constexpr int kAChunkBytes = 64 * kBK * 2;               // 8 KB: 64 M x 64 K
constexpr int kABytes = 2 * kAChunkBytes;                // 16 KB
constexpr int kBBytesMax = kMaxBN * kBK * 2;             // 32 KB
constexpr int kStageBytes = kABytes + kBBytesMax;        // 48 KB
constexpr int kNumBoxes = 4;                             // B box heights 32/64/128/256
constexpr int kEpiThreads = 128;
constexpr int kThreads = 64 + kEpiThreads;
constexpr uint32_t kTmemCols = 512;                      // 2 x 256-column accumulators
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kMaxExperts = 1024;

// Epilogue staging (per 32-column chunk)
constexpr int kUPitch = 33;                              // floats per row of the up buffer
constexpr int kUBytes = 64 * kUPitch * 4;                // 8448
constexpr int kOutBytes = 32 * 256;                      // 32 token rows x up to 128 bf16

struct Smem {
  // offsets inside the 1024-aligned dynamic smem block
  static constexpr int stages = 0;
  static constexpr int u = kStages * kStageBytes;
  static constexpr int out = u + kUBytes;
  static constexpr int bars = out + kOutBytes;                    // 8-byte aligned
  static constexpr int nbars = 2 * kStages + 4 + 1;
  static constexpr int tmem_slot = bars + nbars * 8;
  static constexpr int abort_flag = tmem_slot + 4;
  static constexpr int epi_ok = abort_flag + 4;
  static constexpr int tile_prefix = epi_ok + 4;                  // int[kMaxExperts + 1]
  static constexpr int total = tile_prefix + (kMaxExperts + 1) * 4;
};
constexpr int kSmemBytes = Smem::total + 1024;  // + alignment slack

struct TcParams {
  const int32_t *offsets;  // [N+1]
  int N;                   // experts
  int K;                   // reduction length (d or f)
  int M;                   // weight columns (f for GEMM1, d for GEMM2)
  int slabs;               // tiles along M per expert
  int gemm1;               // 1: gate/up + SwiGLU, 0: down + row scale
  __nv_bfloat16 *out;      // h [*, f] or y_perm [*, d]
  int out_ld;              // = M
  const float *row_scale;  // GEMM2 only (nullable)
  int32_t *status;
};

struct TileInfo {
  int e, slab, row0, rows;  // rows of this tile: [row0, row0 + rows) of the permuted rows
};

// Token tiles of an expert with n rows: ceil(n/256) tiles of equal width
// (rounded up to 16).
__device__ __forceinline__ int token_tiles(int n) { return (n + kMaxBN - 1) / kMaxBN; }
__device__ __forceinline__ int tile_width(int n, int jt) {
  int w = (n + jt - 1) / jt;
  return (w + 15) & ~15;
}

// prefix[e] = first global tile of expert e (slab-major inside an expert).
__device__ void build_tile_prefix(const TcParams &p, int *prefix) {
  // one warp scans the experts 32 at a time
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int base = 0;
    for (int e0 = 0; e0 < p.N; e0 += 32) {
      int e = e0 + lane;
      int n = 0;
      if (e < p.N) n = p.offsets[e + 1] - p.offsets[e];
      int cnt = n > 0 ? token_tiles(n) * p.slabs : 0;
      int incl = cnt;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < p.N) prefix[e] = base + incl - cnt;
      base += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[p.N] = base;
  }
}

__device__ __forceinline__ TileInfo decode_tile(const TcParams &p, const int *prefix, int t) {
  // binary search: last e with prefix[e] <= t (experts with no tiles share prefixes)
  int lo = 0, hi = p.N - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (prefix[mid] <= t) lo = mid; else hi = mid - 1;
  }
  const int e = lo;
  const int base = p.offsets[e];
  const int n = p.offsets[e + 1] - base;
  const int jt = token_tiles(n);
  const int local = t - prefix[e];
  const int slab = local / jt;
  const int j = local % jt;
  const int w = tile_width(n, jt);
  TileInfo ti;
  ti.e = e;
  ti.slab = slab;
  ti.row0 = base + j * w;
  ti.rows = min(w, n - j * w);
  return ti;
}

__device__ __forceinline__ int box_index(int rows) {
  return rows <= 32 ? 0 : rows <= 64 ? 1 : rows <= 128 ? 2 : 3;
}

__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_tc(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmB2,
                    const __grid_constant__ CUtensorMap tmB3, const TcParams p) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Smem::bars);
  uint64_t *full = bars;                   // [kStages]
  uint64_t *empty = bars + kStages;        // [kStages]
  uint64_t *acc_full = bars + 2 * kStages; // [2]
  uint64_t *acc_empty = acc_full + 2;      // [2]
  uint64_t *drain = acc_empty + 2;         // [1]
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::tmem_slot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Smem::abort_flag);
  int *prefix = reinterpret_cast<int *>(smem + Smem::tile_prefix);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      tc::mbar_init(&acc_full[b], 1);
      tc::mbar_init(&acc_empty[b], kEpiThreads / 32);
    }
    tc::mbar_init(drain, 1);
    *abort_flag = 0;
    tc::fence_barrier_init();
    tc::fence_proxy_async();
  }
  if (warp == 0 && lane == 0) {
    tc::tma_prefetch_desc(&tmA0);
    tc::tma_prefetch_desc(&tmA1);
    tc::tma_prefetch_desc(&tmB0);
    tc::tma_prefetch_desc(&tmB1);
    tc::tma_prefetch_desc(&tmB2);
    tc::tma_prefetch_desc(&tmB3);
  }
  if (warp == 1) {
    tc::tmem_alloc(tmem_slot, kTmemCols);
    tc::tmem_relinquish();
  }
  build_tile_prefix(p, prefix);
  tc::tc_fence_before();
  __syncthreads();
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = prefix[p.N];
  const int kblocks = (p.K + kBK - 1) / kBK;

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    if (lane == 0) {
      const uint64_t pol_w = tc::policy_evict_first();  // weights: streamed
      const uint64_t pol_x = tc::policy_evict_last();   // token rows: reused across slabs
      const CUtensorMap *tmB[kNumBoxes] = {&tmB0, &tmB1, &tmB2, &tmB3};
      uint32_t it = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x) {
        const TileInfo ti = decode_tile(p, prefix, t);
        const int bi = box_index(ti.rows);
        const uint32_t bbytes = (uint32_t)(32 << bi) * kBK * 2;
        const int m0 = ti.slab * (p.gemm1 ? 64 : kBM);
        const int m1 = p.gemm1 ? m0 : m0 + 64;
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStages;
          const uint32_t ph = (it / kStages) & 1;
          if (!tc::mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, kTimeoutNs)) { ok = false; break; }
          unsigned char *st = smem + Smem::stages + s * kStageBytes;
          tc::mbar_arrive_expect_tx(&full[s], kABytes + bbytes);
          tc::tma_load_3d(st, &tmA0, &full[s], m0, kb * kBK, ti.e, pol_w);
          tc::tma_load_3d(st + kAChunkBytes, &tmA1, &full[s], m1, kb * kBK, ti.e, pol_w);
          tc::tma_load_2d(st + kABytes, tmB[bi], &full[s], kb * kBK, ti.row0, pol_x);
        }
      }
      if (!ok) {
        // Drain: wait (bounded) for every stage still being filled.
        for (uint32_t q = (it >= kStages ? it - kStages : 0); q < it; ++q) {
          volatile int dummy = 0;
          tc::mbar_wait_bounded(&full[q % kStages], (q / kStages) & 1, &dummy, kTimeoutNs / 4);
        }
      }
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer --
    if (lane == 0) {
      uint32_t it = 0, tcount = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < total_tiles && ok; t += gridDim.x, ++tcount) {
        const TileInfo ti = decode_tile(p, prefix, t);
        const int n_mma = max(16, (ti.rows + 15) & ~15);
        const uint32_t idesc = tc::idesc_bf16(kBM, n_mma, /*a_mn=*/1, /*b_mn=*/0);
        const int buf = tcount & 1;
        const uint32_t d_tmem = tmem_base + buf * 256;
        if (!tc::mbar_wait_bounded(&acc_empty[buf], ((tcount >> 1) & 1) ^ 1, abort_flag,
                                   kTimeoutNs)) { ok = false; break; }
        tc::tc_fence_after();
        for (int kb = 0; kb < kblocks; ++kb, ++it) {
          const int s = it % kStages;
          if (!tc::mbar_wait_bounded(&full[s], (it / kStages) & 1, abort_flag, kTimeoutNs)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          const uint32_t a_addr = tc::smem_u32(smem + Smem::stages + s * kStageBytes);
          const uint32_t b_addr = a_addr + kABytes;
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k) {
            // A MN-major: 16 k-rows = two 1024-B atoms further; chunks 8 KB apart.
            const uint64_t ad = tc::sdesc_sw128(a_addr + k * 2048, kAChunkBytes, 1024);
            // B K-major: 16 k = 32 B further inside the 128-B swizzled row.
            const uint64_t bd = tc::sdesc_sw128(b_addr + k * 32, 16, 1024);
            tc::mma_f16(d_tmem, ad, bd, idesc, (kb > 0 || k > 0) ? 1u : 0u);
          }
          tc::mma_commit(&empty[s]);  // frees the stage once these MMAs finish
        }
        if (!ok) break;
        tc::mma_commit(&acc_full[buf]);
      }
      // Drain: make sure no MMA is still writing tensor memory.
      tc::mma_commit(drain);
      volatile int dummy = 0;
      tc::mbar_wait_bounded(drain, 0, &dummy, kTimeoutNs);
    }
  } else {
    // ------------------------------------------------------------ epilogue --
    const int ew = warp - 2;                 // 0..3
    const int lane_grp = warp % 4;           // TMEM lanes 32*lane_grp .. +31
    const int etid = threadIdx.x - 64;       // 0..127
    volatile int *epi_ok = reinterpret_cast<volatile int *>(smem + Smem::epi_ok);
    float *ubuf = reinterpret_cast<float *>(smem + Smem::u);
    __nv_bfloat16 *obuf = reinterpret_cast<__nv_bfloat16 *>(smem + Smem::out);
    uint32_t tcount = 0;
    for (int t = blockIdx.x; t < total_tiles; t += gridDim.x, ++tcount) {
      const TileInfo ti = decode_tile(p, prefix, t);
      const int buf = tcount & 1;
      // One thread waits (bounded) and the outcome is shared, so the four
      // epilogue warps always leave the loop together.
      if (etid == 0)
        *epi_ok = tc::mbar_wait_bounded(&acc_full[buf], (tcount >> 1) & 1, abort_flag,
                                        kTimeoutNs) ? 1 : 0;
      tc::named_bar(1, kEpiThreads);
      const int go = *epi_ok;
      tc::named_bar(1, kEpiThreads);
      if (!go) break;
      tc::tc_fence_after();
      const uint32_t t_base = tmem_base + ((uint32_t)(lane_grp * 32) << 16) + buf * 256;
      const int nchunks = (ti.rows + 31) / 32;
      for (int cc = 0; cc < nchunks; ++cc) {
        uint32_t r[32];
        tc::tmem_ld_32x32b_x32(t_base + cc * 32, r);
        tc::tmem_ld_wait();
        const int ncols = min(32, ti.rows - cc * 32);
        if (p.gemm1) {
          // lanes 64..127 (up) hand their values to lanes 0..63 (gate)
          if (lane_grp >= 2) {
            float *urow = ubuf + ((lane_grp - 2) * 32 + lane) * kUPitch;
#pragma unroll
            for (int c = 0; c < 32; ++c) urow[c] = __uint_as_float(r[c]);
          }
          tc::named_bar(1, kEpiThreads);
          if (lane_grp < 2) {
            const int hr = lane_grp * 32 + lane;          // hidden unit within the slab
            const float *urow = ubuf + hr * kUPitch;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float g = __uint_as_float(r[c]);
              const float h = g / (1.f + __expf(-g)) * urow[c];
              obuf[c * 64 + hr] = __float2bfloat16_rn(h);
            }
          }
          tc::named_bar(1, kEpiThreads);
          // copy out: ncols token rows x 64 hidden units (128 B) each
          const int m0 = ti.slab * 64;
          const int vec_valid = min(8, (p.M - m0) / 8);
          for (int q = etid; q < ncols * 8; q += kEpiThreads) {
            const int c = q / 8, v = q % 8;
            if (v < vec_valid) {
              const uint4 val = *reinterpret_cast<const uint4 *>(obuf + c * 64 + v * 8);
              *reinterpret_cast<uint4 *>(p.out + (size_t)(ti.row0 + cc * 32 + c) * p.out_ld +
                                         m0 + v * 8) = val;
            }
          }
          tc::named_bar(1, kEpiThreads);
        } else {
          // scale each token column by its gate weight
          float sc = 1.f;
          if (p.row_scale && lane < ncols) sc = p.row_scale[ti.row0 + cc * 32 + lane];
          const int dr = lane_grp * 32 + lane;             // output column within the slab
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float s = __shfl_sync(0xffffffffu, sc, c);
            obuf[c * 128 + dr] = __float2bfloat16_rn(__uint_as_float(r[c]) * s);
          }
          tc::named_bar(1, kEpiThreads);
          const int m0 = ti.slab * kBM;
          const int vec_valid = min(16, (p.M - m0) / 8);
          for (int q = etid; q < ncols * 16; q += kEpiThreads) {
            const int c = q / 16, v = q % 16;
            if (v < vec_valid) {
              const uint4 val = *reinterpret_cast<const uint4 *>(obuf + c * 128 + v * 8);
              *reinterpret_cast<uint4 *>(p.out + (size_t)(ti.row0 + cc * 32 + c) * p.out_ld +
                                         m0 + v * 8) = val;
            }
          }
          tc::named_bar(1, kEpiThreads);
        }
      }
      tc::tc_fence_before();
      if (lane == 0) tc::mbar_arrive(&acc_empty[buf]);
      (void)ew;
    }
  }

  __syncthreads();
  if (*abort_flag && threadIdx.x == 0) report(p.status, MOE_DEV_TIMEOUT);
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc(tmem_base, kTmemCols);
  }
}

// ----------------------------------------------------------------- host ----
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// Weights W[N][K][M] (M contiguous), box 64(M) x 64(K) x 1.
bool make_weight_map(CUtensorMap *m, const void *W, int N, int K, int M) {
  cuuint64_t dims[3] = {(cuuint64_t)M, (cuuint64_t)K, (cuuint64_t)N};
  cuuint64_t strides[2] = {(cuuint64_t)M * 2, (cuuint64_t)K * M * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kBK, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(W), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Token rows X[rows][K] (K contiguous), box 64(K) x box_rows.
bool make_rows_map(CUtensorMap *m, const void *X, int rows, int K, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K * 2};
  cuuint32_t box[2] = {(cuuint32_t)kBK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(X), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int n = 0;
  if (!n) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (n <= 0) n = 148;
  }
  return n;
}

moe_status_t launch_gemm(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap *b,
                         const TcParams &p, cudaStream_t stream) {
  static bool attr_set = false;
  if (!attr_set) {
    MOE_CUDA_TRY(cudaFuncSetAttribute(grouped_gemm_tc,
                                      cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes));
    attr_set = true;
  }
  grouped_gemm_tc<<<num_sms(), kThreads, kSmemBytes, stream>>>(a0, a1, b[0], b[1], b[2], b[3],
                                                               p);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace

// x_perm [A_max, d] -> h [A_max, f] -> y_perm [A_max, d], bf16, per expert.
moe_status_t launch_ffn_tc(const void *x_perm, const int32_t *offsets, const float *row_scale,
                           int A_max, int d, int f, int N, const void *W_gate, const void *W_up,
                           const void *W_down, void *h, void *y_perm, int32_t *device_status,
                           cudaStream_t stream) {
  if (A_max == 0) return MOE_OK;
  if (!encode_fn()) {
    set_error("cuTensorMapEncodeTiled unavailable from the driver");
    return MOE_ERR_CUDA;
  }
  if (N > kMaxExperts) {
    set_error("tensor-core FFN supports N <= %d experts", kMaxExperts);
    return MOE_ERR_UNSUPPORTED;
  }
  CUtensorMap wg, wu, wd, bx[kNumBoxes], bh[kNumBoxes];
  bool ok = make_weight_map(&wg, W_gate, N, d, f) && make_weight_map(&wu, W_up, N, d, f) &&
            make_weight_map(&wd, W_down, N, f, d);
  for (int i = 0; i < kNumBoxes; ++i) {
    ok = ok && make_rows_map(&bx[i], x_perm, A_max, d, 32 << i) &&
         make_rows_map(&bh[i], h, A_max, f, 32 << i);
  }
  if (!ok) {
    set_error("tensor map encoding failed (alignment or size)");
    return MOE_ERR_INVALID_ARG;
  }
  TcParams p1{offsets, N, d, f, (f + 63) / 64, 1, static_cast<__nv_bfloat16 *>(h), f, nullptr,
              device_status};
  moe_status_t s = launch_gemm(wg, wu, bx, p1, stream);
  if (s != MOE_OK) return s;
  TcParams p2{offsets, N, f, d, (d + kBM - 1) / kBM, 0, static_cast<__nv_bfloat16 *>(y_perm), d,
              row_scale, device_status};
  return launch_gemm(wd, wd, bh, p2, stream);
}

}  // namespace moe
