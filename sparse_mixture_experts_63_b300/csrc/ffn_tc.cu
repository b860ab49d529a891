// Grouped SwiGLU expert FFN on the 5th-generation tensor cores (tcgen05).
//
// Source: "MoE 分片：混合專家模型的平行化策略", section 什麼是 MoE 模型 (an
// expert is two linear maps with an activation between) and section 動態 token
// 路由 step 4 (each expert runs on the tokens routed to it);
// "MoE稀疏激活原理与工程实践", 3.1 (tokens regrouped by expert so each expert
// runs once per batch -- here one persistent launch covers every expert).
// SwiGLU reading: h = SiLU(x W_gate) * (x W_up), y_perm = row_scale * (h W_down).
//
// Formulation ("swap AB"): the weights are the M operand and the expert's
// tokens the N operand, so a tile's N is that expert's row count rounded up
// to 16 (no padding of small experts to 128 rows).  Two CTAs of a cluster
// share one MMA (tcgen05 cta_group::2, M = 256): CTA r holds 128 weight rows
// and half of the token rows, and gets its 128 rows of D in its own tensor
// memory.  Per CTA:
//   GEMM1  D[128 x n] = [W_gate[:, f0:f0+64] | W_up[:, f0:f0+64]]^T x x_perm^T
//          lanes 0-63 hold gate, lanes 64-127 up for the same 64 hidden units
//          (f0 = 128 * pair + 64 * r); the epilogue writes h = SiLU(gate) * up.
//   GEMM2  D[128 x n] = W_down[:, m0:m0+128]^T x h^T   (m0 = 256 * pair + 128 * r)
//          the epilogue writes y_perm = row_scale * D (bf16).
// A (weights) is read MN-major straight from W[N, K, M] by 3-D TMA boxes of
// 64(M) x 64(K) with 128-byte swizzle; B (token rows, K contiguous) is read
// K-major by 2-D boxes of 64(K) x {32,64,80,128}(rows), half a sub-tile per CTA.
// Sharing the token tile halves each CTA's bytes per MMA cycle, so 5-9 stages
// of 20-36 KB cover the ~2 us load latency that four 48 KB stages of a one-CTA
// tile could not (the tensor pipe sat ~30% idle waiting for data).
//
// CTA = 6 warps, persistent (one CTA pair per two SMs):
//   warp 0      TMA producer (both CTAs; completions land on the even CTA's barriers)
//   warp 1      tensor-memory allocator; MMA issuer in the even CTA
//   warps 2..5  epilogue (tcgen05.ld of their 32 lanes, math, coalesced stores)
// Pipelines: shared-memory stages (full/empty mbarriers) and a ring of 32-column
// accumulator chunks in tensor memory (acc_full per sub-tile, col_free per
// chunk), so the epilogue of one (sub-)tile overlaps the MMAs of the next.  Every wait is bounded (2 s):
// on timeout the CTA sets MOE_DEV_TIMEOUT, drains what it issued and exits
// cleanly.
#include <cuda.h>
#include <math.h>

#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kBM = 128;          // weight rows per CTA (MMA M = 256 per pair)
constexpr int kBK = 64;           // K per pipeline stage (128 B of bf16)
constexpr int kMaxStages = 10;
constexpr int kAChunkBytes = 64 * kBK * 2;               // 8 KB: 64 M x 64 K
constexpr int kABytes = 2 * kAChunkBytes;                // 16 KB
constexpr int kStageRegion = 192 * 1024;                 // shared memory for all stages
// Token tiling.  A tile is one expert's weight pair times up to tile_cap of its
// token rows: tile_cap 64/128/256, one MMA (N <= 256) per 16 K.  Wide layers
// (experts of ~250-320 rows, where cutting an expert into two tiles would
// stream its weights through the SMs twice) take tile_cap 320: a tile over 256
// rows runs as two balanced token sub-tiles of <= 160 rows that share every
// weight stage (two MMAs per 16 K).
// A stage holds 16 KB of weights and the tile's token rows (half per CTA):
// tile_cap 256 -> 32 KB stages x 6; 128 -> 24 KB x 8; 64 -> 20 KB x 9;
// wide -> 16 KB + 2 x 80 rows = 36 KB x 5.  The stage region holds the weight
// parts of all stages first and the token parts after them (measured ~1%
// faster than keeping each stage's two parts adjacent).  Both parts of a
// stage share one full and one empty barrier: a second barrier pair per
// stage (separate weight and token rings, so the weights could be fetched
// further ahead) put a second wait and commit into the MMA issuer's loop per
// K step and made every layer 3-12% slower.
// Accumulators: tensor memory is a ring of 16 chunks of 32 columns; each
// sub-tile takes ceil(N/32) consecutive chunks (wrapping to chunk 0 when the
// rest of the ring is too short), and the epilogue hands every chunk back as
// soon as it has loaded it, so the next sub-tile's MMAs start while the
// epilogue still works on the previous one.
constexpr int kWideSub = 160;                            // sub-tile cap in a split wide tile
constexpr int kWideTile = 2 * kWideSub;
constexpr int kSubBytes = (kWideSub / 2) * kBK * 2;      // 10 KB: 80 rows per CTA
constexpr int kNumBoxes = 4;                             // B box heights 32/64/80/128
constexpr int kChunks = 16;                              // 32-column chunks of tensor memory
constexpr int kAccRing = 16;                             // acc_full barriers (sub-tile ring)
constexpr int kEpiThreads = 128;
// Warps: 0 TMA producer, 1 MMA issuer (and tensor-memory allocator), with two
// MMA issuers (wide layers) 2 the second issuer; then 4 epilogue warps.
constexpr int epi_warp0(bool dual) { return dual ? 3 : 2; }
constexpr int threads_for(bool dual) { return 32 * epi_warp0(dual) + kEpiThreads; }
constexpr int kMaxThreads = threads_for(true);
constexpr uint32_t kTmemCols = 512;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr int kMaxExperts = 1024;

// Epilogue staging (per 32-column chunk)
constexpr int kXPitch = 20;                              // floats per row of a swap buffer
                                                         // (16-B rows, float4 conflict-free)
constexpr int kXHalf = 64 * kXPitch;                     // floats per swap buffer
constexpr int kXBytes = 2 * kXHalf * 4;                  // 10 KB: gate->up and up->gate
constexpr int kOutHalf = 32 * 128;                       // bf16 per output buffer (8 KB)
constexpr int kOutBytes = 2 * kOutHalf * 2;              // two output buffers

struct Smem {
  // offsets inside the 1024-aligned dynamic smem block
  static constexpr int stages = 0;
  static constexpr int x = kStageRegion;
  static constexpr int out = x + kXBytes;
  static constexpr int bars = out + kOutBytes;                    // 8-byte aligned
  static constexpr int nbars = 2 * kMaxStages + kAccRing + kChunks + 2;
  static constexpr int tmem_slot = bars + nbars * 8;
  static constexpr int abort_flag = tmem_slot + 4;
  static constexpr int epi_ok = abort_flag + 4;
  static constexpr int tile_prefix = epi_ok + 4;                  // int[kMaxExperts + 1]
  static constexpr int total = tile_prefix + (kMaxExperts + 1) * 4;
};
constexpr int kSmemBytes = Smem::total + 1024;  // + alignment slack
static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");

struct TcParams {
  const int32_t *offsets;  // [N+1]
  int N;                   // experts
  int K;                   // reduction length (d or f)
  int M;                   // weight columns (f for GEMM1, d for GEMM2)
  int pairs;               // tiles along M per expert (256 weight rows each)
  int gemm1;               // 1: gate/up + SwiGLU, 0: down + row scale
  __nv_bfloat16 *out;      // h [*, f] or y_perm [*, d]
  int out_ld;              // = M
  const float *row_scale;  // GEMM2 only (nullable)
  int32_t *status;
  int group;               // token tiles per raster group (see decode_tile)
  int tile_cap;            // token rows per tile: 64, 128, 256, or 320 (wide)
  int wide;                // 1: tiles over 256 rows run as two sub-tiles
  int stages;              // pipeline stages (kStageRegion / stage_bytes)
  int kgroup;              // stages per barrier pair (1 or 2; divides stages): selects
                           // the kernel instance
  int stage_bytes;         // kABytes + token rows of a stage (both sub-tiles)
  // FP8 (E4M3 weights and rows, K-major): D is multiplied by the output
  // channel's scale and the row's scale before the epilogue's math
  const float *wscale_g;   // [N, M] channel scales (GEMM1: gate; GEMM2: down)
  const float *wscale_u;   // [N, M] up channel scales (GEMM1)
  const float *xscale;     // row scales: [T] by token (GEMM1) or [A] by permuted row (GEMM2)
  const int32_t *perm_token;  // [A] token of each permuted row (GEMM1), else null
  int out_f32;             // GEMM1: h written in fp32 (out holds floats), else bf16
  // GEMM2: row p of the result goes to out row out_row[p] (null: row p); an
  // index outside [0, rows_out) stores nothing and sets MOE_DEV_BAD_ROW
  const int32_t *out_row;
  int rows_out;
};

// Token sub-tiles of a tile: rows [row0, row0 + rows0) and, for a wide tile
// over 256 rows, [row0 + rows0, row0 + rows0 + rows1).
struct TileInfo {
  int e, pair, row0, rows0, rows1;
};

// Token tiles of an expert with n rows: ceil(n/tile_cap) tiles of equal width
// (rounded up to 32).
__device__ __forceinline__ int token_tiles(int n, int cap) { return (n + cap - 1) / cap; }
__device__ __forceinline__ int tile_width(int n, int jt) {
  int w = (n + jt - 1) / jt;
  return (w + 31) & ~31;
}
// MMA N of a sub-tile: its rows rounded up to 16, at least 64.
__device__ __forceinline__ int mma_n(int rows) { return max(64, (rows + 15) & ~15); }

// prefix[e] = first global tile of expert e (pair-major inside an expert).
__device__ void build_tile_prefix(const TcParams &p, int *prefix) {
  // one warp scans the experts 32 at a time
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    int base = 0;
    for (int e0 = 0; e0 < p.N; e0 += 32) {
      int e = e0 + lane;
      int n = 0;
      if (e < p.N) n = p.offsets[e + 1] - p.offsets[e];
      int cnt = n > 0 ? token_tiles(n, p.tile_cap) * p.pairs : 0;
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

// Tile order inside an expert: token tiles in groups of p.group; for each
// group, every weight pair; inside that, the group's token tiles.  Tiles that
// run at the same time then share both operands through L2 (a group's token
// rows are sized on the host to stay resident), instead of every weight pair
// re-streaming all of a large expert's token rows.
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
  const int jt = token_tiles(n, p.tile_cap);
  const int local = t - prefix[e];
  const int full_groups = jt / p.group;
  const int per_group = p.group * p.pairs;
  int g, gsize, idx;
  if (local < full_groups * per_group) {
    g = local / per_group;
    gsize = p.group;
    idx = local - g * per_group;
  } else {
    g = full_groups;
    gsize = jt - full_groups * p.group;
    idx = local - full_groups * per_group;
  }
  const int pair = idx / gsize;
  const int j = g * p.group + idx % gsize;
  const int w = tile_width(n, jt);
  const int rows = min(w, n - j * w);
  TileInfo ti;
  ti.e = e;
  ti.pair = pair;
  ti.row0 = base + j * w;
  if (p.wide && rows > 256) {
    ti.rows0 = ((rows + 1) / 2 + 15) & ~15;   // 144..160
    ti.rows1 = rows - ti.rows0;                // 113..160
  } else {
    ti.rows0 = rows;
    ti.rows1 = 0;
  }
  return ti;
}

// B box per CTA for a sub-tile of MMA width n: n/2 rows -> 32, 64, 80 or 128.
__device__ __forceinline__ int box_index(int n_mma) {
  const int half = n_mma / 2;
  return half <= 32 ? 0 : half <= 64 ? 1 : half <= 80 ? 2 : 3;
}
__device__ __forceinline__ uint32_t box_bytes(int bi) {
  return (uint32_t)(bi == 0 ? 32 : bi == 1 ? 64 : bi == 2 ? 80 : 128) * kBK * 2;
}

// Tensor-memory chunks of a sub-tile of MMA width n, taken from the ring at
// *pos (wrapping to 0 when fewer than needed remain before the end).
__device__ __forceinline__ int ring_take(int &pos, int n_mma) {
  const int nch = (n_mma + 31) / 32;
  if (pos + nch > kChunks) pos = 0;
  const int c0 = pos;
  pos += nch;
  return c0;
}

// Epilogue of one 32-column chunk of accumulators (r: this thread's TMEM
// lane, 32 token columns): GEMM1 writes h = SiLU(gate) * up, GEMM2 writes
// y_perm = row_scale * D, both staged through shared memory into coalesced
// 16-B row stores.  All 128 epilogue threads call it together.
__device__ __forceinline__ void epilogue_chunk(const TcParams &p, const TileInfo &ti,
                                               uint32_t rank, int lane_grp, int lane, int etid,
                                               float *xbuf, __nv_bfloat16 *obuf, uint32_t &obi,
                                               int srow0, int srows, int cc,
                                               const uint32_t (&r)[32]) {
  const int ncols = min(32, srows - cc * 32);
  if (p.gemm1) {
    // Gate lanes (lane_grp 0,1) and up lanes (2,3) of the same hidden unit
    // hand each other half of the 32 token columns, so all four warps compute
    // SiLU(gate) * up for 16 columns.
    const bool gate_side = lane_grp < 2;
    const int hr = (lane_grp & 1) * 32 + lane;     // hidden unit within the slab
    float4 *mine = reinterpret_cast<float4 *>(xbuf + (gate_side ? kXHalf : 0) + hr * kXPitch);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int c = 4 * q;
      mine[q] = gate_side ? make_float4(__uint_as_float(r[16 + c]), __uint_as_float(r[17 + c]),
                                        __uint_as_float(r[18 + c]), __uint_as_float(r[19 + c]))
                          : make_float4(__uint_as_float(r[c]), __uint_as_float(r[c + 1]),
                                        __uint_as_float(r[c + 2]), __uint_as_float(r[c + 3]));
    }
    tc::named_bar(1, kEpiThreads);
    const float4 *other4 =
        reinterpret_cast<const float4 *>(xbuf + (gate_side ? 0 : kXHalf) + hr * kXPitch);
    // h of token column c (this side's 16) and hidden unit hr at [c * 64 + hr]
    __nv_bfloat16 *ob = obuf + (gate_side ? 0 : 16 * 64);
    float *obf = reinterpret_cast<float *>(obuf) + (gate_side ? 0 : 16 * 64);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float4 o4 = other4[q];
      const float o[4] = {o4.x, o4.y, o4.z, o4.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = 4 * q + i;
        const float g = gate_side ? __uint_as_float(r[c]) : o[i];
        const float u = gate_side ? o[i] : __uint_as_float(r[16 + c]);
        const float h = __fdividef(g, 1.f + __expf(-g)) * u;
        if (p.out_f32)
          obf[c * 64 + hr] = h;
        else
          ob[c * 64 + hr] = __float2bfloat16_rn(h);
      }
    }
    tc::named_bar(1, kEpiThreads);
    // copy out: ncols token rows x 64 hidden units (128 B in bf16, 256 B in
    // fp32) each.  The next chunk writes obuf only after its exchange barrier,
    // which every thread reaches after finishing this copy.
    const int m0 = ti.pair * 128 + rank * 64;
    if (p.out_f32) {
      const float *src = reinterpret_cast<const float *>(obuf);
      float *dst = reinterpret_cast<float *>(p.out);
      const int vec_valid = max(0, min(16, (p.M - m0) / 4));
      for (int q = etid; q < ncols * 16; q += kEpiThreads) {
        const int c = q / 16, v = q % 16;
        if (v < vec_valid) {
          const uint4 val = *reinterpret_cast<const uint4 *>(src + c * 64 + v * 4);
          *reinterpret_cast<uint4 *>(dst + (size_t)(srow0 + cc * 32 + c) * p.out_ld + m0 +
                                     v * 4) = val;
        }
      }
    } else {
      const int vec_valid = max(0, min(8, (p.M - m0) / 8));
      for (int q = etid; q < ncols * 8; q += kEpiThreads) {
        const int c = q / 8, v = q % 8;
        if (v < vec_valid) {
          const uint4 val = *reinterpret_cast<const uint4 *>(obuf + c * 64 + v * 8);
          *reinterpret_cast<uint4 *>(p.out + (size_t)(srow0 + cc * 32 + c) * p.out_ld + m0 +
                                     v * 8) = val;
        }
      }
    }
  } else {
    // scale each token column by its gate weight; two output buffers
    // alternate, so a chunk's writes never meet the previous chunk's copy
    __nv_bfloat16 *ob = obuf + (obi & 1) * kOutHalf;
    ++obi;
    float scl = 1.f;
    if (p.row_scale && lane < ncols) scl = p.row_scale[srow0 + cc * 32 + lane];
    const int dr = lane_grp * 32 + lane;             // output column within the slab
#pragma unroll
    for (int c = 0; c < 32; ++c) {
      const float sv = __shfl_sync(0xffffffffu, scl, c);
      ob[c * 128 + dr] = __float2bfloat16_rn(__uint_as_float(r[c]) * sv);
    }
    tc::named_bar(1, kEpiThreads);
    const int m0 = ti.pair * 256 + rank * kBM;
    const int vec_valid = max(0, min(16, (p.M - m0) / 8));
    for (int q = etid; q < ncols * 16; q += kEpiThreads) {
      const int c = q / 16, v = q % 16;
      if (v < vec_valid) {
        int orow = srow0 + cc * 32 + c;
        if (p.out_row) {
          orow = p.out_row[orow];
          if (orow < 0 || orow >= p.rows_out) {
            if (v == 0) report(p.status, MOE_DEV_BAD_ROW);
            continue;
          }
        }
        const uint4 val = *reinterpret_cast<const uint4 *>(ob + c * 128 + v * 8);
        *reinterpret_cast<uint4 *>(p.out + (size_t)orow * p.out_ld + m0 + v * 8) = val;
      }
    }
  }
}

// FP8: D of a 32-column chunk (permuted rows row0 .. row0 + 31, of which
// `valid` hold rows) times this thread's channel scale and each column's row
// scale (GEMM1: the token's, through perm_token; GEMM2: h's own row scale).
__device__ __forceinline__ void scale_chunk(const TcParams &p, int row0, int valid, int lane,
                                            float wsc, uint32_t (&r)[32]) {
  const float sxl =
      lane < valid ? p.xscale[p.perm_token ? p.perm_token[row0 + lane] : row0 + lane] : 0.f;
#pragma unroll
  for (int c = 0; c < 32; ++c)
    r[c] = __float_as_uint(__uint_as_float(r[c]) * (wsc * __shfl_sync(0xffffffffu, sxl, c)));
}

// FP8: E4M3 weights [N, M, K] and token (or h) rows, both K-major, 128 K per
// stage (the same 128-byte rows as 64 bf16), kind::f8f6f4 MMAs, and the
// channel x row scales applied to D before SwiGLU (GEMM1) or the gate-weight
// scale (GEMM2).
template <bool FP8, int G, bool DUAL>
__global__ void __launch_bounds__(kMaxThreads, 1)
    grouped_gemm_tc(const __grid_constant__ CUtensorMap tmA0,
                    const __grid_constant__ CUtensorMap tmA1,
                    const __grid_constant__ CUtensorMap tmB0,
                    const __grid_constant__ CUtensorMap tmB1,
                    const __grid_constant__ CUtensorMap tmB2,
                    const __grid_constant__ CUtensorMap tmB3, const TcParams p) {
  // the next kernel may start launching; this one's set-up (barriers, tensor
  // memory, descriptor prefetch) overlaps the previous kernel's tail
  pdl_trigger();
  extern __shared__ unsigned char smem_raw[];
  unsigned char *smem = reinterpret_cast<unsigned char *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Smem::bars);
  uint64_t *full = bars;                        // [kMaxStages] (used in the even CTA)
  uint64_t *empty = bars + kMaxStages;          // [kMaxStages]
  uint64_t *acc_full = bars + 2 * kMaxStages;   // [kAccRing] sub-tile accumulated
  uint64_t *col_free = acc_full + kAccRing;     // [kChunks]  chunk loaded by the epilogue
                                                //            (used in the even CTA)
  uint64_t *drain = col_free + kChunks;         // [2] one per MMA issuer
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Smem::tmem_slot);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + Smem::abort_flag);
  int *prefix = reinterpret_cast<int *>(smem + Smem::tile_prefix);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = tc::cluster_ctarank();   // 0: even CTA (issues the MMAs)
  const int cid = (int)tc::cluster_id_x();
  const int ncl = (int)tc::nclusters_x();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kMaxStages; ++s) {
      tc::mbar_init(&full[s], 1);
      tc::mbar_init(&empty[s], DUAL ? 2 : 1);   // each MMA issuer commits every group
    }
    for (int b = 0; b < kAccRing; ++b) tc::mbar_init(&acc_full[b], 1);
    for (int c = 0; c < kChunks; ++c) tc::mbar_init(&col_free[c], 2 * kEpiThreads / 32);
    tc::mbar_init(&drain[0], 1);
    tc::mbar_init(&drain[1], 1);
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
    tc::tmem_alloc_pair(tmem_slot, kTmemCols);
    tc::tmem_relinquish_pair();
  }
  pdl_wait();   // the offsets and rows come from the previous kernels
  build_tile_prefix(p, prefix);
  tc::tc_fence_before();
  __syncthreads();
  tc::cluster_sync();   // the peer's barriers are initialised before any remote use
  tc::tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = prefix[p.N];
  constexpr int kKStage = FP8 ? 128 : kBK;        // K elements per stage (128 B rows)
  const int kblocks = (p.K + kKStage - 1) / kKStage;

  if (warp == 0) {
    // ------------------------------------------------------------ producer --
    // Lane 0 runs a tight loop (stage/phase counters, no divisions); the copies
    // complete on the even CTA's full barrier.
    if (lane == 0) {
      const uint64_t pol_w = tc::policy_evict_normal();  // weights: shared by a group's tiles
      const uint64_t pol_x = tc::policy_evict_last();    // token rows: reused across pairs
      unsigned char *stage0 = smem + Smem::stages;
      // the even CTA's full barriers, in cluster address space (contiguous, 8 B apart)
      const uint32_t full_leader0 = tc::mapa_shared(&full[0], 0);
      const int ngroups = p.stages / G;          // G: stages per barrier pair
      const int bbytes = p.stage_bytes - kABytes;   // token part of a stage
      int g = 0;            // barrier group: stages g*G .. g*G+G-1
      uint32_t ph = 0;
      uint32_t issued = 0;
      bool ok = true;
      for (int t = cid; t < total_tiles && ok; t += ncl) {
        const TileInfo ti = decode_tile(p, prefix, t);
        const int n0 = mma_n(ti.rows0);
        const int bi0 = box_index(n0);
        const CUtensorMap *tb0 = bi0 == 0 ? &tmB0 : bi0 == 1 ? &tmB1 : bi0 == 2 ? &tmB2 : &tmB3;
        const int n1 = ti.rows1 > 0 ? mma_n(ti.rows1) : 0;
        const int bi1 = box_index(n1);
        const CUtensorMap *tb1 = bi1 == 0 ? &tmB0 : bi1 == 1 ? &tmB1 : bi1 == 2 ? &tmB2 : &tmB3;
        uint32_t tx = kABytes + box_bytes(bi0);
        if (n1) tx += box_bytes(bi1);
        tx *= 2u;   // both CTAs' bytes complete on the even CTA's barrier
        const int m0 = p.gemm1 ? ti.pair * 128 + rank * 64 : ti.pair * 256 + rank * kBM;
        const int m1 = p.gemm1 ? m0 : m0 + 64;
        const int brow0 = ti.row0 + (int)rank * (n0 / 2);
        const int brow1 = ti.row0 + ti.rows0 + (int)rank * (n1 / 2);
        // K steps go in groups of G (the last group of a tile may be shorter),
        // one full and one empty barrier per group
        for (int kb = 0; kb < kblocks; kb += G) {
          const int nk = min(G, kblocks - kb);
          if (!tc::mbar_wait_bounded(&empty[g], ph ^ 1, abort_flag, kTimeoutNs)) {
            ok = false;
            break;
          }
          if (rank == 0) tc::mbar_arrive_expect_tx(&full[g], tx * (uint32_t)nk);
          const uint32_t fb = full_leader0 + 8u * g;
          for (int h = 0; h < nk; ++h) {
            const int slot = g * G + h;
            unsigned char *st = stage0 + slot * kABytes;                  // weight part
            unsigned char *stb = stage0 + p.stages * kABytes + slot * bbytes;   // token part
            const int kc = (kb + h) * kKStage;
            if (FP8) {   // K-major weights W[N][M][K]: coordinates (k, m, e)
              tc::tma_load_3d_pair(st, &tmA0, fb, kc, m0, ti.e, pol_w);
              tc::tma_load_3d_pair(st + kAChunkBytes, &tmA1, fb, kc, m1, ti.e, pol_w);
            } else {     // MN-major weights W[N][K][M]: coordinates (m, k, e)
              tc::tma_load_3d_pair(st, &tmA0, fb, m0, kc, ti.e, pol_w);
              tc::tma_load_3d_pair(st + kAChunkBytes, &tmA1, fb, m1, kc, ti.e, pol_w);
            }
            tc::tma_load_2d_pair(stb, tb0, fb, kc, brow0, pol_x);
            if (n1) tc::tma_load_2d_pair(stb + kSubBytes, tb1, fb, kc, brow1, pol_x);
          }
          ++issued;
          if (++g == ngroups) { g = 0; ph ^= 1; }
        }
      }
      if (!ok && rank == 0) {
        // Drain: wait (bounded) for every group still being filled (both CTAs'
        // bytes complete on these barriers).
        const uint32_t ns = (uint32_t)ngroups;
        const uint32_t first = issued >= ns ? issued - ns : 0;
        for (uint32_t q = first; q < issued; ++q) {
          volatile int dummy = 0;
          tc::mbar_wait_bounded(&full[q % ns], (q / ns) & 1, &dummy, kTimeoutNs / 4);
        }
      }
    }
    __syncwarp();
  } else if (warp == 1 || (DUAL && warp == 2)) {
    // --------------------------------------------------------- MMA issuers --
    // Even CTA only.  Lane 0 of warp 1 issues the first token sub-tile's MMAs,
    // lane 0 of warp 2 the second's (wide layers): one tcgen05.mma takes ~72
    // cycles to issue whatever its N, so one thread issuing both sub-tiles'
    // eight MMAs per K step fell behind the tensor pipe.  Both walk the same
    // tiles and stages, wait on every full barrier and commit every stage
    // group (the empty barriers count two arrivals), and both track every
    // tensor-memory chunk's uses, waiting only for their own sub-tile's.
    // Each loop stays tight: the gap between the last MMA of one stage and the
    // first of the next must stay shorter than the work the tensor pipe still
    // has queued, or it idles.
    // Layers without wide tiles have one token sub-tile per tile: their kernel
    // instance has the first issuer only (DUAL false, one arrival per stage).
    const int role = warp - 1;   // 0: sub-tile 0, 1: sub-tile 1
    if (rank == 0 && lane == 0) {
      const uint32_t stage0 = tc::smem_u32(smem + Smem::stages);
      // descriptors of stage 0; stage s adds (s * stage_bytes) >> 4 to the start field
      // A MN-major (bf16) or K-major (FP8: 128 rows of 128 B, 8-row atoms)
      const uint64_t a_desc0 = FP8 ? tc::sdesc_sw128(stage0, 16, 1024)
                                   : tc::sdesc_sw128(stage0, kAChunkBytes, 1024);
      const uint64_t b_desc0 =
          tc::sdesc_sw128(stage0 + (uint32_t)(p.stages * kABytes), 16, 1024);   // K-major B
      const int ngroups = p.stages / G;
      const int bbytes = p.stage_bytes - kABytes;
      int g = 0;            // barrier group, as in the producer
      uint32_t ph = 0;
      int pos = 0;              // tensor-memory ring position (chunks)
      uint32_t cuse = 0;        // bit c: parity of chunk c's uses so far
      uint32_t k = 0;           // token sub-tiles so far
      bool ok = true;
      for (int t = cid; t < total_tiles && ok; t += ncl) {
        const TileInfo ti = decode_tile(p, prefix, t);
        const bool two = ti.rows1 > 0;
        const int n0 = mma_n(ti.rows0), n1 = two ? mma_n(ti.rows1) : 0;
        const uint32_t idesc0 = FP8 ? tc::idesc_e4m3(2 * kBM, n0)
                                    : tc::idesc_bf16(2 * kBM, n0, /*a_mn=*/1, /*b_mn=*/0);
        const uint32_t idesc1 = !two ? 0u
                                : FP8 ? tc::idesc_e4m3(2 * kBM, n1)
                                      : tc::idesc_bf16(2 * kBM, n1, 1, 0);
        const int c0 = ring_take(pos, n0);
        const int c1 = two ? ring_take(pos, n1) : c0;
        // every chunk of the sub-tiles must have been loaded by the epilogue
        // since its previous use
        const int e0 = c0 + (n0 + 31) / 32;
        for (int c = c0; c < e0 && ok; ++c) {
          if (role == 0)
            ok = tc::mbar_wait_bounded(&col_free[c], ((cuse >> c) & 1) ^ 1, abort_flag,
                                       kTimeoutNs);
          cuse ^= 1u << c;
        }
        if (two) {
          const int e1 = c1 + (n1 + 31) / 32;
          for (int c = c1; c < e1 && ok; ++c) {
            if (role == 1)
              ok = tc::mbar_wait_bounded(&col_free[c], ((cuse >> c) & 1) ^ 1, abort_flag,
                                         kTimeoutNs);
            cuse ^= 1u << c;
          }
        }
        if (!ok) break;
        const uint32_t d0 = tmem_base + (uint32_t)(c0 * 32);
        const uint32_t d1 = tmem_base + (uint32_t)(c1 * 32);
        tc::tc_fence_after();
        for (int kb = 0; kb < kblocks; kb += G) {
          const int nk = min(G, kblocks - kb);
          if (!tc::mbar_wait_bounded(&full[g], ph, abort_flag, kTimeoutNs)) {
            ok = false;
            break;
          }
          tc::tc_fence_after();
          for (int h = 0; h < nk; ++h) {
            const int slot = g * G + h;
            const uint64_t ad = a_desc0 + (uint64_t)((slot * kABytes) >> 4);
            const uint64_t bd = b_desc0 + (uint64_t)((slot * bbytes) >> 4);
            const uint32_t acc = (kb + h) > 0 ? 1u : 0u;   // the tile's first K step overwrites
            if (FP8) {
              // both K-major: 32 k of 8 bits = 32 B further inside the 128-B rows (+2)
              if (role == 0) {
                tc::mma_f8_pair(d0, ad, bd, idesc0, acc);
                tc::mma_f8_pair(d0, ad + 2, bd + 2, idesc0, 1u);
                tc::mma_f8_pair(d0, ad + 4, bd + 4, idesc0, 1u);
                tc::mma_f8_pair(d0, ad + 6, bd + 6, idesc0, 1u);
              } else if (two) {
                const uint64_t bd1 = bd + (kSubBytes >> 4);
                tc::mma_f8_pair(d1, ad, bd1, idesc1, acc);
                tc::mma_f8_pair(d1, ad + 2, bd1 + 2, idesc1, 1u);
                tc::mma_f8_pair(d1, ad + 4, bd1 + 4, idesc1, 1u);
                tc::mma_f8_pair(d1, ad + 6, bd1 + 6, idesc1, 1u);
              }
            } else {
              // A MN-major: 16 k-rows = two 1024-B atoms further (+128 in 16-B units);
              // B K-major: 16 k = 32 B further inside the 128-B swizzled row (+2).
              if (role == 0) {
                tc::mma_f16_pair(d0, ad, bd, idesc0, acc);
                tc::mma_f16_pair(d0, ad + 128, bd + 2, idesc0, 1u);
                tc::mma_f16_pair(d0, ad + 256, bd + 4, idesc0, 1u);
                tc::mma_f16_pair(d0, ad + 384, bd + 6, idesc0, 1u);
              } else if (two) {
                const uint64_t bd1 = bd + (kSubBytes >> 4);   // second sub-tile's token rows
                tc::mma_f16_pair(d1, ad, bd1, idesc1, acc);
                tc::mma_f16_pair(d1, ad + 128, bd1 + 2, idesc1, 1u);
                tc::mma_f16_pair(d1, ad + 256, bd1 + 4, idesc1, 1u);
                tc::mma_f16_pair(d1, ad + 384, bd1 + 6, idesc1, 1u);
              }
            }
          }
          tc::mma_commit_pair(&empty[g], 0x3);  // frees the group's stages in both CTAs
          if (++g == ngroups) { g = 0; ph ^= 1; }
        }
        if (!ok) break;
        if (role == 0) tc::mma_commit_pair(&acc_full[k % kAccRing], 0x3);
        if (two && role == 1) tc::mma_commit_pair(&acc_full[(k + 1) % kAccRing], 0x3);
        k += two ? 2 : 1;
      }
      // Drain: make sure none of this issuer's MMAs is still reading shared or
      // writing tensor memory.
      tc::mma_commit_pair(&drain[role], 0x1);
      volatile int dummy = 0;
      tc::mbar_wait_bounded(&drain[role], 0, &dummy, kTimeoutNs);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue --
    const int lane_grp = warp % 4;           // TMEM lanes 32*lane_grp .. +31
    const int etid = threadIdx.x - 32 * epi_warp0(DUAL);   // 0..127
    volatile int *epi_ok = reinterpret_cast<volatile int *>(smem + Smem::epi_ok);
    float *xbuf = reinterpret_cast<float *>(smem + Smem::x);
    __nv_bfloat16 *obuf = reinterpret_cast<__nv_bfloat16 *>(smem + Smem::out);
    int pos = 0;          // tensor-memory ring position, as in the MMA issuer
    uint32_t k = 0;       // token sub-tiles so far
    uint32_t obi = 0;     // output buffer parity (GEMM2 alternates two buffers)
    bool go_on = true;
    for (int t = cid; t < total_tiles && go_on; t += ncl) {
      const TileInfo ti = decode_tile(p, prefix, t);
      const int nsub = ti.rows1 > 0 ? 2 : 1;
      float wsc = 1.f;   // FP8: this thread's output channel scale
      if (FP8) {
        // GEMM1: lanes 0-63 gate, 64-127 up of 64 hidden units; GEMM2: 128 columns of y
        const int ch = p.gemm1 ? ti.pair * 128 + (int)rank * 64 + (lane_grp & 1) * 32 + lane
                               : ti.pair * 256 + (int)rank * kBM + lane_grp * 32 + lane;
        const float *ws = (!p.gemm1 || lane_grp < 2) ? p.wscale_g : p.wscale_u;
        wsc = ch < p.M ? ws[(size_t)ti.e * p.M + ch] : 0.f;
      }
      for (int sub = 0; sub < nsub; ++sub) {
        const int srow0 = ti.row0 + (sub ? ti.rows0 : 0);   // first permuted row of the sub-tile
        const int srows = sub ? ti.rows1 : ti.rows0;
        const int n_mma = mma_n(srows);
        const int c0 = ring_take(pos, n_mma);
        const int nalloc = (n_mma + 31) / 32;
        const uint32_t par = (k / kAccRing) & 1;
        uint64_t *accb = &acc_full[k % kAccRing];
        ++k;
        // One thread waits (bounded) and the outcome is shared, so the four
        // epilogue warps always leave the loop together.
        if (etid == 0)
          *epi_ok = tc::mbar_wait_bounded(accb, par, abort_flag, kTimeoutNs) ? 1 : 0;
        tc::named_bar(1, kEpiThreads);
        const int go = *epi_ok;
        tc::named_bar(1, kEpiThreads);
        if (!go) {
          go_on = false;
          break;
        }
        tc::tc_fence_after();
        const uint32_t t_base = tmem_base + ((uint32_t)(lane_grp * 32) << 16) +
                                (uint32_t)(c0 * 32);
        const int nchunks = (srows + 31) / 32;
        // chunks the MMA wrote but that hold no rows (N rounded up) go back at once
        for (int cc = nchunks; cc < nalloc; ++cc) {
          tc::tc_fence_before();
          if (lane == 0) tc::mbar_arrive_cluster_relaxed(tc::mapa_shared(&col_free[c0 + cc], 0));
        }
        // Chunks are loaded two at a time and handed back to the MMA issuer
        // before any math, so the next sub-tile can take them early.
        for (int c2 = 0; c2 < nchunks; c2 += 2) {
          const bool pair = c2 + 1 < nchunks;
          uint32_t ra[32], rb[32];
          tc::tmem_ld_32x32b_x32(t_base + c2 * 32, ra);
          if (pair) tc::tmem_ld_32x32b_x32(t_base + (c2 + 1) * 32, rb);
          tc::tmem_ld_wait();
          // the chunks are in registers: hand them back (relaxed: the loads
          // have completed; nothing else needs ordering)
          tc::tc_fence_before();
          if (lane == 0) {
            tc::mbar_arrive_cluster_relaxed(tc::mapa_shared(&col_free[c0 + c2], 0));
            if (pair) tc::mbar_arrive_cluster_relaxed(tc::mapa_shared(&col_free[c0 + c2 + 1], 0));
          }
          if (FP8) {
            scale_chunk(p, srow0 + c2 * 32, srows - c2 * 32, lane, wsc, ra);
            if (pair) scale_chunk(p, srow0 + (c2 + 1) * 32, srows - (c2 + 1) * 32, lane, wsc, rb);
          }
          epilogue_chunk(p, ti, rank, lane_grp, lane, etid, xbuf, obuf, obi, srow0, srows, c2, ra);
          if (pair)
            epilogue_chunk(p, ti, rank, lane_grp, lane, etid, xbuf, obuf, obi, srow0, srows,
                           c2 + 1, rb);
        }
      }
    }
  }

  __syncthreads();
  tc::cluster_sync();   // no CTA leaves while its pair may still touch its memory
  if (*abort_flag && threadIdx.x == 0) report(p.status, MOE_DEV_TIMEOUT);
  if (warp == 1) {
    tc::tc_fence_after();
    tc::tmem_dealloc_pair(tmem_base, kTmemCols);
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

// FP8 weights Wq[N][M][K] (K contiguous, E4M3 bytes), box 128(K) x 64(M) x 1.
bool make_weight_map_k8(CUtensorMap *m, const void *Wq, int N, int M, int K) {
  cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)M, (cuuint64_t)N};
  cuuint64_t strides[2] = {(cuuint64_t)K, (cuuint64_t)M * K};
  cuuint32_t box[3] = {128, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(Wq), dims,
                     strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// FP8 token rows Xq[rows][K] (E4M3 bytes), box 128(K) x box_rows.
bool make_rows_map_u8(CUtensorMap *m, const void *Xq, int rows, int K, int box_rows) {
  cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)K};
  cuuint32_t box[2] = {128, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  return encode_fn()(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(Xq), dims,
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

// Token tiles per raster group: a group's token rows (256 rows x K bf16 per
// tile) stay within ~32 MB, a quarter of the 126 MB L2.
int raster_group(int K) {
  const long tile_bytes = 256L * K * 2;
  long g = (32L << 20) / tile_bytes;
  return (int)(g < 1 ? 1 : g > 64 ? 64 : g);
}

// Co-resident CTA pairs on this device (one pair per two SMs at most),
// asked once per device.
int max_pairs() {
  static int cached[kMaxDevicesCached] = {};
  const int dev = current_device();
  if (dev < kMaxDevicesCached && cached[dev]) return cached[dev];
  int sms = 148;
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(2 * (sms / 2));
  cfg.blockDim = dim3(kMaxThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int c = 0;
  if (cudaOccupancyMaxActiveClusters(&c, grouped_gemm_tc<false, 1, true>, &cfg) != cudaSuccess ||
      c <= 0) {
    cudaGetLastError();
    c = sms / 2;
  }
  const int n = c < sms / 2 ? c : sms / 2;
  if (dev < kMaxDevicesCached) cached[dev] = n;
  return n;
}

template <bool FP8>
moe_status_t launch_gemm(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap *b,
                         const TcParams &p, cudaStream_t stream) {
  static bool attr_set[kMaxDevicesCached] = {};
  const int dev = current_device();
  if (dev >= kMaxDevicesCached || !attr_set[dev]) {
    for (auto fn : {grouped_gemm_tc<FP8, 1, false>, grouped_gemm_tc<FP8, 2, false>,
                    grouped_gemm_tc<FP8, 1, true>}) {
      MOE_CUDA_TRY(
          cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes));
      MOE_CUDA_TRY(cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 0));
    }
    if (dev < kMaxDevicesCached) attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;   // see pdl_begin
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.gridDim = dim3(2 * max_pairs());
  cfg.blockDim = dim3(threads_for(p.wide != 0));
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  // wide layers: one barrier pair per stage, two MMA issuers
  auto fn = p.wide ? grouped_gemm_tc<FP8, 1, true>
          : p.kgroup == 2 ? grouped_gemm_tc<FP8, 2, false> : grouped_gemm_tc<FP8, 1, false>;
  MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, fn, a0, a1, b[0], b[1], b[2], b[3], p));
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace

namespace {

struct TileCfg {
  int tile_cap, wide, stages, stage_bytes, kgroup;
};

// Token tile width: the expected largest expert (1.25x the average rows, or
// the capacity when that is smaller) rounded up to 64/128/256, so narrow
// layers fit more, smaller stages.  Layers whose experts run ~250-320 rows
// (many experts just over 256) take wide tiles instead, which keep such an
// expert in one tile.
TileCfg tile_config(int A_max, int N, int capacity) {
  const long avg_rows = ((long)A_max + N - 1) / N;
  long exp_rows = avg_rows + avg_rows / 4;
  if (capacity > 0 && capacity < exp_rows) exp_rows = capacity;
  TileCfg c;
  c.wide = (exp_rows > 256 && avg_rows <= 320) ? 1 : 0;
  c.tile_cap = c.wide ? kWideTile : exp_rows > 128 ? 256 : exp_rows > 64 ? 128 : 64;
  c.stage_bytes = c.wide ? kABytes + 2 * kSubBytes : kABytes + (c.tile_cap / 2) * kBK * 2;
  c.stages = kStageRegion / c.stage_bytes;
  if (c.stages > kMaxStages) c.stages = kMaxStages;
  // Every barrier wait and commit in the MMA issuer's loop costs about as much
  // as issuing an MMA.  Where an expert spans many token tiles (the weights
  // come from L2 and the tensor pipe is the limit) two stages share one
  // barrier pair: one wait and one commit per 128 K (measured: prefill 2%
  // faster).  Where the weights stream from DRAM the finer release of one
  // pair per stage measured faster (DeepSeek-shaped, capacity layers).
  const long tiles = (exp_rows + c.tile_cap - 1) / c.tile_cap;
  c.kgroup = (tiles > 2 && c.stages % 2 == 0) ? 2 : 1;
  return c;
}

moe_status_t check_ffn_launch(int N) {
  if (!encode_fn()) {
    set_error("cuTensorMapEncodeTiled unavailable from the driver");
    return MOE_ERR_CUDA;
  }
  if (N > kMaxExperts) {
    set_error("tensor-core FFN supports N <= %d experts", kMaxExperts);
    return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

// GEMM2 (down projection + gate scale) of either form: h [A_max, f] bf16.
moe_status_t launch_down(const int32_t *offsets, const float *row_scale, int A_max, int d,
                         int f, int N, const TileCfg &tc_, const void *W_down, void *h,
                         void *y_perm, int32_t *device_status, cudaStream_t stream,
                         const int32_t *out_row = nullptr, int rows_out = 0) {
  CUtensorMap wd, bh[kNumBoxes];
  bool ok = make_weight_map(&wd, W_down, N, f, d);
  const int box_rows[kNumBoxes] = {32, 64, 80, 128};
  for (int i = 0; i < kNumBoxes; ++i) ok = ok && make_rows_map(&bh[i], h, A_max, f, box_rows[i]);
  if (!ok) {
    set_error("tensor map encoding failed (alignment or size)");
    return MOE_ERR_INVALID_ARG;
  }
  TcParams p2{offsets, N, f, d, (d + 255) / 256, 0, static_cast<__nv_bfloat16 *>(y_perm), d,
              row_scale, device_status, raster_group(f), tc_.tile_cap, tc_.wide, tc_.stages,
              tc_.kgroup, tc_.stage_bytes};
  p2.out_row = out_row;
  p2.rows_out = rows_out;
  return launch_gemm<false>(wd, wd, bh, p2, stream);
}

}  // namespace

// x_perm [A_max, d] -> h [A_max, f] -> y_perm [A_max, d], bf16, per expert.
moe_status_t launch_ffn_tc(const void *x_perm, const int32_t *offsets, const float *row_scale,
                           int A_max, int d, int f, int N, int capacity, const void *W_gate,
                           const void *W_up, const void *W_down, void *h, void *y_perm,
                           int32_t *device_status, cudaStream_t stream,
                           const int32_t *out_row, int rows_out) {
  if (A_max == 0) return MOE_OK;
  moe_status_t s = check_ffn_launch(N);
  if (s != MOE_OK) return s;
  CUtensorMap wg, wu, bx[kNumBoxes];
  bool ok = make_weight_map(&wg, W_gate, N, d, f) && make_weight_map(&wu, W_up, N, d, f);
  const int box_rows[kNumBoxes] = {32, 64, 80, 128};
  for (int i = 0; i < kNumBoxes; ++i)
    ok = ok && make_rows_map(&bx[i], x_perm, A_max, d, box_rows[i]);
  if (!ok) {
    set_error("tensor map encoding failed (alignment or size)");
    return MOE_ERR_INVALID_ARG;
  }
  const TileCfg c = tile_config(A_max, N, capacity);
  TcParams p1{offsets, N, d, f, (f + 127) / 128, 1, static_cast<__nv_bfloat16 *>(h), f, nullptr,
              device_status, raster_group(d), c.tile_cap, c.wide, c.stages, c.kgroup, c.stage_bytes};
  s = launch_gemm<false>(wg, wu, bx, p1, stream);
  if (s != MOE_OK) return s;
  return launch_down(offsets, row_scale, A_max, d, f, N, c, W_down, h, y_perm, device_status,
                     stream, out_row, rows_out);
}

// h in bf16 (bf16 down projection), or in fp32 followed by its E4M3 codes
// and row scales (E4M3 down projection: the row quantiser sees h unrounded).
size_t ffn_fp8_workspace_bytes(int A_max, int f, bool fp8_down) {
  size_t b = align_up((size_t)A_max * f * (fp8_down ? 4 : 2), 256);
  if (fp8_down)
    b += align_up((size_t)A_max * f, 256) + align_up((size_t)A_max * 4, 256);  // hq, its scales
  return b;
}

// The same with E4M3 gate/up: xq_perm [A_max, d] E4M3 token rows (scale of
// permuted row p: x_scale[perm_token[p]]), Wq_gate / Wq_up [N, f, d] E4M3
// with channel scales [N, f].  The down projection is bf16 from W_down on h
// written in bf16, or, with Wq_down [N, d, f] and its channel scales [N, d],
// E4M3 on h written in fp32 and quantised per row from those values (rows
// past offsets[N] left alone).
moe_status_t launch_ffn_tc_fp8(const void *xq_perm, const float *x_scale,
                               const int32_t *perm_token, const int32_t *offsets,
                               const float *row_scale, int A_max, int d, int f, int N,
                               int capacity, const void *Wq_gate, const float *sw_gate,
                               const void *Wq_up, const float *sw_up, const void *W_down,
                               const void *Wq_down, const float *sw_down, void *workspace,
                               void *y_perm, int32_t *device_status, cudaStream_t stream) {
  if (A_max == 0) return MOE_OK;
  moe_status_t s = check_ffn_launch(N);
  if (s != MOE_OK) return s;
  char *ws = static_cast<char *>(workspace);
  void *h = ws;
  const bool h_f32 = Wq_down != nullptr;
  uint8_t *hq = reinterpret_cast<uint8_t *>(ws + align_up((size_t)A_max * f * (h_f32 ? 4 : 2),
                                                          256));
  float *hs = reinterpret_cast<float *>(reinterpret_cast<char *>(hq) +
                                        align_up((size_t)A_max * f, 256));
  CUtensorMap wg, wu, bx[kNumBoxes];
  bool ok = make_weight_map_k8(&wg, Wq_gate, N, f, d) && make_weight_map_k8(&wu, Wq_up, N, f, d);
  const int box_rows[kNumBoxes] = {32, 64, 80, 128};
  for (int i = 0; i < kNumBoxes; ++i)
    ok = ok && make_rows_map_u8(&bx[i], xq_perm, A_max, d, box_rows[i]);
  CUtensorMap wd, bh[kNumBoxes];
  if (Wq_down) {
    ok = ok && make_weight_map_k8(&wd, Wq_down, N, d, f);
    for (int i = 0; i < kNumBoxes; ++i) ok = ok && make_rows_map_u8(&bh[i], hq, A_max, f, box_rows[i]);
  }
  if (!ok) {
    set_error("tensor map encoding failed (alignment or size)");
    return MOE_ERR_INVALID_ARG;
  }
  const TileCfg c = tile_config(A_max, N, capacity);
  TcParams p1{offsets, N, d, f, (f + 127) / 128, 1, static_cast<__nv_bfloat16 *>(h), f, nullptr,
              device_status, raster_group(d), c.tile_cap, c.wide, c.stages, c.kgroup, c.stage_bytes,
              sw_gate, sw_up, x_scale, perm_token, h_f32 ? 1 : 0};
  s = launch_gemm<true>(wg, wu, bx, p1, stream);
  if (s != MOE_OK) return s;
  if (!Wq_down)
    return launch_down(offsets, row_scale, A_max, d, f, N, c, W_down, h, y_perm, device_status,
                       stream);
  s = launch_quantize_rows_e4m3(h, A_max, f, hq, hs, stream, offsets + N, /*f32_in=*/true);
  if (s != MOE_OK) return s;
  TcParams p2{offsets, N, f, d, (d + 255) / 256, 0, static_cast<__nv_bfloat16 *>(y_perm), d,
              row_scale, device_status, raster_group(f), c.tile_cap, c.wide, c.stages,
              c.kgroup, c.stage_bytes, sw_down, nullptr, hs, nullptr};
  return launch_gemm<true>(wd, wd, bh, p2, stream);
}

}  // namespace moe
