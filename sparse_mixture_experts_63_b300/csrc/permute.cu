// Dispatch: regroup the T*k (token, slot) assignments by expert, stable by
// token index, with an optional per-expert capacity, and gather the rows.
//
// Source: "MoE稀疏激活原理与工程实践", 3.1 (token-level batching: the batch's
// tokens are regrouped by target expert id, {0:[t0,t1,t3], 1:[t2,t5], ...},
// before each expert runs) and 2.2 (a per-expert queue with a hard capacity);
// "MoE 分片：混合專家模型的平行化策略", section 動態 token 路由, step 3.
//
// Deterministic without inter-CTA waits, in four launches:
//   1. hist:    CTA b counts its chunk's assignments per expert -> hist[b][e]
//   2. scan:    one CTA: per expert, prefix over chunks (chunk_base[b][e]),
//               counts[e], kept[e] = min(counts[e], C), offsets = exclusive
//               scan of kept, dropped.
//   3. scatter: CTA b re-reads its chunk; the rank of an assignment inside the
//               chunk (stable by token) comes from warp match + per-warp counts;
//               rank = chunk_base + in-chunk rank; kept iff rank < C.
//   4. copy:    x_perm[inv_pos[t][j]] = x[t] for every kept slot, in token
//               order: each row of x is read once and written k times
//               (16-byte vectors; reading in expert order re-read x from DRAM
//               ~5x once the 0.9 GB write stream had pushed it out of L2).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kChunkTokens = 256;  // tokens per chunk (CTA) in hist / scatter
constexpr int kThreads = 256;
constexpr int kMaxN = 1024;

// neg_one_drops: an id of -1 marks a slot already known to be dropped (no
// report); any other id outside [0, N) is reported as a bad expert id.
__global__ void __launch_bounds__(kThreads) permute_hist(const int32_t *__restrict__ topk_idx,
                                                         int T, int N, int k,
                                                         int32_t *__restrict__ hist,
                                                         int32_t *status, int neg_one_drops) {
  pdl_begin();
  extern __shared__ int32_t sh_hist[];  // [N]
  for (int e = threadIdx.x; e < N; e += blockDim.x) sh_hist[e] = 0;
  __syncthreads();
  const long a0 = (long)blockIdx.x * kChunkTokens * k;
  const long a1 = min((long)T * k, a0 + (long)kChunkTokens * k);
  bool bad = false;
  for (long a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
    int e = topk_idx[a];
    if (e >= 0 && e < N)
      atomicAdd(&sh_hist[e], 1);
    else if (!(neg_one_drops && e == -1))
      bad = true;
  }
  if (bad) report(status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) hist[(size_t)blockIdx.x * N + e] = sh_hist[e];
}

// One CTA of kMaxN threads; thread e owns expert e.
__global__ void __launch_bounds__(kMaxN) permute_scan(int32_t *__restrict__ hist, int nchunks,
                                                      int T, int N, int k, int capacity,
                                                      int32_t *__restrict__ counts,
                                                      int32_t *__restrict__ offsets,
                                                      int32_t *__restrict__ dropped) {
  pdl_begin();
  __shared__ int32_t warp_sums[kMaxN / 32];
  const int e = threadIdx.x;
  int32_t total = 0;
  if (e < N) {
    for (int b = 0; b < nchunks; ++b) {
      int32_t c = hist[(size_t)b * N + e];
      hist[(size_t)b * N + e] = total;  // becomes chunk_base[b][e]
      total += c;
    }
    counts[e] = total;
  }
  int32_t kept = (e < N) ? ((capacity > 0 && total > capacity) ? capacity : total) : 0;
  // Block-wide exclusive scan of kept.
  const int lane = e % 32, w = e / 32;
  int32_t incl = kept;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    int32_t o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  if (w == 0) {
    int32_t s = warp_sums[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int32_t o = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += o;
    }
    warp_sums[lane] = s;  // inclusive over warps
  }
  __syncthreads();
  int32_t excl = incl - kept + (w > 0 ? warp_sums[w - 1] : 0);
  if (e < N) offsets[e] = excl;
  if (e == N - 1) {
    offsets[N] = excl + kept;
    if (dropped) *dropped = (int32_t)((long)T * k - (excl + kept));
  }
}

// CTA b: assignments of tokens [b*256, (b+1)*256).  Processed in rounds of
// kThreads consecutive assignments (token-major, so order = token order).
__global__ void __launch_bounds__(kThreads) permute_scatter(
    const int32_t *__restrict__ topk_idx, const float *__restrict__ topk_w, int T, int N, int k,
    int capacity, const int32_t *__restrict__ chunk_base, const int32_t *__restrict__ offsets,
    int32_t *__restrict__ perm_token, float *__restrict__ row_scale, int32_t *__restrict__ inv_pos) {
  pdl_begin();
  extern __shared__ int32_t sm[];
  int32_t *running = sm;                  // [N] rows of each expert seen in earlier rounds
  int32_t *warp_cnt = sm + N;             // [8][N] per-warp counts of this round
  constexpr int kWarps = kThreads / 32;
  for (int e = threadIdx.x; e < N; e += blockDim.x) running[e] = 0;
  const long a0 = (long)blockIdx.x * kChunkTokens * k;
  const long a1 = min((long)T * k, a0 + (long)kChunkTokens * k);
  const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (long base = a0; base < a1; base += kThreads) {
    for (int q = threadIdx.x; q < kWarps * N; q += blockDim.x) warp_cnt[q] = 0;
    __syncthreads();
    const long a = base + threadIdx.x;
    int e = (a < a1) ? topk_idx[a] : -1;
    const bool valid = (e >= 0 && e < N);
    const int key = valid ? e : -1 - (int)(threadIdx.x);  // invalid lanes match nobody
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank_in_warp = __popc(peers & lt_mask);
    const bool last_of_group = (peers >> lane) == 1u;  // highest lane of its group
    if (valid && last_of_group) warp_cnt[w * N + e] = rank_in_warp + 1;
    __syncthreads();
    if (valid) {
      int32_t r = running[e] + rank_in_warp;
      for (int w2 = 0; w2 < w; ++w2) r += warp_cnt[w2 * N + e];
      r += chunk_base[(size_t)blockIdx.x * N + e];
      if (capacity > 0 && r >= capacity) {
        inv_pos[a] = -1;
      } else {
        int32_t p = offsets[e] + r;
        inv_pos[a] = p;
        perm_token[p] = (int32_t)(a / k);
        if (row_scale) row_scale[p] = topk_w[a];
      }
    } else if (a < a1) {
      inv_pos[a] = -1;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < N; q += blockDim.x) {
      int32_t s = 0;
      for (int w2 = 0; w2 < kWarps; ++w2) s += warp_cnt[w2 * N + q];
      running[q] += s;
    }
    __syncthreads();
  }
}

// All of hist, scan and scatter in one CTA when every token fits one chunk
// (T <= 256) and N <= 256: the same order and ranks as the three kernels
// (assignments in index order = token order), without their launch gaps --
// decode-sized batches spent most of the dispatch time between launches.
constexpr int kSmallThreads = 1024;
constexpr int kSmallMaxN = 256;

__global__ void __launch_bounds__(kSmallThreads) permute_small(
    const int32_t *__restrict__ topk_idx, const float *__restrict__ topk_w, int T, int N, int k,
    int capacity, int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
    int32_t *__restrict__ perm_token, float *__restrict__ row_scale,
    int32_t *__restrict__ inv_pos, int32_t *__restrict__ dropped, int32_t *status,
    int neg_one_drops) {
  pdl_begin();
  constexpr int kWarps = kSmallThreads / 32;
  __shared__ int32_t hist[kSmallMaxN];
  __shared__ int32_t off_s[kSmallMaxN + 1];
  __shared__ int32_t running[kSmallMaxN];
  __shared__ int32_t warp_cnt[kWarps * kSmallMaxN];
  const int A = T * k;
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    hist[e] = 0;
    running[e] = 0;
  }
  __syncthreads();
  bool bad = false;
  for (int a = threadIdx.x; a < A; a += blockDim.x) {
    const int e = topk_idx[a];
    if (e >= 0 && e < N)
      atomicAdd(&hist[e], 1);
    else if (!(neg_one_drops && e == -1))
      bad = true;
  }
  if (bad) report(status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  if (threadIdx.x == 0) {
    int32_t acc = 0;
    for (int e = 0; e < N; ++e) {
      const int32_t c = hist[e];
      counts[e] = c;
      off_s[e] = acc;
      offsets[e] = acc;
      acc += (capacity > 0 && c > capacity) ? capacity : c;
    }
    off_s[N] = acc;
    offsets[N] = acc;
    if (dropped) *dropped = A - acc;
  }
  __syncthreads();
  const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int base = 0; base < A; base += kSmallThreads) {
    for (int q = threadIdx.x; q < kWarps * N; q += blockDim.x) warp_cnt[q] = 0;
    __syncthreads();
    const int a = base + threadIdx.x;
    const int e = (a < A) ? topk_idx[a] : -1;
    const bool valid = (e >= 0 && e < N);
    const int key = valid ? e : -1 - (int)threadIdx.x;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank_in_warp = __popc(peers & lt_mask);
    const bool last_of_group = (peers >> lane) == 1u;
    if (valid && last_of_group) warp_cnt[w * N + e] = rank_in_warp + 1;
    __syncthreads();
    if (valid) {
      int32_t r = running[e] + rank_in_warp;
      for (int w2 = 0; w2 < w; ++w2) r += warp_cnt[w2 * N + e];
      if (capacity > 0 && r >= capacity) {
        inv_pos[a] = -1;
      } else {
        const int32_t p = off_s[e] + r;
        inv_pos[a] = p;
        perm_token[p] = a / k;
        if (row_scale) row_scale[p] = topk_w[a];
      }
    } else if (a < A) {
      inv_pos[a] = -1;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < N; q += blockDim.x) {
      int32_t s2 = 0;
      for (int w2 = 0; w2 < kWarps; ++w2) s2 += warp_cnt[w2 * N + q];
      running[q] += s2;
    }
    __syncthreads();
  }
}

// One warp per token (grid-stride): the row is read once, four 16-byte
// vectors per lane in flight, and written to the position of each kept slot
// (inv_pos < 0: dropped).  Slots are taken 32 at a time (one per lane).
template <typename VecT>
__global__ void __launch_bounds__(256) permute_copy_rows(const VecT *__restrict__ x,
                                                         const int32_t *__restrict__ inv_pos,
                                                         int T, int k, int vecs_per_row,
                                                         VecT *__restrict__ x_perm) {
  pdl_begin();
  constexpr int kUnroll = 4;
  const int lane = threadIdx.x % 32;
  const int warps = blockDim.x / 32;
  for (int t = blockIdx.x * warps + threadIdx.x / 32; t < T; t += gridDim.x * warps) {
    const VecT *src = x + (size_t)t * vecs_per_row;
    for (int j0 = 0; j0 < k; j0 += 32) {
      const int nj = min(32, k - j0);
      const int my = lane < nj ? inv_pos[(size_t)t * k + j0 + lane] : -1;
      for (int v0 = 0; v0 < vecs_per_row; v0 += 32 * kUnroll) {
        VecT val[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < vecs_per_row) val[u] = __ldg(src + v);
        }
        for (int j = 0; j < nj; ++j) {
          const int pos = __shfl_sync(0xffffffffu, my, j);
          if (pos < 0) continue;
          VecT *dst = x_perm + (size_t)pos * vecs_per_row;
#pragma unroll
          for (int u = 0; u < kUnroll; ++u) {
            const int v = v0 + u * 32 + lane;
            if (v < vecs_per_row) dst[v] = val[u];
          }
        }
      }
    }
  }
}

}  // namespace

size_t permute_workspace_bytes(int T, int N, int k) {
  (void)k;
  size_t nchunks = ((size_t)T + kChunkTokens - 1) / kChunkTokens;
  return align_up(nchunks * (size_t)N * sizeof(int32_t), 256);
}

moe_status_t launch_permute(const int32_t *topk_idx, const float *topk_w, const void *x,
                            moe_dtype_t dtype, int T, int d, int N, int k, int capacity,
                            int32_t *counts, int32_t *offsets, int32_t *perm_token,
                            float *row_scale, int32_t *inv_pos, void *x_perm, int32_t *dropped,
                            int32_t *device_status, void *workspace, cudaStream_t stream,
                            bool neg_one_drops) {
  if (N > kMaxN) {
    set_error("moe_permute: N=%d above %d", N, kMaxN);
    return MOE_ERR_UNSUPPORTED;
  }
  int32_t *hist = static_cast<int32_t *>(workspace);
  const int nchunks = (T + kChunkTokens - 1) / kChunkTokens;
  if (nchunks == 1 && N <= kSmallMaxN) {
    MOE_CUDA_TRY(launch_pdl(permute_small, dim3(1), dim3(kSmallThreads), 0, stream, topk_idx,
        topk_w, T, N, k, capacity, counts, offsets, perm_token, row_scale, inv_pos, dropped,
        device_status, neg_one_drops ? 1 : 0));
    MOE_LAUNCH_CHECK();
  } else {
  if (nchunks > 0) {
    MOE_CUDA_TRY(launch_pdl(permute_hist, dim3(nchunks), dim3(kThreads), N * sizeof(int32_t),
        stream, topk_idx, T, N, k, hist, device_status, neg_one_drops ? 1 : 0));
    MOE_LAUNCH_CHECK();
  }
  MOE_CUDA_TRY(launch_pdl(permute_scan, dim3(1), dim3(kMaxN), 0, stream, hist, nchunks, T, N, k,
      capacity, counts, offsets, dropped));
  MOE_LAUNCH_CHECK();
  if (nchunks > 0) {
    size_t smem = (size_t)N * (1 + kThreads / 32) * sizeof(int32_t);
    MOE_CUDA_TRY(launch_pdl(permute_scatter, dim3(nchunks), dim3(kThreads), smem, stream, topk_idx,
        topk_w, T, N, k, capacity, hist, offsets, perm_token, row_scale, inv_pos));
    MOE_LAUNCH_CHECK();
  }
  }
  return launch_copy_rows(x, dtype, inv_pos, T, d, k, x_perm, stream);
}

moe_status_t launch_copy_rows(const void *x, moe_dtype_t dtype, const int32_t *inv_pos, int T,
                              int d, int k, void *x_perm, cudaStream_t stream) {
  return launch_copy_row_bytes(x, (size_t)d * (dtype == MOE_BF16 ? 2 : 4), inv_pos, T, k, x_perm,
                               stream);
}

moe_status_t launch_copy_row_bytes(const void *x, size_t row_bytes, const int32_t *inv_pos,
                                   int T, int k, void *x_perm, cudaStream_t stream) {
  if (x_perm && T > 0) {
    const int vecs = (int)(row_bytes / 16);
    long grid = ((long)T + 7) / 8;
    if (grid > 148L * 16) grid = 148L * 16;
    MOE_CUDA_TRY(launch_pdl(permute_copy_rows<uint4>, dim3((int)grid), dim3(256), 0, stream,
        static_cast<const uint4 *>(x), inv_pos, T, k, vecs, static_cast<uint4 *>(x_perm)));
    MOE_LAUNCH_CHECK();
  }
  return MOE_OK;
}

}  // namespace moe
