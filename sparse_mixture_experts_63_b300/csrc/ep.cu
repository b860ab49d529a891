// Expert-parallel dispatch and combine: the device steps on either side of the
// all-to-all exchanges.
//
// Source: "MoE 分片：混合專家模型的平行化策略", sections 專家平行化詳解 (the
// experts are split over the GPUs, each holding N/G of them) and 動態 token
// 路由 steps 3-5 (tokens are sent to the GPUs of their experts, computed there,
// and the results sent back to the tokens' own GPU); "MoE稀疏激活原理与工程实践",
// 2.2 (an all-to-all per routing step).
//
// Layout.  Rank r holds experts [r*Ne, (r+1)*Ne).  Its dispatch (moe_permute
// over all N experts) already orders its rows by expert, so the rows bound
// for rank q are one contiguous range of x_perm: no packing kernel is needed.
// After the exchange a rank holds, from each source s, the rows of each of
// its experts e in turn: block (s, e) of recv_counts[s][e] rows, blocks in
// (s, e) order.  The grouped GEMM wants each expert's rows together, so the
// regroup moves block (s, e) to expert e's range, after the blocks of the
// earlier sources (stable: a source's rows keep their order), and records
// where each received row went; the return gather undoes it on the outputs.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kEpThreads = 256;
constexpr int kEpMaxBlocks = 4096;   // G * Ne entries scanned in shared memory

// Block starts in the received (source-major) order and in the regrouped
// (expert-major) order, computed by every CTA from the G x Ne counts.
struct EpScan {
  int32_t recv_start[kEpMaxBlocks];   // first received row of block (s, e)
  int32_t local_start[kEpMaxBlocks];  // its first row in the regrouped order
  int32_t total;
};

__device__ void ep_scan(const int32_t *counts, int G, int Ne, EpScan &sc, int32_t *offsets_out) {
  const int nb = G * Ne;
  if (threadIdx.x == 0) {
    // source-major starts
    int32_t acc = 0;
    for (int b = 0; b < nb; ++b) {
      sc.recv_start[b] = acc;
      acc += max(counts[b], 0);
    }
    sc.total = acc;
    // expert-major: expert e's range starts after every earlier expert's rows;
    // inside it, source s's block follows the blocks of sources 0..s-1
    int32_t base = 0;
    for (int e = 0; e < Ne; ++e) {
      if (offsets_out) offsets_out[e] = base;
      for (int s = 0; s < G; ++s) {
        sc.local_start[s * Ne + e] = base;
        base += max(counts[s * Ne + e], 0);
      }
    }
    if (offsets_out) offsets_out[Ne] = base;
  }
  __syncthreads();
}

// The block (s, e) holding received row i: the last block whose start is <= i
// (empty blocks share their start with the next one; the search skips them).
__device__ __forceinline__ int ep_block_of(const EpScan &sc, const int32_t *counts, int nb,
                                           int32_t i) {
  int lo = 0, hi = nb - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (sc.recv_start[mid] <= i) lo = mid; else hi = mid - 1;
  }
  while (lo > 0 && counts[lo] <= 0) --lo;   // an empty block cannot hold row i
  return lo;
}

// One warp per row, 16-byte vectors.
__global__ void __launch_bounds__(kEpThreads) ep_regroup_kernel(
    const int32_t *__restrict__ counts, int G, int Ne, const uint4 *__restrict__ x_recv,
    const float *__restrict__ rs_recv, int R, int vecs, uint4 *__restrict__ x_local,
    float *__restrict__ rs_local, int32_t *__restrict__ offsets_local,
    int32_t *__restrict__ dest, int32_t *__restrict__ src_row, int32_t *device_status) {
  pdl_begin();
  __shared__ EpScan sc;
  ep_scan(counts, G, Ne, sc, blockIdx.x == 0 ? offsets_local : nullptr);
  if (sc.total != R) {                 // the counts do not describe the rows given
    if (blockIdx.x == 0 && threadIdx.x == 0) report(device_status, MOE_DEV_BAD_COUNTS);
    return;
  }
  const int nb = G * Ne;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (long i = (long)blockIdx.x * (kEpThreads / 32) + warp; i < R;
       i += (long)gridDim.x * (kEpThreads / 32)) {
    const int b = ep_block_of(sc, counts, nb, (int32_t)i);
    const int32_t to = sc.local_start[b] + ((int32_t)i - sc.recv_start[b]);
    const uint4 *src = x_recv + (size_t)i * vecs;
    uint4 *dst = x_local + (size_t)to * vecs;
    for (int v = lane; v < vecs; v += 32) dst[v] = src[v];
    if (lane == 0) {
      dest[i] = to;
      if (src_row) src_row[to] = (int32_t)i;
      if (rs_recv) rs_local[to] = rs_recv[i];
    }
  }
}

// y_back[i] = y_local[dest[i]]: the expert outputs back in received order.
__global__ void __launch_bounds__(kEpThreads) ep_return_kernel(const uint4 *__restrict__ y_local,
                                                               const int32_t *__restrict__ dest,
                                                               int R, int vecs,
                                                               uint4 *__restrict__ y_back) {
  pdl_begin();
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  for (long i = (long)blockIdx.x * (kEpThreads / 32) + warp; i < R;
       i += (long)gridDim.x * (kEpThreads / 32)) {
    const int32_t from = dest[i];
    if (from < 0 || from >= R) continue;   // not written by a regroup of these counts
    const uint4 *src = y_local + (size_t)from * vecs;
    uint4 *dst = y_back + (size_t)i * vecs;
    for (int v = lane; v < vecs; v += 32) dst[v] = src[v];
  }
}

int ep_grid(long rows) {
  long g = (rows + kEpThreads / 32 - 1) / (kEpThreads / 32);
  if (g > 148L * 8) g = 148L * 8;
  return (int)(g < 1 ? 1 : g);
}

}  // namespace

int ep_max_blocks() { return kEpMaxBlocks; }

moe_status_t launch_ep_regroup(const int32_t *recv_counts, int G, int Ne, const void *x_recv,
                               const float *row_scale_recv, int R, size_t row_bytes,
                               void *x_local, float *row_scale_local, int32_t *offsets_local,
                               int32_t *dest, int32_t *src_row, int32_t *device_status,
                               cudaStream_t stream) {
  MOE_CUDA_TRY(launch_pdl(ep_regroup_kernel, dim3(ep_grid(R)), dim3(kEpThreads), 0, stream,
                          recv_counts, G, Ne, static_cast<const uint4 *>(x_recv), row_scale_recv,
                          R, (int)(row_bytes / 16), static_cast<uint4 *>(x_local),
                          row_scale_local, offsets_local, dest, src_row, device_status));
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

moe_status_t launch_ep_return(const void *y_local, const int32_t *dest, int R, size_t row_bytes,
                              void *y_back, cudaStream_t stream) {
  if (R == 0) return MOE_OK;
  MOE_CUDA_TRY(launch_pdl(ep_return_kernel, dim3(ep_grid(R)), dim3(kEpThreads), 0, stream,
                          static_cast<const uint4 *>(y_local), dest, R, (int)(row_bytes / 16),
                          static_cast<uint4 *>(y_back)));
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
