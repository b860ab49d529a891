// moe_permute_noalloc: moe_permute without a caller-provided workspace.
//
// Who needs it: callers that cannot allocate device memory at the point where
// they dispatch tokens -- for example an operator plugged into a host
// framework that hands it only its input and output buffers and forbids
// allocations while a model runs, or a fixed-budget serving process that
// reserves all of its memory up front.  moe_permute itself allocates nothing,
// but it needs a small scratch buffer from the caller; this variant takes that
// scratch from a fixed array in the library instead.
//
// The scratch is the per-chunk expert histogram of the dispatch kernels:
// ceil(T / 256) * N int32 entries, at most kNoAllocHistEntries (65536 entries,
// 256 KB; e.g. T = 65536 tokens with N = 256 experts).  Every GPU that loads
// the library holds this array until the process exits.  The kernels write
// every entry they later read, so nothing needs clearing between calls.  All
// calls share the one array: calls that overlap on the GPU (different streams
// or threads without ordering between them) race on it.
#include <mutex>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kNoAllocHistEntries = 65536;
constexpr int kMaxDevices = 64;

// Device-side scratch.  In host code this name is only a stand-in for the
// symbol: its device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) int32_t g_noalloc_hist[kNoAllocHistEntries];

std::mutex g_mu;
void *g_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device, looked up once
// per device (with that device current) and cached.
moe_status_t scratch_address(void **out) {
  int dev = 0;
  MOE_CUDA_TRY(cudaGetDevice(&dev));
  if (dev < 0 || dev >= kMaxDevices) {
    set_error("moe_permute_noalloc: device %d beyond the %d supported", dev, kMaxDevices);
    return MOE_ERR_UNSUPPORTED;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_addr[dev]) {
    void *p = nullptr;
    cudaError_t err = cudaGetSymbolAddress(&p, g_noalloc_hist);
    if (err != cudaSuccess || !p) {
      set_error("moe_permute_noalloc: cudaGetSymbolAddress failed: %s",
                cudaGetErrorString(err));
      return MOE_ERR_CUDA;
    }
    g_addr[dev] = p;
  }
  *out = g_addr[dev];
  return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_permute_noalloc(const int32_t *topk_idx, const float *topk_w,
                                            const void *x, moe_dtype_t dtype, int T, int d,
                                            int N, int k, int capacity, int32_t *counts,
                                            int32_t *offsets, int32_t *perm_token,
                                            float *row_scale, int32_t *inv_pos, void *x_perm,
                                            int32_t *dropped, int32_t *device_status,
                                            void *stream) {
  if (T < 0 || N < 1 || k < 1) {
    set_error("moe_permute_noalloc: bad sizes T=%d N=%d k=%d", T, N, k);
    return MOE_ERR_INVALID_ARG;
  }
  const long need = (((long)T + 255) / 256) * (long)N;   // no int overflow near INT_MAX
  if (need > kNoAllocHistEntries) {
    set_error("moe_permute_noalloc: ceil(T/256)*N = %ld histogram entries exceeds the fixed "
              "scratch of %d (use moe_permute with a workspace)",
              need, kNoAllocHistEntries);
    return MOE_ERR_UNSUPPORTED;
  }
  void *scratch = nullptr;
  moe_status_t s = scratch_address(&scratch);
  if (s != MOE_OK) return s;
  return moe_permute(topk_idx, topk_w, x, dtype, T, d, N, k, capacity, counts, offsets,
                     perm_token, row_scale, inv_pos, x_perm, dropped, device_status, scratch,
                     (size_t)kNoAllocHistEntries * sizeof(int32_t), stream);
}
