// Dispatch with capacity overflow re-routed to the next-best expert.
//
// Source: "MoE稀疏激活原理与工程实践", 2.2 (专家容量的硬约束: once an expert's queue
// holds its capacity, a token that selects it is re-routed to its next-best
// expert; the re-routing rate is the operational signal of 4.1/5).
//
// Reading (the page gives the rule, not the order): the first pass is the
// capacity rule of moe_permute (an expert keeps its first C assignments by
// token index); then, in each of R rounds, every slot still without an expert
// proposes its token's next untried candidate (ranks k, k+1, ... of the
// token's experts, taken in slot order, used up whether granted or not), and
// each expert grants its remaining room to that round's proposals in (token,
// slot) order.  A slot still unplaced after R rounds is dropped.  Gate
// weights: the softmax over the logits of the token's final experts, i.e. the
// router's softmax over its k+R candidates renormalised over them (a dropped
// slot keeps its first choice in the denominator and contributes nothing).
//
// Every round, the first pass included, is three launches, deterministic:
//   propose: CTA b takes the slots of tokens [256b, 256b+256): each unplaced
//            slot's proposal from the round's starting state; per-chunk
//            proposal counts per expert;
//   scan:    per expert, chunk bases, the room left (C - used) and the grants;
//   grant:   a proposal's rank among the round's proposals to its expert
//            (chunk base + rank inside the chunk, token order, as in the
//            dispatch scatter) decides it: granted iff rank < room.
// Then the final selection goes through the dispatch (-1 = dropped).
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kChunkTokens = 256;
constexpr int kThreads = 256;
constexpr int kMaxN = 1024;

struct RerouteState {
  int32_t *hist;     // [nchunks][N] proposal counts, then chunk bases
  int32_t *used;     // [N] capacity taken so far
  int32_t *room;     // [N] room at the start of the round
  int32_t *ptr[2];   // [T] each token's next untried candidate (in / out)
  int32_t *fcand;    // [T*k] candidate granted to each slot, -1 = none yet
  int32_t *prop;     // [T*k] candidate proposed this round, -1 = none
};

__global__ void __launch_bounds__(kThreads) rr_propose(
    const int32_t *__restrict__ cand, int T, int N, int k, int kr,
    const int32_t *__restrict__ fcand, const int32_t *__restrict__ ptr_in,
    int32_t *__restrict__ ptr_out, int32_t *__restrict__ prop, int32_t *__restrict__ hist,
    int32_t *status) {
  extern __shared__ int32_t sh_hist[];  // [N]
  for (int e = threadIdx.x; e < N; e += blockDim.x) sh_hist[e] = 0;
  __syncthreads();
  const long a0 = (long)blockIdx.x * kChunkTokens * k;
  const long a1 = min((long)T * k, a0 + (long)kChunkTokens * k);
  bool bad = false;
  for (long a = a0 + threadIdx.x; a < a1; a += blockDim.x) {
    const long t = a / k;
    const int j = (int)(a - t * k);
    int before = 0;   // unplaced slots of this token before slot j
    for (int jj = 0; jj < j; ++jj) before += fcand[t * k + jj] < 0 ? 1 : 0;
    const bool open = fcand[a] < 0;
    int p = -1;
    if (open) {
      const int c = ptr_in[t] + before;
      if (c < kr) {
        const int e = cand[t * kr + c];
        if (e >= 0 && e < N) {
          p = c;
          atomicAdd(&sh_hist[e], 1);
        } else {
          bad = true;
        }
      }
    }
    prop[a] = p;
    if (j == k - 1) ptr_out[t] = min(kr, ptr_in[t] + before + (open ? 1 : 0));
  }
  if (bad) report(status, MOE_DEV_BAD_EXPERT_ID);
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) hist[(size_t)blockIdx.x * N + e] = sh_hist[e];
}

// One CTA; thread e owns expert e.
__global__ void __launch_bounds__(kMaxN) rr_scan(int32_t *__restrict__ hist, int nchunks, int N,
                                                 int capacity, int32_t *__restrict__ used,
                                                 int32_t *__restrict__ room,
                                                 int32_t *__restrict__ demand) {
  const int e = threadIdx.x;
  if (e >= N) return;
  int32_t total = 0;
  for (int b = 0; b < nchunks; ++b) {
    const int32_t c = hist[(size_t)b * N + e];
    hist[(size_t)b * N + e] = total;  // chunk base
    total += c;
  }
  const int32_t r = capacity - used[e];
  room[e] = r;
  used[e] += total < r ? total : r;
  if (demand) demand[e] = total;
}

__global__ void __launch_bounds__(kThreads) rr_grant(
    const int32_t *__restrict__ cand, int T, int N, int k, int kr,
    const int32_t *__restrict__ prop, const int32_t *__restrict__ chunk_base,
    const int32_t *__restrict__ room, int32_t *__restrict__ fcand, int32_t *rerouted,
    int count_rerouted) {
  extern __shared__ int32_t sm[];
  int32_t *running = sm;                  // [N] proposals of each expert in earlier sub-rounds
  int32_t *warp_cnt = sm + N;             // [8][N]
  constexpr int kWarps = kThreads / 32;
  for (int e = threadIdx.x; e < N; e += blockDim.x) running[e] = 0;
  const long a0 = (long)blockIdx.x * kChunkTokens * k;
  const long a1 = min((long)T * k, a0 + (long)kChunkTokens * k);
  const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
  const unsigned lt_mask = (1u << lane) - 1u;
  int granted = 0;
  for (long base = a0; base < a1; base += kThreads) {
    for (int q = threadIdx.x; q < kWarps * N; q += blockDim.x) warp_cnt[q] = 0;
    __syncthreads();
    const long a = base + threadIdx.x;
    const int p = (a < a1) ? prop[a] : -1;
    const int e = p >= 0 ? cand[(a / k) * kr + p] : -1;
    const bool valid = p >= 0;
    const int key = valid ? e : -1 - (int)threadIdx.x;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank_in_warp = __popc(peers & lt_mask);
    const bool last_of_group = (peers >> lane) == 1u;
    if (valid && last_of_group) warp_cnt[w * N + e] = rank_in_warp + 1;
    __syncthreads();
    if (valid) {
      int32_t r = running[e] + rank_in_warp;
      for (int w2 = 0; w2 < w; ++w2) r += warp_cnt[w2 * N + e];
      r += chunk_base[(size_t)blockIdx.x * N + e];
      if (r < room[e]) {
        fcand[a] = p;
        ++granted;
      }
    }
    __syncthreads();
    for (int q = threadIdx.x; q < N; q += blockDim.x) {
      int32_t s = 0;
      for (int w2 = 0; w2 < kWarps; ++w2) s += warp_cnt[w2 * N + q];
      running[q] += s;
    }
    __syncthreads();
  }
  if (count_rerouted && rerouted && granted) atomicAdd(rerouted, granted);
}

// Final selection per token: each slot's expert (-1 if dropped) and the
// weights renormalised over the final candidates.
__global__ void rr_finalize(const int32_t *__restrict__ cand, const float *__restrict__ cand_w,
                            int T, int k, int kr, const int32_t *__restrict__ fcand,
                            int32_t *__restrict__ final_idx, float *__restrict__ final_w) {
  for (long t = (long)blockIdx.x * blockDim.x + threadIdx.x; t < T;
       t += (long)gridDim.x * blockDim.x) {
    float s = 0.f;
    for (int j = 0; j < k; ++j) {
      const int c = fcand[t * k + j];
      s += cand_w[t * kr + (c >= 0 ? c : j)];
    }
    for (int j = 0; j < k; ++j) {
      const int c = fcand[t * k + j];
      final_idx[t * k + j] = c >= 0 ? cand[t * kr + c] : -1;
      final_w[t * k + j] = cand_w[t * kr + (c >= 0 ? c : j)] / s;
    }
  }
}

RerouteState carve(void *ws, int T, int N, int k) {
  const int nchunks = (T + kChunkTokens - 1) / kChunkTokens;
  char *p = static_cast<char *>(ws);
  auto take = [&](size_t n) {
    int32_t *q = reinterpret_cast<int32_t *>(p);
    p += align_up(n * sizeof(int32_t), 256);
    return q;
  };
  RerouteState s;
  s.hist = take((size_t)(nchunks > 0 ? nchunks : 1) * N);
  s.used = take(N);
  s.room = take(N);
  s.ptr[0] = take((size_t)T + 1);
  s.ptr[1] = take((size_t)T + 1);
  s.fcand = take((size_t)T * k + 1);
  s.prop = take((size_t)T * k + 1);
  return s;
}

}  // namespace

size_t reroute_workspace_bytes(int T, int N, int k) {
  const size_t nchunks = (size_t)(T + kChunkTokens - 1) / kChunkTokens;
  auto a = [](size_t n) { return align_up(n * sizeof(int32_t), 256); };
  return a((nchunks > 0 ? nchunks : 1) * (size_t)N) + 2 * a(N) + 2 * a((size_t)T + 1) +
         2 * a((size_t)T * k + 1);
}

moe_status_t launch_permute_reroute(const int32_t *cand, const float *cand_w, const void *x,
                                    moe_dtype_t dtype, int T, int d, int N, int k, int R,
                                    int capacity, int32_t *final_idx, float *final_w,
                                    int32_t *demand, int32_t *counts, int32_t *offsets,
                                    int32_t *perm_token, float *row_scale, int32_t *inv_pos,
                                    void *x_perm, int32_t *dropped, int32_t *rerouted,
                                    int32_t *device_status, void *workspace,
                                    cudaStream_t stream) {
  if (N > kMaxN) {
    set_error("moe_permute_reroute: N=%d above %d", N, kMaxN);
    return MOE_ERR_UNSUPPORTED;
  }
  const int kr = k + R;
  const int nchunks = (T + kChunkTokens - 1) / kChunkTokens;
  RerouteState st = carve(workspace, T, N, k);
  MOE_CUDA_TRY(cudaMemsetAsync(st.used, 0, sizeof(int32_t) * N, stream));
  MOE_CUDA_TRY(cudaMemsetAsync(st.ptr[0], 0, sizeof(int32_t) * ((size_t)T + 1), stream));
  MOE_CUDA_TRY(cudaMemsetAsync(st.fcand, 0xff, sizeof(int32_t) * ((size_t)T * k + 1), stream));
  if (rerouted) MOE_CUDA_TRY(cudaMemsetAsync(rerouted, 0, sizeof(int32_t), stream));
  if (demand && T == 0) MOE_CUDA_TRY(cudaMemsetAsync(demand, 0, sizeof(int32_t) * N, stream));
  if (T > 0) {
    const size_t grant_smem = (size_t)N * (1 + kThreads / 32) * sizeof(int32_t);
    for (int r = 0; r <= R; ++r) {
      rr_propose<<<nchunks, kThreads, N * sizeof(int32_t), stream>>>(
          cand, T, N, k, kr, st.fcand, st.ptr[r & 1], st.ptr[(r + 1) & 1], st.prop, st.hist,
          device_status);
      MOE_LAUNCH_CHECK();
      rr_scan<<<1, kMaxN, 0, stream>>>(st.hist, nchunks, N, capacity, st.used, st.room,
                                       r == 0 ? demand : nullptr);
      MOE_LAUNCH_CHECK();
      rr_grant<<<nchunks, kThreads, grant_smem, stream>>>(cand, T, N, k, kr, st.prop, st.hist,
                                                          st.room, st.fcand, rerouted, r > 0);
      MOE_LAUNCH_CHECK();
    }
    const int blocks = (int)((T + 255) / 256 < 148 * 8 ? (T + 255) / 256 : 148 * 8);
    rr_finalize<<<blocks, 256, 0, stream>>>(cand, cand_w, T, k, kr, st.fcand, final_idx,
                                            final_w);
    MOE_LAUNCH_CHECK();
  }
  // final selection through the dispatch (no capacity: it holds by construction)
  return launch_permute(final_idx, final_w, x, dtype, T, d, N, k, 0, counts, offsets,
                        perm_token, row_scale, inv_pos, x_perm, dropped, device_status,
                        st.hist, stream, /*neg_one_drops=*/true);
}

}  // namespace moe
