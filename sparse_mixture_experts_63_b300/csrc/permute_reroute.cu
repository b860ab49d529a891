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
// Where every 256-token chunk can hold a CTA at once (N <= 512), the rounds
// and the final grouping run in one cooperative launch with a grid barrier
// per round (rr_fused, below); otherwise each round, the first pass
// included, is three launches.  Both are deterministic and give the same
// result:
//   propose: CTA b takes the slots of tokens [256b, 256b+256): each unplaced
//            slot's proposal from the round's starting state; per-chunk
//            proposal counts per expert;
//   scan:    per expert, chunk bases, the room left (C - used) and the grants;
//   grant:   a proposal's rank among the round's proposals to its expert
//            (chunk base + rank inside the chunk, token order, as in the
//            dispatch scatter) decides it: granted iff rank < room.
// Then the final selection goes through the dispatch (-1 = dropped); the
// single launch does that grouping itself, and the rows are copied after.
#include "moe_internal.cuh"
#include "tc_ptx.cuh"

namespace moe {
namespace {

constexpr int kChunkTokens = 256;
constexpr int kThreads = 256;
constexpr int kMaxN = 1024;

struct GridBar;

struct RerouteState {
  int32_t *hist;     // [nchunks][N] proposal counts, then chunk bases
  int32_t *used;     // [N] capacity taken so far
  int32_t *room;     // [N] room at the start of the round
  int32_t *ptr[2];   // [T] each token's next untried candidate (in / out)
  int32_t *fcand;    // [T*k] candidate granted to each slot, -1 = none yet
  int32_t *prop;     // [T*k] candidate proposed this round, -1 = none
  int32_t *hist2;    // [2][nchunks][N] per-round counts of the single-launch path
  GridBar *bar;      // grid barrier state of the single-launch path
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

// ---------------------------------------------------------------------------
// The same rounds and the final grouping in ONE cooperative launch, one CTA
// per 256-token chunk (all resident).  Every CTA recomputes the per-expert
// scan from the chunks' counts -- its own chunk base, the room, the capacity
// used so far, kept in its shared memory and identical in every CTA -- so a
// round needs one grid barrier (after the proposals) and the final grouping
// one more.  Counts of consecutive rounds alternate between two buffers: the
// next round's proposals never overwrite counts another CTA may still read.
// Counts written by other CTAs are read through L2 (ld.global.cg).
// ---------------------------------------------------------------------------
constexpr int kFusedMaxN = 512;
constexpr int kFusedMaxSmem = 200 * 1024;
constexpr uint64_t kBarrierTimeoutNs = 2000000000ull;

struct GridBar {
  unsigned int count;  // arrivals at the current barrier
  unsigned int gen;    // barriers completed
  int abort;           // set by a CTA that gave up waiting
  int pad;
};

// Grid-wide barrier with a bounded wait: after 2 s it raises MOE_DEV_TIMEOUT
// and sets the abort word; every CTA that sees it returns false.
__device__ bool grid_barrier(GridBar *gb, unsigned int &gen, int32_t *status, int *sh_ok) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    const unsigned int g = gen;
    __threadfence();
    if (atomicAdd(&gb->count, 1u) == gridDim.x - 1) {
      atomicExch(&gb->count, 0u);
      __threadfence();
      atomicExch(&gb->gen, g + 1);
    } else {
      const uint64_t t0 = tc::globaltimer_ns();
      while (atomicAdd(&gb->gen, 0u) == g) {
        if (atomicAdd(&gb->abort, 0) != 0) {
          ok = 0;
          break;
        }
        if (tc::globaltimer_ns() - t0 > kBarrierTimeoutNs) {
          atomicExch(&gb->abort, 1);
          report(status, MOE_DEV_TIMEOUT);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    gen = g + 1;
    *sh_ok = ok;
  }
  __syncthreads();
  return *sh_ok != 0;
}

// Per expert e, over the chunks' counts h[nchunks][N]: the total (tot[e]) and
// the sum over the chunks before chunk c (before[e]).  Small N: the chunks
// are split over G = 256/N thread groups and the groups' sums added after.
// red: 512 ints of shared memory.  All threads call it.
__device__ void scan_chunks(const int32_t *h, int nchunks, int N, int c, int32_t *tot,
                            int32_t *before, int32_t *red) {
  const int G = N >= kThreads ? 1 : kThreads / N;
  if (G == 1) {
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
      int32_t all = 0, lt = 0;
#pragma unroll 8
      for (int b = 0; b < nchunks; ++b) {
        const int32_t v = __ldcg(h + (size_t)b * N + e);
        all += v;
        lt += b < c ? v : 0;
      }
      tot[e] = all;
      before[e] = lt;
    }
  } else {
    const int e = threadIdx.x % N, g = threadIdx.x / N;
    if (g < G) {
      int32_t all = 0, lt = 0;
#pragma unroll 4
      for (int b = g; b < nchunks; b += G) {
        const int32_t v = __ldcg(h + (size_t)b * N + e);
        all += v;
        lt += b < c ? v : 0;
      }
      red[g * N + e] = all;
      red[kThreads + g * N + e] = lt;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < N; q += blockDim.x) {
      int32_t all = 0, lt = 0;
      for (int g2 = 0; g2 < G; ++g2) {
        all += red[g2 * N + q];
        lt += red[kThreads + g2 * N + q];
      }
      tot[q] = all;
      before[q] = lt;
    }
  }
  __syncthreads();
}

// Ranks of this chunk's keyed slots (key = expert, -1 = none) in slot order:
// base[e] + the number of earlier slots of the chunk with the same key;
// calls use(a, e, rank) for every keyed slot.  All threads call it.
template <typename KeyFn, typename UseFn>
__device__ void chunk_ranks(long a0, long a1, int N, const int32_t *base, int32_t *running,
                            int32_t *warp_cnt, KeyFn key_of, UseFn use) {
  constexpr int kWarps = kThreads / 32;
  const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
  const unsigned lt_mask = (1u << lane) - 1u;
  for (int e = threadIdx.x; e < N; e += blockDim.x) running[e] = 0;
  __syncthreads();
  for (long b0 = a0; b0 < a1; b0 += kThreads) {
    for (int q = threadIdx.x; q < kWarps * N; q += blockDim.x) warp_cnt[q] = 0;
    __syncthreads();
    const long a = b0 + threadIdx.x;
    const int e = (a < a1) ? key_of(a) : -1;
    const bool valid = e >= 0;
    const int key = valid ? e : -1 - (int)threadIdx.x;
    const unsigned peers = __match_any_sync(0xffffffffu, key);
    const int rank_in_warp = __popc(peers & lt_mask);
    if (valid && (peers >> lane) == 1u) warp_cnt[w * N + e] = rank_in_warp + 1;
    __syncthreads();
    if (valid) {
      int32_t r = base[e] + running[e] + rank_in_warp;
      for (int w2 = 0; w2 < w; ++w2) r += warp_cnt[w2 * N + e];
      use(a, e, r);
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

struct FusedArgs {
  const int32_t *cand;
  const float *cand_w;
  int T, N, k, kr, R, capacity, nchunks;
  int32_t *final_idx;
  float *final_w;
  int32_t *demand, *counts, *offsets, *perm_token;
  float *row_scale;
  int32_t *inv_pos, *dropped, *rerouted, *status;
  int32_t *hist;    // [2][nchunks][N] proposal counts per chunk, alternating rounds
  int32_t *fhist;   // [nchunks][N] final placements per chunk
  GridBar *bar;     // zeroed before the launch
};

// Shared memory of rr_fused: per-expert state (5 N), the match-and-count
// table (8 N), the scan's group sums (512), the tokens' candidate pointers
// (2 x 256), then this chunk's candidates (256 kr), grants and proposals
// (256 k each).
size_t fused_smem_bytes(int N, int k, int kr) {
  return sizeof(int32_t) * ((size_t)(5 + kThreads / 32) * N + 2 * kThreads + 2 * kChunkTokens +
                            (size_t)kChunkTokens * (kr + 2 * k));
}

__global__ void __launch_bounds__(kThreads) rr_fused(const FusedArgs p) {
  extern __shared__ int32_t sm[];
  const int N = p.N, k = p.k, kr = p.kr;
  int32_t *used = sm;                            // [N] capacity taken so far
  int32_t *room = used + N;                      // [N] room at the round's start; offsets at the end
  int32_t *base = room + N;                      // [N] this chunk's first rank
  int32_t *running = base + N;                   // [N]
  int32_t *cnt = running + N;                    // [N] this chunk's counts; totals after a scan
  int32_t *warp_cnt = cnt + N;                   // [8][N]
  int32_t *red = warp_cnt + (kThreads / 32) * N; // [2][256]
  int32_t *ptr = red + 2 * kThreads;             // [2][256] each token's next untried candidate
  int32_t *cand_s = ptr + 2 * kChunkTokens;      // [256][kr] this chunk's candidates
  int32_t *fcand = cand_s + kChunkTokens * kr;   // [256][k] candidate granted, -1 = none yet
  int32_t *prop = fcand + kChunkTokens * k;      // [256][k] proposal; final expert at the end
  __shared__ int ok_s;
  __shared__ int32_t total_s;
  const int c = blockIdx.x;
  const long t0 = (long)c * kChunkTokens;
  const int ntok = (int)min((long)kChunkTokens, (long)p.T - t0);
  const int A = ntok * k;        // this chunk's slots, local index q = (t - t0) k + j
  const long a0 = t0 * k;        // global index of local slot 0
  unsigned int gen = 0;
  int granted = 0;
  for (int e = threadIdx.x; e < N; e += blockDim.x) used[e] = 0;
  for (int i = threadIdx.x; i < 2 * kChunkTokens; i += blockDim.x) ptr[i] = 0;
  for (int q = threadIdx.x; q < A; q += blockDim.x) fcand[q] = -1;
  for (int i = threadIdx.x; i < ntok * kr; i += blockDim.x) cand_s[i] = p.cand[t0 * kr + i];
  // the re-routed count is added to only after the first barrier
  if (c == 0 && threadIdx.x == 0 && p.rerouted) *p.rerouted = 0;
  __syncthreads();
  for (int r = 0; r <= p.R; ++r) {
    const int32_t *ptr_in = ptr + (r & 1) * kChunkTokens;
    int32_t *ptr_out = ptr + ((r + 1) & 1) * kChunkTokens;
    int32_t *hist = p.hist + (size_t)(r & 1) * p.nchunks * N;
    // proposals from the round's starting state, counted per expert
    for (int e = threadIdx.x; e < N; e += blockDim.x) cnt[e] = 0;
    __syncthreads();
    bool bad = false;
    for (int q = threadIdx.x; q < A; q += blockDim.x) {
      const int tl = q / k;
      const int j = q - tl * k;
      int before = 0;   // unplaced slots of this token before slot j
      for (int jj = 0; jj < j; ++jj) before += fcand[tl * k + jj] < 0 ? 1 : 0;
      const bool open = fcand[q] < 0;
      int pr = -1;
      if (open) {
        const int ci = ptr_in[tl] + before;
        if (ci < kr) {
          const int e = cand_s[tl * kr + ci];
          if (e >= 0 && e < N) {
            pr = ci;
            atomicAdd(&cnt[e], 1);
          } else {
            bad = true;
          }
        }
      }
      prop[q] = pr;
      if (j == k - 1) ptr_out[tl] = min(kr, ptr_in[tl] + before + (open ? 1 : 0));
    }
    if (bad) report(p.status, MOE_DEV_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < N; e += blockDim.x) hist[(size_t)c * N + e] = cnt[e];
    if (!grid_barrier(p.bar, gen, p.status, &ok_s)) return;
    scan_chunks(hist, p.nchunks, N, c, cnt, base, red);
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
      const int32_t tot = cnt[e], rm = p.capacity - used[e];
      room[e] = rm;
      used[e] += tot < rm ? tot : rm;
      if (r == 0 && c == 0 && p.demand) p.demand[e] = tot;
    }
    __syncthreads();
    // grants: a proposal is granted iff its rank among the round's proposals
    // to its expert (chunk base + rank inside the chunk) is below the room
    chunk_ranks(
        0, A, N, base, running, warp_cnt,
        [&](long q) {
          const int pr = prop[q];
          return pr >= 0 ? cand_s[(q / k) * kr + pr] : -1;
        },
        [&](long q, int e, int32_t rank) {
          if (rank < room[e]) {
            fcand[q] = prop[q];
            if (r > 0) ++granted;
          }
        });
  }
  if (p.rerouted && granted) atomicAdd(p.rerouted, granted);
  // final selection for this chunk's tokens; weights renormalised over the
  // final candidates (a dropped slot keeps its first choice in the sum)
  for (int tl = threadIdx.x; tl < ntok; tl += blockDim.x) {
    const long t = t0 + tl;
    float s = 0.f;
    for (int j = 0; j < k; ++j) {
      const int ci = fcand[tl * k + j];
      s += p.cand_w[t * kr + (ci >= 0 ? ci : j)];
    }
    for (int j = 0; j < k; ++j) {
      const int ci = fcand[tl * k + j];
      const int e = ci >= 0 ? cand_s[tl * kr + ci] : -1;
      prop[tl * k + j] = e;
      p.final_idx[t * k + j] = e;
      p.final_w[t * k + j] = p.cand_w[t * kr + (ci >= 0 ? ci : j)] / s;
    }
  }
  for (int e = threadIdx.x; e < N; e += blockDim.x) cnt[e] = 0;
  __syncthreads();
  // final grouping, stable by slot: per-chunk placements, one barrier, scan
  for (int q = threadIdx.x; q < A; q += blockDim.x) {
    const int e = prop[q];
    if (e >= 0) atomicAdd(&cnt[e], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) p.fhist[(size_t)c * N + e] = cnt[e];
  if (!grid_barrier(p.bar, gen, p.status, &ok_s)) return;
  scan_chunks(p.fhist, p.nchunks, N, c, cnt, base, red);
  if (threadIdx.x == 0) {
    int32_t acc = 0;
    for (int e = 0; e < N; ++e) {
      room[e] = acc;
      acc += cnt[e];
    }
    total_s = acc;
  }
  __syncthreads();
  if (c == 0) {
    for (int e = threadIdx.x; e < N; e += blockDim.x) {
      p.counts[e] = cnt[e];
      p.offsets[e] = room[e];
    }
    if (threadIdx.x == 0) {
      p.offsets[N] = total_s;
      if (p.dropped) *p.dropped = (int32_t)((long)p.T * k - total_s);
    }
  }
  for (int q = threadIdx.x; q < A; q += blockDim.x)
    if (prop[q] < 0) p.inv_pos[a0 + q] = -1;
  chunk_ranks(
      0, A, N, base, running, warp_cnt, [&](long q) { return prop[q]; },
      [&](long q, int e, int32_t rank) {
        const int32_t pos = room[e] + rank;
        p.inv_pos[a0 + q] = pos;
        p.perm_token[pos] = (int32_t)(t0 + q / k);
        if (p.row_scale) p.row_scale[pos] = p.final_w[a0 + q];
      });
}

// Blocks of rr_fused resident at once on this device with the given shared
// memory (0 if cooperative launches are not supported); the attribute that
// lets it take more than 48 KB is set once per device.
int fused_max_blocks(size_t smem) {
  static bool coop_known[kMaxDevicesCached];
  static int coop_sms[kMaxDevicesCached];
  const int dev = current_device();
  int sms = 0;
  if (dev >= 0 && dev < kMaxDevicesCached && coop_known[dev]) {
    sms = coop_sms[dev];
  } else {
    int coop = 0, n = 0;
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    cudaFuncSetAttribute(rr_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, kFusedMaxSmem);
    sms = coop ? n : 0;
    if (dev >= 0 && dev < kMaxDevicesCached) {
      coop_sms[dev] = sms;
      coop_known[dev] = true;
    }
  }
  if (sms == 0 || smem > (size_t)kFusedMaxSmem) return 0;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, rr_fused, kThreads, smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return sms * per_sm;
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
  s.hist2 = take((size_t)2 * (nchunks > 0 ? nchunks : 1) * N);
  s.bar = reinterpret_cast<GridBar *>(take(sizeof(GridBar) / sizeof(int32_t)));
  return s;
}

}  // namespace

size_t reroute_workspace_bytes(int T, int N, int k) {
  const size_t nchunks = (size_t)(T + kChunkTokens - 1) / kChunkTokens;
  const size_t nc = nchunks > 0 ? nchunks : 1;
  auto a = [](size_t n) { return align_up(n * sizeof(int32_t), 256); };
  return a(nc * (size_t)N) + 2 * a(N) + 2 * a((size_t)T + 1) + 2 * a((size_t)T * k + 1) +
         a(2 * nc * (size_t)N) + a(sizeof(GridBar) / sizeof(int32_t));
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
  const size_t fsmem = fused_smem_bytes(N, k, kr);
  if (T > 0 && N <= kFusedMaxN && nchunks <= fused_max_blocks(fsmem)) {
    // one cooperative launch for the rounds and the grouping, then the rows
    MOE_CUDA_TRY(cudaMemsetAsync(st.bar, 0, sizeof(GridBar), stream));
    FusedArgs a;
    a.cand = cand;
    a.cand_w = cand_w;
    a.T = T;
    a.N = N;
    a.k = k;
    a.kr = kr;
    a.R = R;
    a.capacity = capacity;
    a.nchunks = nchunks;
    a.final_idx = final_idx;
    a.final_w = final_w;
    a.demand = demand;
    a.counts = counts;
    a.offsets = offsets;
    a.perm_token = perm_token;
    a.row_scale = row_scale;
    a.inv_pos = inv_pos;
    a.dropped = dropped;
    a.rerouted = rerouted;
    a.status = device_status;
    a.hist = st.hist2;
    a.fhist = st.hist;
    a.bar = st.bar;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.gridDim = dim3(nchunks);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = fsmem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, rr_fused, a));
    MOE_LAUNCH_CHECK();
    return launch_copy_rows(x, dtype, inv_pos, T, d, k, x_perm, stream);
  }
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
