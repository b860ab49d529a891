// Routing diagnostics: selection frequencies, their entropy, the most chosen
// experts, std/mean, and the balance statistic N * sum f_i p_i.
//
// Source: "MoE稀疏激活原理与工程实践", 4.2 路由质量诊断 (frequency of each expert
// among the tokens' top-k, entropy in bits against log2 N, top-3 experts and
// their share, single-expert share, std/mean of the frequencies);
// "大模型MoE混合专家架构原理与DeepSeek-V4工程实践解析" (balance statistic with p_i
// the mean routing probability, i.e. the softmax over all N logits).
//
// Two launches, deterministic (fixed reduction orders, no atomics):
//   1. prob_partial (only with logits): kProbCtas CTAs (a constant, so the
//      order does not depend on the device) stride over chunks of 64 tokens;
//      warp w of a CTA sums, token by token in order, softmax(l_t) into its
//      own shared-memory row; the CTA adds its 8 rows in order ->
//      partial[c][N].  Three passes over a token's logits (max, sum of exp,
//      probabilities), the later two from L1.
//   2. finish (one CTA of 1024 threads, thread e = expert e): p_e = sum over
//      chunks in order / T, f_e = counts_e / sum(counts), and the scalars by
//      fixed tree reductions in shared memory.
// HBM-bound on the logits (T * N * 4 bytes); the counts are N integers.
#include <math.h>

#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kTok = 64;         // tokens per chunk in prob_partial (8 per warp)
constexpr int kWarps = 8;
constexpr int kProbCtas = 148;   // CTAs of prob_partial (one wave on 148 SMs)
constexpr int kMaxN = 1024;

__global__ void __launch_bounds__(kWarps * 32) prob_partial(const float *__restrict__ logits,
                                                            int T, int N,
                                                            float *__restrict__ partial) {
  extern __shared__ float rows[];   // [kWarps][N]
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  float *mine = rows + (size_t)warp * N;
  for (int e = lane; e < N; e += 32) mine[e] = 0.f;
  const int nchunks = (T + kTok - 1) / kTok;
  for (int ch = blockIdx.x; ch < nchunks; ch += gridDim.x) {
  const int t0 = ch * kTok + warp * (kTok / kWarps);
  const int t1 = min(T, t0 + kTok / kWarps);
  for (int t = t0; t < t1; ++t) {
    const float *l = logits + (size_t)t * N;
    float m = -INFINITY;
    for (int e = lane; e < N; e += 32) m = fmaxf(m, l[e]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    float s = 0.f;
    for (int e = lane; e < N; e += 32) s += expf(l[e] - m);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    const float inv = 1.f / s;
    for (int e = lane; e < N; e += 32) mine[e] += expf(l[e] - m) * inv;
  }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    float acc = 0.f;
    for (int w = 0; w < kWarps; ++w) acc += rows[(size_t)w * N + e];
    partial[(size_t)blockIdx.x * N + e] = acc;
  }
}

// Sum of v over the first `width` threads (a power of two) in a fixed tree order.
__device__ float tree_sum(float *sh, float v, int width) {
  sh[threadIdx.x] = v;
  __syncthreads();
  for (int s = width / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) sh[threadIdx.x] += sh[threadIdx.x + s];
    __syncthreads();
  }
  const float r = sh[0];
  __syncthreads();
  return r;
}

// Index of the largest key (ties -> lower index; key < 0 never wins).
__device__ int tree_argmax(float *shv, int *shi, float key, int width) {
  shv[threadIdx.x] = key;
  shi[threadIdx.x] = threadIdx.x;
  __syncthreads();
  for (int s = width / 2; s > 0; s >>= 1) {
    if (threadIdx.x < s) {
      const float a = shv[threadIdx.x], b = shv[threadIdx.x + s];
      const int ia = shi[threadIdx.x], ib = shi[threadIdx.x + s];
      if (b > a || (b == a && ib < ia)) {
        shv[threadIdx.x] = b;
        shi[threadIdx.x] = ib;
      }
    }
    __syncthreads();
  }
  const int r = shv[0] >= 0.f ? shi[0] : -1;
  __syncthreads();
  return r;
}

// have_p: logits were given (partial is null only when T == 0: all p_e = 0).
__global__ void __launch_bounds__(kMaxN) finish(const int32_t *__restrict__ counts,
                                                const float *__restrict__ partial, int nchunks,
                                                int have_p, int T, int N,
                                                moe_routing_stats_t *stats, float *freq_out,
                                                float *prob_out) {
  __shared__ float shv[kMaxN];
  __shared__ int shi[kMaxN];
  __shared__ int shc[kMaxN];
  const int e = threadIdx.x;
  const int width = blockDim.x;     // next power of two >= N (>= 32)
  const bool live = e < N;
  // total assignments (integer: any order gives the same sum)
  shc[e] = live ? counts[e] : 0;
  __syncthreads();
  for (int s = width / 2; s > 0; s >>= 1) {
    if (e < s) shc[e] += shc[e + s];
    __syncthreads();
  }
  const int total = shc[0];
  __syncthreads();
  const float f = (live && total > 0) ? (float)counts[e] / (float)total : 0.f;
  float p = 0.f;
  if (partial && live) {
#pragma unroll 8
    for (int c = 0; c < nchunks; ++c) p += partial[(size_t)c * N + e];
    p /= (float)T;
  }
  const float h = tree_sum(shv, f > 0.f ? -f * log2f(f) : 0.f, width);
  const float mean = tree_sum(shv, f, width) / (float)N;
  const float dev = live ? f - mean : 0.f;
  const float var = tree_sum(shv, dev * dev, width) / (float)N;
  const float bal = have_p ? (float)N * tree_sum(shv, f * p, width) : NAN;
  // three most chosen: repeated argmax over the frequencies of the others
  int top[3];
  bool taken = false;
  for (int r = 0; r < 3; ++r) {
    top[r] = tree_argmax(shv, shi, (live && !taken) ? f : -1.f, width);
    if (e == top[r]) taken = true;
  }
  if (live) {
    if (freq_out) freq_out[e] = f;
    if (prob_out && have_p) prob_out[e] = p;
  }
  // top-3 share and largest share from the exact frequencies of the winners
  __shared__ float fsel[3];
  for (int r = 0; r < 3; ++r)
    if (e == top[r]) fsel[r] = f;
  __syncthreads();
  if (e == 0) {
    float share = 0.f;
    for (int r = 0; r < 3; ++r) share += top[r] >= 0 ? fsel[r] : 0.f;
    stats->entropy_bits = h;
    stats->entropy_max_bits = log2f((float)N);
    stats->top3_share = share;
    stats->max_share = top[0] >= 0 ? fsel[0] : 0.f;
    stats->freq_cv = mean > 0.f ? sqrtf(var) / mean : 0.f;
    stats->balance = bal;
    for (int r = 0; r < 3; ++r) stats->top3[r] = top[r];
    stats->assignments = total;
  }
}

}  // namespace

size_t routing_stats_workspace_bytes(int T, int N) {
  const size_t nchunks = (size_t)(T + kTok - 1) / kTok;
  const size_t rows = nchunks < (size_t)kProbCtas ? nchunks : (size_t)kProbCtas;
  return align_up(rows * (size_t)N * sizeof(float), 256);
}

moe_status_t launch_routing_stats(const float *logits, const int32_t *counts, int T, int N,
                                  moe_routing_stats_t *stats, float *freq, float *prob_mean,
                                  void *workspace, cudaStream_t stream) {
  float *partial = nullptr;
  const int nchunks = (T + kTok - 1) / kTok;
  const int ctas = nchunks < kProbCtas ? nchunks : kProbCtas;
  if (logits && T > 0) {
    partial = static_cast<float *>(workspace);
    prob_partial<<<ctas, kWarps * 32, (size_t)kWarps * N * sizeof(float), stream>>>(
        logits, T, N, partial);
    MOE_LAUNCH_CHECK();
  }
  int width = 32;
  while (width < N) width <<= 1;
  finish<<<1, width, 0, stream>>>(counts, partial, partial ? ctas : 0, logits ? 1 : 0, T, N,
                                  stats, freq, prob_mean);
  MOE_LAUNCH_CHECK();
  return MOE_OK;
}

}  // namespace moe
