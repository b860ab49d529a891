/*
 * moe_oracle.c -- plain, slow, fp64 CPU oracle for the forward pass of one
 * sparse Mixture-of-Experts layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the CUDA
 * library; the two meet only through the seeded input generator.
 *
 * Every step is the plain definition written out as loops, in double
 * precision, from the exact input values (bf16 inputs are widened exactly; no
 * intermediate is rounded).  Sources, by page title and section:
 *
 *   [MoE-Sharding]  "MoE 分片：混合專家模型的平行化策略" (optiversetech.com)
 *   [MoE-Infer]     "MoE 推理：激活参数 vs 总参数与专家路由" (inference-learning-path)
 *   [MoE-DSV4]      "大模型MoE混合专家架构原理与DeepSeek-V4工程实践解析" (yunthe.com)
 *   [MoE-Primer]    "MoE 架构科普：为什么大模型要「混合专家」" (lidayun.com)
 *   [MoE-Sparse]    "MoE稀疏激活原理与工程实践：揭秘大模型参数幻觉" (CSDN)
 *
 * Readings taken where the pages are silent or disagree (each one is repeated
 * next to the function that applies it):
 *   - gate weights are the softmax over the k selected logits (renormalised);
 *   - top-k order is descending logit, equal logits -> lower expert id first,
 *     NaN ranks below every number;
 *   - the expert FFN is SwiGLU: (SiLU(x W_gate) * (x W_up)) W_down, no biases;
 *   - capacity C = ceil(cf * T * k / N); an assignment is kept iff its 0-based
 *     rank among the assignments of its expert, ordered by token index, is < C;
 *     a dropped slot contributes zero and the kept weights are not renormalised;
 *   - the optional shared expert is added with weight 1, outside the softmax;
 *   - low-precision expert weights are calibration-free FP8 E4M3 with one
 *     absmax scale per output channel (gate/up) and per token row (x).
 *
 * Parity pins for this file live in tests/test_oracle.py.  The fp64 values of
 * the expert FFN have no printed worked example on the pages; they are pinned
 * by closed-form special cases and invariants only.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1, ORACLE_F64 = 2 };

/* Widen element i of a float32, bf16 or double array to double, exactly. */
static double elem(const void *p, int dtype, size_t i) {
  if (dtype == ORACLE_F32) return (double)((const float *)p)[i];
  if (dtype == ORACLE_F64) return ((const double *)p)[i];
  uint32_t bits = ((uint32_t)((const uint16_t *)p)[i]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ------------------------------------------------------------------------- */
/* A tiny static-partition thread pool: run fn(lo, hi, ctx) over [0, n).       */
/* ------------------------------------------------------------------------- */
typedef void (*range_fn)(long lo, long hi, void *ctx);
typedef struct {
  range_fn fn;
  void *ctx;
  long lo, hi;
} range_job;

static void *range_thread(void *p) {
  range_job *j = (range_job *)p;
  j->fn(j->lo, j->hi, j->ctx);
  return NULL;
}

static void parallel_for(long n, int nthreads, range_fn fn, void *ctx) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (n < nthreads) nthreads = (int)(n > 0 ? n : 1);
  if (nthreads == 1) {
    fn(0, n, ctx);
    return;
  }
  pthread_t th[256];
  range_job jobs[256];
  for (int i = 0; i < nthreads; ++i) {
    jobs[i].fn = fn;
    jobs[i].ctx = ctx;
    jobs[i].lo = n * i / nthreads;
    jobs[i].hi = n * (i + 1) / nthreads;
    pthread_create(&th[i], NULL, range_thread, &jobs[i]);
  }
  for (int i = 0; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* ------------------------------------------------------------------------- */
/* Step 1: router linear layer.                                               */
/* [MoE-Sharding] "動態 token 路由", step 2 (router scores every expert);      */
/* [MoE-Infer] "深入原理" (router is a linear layer giving N gate logits);     */
/* [MoE-DSV4] "MoE核心机制" (g(x) computed from W_g and x).                    */
/*   logits[t,e] = sum_i x[t,i] * W_g[i,e] + bias[e]                          */
/* ------------------------------------------------------------------------- */
typedef struct {
  int d, N, dtype;
  const void *x, *Wg;
  const float *bias;
  double *logits;
} router_ctx;

static void router_rows(long lo, long hi, void *p) {
  router_ctx *c = (router_ctx *)p;
  for (long t = lo; t < hi; ++t) {
    for (int e = 0; e < c->N; ++e) {
      double acc = 0.0;
      for (int i = 0; i < c->d; ++i)
        acc += elem(c->x, c->dtype, (size_t)t * c->d + i) *
               elem(c->Wg, c->dtype, (size_t)i * c->N + e);
      if (c->bias) acc += (double)c->bias[e];
      c->logits[(size_t)t * c->N + e] = acc;
    }
  }
}

int oracle_router_logits(int T, int d, int N, int dtype, const void *x,
                         const void *Wg, const float *bias, double *logits,
                         int nthreads) {
  if (T < 0 || d < 1 || N < 1 || !x || !Wg || !logits) return 1;
  router_ctx c = {d, N, dtype, x, Wg, bias, logits};
  parallel_for(T, nthreads, router_rows, &c);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Steps 2-3: top-k selection and softmax-normalised gate weights.            */
/* [MoE-Infer] "代码" (top-k of the gate logits, then exp(l - max)/sum over   */
/* the selected k) and "深入原理" ("top-k softmax gives the weights");         */
/* [MoE-Sharding] "動態 token 路由", step 6 (0.6 / 0.4 worked example).        */
/* Reading: order by logit descending, equal logits -> lower expert id; NaN   */
/* ranks below every number.  Slot j holds the expert of rank j.              */
/* ------------------------------------------------------------------------- */
static double rank_key(double v) { return isnan(v) ? -INFINITY : v; }

/* Does expert a (logit la) come before expert b (logit lb)? */
static int ranks_before(double la, int a, double lb, int b) {
  double ka = rank_key(la), kb = rank_key(lb);
  if (ka != kb) return ka > kb;
  return a < b;
}

int oracle_topk_softmax(int T, int N, int k, const double *logits,
                        int32_t *topk_idx, double *topk_w) {
  if (T < 0 || N < 1 || k < 1 || k > N || !logits || !topk_idx || !topk_w)
    return 1;
  char *taken = (char *)calloc((size_t)N, 1);
  if (!taken) return 2;
  for (int t = 0; t < T; ++t) {
    const double *l = logits + (size_t)t * N;
    memset(taken, 0, (size_t)N);
    /* Selection: k rounds, each picking the best expert not yet taken. */
    for (int j = 0; j < k; ++j) {
      int best = -1;
      for (int e = 0; e < N; ++e) {
        if (taken[e]) continue;
        if (best < 0 || ranks_before(l[e], e, l[best], best)) best = e;
      }
      taken[best] = 1;
      topk_idx[(size_t)t * k + j] = best;
    }
    /* Softmax over the k selected logits, shifted by the largest (slot 0). */
    double lmax = l[topk_idx[(size_t)t * k]];
    double denom = 0.0;
    for (int j = 0; j < k; ++j)
      denom += exp(l[topk_idx[(size_t)t * k + j]] - lmax);
    for (int j = 0; j < k; ++j)
      topk_w[(size_t)t * k + j] = exp(l[topk_idx[(size_t)t * k + j]] - lmax) / denom;
  }
  free(taken);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Capacity.  [MoE-Sparse] 2.2 "专家容量（Expert Capacity）的硬约束";          */
/* [MoE-DSV4] "MoE训练中的负载均衡" (capacity factor caps tokens per expert). */
/* The pages give no formula; reading: C = ceil(cf * T * k / N), cf <= 0     */
/* meaning no limit (returned as 0).                                          */
/* ------------------------------------------------------------------------- */
int oracle_capacity(double cf, int T, int k, int N) {
  if (!(cf > 0.0) || N < 1) return 0;
  return (int)ceil(cf * (double)T * (double)k / (double)N);
}

/* ------------------------------------------------------------------------- */
/* Step 4-5: grouping tokens by expert ("token-level batching").             */
/* [MoE-Sparse] 3.1 (tokens of a batch are regrouped by target expert id,    */
/* e.g. {0:[t0,t1,t3], 1:[t2,t5], ...}); [MoE-Sharding] "動態 token 路由"     */
/* step 3.  For e = 0..N-1 the list of tokens t (ascending) with e among      */
/* their k experts; with capacity C > 0 only the first C of each list are     */
/* kept.                                                                      */
/*   counts[e]   = number of assignments routed to e (before capacity)        */
/*   offsets[e]  = sum of kept counts of experts < e; offsets[N] = kept total */
/*   perm_token[p] = token of kept row p; perm_slot[p] = its slot j           */
/*   inv_pos[t,j]  = row p of assignment (t,j), or -1 when dropped            */
/* ------------------------------------------------------------------------- */
int oracle_group(int T, int N, int k, int capacity, const int32_t *topk_idx,
                 int32_t *counts, int32_t *offsets, int32_t *perm_token,
                 int32_t *perm_slot, int32_t *inv_pos, int32_t *dropped) {
  if (T < 0 || N < 1 || k < 1 || capacity < 0 || !topk_idx || !counts ||
      !offsets || !inv_pos)
    return 1;
  int32_t n_dropped = 0;
  int32_t next = 0;
  for (int e = 0; e < N; ++e) {
    offsets[e] = next;
    int32_t rank = 0;
    for (int t = 0; t < T; ++t) {
      for (int j = 0; j < k; ++j) {
        if (topk_idx[(size_t)t * k + j] != e) continue;
        if (capacity > 0 && rank >= capacity) {
          inv_pos[(size_t)t * k + j] = -1;
          ++n_dropped;
        } else {
          int32_t p = next + rank;
          inv_pos[(size_t)t * k + j] = p;
          if (perm_token) perm_token[p] = t;
          if (perm_slot) perm_slot[p] = j;
        }
        ++rank;
      }
    }
    counts[e] = rank;
    next += (capacity > 0 && rank > capacity) ? capacity : rank;
  }
  offsets[N] = next;
  /* Assignments whose expert id is outside [0, N) are in no list. */
  for (long a = 0; a < (long)T * k; ++a)
    if (topk_idx[a] < 0 || topk_idx[a] >= N) {
      inv_pos[a] = -1;
      ++n_dropped;
    }
  if (dropped) *dropped = n_dropped;
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Step 6: one expert's FFN on a set of rows, SwiGLU form.                    */
/* [MoE-Sharding] "什麼是 MoE 模型" (an expert is two linear maps with an     */
/* activation between) and step 4 (the expert runs only on its tokens).       */
/* SwiGLU reading: g = x W_gate, u = x W_up, h = SiLU(g) * u with             */
/* SiLU(z) = z / (1 + exp(-z)), out = h W_down.  Layouts: W_gate, W_up [d,f], */
/* W_down [f,d], row-major.                                                   */
/* ------------------------------------------------------------------------- */
typedef struct {
  int d, f, dtype, x_dtype;
  const void *Wg, *Wu, *Wd, *xrows;
  double *out;
} ffn_ctx;

static void ffn_rows(long lo, long hi, void *p) {
  ffn_ctx *c = (ffn_ctx *)p;
  double *g = (double *)malloc(sizeof(double) * (size_t)c->f);
  double *u = (double *)malloc(sizeof(double) * (size_t)c->f);
  double *xr = (double *)malloc(sizeof(double) * (size_t)c->d);
  if (!g || !u || !xr) {
    free(g); free(u); free(xr);
    return;
  }
  for (long r = lo; r < hi; ++r) {
    for (int i = 0; i < c->d; ++i)
      xr[i] = elem(c->xrows, c->x_dtype, (size_t)r * c->d + i);
    for (int j = 0; j < c->f; ++j) g[j] = u[j] = 0.0;
    for (int i = 0; i < c->d; ++i) {
      double xi = xr[i];
      for (int j = 0; j < c->f; ++j) {
        g[j] += xi * elem(c->Wg, c->dtype, (size_t)i * c->f + j);
        u[j] += xi * elem(c->Wu, c->dtype, (size_t)i * c->f + j);
      }
    }
    double *o = c->out + (size_t)r * c->d;
    for (int q = 0; q < c->d; ++q) o[q] = 0.0;
    for (int j = 0; j < c->f; ++j) {
      double h = g[j] / (1.0 + exp(-g[j])) * u[j];
      for (int q = 0; q < c->d; ++q)
        o[q] += h * elem(c->Wd, c->dtype, (size_t)j * c->d + q);
    }
  }
  free(g); free(u); free(xr);
}

/* The hidden activations alone: h[r, j] = SiLU(g) * u for row r (the first
 * half of the expert above; used where h itself is quantised). */
typedef struct {
  int d, f, dtype, x_dtype;
  const void *Wg, *Wu, *xrows;
  double *h;
} hid_ctx;

static void hidden_rows(long lo, long hi, void *p) {
  hid_ctx *c = (hid_ctx *)p;
  for (long r = lo; r < hi; ++r) {
    double *h = c->h + (size_t)r * c->f;
    for (int j = 0; j < c->f; ++j) {
      double g = 0.0, u = 0.0;
      for (int i = 0; i < c->d; ++i) {
        const double xi = elem(c->xrows, c->x_dtype, (size_t)r * c->d + i);
        g += xi * elem(c->Wg, c->dtype, (size_t)i * c->f + j);
        u += xi * elem(c->Wu, c->dtype, (size_t)i * c->f + j);
      }
      h[j] = g / (1.0 + exp(-g)) * u;
    }
  }
}

int oracle_expert_hidden(int d, int f, int dtype, const void *W_gate_e, const void *W_up_e,
                         int R, const void *xrows, int x_dtype, double *h, int nthreads) {
  if (d < 1 || f < 1 || R < 0 || !W_gate_e || !W_up_e || (R > 0 && (!xrows || !h))) return 1;
  hid_ctx c = {d, f, dtype, x_dtype, W_gate_e, W_up_e, xrows, h};
  parallel_for(R, nthreads, hidden_rows, &c);
  return 0;
}

int oracle_expert_rows(int d, int f, int dtype, const void *W_gate_e,
                       const void *W_up_e, const void *W_down_e, int R,
                       const void *xrows, int x_dtype, double *out,
                       int nthreads) {
  if (d < 1 || f < 1 || R < 0 || !W_gate_e || !W_up_e || !W_down_e ||
      (R > 0 && (!xrows || !out)))
    return 1;
  ffn_ctx c = {d, f, dtype, x_dtype, W_gate_e, W_up_e, W_down_e, xrows, out};
  parallel_for(R, nthreads, ffn_rows, &c);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Step 7: gate-weighted combine back in token order.                         */
/* [MoE-Sharding] "動態 token 路由", step 6; [MoE-Infer] "深入原理" (output = */
/* weighted sum of its k experts); [MoE-DSV4] "MoE核心机制" (sum of g_i E_i). */
/* For each row r: y[r] = sum over kept slots j of w[r,j] * o[r,j,:]          */
/*                 (+ shared[r,:] with weight 1 when given).                  */
/* expert_out is [R, k, d]: the output of slot j's expert on row r's token.   */
/* ------------------------------------------------------------------------- */
int oracle_combine_rows(int R, int k, int d, const int32_t *inv_pos_rows,
                        const double *topk_w_rows, const double *expert_out,
                        const double *shared, double *y) {
  if (R < 0 || k < 1 || d < 1 || (R > 0 && (!inv_pos_rows || !topk_w_rows ||
                                           !expert_out || !y)))
    return 1;
  for (long r = 0; r < R; ++r) {
    double *yr = y + (size_t)r * d;
    for (int q = 0; q < d; ++q) yr[q] = 0.0;
    for (int j = 0; j < k; ++j) {
      if (inv_pos_rows[(size_t)r * k + j] < 0) continue; /* dropped slot */
      double w = topk_w_rows[(size_t)r * k + j];
      const double *o = expert_out + ((size_t)r * k + j) * d;
      for (int q = 0; q < d; ++q) yr[q] += w * o[q];
    }
    if (shared)
      for (int q = 0; q < d; ++q) yr[q] += shared[(size_t)r * d + q];
  }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Whole layer, all tokens, weights resident in host memory (small cases).    */
/* Composes steps 1-7 above.  Optional outputs may be NULL.                   */
/* ------------------------------------------------------------------------- */
int oracle_moe_forward(int T, int d, int f, int N, int k, int dtype,
                       const void *x, const void *Wg, const float *bias,
                       const void *W_gate, const void *W_up, const void *W_down,
                       int fs, const void *Ws_gate, const void *Ws_up,
                       const void *Ws_down, double capacity_factor, double *y,
                       double *logits_out, int32_t *topk_idx_out,
                       double *topk_w_out, int32_t *counts_out,
                       int32_t *offsets_out, int32_t *inv_pos_out,
                       int32_t *dropped_out, int nthreads) {
  if (T < 1 || d < 1 || f < 1 || N < 1 || k < 1 || k > N || !x || !Wg ||
      !W_gate || !W_up || !W_down || !y)
    return 1;
  if (fs > 0 && (!Ws_gate || !Ws_up || !Ws_down)) return 1;
  size_t esz = dtype == ORACLE_F32 ? 4 : 2;
  size_t TK = (size_t)T * k;
  double *logits = (double *)malloc(sizeof(double) * (size_t)T * N);
  int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * TK);
  double *w = (double *)malloc(sizeof(double) * TK);
  int32_t *counts = (int32_t *)malloc(sizeof(int32_t) * (size_t)N);
  int32_t *offsets = (int32_t *)malloc(sizeof(int32_t) * ((size_t)N + 1));
  int32_t *inv = (int32_t *)malloc(sizeof(int32_t) * TK);
  double *o = (double *)malloc(sizeof(double) * TK * d);
  double *sh = fs > 0 ? (double *)malloc(sizeof(double) * (size_t)T * d) : NULL;
  int rc = 0;
  if (!logits || !idx || !w || !counts || !offsets || !inv || !o ||
      (fs > 0 && !sh)) {
    rc = 2;
    goto done;
  }
  oracle_router_logits(T, d, N, dtype, x, Wg, bias, logits, nthreads);
  oracle_topk_softmax(T, N, k, logits, idx, w);
  int C = oracle_capacity(capacity_factor, T, k, N);
  int32_t dropped = 0;
  oracle_group(T, N, k, C, idx, counts, offsets, NULL, NULL, inv, &dropped);
  /* Expert outputs for every (t, j), one expert at a time, gathering its rows. */
  memset(o, 0, sizeof(double) * TK * d);
  for (int e = 0; e < N; ++e) {
    int R = 0;
    for (size_t a = 0; a < TK; ++a)
      if (idx[a] == e && inv[a] >= 0) ++R;
    if (R == 0) continue;
    char *xr = (char *)malloc(esz * (size_t)R * d);
    double *orow = (double *)malloc(sizeof(double) * (size_t)R * d);
    size_t *which = (size_t *)malloc(sizeof(size_t) * (size_t)R);
    if (!xr || !orow || !which) {
      free(xr); free(orow); free(which);
      rc = 2;
      goto done;
    }
    int r = 0;
    for (size_t a = 0; a < TK; ++a) {
      if (idx[a] != e || inv[a] < 0) continue;
      size_t t = a / (size_t)k;
      memcpy(xr + esz * (size_t)r * d, (const char *)x + esz * t * d, esz * d);
      which[r++] = a;
    }
    const char *wg = (const char *)W_gate + esz * (size_t)e * d * f;
    const char *wu = (const char *)W_up + esz * (size_t)e * d * f;
    const char *wd = (const char *)W_down + esz * (size_t)e * f * d;
    oracle_expert_rows(d, f, dtype, wg, wu, wd, R, xr, dtype, orow, nthreads);
    for (int q = 0; q < R; ++q)
      memcpy(o + which[q] * d, orow + (size_t)q * d, sizeof(double) * d);
    free(xr); free(orow); free(which);
  }
  if (fs > 0)
    oracle_expert_rows(d, fs, dtype, Ws_gate, Ws_up, Ws_down, T, x, dtype, sh,
                       nthreads);
  oracle_combine_rows(T, k, d, inv, w, o, sh, y);
  if (logits_out) memcpy(logits_out, logits, sizeof(double) * (size_t)T * N);
  if (topk_idx_out) memcpy(topk_idx_out, idx, sizeof(int32_t) * TK);
  if (topk_w_out) memcpy(topk_w_out, w, sizeof(double) * TK);
  if (counts_out) memcpy(counts_out, counts, sizeof(int32_t) * (size_t)N);
  if (offsets_out) memcpy(offsets_out, offsets, sizeof(int32_t) * ((size_t)N + 1));
  if (inv_pos_out) memcpy(inv_pos_out, inv, sizeof(int32_t) * TK);
  if (dropped_out) *dropped_out = dropped;
done:
  free(logits); free(idx); free(w); free(counts); free(offsets); free(inv);
  free(o); free(sh);
  return rc;
}

/*
 * Routing diagnostics (forward only).
 *
 * [MoE-Sparse] 4.2 (路由质量诊断): how often each expert is chosen among the
 * tokens' top-k, the entropy of that frequency distribution in bits (log2 N
 * when the load is even), the three most chosen experts and their combined
 * share, the largest single share, and the calibration term's std/mean of the
 * frequencies.  [MoE-DSV4] (负载均衡损失): N * sum_i f_i * p_i with f_i the
 * selection frequency and p_i the mean routing probability of expert i.
 *
 * Readings: f_i = counts_i / sum(counts), so the f_i sum to 1; the entropy
 * takes 0 log 0 = 0 (the page's "+1e-8" inside the logarithm is a numerical
 * guard); std is the population std over the N experts; p_i is the mean over
 * tokens of the softmax over all N logits (the router's probabilities before
 * the top-k); the three most chosen go by frequency, equal frequencies ->
 * lower expert id, -1 past N.  With no assignments every statistic is 0.
 *
 * stats[0] entropy (bits)  [1] log2 N  [2] top-3 share  [3] largest share
 *      [4] std/mean  [5] balance (NaN when logits is NULL)
 */
int oracle_routing_stats(int T, int N, const double *logits, const int32_t *counts,
                         double *stats, int32_t *top3, double *freq, double *prob) {
  if (T < 0 || N < 1 || !counts || !stats || !top3 || !freq) return 1;
  double total = 0.0;
  for (int e = 0; e < N; ++e) total += counts[e];
  for (int e = 0; e < N; ++e) freq[e] = total > 0 ? counts[e] / total : 0.0;
  double h = 0.0;
  for (int e = 0; e < N; ++e)
    if (freq[e] > 0) h -= freq[e] * log2(freq[e]);
  stats[0] = h;
  stats[1] = log2((double)N);
  double share = 0.0;
  for (int r = 0; r < 3; ++r) {
    int best = -1;
    for (int e = 0; e < N; ++e) {
      int taken = 0;
      for (int q = 0; q < r; ++q) taken |= (top3[q] == e);
      if (taken) continue;
      if (best < 0 || freq[e] > freq[best]) best = e;
    }
    top3[r] = best;
    if (best >= 0) share += freq[best];
  }
  stats[2] = share;
  stats[3] = top3[0] >= 0 ? freq[top3[0]] : 0.0;
  double mean = 0.0, var = 0.0;
  for (int e = 0; e < N; ++e) mean += freq[e];
  mean /= N;
  for (int e = 0; e < N; ++e) var += (freq[e] - mean) * (freq[e] - mean);
  var /= N;
  stats[4] = mean > 0 ? sqrt(var) / mean : 0.0;
  if (!logits) {
    stats[5] = NAN;
    return 0;
  }
  double *p = prob ? prob : (double *)calloc((size_t)N, sizeof(double));
  if (!p) return 2;
  for (int e = 0; e < N; ++e) p[e] = 0.0;
  for (int t = 0; t < T; ++t) {
    const double *l = logits + (size_t)t * N;
    double m = l[0];
    for (int e = 1; e < N; ++e)
      if (l[e] > m) m = l[e];
    double s = 0.0;
    for (int e = 0; e < N; ++e) s += exp(l[e] - m);
    for (int e = 0; e < N; ++e) p[e] += exp(l[e] - m) / s;
  }
  double bal = 0.0;
  for (int e = 0; e < N; ++e) {
    p[e] = T > 0 ? p[e] / T : 0.0;
    bal += freq[e] * p[e];
  }
  stats[5] = N * bal;
  if (!prob) free(p);
  return 0;
}

/*
 * Capacity overflow re-routed to the next-best expert.
 *
 * [MoE-Sparse] 2.2 (专家容量的硬约束): once an expert's queue holds its
 * capacity, a token that selects it is re-routed to its next-best expert.
 * Readings: the first pass is the capacity rule above (rank by token index
 * < C); then, in each of R rounds, every slot still without an expert
 * proposes its token's next-ranked expert not yet tried by the token (ranks
 * k, k+1, ... of the token's candidates, consumed in slot order whether the
 * proposal is granted or not), and each expert grants its remaining room to
 * that round's proposals in (token, slot) order.  A slot still unplaced after
 * R rounds is dropped.  A slot keeps the candidate it was finally granted
 * (or, if dropped, its first choice).
 *
 * Gate weights (reading): the softmax over the logits of the token's k final
 * experts -- the same rule as without re-routing, applied to the final
 * selection; a dropped slot keeps its first choice's logit in the denominator
 * and contributes nothing to the output (weights are not renormalised).
 *
 * cand [T][k+R]: each token's experts by rank (distinct); logits [T][N] or
 * NULL.  Outputs: final_cand [T][k] candidate index of each slot's expert,
 * placed [T][k], *rerouted = slots placed in rounds >= 1, final_w [T][k]
 * (written when logits is given).
 */
int oracle_reroute(int T, int N, int k, int R, int capacity, const int32_t *cand,
                   const double *logits, int32_t *final_cand, int32_t *placed,
                   int32_t *rerouted, double *final_w) {
  if (T < 0 || N < 1 || k < 1 || R < 0 || capacity < 1) return 1;
  const int kr = k + R;
  int32_t *used = (int32_t *)calloc((size_t)N, sizeof(int32_t));
  int32_t *ptr = (int32_t *)malloc(sizeof(int32_t) * ((size_t)T + 1));
  int32_t *prop = (int32_t *)malloc(sizeof(int32_t) * ((size_t)T * k + 1));
  if (!used || !ptr || !prop) { free(used); free(ptr); free(prop); return 2; }
  *rerouted = 0;
  /* first pass: the token's own top-k, by token index */
  for (int t = 0; t < T; ++t) {
    ptr[t] = k;
    for (int j = 0; j < k; ++j) {
      const int e = cand[(size_t)t * kr + j];
      final_cand[(size_t)t * k + j] = j;
      placed[(size_t)t * k + j] = 0;
      if (e >= 0 && e < N && used[e] < capacity) {
        used[e]++;
        placed[(size_t)t * k + j] = 1;
      }
    }
  }
  for (int r = 1; r <= R; ++r) {
    /* proposals: each unplaced slot takes its token's next untried candidate */
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j) {
        size_t a = (size_t)t * k + j;
        prop[a] = -1;
        if (!placed[a] && ptr[t] < kr) prop[a] = ptr[t]++;
      }
    /* grants: remaining room, in (token, slot) order */
    for (int t = 0; t < T; ++t)
      for (int j = 0; j < k; ++j) {
        size_t a = (size_t)t * k + j;
        if (prop[a] < 0) continue;
        const int e = cand[(size_t)t * kr + prop[a]];
        if (e >= 0 && e < N && used[e] < capacity) {
          used[e]++;
          placed[a] = 1;
          final_cand[a] = prop[a];
          (*rerouted)++;
        }
      }
  }
  if (logits && final_w) {
    for (int t = 0; t < T; ++t) {
      double lmax = -INFINITY, denom = 0.0;
      for (int j = 0; j < k; ++j) {
        const int e = cand[(size_t)t * kr + final_cand[(size_t)t * k + j]];
        const double l = logits[(size_t)t * N + e];
        if (l > lmax) lmax = l;
      }
      for (int j = 0; j < k; ++j) {
        const int e = cand[(size_t)t * kr + final_cand[(size_t)t * k + j]];
        denom += exp(logits[(size_t)t * N + e] - lmax);
      }
      for (int j = 0; j < k; ++j) {
        const int e = cand[(size_t)t * kr + final_cand[(size_t)t * k + j]];
        final_w[(size_t)t * k + j] = exp(logits[(size_t)t * N + e] - lmax) / denom;
      }
    }
  }
  free(used); free(ptr); free(prop);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Low-precision expert weights: FP8 E4M3 with absmax scales.                 */
/* [MoE-DSV4] "MoE模型推理部署与显存优化实战" (inference is bound by memory     */
/* bandwidth; the third remedy is quantising the weights to fewer bits, with  */
/* FP8 named for the cached activations); [MoE-Sparse] 4.3 (weights cut from  */
/* 16-bit to fewer bits to shrink memory).  Reading: calibration-free FP8     */
/* E4M3 (OCP 8-bit floating point: 1 sign, 4 exponent bits with bias 7, 3     */
/* mantissa bits, no infinities, S.1111.111 = NaN, largest finite 448).       */
/* A vector v (one token's row of x, or one output channel of a gate/up       */
/* weight matrix over d) is stored as codes q = E4M3(v * (448 / amax|v|)),    */
/* rounded to nearest with ties to an even mantissa and saturated at 448,     */
/* and one fp32 scale amax / 448 (both factors formed in fp32; an all-zero    */
/* vector takes scale 1).  Its value is decode(q) * scale.                    */
/* ------------------------------------------------------------------------- */

/* Value of an E4M3 code, from the format's definition. */
static double e4m3_value(uint8_t c) {
  const int s = c >> 7, e = (c >> 3) & 0xF, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m / 8.0, -6);          /* subnormal: m/8 * 2^-6 */
  else
    v = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: (1 + m/8) * 2^(e-7) */
  return s ? -v : v;
}

/* The 256 code values, filled once from e4m3_value (a lookup, so the loops
 * below need not recompute the definition for every element). */
static double e4m3_tab[256];
static pthread_once_t e4m3_tab_once = PTHREAD_ONCE_INIT;
static void e4m3_tab_fill(void) {
  for (int c = 0; c < 256; ++c) e4m3_tab[c] = e4m3_value((uint8_t)c);
}
static void e4m3_tab_init(void) { pthread_once(&e4m3_tab_once, e4m3_tab_fill); }

/* Nearest finite E4M3 code to v (|v| > 448 -> +-448), ties to the code with
 * an even mantissa.  The finite non-negative codes 0x00..0x7E have increasing
 * values, so a bisection finds the last code whose value is <= |v|; the
 * answer is that code or the next one, whichever is nearer.  Callers run
 * e4m3_tab_init() first. */
static uint8_t e4m3_encode(float vf) {
  const double v = (double)vf;
  const uint8_t sign = (v < 0.0 || (v == 0.0 && signbit(v))) ? 0x80 : 0;
  const double a = fabs(v);
  if (isnan(v)) return (uint8_t)(sign | 0x7F);
  if (a >= 448.0) return (uint8_t)(sign | 0x7E);
  int lo = 0, hi = 0x7E;                       /* value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    const int mid = (lo + hi) / 2;
    if (e4m3_tab[mid] <= a) lo = mid; else hi = mid;
  }
  const double dlo = a - e4m3_tab[lo], dhi = e4m3_tab[hi] - a;
  int c;
  if (dlo < dhi) c = lo;
  else if (dhi < dlo) c = hi;
  else c = (lo & 1) == 0 ? lo : hi;            /* tie: even mantissa */
  return (uint8_t)(sign | c);
}

void oracle_e4m3_decode(long n, const uint8_t *codes, double *out) {
  for (long i = 0; i < n; ++i) out[i] = e4m3_value(codes[i]);
}

void oracle_e4m3_encode(long n, const float *v, uint8_t *codes) {
  e4m3_tab_init();
  for (long i = 0; i < n; ++i) codes[i] = e4m3_encode(v[i]);
}

/* One vector of n elements at stride `stride` (element i at p[i * stride]):
 * codes to q[i * qstride], scale to *scale. */
static void quantize_vector(const void *p, int dtype, size_t base, size_t stride, int n,
                            uint8_t *q, size_t qstride, float *scale) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    const float a = fabsf((float)elem(p, dtype, base + (size_t)i * stride));
    if (a > amax) amax = a;
  }
  const float inv = amax > 0.0f ? 448.0f / amax : 1.0f;
  *scale = amax > 0.0f ? amax / 448.0f : 1.0f;
  for (int i = 0; i < n; ++i) {
    const float v = (float)elem(p, dtype, base + (size_t)i * stride) * inv;
    q[(size_t)i * qstride] = e4m3_encode(v);
  }
}

/* Rows of x [R, C]: codes [R, C], scales [R]. */
int oracle_quantize_rows_e4m3(int R, int C, int dtype, const void *x, uint8_t *q,
                              float *scale) {
  if (R < 0 || C < 1 || (R > 0 && (!x || !q || !scale))) return 1;
  e4m3_tab_init();
  for (int r = 0; r < R; ++r)
    quantize_vector(x, dtype, (size_t)r * C, 1, C, q + (size_t)r * C, 1, scale + r);
  return 0;
}

/* Gate/up weights W [N, d, f] per output channel j (a column over d):
 * codes [N, f, d] (channel-major: each channel's d codes contiguous),
 * scales [N, f].  Channels are independent; they are split over threads. */
typedef struct {
  int d, f, dtype;
  const void *W;
  uint8_t *q;
  float *scale;
} qw_ctx;

static void quantize_channels(long lo, long hi, void *p) {
  qw_ctx *c = (qw_ctx *)p;
  for (long ch = lo; ch < hi; ++ch) {
    const long e = ch / c->f, j = ch % c->f;
    quantize_vector(c->W, c->dtype, (size_t)e * c->d * c->f + j, (size_t)c->f, c->d,
                    c->q + (size_t)ch * c->d, 1, c->scale + ch);
  }
}

int oracle_quantize_weights_e4m3(int N, int d, int f, int dtype, const void *W, uint8_t *q,
                                 float *scale, int nthreads) {
  if (N < 1 || d < 1 || f < 1 || !W || !q || !scale) return 1;
  e4m3_tab_init();
  qw_ctx c = {d, f, dtype, W, q, scale};
  parallel_for((long)N * f, nthreads, quantize_channels, &c);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* The SwiGLU expert with E4M3 operands (same sources and reading as above).  */
/* Every operand is its exact dequantised value, decode(code) * scale, and    */
/* the arithmetic is the expert of step 6 in double precision:                */
/*   x_r[i]   = decode(qx[r, i]) * sx[r]            (token row, per-row scale)  */
/*   g[j]     = sum_i x_r[i] * decode(qg[j, i]) * sg[j]   (gate channel j)      */
/*   u[j]     = sum_i x_r[i] * decode(qu[j, i]) * su[j]   (up channel j)        */
/*   h[j]     = g[j] / (1 + exp(-g[j])) * u[j]                                 */
/* and the down projection either from W_down [f, d] as given,                */
/*   out[m]   = sum_j h[j] * W_down[j, m],                                     */
/* or in E4M3 too: the row h (its exact values, narrowed to fp32 as the       */
/* quantiser's definition takes them) is quantised like a token row, codes    */
/* hq[j] and one scale hs, and with W_down's channel m stored as codes        */
/* qd[m, j] (channel-major [d, f]) and scale sd[m]:                            */
/*   out[m]   = sum_j decode(hq[j]) * hs * decode(qd[m, j]) * sd[m].           */
/* ------------------------------------------------------------------------- */

/* E4M3 down projection of R rows h [R, f] (double): out [R, d]. */
typedef struct {
  int f, d;
  const double *h;
  const uint8_t *qd;
  const float *sd;
  double *out;
} down8_ctx;

static void down8_row(const down8_ctx *c, long r, uint8_t *hq) {
  float hs;
  quantize_vector(c->h, ORACLE_F64, (size_t)r * c->f, 1, c->f, hq, 1, &hs);
  double *o = c->out + (size_t)r * c->d;
  for (int m = 0; m < c->d; ++m) {
    const uint8_t *wq = c->qd + (size_t)m * c->f;
    double acc = 0.0;
    for (int j = 0; j < c->f; ++j)
      acc += (e4m3_tab[hq[j]] * (double)hs) * (e4m3_tab[wq[j]] * (double)c->sd[m]);
    o[m] = acc;
  }
}

static void down8_rows(long lo, long hi, void *p) {
  down8_ctx *c = (down8_ctx *)p;
  uint8_t *hq = (uint8_t *)malloc((size_t)c->f);
  if (!hq) return;
  for (long r = lo; r < hi; ++r) down8_row(c, r, hq);
  free(hq);
}

int oracle_down_rows_e4m3(int R, int f, int d, const double *h, const uint8_t *qd,
                          const float *sd, double *out, int nthreads) {
  if (R < 0 || f < 1 || d < 1 || !qd || !sd || (R > 0 && (!h || !out))) return 1;
  e4m3_tab_init();
  down8_ctx c = {f, d, h, qd, sd, out};
  parallel_for(R, nthreads, down8_rows, &c);
  return 0;
}

/* The whole E4M3 expert on R token rows.  Down projection: Wd [f, d] in
 * wd_dtype when qd is NULL, else the E4M3 form (qd [d, f], sd [d]). */
typedef struct {
  int d, f, wd_dtype;
  const uint8_t *qg, *qu, *qx, *qd;
  const float *sg, *su, *sx, *sd;
  const void *Wd;
  double *out;
} exp8_ctx;

static void exp8_rows(long lo, long hi, void *p) {
  exp8_ctx *c = (exp8_ctx *)p;
  double *xr = (double *)malloc(sizeof(double) * (size_t)c->d);
  double *h = (double *)malloc(sizeof(double) * (size_t)c->f);
  uint8_t *hq = (uint8_t *)malloc((size_t)c->f);
  if (!xr || !h || !hq) {
    free(xr); free(h); free(hq);
    return;
  }
  for (long r = lo; r < hi; ++r) {
    for (int i = 0; i < c->d; ++i)
      xr[i] = e4m3_tab[c->qx[(size_t)r * c->d + i]] * (double)c->sx[r];
    for (int j = 0; j < c->f; ++j) {
      const uint8_t *wg = c->qg + (size_t)j * c->d, *wu = c->qu + (size_t)j * c->d;
      double g = 0.0, u = 0.0;
      for (int i = 0; i < c->d; ++i) {
        g += xr[i] * (e4m3_tab[wg[i]] * (double)c->sg[j]);
        u += xr[i] * (e4m3_tab[wu[i]] * (double)c->su[j]);
      }
      h[j] = g / (1.0 + exp(-g)) * u;
    }
    double *o = c->out + (size_t)r * c->d;
    if (c->qd) {
      down8_ctx dc = {c->f, c->d, h, c->qd, c->sd, o};
      down8_row(&dc, 0, hq);
    } else {
      for (int m = 0; m < c->d; ++m) o[m] = 0.0;
      for (int j = 0; j < c->f; ++j)
        for (int m = 0; m < c->d; ++m)
          o[m] += h[j] * elem(c->Wd, c->wd_dtype, (size_t)j * c->d + m);
    }
  }
  free(xr); free(h); free(hq);
}

int oracle_expert_rows_e4m3(int d, int f, const uint8_t *qg, const float *sg,
                            const uint8_t *qu, const float *su, int R, const uint8_t *qx,
                            const float *sx, int wd_dtype, const void *Wd, const uint8_t *qd,
                            const float *sd, double *out, int nthreads) {
  if (d < 1 || f < 1 || R < 0 || !qg || !sg || !qu || !su || (!Wd && !qd) ||
      (qd && !sd) || (R > 0 && (!qx || !sx || !out)))
    return 1;
  e4m3_tab_init();
  exp8_ctx c = {d, f, wd_dtype, qg, qu, qx, qd, sg, su, sx, sd, Wd, out};
  parallel_for(R, nthreads, exp8_rows, &c);
  return 0;
}
