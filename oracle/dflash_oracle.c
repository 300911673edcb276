/*
 * dflash_oracle.c -- plain, slow, fp64 CPU oracle for the batched
 * draft-verification step of block-drafted speculative decoding.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the
 * benchmark's CPU-baseline leg, never by the GPU library, with which it shares
 * no code. Single-threaded; a caller may run disjoint request ranges on
 * several threads (no global state).
 *
 * What it follows, step by step (page titles and sections; the pages are
 * listed in dflash_oracle.h):
 *  1. Logits are read exactly (bf16 widened to fp32 to fp64).
 *  2. Temperature: z = x / T (model card: temperature 1.0). T == 0 means
 *     greedy decoding for that request.
 *  3. Top-k on the raw logits, order (logit desc, token index asc) (model
 *     card: top-k 20). Softmax over the k survivors.
 *  4. Top-p on that renormalised mass, in the same order: keep a token while
 *     the mass strictly before it is < top_p (model card: top-p 0.95), then
 *     renormalise.
 *  5. Draft/verify loop (bml.asia pseudocode; rytg.cn "裁决" step): for each
 *     draft token in order accept with probability min(1, p/q); at the first
 *     rejection draw from the normalised residual max(0, p - q) and stop; if
 *     every draft is accepted draw a bonus token from the last target
 *     position. Greedy: accept while the draft equals the target argmax,
 *     then emit the argmax ("greedy output matches the target model
 *     exactly").
 *  6. Uniforms from Philox4x32-10 (Salmon et al., SC'11) keyed by
 *     (seed, request, position).
 *
 * Decisions that turn floating point into an integer (the accept test, the
 * top-p cut, the inverse-CDF draw) are taken in fp32: both sides of the
 * comparison are computed in fp64 and rounded to fp32 before comparing, the
 * precision the GPU kernels decide in. Everything else stays in fp64.
 */
#include "dflash_oracle.h"

#include <float.h>
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al. 2011, section 4 "Philox"): ten rounds of a   */
/* multiply-based bijection on four 32-bit words; the two 32-bit key words   */
/* advance by the Weyl constants (golden ratio, sqrt(3)-1) between rounds.   */
/* ------------------------------------------------------------------ */
static const uint32_t PHILOX_MUL_A = 0xD2511F53u;
static const uint32_t PHILOX_MUL_B = 0xCD9E8D57u;
static const uint32_t WEYL_A = 0x9E3779B9u;
static const uint32_t WEYL_B = 0xBB67AE85u;

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += WEYL_A;
      k1 += WEYL_B;
    }
    uint64_t prod_a = (uint64_t)PHILOX_MUL_A * (uint64_t)x0;
    uint64_t prod_b = (uint64_t)PHILOX_MUL_B * (uint64_t)x2;
    uint32_t y0 = (uint32_t)(prod_b >> 32) ^ x1 ^ k0;
    uint32_t y1 = (uint32_t)prod_b;
    uint32_t y2 = (uint32_t)(prod_a >> 32) ^ x3 ^ k1;
    uint32_t y3 = (uint32_t)prod_a;
    x0 = y0;
    x1 = y1;
    x2 = y2;
    x3 = y3;
  }
  out[0] = x0;
  out[1] = x1;
  out[2] = x2;
  out[3] = x3;
}

void oracle_uniforms(uint64_t seed, uint32_t request, uint32_t position, uint32_t stream,
                     float* u_accept, float* u_draw) {
  uint32_t ctr[4] = {position, request, stream, 0u};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t w[4];
  oracle_philox4x32_10(ctr, key, w);
  /* 24-bit dyadic rationals: exact in fp32 */
  if (u_accept) *u_accept = (float)((double)(w[0] >> 8) / 16777216.0);
  if (u_draw) *u_draw = (float)((double)(w[1] >> 8) / 16777216.0);
}

/* ------------------------------------------------------------------ */
/* row access                                                           */
/* ------------------------------------------------------------------ */
static double logit_at(const void* row, int dtype, size_t j) {
  if (dtype == ORC_BF16) {
    uint16_t h = ((const uint16_t*)row)[j];
    uint32_t bits = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  return (double)((const float*)row)[j];
}

static size_t elem_size(int dtype) { return dtype == ORC_BF16 ? 2u : 4u; }

/* A row is unusable when it holds a NaN or its largest logit is infinite. */
static int row_is_bad(const double* x, int V) {
  double m = -INFINITY;
  for (int j = 0; j < V; ++j) {
    if (isnan(x[j])) return 1;
    if (x[j] > m) m = x[j];
  }
  return !isfinite(m);
}

static void update_margin(double* margin, double a, double b) {
  if (!margin) return;
  double scale = fabs(b) > 1e-300 ? fabs(b) : 1e-300;
  double gap = fabs(a - b) / scale;
  if (gap < *margin) *margin = gap;
}

/* The absolute gap |a - b|: the margin of an inverse-CDF decision, whose two
 * sides (u times the total weight, a cumulative weight) are sums of
 * probabilities; an implementation's error on them is bounded in the same
 * units (a multiple of the fp32 rounding unit times the mass summed), not
 * relative to the cumulative weight, which can be tiny. */
static void update_margin_abs(double* margin, double a, double b) {
  if (!margin) return;
  double gap = fabs(a - b);
  if (gap < *margin) *margin = gap;
}

int32_t oracle_argmax_row(const void* row, int V, int dtype, uint32_t* status) {
  int32_t best = 0;
  double best_x = logit_at(row, dtype, 0);
  int bad = isnan(best_x);
  for (int j = 1; j < V; ++j) {
    double x = logit_at(row, dtype, (size_t)j);
    if (isnan(x)) bad = 1;
    if (x > best_x) { /* strictly greater: equal values keep the lower index */
      best_x = x;
      best = j;
    }
  }
  if (!isfinite(best_x)) bad = 1;
  if (bad && status) *status |= ORC_STATUS_BAD_ROW;
  return best;
}

/* ------------------------------------------------------------------ */
/* filtering: temperature -> top-k -> softmax -> top-p -> renormalise   */
/* ------------------------------------------------------------------ */
typedef struct {
  double x;
  int32_t j;
} entry_t;

/* (logit desc, index asc) */
static int entry_cmp(const void* a, const void* b) {
  const entry_t* ea = (const entry_t*)a;
  const entry_t* eb = (const entry_t*)b;
  if (ea->x > eb->x) return -1;
  if (ea->x < eb->x) return 1;
  return (ea->j < eb->j) ? -1 : (ea->j > eb->j) ? 1 : 0;
}

/* Returns the kept-set size, or -1 for a bad row / allocation failure.
 * order[0..n-1] receives the kept tokens (logit desc, index asc) and
 * p[0..n-1] their filtered probabilities. order/p need V entries. */
static int filter_core(const void* row, int V, int dtype, double T, int top_k, float top_p,
                       int32_t* order, double* p, double* margin) {
  double* x = (double*)malloc(sizeof(double) * (size_t)V);
  entry_t* e = (entry_t*)malloc(sizeof(entry_t) * (size_t)V);
  if (!x || !e) {
    free(x);
    free(e);
    return -1;
  }
  for (int j = 0; j < V; ++j) x[j] = logit_at(row, dtype, (size_t)j);
  if (row_is_bad(x, V)) {
    free(x);
    free(e);
    return -1;
  }
  const int k = (top_k <= 0 || top_k >= V) ? V : top_k;
  const int cut = top_p < 1.0f;
  for (int j = 0; j < V; ++j) {
    e[j].x = x[j];
    e[j].j = j;
  }
  if (k < V || cut) qsort(e, (size_t)V, sizeof(entry_t), entry_cmp);

  double xmax = x[0];
  for (int j = 1; j < V; ++j)
    if (x[j] > xmax) xmax = x[j];
  const double zmax = xmax / T;

  /* softmax over the k survivors (the weights are kept unnormalised) */
  int n = k;
  double W = 0.0;
  for (int t = 0; t < n; ++t) {
    order[t] = e[t].j;
    p[t] = exp(e[t].x / T - zmax);
    W += p[t];
  }
  /* top-p: keep token t while the mass strictly before it is < top_p */
  if (cut) {
    double before = 0.0;
    for (int t = 0; t < n; ++t) {
      float before_f = (float)before;
      update_margin(margin, before, (double)top_p);
      if (!(before_f < top_p)) {
        n = t;
        break;
      }
      before += p[t] / W;
    }
  }
  double Wkept = 0.0;
  for (int t = 0; t < n; ++t) Wkept += p[t];
  for (int t = 0; t < n; ++t) p[t] = p[t] / Wkept;
  free(x);
  free(e);
  return n;
}

int oracle_filter_row_sparse(const void* row, int V, int dtype, double temperature, int top_k,
                             float top_p, int32_t* idx, double* prob) {
  if (!row || V <= 0 || !(temperature > 0.0) || !isfinite(temperature) || !(top_p > 0.0f))
    return -1;
  return filter_core(row, V, dtype, temperature, top_k, top_p, idx, prob, NULL);
}

static int filter_dense(const void* row, int V, int dtype, double T, int top_k, float top_p,
                        double* dense, double* margin) {
  int32_t* order = (int32_t*)malloc(sizeof(int32_t) * (size_t)V);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  if (!order || !p) {
    free(order);
    free(p);
    return -1;
  }
  int n = filter_core(row, V, dtype, T, top_k, top_p, order, p, margin);
  if (n >= 0) {
    for (int j = 0; j < V; ++j) dense[j] = 0.0;
    for (int t = 0; t < n; ++t) dense[order[t]] = p[t];
  }
  free(order);
  free(p);
  return n;
}

int oracle_filter_row(const void* row, int V, int dtype, double temperature, int top_k,
                      float top_p, double* prob) {
  if (!row || !prob || V <= 0 || !(temperature > 0.0) || !isfinite(temperature) ||
      !(top_p > 0.0f))
    return -1;
  return filter_dense(row, V, dtype, temperature, top_k, top_p, prob, NULL);
}

/* Inverse CDF in ascending token order: the smallest token j whose
 * cumulative weight exceeds u * (total weight); if rounding leaves none, the
 * last token with positive weight. */
static int32_t draw_ascending(const double* w, int V, float u, double* margin) {
  double Z = 0.0;
  for (int j = 0; j < V; ++j) Z += w[j];
  const double target = (double)u * Z;
  const float target_f = (float)target;
  double cum = 0.0, prev = 0.0;
  int32_t last_positive = -1;
  for (int j = 0; j < V; ++j) {
    if (!(w[j] > 0.0)) continue;
    last_positive = j;
    prev = cum;
    cum += w[j];
    if (target_f < (float)cum) {
      update_margin_abs(margin, target, cum);
      if (prev > 0.0) update_margin_abs(margin, target, prev);
      return j;
    }
  }
  return last_positive;
}

static int temperature_kind(float T, uint32_t* status) {
  /* 1 = sampling, 0 = greedy */
  if (T == 0.0f) return 0;
  if (T > 0.0f && isfinite(T)) return 1;
  if (status) *status |= ORC_STATUS_BAD_TEMPERATURE;
  return 0;
}

static void greedy_request(const void* target_b, const int32_t* d, int gamma, int V, int dtype,
                           int32_t* out, int32_t* len, uint32_t* status) {
  const size_t row_bytes = (size_t)V * elem_size(dtype);
  for (int t = 0; t <= gamma; ++t) out[t] = -1;
  int32_t argmax[gamma + 1];
  for (int i = 0; i <= gamma; ++i)
    argmax[i] = oracle_argmax_row((const char*)target_b + (size_t)i * row_bytes, V, dtype, status);
  int n = 0;
  for (int i = 0; i < gamma; ++i) {
    if (d[i] < 0 || d[i] >= V) *status |= ORC_STATUS_BAD_TOKEN;
  }
  while (n < gamma && d[n] == argmax[n]) {
    out[n] = d[n];
    ++n;
  }
  out[n] = argmax[n];
  *len = n + 1;
}

int oracle_verify_greedy(const void* target, const int32_t* draft_tokens, int B, int gamma, int V,
                         int dtype, int32_t* out_tokens, int32_t* out_accept_len,
                         uint32_t* status, int b_begin, int b_end) {
  if (!target || !draft_tokens || !out_tokens || !out_accept_len || B < 0 || gamma < 1 || V < 1)
    return ORC_ERR_INVALID_ARG;
  if (b_begin < 0) b_begin = 0;
  if (b_end > B) b_end = B;
  const size_t row_bytes = (size_t)V * elem_size(dtype);
  uint32_t st = 0;
  for (int b = b_begin; b < b_end; ++b) {
    greedy_request((const char*)target + (size_t)b * (size_t)(gamma + 1) * row_bytes,
                   draft_tokens + (size_t)b * gamma, gamma, V, dtype,
                   out_tokens + (size_t)b * (gamma + 1), out_accept_len + b, &st);
  }
  if (status) *status |= st;
  return ORC_OK;
}

/* A request's margins: with margin_cut given, the accept tests' and the
 * top-p cuts' apart; without it, margin_accept holds the smaller of the two. */
static void store_margins(int b, double accept, double cut, double draw, double* margin_accept,
                          double* margin_cut, double* margin_draw) {
  if (margin_cut) {
    margin_cut[b] = cut;
    if (margin_accept) margin_accept[b] = accept;
  } else if (margin_accept) {
    margin_accept[b] = accept < cut ? accept : cut;
  }
  if (margin_draw) margin_draw[b] = draw;
}

int oracle_verify_margins(const void* target, const void* draft, const int32_t* draft_tokens,
                          int B, int gamma, int V, int dtype, const float* temperature, int top_k,
                          float top_p, uint64_t seed, int32_t* out_tokens,
                          int32_t* out_accept_len, double* margin_accept, double* margin_draw,
                          double* margin_cut, uint32_t* status, int b_begin, int b_end) {
  if (!target || !draft || !draft_tokens || !temperature || !out_tokens || !out_accept_len ||
      B < 0 || gamma < 1 || V < 1 || !(top_p > 0.0f))
    return ORC_ERR_INVALID_ARG;
  if (b_begin < 0) b_begin = 0;
  if (b_end > B) b_end = B;
  const size_t row_bytes = (size_t)V * elem_size(dtype);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  double* x = (double*)malloc(sizeof(double) * (size_t)V);
  if (!p || !q || !r || !x) {
    free(p);
    free(q);
    free(r);
    free(x);
    return ORC_ERR_NOMEM;
  }
  uint32_t st = 0;
  for (int b = b_begin; b < b_end; ++b) {
    const char* Xb = (const char*)target + (size_t)b * (size_t)(gamma + 1) * row_bytes;
    const char* Yb = (const char*)draft + (size_t)b * (size_t)gamma * row_bytes;
    const int32_t* d = draft_tokens + (size_t)b * gamma;
    int32_t* out = out_tokens + (size_t)b * (gamma + 1);
    double mg = DBL_MAX;   /* accept tests */
    double mgc = DBL_MAX;  /* top-p cuts */
    double mgd = DBL_MAX;  /* the final inverse-CDF draw */
    if (!temperature_kind(temperature[b], &st)) {
      greedy_request(Xb, d, gamma, V, dtype, out, out_accept_len + b, &st);
      store_margins(b, mg, mgc, mgd, margin_accept, margin_cut, margin_draw);
      continue;
    }
    const double T = (double)temperature[b];
    /* every row the step reads is checked, whatever the accept loop uses */
    for (int i = 0; i <= gamma; ++i) {
      for (int j = 0; j < V; ++j) x[j] = logit_at(Xb + (size_t)i * row_bytes, dtype, (size_t)j);
      if (row_is_bad(x, V)) st |= ORC_STATUS_BAD_ROW;
    }
    for (int i = 0; i < gamma; ++i) {
      for (int j = 0; j < V; ++j) x[j] = logit_at(Yb + (size_t)i * row_bytes, dtype, (size_t)j);
      if (row_is_bad(x, V)) st |= ORC_STATUS_BAD_ROW;
      if (d[i] < 0 || d[i] >= V) st |= ORC_STATUS_BAD_TOKEN;
    }
    for (int t = 0; t <= gamma; ++t) out[t] = -1;
    int n = 0;
    int32_t last = -1;
    int rejected = 0;
    for (int i = 0; i < gamma; ++i) {
      int np = filter_dense(Xb + (size_t)i * row_bytes, V, dtype, T, top_k, top_p, p, &mgc);
      int nq = filter_dense(Yb + (size_t)i * row_bytes, V, dtype, T, top_k, top_p, q, &mgc);
      if (np < 0 || nq < 0) { /* bad row: output unspecified, keep it in range */
        last = oracle_argmax_row(Xb + (size_t)i * row_bytes, V, dtype, NULL);
        rejected = 1;
        break;
      }
      const int32_t tok = d[i];
      const double p_d = (tok >= 0 && tok < V) ? p[tok] : 0.0;
      const double q_d = (tok >= 0 && tok < V) ? q[tok] : 0.0;
      float u_acc, u_draw;
      oracle_uniforms(seed, (uint32_t)b, (uint32_t)i, 0u, &u_acc, &u_draw);
      const double ratio = p_d / q_d; /* q_d == 0: +inf if p_d > 0, NaN if p_d == 0 */
      if (isfinite(ratio)) update_margin(&mg, (double)u_acc, ratio);
      if (u_acc < (float)ratio) {
        out[n++] = tok;
        continue;
      }
      /* rejected: residual max(0, p - q), normalised by the draw */
      double Zr = 0.0;
      for (int j = 0; j < V; ++j) {
        r[j] = p[j] - q[j] > 0.0 ? p[j] - q[j] : 0.0;
        Zr += r[j];
      }
      last = draw_ascending(Zr > 0.0 ? r : p, V, u_draw, &mgd);
      rejected = 1;
      break;
    }
    if (!rejected) {
      int np = filter_dense(Xb + (size_t)gamma * row_bytes, V, dtype, T, top_k, top_p, p, &mgc);
      if (np < 0) {
        last = oracle_argmax_row(Xb + (size_t)gamma * row_bytes, V, dtype, NULL);
      } else {
        float u_draw;
        oracle_uniforms(seed, (uint32_t)b, (uint32_t)gamma, 0u, NULL, &u_draw);
        last = draw_ascending(p, V, u_draw, &mgd);
      }
    }
    out[n] = last;
    out_accept_len[b] = n + 1;
    store_margins(b, mg, mgc, mgd, margin_accept, margin_cut, margin_draw);
  }
  free(p);
  free(q);
  free(r);
  free(x);
  if (status) *status |= st;
  return ORC_OK;
}

/* Verification of deterministic drafts: the drafter's distribution at
 * position i is the point mass at d_i (q = delta_d), as for a greedy drafter
 * (bml.asia, the speculative-decoding listing's drafter) or a path selector
 * (rytg.cn, the lightweight-selector paragraph). The rule is the general one with that q: accept d_i when
 * u < min(1, p_i(d_i) / 1), and at the first rejection draw from the
 * normalised residual max(0, p_i - delta_{d_i}), which is p_i with d_i taken
 * out; when every draft is accepted, the bonus token from p_gamma. No draft
 * logits are read. */
int oracle_verify_det_margins(const void* target, const int32_t* draft_tokens, int B, int gamma,
                              int V, int dtype, const float* temperature, int top_k, float top_p,
                              uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len,
                              double* margin_accept, double* margin_draw, double* margin_cut,
                              uint32_t* status, int b_begin, int b_end) {
  if (!target || !draft_tokens || !temperature || !out_tokens || !out_accept_len || B < 0 ||
      gamma < 1 || V < 1 || !(top_p > 0.0f))
    return ORC_ERR_INVALID_ARG;
  if (b_begin < 0) b_begin = 0;
  if (b_end > B) b_end = B;
  const size_t row_bytes = (size_t)V * elem_size(dtype);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  double* r = (double*)malloc(sizeof(double) * (size_t)V);
  double* x = (double*)malloc(sizeof(double) * (size_t)V);
  if (!p || !r || !x) {
    free(p);
    free(r);
    free(x);
    return ORC_ERR_NOMEM;
  }
  uint32_t st = 0;
  for (int b = b_begin; b < b_end; ++b) {
    const char* Xb = (const char*)target + (size_t)b * (size_t)(gamma + 1) * row_bytes;
    const int32_t* d = draft_tokens + (size_t)b * gamma;
    int32_t* out = out_tokens + (size_t)b * (gamma + 1);
    double mg = DBL_MAX, mgc = DBL_MAX, mgd = DBL_MAX;  /* accept tests, top-p cuts, the draw */
    if (!temperature_kind(temperature[b], &st)) {
      greedy_request(Xb, d, gamma, V, dtype, out, out_accept_len + b, &st);
      store_margins(b, mg, mgc, mgd, margin_accept, margin_cut, margin_draw);
      continue;
    }
    const double T = (double)temperature[b];
    for (int i = 0; i <= gamma; ++i) {
      for (int j = 0; j < V; ++j) x[j] = logit_at(Xb + (size_t)i * row_bytes, dtype, (size_t)j);
      if (row_is_bad(x, V)) st |= ORC_STATUS_BAD_ROW;
    }
    for (int i = 0; i < gamma; ++i)
      if (d[i] < 0 || d[i] >= V) st |= ORC_STATUS_BAD_TOKEN;
    for (int t = 0; t <= gamma; ++t) out[t] = -1;
    int n = 0, rejected = 0;
    int32_t last = -1;
    for (int i = 0; i < gamma; ++i) {
      if (filter_dense(Xb + (size_t)i * row_bytes, V, dtype, T, top_k, top_p, p, &mgc) < 0) {
        last = oracle_argmax_row(Xb + (size_t)i * row_bytes, V, dtype, NULL);
        rejected = 1;
        break;
      }
      const int32_t tok = d[i];
      const double p_d = (tok >= 0 && tok < V) ? p[tok] : 0.0;
      float u_acc, u_draw;
      oracle_uniforms(seed, (uint32_t)b, (uint32_t)i, 0u, &u_acc, &u_draw);
      update_margin(&mg, (double)u_acc, p_d);
      if (u_acc < (float)p_d) { /* q(d) = 1: the ratio is p(d) */
        out[n++] = tok;
        continue;
      }
      double Zr = 0.0;
      for (int j = 0; j < V; ++j) {
        r[j] = j == tok ? 0.0 : p[j];
        Zr += r[j];
      }
      /* after a rejection p(d) < 1, so Zr = 1 - p(d) > 0; p is only a guard */
      const double* w = Zr > 0.0 ? r : p;
      last = draw_ascending(w, V, u_draw, &mgd);
      rejected = 1;
      break;
    }
    if (!rejected) {
      if (filter_dense(Xb + (size_t)gamma * row_bytes, V, dtype, T, top_k, top_p, p, &mgc) < 0) {
        last = oracle_argmax_row(Xb + (size_t)gamma * row_bytes, V, dtype, NULL);
      } else {
        float u_draw;
        oracle_uniforms(seed, (uint32_t)b, (uint32_t)gamma, 0u, NULL, &u_draw);
        last = draw_ascending(p, V, u_draw, &mgd);
      }
    }
    out[n] = last;
    out_accept_len[b] = n + 1;
    store_margins(b, mg, mgc, mgd, margin_accept, margin_cut, margin_draw);
  }
  free(p);
  free(r);
  free(x);
  if (status) *status |= st;
  return ORC_OK;
}

int oracle_verify(const void* target, const void* draft, const int32_t* draft_tokens, int B,
                  int gamma, int V, int dtype, const float* temperature, int top_k, float top_p,
                  uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len, double* margin,
                  uint32_t* status, int b_begin, int b_end) {
  if (!margin)
    return oracle_verify_margins(target, draft, draft_tokens, B, gamma, V, dtype, temperature,
                                 top_k, top_p, seed, out_tokens, out_accept_len, NULL, NULL, NULL,
                                 status, b_begin, b_end);
  if (b_begin < 0) b_begin = 0;
  if (b_end > B) b_end = B;
  const int n = b_end > b_begin ? b_end - b_begin : 0;
  double* md = (double*)malloc(sizeof(double) * (size_t)(B > 0 ? B : 1));
  if (!md) return ORC_ERR_NOMEM;
  int rc = oracle_verify_margins(target, draft, draft_tokens, B, gamma, V, dtype, temperature,
                                 top_k, top_p, seed, out_tokens, out_accept_len, margin, md, NULL,
                                 status, b_begin, b_end);
  for (int i = 0; i < n && rc == ORC_OK; ++i)
    if (md[b_begin + i] < margin[b_begin + i]) margin[b_begin + i] = md[b_begin + i];
  free(md);
  return rc;
}

int oracle_sample_rows(const void* logits, int R, int V, int dtype, const float* temperature,
                       int top_k, float top_p, uint64_t seed, int32_t* out_tokens,
                       double* margin, uint32_t* status, int r_begin, int r_end) {
  if (!logits || !temperature || !out_tokens || R < 0 || V < 1 || !(top_p > 0.0f))
    return ORC_ERR_INVALID_ARG;
  if (r_begin < 0) r_begin = 0;
  if (r_end > R) r_end = R;
  const size_t row_bytes = (size_t)V * elem_size(dtype);
  double* p = (double*)malloc(sizeof(double) * (size_t)V);
  if (!p) return ORC_ERR_NOMEM;
  uint32_t st = 0;
  for (int r = r_begin; r < r_end; ++r) {
    const char* row = (const char*)logits + (size_t)r * row_bytes;
    double mg = DBL_MAX;
    if (!temperature_kind(temperature[r], &st)) {
      out_tokens[r] = oracle_argmax_row(row, V, dtype, &st);
    } else {
      int n = filter_dense(row, V, dtype, (double)temperature[r], top_k, top_p, p, &mg);
      if (n < 0) {
        st |= ORC_STATUS_BAD_ROW;
        out_tokens[r] = oracle_argmax_row(row, V, dtype, NULL);
      } else {
        float u;
        oracle_uniforms(seed, 0u, (uint32_t)r, 1u, &u, NULL);
        out_tokens[r] = draw_ascending(p, V, u, &mg);
      }
    }
    if (margin) margin[r] = mg;
  }
  free(p);
  if (status) *status |= st;
  return ORC_OK;
}
