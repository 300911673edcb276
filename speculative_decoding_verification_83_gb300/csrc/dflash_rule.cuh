// dflash_rule.cuh -- the verification rule on filtered rows, shared by the
// stream kernel's finals (dflash_sweep.cu) and the verification from
// vocabulary-shard candidates (dflash_candidates.cu): the row filter
// (temperature, softmax over the top k, top-p, renormalisation), the inverse
// CDF in ascending token order, and the accept test and draw of a sampling
// request.
//
// The rule is standard speculative sampling as "DFlash2 用投机解码给 Qwen 提速"
// (bml.asia, the draft/verify loop) and "无损加速是真的吗？Qwen3.8-27B-DFlash2
// 如何保证输出与目标模型完全一致" (rytg.cn, section 投机解码如何白嫖速度, step 3)
// describe it: accept d with probability min(1, p(d)/q(d)), at the first
// rejection draw from the normalised max(0, p - q), else the bonus token
// from the last target row.
#pragma once

#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "dflash_device.cuh"
#include "dflash_ff.cuh"
#include "dflash_internal.h"

namespace dflash {

constexpr uint32_t kStatusBadToken = 1u, kStatusBadRow = 2u, kStatusTimeout = 4u,
                   kStatusBadTemperature = 8u;

__device__ __forceinline__ bool sampling_temperature(float t) { return t > 0.0f && t < INFINITY; }

// ---- filtering and drawing ---------------------------------------------------------
// Every decision here turns sums of probabilities into an integer (the top-p
// cut, the accept test, the inverse CDF), and is taken in fp32 on the fp32
// rounding of nearly exact quantities: the weights and prefix sums are
// float-float (dflash_ff.cuh), so the only error a decision sees is the
// final rounding of its operands. Sorts place each element by its rank
// (independent loads from a small shared scratch) rather than through a
// sorting network; sums and prefix sums over a warp are five shuffle steps.

// Filters one row's sorted top-k (lane j holds rank j): temperature, softmax
// over the survivors, top-p cut, renormalisation. Returns this lane's
// probability (0 outside the kept set) and sets idx to -1 there.
// The weight of rank j is exp((x_j - x_0) / T): the difference to the
// largest logit is exact as a pair, its quotient by T a pair (the rounded
// quotient and the exact remainder over T), and exp() float-float (th, tl:
// Tang's table). The mass before rank j is its exclusive prefix over the
// total, rounded to fp32 for the cut (kept while below top_p, so the kept
// ranks are a prefix that always holds rank 0); a kept probability is its
// weight over the kept total, rounded once to fp32.
__device__ __forceinline__ float filter_lane(uint32_t key, int32_t& idx, int k_eff, float T, float top_p,
                                             int lane, const float* th, const float* tl) {
  const bool in_k = lane < k_eff && idx >= 0;
  const float x = value_of_key(key);
  const float x0 = __shfl_sync(0xffffffffu, x, 0);  // the largest
  const ff delta = two_sum(x, -x0);                 // x - x0, exactly
  const float q_hi = __fdiv_rn(delta.hi, T);
  const float rem = __fmaf_rn(-q_hi, T, delta.hi);  // delta.hi - q_hi T, exactly
  const ff d = fast_two_sum(q_hi, __fdiv_rn(__fadd_rn(rem, delta.lo), T));
  const ff w = in_k ? exp_ff(d, th, tl) : ff{0.0f, 0.0f};
  const ff incl = warp_inclusive_scan_ff(w, lane);
  bool keep = in_k;
  if (top_p < 1.0f) {
    // every lane takes part in both shuffles (none may sit in a
    // short-circuited operand: a lane skipping a full-mask shuffle leaves
    // the others waiting for it)
    const ff total = shfl_ff(incl, 31);
    ff before = shfl_up_ff(incl, 1);  // mass of the higher ranks
    if (lane == 0) before = ff{0.0f, 0.0f};
    const float before_f = ff_round(ff_mul(before, ff_recip(total)));
    keep = keep && before_f < top_p;
  }
  const uint32_t kept = __ballot_sync(0xffffffffu, keep);
  const ff Wk = shfl_ff(incl, kept ? 31 - __clz(kept) : 0);  // the kept total
  if (!keep) idx = -1;
  return keep ? ff_round(ff_mul(w, ff_recip(Wk))) : 0.0f;
}

// Inverse CDF in ascending token order: the smallest token whose cumulative
// weight exceeds u * total; if rounding leaves none, the last token with
// positive weight; tokens marked -1 have no weight. The lanes are put in
// token order by rank (ties, only among the -1 marks, by lane); the
// cumulative weights and the total are float-float prefix sums, and the
// comparison is taken on the fp32 roundings of the cumulative weight and of
// u * total. sk, sw: 32 words each of warp scratch, 16-byte aligned.
__device__ __forceinline__ int32_t draw_ascending(int32_t tok, float w, float u, int lane, int32_t* sk,
                                                  float* sw) {
  const int32_t key = tok >= 0 ? tok : INT_MAX;
  const float wt = tok >= 0 ? w : 0.0f;
  sk[lane] = key;
  __syncwarp();
  int r = 0;
  const int4* k4 = reinterpret_cast<const int4*>(sk);
#pragma unroll 1
  for (int q = 0; q < 8; ++q) {
    const int4 v = k4[q];
    const int32_t e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) r += (e[i] < key || (e[i] == key && 4 * q + i < lane)) ? 1 : 0;
  }
  __syncwarp();
  sk[r] = key;
  sw[r] = wt;
  __syncwarp();
  // lane l now stands for rank l
  const float wl = sw[lane];
  const ff cum = warp_inclusive_scan_ff(ff{wl, 0.0f}, lane);
  const float t = ff_round(ff_scale(u, shfl_ff(cum, 31)));
  const uint32_t hit = __ballot_sync(0xffffffffu, wl > 0.0f && t < ff_round(cum));
  int chosen;
  if (hit) {
    chosen = __ffs(hit) - 1;
  } else {
    const uint32_t pos = __ballot_sync(0xffffffffu, wl > 0.0f);
    chosen = pos ? 31 - __clz(pos) : 0;
  }
  const int32_t res = sk[chosen];
  __syncwarp();
  return res == INT_MAX ? -1 : res;
}

// Home slot of a token in a 64-slot table (Fibonacci hashing).
__device__ __forceinline__ uint32_t token_slot(int32_t t) { return ((uint32_t)t * 2654435761u) >> 26; }
static_assert(2 * kMaxTopK == 64, "token_slot hashes into 64 slots");

// ---- the accept test and the draw of one sampling request (one warp) ----------------
// idx / prob: the request's rows' filtered lists, rows padded to 33 words:
// lane j of row r is the rank-j kept token (-1 past the kept set) and its
// probability; column 32 holds the probability the row gives its position's
// draft token (prob) and the row's bad flag (idx). Rows go target 0, draft 0,
// target 1, ..., target gamma, or with deterministic drafts (det: q is the
// point mass at each draft) the gamma + 1 target rows alone. d_lane: lane i's
// draft token (i < gamma); wd: lane i's counter-based words for position i
// (accept: x, draw: y). scratch: 64 words of warp scratch, 16-byte aligned.
// Writes out[0..gamma] (the request's tokens), out_len[b] (its accept length)
// and ORs its status bits into *status; audit_pq (optional, [gamma][2])
// receives each position's p(d) and q(d) as the accept test used them.
__device__ __forceinline__ void sampling_rule(const int32_t (*idx)[33], const float (*prob)[33], int per_s,
                                              bool det, int gamma, int V, int32_t d_lane, uint4 wd,
                                              unsigned long long seed, int b, int lane,
                                              unsigned long long* scratch, int32_t* out, int32_t* out_len,
                                              uint32_t* status, float* audit_pq = nullptr) {
  uint32_t st = 0;
  for (int r = lane; r < per_s; r += 32)
    if (idx[r][32]) st |= kStatusBadRow;
  bool reject = false;
  if (lane < gamma) {
    const int32_t di = d_lane;
    if (di < 0 || di >= V) st |= kStatusBadToken;
    // p(d) and q(d), found by the rows' finals (0 when the token is not kept)
    const float p_d = prob[det ? lane : 2 * lane][32];
    const float q_d = det ? 1.0f : prob[2 * lane + 1][32];
    const float ratio = p_d / q_d;  // q = 0: +inf if p > 0, NaN if p == 0
    reject = !(uniform24(wd.x) < ratio);
    if (audit_pq) {
      audit_pq[2 * lane] = p_d;
      audit_pq[2 * lane + 1] = q_d;
    }
  }
  const uint32_t rej = __ballot_sync(0xffffffffu, reject);
  const int n = rej ? __ffs(rej) - 1 : gamma;  // drafts accepted
  uint32_t u_draw = __shfl_sync(0xffffffffu, wd.y, n & 31);
  if (n >= 32) u_draw = step_uniform_words(seed, (uint32_t)b, (uint32_t)n, 0u).y;  // gamma = 32, all kept
  const int row = det ? n : 2 * n;  // target row of position n (the bonus row when n == gamma)
  const int32_t ti = idx[row][lane];
  const float pi = prob[row][lane];
  float wt = pi;
  if (n < gamma && det) {
    // residual p - delta_d: the target's kept tokens other than the draft
    const int32_t dn = __shfl_sync(0xffffffffu, d_lane, n);
    const float r = (ti >= 0 && ti != dn) ? pi : 0.0f;
    if (__ballot_sync(0xffffffffu, r > 0.0f) != 0u) wt = r;
  } else if (n < gamma) {
    // residual max(0, p - q) over the target's kept tokens: q from the
    // draft row's list through a 64-slot open-addressing table in the
    // scratch (keys, then values)
    int32_t* hk = reinterpret_cast<int32_t*>(scratch);
    float* hv = reinterpret_cast<float*>(scratch) + 2 * kMaxTopK;
    hk[lane] = -1;
    hk[lane + kMaxTopK] = -1;
    __syncwarp();
    const int32_t dt = idx[row + 1][lane];
    if (dt >= 0) {
      uint32_t h = token_slot(dt);
      for (int probe = 0; probe < 2 * kMaxTopK; ++probe, h = (h + 1u) & (2 * kMaxTopK - 1)) {
        if (atomicCAS(&hk[h], -1, dt) == -1) {
          hv[h] = prob[row + 1][lane];
          break;
        }
      }
    }
    __syncwarp();
    float q_of_t = 0.0f;
    if (ti >= 0) {
      uint32_t h = token_slot(ti);
      for (int probe = 0; probe < 2 * kMaxTopK; ++probe, h = (h + 1u) & (2 * kMaxTopK - 1)) {
        const int32_t key = hk[h];
        if (key == ti) {
          q_of_t = hv[h];
          break;
        }
        if (key == -1) break;
      }
    }
    __syncwarp();  // the table's slots are the draw's scratch next
    const float r = ti >= 0 ? fmaxf(pi - q_of_t, 0.0f) : 0.0f;
    if (__ballot_sync(0xffffffffu, r > 0.0f) != 0u) wt = r;
  }
  int32_t last = draw_ascending(ti, wt, uniform24(u_draw), lane, reinterpret_cast<int32_t*>(scratch),
                                reinterpret_cast<float*>(scratch) + 32);
  if (last < 0) last = __shfl_sync(0xffffffffu, ti, 0);
  // gamma <= 32: a position i < n is this lane's own (i == lane)
  for (int i = lane; i <= gamma; i += 32) out[i] = i < n ? d_lane : (i == n ? last : -1);
  st = __reduce_or_sync(0xffffffffu, st);
  if (lane == 0) {
    if (out_len) out_len[b] = n + 1;
    if (st && status) atomicOr(status, st);
  }
}

}  // namespace dflash
