// dflash_ff.cuh -- float-float arithmetic (pairs hi + lo of fp32 values,
// about 44 significant bits) for the decisions of the verification step that
// must be taken on nearly exact sums: the filtered probabilities of a row's
// kept tokens, the top-p cut, the inverse CDF of a draw, and the
// full-vocabulary draw. Error-free transformations after Knuth (two-sum) and
// Dekker (fast two-sum, products through fma), and exp() by Tang's
// table-driven method ("Table-driven implementation of the exponential
// function in IEEE floating-point arithmetic", ACM TOMS 15(2), 1989)
// evaluated in float-float: exp(a) = 2^m * 2^(j/64) * exp(r) with
// N = 64 m + j = round(a * 64/ln2), |r| <= ln2/128, and exp(r) - 1 by its
// Taylor series to r^4 (relative error about 1e-9). Every operation is an
// explicitly rounded intrinsic, so a weight recomputed anywhere is
// bit-identical.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "dflash_internal.h"

namespace dflash {

// ---- float-float arithmetic (Dekker / Knuth error-free transformations) --------------
struct ff {
  float hi, lo;
};

__device__ __forceinline__ ff two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}
// requires |a| >= |b| (or a == 0)
__device__ __forceinline__ ff fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
  const ff s = two_sum(a.hi, b.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ ff ff_neg(ff a) { return {-a.hi, -a.lo}; }
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
  const float p = __fmul_rn(a.hi, b.hi);
  float e = __fmaf_rn(a.hi, b.hi, -p);
  e = __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, e));
  return fast_two_sum(p, e);
}
// x * b for a plain float x
__device__ __forceinline__ ff ff_scale(float x, ff b) {
  const float p = __fmul_rn(x, b.hi);
  const float e = __fmaf_rn(x, b.lo, __fmaf_rn(x, b.hi, -p));
  return {p, e};
}
// 1 / a; the remainder 1 - a.hi * RN(1/a.hi) is exact in fp32
__device__ __forceinline__ ff ff_recip(ff a) {
  const float r = __frcp_rn(a.hi);
  const float e = __fmaf_rn(-a.lo, r, __fmaf_rn(-a.hi, r, 1.0f));
  return fast_two_sum(r, __fmul_rn(e, r));
}
// the fp32 value nearest to hi + lo (one correctly rounded addition)
__device__ __forceinline__ float ff_round(ff a) { return __fadd_rn(a.hi, a.lo); }

__device__ __forceinline__ ff shfl_down_ff(ff a, int o) {
  return {__shfl_down_sync(0xffffffffu, a.hi, o), __shfl_down_sync(0xffffffffu, a.lo, o)};
}
__device__ __forceinline__ ff shfl_up_ff(ff a, int o) {
  return {__shfl_up_sync(0xffffffffu, a.hi, o), __shfl_up_sync(0xffffffffu, a.lo, o)};
}
// warp sum in a fixed tree; the result is valid in lane 0
__device__ __forceinline__ ff warp_sum_ff(ff a) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const ff b = shfl_down_ff(a, o);
    if ((threadIdx.x & 31) + o < 32) a = ff_add(a, b);
  }
  return a;
}

// ---- exp in float-float ------------------------------------------------------------
constexpr double kInvLn2x64 = 92.33248261689366;        // 64 / ln 2
constexpr double kLn2Div64 = 0.010830424696249145;      // ln 2 / 64
constexpr float kK_hi = (float)kInvLn2x64;
constexpr float kK_lo = (float)(kInvLn2x64 - (double)(float)kInvLn2x64);
constexpr float kL_hi = (float)kLn2Div64;
constexpr float kL_lo = (float)(kLn2Div64 - (double)(float)kLn2Div64);
constexpr float kRoundMagic = 12582912.0f;              // 1.5 * 2^23

// exp(a) for a <= 0 (a.hi >= -87: below that the weight is under 2^-125 of
// the row's largest and is taken as 0). th/tl: 2^(j/64) as fp32 pairs.
__device__ __forceinline__ ff exp_ff(ff a, const float* th, const float* tl) {
  if (!(a.hi >= -87.0f)) return {0.0f, 0.0f};
  // t = a * 64/ln2 as a pair; N = round(t) = 64 m + j
  const float t_hi = __fmul_rn(a.hi, kK_hi);
  float t_lo = __fmaf_rn(a.hi, kK_hi, -t_hi);
  t_lo = __fmaf_rn(a.hi, kK_lo, __fmaf_rn(a.lo, kK_hi, t_lo));
  const float v = __fadd_rn(t_hi, kRoundMagic);  // |t_hi| < 2^22: v's last bit is N's
  const int N = __float_as_int(v) - __float_as_int(kRoundMagic);
  const float Nf = __fsub_rn(v, kRoundMagic);
  const float g = __fadd_rn(__fsub_rn(t_hi, Nf), t_lo);  // t - N, |g| <= 1/2; t_hi - Nf is exact
  const float r = __fmaf_rn(g, kL_hi, __fmul_rn(g, kL_lo));  // r = g * ln2/64
  // exp(r) - 1 = r + r^2 (1/2 + r (1/6 + r/24)) + O(r^5), |r| <= 0.0055
  const float c4 = __fmaf_rn(r, 1.0f / 24.0f, 1.0f / 6.0f);
  const float c2 = __fmaf_rn(r, c4, 0.5f);
  const float P = __fmaf_rn(__fmul_rn(r, r), c2, r);
  const int j = N & (kExpTable - 1), m = N >> 6;
  const float Th = th[j], Tl = tl[j];
  const ff w = fast_two_sum(Th, __fmaf_rn(Th, P, Tl));  // 2^(j/64) (1 + P)
  const float sc = __int_as_float((m + 127) << 23);      // 2^m, m >= -126
  return {__fmul_rn(w.hi, sc), __fmul_rn(w.lo, sc)};
}


// (a_hi + a_lo) / T as a pair: the rounded quotient of a_hi, the exact
// remainder of that division plus a_lo, divided by T (the low part's own
// rounding is below 2^-48 of the quotient)
__device__ __forceinline__ ff quot_ff(float a_hi, float a_lo, float T) {
  const float q = __fdiv_rn(a_hi, T);
  const float rem = __fmaf_rn(-q, T, a_hi);
  return fast_two_sum(q, __fdiv_rn(__fadd_rn(rem, a_lo), T));
}
// exp((x - m) / T) for x <= m, as a pair (0 for x = -inf)
__device__ __forceinline__ ff exp_diff_ff(float x, float m, float T, const float* th, const float* tl) {
  const ff d = two_sum(x, -m);
  return exp_ff(quot_ff(d.hi, d.lo, T), th, tl);
}

// warp-wide inclusive prefix sum of pairs over lanes (five shuffle steps)
__device__ __forceinline__ ff warp_inclusive_scan_ff(ff a, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff b = shfl_up_ff(a, o);
    if (lane >= o) a = ff_add(a, b);
  }
  return a;
}
__device__ __forceinline__ ff shfl_ff(ff a, int src) {
  return {__shfl_sync(0xffffffffu, a.hi, src), __shfl_sync(0xffffffffu, a.lo, src)};
}

}  // namespace dflash
