// dflash_fullvocab.cu -- second pass of the full-vocabulary mode (top-k off,
// top-p 1): the residual or bonus draw over the whole vocabulary.
//
// With no top-k the filtered distributions are the plain softmax
// p_j = exp(x_j/T - max/T) / S over all V tokens, so the residual
// max(0, p - q) at the first rejected position spans the vocabulary too (the
// accept rule min(1, p/q), the residual and the bonus token of standard
// speculative sampling; "DFlash2 用投机解码给 Qwen 提速", bml.asia, the
// draft/verify loop, and "无损加速是真的吗？Qwen3.8-27B-DFlash2 如何保证输出与
// 目标模型完全一致", rytg.cn, section 投机解码如何白嫖速度, step 3). The first
// pass (the stream in dflash_sweep.cu) ran the accept tests and left, per
// request, the accepted count n and the row maxima; this pass draws the token
// at position n by the inverse CDF in ascending token order.
//
// Precision. At V = 248320 a token holds a few parts per million of the mass,
// so the draw compares a cumulative sum with u * total to far better than
// fp32 resolution: every weight here is a float-float pair (about 44 bits),
// and exp() is Tang's table-driven method ("Table-driven implementation of
// the exponential function in IEEE floating-point arithmetic", ACM TOMS 15(2),
// 1989) evaluated in float-float: exp(a) = 2^m * 2^(j/64) * exp(r) with
// N = 64 m + j = round(a * 64/ln2), |r| <= ln2/128 and exp(r) - 1 by its
// Taylor series to r^4, relative error about 1e-9. The decision itself is
// taken in fp32 like every other decision of the step: the smallest token
// whose cumulative weight, rounded to fp32, exceeds u * total rounded to fp32.
// All arithmetic uses explicitly rounded intrinsics, so the per-token weights
// are bit-identical wherever they are recomputed.
//
// Two launches, no waits between CTAs:
//  1. fv_sums: per (slice, request), the slice's sums of the exp weights of
//              the target and draft rows (-> the normalisers S_x, S_y), the
//              same sums over the tokens with p > q (-> the residual's slice
//              sums), and the slice's last token with weight.
//  2. fv_pick: per request, the slice where the cumulative weight crosses
//              u * total, then a block scan inside that slice.

#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "dflash_device.cuh"
#include "dflash_ff.cuh"
#include "dflash_internal.h"

namespace dflash {
namespace {

__device__ __forceinline__ float fv_load(const unsigned char* row, int j, int dtype) {
  if (dtype == 0) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + j);
    return __uint_as_float((uint32_t)h << 16);
  }
  return __ldg(reinterpret_cast<const float*>(row) + j);
}

// ---- per-request context -------------------------------------------------------------
struct Req {
  bool live;
  bool residual;
  int n;
  const unsigned char* x;  // target row n
  const unsigned char* y;  // draft row n (residual)
  ff inv_t;                // 1 / T
  ff zmx, zmy;             // row maxima / T
  float sx0, sy0;          // the stream's fp32 normalisers (residual: which side of p = q)
  int excl;                // token with no weight in this draw (-1: none)
  bool cut;                // top-p over the full vocabulary: only the kept sets weigh
  uint32_t kx, ky;         // ... the key of each row's last kept token
  int jx, jy;              // ... and the last kept index among that key's tokens
};

// whether token j (logit x) is in a row's kept set: every key above kappa,
// and key kappa's tokens up to index j_cut
__device__ __forceinline__ bool in_kept(bool cut, uint32_t kappa, int j_cut, float x, int j) {
  if (!cut) return true;
  const uint32_t k = key_of(x);
  return k > kappa || (k == kappa && j <= j_cut);
}

__device__ __forceinline__ Req load_req(const FvParams& f, int b) {
  Req q;
  q.live = false;
  if (*reinterpret_cast<const volatile uint32_t*>(f.abort_flag) != 0u) return q;
  const FvDraw d = f.draw[b];
  // a request drawn by the first pass has 0 <= n <= gamma; a residual needs n < gamma
  if (d.mode != kFvResidual && d.mode != kFvBonus) return q;
  if (d.n < 0 || d.n > f.gamma || (d.mode == kFvResidual && d.n >= f.gamma)) return q;
  const float T = __ldg(f.temperature + b);
  if (!(T > 0.0f) || !(T < INFINITY)) return q;
  q.live = true;
  q.residual = d.mode == kFvResidual;
  q.n = d.n;
  const size_t row_bytes = (size_t)f.V * (f.dtype == 0 ? 2 : 4);
  q.x = f.target + ((size_t)b * (f.gamma + 1) + d.n) * row_bytes;
  q.y = q.residual ? f.draft + ((size_t)b * f.gamma + d.n) * row_bytes : nullptr;
  const float r = __frcp_rn(T);
  q.inv_t = fast_two_sum(r, __fmul_rn(__fmaf_rn(-T, r, 1.0f), r));
  q.zmx = ff_scale(d.mx, q.inv_t);
  q.zmy = ff_scale(d.my, q.inv_t);
  q.sx0 = d.sx0;
  q.sy0 = d.sy0;
  q.excl = d.mode == kFvBonus ? d.excl : -1;
  q.cut = f.cut != nullptr;
  if (q.cut) {
    const FvtpDrawCut c = f.cut[b];
    q.kx = c.kappa_x;
    q.ky = c.kappa_y;
    q.jx = c.jcut_x;
    q.jy = c.jcut_y;
  } else {
    q.kx = q.ky = 0u;
    q.jx = q.jy = 0;
  }
  return q;
}

// unnormalised weight exp(x/T - max/T) of logit x
__device__ __forceinline__ ff weight(float x, ff inv_t, ff zmax, const float* th, const float* tl) {
  const ff z = ff_scale(x, inv_t);
  const ff s = two_sum(z.hi, -zmax.hi);
  const ff a = {s.hi, __fadd_rn(s.lo, __fsub_rn(z.lo, zmax.lo))};
  return exp_ff(a, th, tl);
}

// running sum of non-negative pairs: the low parts gather the rounding errors
// and the pair is renormalised once at the end (acc_done)
__device__ __forceinline__ void acc_add(ff& acc, ff w) {
  const ff s = two_sum(acc.hi, w.hi);
  acc.hi = s.hi;
  acc.lo = __fadd_rn(acc.lo, __fadd_rn(s.lo, w.lo));
}
__device__ __forceinline__ ff acc_done(ff acc) { return fast_two_sum(acc.hi, acc.lo); }

struct Norm {
  ff inv_sx, inv_sy;
};

// 1/S_x and 1/S_y of request b from the slice sums, summed in a fixed order
// (the same wherever they are needed). Run by warp 0; lane 0 writes *out.
__device__ __forceinline__ void load_norm(const FvParams& f, int b, bool residual, Norm* out) {
  const int lane = threadIdx.x & 31;
  ff sx = {0.0f, 0.0f}, sy = {0.0f, 0.0f};
  const float4* part = f.part + (size_t)b * f.n_slices;
  for (int s = lane; s < f.n_slices; s += 32) {
    const float4 v = part[s];
    sx = ff_add(sx, ff{v.x, v.y});
    sy = ff_add(sy, ff{v.z, v.w});
  }
  sx = warp_sum_ff(sx);
  sy = warp_sum_ff(sy);
  if (lane == 0) {
    out->inv_sx = ff_recip(sx);
    out->inv_sy = residual ? ff_recip(sy) : ff{0.0f, 0.0f};
  }
}

// block sum (kFvThreads threads) in a fixed order; valid in thread 0
__device__ __forceinline__ ff block_sum_ff(ff a, ff* scratch) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  a = warp_sum_ff(a);
  if (lane == 0) scratch[w] = a;
  __syncthreads();
  ff t = {0.0f, 0.0f};
  if (threadIdx.x == 0)
    for (int i = 0; i < kFvThreads / 32; ++i) t = ff_add(t, scratch[i]);
  __syncthreads();
  return t;
}

__device__ __forceinline__ void load_table(const FvParams& f, float* th, float* tl) {
  for (int i = threadIdx.x; i < kExpTable; i += blockDim.x) {
    th[i] = f.exp_hi[i];
    tl[i] = f.exp_lo[i];
  }
}

// exclusive warp scan of a pair (fixed order)
__device__ __forceinline__ ff warp_exclusive_ff(ff v, ff& inclusive) {
  const int lane = threadIdx.x & 31;
  ff incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const ff n = shfl_up_ff(incl, o);
    if (lane >= o) incl = ff_add(n, incl);
  }
  inclusive = incl;
  ff ex = shfl_up_ff(incl, 1);
  if (lane == 0) ex = {0.0f, 0.0f};
  return ex;
}

// ---- launch 1: slice sums --------------------------------------------------------------
// Per (slice, request): S_x and S_y over the slice, and for a residual the
// same sums over the tokens with p > q, A = sum w_x and B = sum w_y. The
// residual's slice sum is then A / S_x - B / S_y with the exact normalisers,
// known only after every slice is summed. Which side of p = q a token is on
// comes from the stream's fp32 normalisers (w_x S_y0 > w_y S_x0); a token
// they place wrongly has |p - q| below about 1e-6 p and carries under 1e-11 of
// the mass.
template <int DT, bool kCut>
__global__ void __launch_bounds__(kFvThreads) fv_sums_kernel(const FvParams f) {
  __shared__ float th[kExpTable], tl[kExpTable];
  __shared__ ff scratch[kFvThreads / 32];
  __shared__ int last_r, last_p;
  const int s = blockIdx.x, b = blockIdx.y;
  grid_dependency_sync();
  const Req q = load_req(f, b);
  // one decision for the block: the abort flag can be raised while it runs
  if (!__syncthreads_and(q.live)) return;
  load_table(f, th, tl);
  if (threadIdx.x == 0) {
    last_r = -1;
    last_p = -1;
  }
  __syncthreads();
  ff sx = {0.0f, 0.0f}, sy = {0.0f, 0.0f}, ax = {0.0f, 0.0f}, by = {0.0f, 0.0f};
  int lr = -1, lp = -1;
  const int j0 = s * kFvSlice + threadIdx.x;
  const int jn = min(f.V, (s + 1) * kFvSlice);
  float xs[kFvPerThread], ys[kFvPerThread];
#pragma unroll
  for (int k = 0; k < kFvPerThread; ++k) {
    const int j = j0 + k * kFvThreads;
    xs[k] = j < jn ? fv_load(q.x, j, DT) : -INFINITY;
    ys[k] = (q.residual && j < jn) ? fv_load(q.y, j, DT) : -INFINITY;
  }
  if (q.residual) {
#pragma unroll
    for (int k = 0; k < kFvPerThread; ++k) {
      const int j = j0 + k * kFvThreads;
      const ff wx = in_kept(kCut, q.kx, q.jx, xs[k], j) ? weight(xs[k], q.inv_t, q.zmx, th, tl) : ff{0.0f, 0.0f};
      const ff wy = in_kept(kCut, q.ky, q.jy, ys[k], j) ? weight(ys[k], q.inv_t, q.zmy, th, tl) : ff{0.0f, 0.0f};
      acc_add(sx, wx);
      acc_add(sy, wy);
      if (__fmul_rn(wx.hi, q.sy0) > __fmul_rn(wy.hi, q.sx0)) {
        acc_add(ax, wx);
        acc_add(by, wy);
        lr = j0 + k * kFvThreads;
      }
      if (wx.hi > 0.0f) lp = j0 + k * kFvThreads;
    }
  } else {
#pragma unroll
    for (int k = 0; k < kFvPerThread; ++k) {
      const int j = j0 + k * kFvThreads;
      ff wx = in_kept(kCut, q.kx, q.jx, xs[k], j) ? weight(xs[k], q.inv_t, q.zmx, th, tl) : ff{0.0f, 0.0f};
      if (j == q.excl) wx = {0.0f, 0.0f};  // p without the deterministic draft
      acc_add(sx, wx);
      if (wx.hi > 0.0f) lp = j0 + k * kFvThreads;
    }
  }
  if (lr >= 0) atomicMax(&last_r, lr);
  if (lp >= 0) atomicMax(&last_p, lp);
  sx = block_sum_ff(acc_done(sx), scratch);  // its barriers also order the atomics above
  sy = block_sum_ff(acc_done(sy), scratch);
  ax = block_sum_ff(acc_done(ax), scratch);
  by = block_sum_ff(acc_done(by), scratch);
  if (threadIdx.x == 0) {
    const size_t c = (size_t)b * f.n_slices + s;
    f.part[c] = make_float4(sx.hi, sx.lo, sy.hi, sy.lo);
    f.pos[c] = make_float4(ax.hi, ax.lo, by.hi, by.lo);
    f.last[c] = make_int2(last_r, last_p);
  }
}

// ---- launch 2: the draw -----------------------------------------------------------------
// p_j and r_j = max(0, p_j - q_j) of a token with target logit x and draft
// logit y (r = 0 for a bonus draw), normalised exactly
__device__ __forceinline__ void token_weights(const Req& q, const Norm& nm, float x, float y, int j, const float* th,
                                              const float* tl, ff& p, ff& r) {
  p = in_kept(q.cut, q.kx, q.jx, x, j) ? ff_mul(weight(x, q.inv_t, q.zmx, th, tl), nm.inv_sx) : ff{0.0f, 0.0f};
  r = {0.0f, 0.0f};
  if (q.residual) {
    const ff qq =
        in_kept(q.cut, q.ky, q.jy, y, j) ? ff_mul(weight(y, q.inv_t, q.zmy, th, tl), nm.inv_sy) : ff{0.0f, 0.0f};
    const ff d = ff_add(p, ff_neg(qq));
    if (d.hi > 0.0f) r = d;
  }
}

__global__ void __launch_bounds__(kFvThreads) fv_pick_kernel(const FvParams f) {
  __shared__ float th[kExpTable], tl[kExpTable];
  __shared__ Norm nm_s;
  __shared__ ff warp_tot[kFvThreads / 32];
  __shared__ int sel_slice, use_r, hit, last_any;
  __shared__ float target_f;
  __shared__ ff slice_base;
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  grid_dependency_sync();
  const Req q = load_req(f, b);
  // every call leaves the workspace at zero (its regions move with the
  // shape): this launch is the last reader of the request's draw state
  FvDraw* draw_w = const_cast<FvDraw*>(f.draw) + b;
  if (!__syncthreads_and(q.live)) {  // one decision for the block, as in fv_sums
    if (tid == 0 && *reinterpret_cast<const volatile uint32_t*>(f.abort_flag) == 0u) {
      *draw_w = FvDraw{};
      if (f.cut) f.cut[b] = FvtpDrawCut{};
    }
    return;
  }
  load_table(f, th, tl);
  if (tid < 32) load_norm(f, b, q.residual, &nm_s);
  __syncthreads();
  const Norm nm = nm_s;
  const size_t c0 = (size_t)b * f.n_slices;

  if (w == 0) {
    // slice sums of the residual (A/S_x - B/S_y, never below 0) and of p
    // (S_x slice / S_x); the draw uses the residual unless it is zero
    // everywhere (or this is the bonus draw)
    auto slice_r = [&](int s) {
      const float4 v = f.pos[c0 + s];
      const ff d = ff_add(ff_mul(ff{v.x, v.y}, nm.inv_sx), ff_neg(ff_mul(ff{v.z, v.w}, nm.inv_sy)));
      return d.hi > 0.0f ? d : ff{0.0f, 0.0f};
    };
    auto slice_p = [&](int s) {
      const float4 v = f.part[c0 + s];
      return ff_mul(ff{v.x, v.y}, nm.inv_sx);
    };
    ff zr = {0.0f, 0.0f}, zp = {0.0f, 0.0f};
    int lr = -1, lp = -1;
    for (int s = lane; s < f.n_slices; s += 32) {
      if (q.residual) zr = ff_add(zr, slice_r(s));
      zp = ff_add(zp, slice_p(s));
      const int2 l = f.last[c0 + s];
      lr = max(lr, l.x);
      lp = max(lp, l.y);
    }
    zr = warp_sum_ff(zr);
    zp = warp_sum_ff(zp);
    const bool resid = __shfl_sync(0xffffffffu, (int)(q.residual && zr.hi > 0.0f), 0) != 0;
    const ff z = resid ? zr : zp;
    lr = __reduce_max_sync(0xffffffffu, lr);
    lp = __reduce_max_sync(0xffffffffu, lp);
    // verification: word 1 of (position n, request b, stream 0); the sampler:
    // word 0 of (row, 0, stream 1), rows counted across the call's launches
    const float u = f.sampler ? uniform24(step_uniform_words(f.seed, 0u, (uint32_t)(f.row_base + b), 1u).x)
                              : uniform24(step_uniform_words(f.seed, (uint32_t)b, (uint32_t)q.n, 0u).y);
    const float tf = __shfl_sync(0xffffffffu, ff_round(ff_scale(u, z)), 0);
    // first slice whose cumulative weight (rounded to fp32) exceeds tf
    ff carry = {0.0f, 0.0f};
    int found = -1;
    ff found_base = {0.0f, 0.0f};
    for (int s0 = 0; s0 < f.n_slices && found < 0; s0 += 32) {
      const int s = s0 + lane;
      ff v = {0.0f, 0.0f};
      if (s < f.n_slices) v = resid ? slice_r(s) : slice_p(s);
      ff incl;  // scans over the 32 slices of this round
      const ff excl = ff_add(carry, warp_exclusive_ff(v, incl));
      const ff cum = ff_add(carry, incl);
      const uint32_t ball = __ballot_sync(0xffffffffu, s < f.n_slices && tf < ff_round(cum));
      if (ball) {
        const int l = __ffs(ball) - 1;
        found = s0 + l;  // the cumulative weight before it is lane l's excl
        found_base = {__shfl_sync(0xffffffffu, excl.hi, l), __shfl_sync(0xffffffffu, excl.lo, l)};
      }
      carry = {__shfl_sync(0xffffffffu, cum.hi, 31), __shfl_sync(0xffffffffu, cum.lo, 31)};
    }
    if (lane == 0) {
      sel_slice = found;
      use_r = resid ? 1 : 0;
      target_f = tf;
      slice_base = found_base;
      last_any = resid ? lr : lp;
      hit = INT_MAX;
    }
  }
  __syncthreads();
  const int s = sel_slice;
  int32_t* out = f.out_tokens + (size_t)b * (f.gamma + 1) + q.n;
  for (int c = tid; c < f.n_slices; c += kFvThreads) {  // the slice sums are used up
    f.part[c0 + c] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    f.pos[c0 + c] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
  }
  if (tid == 0) {
    *draw_w = FvDraw{};
    if (f.cut) f.cut[b] = FvtpDrawCut{};
  }
  if (s < 0) {  // rounding left no token above u * total: the last with weight
    if (tid == 0) *out = last_any >= 0 ? last_any : 0;
    for (int c = tid; c < f.n_slices; c += kFvThreads) f.last[c0 + c] = make_int2(0, 0);
    return;
  }
  // inside slice s: thread t owns tokens s*kFvSlice + t*kFvPerThread + k, in order
  const bool resid = use_r != 0;
  const int jb = s * kFvSlice + tid * kFvPerThread;
  float xs[kFvPerThread], ys[kFvPerThread];
#pragma unroll
  for (int k = 0; k < kFvPerThread; ++k) {
    const int j = jb + k;
    xs[k] = j < f.V ? fv_load(q.x, j, f.dtype) : -INFINITY;
    ys[k] = (q.residual && j < f.V) ? fv_load(q.y, j, f.dtype) : -INFINITY;
  }
  ff wk[kFvPerThread];
  ff mine = {0.0f, 0.0f};
#pragma unroll
  for (int k = 0; k < kFvPerThread; ++k) {
    ff p, r;
    token_weights(q, nm, xs[k], ys[k], jb + k, th, tl, p, r);
    if (jb + k == q.excl) p = {0.0f, 0.0f};
    wk[k] = resid ? r : p;
    mine = ff_add(mine, wk[k]);
  }
  // exclusive block scan of the threads' sums
  ff incl;
  const ff ex = warp_exclusive_ff(mine, incl);
  if (lane == 31) warp_tot[w] = incl;
  __syncthreads();
  ff cum = slice_base;
  for (int i = 0; i < w; ++i) cum = ff_add(cum, warp_tot[i]);
  cum = ff_add(cum, ex);
  const float tf = target_f;
  int first = INT_MAX;
#pragma unroll
  for (int k = 0; k < kFvPerThread; ++k) {
    cum = ff_add(cum, wk[k]);
    if (first == INT_MAX && wk[k].hi > 0.0f && tf < ff_round(cum)) first = jb + k;
  }
  if (first != INT_MAX) atomicMin(&hit, first);
  __syncthreads();
  if (tid == 0) {
    int j = hit;
    if (j == INT_MAX) {
      // the slice sums put the crossing here but the in-slice order rounded
      // past it: the slice's last token with weight
      const int2 l = f.last[c0 + s];
      j = resid ? l.x : l.y;
      if (j < 0) j = last_any >= 0 ? last_any : 0;
    }
    *out = j;
  }
  __syncthreads();
  for (int c = tid; c < f.n_slices; c += kFvThreads) f.last[c0 + c] = make_int2(0, 0);
}

}  // namespace

int launch_fullvocab_draw(const FvParams& f, void* stream) {
  if (f.B <= 0 || f.n_slices <= 0) return 0;
  // both launches may start while the kernel before them ends (programmatic
  // dependent launch); each waits for it before its first global access
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kFvThreads);
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cfg.gridDim = dim3((unsigned)f.n_slices, (unsigned)f.B);
  // the storage type and whether a top-p cut masks the weights are the
  // launch's: one instantiation each, no per-logit test of either
  void (*sums)(const FvParams) = f.dtype == 0 ? (f.cut ? fv_sums_kernel<0, true> : fv_sums_kernel<0, false>)
                                              : (f.cut ? fv_sums_kernel<1, true> : fv_sums_kernel<1, false>);
  cudaError_t e = cudaLaunchKernelEx(&cfg, sums, f);
  if (e != cudaSuccess) return (int)e;
  cfg.gridDim = dim3((unsigned)f.B);
  e = cudaLaunchKernelEx(&cfg, fv_pick_kernel, f);
  return (int)e;
}

}  // namespace dflash
