// dflash_fvtp.cu -- top-p over the whole vocabulary (top-k off, 0 < top_p < 1):
// the cut of every sampling row, then the accept tests.
//
// With no top-k, the top-p filter keeps the shortest prefix of a row's order
// (logit descending, token index ascending) whose softmax mass reaches
// top_p: token j is kept while the mass of the tokens before it is below
// top_p, and the kept probabilities are renormalised. This is the filter
// setting of "DFlash2 用投机解码给 Qwen 提速" (bml.asia, the model-card
// paragraph: temperature 1.0, top-p 0.95, top-k 20) with its top-k switched
// off; the accept rule, residual and bonus token are those of the draft/verify
// loop there and of step 3 of rytg.cn's section 投机解码如何白嫖速度.
//
// At V = 248320 the kept set holds a large share of the vocabulary, so no
// sort of candidates finds it. Instead the cut is found by radix selection on
// the order keys, weighted by mass:
//  * every weight is exp((x - m) / T) in float-float (Tang's method,
//    dflash_ff.cuh; m the row's largest logit from the stream), rounded to
//    fixed point with frac_bits fractional bits: the sums below are then
//    exact integers, identical wherever they are taken;
//  * round k (8 bits of the key at a time, from the top: two rounds for bf16
//    keys, four for fp32) builds, per row, the mass and count histogram of
//    the next key byte over the tokens whose key matches the bits found so
//    far (one CTA per 4096-token slice, shared-memory histograms per warp,
//    then global 64-bit atomics);
//  * the select step scans that histogram from the top: the key group
//    holding the last kept token is the lowest non-empty bin whose mass above
//    it, over the row's total, rounds (fp32) below top_p;
//  * after the last round the key kappa of the last kept token is known,
//    with the mass of the keys above it, and how many of the tokens with key
//    kappa are kept (they all weigh the same: the largest t with
//    RN32((above + t w_kappa) / total) < top_p); when only some are kept, a
//    count per slice and a scan of one slice give the index j_cut of the last
//    kept one.
// The accept test at position i takes p(d) = w(d) / (kept mass) (0 when d is
// not kept) from the target row, and q(d) likewise from the draft row (1 for
// a deterministic draft), and leaves the draw descriptors for the second pass
// (dflash_fullvocab.cu), which draws over the kept sets.

#include <cuda_runtime.h>

#include <climits>
#include <cstdint>

#include "dflash_device.cuh"
#include "dflash_ff.cuh"
#include "dflash_internal.h"
#include "dflash_rule.cuh"

namespace dflash {
namespace {

constexpr int kTpThreads = 256;
constexpr int kTpWarps = kTpThreads / 32;
static_assert(kFvSlice % kTpThreads == 0, "a slice is whole rounds of the block");

struct RowRef {
  int b;                     // request
  const unsigned char* ptr;  // the row's logits
  bool live;                 // a sampling request's row that the stream found usable
  float m;                   // the row's largest logit
  float T;
};

__device__ __forceinline__ RowRef row_ref(const FvtpParams& t, int rho) {
  RowRef rr;
  rr.b = rho / t.per_s;
  const int r = rho - rr.b * t.per_s;
  const size_t row_bytes = (size_t)t.V * (t.dtype == 0 ? 2 : 4);
  // rows of a request: target 0, draft 0, target 1, ..., target gamma; or with
  // deterministic drafts the gamma + 1 target rows
  if (t.det || (r & 1) == 0) {
    const int i = t.det ? r : r >> 1;
    rr.ptr = t.target + ((size_t)rr.b * (t.gamma + 1) + i) * row_bytes;
  } else {
    rr.ptr = t.draft + ((size_t)rr.b * t.gamma + (r >> 1)) * row_bytes;
  }
  rr.T = __ldg(t.temperature + rr.b);
  const float4 st = t.rows[rho];
  rr.m = st.x;
  rr.live = sampling_temperature(rr.T) && st.w == 0.0f &&
            *reinterpret_cast<const volatile uint32_t*>(t.abort_flag) == 0u;
  return rr;
}
// Whether the block works on its row. The abort flag can be raised from the
// host while a kernel runs, so threads may read it differently; the block
// takes one decision (every thread calls this, before any other barrier).
__device__ __forceinline__ bool block_live(const RowRef& rr) { return __syncthreads_and(rr.live) != 0; }

__device__ __forceinline__ float tp_load(const unsigned char* row, int j, int dtype) {
  if (dtype == 0) return __uint_as_float((uint32_t)__ldg(reinterpret_cast<const unsigned short*>(row) + j) << 16);
  return __ldg(reinterpret_cast<const float*>(row) + j);
}

// v * 2^frac rounded to an integer (v >= 0 and small, or a small negative
// correction): integer arithmetic on the float's fields, the same everywhere
__device__ __forceinline__ long long fixed_of(float v, int frac) {
  const uint32_t u = __float_as_uint(v);
  const int e = (int)((u >> 23) & 255u);
  if (e == 0) return 0;  // zero (and denormals, far below 2^-frac)
  const long long mant = (long long)((u & 0x7fffffu) | 0x800000u);
  const int shift = e - 150 + frac;  // v = mant 2^(e - 150)
  long long r;
  if (shift >= 0)
    r = mant << shift;
  else if (shift > -40)
    r = (mant + (1ll << (-shift - 1))) >> (-shift);
  else
    r = 0;
  return (u & 0x80000000u) ? -r : r;
}
__device__ __forceinline__ unsigned long long weight_fixed(ff w, int frac) {
  const long long v = fixed_of(w.hi, frac) + fixed_of(w.lo, frac);
  return v > 0 ? (unsigned long long)v : 0ull;
}
// a fixed-point mass as a float-float value (exact to the pair's precision)
__device__ __forceinline__ ff ff_of_fixed(unsigned long long v, int frac) {
  const float hi = __ull2float_rn(v);
  const long long rest = (long long)(v - (unsigned long long)hi);  // |rest| < 2^40 here
  const float sc = __int_as_float((127 - frac) << 23);              // 2^-frac (frac < 127)
  return fast_two_sum(__fmul_rn(hi, sc), __fmul_rn(__ll2float_rn(rest), sc));
}
// whether RN32(mass / total) < top_p: the ratio of the two exact integers is
// taken in double precision (relative error below 2^-52), then rounded to fp32;
// monotone in mass, so every step of the search takes the same decision
__device__ __forceinline__ bool below_top_p(unsigned long long mass, unsigned long long total, float top_p) {
  return __double2float_rn((double)mass / (double)total) < top_p;
}

// ---- one radix round: the next key byte's mass and count histogram per row --------
__global__ void __launch_bounds__(kTpThreads) fvtp_hist_kernel(const FvtpParams t) {
  __shared__ unsigned long long hm[kTpWarps][256];
  __shared__ uint32_t hc[kTpWarps][256];
  __shared__ float th[kExpTable], tl[kExpTable];
  grid_dependency_sync();
  const int rho = blockIdx.x, s = blockIdx.y, tid = threadIdx.x, w = tid >> 5;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;
  const FvtpCut c = t.cut[rho];
  const uint32_t prefix = t.round == 0 ? 0u : c.prefix, mask = t.round == 0 ? 0u : c.mask;
  const int shift = 24 - 8 * t.round;
  if (tid < kExpTable) {
    th[tid] = t.exp2.hi[tid];
    tl[tid] = t.exp2.lo[tid];
  }
#pragma unroll
  for (int i = 0; i < kTpWarps; ++i) {
    hm[i][tid] = 0ull;
    hc[i][tid] = 0u;
  }
  __syncthreads();
  const int j0 = s * kFvSlice + tid, jn = min(t.V, (s + 1) * kFvSlice);
  float xs[kFvSlice / kTpThreads];
#pragma unroll
  for (int k = 0; k < kFvSlice / kTpThreads; ++k) {
    const int j = j0 + k * kTpThreads;
    xs[k] = j < jn ? tp_load(rr.ptr, j, t.dtype) : 0.0f;
  }
#pragma unroll 4
  for (int k = 0; k < kFvSlice / kTpThreads; ++k) {
    const int j = j0 + k * kTpThreads;
    if (j >= jn) break;
    const uint32_t key = key_of(xs[k]);
    if ((key & mask) != prefix) continue;
    const uint32_t d = (key >> shift) & 255u;
    atomicAdd(&hm[w][d], weight_fixed(exp_diff_ff(xs[k], rr.m, rr.T, th, tl), t.frac_bits));
    atomicAdd(&hc[w][d], 1u);
  }
  __syncthreads();
  unsigned long long sm = 0ull;
  uint32_t sc = 0u;
#pragma unroll
  for (int i = 0; i < kTpWarps; ++i) {
    sm += hm[i][tid];
    sc += hc[i][tid];
  }
  if (sc) {
    atomicAdd(t.hist_m + (size_t)rho * 256 + tid, sm);
    atomicAdd(t.hist_c + (size_t)rho * 256 + tid, sc);
  }
}

// ---- the select step of a round: the bin that holds the last kept token --------------
__global__ void __launch_bounds__(kTpThreads) fvtp_select_kernel(const FvtpParams t) {
  __shared__ unsigned long long suf[256];
  __shared__ unsigned long long tot[kTpWarps];
  __shared__ int best;
  __shared__ float th[kExpTable], tl[kExpTable];
  grid_dependency_sync();
  const int rho = blockIdx.x, tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const RowRef rr = row_ref(t, rho);
  const bool last_round = t.round == t.rounds - 1;
  unsigned long long* hmp = t.hist_m + (size_t)rho * 256;
  uint32_t* hcp = t.hist_c + (size_t)rho * 256;
  if (!block_live(rr)) return;  // nothing was counted for this row; its cut stays empty
  if (tid < kExpTable) {
    th[tid] = t.exp2.hi[tid];
    tl[tid] = t.exp2.lo[tid];
  }
  const unsigned long long H = hmp[tid];
  const uint32_t C = hcp[tid];
  hmp[tid] = 0ull;  // ready for the next round (and the next call)
  hcp[tid] = 0u;
  FvtpCut c = t.cut[rho];
  if (t.round == 0) {
    c.prefix = 0u;
    c.mask = 0u;
    c.above = 0ull;
    // the row's total mass
    unsigned long long v = H;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) tot[w] = v;
    __syncthreads();
    unsigned long long total = 0ull;
#pragma unroll
    for (int i = 0; i < kTpWarps; ++i) total += tot[i];
    c.total = total;
  }
  // A_d = mass above bin d's keys = above + sum of the bins over d (an
  // exclusive suffix sum, bins in descending order)
  suf[tid] = H;
  if (tid == 0) best = 256;
  __syncthreads();
  for (int o = 1; o < 256; o <<= 1) {
    const unsigned long long add = tid + o < 256 ? suf[tid + o] : 0ull;
    __syncthreads();
    suf[tid] += add;
    __syncthreads();
  }
  const unsigned long long A = c.above + (suf[tid] - H);
  const bool cond = C > 0u && below_top_p(A, c.total, t.top_p);
  if (cond) atomicMin(&best, tid);
  __syncthreads();
  const int dstar = best;  // always found: the bin of the group's largest key qualifies
  if (tid != dstar) return;
  const int shift = 24 - 8 * t.round;
  c.prefix |= (uint32_t)dstar << shift;
  c.mask |= 255u << shift;
  c.above = A;
  c.count = C;
  if (last_round) {
    // the key kappa of the last kept token (bf16 keys are known after their
    // upper 16 bits: a value's key is its 16-bit key shifted up, the low half
    // all ones for a negative value)
    uint32_t kappa = c.prefix;
    if (t.dtype == 0) {
      const uint32_t k16 = kappa >> 16;
      const uint32_t h = (k16 & 0x8000u) ? (k16 & 0x7fffu) : (~k16 & 0xffffu);
      kappa = key_of(__uint_as_float(h << 16));
    }
    c.prefix = kappa;
    c.mask = 0xffffffffu;
    const unsigned long long wk =
        weight_fixed(exp_diff_ff(value_of_key(kappa), rr.m, rr.T, th, tl), t.frac_bits);
    // the largest t < count with RN32((above + t wk) / total) < top_p (t = 0 holds)
    uint32_t lo = 0u, hi = C - 1u;
    while (lo < hi) {
      const uint32_t mid = lo + (hi - lo + 1u) / 2u;
      if (below_top_p(c.above + (unsigned long long)mid * wk, c.total, t.top_p))
        lo = mid;
      else
        hi = mid - 1u;
    }
    c.keep = lo + 1u;
    c.kept = c.above + (unsigned long long)c.keep * wk;
    c.j_cut = c.keep == c.count ? t.V : -1;
    c.state = 1;
  }
  t.cut[rho] = c;
}

// ---- the index of the last kept token of key kappa (when only some are kept) ---------
__global__ void __launch_bounds__(kTpThreads) fvtp_kcount_kernel(const FvtpParams t) {
  __shared__ uint32_t wsum[kTpWarps];
  grid_dependency_sync();
  const int rho = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;
  const FvtpCut c = t.cut[rho];
  if (c.state != 1 || c.keep == c.count) return;
  uint32_t n = 0u;
  const int jn = min(t.V, (s + 1) * kFvSlice);
  for (int j = s * kFvSlice + tid; j < jn; j += kTpThreads) n += key_of(tp_load(rr.ptr, j, t.dtype)) == c.prefix;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
  if ((tid & 31) == 0) wsum[tid >> 5] = n;
  __syncthreads();
  if (tid == 0) {
    uint32_t tot = 0u;
    for (int i = 0; i < kTpWarps; ++i) tot += wsum[i];
    t.kcount[(size_t)rho * t.n_slices + s] = tot;
  }
}

__global__ void __launch_bounds__(kTpThreads) fvtp_kpos_kernel(const FvtpParams t) {
  __shared__ uint32_t cnt[kTpThreads];
  __shared__ int slice_s;
  __shared__ uint32_t before_s;
  grid_dependency_sync();
  const int rho = blockIdx.x, tid = threadIdx.x;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;
  FvtpCut c = t.cut[rho];
  if (c.state != 1 || c.keep == c.count) return;
  uint32_t* kc = t.kcount + (size_t)rho * t.n_slices;
  // the slice holding the keep-th token of key kappa (one thread walks the
  // slice counts, then returns them to zero)
  if (tid == 0) {
    uint32_t acc = 0u;
    int sl = t.n_slices - 1;
    for (int s = 0; s < t.n_slices; ++s) {
      if (acc + kc[s] >= c.keep) {
        sl = s;
        break;
      }
      acc += kc[s];
    }
    slice_s = sl;
    before_s = acc;
    for (int s = 0; s < t.n_slices; ++s) kc[s] = 0u;
  }
  __syncthreads();
  // in that slice, thread i takes kFvSlice / 256 consecutive tokens; an
  // exclusive scan of the counts finds the thread, then the token
  constexpr int per = kFvSlice / kTpThreads;
  const int j0 = slice_s * kFvSlice + tid * per;
  uint32_t mine = 0u;
  for (int e = 0; e < per; ++e) {
    const int j = j0 + e;
    if (j < t.V) mine += key_of(tp_load(rr.ptr, j, t.dtype)) == c.prefix;
  }
  cnt[tid] = mine;
  __syncthreads();
  for (int o = 1; o < kTpThreads; o <<= 1) {
    const uint32_t add = tid >= o ? cnt[tid - o] : 0u;
    __syncthreads();
    cnt[tid] += add;
    __syncthreads();
  }
  const uint32_t incl = cnt[tid], excl = incl - mine;
  const uint32_t want = c.keep - before_s;  // 1-based rank within the slice
  if (mine && excl < want && want <= incl) {
    uint32_t seen = excl;
    for (int e = 0; e < per; ++e) {
      const int j = j0 + e;
      if (j < t.V && key_of(tp_load(rr.ptr, j, t.dtype)) == c.prefix && ++seen == want) {
        c.j_cut = j;
        t.cut[rho] = c;
        break;
      }
    }
  }
}

// ---- the accept tests (one warp per request) --------------------------------------------
// probability of token d in row rho's kept set (0 outside it)
__device__ __forceinline__ float kept_prob(const FvtpParams& t, int rho, int d, const float* th, const float* tl) {
  const RowRef rr = row_ref(t, rho);
  const FvtpCut c = t.cut[rho];
  const float x = tp_load(rr.ptr, d, t.dtype);
  const uint32_t key = key_of(x);
  const bool kept = key > c.prefix || (key == c.prefix && d <= c.j_cut);
  if (!kept) return 0.0f;
  return ff_round(ff_mul(exp_diff_ff(x, rr.m, rr.T, th, tl), ff_recip(ff_of_fixed(c.kept, t.frac_bits))));
}

__global__ void __launch_bounds__(32) fvtp_accept_kernel(const FvtpParams t) {
  __shared__ float th[kExpTable], tl[kExpTable];
  grid_dependency_sync();
  const int b = blockIdx.x, lane = threadIdx.x;
  const int gamma = t.gamma, V = t.V, per_s = t.per_s;
  const bool det = t.det != 0;
  const float T = __ldg(t.temperature + b);
  if (!sampling_temperature(T)) return;  // greedy requests: decided in the stream
  // one decision for the warp (the flag can be raised while the kernel runs)
  if (__any_sync(0xffffffffu, *reinterpret_cast<const volatile uint32_t*>(t.abort_flag) != 0u)) return;
  for (int i = lane; i < kExpTable; i += 32) {
    th[i] = t.exp2.hi[i];
    tl[i] = t.exp2.lo[i];
  }
  __syncwarp();
  const int rho0 = b * per_s;
  uint32_t st = 0u;
  for (int r = lane; r < per_s; r += 32)
    if (t.rows[rho0 + r].w != 0.0f) st |= kStatusBadRow;
  const int32_t d_lane = lane < gamma ? __ldg(t.draft_tokens + (size_t)b * gamma + lane) : -1;
  bool stop = false;
  if (lane < gamma) {
    const int i = lane, rx = det ? i : 2 * i, ry = 2 * i + 1;
    const bool valid = d_lane >= 0 && d_lane < V;
    if (!valid) st |= kStatusBadToken;
    if (t.rows[rho0 + rx].w != 0.0f || (!det && t.rows[rho0 + ry].w != 0.0f)) {
      stop = true;  // a bad row ends the loop at its position
    } else {
      float p_d = 0.0f, q_d = det ? 1.0f : 0.0f;
      if (valid) {
        p_d = kept_prob(t, rho0 + rx, d_lane, th, tl);
        if (!det) q_d = kept_prob(t, rho0 + ry, d_lane, th, tl);
      }
      const uint4 wd = step_uniform_words(t.seed, (uint32_t)b, (uint32_t)i, 0u);
      stop = !(uniform24(wd.x) < p_d / q_d);  // q = 0: +inf if p > 0, NaN if p == 0
      if (t.audit_pq) {
        t.audit_pq[((size_t)b * gamma + i) * 2] = p_d;
        t.audit_pq[((size_t)b * gamma + i) * 2 + 1] = q_d;
      }
    }
  }
  const uint32_t ball = __ballot_sync(0xffffffffu, stop);
  const int n = ball ? __ffs(ball) - 1 : gamma;
  const int tn = det ? n : 2 * n;  // position n's target row (the bonus row when n == gamma)
  const bool resid = n < gamma && !det;
  const bool bad_n = t.rows[rho0 + tn].w != 0.0f || (resid && t.rows[rho0 + 2 * n + 1].w != 0.0f);
  const int mode = bad_n ? kFvNone : (resid ? kFvResidual : kFvBonus);
  const int32_t d_n = __shfl_sync(0xffffffffu, d_lane, n & 31);
  const int excl = det && n < gamma ? d_n : -1;
  int32_t* out = t.out_tokens + (size_t)b * (gamma + 1);
  for (int i = lane; i <= gamma; i += 32) out[i] = i < n ? d_lane : (i == n ? 0 : -1);
  st = __reduce_or_sync(0xffffffffu, st);
  if (lane == 0) {
    const FvtpCut cx = t.cut[rho0 + tn];
    const FvtpCut cy = resid ? t.cut[rho0 + 2 * n + 1] : FvtpCut{};
    // the kept masses, in units of exp((x - m) / T), are the draw's normalisers
    const float sx = ff_round(ff_of_fixed(cx.kept, t.frac_bits));
    const float sy = resid ? ff_round(ff_of_fixed(cy.kept, t.frac_bits)) : 0.0f;
    t.draw[b] = FvDraw{n, mode, t.rows[rho0 + tn].x, resid ? t.rows[rho0 + 2 * n + 1].x : 0.0f, sx, sy, excl};
    t.draw_cut[b] = FvtpDrawCut{cx.prefix, resid ? cy.prefix : 0u, cx.j_cut, resid ? cy.j_cut : -1};
    if (t.out_len) t.out_len[b] = n + 1;
    if (st && t.status) atomicOr(t.status, st);
  }
  __syncwarp();
  // every call leaves the workspace at zero: the rows' statistics and cuts
  for (int r = lane; r < per_s; r += 32) {
    t.rows[rho0 + r] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    t.cut[rho0 + r] = FvtpCut{};
  }
}

}  // namespace

int launch_fvtp_cut(const FvtpParams& t0, void* stream) {
  if (t0.B <= 0) return 0;
  FvtpParams t = t0;
  const int n_rows = t.B * t.per_s;
  cudaLaunchConfig_t cfg = {};
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e;
  for (int round = 0; round < t.rounds; ++round) {
    t.round = round;
    cfg.blockDim = dim3(kTpThreads);
    cfg.gridDim = dim3((unsigned)n_rows, (unsigned)t.n_slices);  // slices <= 1024: V <= 2^22
    if ((e = cudaLaunchKernelEx(&cfg, fvtp_hist_kernel, t)) != cudaSuccess) return (int)e;
    cfg.gridDim = dim3((unsigned)n_rows);
    if ((e = cudaLaunchKernelEx(&cfg, fvtp_select_kernel, t)) != cudaSuccess) return (int)e;
  }
  cfg.gridDim = dim3((unsigned)n_rows, (unsigned)t.n_slices);
  if ((e = cudaLaunchKernelEx(&cfg, fvtp_kcount_kernel, t)) != cudaSuccess) return (int)e;
  cfg.gridDim = dim3((unsigned)n_rows);
  if ((e = cudaLaunchKernelEx(&cfg, fvtp_kpos_kernel, t)) != cudaSuccess) return (int)e;
  cfg.blockDim = dim3(32);
  cfg.gridDim = dim3((unsigned)t.B);
  return (int)cudaLaunchKernelEx(&cfg, fvtp_accept_kernel, t);
}

}  // namespace dflash
