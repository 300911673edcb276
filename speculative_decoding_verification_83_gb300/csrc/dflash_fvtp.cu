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
// sort of candidates finds it. Instead the cut is found by a selection over
// the order, weighted by mass:
//  * every weight is exp((x - m) / T) in float-float (Tang's method,
//    dflash_ff.cuh; m the row's largest logit from the stream), rounded to
//    fixed point with frac_bits fractional bits: the sums below are then
//    exact integers, identical wherever they are taken (in any order);
//  * the first round builds, per row, the mass and count histogram of
//    bin0 = floor(8 (m - x) / T) (1/8 of the weight's logarithm per bin),
//    with each bin's smallest and largest key: one CTA per 4096-token slice,
//    a shared-memory histogram, then global 64-bit atomics. Its select step
//    takes the last non-empty bin (from the largest logit down) whose mass
//    above, over the row's mass, rounds (fp32) below top_p: it holds the last
//    kept token, and its tokens are exactly the keys kmin..kmax;
//  * refinement rounds take the offset key - kmin a byte at a time from its
//    top (as many rounds as the bin's key span has bytes) over the tokens
//    whose higher offset bits match those found so far; each select step
//    keeps the lowest non-empty digit whose mass above rounds below top_p;
//  * then the key kappa of the last kept token is known, with the mass of
//    the keys above it, and how many of the tokens with key kappa are kept
//    (they all weigh the same: the largest t with
//    RN32((above + t w_kappa) / total) < top_p); when only some are kept, a
//    count per slice and a scan of one slice give the index j_cut of the last
//    kept one.
// The accept test at position i takes p(d) = w(d) / (kept mass) (0 when d is
// not kept) from the target row, and q(d) likewise from the draft row (1 for
// a deterministic draft), and leaves the draw descriptors for the second pass
// (dflash_fullvocab.cu), which draws over the kept sets.

#include <cuda_runtime.h>

#include <algorithm>
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
  ff inv_t;                  // 1 / T as a pair
  float c8;                  // 8 RN(1/T): the first round's bin scale
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
  rr.inv_t = ff_recip(ff{rr.T, 0.0f});
  rr.c8 = __fmul_rn(__frcp_rn(rr.T), 8.0f);
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

// ---- weights -----------------------------------------------------------------------------
// exp((x - m) / T) as a pair: x - m exactly (two-sum), times 1/T in
// float-float, then Tang's exp. Every weight of the cut and of its accept
// tests comes from here, so equal logits weigh exactly the same.
__device__ __forceinline__ ff tp_weight(float x, const RowRef& rr, const float* th, const float* tl) {
  return exp_ff(ff_mul(two_sum(x, -rr.m), rr.inv_t), th, tl);
}
// v * 2^frac rounded to an integer (half away from zero), for |v| < 2^(63 - frac):
// integer arithmetic on the float's fields (a float-to-64-bit conversion
// would run on the FP64 pipe, which this GPU has little of)
__device__ __forceinline__ long long fixed_part(float v, int frac) {
  const uint32_t u = __float_as_uint(v);
  const int e = (int)((u >> 23) & 255u);
  if (e == 0) return 0;  // zero, and denormals (far below 2^-frac)
  const unsigned long long mant = (u & 0x7fffffu) | 0x800000u;
  const int shift = e - 150 + frac;  // v = mant 2^(e - 150)
  unsigned long long r;
  if (shift >= 0)
    r = mant << shift;
  else if (shift > -26)
    r = (mant + (1ull << (-shift - 1))) >> (-shift);
  else
    r = 0ull;
  return (u & 0x80000000u) ? -(long long)r : (long long)r;
}
// a weight in fixed point (frac fractional bits): the sum of its two parts'
// roundings, never negative
__device__ __forceinline__ unsigned long long to_fixed(ff w, int frac) {
  const long long v = fixed_part(w.hi, frac) + fixed_part(w.lo, frac);
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

// ---- order keys in the units of the refinement -------------------------------------------
// fp32 logits: the 32-bit order key. bf16 logits: its upper half (the
// 16-bit order key of the bf16 value; the lower half of a bf16 value's key
// is all ones for a negative value, zero otherwise).
__device__ __forceinline__ uint32_t okey_of(uint32_t key, int dtype) { return dtype == 0 ? key >> 16 : key; }
__device__ __forceinline__ uint32_t full_key(uint32_t ok, int dtype) {
  return dtype == 0 ? ((ok << 16) | ((ok & 0x8000u) ? 0u : 0xffffu)) : ok;
}

// ---- the first round's bins ------------------------------------------------------------
// bin0(x) = floor(RN(RN(m - x) * 8 RN(1/T))), at most 255: bins of about 1/8
// in the weight's logarithm, from the row's largest logit down. Each step is
// a correctly rounded monotone operation, so bin0 does not increase with x
// (equal logits share a bin) and each bin is an interval of the order; the
// tokens of N(0, sigma) logits spread over about a hundred bins, so the
// histogram's shared atomics rarely collide (the top key byte would put them
// in a handful).
__device__ __forceinline__ int bin0_of(float x, const RowRef& rr) {
  const float b = __fmul_rn(__fsub_rn(rr.m, x), rr.c8);  // +inf for x = -inf
  return b < 255.0f ? (b > 0.0f ? (int)b : 0) : 255;
}
// The order keys (refinement units) of bin d: an interval, found by
// bisection over the finite keys (bin0 of -inf is 255, of +inf 0).
__device__ __forceinline__ void bin_key_range(int d, const RowRef& rr, int dtype, uint32_t* kmin, uint32_t* kmax) {
  const uint32_t lo0 = okey_of(kKeyNegInf, dtype), hi0 = okey_of(kKeyPosInf, dtype);
  uint32_t lo = lo0, hi = hi0;  // smallest key with bin0 <= d
  while (lo < hi) {
    const uint32_t mid = lo + (hi - lo) / 2u;
    if (bin0_of(value_of_key(full_key(mid, dtype)), rr) <= d)
      hi = mid;
    else
      lo = mid + 1u;
  }
  *kmin = lo;
  lo = lo0;
  hi = hi0;  // largest key with bin0 >= d
  while (lo < hi) {
    const uint32_t mid = lo + (hi - lo + 1u) / 2u;
    if (bin0_of(value_of_key(full_key(mid, dtype)), rr) >= d)
      lo = mid;
    else
      hi = mid - 1u;
  }
  *kmax = lo;
}

// ---- slices ------------------------------------------------------------------------------
// A thread's 16 tokens of a 4096-token slice, all loads issued before any
// is used. Rows on a 16-byte boundary are read in 16-byte vectors (thread t
// takes vectors t, t + 256, ...: 8 bf16 or 4 fp32 logits each), others one
// logit at a time (tokens t, t + 256, ...). Past the row's end: j >= jn.
constexpr int kTpPer = kFvSlice / kTpThreads;  // 16
__device__ __forceinline__ int tok_index(int s, int tid, int e, int dtype, bool vec) {
  if (!vec) return s * kFvSlice + tid + e * kTpThreads;
  if (dtype == 0) return s * kFvSlice + (tid + (e >> 3) * kTpThreads) * 8 + (e & 7);
  return s * kFvSlice + (tid + (e >> 2) * kTpThreads) * 4 + (e & 3);
}
__device__ __forceinline__ void load_tokens(const unsigned char* row, int s, int tid, int jn, int dtype, bool vec,
                                            float (&x)[kTpPer]) {
  if (vec && dtype == 0) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int j = tok_index(s, tid, 8 * c, 0, true);
      if (j + 8 <= jn) {
        const uint4 v = __ldg(reinterpret_cast<const uint4*>(row + 2 * (size_t)j));
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          x[8 * c + 2 * i] = __uint_as_float(w[i] << 16);
          x[8 * c + 2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) x[8 * c + i] = j + i < jn ? tp_load(row, j + i, 0) : 0.0f;
      }
    }
  } else if (vec) {
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int j = tok_index(s, tid, 4 * c, 1, true);
      if (j + 4 <= jn) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(row + 4 * (size_t)j));
        x[4 * c] = v.x;
        x[4 * c + 1] = v.y;
        x[4 * c + 2] = v.z;
        x[4 * c + 3] = v.w;
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) x[4 * c + i] = j + i < jn ? tp_load(row, j + i, 1) : 0.0f;
      }
    }
  } else {
#pragma unroll
    for (int e = 0; e < kTpPer; ++e) {
      const int j = tok_index(s, tid, e, dtype, false);
      x[e] = j < jn ? tp_load(row, j, dtype) : 0.0f;
    }
  }
}
// The slice's logits (as fp32) into shared memory, in token order; returns
// how many tokens the slice has. The caller synchronises before reading.
__device__ __forceinline__ int stage_slice(const unsigned char* row, int s, int V, int dtype, float* xs_s) {
  const int tid = threadIdx.x, base = s * kFvSlice, jn = min(V, base + kFvSlice);
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15u) == 0u;
  float x[kTpPer];
  load_tokens(row, s, tid, jn, dtype, vec, x);
#pragma unroll
  for (int e = 0; e < kTpPer; ++e) {
    const int j = tok_index(s, tid, e, dtype, vec);
    if (j < jn) xs_s[j - base] = x[e];
  }
  return jn - base;
}

__device__ __forceinline__ void load_exp_table(const FvtpParams& t, float* th, float* tl) {
  if (threadIdx.x < kExpTable) {
    th[threadIdx.x] = t.exp2.hi[threadIdx.x];
    tl[threadIdx.x] = t.exp2.lo[threadIdx.x];
  }
}

// ---- the first round: masses by bin0 ------------------------------------------------------
__global__ void __launch_bounds__(kTpThreads) fvtp_hist0_kernel(const FvtpParams t) {
  __shared__ __align__(16) float xs_s[kFvSlice];
  __shared__ unsigned long long hm[256];
  __shared__ float th[kExpTable], tl[kExpTable];
  grid_dependency_sync();
  const int rho = blockIdx.x, tid = threadIdx.x;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;
  load_exp_table(t, th, tl);
  hm[tid] = 0ull;
  // slices blockIdx.y, blockIdx.y + gridDim.y, ... of the row
  for (int s = blockIdx.y; s < t.n_slices; s += gridDim.y) {
    const int n = stage_slice(rr.ptr, s, t.V, t.dtype, xs_s);
    __syncthreads();
    for (int l = tid; l < n; l += kTpThreads) {
      const float x = xs_s[l];
      atomicAdd(&hm[bin0_of(x, rr)], to_fixed(tp_weight(x, rr, th, tl), t.frac_bits));
    }
    __syncthreads();  // before the next slice overwrites the stage
  }
  if (hm[tid]) atomicAdd(t.hist_m + (size_t)rho * 256 + tid, hm[tid]);
}

// ---- a refinement round: the next byte of (key - kmin) inside the crossing bin -------
// Refinement round i (1 <= i <= nref) takes bits [8 (nref - i), 8 (nref - i) + 8)
// of the offset ok - kmin (ok: the key in refinement units); the tokens in
// the bin are exactly those with kmin <= ok <= kmax, and of them the ones
// whose higher offset bits match the bits found so far take part. Few tokens
// do: a thread marks its 16 tokens that take part, a warp with any gathers
// them into a queue (a scan of its lanes' counts) and weighs them with every
// lane busy (weighing them where they lie would run the float-float weight
// in many warps for one or two lanes).
__global__ void __launch_bounds__(kTpThreads) fvtp_histr_kernel(const FvtpParams t) {
  __shared__ __align__(16) float xs_s[kFvSlice];
  __shared__ unsigned long long hm[256];
  __shared__ float th[kExpTable], tl[kExpTable];
  __shared__ float queue[kTpWarps][32 * kTpPer];
  grid_dependency_sync();
  const int rho = blockIdx.x, tid = threadIdx.x, lane = tid & 31;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;
  const FvtpCut c = t.cut[rho];
  if (c.state != 1 || c.nref < t.round) return;  // the same for every thread of the block
  const int shift = 8 * (c.nref - t.round);
  const unsigned long long known = (unsigned long long)c.prefix >> (shift + 8);
  load_exp_table(t, th, tl);
  hm[tid] = 0ull;
  float* q = queue[tid >> 5];
  for (int s = blockIdx.y; s < t.n_slices; s += gridDim.y) {
    const int n = stage_slice(rr.ptr, s, t.V, t.dtype, xs_s);
    __syncthreads();
    uint32_t mine = 0u;  // bit e: token tid + e kTpThreads of the slice takes part
#pragma unroll
    for (int e = 0; e < kTpPer; ++e) {
      const int l = tid + e * kTpThreads;
      const uint32_t ok = okey_of(key_of(xs_s[l]), t.dtype);
      const bool in = l < n && ok >= c.kmin && ok <= c.kmax &&
                      ((unsigned long long)(ok - c.kmin) >> (shift + 8)) == known;
      mine |= (in ? 1u : 0u) << e;
    }
    if (__any_sync(0xffffffffu, mine != 0u)) {
      // the warp's queue: each lane's tokens after those of the lanes below
      const int cnt = __popc(mine);
      int incl = cnt;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      const int nq = __shfl_sync(0xffffffffu, incl, 31);
      int pos = incl - cnt;
      for (uint32_t m = mine; m; m &= m - 1u) q[pos++] = xs_s[tid + (__ffs(m) - 1) * kTpThreads];
      __syncwarp();
      for (int i = lane; i < nq; i += 32) {
        const float v = q[i];
        const uint32_t ok = okey_of(key_of(v), t.dtype);
        atomicAdd(&hm[((ok - c.kmin) >> shift) & 255u], to_fixed(tp_weight(v, rr, th, tl), t.frac_bits));
      }
      __syncwarp();  // the queue is refilled for the next slice
    }
    __syncthreads();  // before the next slice overwrites the stage
  }
  if (hm[tid]) atomicAdd(t.hist_m + (size_t)rho * 256 + tid, hm[tid]);
}

// ---- bf16 rows: counts per value instead of a weight per token -----------------------
// A bf16 logit's weight depends only on its 16-bit value, so a block counts
// its tokens per 16-bit order key (all 65 536 of them: two 16-bit counts to a
// shared word, a block taking at most 65 535 tokens) and then weighs each
// key it saw once: mass = count x weight, the same integer as the sum of the
// tokens' own fixed-point weights. A block takes a contiguous range of the
// row, in 16-byte vectors when the row is aligned.
constexpr int kB16Threads = 1024;
constexpr int kB16Words = 32768;  // 65 536 packed 16-bit counts
constexpr size_t kB16Smem = (size_t)kB16Words * 4;

// the block's token range of the row: group g of G, cut at multiples of 8
__device__ __forceinline__ void b16_range(int V, int g, int G, int* j0, int* j1) {
  const long long per = (((long long)V + G - 1) / G + 7) / 8 * 8;
  const long long a = per * g, b = per * (g + 1);
  *j0 = (int)(a < V ? a : V);
  *j1 = (int)(b < V ? b : V);
}

// hand each of the range's tokens to count(k16), its 16-bit key
template <class Count>
__device__ __forceinline__ void b16_count(const unsigned char* row, int j0, int j1, Count count) {
  const unsigned short* r16 = reinterpret_cast<const unsigned short*>(row);
  auto add = [&](uint32_t bits) { count(okey_of(key_of(__uint_as_float(bits << 16)), 0)); };
  const bool vec = ((reinterpret_cast<uintptr_t>(row) + 2 * (uintptr_t)j0) & 15u) == 0u;
  int j = j0 + (int)threadIdx.x * 8;
  if (vec) {
    // a block takes at most 65 528 tokens: at most 8 vectors a thread, all
    // loaded before any is counted (one memory latency, not eight)
    constexpr int kMaxVec = (65528 + kB16Threads * 8 - 1) / (kB16Threads * 8);
    uint4 v[kMaxVec];
#pragma unroll
    for (int r = 0; r < kMaxVec; ++r) {
      const int jr = j + r * kB16Threads * 8;
      v[r] = jr + 8 <= j1 ? __ldg(reinterpret_cast<const uint4*>(r16 + jr)) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int r = 0; r < kMaxVec; ++r) {
      if (j + r * kB16Threads * 8 + 8 > j1) continue;
      add(v[r].x & 0xffffu);
      add(v[r].x >> 16);
      add(v[r].y & 0xffffu);
      add(v[r].y >> 16);
      add(v[r].z & 0xffffu);
      add(v[r].z >> 16);
      add(v[r].w & 0xffffu);
      add(v[r].w >> 16);
    }
    while (j + 8 <= j1) j += kB16Threads * 8;  // to the first vector not counted
  }
  for (; j < j1; j += kB16Threads * 8)  // the ragged end, or an unaligned row
    for (int i = 0; i < 8 && j + i < j1; ++i) add(__ldg(r16 + j + i));
}

// weigh each key seen: bin(k16, x) receives count x weight (bin < 0: the
// key does not take part)
template <class Bin>
__device__ __forceinline__ void b16_weigh(const uint32_t* cnt, const RowRef& rr, int frac, const float* th,
                                          const float* tl, unsigned long long* hm, Bin bin) {
  for (int w = threadIdx.x; w < kB16Words; w += kB16Threads) {
    const uint32_t v = cnt[w];
    if (!v) continue;
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const uint32_t n = half ? v >> 16 : v & 0xffffu;
      if (!n) continue;
      const uint32_t k16 = 2u * (uint32_t)w + (uint32_t)half;
      const float x = value_of_key(full_key(k16, 0));
      const int b = bin(k16, x);
      if (b < 0) continue;
      const unsigned long long wk = to_fixed(tp_weight(x, rr, th, tl), frac);
      if (wk) atomicAdd(&hm[b], (unsigned long long)n * wk);
    }
  }
}

__global__ void __launch_bounds__(kB16Threads) fvtp_hist0_b16_kernel(const FvtpParams t) {
  extern __shared__ __align__(16) uint32_t cnt[];
  __shared__ unsigned long long hm[256];
  __shared__ float th[kExpTable], tl[kExpTable];
  grid_dependency_sync();
  const int rho = blockIdx.x, tid = threadIdx.x;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;
  load_exp_table(t, th, tl);
  if (tid < 256) hm[tid] = 0ull;
  for (int w = tid; w < kB16Words; w += kB16Threads) cnt[w] = 0u;
  int j0, j1;
  b16_range(t.V, blockIdx.y, gridDim.y, &j0, &j1);
  __syncthreads();
  b16_count(rr.ptr, j0, j1, [&](uint32_t k16) { atomicAdd(&cnt[k16 >> 1], (k16 & 1u) ? 0x10000u : 1u); });
  __syncthreads();
  b16_weigh(cnt, rr, t.frac_bits, th, tl, hm, [&](uint32_t, float x) { return bin0_of(x, rr); });
  __syncthreads();
  if (tid < 256 && hm[tid]) atomicAdd(t.hist_m + (size_t)rho * 256 + tid, hm[tid]);
}

// A refinement round on bf16 rows. In the round that takes the last byte of
// the offset (shift 0) the tokens that take part have at most 256 keys,
// kmin + 256 known + d: the block counts them per digit d in 256 words, and
// neither clears nor scans the 65 536 counts.
__global__ void __launch_bounds__(kB16Threads) fvtp_histr_b16_kernel(const FvtpParams t) {
  extern __shared__ __align__(16) uint32_t cnt[];
  __shared__ unsigned long long hm[256];
  __shared__ float th[kExpTable], tl[kExpTable];
  grid_dependency_sync();
  const int rho = blockIdx.x, tid = threadIdx.x;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;
  const FvtpCut c = t.cut[rho];
  if (c.state != 1 || c.nref < t.round) return;  // the same for every thread of the block
  const int shift = 8 * (c.nref - t.round);
  const unsigned long long known = (unsigned long long)c.prefix >> (shift + 8);
  const bool last_byte = shift == 0;
  load_exp_table(t, th, tl);
  if (tid < 256) hm[tid] = 0ull;
  for (int w = tid; w < (last_byte ? 256 : kB16Words); w += kB16Threads) cnt[w] = 0u;
  int j0, j1;
  b16_range(t.V, blockIdx.y, gridDim.y, &j0, &j1);
  __syncthreads();
  auto in_group = [&](uint32_t k16) {
    return k16 >= c.kmin && k16 <= c.kmax && ((unsigned long long)(k16 - c.kmin) >> (shift + 8)) == known;
  };
  if (last_byte) {
    b16_count(rr.ptr, j0, j1, [&](uint32_t k16) {
      if (in_group(k16)) atomicAdd(&cnt[(k16 - c.kmin) & 255u], 1u);
    });
    __syncthreads();
    if (tid < 256 && cnt[tid]) {  // digit tid: one key, all its tokens weigh the same
      const uint32_t k16 = c.kmin + (uint32_t)((known << 8) | (unsigned)tid);
      hm[tid] = (unsigned long long)cnt[tid] *
                to_fixed(tp_weight(value_of_key(full_key(k16, 0)), rr, th, tl), t.frac_bits);
    }
  } else {
    b16_count(rr.ptr, j0, j1, [&](uint32_t k16) {
      if (in_group(k16)) atomicAdd(&cnt[k16 >> 1], (k16 & 1u) ? 0x10000u : 1u);
    });
    __syncthreads();
    b16_weigh(cnt, rr, t.frac_bits, th, tl, hm, [&](uint32_t k16, float) {
      return in_group(k16) ? (int)(((k16 - c.kmin) >> shift) & 255u) : -1;
    });
  }
  __syncthreads();
  if (tid < 256 && hm[tid]) atomicAdd(t.hist_m + (size_t)rho * 256 + tid, hm[tid]);
}

// The last kept token's key kappa is known (refinement units: okappa), with
// the mass of its group: how many of its tokens there are (they weigh the
// same, so the group's mass is their count times that weight), how many are
// kept (the largest t < count with RN32((above + t wk) / total) < top_p; t = 0
// holds), the kept mass, and j_cut when all of them are kept.
__device__ __forceinline__ void resolve(FvtpCut& c, unsigned long long group_mass, uint32_t okappa, const RowRef& rr,
                                        const FvtpParams& t, const float* th, const float* tl) {
  c.kappa = full_key(okappa, t.dtype);
  const unsigned long long wk = to_fixed(tp_weight(value_of_key(c.kappa), rr, th, tl), t.frac_bits);
  c.count = wk ? (uint32_t)(group_mass / wk) : 1u;
  uint32_t lo = 0u, hi = c.count - 1u;
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
  c.state = 2;
}

// block-wide exclusive prefix sum over the 256 bins in the order given by
// pos (the bin with pos 0 first); returns the sum of the bins before this
// thread's, and leaves the inclusive sums in buf
__device__ __forceinline__ unsigned long long bins_before(unsigned long long H, int pos, unsigned long long* buf) {
  buf[pos] = H;
  __syncthreads();
  for (int o = 1; o < 256; o <<= 1) {
    const unsigned long long add = pos >= o ? buf[pos - o] : 0ull;
    __syncthreads();
    buf[pos] += add;
    __syncthreads();
  }
  return buf[pos] - H;
}

// ---- the select step of the first round ----------------------------------------------
// A bin's mass is 0 only below every token that weighs (weights fall with
// the bin), where the mass above is the row's: no such bin holds the cut.
__global__ void __launch_bounds__(kTpThreads) fvtp_select0_kernel(const FvtpParams t) {
  __shared__ unsigned long long buf[256];
  __shared__ int best;
  __shared__ float th[kExpTable], tl[kExpTable];
  grid_dependency_sync();
  const int rho = blockIdx.x, tid = threadIdx.x;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;  // nothing was counted for this row; its cut stays empty
  load_exp_table(t, th, tl);
  unsigned long long* hmp = t.hist_m + (size_t)rho * 256;
  const unsigned long long H = hmp[tid];
  hmp[tid] = 0ull;  // ready for the next round (and the next call)
  if (tid == 0) best = -1;
  // bins ascend from the row's largest logit: the mass above bin d is the
  // sum of bins 0..d-1; the row's mass is the sum of all
  const unsigned long long A = bins_before(H, tid, buf);
  const unsigned long long total = buf[255];
  // the last kept token lies in the last bin with mass whose mass above,
  // over the row's mass, rounds below top_p (bin 0 holds the largest logit,
  // weight 1, and qualifies, since 0 < top_p)
  if (H > 0ull && below_top_p(A, total, t.top_p)) atomicMax(&best, tid);
  __syncthreads();
  if (tid != best) return;
  FvtpCut c = {};
  c.total = total;
  c.above = A;
  c.prefix = 0u;
  c.state = 1;
  bin_key_range(tid, rr, t.dtype, &c.kmin, &c.kmax);
  const uint32_t span = c.kmax - c.kmin;
  c.nref = span == 0u ? 0 : (32 - __clz(span) + 7) / 8;
  if (c.nref == 0) resolve(c, H, c.kmin, rr, t, th, tl);
  t.cut[rho] = c;
}

// ---- the select step of refinement round t.round -------------------------------------
__global__ void __launch_bounds__(kTpThreads) fvtp_selectr_kernel(const FvtpParams t) {
  __shared__ unsigned long long buf[256];
  __shared__ int best;
  __shared__ float th[kExpTable], tl[kExpTable];
  grid_dependency_sync();
  const int rho = blockIdx.x, tid = threadIdx.x;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;
  FvtpCut c = t.cut[rho];
  if (c.state != 1 || c.nref < t.round) return;
  load_exp_table(t, th, tl);
  unsigned long long* hmp = t.hist_m + (size_t)rho * 256;
  const unsigned long long H = hmp[tid];
  hmp[tid] = 0ull;
  if (tid == 0) best = 256;
  // digits ascend with the key, so digit d's mass above is that of the
  // group's keys above it, digits d+1..255 (prefix order 255 - d)
  const unsigned long long A = c.above + bins_before(H, 255 - tid, buf);
  // the lowest digit with mass whose mass above rounds below top_p (the
  // group's largest digit with mass qualifies: its mass above is the group's)
  if (H > 0ull && below_top_p(A, c.total, t.top_p)) atomicMin(&best, tid);
  __syncthreads();
  if (tid != best) return;
  const int shift = 8 * (c.nref - t.round);
  c.prefix |= (uint32_t)tid << shift;
  c.above = A;
  if (t.round == c.nref) resolve(c, H, c.kmin + c.prefix, rr, t, th, tl);
  t.cut[rho] = c;
}

// ---- the index of the last kept token of key kappa (when only some are kept) ---------
__global__ void __launch_bounds__(kTpThreads) fvtp_kcount_kernel(const FvtpParams t) {
  __shared__ uint32_t wsum[kTpWarps];
  grid_dependency_sync();
  const int rho = blockIdx.x, tid = threadIdx.x;
  const RowRef rr = row_ref(t, rho);
  if (!block_live(rr)) return;
  const FvtpCut c = t.cut[rho];
  if (c.state != 2 || c.keep == c.count) return;
  const bool vec = (reinterpret_cast<uintptr_t>(rr.ptr) & 15u) == 0u;
  for (int s = blockIdx.y; s < t.n_slices; s += gridDim.y) {
    uint32_t n = 0u;
    const int jn = min(t.V, (s + 1) * kFvSlice);
    float xs[kTpPer];
    load_tokens(rr.ptr, s, tid, jn, t.dtype, vec, xs);
#pragma unroll
    for (int e = 0; e < kTpPer; ++e) n += tok_index(s, tid, e, t.dtype, vec) < jn && key_of(xs[e]) == c.kappa;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) n += __shfl_xor_sync(0xffffffffu, n, o);
    if ((tid & 31) == 0) wsum[tid >> 5] = n;
    __syncthreads();
    if (tid == 0) {
      uint32_t tot = 0u;
      for (int i = 0; i < kTpWarps; ++i) tot += wsum[i];
      t.kcount[(size_t)rho * t.n_slices + s] = tot;
    }
    __syncthreads();  // wsum is rewritten for the next slice
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
  if (c.state != 2 || c.keep == c.count) return;
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
    if (j < t.V) mine += key_of(tp_load(rr.ptr, j, t.dtype)) == c.kappa;
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
      if (j < t.V && key_of(tp_load(rr.ptr, j, t.dtype)) == c.kappa && ++seen == want) {
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
  const bool kept = c.state == 2 && (key > c.kappa || (key == c.kappa && d <= c.j_cut));
  if (!kept) return 0.0f;
  return ff_round(ff_mul(tp_weight(x, rr, th, tl), ff_recip(ff_of_fixed(c.kept, t.frac_bits))));
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
    t.draw_cut[b] = FvtpDrawCut{cx.kappa, resid ? cy.kappa : 0u, cx.j_cut, resid ? cy.j_cut : -1};
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
  // Blocks over (row, group of slices): about 2048 blocks in all, each
  // looping over its row's slices blockIdx.y, blockIdx.y + groups, ...
  // (thousands of one-slice blocks cost more to schedule than their work).
  const int groups = (int)std::max(1, std::min(t.n_slices, (2048 + n_rows - 1) / n_rows));
  // bf16 rows count per value: one 1024-thread block per SM (128 KB of
  // counts), at most 65 528 tokens each (ranges are cut at multiples of 8,
  // so no count can reach 65 536), about four blocks per SM in all
  const bool b16 = t.dtype == 0;
  const int g16 = std::max((t.V + 65527) / 65528, std::min(32, (4 * 152 + n_rows - 1) / n_rows));
  static bool b16_ready[kMaxDevices] = {false};
  int dev = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return (int)e;
  if (b16 && dev >= 0 && dev < kMaxDevices && !b16_ready[dev]) {
    if ((e = cudaFuncSetAttribute(fvtp_hist0_b16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kB16Smem)) != cudaSuccess ||
        (e = cudaFuncSetAttribute(fvtp_histr_b16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                  (int)kB16Smem)) != cudaSuccess)
      return (int)e;
    b16_ready[dev] = true;
  }
  // the first round, then the refinement rounds: up to four for fp32 keys
  // (a span of at most 32 bits), two for bf16 (16 bits); rows already
  // resolved leave the later launches at once
  const int last_round = b16 ? 2 : 4;
  for (int round = 0; round <= last_round; ++round) {
    t.round = round;
    if (b16) {
      cfg.blockDim = dim3(kB16Threads);
      cfg.gridDim = dim3((unsigned)n_rows, (unsigned)g16);
      cfg.dynamicSmemBytes = kB16Smem;
      e = cudaLaunchKernelEx(&cfg, round == 0 ? fvtp_hist0_b16_kernel : fvtp_histr_b16_kernel, t);
      cfg.dynamicSmemBytes = 0;
    } else {
      cfg.blockDim = dim3(kTpThreads);
      cfg.gridDim = dim3((unsigned)n_rows, (unsigned)groups);
      e = cudaLaunchKernelEx(&cfg, round == 0 ? fvtp_hist0_kernel : fvtp_histr_kernel, t);
    }
    if (e != cudaSuccess) return (int)e;
    cfg.blockDim = dim3(kTpThreads);
    cfg.gridDim = dim3((unsigned)n_rows);
    if ((e = cudaLaunchKernelEx(&cfg, round == 0 ? fvtp_select0_kernel : fvtp_selectr_kernel, t)) != cudaSuccess)
      return (int)e;
  }
  cfg.blockDim = dim3(kTpThreads);
  cfg.gridDim = dim3((unsigned)n_rows, (unsigned)groups);
  if ((e = cudaLaunchKernelEx(&cfg, fvtp_kcount_kernel, t)) != cudaSuccess) return (int)e;
  cfg.gridDim = dim3((unsigned)n_rows);
  if ((e = cudaLaunchKernelEx(&cfg, fvtp_kpos_kernel, t)) != cudaSuccess) return (int)e;
  cfg.blockDim = dim3(32);
  cfg.gridDim = dim3((unsigned)t.B);
  return (int)cudaLaunchKernelEx(&cfg, fvtp_accept_kernel, t);
}

}  // namespace dflash
