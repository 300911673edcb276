// dflash_candidates.cu -- verification from the candidates of vocabulary shards.
//
// When the logits rows are split by vocabulary across ranks (a
// vocabulary-parallel LM head), each rank reduces its shard to a record: per
// row the shard's k largest (logit, token) pairs and its largest logit
// (sweep_kernel's candidates task). After one all-gather of those records
// every rank holds, per row, the union of the shards' top k, which contains
// the row's global top k: a token among the k largest of a row is among the k
// largest of its own shard, since the order (logit desc, token asc) within a
// shard is the global order restricted to it. This kernel merges the union
// into the row's top k and applies the filter and the accept rule of the
// stream kernel's finals to the same values, so every rank computes the
// outputs of the unsharded step, bit for bit, from identical Philox uniforms
// and with no second exchange.
//
// One CTA of four warps per request. A sampling request's warps take its rows
// in turn (target 0, draft 0, ..., target gamma): rank the row's candidates
// (larger composite first; a token listed twice keeps its first place),
// filter the top k into the request's lists, then warp 0 runs the accept test
// and the draw. A greedy request's warp 0 takes each target row's largest
// candidate and prefix-matches the drafts.

#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "dflash_device.cuh"
#include "dflash_internal.h"
#include "dflash_rule.cuh"

namespace dflash {
namespace {

constexpr int kCandWarps = 4;

struct CandSmem {
  int32_t idx[kMaxRowsPerRequest][33];
  float prob[kMaxRowsPerRequest][33];
  unsigned long long comp[kCandWarps][kMaxShardCand];
  unsigned long long sorted[kCandWarps][kMaxTopK];
  alignas(16) unsigned long long scratch[2 * kMaxTopK];
  float exp_hi[kExpTable], exp_lo[kExpTable];  // 2^(j/64) for the filter's float-float exp
};

// candidate j of shard s for row `row` of the target (or draft) rows
struct RowCands {
  const uint32_t* logit;  // shard 0's block; shard s at + s * words
  const uint32_t* token;
  const uint32_t* rmax;
};

__device__ __forceinline__ RowCands row_cands(const CandParams& c, bool target, size_t row) {
  const CandidateLayout& L = c.L;
  RowCands r;
  r.logit = c.records + (target ? L.t_logit : L.d_logit) + row * c.k;
  r.token = c.records + (target ? L.t_token : L.d_token) + row * c.k;
  r.rmax = c.records + (target ? L.t_max : L.d_max) + row;
  return r;
}

// composite of candidate i (shard i / k, rank i % k); 0 for an empty slot
__device__ __forceinline__ unsigned long long cand_composite(const CandParams& c, const RowCands& r, int i) {
  const int s = i / c.k, j = i - s * c.k;
  const size_t off = (size_t)s * c.words + j;
  const int32_t t = (int32_t)__ldg(r.token + off);
  if (t < 0 || t >= c.V) return 0ull;
  return composite(key_of(__uint_as_float(__ldg(r.logit + off))), t);
}

// whether a row is unusable (as the stream kernel judges a whole row): a
// shard holds a NaN, or the row's largest logit is infinite
__device__ __forceinline__ bool row_is_bad(const CandParams& c, const RowCands& r) {
  bool nan = false;
  float m = -INFINITY;
  for (int s = 0; s < c.n_shards; ++s) {
    const float v = __uint_as_float(__ldg(r.rmax + (size_t)s * c.words));
    nan |= isnan(v);
    m = fmaxf(m, v);
  }
  return nan || !(fabsf(m) < INFINITY);
}

__global__ void __launch_bounds__(kCandWarps * 32) verify_candidates_kernel(const CandParams c) {
  __shared__ CandSmem S;
  const int b = blockIdx.x, lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int gamma = c.gamma, V = c.V, k = c.top_k, n_cand = c.n_shards * c.k;
  const float T = __ldg(c.temperature + b);
  int32_t* out = c.out_tokens + (size_t)b * (gamma + 1);
  const int32_t* d = c.draft_tokens + (size_t)b * gamma;
  for (int j = threadIdx.x; j < kExpTable; j += blockDim.x) {
    S.exp_hi[j] = c.exp2.hi[j];
    S.exp_lo[j] = c.exp2.lo[j];
  }
  __syncthreads();

  if (!sampling_temperature(T)) {
    // greedy: the argmax of each target row is its largest candidate
    if (w != 0) return;
    uint32_t st = T != 0.0f ? kStatusBadTemperature : 0u;
    const int32_t d_lane = lane < gamma ? __ldg(d + lane) : -1;
    int n = gamma;
    int32_t am[2] = {-1, -1};
    for (int base = 0, u = 0; base <= gamma; base += 32, ++u) {
      const int i = base + lane;
      bool mismatch = false;
      if (i <= gamma) {
        const RowCands r = row_cands(c, true, (size_t)b * (gamma + 1) + i);
        if (row_is_bad(c, r)) st |= kStatusBadRow;
        unsigned long long best = 0ull;
        for (int j = 0; j < n_cand; ++j) {
          const unsigned long long x = cand_composite(c, r, j);
          best = x > best ? x : best;
        }
        am[u] = best ? composite_idx(best) : 0;
        if (am[u] < 0 || am[u] >= V) am[u] = 0;
      }
      if (i < gamma) {  // gamma <= 32: i == lane
        if (d_lane < 0 || d_lane >= V) st |= kStatusBadToken;
        mismatch = d_lane != am[u];
      }
      const uint32_t mm = __ballot_sync(0xffffffffu, mismatch);
      if (mm && n == gamma) n = base + __ffs(mm) - 1;
    }
    for (int base = 0, u = 0; base <= gamma; base += 32, ++u) {
      const int i = base + lane;
      if (i <= gamma) out[i] = i < n ? d_lane : (i == n ? am[u] : -1);
    }
    st = __reduce_or_sync(0xffffffffu, st);
    if (lane == 0) {
      c.out_len[b] = n + 1;
      if (st && c.status) atomicOr(c.status, st);
    }
    return;
  }

  // sampling: every row's filtered list, as the stream kernel's row finals
  // write it (lane j: the rank-j kept token and its probability; column 32:
  // the probability of the position's draft token, and the bad flag)
  const int per_s = 2 * gamma + 1;
  unsigned long long* cm = S.comp[w];
  for (int r = w; r < per_s; r += kCandWarps) {
    const bool target = (r & 1) == 0;
    const int i = r >> 1;  // position (the bonus row has no draft token)
    const RowCands rc = row_cands(c, target, target ? (size_t)b * (gamma + 1) + i : (size_t)b * gamma + i);
    const bool bad = row_is_bad(c, rc);
    for (int j = lane; j < n_cand; j += 32) cm[j] = cand_composite(c, rc, j);
    __syncwarp();
    int n_valid = 0;
    for (int j = lane; j < n_cand; j += 32) {
      const unsigned long long x = cm[j];
      if (x == 0ull) continue;
      ++n_valid;
      int rank = 0;
      for (int m = 0; m < n_cand; ++m) {
        const unsigned long long y = cm[m];
        rank += (y > x || (y == x && m < j)) ? 1 : 0;
      }
      if (rank < k) S.sorted[w][rank] = x;
    }
    n_valid = __reduce_add_sync(0xffffffffu, n_valid);
    __syncwarp();
    const int n_c = min(n_valid, k);
    const unsigned long long a = lane < n_c ? S.sorted[w][lane] : 0ull;
    const bool valid = lane < k && lane < n_c;
    int32_t idx = valid ? composite_idx(a) : -1;
    const float pr = filter_lane(valid ? composite_key(a) : 0u, idx, k, T, c.top_p, lane, S.exp_hi, S.exp_lo);
    const int32_t d_row = i < gamma ? __ldg(d + i) : -1;
    const uint32_t hit = __ballot_sync(0xffffffffu, idx >= 0 && idx == d_row);
    const float pd = hit ? __shfl_sync(0xffffffffu, pr, __ffs(hit) - 1) : 0.0f;
    S.idx[r][lane] = idx;
    S.prob[r][lane] = pr;
    if (lane == 0) {
      S.idx[r][32] = bad ? 1 : 0;
      S.prob[r][32] = pd;
    }
    __syncwarp();  // the warp's candidate scratch is reused by its next row
  }
  __syncthreads();
  if (w == 0) {
    const int32_t d_lane = lane < gamma ? __ldg(d + lane) : -1;
    uint4 wd = make_uint4(0u, 0u, 0u, 0u);
    if (lane <= gamma) wd = step_uniform_words(c.seed, (uint32_t)b, (uint32_t)lane, 0u);
    sampling_rule(S.idx, S.prob, per_s, false, gamma, V, d_lane, wd, c.seed, b, lane, S.scratch, out, c.out_len,
                  c.status);
  }
}

}  // namespace

int launch_verify_candidates(const CandParams& c, void* stream) {
  verify_candidates_kernel<<<c.B, kCandWarps * 32, 0, (cudaStream_t)stream>>>(c);
  return (int)cudaGetLastError();
}

}  // namespace dflash
