// dflash_sweep.cu -- the draft-verification step as one persistent kernel.
//
// Pass structure (one launch, one CTA per SM, four warp roles):
//  1. Stream. Every row the step needs (target rows of every request, draft
//     rows of sampling requests) is cut into 16 KB pieces of its aligned body.
//     The producer warp moves pieces into a 12-stage shared-memory ring with
//     1-D bulk copies (TMA) and records what each stage holds. Each of the 8
//     consumer warps takes whole pieces and reduces every 256-element tile of
//     them to its largest logit (packed bf16x2 / fp32 max that propagates
//     NaN), storing the tile's order key to the workspace; for greedy rows it
//     folds the piece's best (logit, lowest index) into the row's running
//     argmax, and for full-vocabulary rows it reduces the piece to (max, sum
//     of exp). Consumers never fence and never wait on each other. Pieces are
//     dealt round-robin to the CTAs, request by request (sampling requests
//     first), so rows complete progressively.
//  2. Publish. For the rows whose finals wait on counts (greedy rows,
//     full-vocabulary rows) the publisher warp takes the finished pieces in
//     batches: one GPU-scope fence per batch, then a fire-and-forget counter
//     increment per piece.
//  3. Finals (the 4-warp finals group of every CTA draws jobs from a counter
//     in the workspace, in the order rows finish). A row final gives a row's
//     top-k in (logit desc, index asc) order: it polls the row's tile keys
//     (zero until written), and a lower bound tau of the k-th largest tile
//     maximum (also a lower bound of the row's k-th largest logit: the k
//     tiles with the largest maxima hold k logits >= it) leaves about k tiles
//     to re-read from L2; the head and tail logits outside the aligned body
//     are always candidates, and a row whose ties leave too many candidates
//     falls back to an exact radix selection. It then filters the row
//     (temperature, softmax over the survivors, top-p, renormalise) into
//     words that are never zero, plus one with the probability it gives the
//     position's draft token. A sampling request's final polls its rows'
//     words and runs the accept test at every draft position at once (Philox
//     uniforms), then the residual or bonus draw. A greedy request's final
//     prefix-matches the streamed argmax. A group draws its next job once the
//     current one's inputs are ready.
// Every wait is time-bounded; row finals wait only on the stream, and a
// request final only on row finals drawn before it, so there is no cycle of
// waits and no grid-wide barrier. Every successful call leaves the workspace
// at zero. A CTA that finds the workspace's abort flag set in its prologue
// (a cancelled workspace) reports a timeout and returns before any copy;
// otherwise the producer waits for its last copies to land before it returns.
//
// The same kernel serves deterministic drafts (sampling requests stream their
// target rows only) and, as rows tasks, the filtered rows, the sampler and a
// vocabulary shard's top-k candidates.
//
// The method follows "DFlash2 用投机解码给 Qwen 提速" (bml.asia, draft/verify
// loop and model-card settings) and "无损加速是真的吗？Qwen3.8-27B-DFlash2
// 如何保证输出与目标模型完全一致" (rytg.cn, section 投机解码如何白嫖速度, step 3,
// and the lossless definition), with the standard accept rule min(1, p/q),
// residual max(0, p - q) and bonus token.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cfloat>
#include <climits>
#include <cstdint>
#include <mutex>

#include "dflash_device.cuh"
#include "dflash_ff.cuh"
#include "dflash_internal.h"
#include "dflash_rule.cuh"

namespace dflash {
namespace {


// what the producer loaded into a ring stage (read by the consumers)
struct PieceDesc {
  int slot;
  int pp;      // piece index within the row
  int nvec;    // 16-byte vectors in the stage
  int head;    // logits before the row's aligned body; + kDescArgmax / kDescStats
  int ord;     // request ordinal of the row (verification)
};
constexpr int kDescArgmax = 256;  // the consumers track this row's argmax in-stream
constexpr int kDescStats = 512;   // the consumers reduce the piece to (max, sum of exp)
constexpr float kLog2eHi = 1.4426950216293335f;  // log2(e), the nearest float

struct Smem {
  alignas(128) unsigned char ring[kStages][kPieceBytes];
  PieceDesc desc[kStages];
  uint64_t full[kStages];       // ring stage loaded (producer expect_tx + bytes)
  uint64_t empty[kStages];      // ring stage read (by the piece's consumer warp)
  uint64_t kfull[kKeyQueue];    // piece's tile keys stored (by the piece's consumer warp)
  uint64_t kempty[kKeyQueue];   // piece published (publisher)
  int16_t req_of_ord[kMaxB];
  union {
    uint32_t key_cache[kKeyCache];
    struct {  // rows padded to 33 words: lane i reading row 2i hits bank 2i
      int32_t idx[kMaxRowsPerRequest][33];
      float prob[kMaxRowsPerRequest][33];
    } lists;
    struct {  // full-vocabulary request final: per row max, sum of exp (a pair), bad flag
      float m[kMaxRowsPerRequest];
      float s[kMaxRowsPerRequest];
      float s_lo[kMaxRowsPerRequest];
      int bad[kMaxRowsPerRequest];
    } fv;
  } u;
  alignas(16) uint32_t hist[256];              // a row final's tau histogram
  alignas(16) unsigned long long cand[kCandCap];  // also a warp's draw scratch
  alignas(16) unsigned long long sorted[32];      // a row final's top 32 candidates, in order
  float exp_hi[kExpTable], exp_lo[kExpTable];   // 2^(j/64) for the filter's float-float exp
  int32_t cand_tiles[kCandTileCap];
  int fin_slot;
  int fin_cmd;
  uint32_t warp_red[kConsumerWarps];
  int n_cand;
  int n_cand_tiles;
  int flag;
  int n_samp;
  uint32_t digit;
  uint32_t digit_above;
  int bad_head_tail;
  int cancelled;  // the workspace's abort flag was set before the call
};

// ---- row geometry ---------------------------------------------------------------
struct RowBody {
  const unsigned char* row;  // first logit of the row
  int head;                  // logits before the first 16-byte boundary
  int nvec;                  // 16-byte vectors of the body
  int tail_start;            // first logit after the body
};

__device__ __forceinline__ RowBody row_body(const unsigned char* row, int V, int esize) {
  RowBody r;
  r.row = row;
  const uint32_t mis = (uint32_t)((uintptr_t)row & 15u);
  int head = (int)(((16u - mis) & 15u) / (uint32_t)esize);
  if (head > V) head = V;
  r.head = head;
  r.nvec = (int)(((long long)(V - head) * esize) >> 4);
  r.tail_start = head + r.nvec * (16 / esize);
  return r;
}

__device__ __forceinline__ float load_logit(const unsigned char* row, int j, int dtype) {
  if (dtype == 0) {
    const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + j);
    return __uint_as_float((uint32_t)h << 16);
  }
  return __ldg(reinterpret_cast<const float*>(row) + j);
}

// ---- work enumeration -----------------------------------------------------------
// Verification: requests are ordered sampling-first (by index), then greedy.
// A sampling request owns 2*gamma+1 slots (target 0, draft 0, target 1, ...,
// target gamma), or with deterministic drafts gamma+1 (its target rows: the
// drafter's distribution is a point mass, so no draft row is read); a greedy
// one owns gamma+1 (its target rows). Rows tasks: slot = row.
struct SlotInfo {
  int ord;        // request ordinal (verify) or row (rows tasks)
  int r;          // row within the request
  bool sampling;  // request samples (vs greedy)
  const unsigned char* ptr;
  int k_eff;
};

// slots of a sampling request
__device__ __forceinline__ int samp_slots(const Params& p) { return p.det ? p.gamma + 1 : 2 * p.gamma + 1; }
// position of row r of a sampling request (target row i, or draft row i)
__device__ __forceinline__ int samp_position(const Params& p, int r) { return p.det ? r : r >> 1; }

__device__ __forceinline__ SlotInfo slot_info(const Params& p, const Smem& S, int slot) {
  SlotInfo s;
  const size_t row_bytes = (size_t)p.geo.V * p.geo.esize;
  if (p.task == kTaskVerify || p.task == kTaskVerifyGreedy) {
    const int per_s = samp_slots(p), per_g = p.gamma + 1;
    const int samp_end = S.n_samp * per_s;
    if (slot < samp_end) {
      s.ord = slot / per_s;
      s.r = slot - s.ord * per_s;
      s.sampling = true;
      const int b = S.req_of_ord[s.ord];
      const int i = samp_position(p, s.r);
      if (p.det || (s.r & 1) == 0)
        s.ptr = p.target + ((size_t)b * (p.gamma + 1) + i) * row_bytes;
      else
        s.ptr = p.draft + ((size_t)b * p.gamma + i) * row_bytes;
      s.k_eff = p.top_k;
    } else {
      const int s2 = slot - samp_end;
      const int g = s2 / per_g;
      s.ord = S.n_samp + g;
      s.r = s2 - g * per_g;
      s.sampling = false;
      const int b = S.req_of_ord[s.ord];
      s.ptr = p.target + ((size_t)b * (p.gamma + 1) + s.r) * row_bytes;
      s.k_eff = 1;
    }
  } else {
    s.ord = slot;
    s.r = 0;
    s.sampling = p.task == kTaskCandidates || sampling_temperature(__ldg(p.temperature + slot));
    s.ptr = p.target + (size_t)slot * row_bytes;
    s.k_eff = s.sampling ? p.top_k : 1;
  }
  return s;
}

__device__ __forceinline__ int active_slots(const Params& p, const Smem& S) {
  if (p.task == kTaskVerify || p.task == kTaskVerifyGreedy)
    return S.n_samp * samp_slots(p) + (p.B - S.n_samp) * (p.gamma + 1);
  return p.B;
}

// Request order (sampling first), built by all threads of the CTA.
__device__ void build_request_order(const Params& p, Smem& S) {
  const int t = threadIdx.x;
  if (t == 0) S.cancelled = *reinterpret_cast<const volatile uint32_t*>(p.abort_flag) != 0u ? 1 : 0;
  if (p.task != kTaskVerify && p.task != kTaskVerifyGreedy) {
    if (t == 0) S.n_samp = 0;
    return;
  }
  const int B = p.B;
  const int chunk = (B + kConsumers - 1) / kConsumers;
  const int lo = min(B, t * chunk), hi = min(B, lo + chunk);
  int mine = 0;
  if (t < kConsumers && p.task == kTaskVerify)
    for (int b = lo; b < hi; ++b) mine += sampling_temperature(__ldg(p.temperature + b)) ? 1 : 0;
  // exclusive scan of per-thread counts over the 256 consumer threads
  const int lane = t & 31, warp = t >> 5;
  int incl = mine;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31 && warp < kConsumerWarps) S.warp_red[warp] = (uint32_t)incl;
  __syncthreads();
  int warp_base = 0, total = 0;
  for (int w = 0; w < kConsumerWarps; ++w) {
    if (w < warp) warp_base += (int)S.warp_red[w];
    total += (int)S.warp_red[w];
  }
  if (t < kConsumers) {
    int samp_before = warp_base + incl - mine;
    int greedy_before = lo - samp_before;
    for (int b = lo; b < hi; ++b) {
      const bool s = p.task == kTaskVerify && sampling_temperature(__ldg(p.temperature + b));
      if (s)
        S.req_of_ord[samp_before++] = b;
      else
        S.req_of_ord[total + greedy_before++] = b;
    }
  }
  if (t == 0) S.n_samp = total;
  __syncthreads();
}

// ---- finals-group helpers (128 threads, gt = thread index in the group) ----------
__device__ __forceinline__ int fin_tid() { return (int)threadIdx.x - kFinBase; }
// The thread that draws the group's finals jobs (one of the last warp, which
// issues no fences). A group draws its next job once the current one is
// ready to run, so jobs go to the groups that are actually working through
// theirs rather than to those still waiting for a row.
constexpr int kFinDrawer = kFin - 32;
__device__ __forceinline__ void draw_next_job(const Params& p, uint32_t& next) {
  if (fin_tid() == kFinDrawer) next = atomicAdd(p.job_cnt, 1u);  // read only when the job ends
}

// Finds, in S.hist, the digit holding the krem-th largest element (counts
// from the top); sets S.digit and S.digit_above (elements in larger digits).
// Run by the group's first warp.
__device__ __forceinline__ void find_digit(Smem& S, uint32_t krem) {
  const int gt = fin_tid(), lane = gt & 31;
  if (gt < 32) {
    uint32_t c[8];
    uint32_t s = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      c[i] = S.hist[lane * 8 + i];
      s += c[i];
    }
    uint32_t v = s;  // sum over lanes >= lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      uint32_t n = __shfl_down_sync(0xffffffffu, v, o);
      if (lane + o < 32) v += n;
    }
    const uint32_t above = v - s;
    const bool here = above < krem && krem <= v;
    const uint32_t ball = __ballot_sync(0xffffffffu, here);
    if (here && lane == 31 - __clz(ball)) {
      uint32_t acc = above;
      uint32_t d = (uint32_t)lane * 8u;
      for (int i = 7; i >= 0; --i) {
        if (acc + c[i] >= krem) {
          d = (uint32_t)lane * 8u + (uint32_t)i;
          break;
        }
        acc += c[i];
      }
      S.digit = d;
      S.digit_above = acc;
    }
    if (ball == 0u && lane == 0) {  // krem exceeds the count: cannot happen for valid k
      S.digit = 0;
      S.digit_above = 0;
    }
  }
}

// The k-th largest of n uint32 keys (MSB-first radix select, 8-bit digits).
// Keys come from the shared cache when it holds them, else from global (L2).
__device__ uint32_t select_kth_key(Smem& S, const uint32_t* gkeys, int n, bool cached, int k) {
  const int gt = fin_tid();
  uint32_t prefix = 0, mask = 0, krem = (uint32_t)k;
  for (int shift = 24; shift >= 0; shift -= 8) {
    S.hist[gt] = 0u;
    S.hist[gt + kFin] = 0u;
    fin_sync();
    for (int i = gt; i < n; i += kFin) {
      const uint32_t key = cached ? S.u.key_cache[i] : __ldcg(gkeys + i);
      if ((key & mask) == prefix) atomicAdd(&S.hist[(key >> shift) & 255u], 1u);
    }
    fin_sync();
    find_digit(S, krem);
    fin_sync();
    krem -= S.digit_above;
    prefix |= S.digit << shift;
    mask |= 255u << shift;
  }
  return prefix;
}

// Visits every logit of a row with key >= tau (head, body, tail), finals-group
// threads in parallel. Used by the exact fallback when the tile filter leaves
// too many candidates (heavily tied rows).
template <int DT, class F>
__device__ __forceinline__ void for_each_row_logit(const RowBody& rb, int V, uint32_t tau, F&& f) {
  constexpr int dtype = DT;
  const int gt = fin_tid();
  const int esize = dtype == 0 ? 2 : 4;
  const int per_vec = 16 / esize;
  for (int j = gt; j < rb.head; j += kFin) {
    uint32_t k = key_of(load_logit(rb.row, j, dtype));
    if (k >= tau) f(k, j);
  }
  for (int j = rb.tail_start + gt; j < V; j += kFin) {
    uint32_t k = key_of(load_logit(rb.row, j, dtype));
    if (k >= tau) f(k, j);
  }
  const uint4* body = reinterpret_cast<const uint4*>(rb.row + (size_t)rb.head * esize);
  for (int v = gt; v < rb.nvec; v += kFin) {
    const uint4 w = __ldg(body + v);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
    const int base = rb.head + v * per_vec;
    if (dtype == 0) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t h = (ws[e >> 1] >> ((e & 1) * 16)) & 0xffffu;
        const uint32_t k = key_of(__uint_as_float(h << 16));
        if (k >= tau) f(k, base + e);
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint32_t k = key_of(__uint_as_float(ws[e]));
        if (k >= tau) f(k, base + e);
      }
    }
  }
}

// Largest of a 16-byte vector of logits (NaN if one is NaN).
template <int DT>
__device__ __forceinline__ float vector_max(const uint4& wv) {
  if (DT == 0) {
    __nv_bfloat162 a = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&wv.x),
                                   *reinterpret_cast<const __nv_bfloat162*>(&wv.y));
    const __nv_bfloat162 b = __hmax2_nan(*reinterpret_cast<const __nv_bfloat162*>(&wv.z),
                                         *reinterpret_cast<const __nv_bfloat162*>(&wv.w));
    a = __hmax2_nan(a, b);
    return max_nan(__low2float(a), __high2float(a));
  }
  return max_nan(max_nan(__uint_as_float(wv.x), __uint_as_float(wv.y)),
                 max_nan(__uint_as_float(wv.z), __uint_as_float(wv.w)));
}

// Body vector of the f-th gathered vector: f / 32 picks the candidate tile,
// f % 32 the vector within it.
__device__ __forceinline__ int candidate_vector(const Smem& S, int f) {
  const int tile = S.cand_tiles[f >> 5];
  const int pc = tile / kTilesPerPiece;
  return pc * kVecPerPiece + tile_vector(tile - pc * kTilesPerPiece, f & 31);
}

// Exclusive prefix over the warp of a count c (0 <= c < 128), from one
// ballot per bit, and the warp's total.
__device__ __forceinline__ int warp_exclusive_count(int c, int lane, int& total) {
  const uint32_t below = (1u << lane) - 1u;
  int pre = 0;
  total = 0;
#pragma unroll
  for (int b = 0; b < 7; ++b) {
    const uint32_t m = __ballot_sync(0xffffffffu, (c >> b) & 1);
    pre += __popc(m & below) << b;
    total += __popc(m) << b;
  }
  return pre;
}

static_assert(sizeof(decltype(Smem::u)) >= sizeof(uint4) * 8 * kFin, "the gather's stage fits the union");

// Bits (as a uint32) of the smallest logit value whose order key is at least
// tau (key of -inf < tau <= key of +inf). A bf16 logit's key is its 16-bit
// key k16 shifted up, with the low half all ones for a negative value and
// zero otherwise (zeros share +0's key); so a negative k16 equal to tau's
// upper half always passes, a non-negative one only when tau's lower half is
// zero. The value of a 16-bit key is the inverse map; the key that -0 would
// have maps to -0, which compares equal to +0 and above every negative.
template <int DT>
__device__ __forceinline__ uint32_t threshold_bits(uint32_t tau) {
  if (DT == 0) {
    const uint32_t t16 = tau >> 16;
    const uint32_t k16 = t16 < 0x8000u ? t16 : t16 + ((tau & 0xffffu) ? 1u : 0u);
    return (k16 & 0x8000u) ? (k16 & 0x7fffu) : (~k16 & 0xffffu);
  }
  return __float_as_uint(value_of_key(tau));
}

// Marks (bit e) of the logits of a 16-byte vector that are >= the threshold
// value: packed bf16 compares, or fp32 compares. NaNs are never marked (a row
// holding one is flagged bad).
template <int DT>
__device__ __forceinline__ uint32_t mark_at_least(const uint4& x, uint32_t thr) {
  if (DT == 0) {
    const __nv_bfloat162 t2 = __halves2bfloat162(__ushort_as_bfloat16((unsigned short)thr),
                                                  __ushort_as_bfloat16((unsigned short)thr));
    const uint32_t ws[4] = {x.x, x.y, x.z, x.w};
    uint32_t m = 0u;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t c = __hge2_mask(*reinterpret_cast<const __nv_bfloat162*>(&ws[q]), t2);
      m |= ((c & 1u) | ((c >> 15) & 2u)) << (2 * q);
    }
    return m;
  }
  const float tf = __uint_as_float(thr);
  return (__uint_as_float(x.x) >= tf ? 1u : 0u) | (__uint_as_float(x.y) >= tf ? 2u : 0u) |
         (__uint_as_float(x.z) >= tf ? 4u : 0u) | (__uint_as_float(x.w) >= tf ? 8u : 0u);
}

// The same marks by order keys (any tau; NaNs compare by their keys).
template <int DT>
__device__ __forceinline__ uint32_t mark_keys_at_least(const uint4& x, uint32_t tau) {
  const uint32_t ws[4] = {x.x, x.y, x.z, x.w};
  constexpr int per_vec = DT == 0 ? 8 : 4;
  uint32_t m = 0u;
#pragma unroll
  for (int e = 0; e < per_vec; ++e) {
    const uint32_t key = DT == 0 ? key_of(__uint_as_float(((ws[e >> 1] >> ((e & 1) * 16)) & 0xffffu) << 16))
                                 : key_of(__uint_as_float(ws[e]));
    m |= (key >= tau ? 1u : 0u) << e;
  }
  return m;
}

// ---- row final ----------------------------------------------------------------------
// Leaves the row's sorted top-k composites in the group's first warp (lane l:
// rank l in `top_a`) and in the workspace.
template <int DT>
__device__ bool row_final(const Params& p, Smem& S, int slot, const SlotInfo& si, unsigned long long& top_a,
                          float& T_row, uint32_t& next) {
  const int gt = fin_tid(), lane = gt & 31, w = gt >> 5;
  const int V = p.geo.V;
  constexpr int dtype = DT;  // the kernel's logit type
  // the row's temperature, loaded now and used last: a global load at the
  // end of the final would add a full round trip to it
  T_row = p.task == kTaskCandidates  // no temperatures: raw logits out
              ? 1.0f
              : ld_nc_now(p.temperature + (p.task == kTaskVerify ? S.req_of_ord[si.ord] : slot));
  // a verification row's position's draft token (target row 2i and draft row
  // 2i + 1 of a request, or target row i with deterministic drafts, are
  // position i's; the bonus row has none)
  const int pos = samp_position(p, si.r);
  const int32_t d_row = (p.task == kTaskVerify && pos < p.gamma)
                            ? ld_nc_now(p.draft_tokens + (size_t)S.req_of_ord[si.ord] * p.gamma + pos)
                            : -1;
  const RowBody rb = row_body(si.ptr, V, p.geo.esize);
  const int n_tiles = p.geo.tiles;
  const uint32_t* gkeys = p.tile_keys + (size_t)slot * n_tiles;
  const bool cached = n_tiles <= kKeyCache;
  const int k = si.k_eff;

  // tile keys (cached) and the logits outside the aligned body, loaded in
  // one round trip; the edges' maximum is all ones when one of them is NaN
  const int n_edge = rb.head + (V - rb.tail_start);
  const int edge_j = gt < rb.head ? gt : rb.tail_start + (gt - rb.head);
  float edge_x = 0.0f;
  if (gt < n_edge) {  // inline-assembly loads stay here, ahead of the poll
    if (DT == 0)
      edge_x = __uint_as_float((uint32_t)ld_nc_now(reinterpret_cast<const unsigned short*>(rb.row) + edge_j) << 16);
    else
      edge_x = ld_nc_now(reinterpret_cast<const float*>(rb.row) + edge_j);
  }
  // The row is ready when every tile key is written: the keys start the call
  // at zero (no tile key is zero: a NaN maximum is the canonical NaN) and a
  // consumer warp stores each one once. So the polls are the final's own key
  // loads, and no counter, fence or second round trip stands between the
  // stream and the final.
  uint32_t mx = 0u;
  const volatile uint32_t* abort_flag = p.abort_flag;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    bool mine = true;
    mx = 0u;
    for (int i = gt; i < n_tiles; i += kFin) {
      const uint32_t key = ld_relaxed_gpu(gkeys + i);
      mine = mine && key != 0u;
      if (cached) S.u.key_cache[i] = key;
      mx = max(mx, key);
    }
    if (fin_sync_and(mine)) break;
    if (fin_sync_or(*abort_flag != 0u || global_timer_ns() - t0 > kWaitLimitNs)) return false;
    __nanosleep(128);
  }
  draw_next_job(p, next);
  const uint32_t emx = gt < n_edge ? (isnan(edge_x) ? 0xffffffffu : key_of(edge_x)) : 0u;
  // the group's largest tile key and edge key (warp maxima in one
  // instruction each), and this job's shared counters reset, behind one
  // barrier; no barrier follows the read of S.warp_red, whose next writer is
  // past a later group barrier
  {
    const uint32_t wm = __reduce_max_sync(0xffffffffu, mx);
    const uint32_t we = __reduce_max_sync(0xffffffffu, emx);
    if (lane == 0) {
      S.warp_red[w] = wm;
      S.warp_red[kFinWarps + w] = we;
    }
    S.hist[gt] = 0u;
    S.hist[gt + kFin] = 0u;
    if (gt == 0) {
      S.n_cand_tiles = 0;
      S.n_cand = 0;
    }
  }
  fin_sync();
  uint32_t tile_max = 0u, edge_max = 0u;
#pragma unroll
  for (int i = 0; i < kFinWarps; ++i) {
    tile_max = max(tile_max, S.warp_red[i]);
    edge_max = max(edge_max, S.warp_red[kFinWarps + i]);
  }
  const bool bad = !key_is_finite(max(tile_max, edge_max));

  // tau: a lower bound of the k-th largest tile key (0 keeps everything when
  // tiles < k). Each thread's largest key counts once: the k largest of those
  // are k distinct tile keys, so the k-th largest of them is at most the
  // row's k-th largest tile key, and that is at most its k-th largest logit.
  // They are counted per bucket of 2^16 key units below the largest (one
  // shared atomic per thread); the bucket where the count from the top
  // reaches k gives tau (exact for bf16 logits, whose keys have zero low 16
  // bits). When they spread wider, an exact radix selection over the tile
  // keys runs instead.
  uint32_t tau = 0u;
  if (k == 1) {
    tau = tile_max;
  } else if (n_tiles >= k) {
    const uint32_t bucket = (tile_max - mx) >> 16;
    if (mx != 0u && bucket < 255u) atomicAdd(&S.hist[bucket], 1u);
    fin_sync();
    if (gt < 32) {
      // inclusive count over buckets 0..b, eight buckets per lane
      uint32_t c[8], run = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = S.hist[lane * 8 + i];
        run += c[i];
      }
      uint32_t incl = run;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t nb = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += nb;
      }
      const uint32_t before = incl - run;
      const bool here = before < (uint32_t)k && (uint32_t)k <= incl;
      if (here) {
        uint32_t acc = before;
        int bkt = lane * 8;
        for (int i = 0; i < 8; ++i) {
          acc += c[i];
          if (acc >= (uint32_t)k) {
            bkt = lane * 8 + i;
            break;
          }
        }
        S.digit = (uint32_t)bkt;
      }
      if (lane == 31 && incl < (uint32_t)k) S.digit = 0xffffffffu;  // top k spread too wide
    }
    fin_sync();
    const uint32_t bkt = S.digit;
    if (bkt != 0xffffffffu) {
      const uint32_t span = (bkt + 1u) << 16;
      tau = tile_max >= span ? tile_max - span + 1u : 0u;
    } else {
      tau = select_kth_key(S, gkeys, n_tiles, cached, k);
    }
  }

  // candidate tiles: each thread marks its tiles (every kFin-th) in a mask;
  // a warp reserves its slots with one atomic (shared atomics on one address
  // serialise) and places its lanes by a prefix of their counts
  for (int base = 0; base < n_tiles; base += kFin * 32) {
    uint32_t mask = 0u;
    const int n_u = min(32, (n_tiles - base - gt + kFin - 1) / kFin);  // this thread's tiles here
    if (cached) {
#pragma unroll 8
      for (int u = 0; u < n_u; ++u)
        if (S.u.key_cache[base + u * kFin + gt] >= tau) mask |= 1u << u;
    } else {
      for (int u = 0; u < n_u; ++u)
        if (__ldcg(gkeys + base + u * kFin + gt) >= tau) mask |= 1u << u;
    }
    int wtotal;
    const int pre = warp_exclusive_count(__popc(mask), lane, wtotal);
    int first = 0;
    if (lane == 0 && wtotal) first = atomicAdd(&S.n_cand_tiles, wtotal);
    int pos = __shfl_sync(0xffffffffu, first, 0) + pre;
    for (; mask; mask &= mask - 1u, ++pos)
      if (pos < kCandTileCap) S.cand_tiles[pos] = base + (__ffs(mask) - 1) * kFin + gt;
  }
  fin_sync();
  const int n_ct = S.n_cand_tiles;
  bool overflow = n_ct > kCandTileCap;
  if (!overflow) {
    // gather: the candidate tiles' 32 vectors each, spread over the group,
    // every load of a round issued before any is used (inline-assembly loads,
    // which the compiler keeps where they stand).
    constexpr int esize = DT == 0 ? 2 : 4, per_vec = 16 / esize;
    const uint4* body = reinterpret_cast<const uint4*>(rb.row + (size_t)rb.head * esize);
    const int n_vec_all = n_ct * 32;
    // The round's vectors wait in shared memory (the key cache is done with,
    // each thread has its own slots), so the marking below is a rolled loop:
    // its code is fetched once and run eight times, where an unrolled one is
    // fetched line by line once per row final.
    uint4* stage = reinterpret_cast<uint4*>(&S.u);  // [8][kFin]
    // key >= tau as a value comparison (one packed compare per two bf16
    // logits): thr is the smallest value whose key is at least tau; a tau at
    // or below the key of -inf, or above that of +inf, keeps the key
    // comparison
    const bool plain_thr = tau > kKeyNegInf && tau <= kKeyPosInf;
    const uint32_t thr = threshold_bits<DT>(tau);
    for (int base = 0; base < n_vec_all; base += kFin * 8) {
      uint4 wv[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int f = base + u * kFin + gt;
        wv[u] = make_uint4(0u, 0u, 0u, 0u);
        if (f < n_vec_all) {
          const int v = candidate_vector(S, f);
          if (v < rb.nvec) wv[u] = ld_nc_now(body + v);
        }
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) stage[u * kFin + gt] = wv[u];
      // marks of the logits at or above tau (bit per_vec u + e), without branches per logit
      unsigned long long cm = 0ull;
#pragma unroll 1
      for (int u = 0; u < 8; ++u) {
        const int f = base + u * kFin + gt;
        if (f >= n_vec_all) break;
        if (candidate_vector(S, f) >= rb.nvec) continue;
        const uint4 x = stage[u * kFin + gt];
        cm |= (unsigned long long)(plain_thr ? mark_at_least<DT>(x, thr) : mark_keys_at_least<DT>(x, tau))
              << (u * per_vec);
      }
      if (cm) {  // few threads: one slot reservation, then the marked logits
        int pos = atomicAdd(&S.n_cand, __popcll(cm));
        for (; cm; cm &= cm - 1ull, ++pos) {
          const int bit = __ffsll(cm) - 1, u = bit / per_vec, e = bit - u * per_vec;
          const uint4 x = stage[u * kFin + gt];
          const int q = dtype == 0 ? e >> 1 : e;
          const uint32_t word = q == 0 ? x.x : q == 1 ? x.y : q == 2 ? x.z : x.w;
          const uint32_t key = key_of(__uint_as_float(dtype == 0 ? (word >> ((e & 1) * 16)) << 16 : word));
          const int v = candidate_vector(S, base + u * kFin + gt);
          if (pos < kCandCap) S.cand[pos] = composite(key, rb.head + v * per_vec + e);
        }
      }
    }
    if (gt < n_edge) {  // head and tail logits are always candidates
      const int pos = atomicAdd(&S.n_cand, 1);
      if (pos < kCandCap) S.cand[pos] = composite(key_of(edge_x), edge_j);
    }
    fin_sync();
    overflow = S.n_cand > kCandCap;
  }
  if (overflow) {
    // exact fallback: radix-select the k-th largest composite over all logits >= tau
    unsigned long long prefix = 0ull, mask = 0ull;
    uint32_t krem = (uint32_t)k;
    for (int shift = 56; shift >= 0; shift -= 8) {
      S.hist[gt] = 0u;
      S.hist[gt + kFin] = 0u;
      fin_sync();
      for_each_row_logit<DT>(rb, V, tau, [&](uint32_t key, int j) {
        const unsigned long long c = composite(key, j);
        if ((c & mask) == prefix) atomicAdd(&S.hist[(uint32_t)(c >> shift) & 255u], 1u);
      });
      fin_sync();
      find_digit(S, krem);
      fin_sync();
      krem -= S.digit_above;
      prefix |= (unsigned long long)S.digit << shift;
      mask |= 255ull << shift;
    }
    if (gt == 0) S.n_cand = 0;
    fin_sync();
    const unsigned long long thr = prefix;
    for_each_row_logit<DT>(rb, V, tau, [&](uint32_t key, int j) {
      const unsigned long long c = composite(key, j);
      if (c >= thr) {
        const int pos = atomicAdd(&S.n_cand, 1);
        if (pos < kCandCap) S.cand[pos] = c;
      }
    });
    fin_sync();
  }
  // sort the (<= 64) candidates: the composites are distinct (each carries
  // its logit's index), so a composite's rank is the number of larger ones;
  // thread c ranks candidate c, and ranks < 32 (k <= 32) are kept in order
  const int n_c = min(S.n_cand, kCandCap);
  if (gt < n_c) {
    const unsigned long long c = S.cand[gt];
    const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(S.cand);
    int r = 0;
#pragma unroll 2
    for (int m = 0; m < (n_c >> 1); ++m) {
      const ulonglong2 v = c2[m];
      r += (v.x > c ? 1 : 0) + (v.y > c ? 1 : 0);
    }
    if (n_c & 1) r += S.cand[n_c - 1] > c ? 1 : 0;
    if (r < 32) S.sorted[r] = c;
  }
  fin_sync();
  if (w == 0) {
    const unsigned long long a = lane < n_c ? S.sorted[lane] : 0ull;
    top_a = a;
    if (p.task == kTaskVerify) {
      // the row's filtered distribution (ranks < k, k <= 32), which the
      // request final reads
      const bool valid = lane < k && lane < n_c;
      int32_t idx = valid ? composite_idx(a) : -1;
      const float pr = filter_lane(valid ? composite_key(a) : 0u, idx, k, T_row, p.top_p, lane, S.exp_hi, S.exp_lo);
      const uint32_t lo = __float_as_uint(pr) | ((bad && lane == 0) ? 0x80000000u : 0u);
      unsigned long long* list = p.res_list + (size_t)slot * kListWords;
      list[lane] = ((unsigned long long)(uint32_t)(idx + 2) << 32) | lo;
      // the probability of the position's draft token, for the accept test
      const uint32_t hit = __ballot_sync(0xffffffffu, idx >= 0 && idx == d_row);
      const float pd = hit ? __shfl_sync(0xffffffffu, pr, __ffs(hit) - 1) : 0.0f;
      if (lane == 0) list[kMaxTopK] = (1ull << 32) | __float_as_uint(pd);
    }
    if (p.task == kTaskCandidates) {
      // a vocabulary shard's top k as (logit, global token), then its largest
      // logit: whether the whole row is bad is decided once the shards meet
      const bool valid = lane < k && lane < n_c;
      if (lane < k) {
        p.out_prob[(size_t)slot * k + lane] = valid ? value_of_key(composite_key(a)) : -INFINITY;
        p.out_idx[(size_t)slot * k + lane] = valid ? composite_idx(a) + p.vocab_offset : -1;
      }
      if (lane == 0) p.out_rowmax[slot] = value_of_key(max(tile_max, edge_max));
    } else if (bad && lane == 0 && p.status) {
      atomicOr(p.status, kStatusBadRow);
    }
  }
  // leave the keys at zero for the next call
  uint32_t* wkeys = p.tile_keys + (size_t)slot * n_tiles;
  for (int i = gt; i < n_tiles; i += kFin) wkeys[i] = 0u;
  fin_sync();
  return true;
}

// ---- request final (sampling verification) -------------------------------------------
// The rows arrive filtered (kept tokens and probabilities). One lane per draft
// position runs the accept test u < p(d)/q(d); the first failing position (or
// gamma when none fails) is where the residual max(0, p - q) (or the bonus
// distribution p) is drawn from. With deterministic drafts q is the point
// mass at d: the test is u < p(d) and the residual is p with d taken out.
__device__ bool request_final(const Params& p, Smem& S, int ord, uint32_t& next) {
  const int gt = fin_tid(), lane = gt & 31, w = gt >> 5;
  const int gamma = p.gamma, V = p.geo.V;
  const int b = S.req_of_ord[ord];
  int32_t* out = p.out_tokens + (size_t)b * (gamma + 1);
  const int32_t* d = p.draft_tokens + (size_t)b * gamma;
  const int per_s = samp_slots(p);
  const int slot0 = ord * per_s;
  // The rows' filtered lists are ready when every word is written (no
  // written word is zero): the polls are the final's own loads.
  unsigned long long* words = p.res_list + (size_t)slot0 * kListWords;
  const int n_words = per_s * kListWords;
  // the drafts, loaded before the wait (after it they would add a round trip),
  // and lane l's counter-based words for position l (accept: x, draw: y)
  const int32_t d_lane = (w == 0 && lane < gamma) ? ld_nc_now(d + lane) : -1;
  uint4 wd = make_uint4(0u, 0u, 0u, 0u);
  if (w == 0 && lane <= gamma) wd = step_uniform_words(p.seed, (uint32_t)b, (uint32_t)lane, 0u);
  const volatile uint32_t* abort_flag = p.abort_flag;
  const unsigned long long t0 = global_timer_ns();
  for (;;) {
    bool mine = true;
    for (int i = gt; i < n_words; i += kFin) {
      const unsigned long long v = ld_relaxed_gpu_u64(words + i);
      mine = mine && v != 0ull;
      const int r = i / kListWords, l = i - r * kListWords;
      // column 32: the prob. of the row's draft token (prob) and the row's bad flag (idx)
      S.u.lists.prob[r][l] = __uint_as_float((uint32_t)v & 0x7fffffffu);
      if (l < kMaxTopK) S.u.lists.idx[r][l] = (int32_t)(uint32_t)(v >> 32) - 2;
      if (l == 0) S.u.lists.idx[r][32] = (int32_t)((uint32_t)v >> 31);
    }
    if (fin_sync_and(mine)) break;
    if (fin_sync_or(*abort_flag != 0u || global_timer_ns() - t0 > kWaitLimitNs)) return false;
    __nanosleep(128);
  }
  draw_next_job(p, next);
  // every call leaves the workspace at zero: its regions move with the
  // shape, and another shape's tile keys may lie here next time
  for (int i = gt; i < n_words; i += kFin) words[i] = 0ull;
  if (w == 0)
    sampling_rule(S.u.lists.idx, S.u.lists.prob, per_s, p.det != 0, gamma, V, d_lane, wd, p.seed, b, lane,
                  S.cand, out, p.out_len, p.status, p.audit_pq ? p.audit_pq + (size_t)b * gamma * 2 : nullptr);
  fin_sync();
  return true;
}

// ---- row final of the rows tasks: filtered distribution / one sample ----------------
__device__ void rows_final(const Params& p, Smem& S, int r, unsigned long long top_a, float T) {
  const int gt = fin_tid(), lane = gt & 31;
  if ((gt >> 5) == 0) {
    const bool samp = sampling_temperature(T);
    const uint32_t st = (!samp && T != 0.0f) ? kStatusBadTemperature : 0u;
    const int k_eff = samp ? p.top_k : 1;
    const int n_c = min(S.n_cand, kCandCap);
    const uint32_t key = (lane < k_eff && lane < n_c) ? composite_key(top_a) : 0u;
    int32_t idx = (lane < k_eff && lane < n_c) ? composite_idx(top_a) : -1;
    float pr;
    if (samp) {
      pr = filter_lane(key, idx, k_eff, T, p.top_p, lane, S.exp_hi, S.exp_lo);
    } else {
      pr = lane == 0 ? 1.0f : 0.0f;
      if (lane != 0) idx = -1;
    }
    if (p.task == kTaskFilter) {
      const int cnt = __popc(__ballot_sync(0xffffffffu, idx >= 0));
      if (lane < p.top_k) {
        p.out_idx[(size_t)r * p.top_k + lane] = idx;
        p.out_prob[(size_t)r * p.top_k + lane] = idx >= 0 ? pr : 0.0f;
      }
      if (lane == 0) p.out_count[r] = cnt;
    } else {
      int32_t tok;
      if (samp) {
        const uint4 wd = step_uniform_words(p.seed, 0u, (uint32_t)(p.row_base + r), 1u);
        tok = draw_ascending(idx, pr, uniform24(wd.x), lane, reinterpret_cast<int32_t*>(S.cand),
                             reinterpret_cast<float*>(S.cand) + 32);
        if (tok < 0) tok = __shfl_sync(0xffffffffu, idx, 0);
      } else {
        tok = __shfl_sync(0xffffffffu, idx, 0);
      }
      if (lane == 0) p.out_tokens[r] = tok;
    }
    if (lane == 0 && st && p.status) atomicOr(p.status, st);
  }
  fin_sync();
}

// ---- roles ---------------------------------------------------------------------------
__device__ __forceinline__ void raise_timeout(const Params& p) {
  atomicExch(p.abort_flag, 1u);
  if (p.status) atomicOr(p.status, kStatusTimeout);
}

// Greedy rows of a verification get their argmax in the stream (no row final).
__device__ __forceinline__ bool in_stream_argmax(const Params& p, const SlotInfo& si) {
  return (p.task == kTaskVerify || p.task == kTaskVerifyGreedy) && !si.sampling;
}

// A CTA's pieces are blockIdx.x, blockIdx.x + G, ... (G = gridDim.x); their
// (slot, piece-in-row) pairs advance without divisions.
struct PieceWalk {
  int slot, pp, dslot, dpp, ppr;
  __device__ __forceinline__ PieceWalk(int ppr_) : ppr(ppr_) {
    slot = (int)(blockIdx.x / (unsigned)ppr_);
    pp = (int)(blockIdx.x - (unsigned)slot * ppr_);
    dslot = (int)(gridDim.x / (unsigned)ppr_);
    dpp = (int)(gridDim.x - (unsigned)dslot * ppr_);
  }
  __device__ __forceinline__ void next() {
    slot += dslot;
    pp += dpp;
    if (pp >= ppr) {
      pp -= ppr;
      ++slot;
    }
  }
};

// Producer warp: lane 0 issues the bulk copies, one per piece. The index
// arithmetic of a piece (slot, request, row pointer, body geometry, flags) is
// a few hundred cycles of dependent scalar work, which on one thread would
// cap the stream well below HBM bandwidth; so the warp prepares the next 32
// pieces in parallel, one per lane, and lane 0 only waits for the stage,
// writes its descriptor and issues the copy.
__device__ void producer(const Params& p, Smem& S, long long total) {
  const int lane = threadIdx.x & 31;
  const volatile uint32_t* abort_flag = p.abort_flag;
  const long long mine = total > blockIdx.x ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  const int ppr = p.geo.ppr;
  bool aborted = false;
  long long it = 0;
  for (long long base = 0; base < mine && !aborted; base += 32) {
    // lane l: piece base + l of this CTA
    const unsigned char* src = nullptr;
    int slot = 0, pp = 0, nvec = 0, head = 0, ord = 0;
    if (base + lane < mine) {
      const long long piece = blockIdx.x + (base + lane) * (long long)gridDim.x;
      slot = (int)(piece / ppr);
      pp = (int)(piece - (long long)slot * ppr);
      const SlotInfo si = slot_info(p, S, slot);
      const RowBody rb = row_body(si.ptr, p.geo.V, p.geo.esize);
      const int v0 = pp * kVecPerPiece;
      nvec = max(0, min(kVecPerPiece, rb.nvec - v0));
      int flags = 0;
      if (in_stream_argmax(p, si))
        flags = kDescArgmax;
      else if (p.fullvocab && si.sampling)
        flags = kDescStats;
      head = rb.head + flags;
      ord = si.ord;
      src = rb.row + (size_t)rb.head * p.geo.esize + (size_t)v0 * 16;
    }
    const int n = (int)min(32ll, mine - base);
    for (int j = 0; j < n; ++j, ++it) {
      const unsigned char* src_j = reinterpret_cast<const unsigned char*>(
          __shfl_sync(0xffffffffu, reinterpret_cast<unsigned long long>(src), j));
      const int slot_j = __shfl_sync(0xffffffffu, slot, j);
      const int pp_j = __shfl_sync(0xffffffffu, pp, j);
      const int nvec_j = __shfl_sync(0xffffffffu, nvec, j);
      const int head_j = __shfl_sync(0xffffffffu, head, j);
      const int ord_j = __shfl_sync(0xffffffffu, ord, j);
      int ok = 1;
      if (lane == 0) {
        const int stage = (int)(it % kStages);
        const uint32_t round = (uint32_t)(it / kStages);
        if (!mbar_wait(&S.empty[stage], (round & 1u) ^ 1u, abort_flag)) {
          ok = 0;
        } else {
          S.desc[stage].slot = slot_j;
          S.desc[stage].pp = pp_j;
          S.desc[stage].nvec = nvec_j;
          S.desc[stage].head = head_j;
          S.desc[stage].ord = ord_j;
          if (nvec_j > 0) {
            mbar_arrive_expect_tx(&S.full[stage], (uint32_t)nvec_j * 16u);
            bulk_load(S.ring[stage], src_j, (uint32_t)nvec_j * 16u, &S.full[stage]);
          } else {
            mbar_arrive(&S.full[stage]);
          }
        }
      }
      if (!__shfl_sync(0xffffffffu, ok, 0)) {
        aborted = true;
        break;
      }
    }
  }
  if (lane == 0) {
    // Every copy issued must land before the CTA's shared memory goes away,
    // also when the consumers stopped early (abort or timeout, possibly after
    // the last copy was issued). Only the last kStages can be in flight; in
    // a call that ran through, they have landed already.
    const long long first = it > kStages ? it - kStages : 0;
    for (long long q = first; q < it; ++q)
      (void)mbar_wait_landed(&S.full[q % kStages], (uint32_t)((q / kStages) & 1));
  }
}


// Tile keys of a piece: per block of 4 rounds, each 8-lane group's maximum is
// one tile key. For greedy rows (argmax) the warp instead folds the piece's
// (largest key, lowest vector holding it) into the row's running argmax.
template <int DT>
__device__ __forceinline__ void piece_keys(const Params& p, const uint4* st4, int nvec, int slot, int pp,
                                           bool argmax, int head, int lane) {
  uint32_t* keys_out = p.tile_keys + (size_t)slot * p.geo.tiles + pp * kTilesPerPiece;
  uint32_t best_key = 0u;  // greedy: this lane's largest key, its lowest vector and that vector
  int best_v = 0;
  uint4 best_w = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll 2
  for (int blk = 0; blk < kTilesPerPiece / 4; ++blk) {
    uint4 wv[4];
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int v = 32 * (4 * blk + rr) + lane;
      if (v < nvec) wv[rr] = st4[v];
    }
    float m = -INFINITY;
    if (DT == 0 && !argmax && 32 * (4 * blk + 3) + lane < nvec) {
      // a whole block of bf16 logits: one packed maximum over its 16 words,
      // converted to fp32 once (NaN propagates through every step)
      __nv_bfloat162 acc = *reinterpret_cast<const __nv_bfloat162*>(&wv[0].x);
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        acc = __hmax2_nan(acc, *reinterpret_cast<const __nv_bfloat162*>(&wv[rr].x));
        acc = __hmax2_nan(acc, *reinterpret_cast<const __nv_bfloat162*>(&wv[rr].y));
        acc = __hmax2_nan(acc, *reinterpret_cast<const __nv_bfloat162*>(&wv[rr].z));
        acc = __hmax2_nan(acc, *reinterpret_cast<const __nv_bfloat162*>(&wv[rr].w));
      }
      m = max_nan(__low2float(acc), __high2float(acc));
    } else {
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int v = 32 * (4 * blk + rr) + lane;
        if (v < nvec) {
          const float vmax = vector_max<DT>(wv[rr]);
          m = max_nan(m, vmax);
          if (argmax) {
            const uint32_t k = key_of(vmax);
            if (k > best_key) {
              best_key = k;
              best_v = v;
              best_w = wv[rr];
            }
          }
        }
      }
    }
    if (!argmax) {
      uint32_t key = key_of(m);
      key = max(key, __shfl_xor_sync(0xffffffffu, key, 1));
      key = max(key, __shfl_xor_sync(0xffffffffu, key, 2));
      key = max(key, __shfl_xor_sync(0xffffffffu, key, 4));
      if ((lane & (kTileLanes - 1)) == 0) keys_out[4 * blk + (lane >> 3)] = key;
    }
  }
  if (argmax) {
    // the lowest logit of the best vector that holds its key (none does for a
    // NaN maximum: its first logit stands in, and the row is flagged bad)
    constexpr int per_vec = DT == 0 ? 8 : 4;
    const uint32_t ws[4] = {best_w.x, best_w.y, best_w.z, best_w.w};
    int e_hit = 0;
#pragma unroll
    for (int e = per_vec - 1; e >= 0; --e) {
      const float x = DT == 0 ? __uint_as_float(((ws[e >> 1] >> ((e & 1) * 16)) & 0xffffu) << 16) : __uint_as_float(ws[e]);
      if (key_of(x) == best_key) e_hit = e;
    }
    unsigned long long comp =
        best_key ? composite(best_key, head + (pp * kVecPerPiece + best_v) * per_vec + e_hit) : 0ull;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const unsigned long long oc = shfl_xor_u64(comp, o);
      comp = oc > comp ? oc : comp;
    }
    if (lane == 0 && comp) red_max_gpu(p.row_best + slot, comp);
  }
}

// Full-vocabulary rows: a piece's largest logit m and its sum of
// exp((x - m) / T) = 2^((x - m) s), s = log2(e) / T, written as one float4
// per piece (m, the sum as a float-float pair, NaN flag).
//
// bf16 rows (two passes over the stage): the piece's maximum comes first,
// so no sum is rescaled; the weights (2^x on the special-function unit) of
// a lane's block are added pairwise, the block sums are accumulated and the
// lanes merged in float-float.
template <int DT>
__device__ __forceinline__ void piece_stats_two_pass(const uint4* st4, int nvec, const float* temperature, float4* out,
                                            int lane) {
  const float s = __fdiv_rn(kLog2eHi, __ldg(temperature));  // log2(e) / T, rounded
  float m = -INFINITY;
#pragma unroll 4
  for (int r = 0; r < kRoundsPerPiece; ++r) {
    const int v = 32 * r + lane;
    if (v < nvec) m = max_nan(m, vector_max<DT>(st4[v]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
  ff acc = {0.0f, 0.0f};
  if (m > -INFINITY && m < INFINITY) {  // the same in every lane
#pragma unroll 2
    for (int blk = 0; blk < kTilesPerPiece / 4; ++blk) {
      float bs[4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const int v = 32 * (4 * blk + rr) + lane;
        bs[rr] = 0.0f;
        if (v < nvec) {
          const uint4 wv = st4[v];
          const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
          float e[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (DT == 0)
              e[q] = __fadd_rn(ex2_approx(__fmul_rn(__uint_as_float(ws[q] << 16) - m, s)),
                               ex2_approx(__fmul_rn(__uint_as_float(ws[q] & 0xffff0000u) - m, s)));
            else
              e[q] = ex2_approx(__fmul_rn(__uint_as_float(ws[q]) - m, s));
          }
          bs[rr] = __fadd_rn(__fadd_rn(e[0], e[1]), __fadd_rn(e[2], e[3]));
        }
      }
      acc = ff_add(acc, two_sum(__fadd_rn(bs[0], bs[1]), __fadd_rn(bs[2], bs[3])));
    }
  }
  // the lanes share m: a float-float tree, lane 0's result
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const ff b = shfl_down_ff(acc, o);
    if (lane + o < 32) acc = ff_add(acc, b);
  }
  if (lane == 0) *out = make_float4(m, acc.hi, acc.lo, isnan(m) ? 1.0f : 0.0f);
}

// fp32 rows (one pass over the stage, which their stream needs: a second
// pass over 4 bytes a logit costs more issue slots than the stream has to
// spare): per block of 4 rounds each lane takes its 16 logits' maximum b and
// their weights 2^((x - b) s) (the special-function unit's 2^x), added
// pairwise; once the piece's maximum is known each block sum is scaled once
// by 2^((b - m) s) and the products are accumulated and the lanes merged in
// float-float. Every weight then carries two 2^x roundings instead of one,
// and its exponent the same roundings as (x - m) s, split in two parts of one
// sign.
template <int DT>
__device__ __forceinline__ void piece_stats_one_pass(const uint4* st4, int nvec, const float* temperature, float4* out,
                                            int lane) {
  const float s = __fdiv_rn(kLog2eHi, __ldg(temperature));  // log2(e) / T, rounded
  constexpr int kBlocks = kTilesPerPiece / 4;
  float bmax[kBlocks], bsum[kBlocks];
  float m = -INFINITY;
#pragma unroll
  for (int blk = 0; blk < kBlocks; ++blk) {
    uint4 wv[4];
    float b = -INFINITY;
#pragma unroll
    for (int rr = 0; rr < 4; ++rr) {
      const int v = 32 * (4 * blk + rr) + lane;
      const uint32_t pad = DT == 0 ? 0xff80ff80u : 0xff800000u;  // -inf past the piece: weight 0
      wv[rr] = v < nvec ? st4[v] : make_uint4(pad, pad, pad, pad);
      b = max_nan(b, vector_max<DT>(wv[rr]));
    }
    float bs = 0.0f;
    if (b > -INFINITY && b < INFINITY) {
      float r4[4];
#pragma unroll
      for (int rr = 0; rr < 4; ++rr) {
        const uint32_t ws[4] = {wv[rr].x, wv[rr].y, wv[rr].z, wv[rr].w};
        float e[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (DT == 0)
            e[q] = __fadd_rn(ex2_approx(__fmul_rn(__uint_as_float(ws[q] << 16) - b, s)),
                             ex2_approx(__fmul_rn(__uint_as_float(ws[q] & 0xffff0000u) - b, s)));
          else
            e[q] = ex2_approx(__fmul_rn(__uint_as_float(ws[q]) - b, s));
        }
        r4[rr] = __fadd_rn(__fadd_rn(e[0], e[1]), __fadd_rn(e[2], e[3]));
      }
      bs = __fadd_rn(__fadd_rn(r4[0], r4[1]), __fadd_rn(r4[2], r4[3]));
    }
    bmax[blk] = b;
    bsum[blk] = bs;
    m = max_nan(m, b);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = max_nan(m, __shfl_xor_sync(0xffffffffu, m, o));
  ff acc = {0.0f, 0.0f};
  if (m > -INFINITY && m < INFINITY) {  // the same in every lane
#pragma unroll
    for (int blk = 0; blk < kBlocks; ++blk)
      if (bsum[blk] > 0.0f) {
        const float sc = ex2_approx(__fmul_rn(bmax[blk] - m, s));
        const float prod = __fmul_rn(bsum[blk], sc);
        acc = ff_add(acc, ff{prod, __fmaf_rn(bsum[blk], sc, -prod)});
      }
  }
  // the lanes share m: a float-float tree, lane 0's result
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const ff b = shfl_down_ff(acc, o);
    if (lane + o < 32) acc = ff_add(acc, b);
  }
  if (lane == 0) *out = make_float4(m, acc.hi, acc.lo, isnan(m) ? 1.0f : 0.0f);
}

// Both forms keep the per-weight error within the accept test's derived
// bound. The request's temperature is fetched here, by the consumer warp,
// not by the producer: a dependent load per piece on the single thread that
// issues the bulk copies slows the whole stream. (The one-pass form takes 34
// more registers, which the bf16 instantiation, the headline's, is spared.)
template <int DT>
__device__ __forceinline__ void piece_stats(const uint4* st4, int nvec, const float* temperature, float4* out,
                                            int lane) {
  if constexpr (DT == 0)
    piece_stats_two_pass<DT>(st4, nvec, temperature, out, lane);
  else
    piece_stats_one_pass<DT>(st4, nvec, temperature, out, lane);
}

// Consumer warp: reduces whole pieces (this warp takes every 8th piece of the
// CTA) to tile keys, a greedy row's running argmax, or a full-vocabulary
// row's (max, sum of exp).
template <int DT>
__device__ void consumer(const Params& p, Smem& S, long long total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const volatile uint32_t* abort_flag = p.abort_flag;
  const long long mine = total > blockIdx.x ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  for (long long it = warp; it < mine; it += kConsumerWarps) {
    const int stage = (int)(it % kStages);
    const int q = (int)(it % kKeyQueue);
    const uint32_t round = (uint32_t)(it / kStages);
    // A parity wait only tells adjacent phases apart. Bulk copies may land
    // out of order, so this stage's previous piece (it - kStages, another
    // warp's) might not have landed yet, and a full-barrier wait for piece it
    // would then match the phase before and pass at once. Waiting first for
    // that piece to be consumed (empty barrier) closes the gap; that wait is
    // itself unambiguous because piece it - 2 kStages was this warp's own.
    bool landed = true;
    if (it >= kStages) landed = mbar_wait(&S.empty[stage], (round & 1u) ^ 1u, abort_flag);
    landed = landed && mbar_wait(&S.full[stage], round & 1u, abort_flag);
    if (!__all_sync(0xffffffffu, landed)) {
      if (lane == 0) raise_timeout(p);
      return;
    }
    const PieceDesc dsc = S.desc[stage];
    const int nvec = dsc.nvec;
    const uint4* st4 = reinterpret_cast<const uint4*>(S.ring[stage]);
    if (dsc.head & kDescStats)
      piece_stats<DT>(st4, nvec, p.temperature + S.req_of_ord[dsc.ord],
                      reinterpret_cast<float4*>(p.tile_keys + (size_t)dsc.slot * p.geo.tiles) + dsc.pp, lane);
    else
      piece_keys<DT>(p, st4, nvec, dsc.slot, dsc.pp, (dsc.head & kDescArgmax) != 0, dsc.head & (kDescArgmax - 1),
                     lane);
    __syncwarp();  // the stage is read and the keys are stored before lane 0 signals
    int ok = 1;
    if (lane == 0) {
      mbar_arrive(&S.empty[stage]);
      // the publisher must have taken queue slot q's previous piece
      if (!mbar_wait(&S.kempty[q], ((uint32_t)(it / kKeyQueue) & 1u) ^ 1u, abort_flag)) {
        raise_timeout(p);
        ok = 0;
      } else {
        mbar_arrive(&S.kfull[q]);
      }
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return;
  }
}

// Rows whose finals wait for their pieces to be counted: greedy rows of a
// verification (argmax in the stream) and full-vocabulary sampling rows. Rows
// with a row final (top-k sampling rows, rows tasks) signal readiness through
// their tile keys instead.
__device__ __forceinline__ bool counted_slot(const Params& p, const Smem& S, int slot) {
  if (p.task != kTaskVerify && p.task != kTaskVerifyGreedy) return false;
  return slot >= S.n_samp * samp_slots(p) || p.fullvocab != 0;
}

// Publisher (one thread): takes the pieces the consumers finished in batches,
// releases their tile keys (and greedy argmax updates) to the other CTAs with
// one fence per batch, then counts the pieces on their rows with
// fire-and-forget reductions, so it never waits for a reply.
__device__ void publisher(const Params& p, Smem& S, long long total) {
  if ((threadIdx.x & 31) != 0) return;
  const int ppr = p.geo.ppr;
  const volatile uint32_t* abort_flag = p.abort_flag;
  const long long mine = total > blockIdx.x ? (total - blockIdx.x + gridDim.x - 1) / gridDim.x : 0;
  PieceWalk w(ppr);
  long long q = 0;
  while (q < mine) {
    int n = 0;
    if (mbar_wait(&S.kfull[q % kKeyQueue], (uint32_t)((q / kKeyQueue) & 1), abort_flag)) {
      n = 1;
      while (q + n < mine && n < kKeyQueue &&
             mbar_test_wait(&S.kfull[(q + n) % kKeyQueue], (uint32_t)(((q + n) / kKeyQueue) & 1)))
        ++n;
    }
    if (n == 0) {
      raise_timeout(p);
      return;
    }
    // rows whose finals wait on counts: release what the batch's consumers
    // wrote (greedy argmax, full-vocabulary statistics), then count
    PieceWalk w2 = w;
    bool counted = false;
    for (int j = 0; j < n; ++j, w2.next()) counted = counted || counted_slot(p, S, w2.slot);
    if (counted) fence_acq_rel_gpu();
    for (int j = 0; j < n; ++j) {
      if (counted_slot(p, S, w.slot)) red_add_gpu(p.row_cnt + w.slot, 1u);
      w.next();
      mbar_arrive(&S.kempty[(q + j) % kKeyQueue]);
    }
    q += n;
  }
}

// Waits (bounded) until `n` consecutive rows from `slot0` have all their
// pieces counted, then returns their counters to zero. Run by one warp.
__device__ __forceinline__ bool wait_rows(const Params& p, int slot0, int n) {
  if (p.keys_ready) return true;  // written by the kernel before this one; nothing was counted
  const int lane = threadIdx.x & 31;
  const volatile uint32_t* abort_flag = p.abort_flag;
  const uint32_t need = (uint32_t)p.geo.ppr;
  const unsigned long long t0 = global_timer_ns();
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    bool done = i >= n || ld_acquire_gpu(p.row_cnt + slot0 + i) >= need;
    while (!__all_sync(0xffffffffu, done)) {
      // the give-up decision is the warp's, so every lane leaves together
      const bool stop = *abort_flag != 0u || global_timer_ns() - t0 > kWaitLimitNs;
      if (__any_sync(0xffffffffu, stop)) return false;
      __nanosleep(64);
      if (!done) done = ld_acquire_gpu(p.row_cnt + slot0 + i) >= need;
    }
  }
  for (int i = lane; i < n; i += 32) p.row_cnt[slot0 + i] = 0u;  // ready for the next call
  return true;
}

// Final of a greedy request: its rows' argmax came from the stream (plus the
// logits outside each row's aligned body); prefix-match the drafts.
template <int DT>
__device__ void greedy_request_final(const Params& p, Smem& S, int ord) {
  const int lane = fin_tid() & 31;
  const int gamma = p.gamma, V = p.geo.V;
  const int b = S.req_of_ord[ord];
  const int slot0 = S.n_samp * samp_slots(p) + (ord - S.n_samp) * (gamma + 1);
  int32_t* out = p.out_tokens + (size_t)b * (gamma + 1);
  const int32_t* d = p.draft_tokens + (size_t)b * gamma;
  const size_t row_bytes = (size_t)V * p.geo.esize;
  // inputs loaded first, so none of them adds a round trip at the end
  const float T_b = p.task == kTaskVerify ? ld_nc_now(p.temperature + b) : 0.0f;  // greedy task: no temperatures
  const int32_t d_lane = lane < gamma ? ld_nc_now(d + lane) : -1;
  uint32_t st = 0;
  if (p.task == kTaskVerify && T_b != 0.0f) st |= kStatusBadTemperature;
  int n = gamma;  // length of the matching prefix
  int32_t am[2] = {-1, -1};  // argmax of rows lane and lane + 32
  for (int base = 0, u = 0; base <= gamma; base += 32, ++u) {
    const int i = base + lane;
    bool mismatch = false;
    if (i <= gamma) {
      // the stream left (largest key, lowest logit of the body holding it)
      const unsigned long long vbest = ld_acquire_gpu_u64(p.row_best + slot0 + i);
      p.row_best[slot0 + i] = 0ull;  // ready for the next call
      const RowBody rb = row_body(p.target + ((size_t)b * (gamma + 1) + i) * row_bytes, V, p.geo.esize);
      bool nan = false;
      unsigned long long comp = vbest;
      for (int j = 0; j < rb.head; ++j) {
        const float x = load_logit(rb.row, j, DT);
        nan |= isnan(x);
        const unsigned long long c = composite(key_of(x), j);
        comp = c > comp ? c : comp;
      }
      for (int j = rb.tail_start; j < V; ++j) {
        const float x = load_logit(rb.row, j, DT);
        nan |= isnan(x);
        const unsigned long long c = composite(key_of(x), j);
        comp = c > comp ? c : comp;
      }
      if (nan || !key_is_finite(composite_key(comp))) st |= kStatusBadRow;
      am[u] = composite_idx(comp);
      if (am[u] < 0 || am[u] >= V) am[u] = 0;
    }
    if (i < gamma) {  // gamma <= 32: i == lane
      const int32_t di = d_lane;
      if (di < 0 || di >= V) st |= kStatusBadToken;
      mismatch = di != am[u];
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
    if (p.out_len) p.out_len[b] = n + 1;
    if (st && p.status) atomicOr(p.status, st);
    if (p.fullvocab) p.fv_draw[b] = FvDraw{n, kFvNone, 0.0f, 0.0f, 0.0f, 0.0f, -1};
  }
}

// Final of a full-vocabulary sampling request (finals group): each row's
// (max, sum of exp) from its pieces' statistics and the logits outside its
// aligned body, then the accept test at every draft position at once (lane i:
// u_i < p_i(d_i) / q_i(d_i)). Emits the accepted drafts and the accept length
// and leaves the draw at the first rejected position (residual) or at the
// bonus position to the second pass, with the rows' maxima.
template <int DT>
__device__ void fullvocab_request_final(const Params& p, Smem& S, int ord) {
  const int gt = fin_tid(), lane = gt & 31, w = gt >> 5;
  const int gamma = p.gamma, V = p.geo.V, per_s = samp_slots(p);
  const bool det = p.det != 0;  // deterministic drafts: target rows only, q(d) = 1
  const int b = S.req_of_ord[ord];
  const int slot0 = ord * per_s;
  const float T_b = ld_nc_now(p.temperature + b);
  const int32_t d_lane = (w == 0 && lane < gamma) ? ld_nc_now(p.draft_tokens + (size_t)b * gamma + lane) : -1;
  // each row's largest logit m and normaliser sum exp((x - m) / T), from its
  // pieces' (m_p, sum_p) and the logits outside its aligned body: every
  // piece's sum is rescaled by exp((m_p - m) / T) and added in float-float
  for (int r = w; r < per_s; r += kFinWarps) {
    const SlotInfo si = slot_info(p, S, slot0 + r);
    const RowBody rb = row_body(si.ptr, V, p.geo.esize);
    float4* st = reinterpret_cast<float4*>(p.tile_keys + (size_t)(slot0 + r) * p.geo.tiles);
    const int n_edge = rb.head + (V - rb.tail_start);
    bool nan = false;
    float m = -INFINITY;
    for (int pp = lane; pp < p.geo.ppr; pp += 32) {
      const float4 v = __ldcg(st + pp);
      nan |= v.w != 0.0f || isnan(v.x);
      m = fmaxf(m, v.x);
    }
    for (int e = lane; e < n_edge; e += 32) {
      const float x = load_logit(rb.row, e < rb.head ? e : rb.tail_start + (e - rb.head), DT);
      nan |= isnan(x);
      m = fmaxf(m, x);
    }
    m = warp_max_f32(m);
    nan = __any_sync(0xffffffffu, nan);
    ff sum = {0.0f, 0.0f};
    if (!nan && m > -INFINITY && m < INFINITY) {
      for (int pp = lane; pp < p.geo.ppr; pp += 32) {
        const float4 v = __ldcg(st + pp);
        if (v.x > -INFINITY) sum = ff_add(sum, ff_mul(ff{v.y, v.z}, exp_diff_ff(v.x, m, T_b, S.exp_hi, S.exp_lo)));
      }
      for (int e = lane; e < n_edge; e += 32) {
        const float x = load_logit(rb.row, e < rb.head ? e : rb.tail_start + (e - rb.head), DT);
        sum = ff_add(sum, exp_diff_ff(x, m, T_b, S.exp_hi, S.exp_lo));
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const ff o2 = shfl_down_ff(sum, o);
      if (lane + o < 32) sum = ff_add(sum, o2);
    }
    // leave the region at zero: rows of later calls take tile keys there
    for (int pp = lane; pp < p.geo.ppr; pp += 32) st[pp] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
    if (lane == 0) {
      const int bad = (nan || !(fabsf(m) < INFINITY) || !(sum.hi > 0.0f)) ? 1 : 0;
      S.u.fv.m[r] = m;
      S.u.fv.s[r] = sum.hi;
      S.u.fv.s_lo[r] = sum.lo;
      S.u.fv.bad[r] = bad;
      // top-p over the full vocabulary: the rows' cuts come first (other
      // kernels), and with them the accept tests
      if (p.fvtp) p.fvtp_rows[(size_t)b * per_s + r] = make_float4(m, sum.hi, sum.lo, bad ? 1.0f : 0.0f);
    }
  }
  fin_sync();
  if (p.fvtp) return;
  if (w == 0) {
    int32_t* out = p.out_tokens + (size_t)b * (gamma + 1);
    uint32_t st = 0;
    for (int r = lane; r < per_s; r += 32)
      if (S.u.fv.bad[r]) st |= kStatusBadRow;
    bool stop = false;
    if (lane < gamma) {
      const int i = lane;
      const int ti = det ? i : 2 * i;  // position i's target row
      const int32_t di = d_lane;
      const bool valid = di >= 0 && di < V;
      if (!valid) st |= kStatusBadToken;
      if (S.u.fv.bad[ti] || (!det && S.u.fv.bad[2 * i + 1])) {
        stop = true;  // a bad row ends the loop at its position
      } else {
        // a token outside the vocabulary has p = q = 0; a deterministic draft has q = 1
        // p(d) = exp((x_d - m) / T) / sum, in float-float, rounded once
        float p_d = 0.0f, q_d = det ? 1.0f : 0.0f;
        if (valid) {
          const SlotInfo sx = slot_info(p, S, slot0 + ti);
          p_d = ff_round(ff_mul(exp_diff_ff(load_logit(sx.ptr, di, DT), S.u.fv.m[ti], T_b, S.exp_hi, S.exp_lo),
                                ff_recip(ff{S.u.fv.s[ti], S.u.fv.s_lo[ti]})));
          if (!det) {
            const int ty = 2 * i + 1;
            const SlotInfo sy = slot_info(p, S, slot0 + ty);
            q_d = ff_round(ff_mul(exp_diff_ff(load_logit(sy.ptr, di, DT), S.u.fv.m[ty], T_b, S.exp_hi, S.exp_lo),
                                  ff_recip(ff{S.u.fv.s[ty], S.u.fv.s_lo[ty]})));
          }
        }
        const uint4 wd = step_uniform_words(p.seed, (uint32_t)b, (uint32_t)i, 0u);
        stop = !(uniform24(wd.x) < p_d / q_d);  // q = 0: +inf if p > 0, NaN if p == 0
        if (p.audit_pq) {
          p.audit_pq[((size_t)b * gamma + i) * 2] = p_d;
          p.audit_pq[((size_t)b * gamma + i) * 2 + 1] = q_d;
        }
      }
    }
    const uint32_t ball = __ballot_sync(0xffffffffu, stop);
    const int n = ball ? __ffs(ball) - 1 : gamma;
    const int tn = det ? n : 2 * n;  // position n's target row (the bonus row when n == gamma)
    const bool resid = n < gamma && !det;
    const bool bad_n = S.u.fv.bad[tn] || (resid && S.u.fv.bad[2 * n + 1]);
    // a deterministic draft's residual is p without d: the bonus-style draw
    // over target row n with d left out
    const int mode = bad_n ? kFvNone : (resid ? kFvResidual : kFvBonus);
    const int32_t d_n = __shfl_sync(0xffffffffu, d_lane, n & 31);
    const int excl = det && n < gamma ? d_n : -1;
    // the token at position n is the second pass's (0 when a bad row leaves no draw)
    for (int i = lane; i <= gamma; i += 32) out[i] = i < n ? d_lane : (i == n ? 0 : -1);
    st = __reduce_or_sync(0xffffffffu, st);
    if (lane == 0) {
      if (p.out_len) p.out_len[b] = n + 1;
      p.fv_draw[b] = FvDraw{n, mode, S.u.fv.m[tn], resid ? S.u.fv.m[2 * n + 1] : 0.0f, S.u.fv.s[tn],
                            resid ? S.u.fv.s[2 * n + 1] : 0.0f, excl};
      if (st && p.status) atomicOr(p.status, st);
    }
  }
  fin_sync();
}

// Finals group (4 warps): runs finals jobs, which it draws one at a time from
// a counter in the workspace: first the rows that need a top-k (sampling
// rows, every row of the rows tasks) in the order rows finish, then one job
// per request (sampling requests, then greedy ones). A group draws its next
// job while it works on the current one (once that one's inputs are ready),
// so a job goes to whichever group frees up first. A row final waits only on
// the stream; a sampling request's final may wait on its rows' finals, which
// were all drawn before it, so no two groups can wait on each other in a
// cycle.
template <int DT>
__device__ bool finals_job(const Params& p, Smem& S, bool row_job, int j, int ord, uint32_t& next) {
  const int gt = fin_tid(), w = gt >> 5;
  const int per_s = samp_slots(p), per_g = p.gamma + 1;
  // A row job's row final, and a top-k sampling request's final, wait on the
  // words they read (tile keys, filtered lists). A full-vocabulary or greedy
  // request's final waits for its rows' pieces to be counted.
  const bool counted = !row_job && (ord >= S.n_samp || p.fullvocab);
  if (w == 0 && counted) {
    const bool samp = ord < S.n_samp;
    const bool ok = wait_rows(p, samp ? ord * per_s : S.n_samp * per_s + (ord - S.n_samp) * per_g,
                              samp ? per_s : per_g);
    if (gt == 0) {
      if (!ok) raise_timeout(p);
      S.fin_cmd = ok ? 1 : 2;
    }
    if (ok) fence_acq_rel_gpu();  // acquire what the rows' consumers wrote
  }
  if (!counted && gt == 0) S.fin_cmd = 1;
  fin_sync();
  if (S.fin_cmd != 1) return false;
  if (counted) draw_next_job(p, next);  // the others draw when their polls succeed
  bool ok = true;
  if (!row_job) {
    if (ord >= S.n_samp) {
      if (w == 0) greedy_request_final<DT>(p, S, ord);
      fin_sync();
    } else if (p.fullvocab) {
      fullvocab_request_final<DT>(p, S, ord);
    } else {
      ok = request_final(p, S, ord, next);
    }
  } else {
    const SlotInfo si = slot_info(p, S, j);
    unsigned long long top_a = 0ull;
    float T_row;
    ok = row_final<DT>(p, S, j, si, top_a, T_row, next);
    if (ok && (p.task == kTaskFilter || p.task == kTaskSample)) rows_final(p, S, j, top_a, T_row);
  }
  if (!ok && gt == 0) raise_timeout(p);
  return ok;
}

template <int DT>
__device__ void finals(const Params& p, Smem& S) {
  const int gt = fin_tid();
  const bool verify = p.task == kTaskVerify || p.task == kTaskVerifyGreedy;
  const bool fv = verify && p.fullvocab;
  // row jobs: top-k sampling rows, or every row of a rows task; then request
  // jobs from request ordinal ord0 on
  const int n_row_jobs = fv ? 0 : (verify ? S.n_samp * samp_slots(p) : p.B);
  const int ord0 = 0;  // every request has a final job (sampling first, then greedy)
  const int n_jobs = n_row_jobs + (verify ? p.B - ord0 : 0);
  if (gt == kFinDrawer) S.fin_slot = (int)atomicAdd(p.job_cnt, 1u);
  fin_sync();
  int j = S.fin_slot;
  while (j < n_jobs) {
    uint32_t next = 0u;  // drawn by the job once it is ready to run
    const bool ok = j < n_row_jobs ? finals_job<DT>(p, S, true, j, 0, next)
                                   : finals_job<DT>(p, S, false, 0, ord0 + (j - n_row_jobs), next);
    if (!ok) return;  // timed out: the workspace must be prepared again anyway
    if (gt == kFinDrawer) S.fin_slot = (int)next;
    fin_sync();
    j = S.fin_slot;
  }
  // every group's last draw is past the jobs; the very last of all draws
  // returns the counter to zero for the next call
  if (gt == kFinDrawer && j == n_jobs + (int)gridDim.x - 1) *p.job_cnt = 0u;
}

// ---- the kernel ---------------------------------------------------------------------------
template <int DT>
__global__ void __launch_bounds__(kThreads, kCtasPerSm) sweep_kernel(const Params p) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem& S = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x, warp = tid >> 5;

  // Tang's exp table (float-float exp of the filters and the full-vocabulary
  // statistics), from the kernel parameters
  if (tid < kExpTable) {
    S.exp_hi[tid] = p.exp2.hi[tid];
    S.exp_lo[tid] = p.exp2.lo[tid];
  }
  // the mbarriers, one per thread of the warps that load no temperatures
  // (the consumer threads' loads of the request order are in flight meanwhile)
  static_assert(kThreads - kConsumers >= 2 * (kStages + kKeyQueue), "one thread per mbarrier");
  {
    const int b = tid - kConsumers;
    if (b >= 0 && b < 2 * (kStages + kKeyQueue)) {
      uint64_t* bar = b < kStages ? &S.full[b]
                      : b < 2 * kStages ? &S.empty[b - kStages]
                      : b < 2 * kStages + kKeyQueue ? &S.kfull[b - 2 * kStages]
                                                    : &S.kempty[b - 2 * kStages - kKeyQueue];
      mbar_init(bar, 1);
      fence_barrier_init();
    }
  }
  // Programmatic dependent launch: everything above touches only this CTA's
  // shared memory, so it may overlap the end of the kernel before this one in
  // the stream; every global load and store (the inputs may be that kernel's
  // outputs, and the workspace its leftovers) comes after the wait. The next
  // kernel may be scheduled at once: its CTAs only start on SMs this grid has
  // left, and they wait in the same place.
  grid_dependency_sync();
  build_request_order(p, S);  // contains __syncthreads
  __syncthreads();
  if (S.cancelled) {  // a cancelled workspace: report, and leave before any copy is issued
    if (tid == 0 && p.status) atomicOr(p.status, kStatusTimeout);
    return;
  }
  // with keys from the LM head's epilogue nothing is streamed: only the finals run
  const long long total = p.keys_ready ? 0 : (long long)active_slots(p, S) * p.geo.ppr;

  if (warp < kConsumerWarps)
    consumer<DT>(p, S, total);
  else if (warp == kProducerWarp)
    producer(p, S, total);
  else if (warp == kPublisherWarp)
    publisher(p, S, total);
  else
    finals<DT>(p, S);
}

__global__ void uniforms_kernel(unsigned long long seed, int B, int npos, int stream_id, float* ua, float* ud) {
  const long long n = (long long)B * npos;
  for (long long i = blockIdx.x * (long long)blockDim.x + threadIdx.x; i < n; i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / npos), pos = (int)(i - (long long)b * npos);
    const uint4 w = step_uniform_words(seed, (uint32_t)b, (uint32_t)pos, (uint32_t)stream_id);
    if (ua) ua[i] = uniform24(w.x);
    if (ud) ud[i] = uniform24(w.y);
  }
}

}  // namespace

int sweep_smem_bytes() { return (int)sizeof(Smem); }

namespace {
// The kernel's shared-memory opt-in, set once per device (the attribute is a
// property of the function on the current device).
std::mutex g_attr_mu;
bool g_attr_set[2][kMaxDevices] = {};

template <int DT>
cudaError_t prepare_sweep(int dev) {
  std::lock_guard<std::mutex> lock(g_attr_mu);
  if (g_attr_set[DT][dev]) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(sweep_kernel<DT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sizeof(Smem));
  if (e == cudaSuccess) g_attr_set[DT][dev] = true;
  return e;
}

template <int DT>
int launch_sweep_t(const Params& p, int grid, void* stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return (int)e;
  if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  if ((e = prepare_sweep<DT>(dev)) != cudaSuccess) return (int)e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = (cudaStream_t)stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return (int)cudaLaunchKernelEx(&cfg, sweep_kernel<DT>, p);
}

template <int DT>
int occupancy_t(int dev, int* ctas_per_sm) {
  cudaError_t e = prepare_sweep<DT>(dev);
  if (e != cudaSuccess) return (int)e;
  return (int)cudaOccupancyMaxActiveBlocksPerMultiprocessor(ctas_per_sm, sweep_kernel<DT>, kThreads,
                                                            sizeof(Smem));
}
}  // namespace

int launch_sweep(const Params& p, int grid, void* stream) {
  return p.dtype == 0 ? launch_sweep_t<0>(p, grid, stream) : launch_sweep_t<1>(p, grid, stream);
}

int sweep_occupancy(int dtype, int dev, int* ctas_per_sm) {
  if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
  return dtype == 0 ? occupancy_t<0>(dev, ctas_per_sm) : occupancy_t<1>(dev, ctas_per_sm);
}

int launch_uniforms(unsigned long long seed, int B, int npos, int stream_id, float* ua, float* ud, void* stream) {
  const long long n = (long long)B * npos;
  if (n <= 0) return 0;
  const int block = 256;
  const int grid = (int)((n + block - 1) / block < 1024 ? (n + block - 1) / block : 1024);
  uniforms_kernel<<<grid, block, 0, (cudaStream_t)stream>>>(seed, B, npos, stream_id, ua, ud);
  return (int)cudaGetLastError();
}

}  // namespace dflash
