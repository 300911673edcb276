// dflash_internal.h -- shapes, workspace layout and kernel parameters shared by
// the host side (dflash_abi.cu) and the kernels (dflash_sweep.cu).
#pragma once

#include <vector_types.h>

#include <cstddef>
#include <cstdint>

namespace dflash {

// ---- fixed tiling -------------------------------------------------------------
// One "piece" is a 16 KB contiguous run of a row's 16-byte-aligned body, moved
// into shared memory by one bulk (TMA) copy and reduced by one consumer warp:
// lane l reads vectors 32*r + l for r = 0..31, in 8 blocks of 4 rounds. A
// "tile" is what 8 neighbouring lanes read in one block: vectors
// 32*(4*blk + rr) + 8*g + l (rr < 4, l < 8) for tile 4*blk + g, i.e. 32
// vectors (256 bf16 or 128 fp32 logits); its largest logit is recorded for the
// row-level selection.
//
// A CTA (one per SM) has four roles: warps 0-7 consume pieces, warp 8 is the
// producer (bulk copies), warp 9 publishes finished pieces to the other CTAs,
// warps 10-13 are the finals group (row and request finals).
constexpr int kConsumerWarps = 8;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kPublisherWarp = kConsumerWarps + 1;
constexpr int kFinWarps = 4;
constexpr int kFin = kFinWarps * 32;
constexpr int kFinBase = (kConsumerWarps + 2) * 32;
constexpr int kThreads = kFinBase + kFin;
constexpr int kPieceBytes = 16384;
constexpr int kVecPerPiece = kPieceBytes / 16;
constexpr int kRoundsPerPiece = kVecPerPiece / 32;   // vectors per lane
constexpr int kTileLanes = 8;
constexpr int kTilesPerPiece = kRoundsPerPiece;       // 8 blocks x 4 lane groups
constexpr int kStages = 12;      // ring of bulk-copy stages
constexpr int kKeyQueue = 32;    // pieces the publisher may lag behind
// Consumer warp w waits for piece it = w + 8 k on stage it % kStages with the
// phase parity of round it / kStages. A parity wait only tells adjacent
// phases apart, so it names the right phase only if the stage's previous
// piece (it - kStages) has landed. Bulk copies can land out of order, so the
// consumer first waits for that piece to be consumed (the stage's empty
// barrier). That wait is unambiguous when piece it - 2 kStages was the warp's
// own, i.e. 2 kStages is a multiple of kConsumerWarps. With fewer stages than
// warps, or without that first wait, a consumer can read a stage before its
// copy lands. The key queue is safe with kKeyQueue >= kConsumerWarps: the
// warp's own previous piece already waited for the publisher to be within
// kKeyQueue + kConsumerWarps pieces.
static_assert(kStages >= kConsumerWarps, "ring stages must cover every consumer warp's piece");
static_assert((2 * kStages) % kConsumerWarps == 0, "piece it - 2 kStages must be the consumer warp's own");
static_assert(kKeyQueue >= kConsumerWarps, "key-queue slots must cover every consumer warp's piece");
constexpr int kCtasPerSm = 1;
constexpr int kMaxDevices = 64;

// Grid of the persistent stream kernel. Its CTAs wait on each other (a row's
// final polls tile keys that other CTAs' consumers write), so every CTA must
// be resident at once: the grid is at most the CTAs the SMs available to the
// calling context hold together (SMs x CTAs per SM at the kernel's shared
// memory and thread counts), and never more than there are pieces. 0 when
// no CTA fits at all.
inline long long persistent_grid(long long pieces, int sms_available, int ctas_per_sm) {
  if (sms_available < 1 || ctas_per_sm < 1) return 0;
  long long g = (long long)sms_available * ctas_per_sm;
  if (g > pieces) g = pieces;
  return g < 1 ? 1 : g;
}

constexpr int kMaxTopK = 32;     // one kept token per lane of a warp
constexpr int kListWords = kMaxTopK + 1;  // a row's filtered list, then its draft token's probability
constexpr int kCandCap = 64;     // candidates sorted in registers (2 per lane)
constexpr int kCandTileCap = 128;
constexpr int kKeyCache = 2048;  // tile keys of one row cached in shared memory
constexpr int kMaxGamma = 32;
constexpr int kMaxRowsPerRequest = 2 * kMaxGamma + 1;
constexpr int kMaxB = 2048;

// body vector (within its piece) of vector t (< 32) of tile `tile`
inline __host__ __device__ int tile_vector(int tile, int t) {
  return 32 * (4 * (tile >> 2) + (t >> 3)) + 8 * (tile & 3) + (t & 7);
}

enum Task : int { kTaskVerify = 0, kTaskVerifyGreedy = 1, kTaskFilter = 2, kTaskSample = 3, kTaskCandidates = 4 };

// Row geometry: the head (elements before the first 16-byte boundary) and
// tail (after the last one) are read with plain loads by the row-final stage;
// the body goes through the pieces. Rows of one tensor may have different
// heads when V * element size is not a multiple of 16, so every count is per
// row and ppr (pieces per row) is the maximum over rows.
struct Geometry {
  int V;
  int esize;     // 2 (bf16) or 4 (fp32)
  int ppr;       // pieces per row (>= 1)
  int tiles;     // ppr * kTilesPerPiece
};

// ---- full-vocabulary mode (top-k off, top-p 1) --------------------------------------
// The stream reduces each piece of a sampling row to (max, sum of exp) for the
// accept test; the residual or bonus draw then runs as a second pass over the
// one or two rows it needs, cut into slices of kFvSlice logits.
constexpr int kFvSlice = 4096;
constexpr int kFvThreads = 256;
constexpr int kFvPerThread = kFvSlice / kFvThreads;
constexpr int kExpTable = 64;  // 2^(j/64), j < 64, as fp32 pairs

enum FvMode : int { kFvNone = 0, kFvResidual = 1, kFvBonus = 2 };

// 2^(j/64) = hi[j] + lo[j] (j < 64) for the float-float exp (computed on the
// host in double precision)
struct ExpTable {
  float hi[kExpTable];
  float lo[kExpTable];
};

// what the accept test left for the draw of request b
struct FvDraw {
  int n;       // drafts accepted: the token drawn goes to position n
  int mode;    // FvMode
  float mx;    // largest logit of target row n
  float my;    // largest logit of draft row n (residual)
  float sx0;   // the stream's (fp32) sum of exp((x - mx) / T) over target row n
  float sy0;   // the same over draft row n (residual)
  int excl;    // a token the draw leaves out (a deterministic draft's residual), -1 for none
};

inline int fv_slices(int V) { return (V + kFvSlice - 1) / kFvSlice; }

struct Params {
  // inputs
  const unsigned char* target;  // verify: [B, gamma+1, V]; rows tasks: [R, V]
  const unsigned char* draft;   // verify: [B, gamma, V]; unused with deterministic drafts
  const int32_t* draft_tokens;  // [B, gamma]
  const float* temperature;     // [B] or [R]
  int B;                        // requests (verify) or rows (rows tasks)
  int gamma;
  int dtype;                    // 0 bf16, 1 fp32
  int top_k;                    // effective k for sampling rows, 1..kMaxTopK
  float top_p;
  unsigned long long seed;
  int task;
  int fullvocab;                // top-k off and top-p 1: softmax over the whole vocabulary
  int det;                      // verify: deterministic drafts (q = point mass at the draft; no draft rows)
  int keys_ready;               // verify: the tile keys and greedy argmaxes were written by the LM head's
                                // epilogue (before this launch); stream nothing, run the finals
  int row_base;                 // rows tasks: index of this launch's first row
  int vocab_offset;             // candidates task: token id of the shard's first logit
  Geometry geo;
  // outputs
  int32_t* out_tokens;
  int32_t* out_len;
  int32_t* out_idx;
  float* out_prob;
  int32_t* out_count;
  float* out_rowmax;            // candidates task: each row's largest logit (NaN if it holds one)
  float* audit_pq;              // verify, optional [B, gamma, 2]: p(d), q(d) each accept test used
  uint32_t* status;
  // workspace (zero-initialised once; counters reset by their last user)
  uint32_t* row_cnt;    // [n_slots]
  uint32_t* abort_flag; // [1]
  uint32_t* job_cnt;    // [1]: next finals job to hand out (beside the abort flag)
  unsigned long long* row_best;  // [kMaxCounterSlots]: greedy rows' best (key, index) composite
  uint32_t* tile_keys;  // [n_slots, geo.tiles]; full-vocabulary rows: float2 (max, sum) per piece
  // [n_slots, kListWords]: a verification sampling row's filtered list, one
  // word per rank: (token + 2) << 32 | probability bits, the sign bit of
  // rank 0 set for a bad row; then 1 << 32 | the probability the row gives
  // its position's draft token (0 when not kept, and for the bonus row). No
  // written word is zero, so the request final polls the words themselves.
  unsigned long long* res_list;
  FvDraw* fv_draw;      // [B]: full-vocabulary mode
  int fvtp;             // full-vocabulary top-p (top-k off, top_p < 1): the stream leaves the rows' statistics
  float4* fvtp_rows;    // [B * rows per request]: (max, normaliser pair, bad flag) of each sampling row
  int n_slots;
  ExpTable exp2;        // for the filter's float-float exp
};

// ---- full-vocabulary top-p (top-k off, 0 < top_p < 1) --------------------------------
// The kept set of a row is the shortest prefix of its (logit desc, index asc)
// order whose mass reaches top_p: every token whose order key is above kappa,
// and the tokens whose key is kappa up to index j_cut. The masses are sums of
// float-float weights exp((x - m) / T) rounded to fixed point (frac_bits
// fractional bits), so every sum is exact and the same wherever it is taken.
struct FvtpCut {
  uint32_t kmin, kmax;           // the first round's crossing bin: its keys (refinement units)
  uint32_t prefix;               // bits of (key - kmin) found by the refinement rounds
                                 // (refinement units: the key, or for bf16 its upper half)
  uint32_t kappa;                // the last kept token's key (state 2)
  int32_t nref;                  // refinement rounds the crossing bin needs (bytes of its key span)
  unsigned long long above;      // mass of the keys above the current group
  unsigned long long total;      // mass of the row
  unsigned long long kept;       // mass of the kept set (state 2)
  uint32_t count;                // tokens in the current group (key kappa's, state 2)
  uint32_t keep;                 // of key kappa's tokens, how many are kept (first in index order)
  int32_t j_cut;                 // last kept index among key kappa's tokens (V: all of them)
  int32_t state;                 // 0 = no cut (not a sampling row, or bad), 1 = searching, 2 = found
};
// what the draw needs of the kept sets of the two rows it reads
struct FvtpDrawCut {
  uint32_t kappa_x, kappa_y;
  int32_t jcut_x, jcut_y;
};

// Second pass of the full-vocabulary draw (dflash_fullvocab.cu).
struct FvParams {
  const unsigned char* target;  // [B, gamma+1, V]
  const unsigned char* draft;   // [B, gamma, V]
  const float* temperature;     // [B]
  int B, gamma, V, dtype, n_slices;
  unsigned long long seed;
  int sampler;                  // the filtered sampler's uniforms (counter (row_base + b, 0, 1, 0), word 0)
  int row_base;
  int32_t* out_tokens;          // [B, gamma+1]
  const FvDraw* draw;           // [B]
  float4* part;                 // [B, n_slices]: slice sums of the two rows' exp weights
  float4* pos;                  // [B, n_slices]: the same sums over the tokens with p > q
  int2* last;                   // [B, n_slices]: last token with p > q / with p > 0
  FvtpDrawCut* cut;             // top-p over the full vocabulary: the kept sets ([B]); null otherwise
  const uint32_t* abort_flag;
  float exp_hi[kExpTable];      // 2^(j/64) = exp_hi[j] + exp_lo[j]
  float exp_lo[kExpTable];
};

// Kernels between the stream and the draw under top-p over the full
// vocabulary (dflash_fvtp.cu): the cut of every sampling row, then the accept
// tests, which leave the draw descriptors for the second pass.
struct FvtpParams {
  const unsigned char* target;  // [B, gamma+1, V]
  const unsigned char* draft;   // [B, gamma, V] (unused with deterministic drafts)
  const int32_t* draft_tokens;  // [B, gamma]
  const float* temperature;     // [B]
  int B, gamma, V, dtype, det, per_s, n_slices, frac_bits, round;
  float top_p;
  unsigned long long seed;
  int sampler, row_base;        // the sampler's uniforms (as for FvParams)
  int32_t* out_tokens;          // [B, gamma+1]
  int32_t* out_len;             // [B] (may be null: the sampler)
  uint32_t* status;
  float* audit_pq;              // optional [B, gamma, 2]
  float4* rows;                 // [B * per_s] from the stream
  FvtpCut* cut;                 // [B * per_s]
  unsigned long long* hist_m;   // [B * per_s, 256] masses of the current round's bins
  uint32_t* kcount;             // [B * per_s, n_slices]
  FvDraw* draw;                 // [B]
  FvtpDrawCut* draw_cut;        // [B]
  const uint32_t* abort_flag;
  ExpTable exp2;
};

// ---- vocabulary-shard candidates ----------------------------------------------------
// A shard's record for a batch (B requests, gamma drafts, k candidates per
// row), 32-bit words: the target rows' [B * (gamma+1), k] candidate logits
// (fp32 bits, -inf past the shard's tokens), their [B * (gamma+1), k] global
// token ids (-1 there), the target rows' maxima [B * (gamma+1)] (fp32), then
// the same three arrays for the draft rows [B * gamma].
constexpr int kMaxShardCand = 256;  // shards x k candidates merged per row
struct CandidateLayout {
  size_t t_logit, t_token, t_max, d_logit, d_token, d_max, words;
};
inline CandidateLayout candidate_layout(int B, int gamma, int k) {
  CandidateLayout L;
  const size_t rt = (size_t)B * (gamma + 1), rd = (size_t)B * gamma;
  L.t_logit = 0;
  L.t_token = L.t_logit + rt * k;
  L.t_max = L.t_token + rt * k;
  L.d_logit = L.t_max + rt;
  L.d_token = L.d_logit + rd * k;
  L.d_max = L.d_token + rd * k;
  L.words = L.d_max + rd;
  return L;
}

struct CandParams {
  const uint32_t* records;      // [n_shards, words]
  size_t words;                 // one record's words
  CandidateLayout L;
  int n_shards, k;              // shards, candidates per shard and row
  const int32_t* draft_tokens;  // [B, gamma]
  const float* temperature;     // [B]
  int B, gamma, V, top_k;
  float top_p;
  unsigned long long seed;
  int32_t* out_tokens;          // [B, gamma+1]
  int32_t* out_len;             // [B]
  uint32_t* status;
  ExpTable exp2;                // for the filter's float-float exp
};

struct WorkspaceLayout {
  size_t row_cnt, abort_flag, row_best, tile_keys, res_list;
  size_t fv_draw, fv_part, fv_pos, fv_last;
  size_t tp_rows, tp_cut, tp_hist_m, tp_kcount, tp_draw, total;
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline Geometry make_geometry(int V, int esize) {
  Geometry g;
  g.V = V;
  g.esize = esize;
  long long body_vec_max = (long long)V * esize / 16;
  long long ppr = (body_vec_max + kVecPerPiece - 1) / kVecPerPiece;
  g.ppr = (int)(ppr < 1 ? 1 : ppr);
  g.tiles = g.ppr * kTilesPerPiece;
  return g;
}

// The hand-off counters and the greedy rows' running argmax live in a fixed header
// at the start of every workspace, at offsets that do not depend on the
// call's shape: every call returns what it used to zero, so a workspace stays
// ready for the next call of any shape. The per-row data follows the header.
constexpr int kMaxCounterSlots = kMaxB * kMaxRowsPerRequest;  // also the rows-task chunk

inline WorkspaceLayout make_layout(int n_slots, int n_requests, const Geometry& g, bool fullvocab = false,
                                   bool fvtp = false) {
  WorkspaceLayout L;
  size_t off = 0;
  L.row_cnt = off;    off = align_up(off + sizeof(uint32_t) * (size_t)kMaxCounterSlots, 256);
  L.abort_flag = off; off = align_up(off + 2 * sizeof(uint32_t), 256);  // abort flag, job counter
  L.row_best = off;   off = align_up(off + sizeof(unsigned long long) * (size_t)kMaxCounterSlots, 256);
  L.tile_keys = off;  off = align_up(off + sizeof(uint32_t) * (size_t)n_slots * g.tiles, 256);
  L.res_list = off;   off = align_up(off + sizeof(unsigned long long) * (size_t)n_slots * kListWords, 256);
  const size_t fv_req = fullvocab ? (size_t)n_requests : 0;
  const size_t fv_cells = fv_req * (size_t)fv_slices(g.V);
  L.fv_draw = off;    off = align_up(off + sizeof(FvDraw) * fv_req, 256);
  L.fv_part = off;    off = align_up(off + 16 * fv_cells, 256);
  L.fv_pos = off;     off = align_up(off + 16 * fv_cells, 256);
  L.fv_last = off;    off = align_up(off + 8 * fv_cells, 256);
  // top-p over the full vocabulary: per row (n_slots of them) its statistics,
  // cut state, 256-bin mass and count histograms and per-slice counts; per
  // request the draw's kept sets
  const size_t tp_rows = fvtp ? (size_t)n_slots : 0, tp_req = fvtp ? (size_t)n_requests : 0;
  L.tp_rows = off;    off = align_up(off + 16 * tp_rows, 256);
  L.tp_cut = off;     off = align_up(off + sizeof(FvtpCut) * tp_rows, 256);
  L.tp_hist_m = off;  off = align_up(off + 8 * 256 * tp_rows, 256);
  L.tp_kcount = off;  off = align_up(off + 4 * tp_rows * (size_t)fv_slices(g.V), 256);
  L.tp_draw = off;    off = align_up(off + sizeof(FvtpDrawCut) * tp_req, 256);
  L.total = off;
  return L;
}

// sets the message dflash_last_error() returns on this thread (dflash_abi.cu)
void set_last_error(const char* msg);

// launches (dflash_sweep.cu); return a cudaError_t value
int launch_sweep(const Params& p, int grid, void* stream);
int sweep_smem_bytes();
// CTAs of the stream kernel (dtype 0 bf16, 1 fp32) one SM of device `dev` holds
int sweep_occupancy(int dtype, int dev, int* ctas_per_sm);
int launch_fullvocab_draw(const FvParams& f, void* stream);
struct FvtpParams;
int launch_fvtp_cut(const FvtpParams& t, void* stream);  // dflash_fvtp.cu

// ---- the LM head on the tensor cores (dflash_lmhead.cu) -----------------------------
// logits [M, V] = h [M, K] W^T (W [V, K]), bf16 in and out, fp32 accumulation;
// M <= kLmMaxRows (four 128-row token tiles), K a multiple of 64. Fused: the
// rows are a verification's target rows (Mt = B (gamma + 1)) then its draft
// rows (B gamma), and the epilogue also writes the top-k rows' tile keys and
// the greedy rows' argmax composites into the verification's workspace.
constexpr int kLmMaxRows = 512;
struct LmParams {
  int M, Mt, V, K;
  uint16_t* logits;               // [M, V] bf16 bits
  int B, gamma, tiles;            // fused: the verification's shape and tiles per row
  const float* temperature;       // fused: [B]
  uint32_t* tile_keys;            // fused: [slots, tiles]
  unsigned long long* row_best;   // fused: [slots]
  uint32_t* status;
};
int launch_lmhead(const LmParams& p, const void* h, const void* w, bool fused, int grid, void* stream);
int lmhead_smem_bytes();
int launch_uniforms(unsigned long long seed, int B, int npos, int stream_id, float* out_accept,
                    float* out_draw, void* stream);
int launch_verify_candidates(const CandParams& c, void* stream);  // dflash_candidates.cu

}  // namespace dflash
