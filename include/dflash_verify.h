/*
 * dflash_verify.h -- C ABI of the GB300 (sm_103a) draft-verification library.
 *
 * The library performs the verification step of block-drafted speculative
 * decoding (DFlash / DFlash2) on a batch of requests: a block of gamma draft
 * tokens per request is checked against the target model's logits at every
 * draft position, and the step emits the accepted tokens, one corrected or
 * bonus token, and the accept length.
 *
 * Sources of the operation (page title, then section):
 *  - "DFlash2 用投机解码给 Qwen 提速" (bml.asia): the draft/verify loop
 *    (one target forward over prefix + drafts, then accept each draft token
 *    in order, resample from the target at the first rejection and stop);
 *    the model-card settings (block size 8, temperature 1.0, top-p 0.95,
 *    top-k 20); rejection sampling keeps the output distribution identical.
 *  - "无损加速是真的吗？Qwen3.8-27B-DFlash2如何保证输出与目标模型完全一致"
 *    (rytg.cn): section "投机解码如何白嫖速度" (a block of 8, 7 tokens
 *    verified per step; step 3 "裁决": from the first mismatch the target
 *    resamples from its own distribution), the lossless definition (greedy
 *    output identical to the target, sampling preserves its distribution) and
 *    the acceptance length (tokens produced per verification step).
 *  - Standard speculative sampling: accept a draft token d with probability
 *    min(1, p(d)/q(d)); at the first rejection draw from the normalised
 *    residual max(0, p - q); when every draft is accepted draw a bonus token
 *    from the target distribution of the last position.
 *  - Philox4x32-10 (Salmon et al., "Parallel Random Numbers: As Easy as 1, 2,
 *    3", SC'11) for the uniforms, keyed by (seed, request, position).
 *
 * Conventions for every entry point:
 *  - Pointers marked [device] are CUDA device pointers; [host] are host
 *    pointers. The caller owns every buffer; the library keeps no pointer
 *    after a call returns and allocates no device memory. Inputs are not
 *    modified.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Device work is enqueued on it; calls with only [device]
 *    buffers return without waiting for the GPU.
 *  - Logits are dense row-major arrays of bf16 (dtype DFLASH_BF16, raw
 *    bfloat16) or fp32 (DFLASH_F32). Rows need no particular alignment.
 *  - Return value: DFLASH_OK, or an error code when the arguments are
 *    rejected (nothing is enqueued) or a CUDA launch fails;
 *    dflash_last_error() describes the last error of the calling thread.
 *  - Data problems found on the GPU never trap: they OR DFLASH_STATUS_* bits
 *    into *status (a [device] uint32, optional, never cleared by the
 *    library), and the outputs stay in range.
 *  - Filtering: temperature T > 0 scales logits as x / T; top-k keeps the k
 *    largest logits, ties to the lower token index (top_k <= 0 or >= V:
 *    off); softmax over the survivors; top-p keeps the shortest prefix of
 *    that order whose mass reaches top_p (top_p >= 1: off) and renormalises.
 *    Supported: 1 <= top_k <= DFLASH_MAX_TOP_K with any top_p in (0, 1], or
 *    top-k off with any top_p (the full-vocabulary softmax, with top_p < 1
 *    cut by mass over the whole vocabulary, V <= 2^22; the verification entry
 *    points and dflash_sample). Other combinations return
 *    DFLASH_ERR_UNSUPPORTED.
 *    Over the full vocabulary with top_p < 1 the cut is taken on exact
 *    fixed-point sums of the float-float weights, the decision "mass before
 *    token j, over the row's mass, rounds (fp32) below top_p" in the order
 *    logit descending, token index ascending.
 */
#ifndef DFLASH_VERIFY_H
#define DFLASH_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DFLASH_ABI_VERSION 1
#define DFLASH_MAX_TOP_K 32

/* logits storage type */
enum { DFLASH_BF16 = 0, DFLASH_F32 = 1 };

/* return codes */
enum {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = 1, /* null pointer, bad size, bad top_p, small workspace */
  DFLASH_ERR_UNSUPPORTED = 2, /* filter combination outside the supported set */
  DFLASH_ERR_CUDA = 3         /* a CUDA call failed (message in dflash_last_error) */
};

/* device status bits (OR-ed into *status) */
#define DFLASH_STATUS_BAD_TOKEN 1u       /* a draft token outside [0, V): never accepted */
#define DFLASH_STATUS_BAD_ROW 2u         /* a row read by the step holds a NaN or has an
                                            infinite maximum; that request's output is
                                            unspecified but in range */
#define DFLASH_STATUS_TIMEOUT 4u         /* a bounded on-chip wait gave up (the call's
                                            outputs are then unspecified) */
#define DFLASH_STATUS_BAD_TEMPERATURE 8u /* temperature negative, NaN or infinite: the
                                            request is verified greedily */

/* ABI version of the loaded library (DFLASH_ABI_VERSION). */
int dflash_abi_version(void);

/* Message of the last error returned to the calling thread ("" if none). */
const char* dflash_last_error(void);

/* Bytes of device workspace dflash_verify / dflash_verify_greedy need for a
 * batch of this shape (greedy: pass top_k = 1, top_p = 1). 0 when the
 * arguments are invalid or unsupported. */
size_t dflash_workspace_bytes(int B, int gamma, int V, int dtype, int top_k, float top_p);

/* Bytes of device workspace dflash_filter / dflash_sample need for R rows. */
size_t dflash_rows_workspace_bytes(int R, int V, int dtype, int top_k, float top_p);

/* Prepares a workspace for first use (zero-fills it on `stream`). Needed once
 * per allocation, and again after any call on it returned DFLASH_ERR_CUDA or
 * raised DFLASH_STATUS_TIMEOUT; every successful call leaves it ready for the
 * next. Calls sharing one workspace must be ordered (same stream, or
 * synchronised). */
int dflash_workspace_init(void* workspace, size_t bytes, void* stream);

/* Cancels the calls on a workspace: sets its abort flag on `stream`. Every
 * bounded wait of a call on this workspace that starts after the flag is set
 * (in stream order), or that runs meanwhile on another stream, gives up at
 * once: the call ORs DFLASH_STATUS_TIMEOUT into its status word, lets its
 * issued copies land, and returns with unspecified outputs. The workspace
 * must be prepared again (dflash_workspace_init) before its next use. */
int dflash_workspace_cancel(void* workspace, size_t bytes, void* stream);

/* Batched verification (sampling, with greedy requests mixed in).
 *
 * target_logits [device] [B, gamma+1, V] dtype: target logits at the gamma
 *     draft positions and the bonus position.
 * draft_logits  [device] [B, gamma, V] dtype: the drafter's logits at each
 *     draft position. Rows of greedy requests are not read (may be garbage).
 * draft_tokens  [device] int32 [B, gamma]: the drafts, which must be samples
 *     from the drafter's filtered distribution for the step to be lossless.
 * temperature   [device] float [B]: T > 0 samples; T == 0 verifies that
 *     request greedily (argmax prefix match); other values: greedy plus
 *     DFLASH_STATUS_BAD_TEMPERATURE.
 * top_k, top_p: the filter applied to both target and draft distributions.
 * seed: Philox key; request b at position i uses counter (i, b, 0, 0):
 *     output word 0 -> the accept uniform, word 1 -> the residual / bonus
 *     uniform, each (w >> 8) * 2^-24.
 * out_tokens     [device] int32 [B, gamma+1]: accepted drafts, then the
 *     corrected or bonus token, then -1 padding.
 * out_accept_len [device] int32 [B]: tokens emitted, in [1, gamma+1].
 * workspace [device], workspace_bytes >= dflash_workspace_bytes(...),
 *     prepared by dflash_workspace_init.
 * Accept test at position i: u < p_i(d_i) / q_i(d_i) in fp32 (q = 0 with
 * p > 0 accepts; p = q = 0 rejects). The residual and bonus draws take the
 * smallest token index whose cumulative weight (ascending token order)
 * exceeds u * total; over the full vocabulary (top-k off) the cumulative
 * weights are carried in float-float and the comparison is taken on their
 * fp32 roundings (with top_p < 1 only the kept tokens weigh). 1 <= gamma <= 32, 1 <= V < 2^31, 1 <= B <= 2048. */
int dflash_verify(const void* target_logits, const void* draft_logits,
                  const int32_t* draft_tokens, int B, int gamma, int V, int dtype,
                  const float* temperature, int top_k, float top_p, uint64_t seed,
                  int32_t* out_tokens, int32_t* out_accept_len, void* workspace,
                  size_t workspace_bytes, uint32_t* status, void* stream);

/* dflash_verify that also reports, for audits, the two probabilities each
 * accept test compared: audit_pq [device] float [B, gamma, 2] receives, for
 * every sampling request b and draft position i, p_i(d_i) (the filtered
 * target probability of the draft token) and q_i(d_i) (the filtered draft
 * probability; both 0 when the token is outside the kept set) as the test
 * u < p/q used them, in fp32. Every position of a sampling request is
 * written (the tests run at all positions at once); greedy requests' entries
 * are left untouched. Otherwise identical to dflash_verify: same arguments,
 * outputs, errors and results. The accept rule is standard speculative
 * sampling as the draft/verify loop of "DFlash2 用投机解码给 Qwen 提速"
 * (bml.asia) and step 3 of rytg.cn's "投机解码如何白嫖速度" apply it. */
int dflash_verify_audit(const void* target_logits, const void* draft_logits,
                        const int32_t* draft_tokens, int B, int gamma, int V, int dtype,
                        const float* temperature, int top_k, float top_p, uint64_t seed,
                        int32_t* out_tokens, int32_t* out_accept_len, float* audit_pq,
                        void* workspace, size_t workspace_bytes, uint32_t* status,
                        void* stream);

/* Greedy verification of every request: a_i = argmax target_logits[b, i, :]
 * (lowest index on ties); n = length of the prefix with draft_tokens[b, i] ==
 * a_i; emits d_0..d_{n-1}, a_n and accept length n + 1. This is the greedy
 * half of the lossless guarantee of "无损加速是真的吗？Qwen3.8-27B-DFlash2如何
 * 保证输出与目标模型完全一致" (rytg.cn, the lossless definition: under greedy
 * decoding the output is identical to the target's own), applied to the
 * draft/verify loop of "DFlash2 用投机解码给 Qwen 提速" (bml.asia). Draft
 * logits are not needed. Arguments as for dflash_verify (workspace sized with
 * top_k = 1, top_p = 1). */
int dflash_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B,
                         int gamma, int V, int dtype, int32_t* out_tokens,
                         int32_t* out_accept_len, void* workspace, size_t workspace_bytes,
                         uint32_t* status, void* stream);

/* Verification of deterministic drafts: the drafter proposes d_i with
 * certainty, as a greedy drafter does ("DFlash2 用投机解码给 Qwen 提速",
 * bml.asia: the drafter of the speculative-decoding listing) or a path
 * selector does (rytg.cn, section "轻量选择器": one coherent path picked
 * from the top-16 candidates per position). Its distribution is then the
 * point mass q_i = delta_{d_i}, and the standard rule with that q reads:
 * accept d_i when u < p_i(d_i) (fp32); at the first rejection draw from p_i
 * with d_i taken out (max(0, p_i - delta_{d_i}), renormalised); when every
 * draft is accepted draw the bonus token from p_gamma. The output follows the
 * target distribution whatever the drafts are. No draft logits are read, so
 * a sampling request reads gamma + 1 rows instead of 2 gamma + 1.
 * Arguments, uniforms, draws, greedy requests (T == 0), outputs and status
 * bits as for dflash_verify without draft_logits; workspace_bytes >=
 * dflash_workspace_bytes(...) of the same shape and filter. Filters as for
 * dflash_verify: top-k on (1 <= top_k <= DFLASH_MAX_TOP_K, top_k < V) with any
 * top_p, or top-k off with any top_p, where the residual p without d is
 * drawn over the whole vocabulary (its kept set when top_p < 1) in
 * float-float. */
int dflash_verify_det(const void* target_logits, const int32_t* draft_tokens, int B, int gamma,
                      int V, int dtype, const float* temperature, int top_k, float top_p,
                      uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len,
                      void* workspace, size_t workspace_bytes, uint32_t* status, void* stream);

/* dflash_verify with [host] inputs and outputs: copies the logits (the draft
 * rows of sampling requests only), drafts and temperatures into the caller's
 * [device] staging buffer, verifies, copies tokens, accept lengths and the
 * status word back, and waits for `stream`. Pinned host memory makes the
 * copies asynchronous. staging_bytes >= dflash_host_staging_bytes(...). */
size_t dflash_host_staging_bytes(int B, int gamma, int V, int dtype);
int dflash_verify_host(const void* target_logits, const void* draft_logits,
                       const int32_t* draft_tokens, int B, int gamma, int V, int dtype,
                       const float* temperature, int top_k, float top_p, uint64_t seed,
                       int32_t* out_tokens, int32_t* out_accept_len, uint32_t* out_status,
                       void* staging, size_t staging_bytes, void* workspace,
                       size_t workspace_bytes, void* stream);

/* ---- Vocabulary-sharded verification ----------------------------------------
 * When each rank holds a slice of the vocabulary of every logits row (a
 * vocabulary-parallel LM head under tensor parallelism, as the target runs in
 * the TP=4 measurement of "DFlash2 用投机解码给 Qwen 提速" (bml.asia, the
 * 8xRTX 3090 paragraph) and in the --tp-size 8 launch command of "你的大模型
 * 为啥突然快了，下一代投机解码 DFlash 拆给你看" (xiaodao.ai), the step needs
 * one exchange: every rank reduces its shard to a record (per row its k
 * largest (logit, token) pairs and its largest logit), the ranks all-gather
 * the records, and every rank verifies from the gathered records with
 * identical uniforms. The union of
 * the shards' top k of a row holds the row's global top k, so the outputs
 * (tokens, accept lengths, status bits) equal dflash_verify's on the whole
 * rows, bit for bit, whenever k >= top_k.
 *
 * A record is dflash_candidates_words(B, gamma, k) 32-bit words: the target
 * rows' [B*(gamma+1), k] candidate logits (fp32 bits; -inf past the shard's
 * tokens), their [B*(gamma+1), k] global token ids (int32; -1 there), the
 * target rows' largest logits [B*(gamma+1)] (fp32; NaN when the shard row
 * holds a NaN), then the same three arrays for the draft rows [B*gamma].
 * Candidates are in (logit desc, token asc) order. 0 for invalid arguments
 * (1 <= k <= DFLASH_MAX_TOP_K). */
size_t dflash_candidates_words(int B, int gamma, int k);

/* Device workspace dflash_shard_candidates needs (0 if invalid; needs
 * k < V_shard). */
size_t dflash_shard_workspace_bytes(int B, int gamma, int V_shard, int dtype, int k);

/* One rank's record. target_shard [device] [B, gamma+1, V_shard] and
 * draft_shard [device] [B, gamma, V_shard] (dtype) hold the logits of tokens
 * vocab_offset .. vocab_offset + V_shard - 1 of every row; record [device]
 * (4-byte aligned) receives dflash_candidates_words(B, gamma, k) words.
 * Draft rows of greedy requests are read like the others (any finite values
 * will do). Needs 1 <= k <= DFLASH_MAX_TOP_K, k < V_shard. Raises no status
 * bits: whether a row is bad is decided from all shards' records. */
int dflash_shard_candidates(const void* target_shard, const void* draft_shard, int B, int gamma,
                            int V_shard, int dtype, int vocab_offset, int k, uint32_t* record,
                            void* workspace, size_t workspace_bytes, uint32_t* status,
                            void* stream);

/* Verification from the records of n_shards shards that cover [0, V)
 * without overlap. records [device] [n_shards, dflash_candidates_words(B,
 * gamma, k)], in any shard order. Needs 1 <= top_k <= k and top_k < V,
 * n_shards * k <= 256. Other arguments, outputs, uniforms and status bits as
 * for dflash_verify (no workspace). The full-vocabulary filter (top-k off)
 * returns DFLASH_ERR_UNSUPPORTED. */
int dflash_verify_candidates(const uint32_t* records, int n_shards, int k,
                             const int32_t* draft_tokens, int B, int gamma, int V,
                             const float* temperature, int top_k, float top_p, uint64_t seed,
                             int32_t* out_tokens, int32_t* out_accept_len, uint32_t* status,
                             void* stream);

/* Filtered distribution of R rows: for row r, the kept tokens in (logit
 * desc, index asc) order, out_idx[r, 0..n-1], their probabilities
 * out_prob[r, 0..n-1] (fp32) and n = out_count[r] (slots n..top_k-1 hold -1
 * and 0). temperature [device] [R] > 0. Requires 1 <= top_k <=
 * DFLASH_MAX_TOP_K. logits [device] [R, V]. */
int dflash_filter(const void* logits, int R, int V, int dtype, const float* temperature,
                  int top_k, float top_p, int32_t* out_idx, float* out_prob,
                  int32_t* out_count, void* workspace, size_t workspace_bytes,
                  uint32_t* status, void* stream);

/* One token per row from its filtered distribution (the drafter's side of
 * the loop): temperature[r] == 0 takes the argmax; otherwise the inverse CDF
 * in ascending token order with the accept uniform of Philox counter
 * (r, 0, 1, 0). out_tokens [device] int32 [R]. Filters: top-k on as for
 * dflash_verify, or top-k off with any top_p (drawn over the whole
 * vocabulary, or its top-p set, in float-float). */
int dflash_sample(const void* logits, int R, int V, int dtype, const float* temperature,
                  int top_k, float top_p, uint64_t seed, int32_t* out_tokens, void* workspace,
                  size_t workspace_bytes, uint32_t* status, void* stream);

/* The uniforms the step draws: out_accept[b * npos + i] and
 * out_draw[b * npos + i] for counter (i, b, stream_id, 0) under `seed`
 * ([device] float arrays of B * npos). For audits and tests. */
int dflash_uniforms(uint64_t seed, int B, int npos, int stream_id, float* out_accept,
                    float* out_draw, void* stream);

/* dflash_verify without a caller-provided workspace, for callers that cannot
 * allocate device memory: code running under another framework's memory pool
 * that forbids foreign cudaMalloc calls, plugins loaded into a process whose
 * allocator they do not own, or paths where an allocation (or the device-wide
 * synchronisation a cudaFree can cause) is not allowed. The pages describe no
 * such entry point; it is a convenience of this library.
 *
 * Scratch comes from a fixed array of dflash_noalloc_scratch_bytes() bytes
 * (4 MiB) that the library keeps on every GPU that loads it, until the process
 * exits. Shapes whose workspace (dflash_workspace_bytes) exceeds it return
 * DFLASH_ERR_INVALID_ARG with a message naming the sizes. The first call on a
 * device looks the array up with that device current; make that first call
 * before any stream capture. Each call clears the part of the array it uses
 * on `stream` before the kernel runs (one memset of dflash_workspace_bytes()
 * of its shape: about 3.6 MB at B = 32, block 8, V = 248320 bf16), and every
 * call on a device shares the one array: calls that may overlap on the GPU
 * (other streams, other threads) race and must be ordered by the caller.
 * dflash_workspace_cancel cannot reach this array (its address is not
 * handed out), so such a call cannot be cancelled: it ends when its work is
 * done or its bounded waits (2 s each) give up. Nothing here allocates or
 * frees memory. Arguments and results as for dflash_verify, including the
 * code and message for an invalid or unsupported shape or filter. */
size_t dflash_noalloc_scratch_bytes(void);
int dflash_verify_noalloc(const void* target_logits, const void* draft_logits,
                          const int32_t* draft_tokens, int B, int gamma, int V, int dtype,
                          const float* temperature, int top_k, float top_p, uint64_t seed,
                          int32_t* out_tokens, int32_t* out_accept_len, uint32_t* status,
                          void* stream);

/* ---- the LM head on the tensor cores -------------------------------------------------
 * The draft/verify loop ("DFlash2 用投机解码给 Qwen 提速", bml.asia, the
 * listing of the loop) runs the target over the block and verifies from its
 * logits: logits = h W^T, with h the positions' last hidden states and W the
 * vocabulary projection.
 *
 * dflash_lmhead_logits: logits [M, V] = h [M, K] W^T for h [M, K] and W [V, K],
 * all bf16 row-major [device], fp32 accumulation on the tensor cores, each
 * logit rounded to the nearest bf16 (ties to even). 1 <= M <= 512; V a
 * positive multiple of 8; K a positive multiple of 64; h, W and logits
 * 16-byte aligned (caller-owned; logits is overwritten). status may be NULL
 * (a bounded wait that gave up ORs DFLASH_STATUS_TIMEOUT into it). */
int dflash_lmhead_logits(const void* h, const void* w, int M, int V, int K, void* logits, uint32_t* status,
                         void* stream);

/* dflash_lmhead_verify: the LM head and dflash_verify in one, without the
 * verification's pass over the logits. h holds the B (gamma + 1) target rows
 * ([B, gamma + 1, K]) and then the B gamma draft rows ([B, gamma, K]), bf16;
 * logits [B (2 gamma + 1), V] bf16 receives the target logits and then the
 * draft logits (the verification's target_logits and draft_logits). The
 * GEMM's epilogue writes the statistics the verification would have taken
 * from them (each 256-logit tile's maximum for the top-k rows, the argmax of
 * the greedy rows) into the workspace; the verification then runs only its
 * row and request finals. Outputs, uniforms, status bits and workspace rules
 * are those of dflash_verify on the same logits (the outputs equal
 * dflash_lmhead_logits followed by dflash_verify bit for bit). Shape limits
 * as for dflash_lmhead_logits with M = B (2 gamma + 1) <= 512; the top-k
 * filter only (1 <= top_k <= DFLASH_MAX_TOP_K, top_k < V, any top_p; others
 * return DFLASH_ERR_UNSUPPORTED). workspace_bytes >= dflash_workspace_bytes(B,
 * gamma, V, DFLASH_BF16, top_k, top_p). */
int dflash_lmhead_verify(const void* h, const void* w, int B, int gamma, int V, int K,
                         const int32_t* draft_tokens, const float* temperature, int top_k, float top_p,
                         uint64_t seed, void* logits, int32_t* out_tokens, int32_t* out_accept_len,
                         void* workspace, size_t workspace_bytes, uint32_t* status, void* stream);

#ifdef __cplusplus
}
#endif
#endif /* DFLASH_VERIFY_H */
