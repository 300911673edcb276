/*
 * dflash_oracle.h -- CPU oracle for the batched draft-verification step of
 * block-drafted speculative decoding.
 *
 * TEST INFRASTRUCTURE. This library exists only to check the GPU library
 * against a plain, slow, fp64 restatement of the method. Only the tests, the
 * smoke check and the CPU-baseline leg of the benchmark load it. It shares no
 * code, header, table or constant with the GPU library.
 *
 * Sources the arithmetic follows (see dflash_oracle.c for per-function notes):
 *  - "DFlash2 用投机解码给 Qwen 提速" (bml.asia), the draft/verify loop
 *    pseudocode: verify draft tokens in order, accept or resample from the
 *    target's own distribution at the first rejection and stop; and the
 *    model-card sampling settings (temperature 1.0, top-p 0.95, top-k 20,
 *    block size 8).
 *  - "无损加速是真的吗？Qwen3.8-27B-DFlash2如何保证输出与目标模型完全一致"
 *    (rytg.cn), section "投机解码如何白嫖速度" (steps 1-4, step 3 "裁决")
 *    and the lossless definition: greedy output identical to the target,
 *    sampling preserves the target distribution.
 *  - Standard speculative sampling: accept with probability min(1, p/q),
 *    otherwise sample the normalised residual max(0, p - q); a bonus token from
 *    the target's last position when every draft is accepted.
 *  - Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As
 *    Easy as 1, 2, 3", SC'11.
 */
#ifndef DFLASH_ORACLE_H
#define DFLASH_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BF16 = 0, ORC_F32 = 1 };

/* status bits, OR-ed per call */
enum {
  ORC_STATUS_BAD_TOKEN = 1u,       /* a draft token outside [0, V) */
  ORC_STATUS_BAD_ROW = 2u,         /* a logits row with a NaN, or a non-finite max */
  ORC_STATUS_BAD_TEMPERATURE = 8u  /* temperature negative, NaN or infinite */
};

/* return codes */
enum { ORC_OK = 0, ORC_ERR_INVALID_ARG = 1, ORC_ERR_NOMEM = 3 };

/* Philox4x32-10 block function: out = philox(ctr, key). */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* The two uniforms in [0,1) drawn for (seed, request, position, stream):
 * key = (seed low word, seed high word), counter = (position, request,
 * stream, 0); u_accept from output word 0, u_draw from output word 1, each
 * as (w >> 8) * 2^-24. Verification uses stream 0, filtered sampling stream 1. */
void oracle_uniforms(uint64_t seed, uint32_t request, uint32_t position, uint32_t stream,
                     float* u_accept, float* u_draw);

/* Largest logit of a row with the lowest index among equal values.
 * Returns the index; *status gets ORC_STATUS_BAD_ROW for a NaN or a
 * non-finite maximum. */
int32_t oracle_argmax_row(const void* row, int V, int dtype, uint32_t* status);

/* The filtered distribution of one row, dense over the vocabulary:
 * prob[j] = filtered probability of token j in fp64 (0 outside the kept set).
 * temperature > 0; top_k <= 0 or >= V disables top-k; top_p >= 1 disables
 * top-p. Returns the kept-set size (>= 1) or -1 for a bad row. */
int oracle_filter_row(const void* row, int V, int dtype, double temperature, int top_k,
                      float top_p, double* prob);

/* The kept set of a row in (logit desc, index asc) order: idx[0..n-1] and
 * their probabilities; returns n or -1. idx/prob need V entries. */
int oracle_filter_row_sparse(const void* row, int V, int dtype, double temperature, int top_k,
                             float top_p, int32_t* idx, double* prob);

/* Batched verification for requests [b_begin, b_end) of a batch of B.
 * target: [B, gamma+1, V]; draft: [B, gamma, V]; draft_tokens: [B, gamma];
 * temperature: [B] (0 = greedy for that request).
 * out_tokens: [B, gamma+1] (-1 padded), out_accept_len: [B].
 * margin (optional, [B]): the smallest gap between the two sides of any fp32
 * decision the request took (diagnostic for near-boundary rows): relative
 * for the accept tests (|u - p/q| / (p/q)) and the top-p cuts
 * (|mass before - top_p| / top_p), absolute for the inverse-CDF draw
 * (|u * total - cumulative weight|, the weights being probabilities).
 * status (optional): OR of ORC_STATUS_* over the processed requests. */
int oracle_verify(const void* target, const void* draft, const int32_t* draft_tokens, int B,
                  int gamma, int V, int dtype, const float* temperature, int top_k, float top_p,
                  uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len, double* margin,
                  uint32_t* status, int b_begin, int b_end);

/* oracle_verify with the decision margins split: margin_draw ([B], optional)
 * covers the final residual or bonus draw; margin_cut ([B], optional) the
 * top-p cuts of every row the request filters (the mass before a token
 * grows along the sorted order, so the smallest gap is at the cut itself);
 * margin_accept ([B], optional) the accept tests, and also the cuts when
 * margin_cut is NULL. Over the full vocabulary neighbouring cumulative
 * weights are a few parts per million apart, so the draw's and the cuts'
 * margins are small on every row while the accept margins are not. */
int oracle_verify_margins(const void* target, const void* draft, const int32_t* draft_tokens,
                          int B, int gamma, int V, int dtype, const float* temperature, int top_k,
                          float top_p, uint64_t seed, int32_t* out_tokens,
                          int32_t* out_accept_len, double* margin_accept, double* margin_draw,
                          double* margin_cut, uint32_t* status, int b_begin, int b_end);

/* Verification of deterministic drafts (q = the point mass at d_i): accept
 * d_i when u < p_i(d_i); at the first rejection draw from p_i with d_i taken
 * out; otherwise the bonus token from p_gamma. No draft logits. Arguments and
 * outputs as oracle_verify_margins without `draft`. */
int oracle_verify_det_margins(const void* target, const int32_t* draft_tokens, int B, int gamma,
                              int V, int dtype, const float* temperature, int top_k, float top_p,
                              uint64_t seed, int32_t* out_tokens, int32_t* out_accept_len,
                              double* margin_accept, double* margin_draw, double* margin_cut,
                              uint32_t* status, int b_begin, int b_end);

/* Greedy verification: argmax prefix match, requests [b_begin, b_end). */
int oracle_verify_greedy(const void* target, const int32_t* draft_tokens, int B, int gamma, int V,
                         int dtype, int32_t* out_tokens, int32_t* out_accept_len,
                         uint32_t* status, int b_begin, int b_end);

/* One token per row from that row's filtered distribution (rows [r_begin,
 * r_end) of R): temperature[r] == 0 gives the argmax; otherwise the inverse
 * CDF in ascending token order with u_accept of (seed, request=0,
 * position=r, stream=1). */
int oracle_sample_rows(const void* logits, int R, int V, int dtype, const float* temperature,
                       int top_k, float top_p, uint64_t seed, int32_t* out_tokens,
                       double* margin, uint32_t* status, int r_begin, int r_end);

#ifdef __cplusplus
}
#endif
#endif
