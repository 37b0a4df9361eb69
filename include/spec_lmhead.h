/*
 * spec_lmhead.h -- C ABI of speculative-sampling verification with the
 * target's LM head fused in, on GB300 (sm_103a).
 *
 * The verify step scores all k+1 positions with one target forward pass
 * ("Speculative Decoding and the Art of Fast LLM Inference", "The Algorithm,
 * Step by Step", the verify step; the techaiinterview answer "How does
 * speculative decoding work, why is it lossless, and how much does it speed
 * things up?", "Algorithm (one round)", step 2).  The last layer of that pass
 * maps each position's hidden state h (length d) to the target logits
 * t = h W^T over the vocabulary (W is the [V, d] LM-head matrix).  Here that
 * product runs on the tensor cores and is reduced to row statistics in the
 * GEMM epilogue, so the logits never reach HBM; only the one row per
 * sequence that a draw needs is computed a second time.
 *
 * What is computed is spec_verify (include/spec_verify.h) on
 * target_logits[b][i][x] = sum_j hidden[b][i][j] * lm_head[x][j]
 * (bf16 inputs, products exact, fp32 accumulation): the accept tests, the
 * first rejection, the residual max(0, p - q) or bonus draw by inverse CDF,
 * the greedy rule at T = 0, and the same sequence errors.  The draft side is
 * given as logits, as for spec_verify.
 *
 * Layouts (all device memory, row-major, caller-owned):
 *   hidden       bf16 [B, k+1, d]   the target's hidden states at the k+1
 *                                   positions, 16-byte aligned base
 *   lm_head      bf16 [V, d]        W, 16-byte aligned base
 *   draft_logits [B, k, V] of draft_dtype (SPEC_F32 or SPEC_BF16), 16-byte
 *                                   aligned base
 *   other arguments as spec_verify.
 * Sizes: B >= 1, 1 <= k <= 31 (the accept scan holds a sequence's k+1
 * positions in one warp), 2 <= V <= SPEC_MAX_V, d a multiple of 64 in
 * [64, 16384], and at most 2^30 GEMM tiles of 128 rows x 256 columns over
 * the B(k+1) x V target logits.
 *
 * Calls may come from several host threads at once, each with its own
 * workspace.
 */
#ifndef SPEC_LMHEAD_H
#define SPEC_LMHEAD_H

#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Bytes of device workspace one spec_verify_lmhead call needs (the 256-byte
 * status header, per-tile row statistics of the B(k+1) target rows, the
 * draft chunk records, the draw rows' hidden vectors and group sums).
 * Returns 0 for sizes out of range.  Host-only.
 */
size_t spec_verify_lmhead_workspace_size(int32_t B, int32_t k, int32_t V, int32_t d,
                                         int32_t draft_dtype);

/*
 * The verification step with the LM head fused in.  Asynchronous on `stream`
 * (cudaStream_t as void*); returns SPEC_OK once the five kernels are launched
 * (draft chunk records, GEMM with the statistics epilogue, accept scan, GEMM
 * of the draw rows, final search).  SPEC_EINVAL for bad sizes, null or
 * misaligned pointers; SPEC_ENOSPACE for a short workspace; SPEC_ECUDA for a
 * failed launch or a failed tensor-map encoding.  Outputs and sequence errors
 * as spec_verify; the workspace's status word must be zero beforehand
 * (SPEC_DEV_OK) and reads SPEC_DEV_WAIT_TIMEOUT if a bounded wait gave up.
 * Two calls in flight must not share a workspace.
 */
int32_t spec_verify_lmhead(const void *hidden, const void *lm_head, const void *draft_logits,
                           const int32_t *draft_tokens, const float *u_accept,
                           const float *u_resample, const float *temperature,
                           int32_t *out_tokens, int32_t *out_num_accepted,
                           int32_t B, int32_t k, int32_t V, int32_t d, int32_t draft_dtype,
                           void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify_lmhead recording the caller's cudaEvent_t handles after each
 * of its SPEC_LMHEAD_STAGES kernels (NULL entries skipped), in the order
 * above; kernels then start in plain stream order.  `out_probs` (device
 * float32 [B, k, 2], or NULL) receives P = p_i(g_i) and Q = q_i(g_i) of
 * every position of a sampled sequence (NaN elsewhere).
 */
#define SPEC_LMHEAD_STAGES 5
int32_t spec_verify_lmhead_timed(const void *hidden, const void *lm_head,
                                 const void *draft_logits, const int32_t *draft_tokens,
                                 const float *u_accept, const float *u_resample,
                                 const float *temperature, int32_t *out_tokens,
                                 int32_t *out_num_accepted, float *out_probs,
                                 int32_t B, int32_t k, int32_t V, int32_t d,
                                 int32_t draft_dtype, void *workspace, size_t workspace_bytes,
                                 void *stream, void *const *stage_events);

/*
 * The fused GEMM alone, storing its fp32 result: out[r][x] = sum_j
 * hidden[r][j] * lm_head[x][j] for r < M, x < V (out device float32 [M, V]).
 * For checking the tensor-core product; the verification never stores it.
 * hidden bf16 [M, d], lm_head bf16 [V, d]; `status` device int32 (the bounded
 * waits' status word, zero beforehand).  M >= 1, V and d as above, with the
 * same tile-count limit.  Returns a SPEC_* code as above.
 */
int32_t spec_lmhead_logits(const void *hidden, const void *lm_head, float *out, int32_t M,
                           int32_t V, int32_t d, int32_t *status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_LMHEAD_H */
