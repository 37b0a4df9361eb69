/*
 * spec_sample.h -- C ABI of batched token sampling on GB300 (sm_103a): one
 * token per row drawn from softmax(logits / T) by inverse CDF with a caller
 * uniform, reading every logit once.
 *
 * This is the drafting step that precedes verification in speculative
 * decoding: the draft model proposes each of its k tokens by sampling from its
 * own next-token distribution q ("Speculative Decoding and the Art of Fast LLM
 * Inference", "The Algorithm, Step by Step", the drafting step; the
 * techaiinterview answer "How does speculative decoding work, why is it
 * lossless, and how much does it speed things up?", "Algorithm (one round)",
 * step 1).  The pages do not spell the sampler out; it uses the same reading
 * as the verification's correction and bonus draws (spec_verify.h):
 *
 *   T > 0:  w(x) = exp((l(x) - m) / T) with m the row maximum (any positive
 *           multiple of softmax(l / T) gives the same draw);
 *           C(x) = sum_{y <= x} w(y), R = C(V-1);
 *           token = the smallest x with C(x) > u * R, or, if rounding leaves
 *           no such x, the largest x with w(x) > 0.
 *   T == 0: token = argmax l, the lowest index on ties; u is not read.
 *
 * Row errors (token -1): T NaN, negative, infinite or positive below
 * FLT_MIN; a NaN or +inf logit in the row; every logit of the row -inf.
 * -inf logits are allowed and are never drawn.
 *
 * Errors, status codes, dtypes and the device status word are those of
 * spec_verify.h; spec_verify_read_status and spec_verify_workspace_reset work
 * on a sampling workspace too (its first 256 bytes are the same header).
 */
#ifndef SPEC_SAMPLE_H
#define SPEC_SAMPLE_H

#include <stddef.h>
#include <stdint.h>

#include "spec_verify.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * Bytes of device workspace one spec_sample call needs: the 256-byte header,
 * an 8-byte record per 4 KB chunk of every row (R * ceil(V * elem / 4096)
 * records), and room for the exact draw of every row (100 bytes plus 32 bytes
 * per 2048 elements of a row).  Returns 0 for sizes out of range (R < 0,
 * V < 2, V > SPEC_MAX_V, unknown dtype).  Host-only; needs no GPU.
 */
size_t spec_sample_workspace_size(int32_t R, int32_t V, int32_t dtype);

/*
 * Sample one token per row.
 *   logits       device, [R, V] of dtype, row-major, 16-byte aligned base
 *   u            device float32 [R], each in [0, 1): the row's uniform
 *   temperature  device float32 [R] >= 0; 0 selects the argmax
 *   out_tokens   device int32 [R]: the drawn token, or -1 on a row error
 *   workspace    device scratch, >= spec_sample_workspace_size(R, V, dtype)
 *                bytes, 16-byte aligned; only its status word must be zero
 *                beforehand (see SPEC_DEV_OK).  Two calls in flight at once
 *                must not share one.
 *   stream       cudaStream_t as void*.
 * Four kernels run in order on `stream`: chunk records (the one read of the
 * logits), the per-row pick, and the exact draws (two kernels) of the rows
 * whose fp32 pick landed within 1.2e-6 of R of a cell edge: their weights in
 * float-float arithmetic and exact fixed-point sums (about 1e-12 of R), so a
 * token equals the exactly rounded draw unless u lies within ~1e-12 of an
 * edge.  With no row listed the last two only read the count.  Returns
 * SPEC_OK once they are launched
 * (R == 0 launches nothing); SPEC_EINVAL for bad sizes, null or misaligned
 * pointers; SPEC_ENOSPACE for a short workspace; SPEC_ECUDA for a failed
 * launch.
 */
int32_t spec_sample(const void *logits, const float *u, const float *temperature,
                    int32_t *out_tokens, int32_t R, int32_t V, int32_t dtype,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_sample recording the caller's cudaEvent_t handles (SPEC_SAMPLE_STAGES
 * of them; the array and its entries may be NULL) on `stream` after each
 * stage: chunk records, pick, exact draws.  Used to time the HBM-bound first
 * kernel.
 */
#define SPEC_SAMPLE_STAGES 3
int32_t spec_sample_timed(const void *logits, const float *u, const float *temperature,
                          int32_t *out_tokens, int32_t R, int32_t V, int32_t dtype,
                          void *workspace, size_t workspace_bytes, void *stream,
                          void *const *stage_events);

/*
 * Bytes of caller-owned device arena spec_sample_host needs: device copies of
 * the inputs and the output plus the workspace, each 256-byte aligned.
 * Returns 0 for sizes out of range.
 */
size_t spec_sample_host_arena_size(int32_t R, int32_t V, int32_t dtype);

/*
 * End-to-end variant on HOST buffers: copies logits, u and temperature
 * host->device into the caller's device arena (one cudaMemcpyAsync each),
 * runs spec_sample, copies out_tokens back to the host buffer, all on
 * `stream`, and synchronises the stream before returning.  Pinned host memory
 * makes the copies asynchronous DMA.  The arena must be
 * >= spec_sample_host_arena_size(...) bytes and 256-byte aligned; the status
 * word of its workspace part is zeroed by this call.
 */
int32_t spec_sample_host(const void *logits, const float *u, const float *temperature,
                         int32_t *out_tokens, int32_t R, int32_t V, int32_t dtype,
                         void *device_arena, size_t arena_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_SAMPLE_H */
