/*
 * spec_verify.h -- C ABI of the GB300 speculative-sampling verification library
 * (libspecverify.so).
 *
 * The operation (one round of speculative decoding's verification step, for a
 * batch of B independent sequences):
 *   - p_i = softmax(t_i / T) and q_i = softmax(d_i / T) with the same per-
 *     sequence temperature T for target and draft ("Speculative Decoding and
 *     the Art of Fast LLM Inference", "Why It Stays Exact", key limitation on
 *     identical sampling parameters);
 *   - left to right, draft token g_i is accepted when u_accept[b,i] is strictly
 *     below p_i(g_i)/q_i(g_i) (always when p_i(g_i) >= q_i(g_i)); the first
 *     rejection ends the scan (same page, "The Algorithm, Step by Step";
 *     thelatentsource "speculative-decoding-llm-speed", "The correction that
 *     keeps the target in charge", the accept_token snippet);
 *   - at the rejected position j one correction token is drawn from
 *     norm(max(0, p_j - q_j)) (second page, equation r(x)); if all k drafts are
 *     accepted a bonus token is drawn from p_{k+1} (first page, step "Bonus
 *     token");
 *   - a draw is inverse-CDF with u_resample[b]: the smallest token x whose
 *     running mass C(x) exceeds u * R, R the total mass (the pages say
 *     "sample"; this is the plain reading).  Draws are computed in fp32; a
 *     draw whose u * R falls within ~1e-6 of its cell's edge in fp32 is
 *     computed again in float-float arithmetic with exact fixed-point sums
 *     (about 1e-12 of R), so the token equals the exactly rounded result
 *     except for uniforms within ~1e-12 of an edge;
 *   - T == 0 is greedy mode: g_i is accepted while it equals argmax t_i, and the
 *     correction or bonus is the target argmax ("How does speculative decoding
 *     work, why is it lossless, and how much does it speed things up?",
 *     techaiinterview, "Deep dive: correctness and speedup").  Argmax ties go to
 *     the lowest index.  Draft logits are not read for greedy sequences.
 *
 * Conventions shared by every entry point:
 *   - Sizes are int32; B >= 0 (B == 0 is a no-op), 1 <= k <= SPEC_MAX_K,
 *     2 <= V <= SPEC_MAX_V.
 *   - Logits are row-major; target [B, k+1, V], draft [B, k, V]; one dtype per
 *     call (SPEC_F32 = IEEE binary32, SPEC_BF16 = bfloat16 bit patterns).
 *     Their base addresses must be 16-byte aligned; V is arbitrary.
 *   - Device entry points take device pointers and a cudaStream_t passed as
 *     void* (NULL = the legacy default stream).  They launch on that stream and
 *     return without synchronising; results are valid once the stream has
 *     reached that point.
 *   - The library allocates no memory and keeps no per-call global state.  The
 *     caller owns every buffer.  Inputs are read-only; outputs are overwritten.
 *   - Entry points may be called from several host threads at once, each call
 *     with its own workspace (the library's only shared state is a per-device
 *     cache of launch facts, published atomically).
 *   - The return value reports host-checkable errors only (spec_status_t).
 *     Data-dependent problems are reported per sequence on the device:
 *     out_num_accepted[b] = -1 and out_tokens[b, :] = -1 when T is NaN,
 *     negative, infinite or positive below FLT_MIN; a draft token lies outside
 *     [0, V); a logit the call reads is NaN or +inf; such a row is entirely
 *     -inf; or the draft probability of a draft token the scan reaches is zero
 *     (the accept_token snippet's ValueError).  Nothing traps and nothing
 *     prints on the device.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_VERIFY_ABI_VERSION 2
#define SPEC_MAX_K 32
#define SPEC_MAX_V (1 << 20)

typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype_t;

typedef enum {
    SPEC_OK = 0,
    SPEC_EINVAL = 1,   /* a null pointer, a size out of range, misalignment, unknown dtype */
    SPEC_ECUDA = 2,    /* a CUDA runtime call or the launch failed */
    SPEC_ENOSPACE = 3  /* workspace (or arena) smaller than the size query returned */
} spec_status_t;

/* Device-side status word, the first 4 bytes of the workspace (read it with
 * spec_verify_read_status).  Nonzero means a kernel stopped early after a
 * bounded wait ran out: the outputs of that call are undefined.  Only a
 * timed-out wait writes it; zero it (spec_verify_workspace_reset) to clear. */
#define SPEC_DEV_OK 0
#define SPEC_DEV_WAIT_TIMEOUT 1

/* ABI version of the loaded library (SPEC_VERIFY_ABI_VERSION). */
int32_t spec_verify_abi_version(void);

/* Human-readable name of a spec_status_t value (static string). */
const char *spec_verify_strerror(int32_t status);

/*
 * Bytes of device workspace one spec_verify call needs for these sizes: a
 * 256-byte header (the status word), one 16-byte partial per 128 KB of every
 * row, and per sequence an 80-byte draw record, its inverse-CDF chunk totals
 * (32 bytes per 16 KB of a row), its bonus row's chunk records (8 bytes per
 * 4 KB of a row), a 16-byte top-k / top-p record per row (read by
 * spec_verify_filtered only), and room for its exact draw (2148 bytes plus
 * 32 bytes per 2048 elements of a row).  Returns 0 for sizes out of range.
 * Host-only; needs no GPU.
 */
size_t spec_verify_workspace_size(int32_t B, int32_t k, int32_t V, int32_t dtype);

/*
 * Zero a workspace on `stream` (cudaMemsetAsync).  Only the status word is
 * read across calls: zero it once after allocation, and again after a call
 * whose device status was nonzero.  Nothing else in the workspace carries
 * over from one call to the next.
 */
int32_t spec_verify_workspace_reset(void *workspace, size_t workspace_bytes, void *stream);

/*
 * The verification step (see the file comment for the operation).
 *   target_logits    device, [B, k+1, V] of dtype; t_1..t_k then the bonus row t_{k+1}
 *   draft_logits     device, [B, k, V] of dtype; never read for sequences with T == 0
 *   draft_tokens     device int32 [B, k]: g_1..g_k
 *   u_accept         device float32 [B, k], each in [0, 1): accept test i uses u_accept[b, i]
 *   u_resample       device float32 [B] in [0, 1): the one correction or bonus draw
 *   temperature      device float32 [B] >= 0; 0 selects greedy mode
 *   out_tokens       device int32 [B, k+1]: accepted prefix, then the correction or
 *                    bonus token, then -1 padding (all -1 on a sequence error)
 *   out_num_accepted device int32 [B]: accepted drafts in [0, k]; -1 = sequence error.
 *                    The sequence emits out_num_accepted[b] + 1 tokens.
 *   workspace        device scratch, >= spec_verify_workspace_size(...) bytes, 16-byte
 *                    aligned.  Its contents need no initialisation apart from the status
 *                    word (see SPEC_DEV_OK).  Two calls in flight at once must not share
 *                    one (the same stream runs calls in order, so one per stream suffices).
 *   stream           cudaStream_t as void*.
 * Five kernels run in order on `stream`: row statistics, accept scan, draw
 * tiles, final search, exact draws (of the sequences the final search listed;
 * with none listed it only reads the count).  Returns SPEC_OK once they are
 * launched; errors are listed above.
 */
int32_t spec_verify(const void *target_logits, const void *draft_logits,
                    const int32_t *draft_tokens, const float *u_accept,
                    const float *u_resample, const float *temperature,
                    int32_t *out_tokens, int32_t *out_num_accepted,
                    int32_t B, int32_t k, int32_t V, int32_t dtype,
                    void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify plus the intermediate probabilities P = p_i(g_i) and
 * Q = q_i(g_i) for every draft position, written to out_probs (device float32
 * [B, k, 2]; NaN for greedy and error sequences).  Same arguments otherwise;
 * used to check intermediates against an fp64 reference.
 */
int32_t spec_verify_probs(const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *u_accept,
                          const float *u_resample, const float *temperature,
                          int32_t *out_tokens, int32_t *out_num_accepted, float *out_probs,
                          int32_t B, int32_t k, int32_t V, int32_t dtype,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify with a trace of each draw, for checking the draw against a
 * reference: out_draw (device int32 [B, 4]) receives, for every sequence that
 * draws from a distribution (T > 0, no sequence error), [0] the token of the
 * fp32 search, [1] 1 if the draw was listed for the exact recomputation,
 * [2] the token written to out_tokens, [3] the bits of a float: the fp32
 * search's distance from u to the nearer edge of the cell it chose, as a
 * fraction of the total mass R (0 when a rounding fallback was taken).
 * Other sequences' entries
 * are left as they were.  resolve_all != 0 lists every draw (the exact draw
 * then decides every token).  out_probs as spec_verify_probs, or NULL.
 * Same arguments and behaviour as spec_verify otherwise.
 */
int32_t spec_verify_trace(const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *u_accept,
                          const float *u_resample, const float *temperature,
                          int32_t *out_tokens, int32_t *out_num_accepted, float *out_probs,
                          int32_t *out_draw, int32_t resolve_all,
                          int32_t B, int32_t k, int32_t V, int32_t dtype,
                          void *workspace, size_t workspace_bytes, void *stream);

/*
 * Bytes of workspace with which spec_verify_filtered cuts top-k rows from
 * group maxima: spec_verify_workspace_size rounded up to 256, plus, for each
 * of the B (2k+1) rows, 4 bytes per 64 bf16 (32 fp32) logits (the group
 * maxima), 2048 bytes (up to 256 kept tokens, which the kept-set draws read
 * back) and 4 bytes (their count), each region starting on a 256-byte
 * boundary.  Returns 0 for sizes out of range.  Host-only; needs no GPU.
 */
size_t spec_verify_filtered_workspace_size(int32_t B, int32_t k, int32_t V, int32_t dtype);

/*
 * spec_verify with top-k / top-p filtered distributions.  The pages require
 * draft and target to share their sampling parameters, top-p among them
 * ("Speculative Decoding and the Art of Fast LLM Inference", "Why It Stays
 * Exact", key limitation), without defining the filters; the reading taken:
 * the tokens of a row are ranked by logit, descending, ties by index
 * ascending; top-k keeps the first K of them; top-p keeps, among those, a
 * token while the mass ranked before it is below P times the top-k mass (at
 * least one token stays); p and q are renormalised over their kept sets before
 * the accept test, the residual and the bonus draw.  Greedy sequences (T = 0)
 * are unaffected.
 *   top_k  device int32 [B] or NULL: 0 or >= V = no top-k; < 0 = sequence error
 *   top_p  device float32 [B] or NULL: >= 1 = no top-p; NaN or <= 0 = sequence error
 *   out_probs  device float32 [B, k, 2] or NULL: the filtered P = p~_i(g_i),
 *          Q = q~_i(g_i) (NaN for greedy and error sequences)
 * A draft token outside the draft's kept set (q~(g) = 0) is a sequence error.
 * Other arguments and errors as spec_verify.  The workspace is at least
 * spec_verify_workspace_size bytes; with spec_verify_filtered_workspace_size
 * bytes the rows with top-k (1 <= K <= 256) are cut from per-group maxima the
 * statistics kernel leaves in the extra room (only the groups that can hold
 * a kept token are read again), otherwise every row takes the streaming
 * filter, and those rows' draws come from their kept sets (fp64 weights over
 * at most K tokens) instead of a pass over the row.  The kernels: statistics;
 * the filter (the group-maximum cut of top-k rows when there is room; one
 * streaming pass over each other row; then the rows neither could cut, by a
 * second pass or a radix search over the order key); accept scan; draw tiles
 * and the kept-set draws; final search; exact draws.
 */
int32_t spec_verify_filtered(const void *target_logits, const void *draft_logits,
                             const int32_t *draft_tokens, const float *u_accept,
                             const float *u_resample, const float *temperature,
                             const int32_t *top_k, const float *top_p,
                             int32_t *out_tokens, int32_t *out_num_accepted, float *out_probs,
                             int32_t B, int32_t k, int32_t V, int32_t dtype,
                             void *workspace, size_t workspace_bytes, void *stream);

/*
 * spec_verify_filtered with stage events as in spec_verify_timed:
 * SPEC_FILTERED_STAGES of them, after the statistics, the filter (all of
 * its kernels), the accept scan, the draw tiles (with the kept-set draws),
 * the final search and the exact draws.
 */
#define SPEC_FILTERED_STAGES 6
int32_t spec_verify_filtered_timed(const void *target_logits, const void *draft_logits,
                                   const int32_t *draft_tokens, const float *u_accept,
                                   const float *u_resample, const float *temperature,
                                   const int32_t *top_k, const float *top_p,
                                   int32_t *out_tokens, int32_t *out_num_accepted,
                                   int32_t B, int32_t k, int32_t V, int32_t dtype,
                                   void *workspace, size_t workspace_bytes, void *stream,
                                   void *const *stage_events);

/*
 * spec_verify with per-stage timing: `stage_events` (nullable; entries may be
 * NULL) holds SPEC_STAGES cudaEvent_t handles, created by the caller, that are
 * recorded on `stream` after each stage: row statistics, accept scan, draw
 * tiles, final search, exact draws.  Same arguments and behaviour as
 * spec_verify otherwise.  Lets a benchmark time the HBM-bound statistics
 * stage alone.
 */
#define SPEC_STAGES 5
int32_t spec_verify_timed(const void *target_logits, const void *draft_logits,
                          const int32_t *draft_tokens, const float *u_accept,
                          const float *u_resample, const float *temperature,
                          int32_t *out_tokens, int32_t *out_num_accepted,
                          int32_t B, int32_t k, int32_t V, int32_t dtype,
                          void *workspace, size_t workspace_bytes, void *stream,
                          void *const *stage_events);

/*
 * spec_verify for callers that cannot allocate device memory at the point of
 * the call: for example a plugin inside a host runtime that owns all device
 * memory through its own pool and hands the plugin none, or a latency-critical
 * loop that must not call cudaMalloc (which can synchronise the device).
 * The pages describe no such entry point; it has no counterpart there.
 *
 * Instead of a caller workspace it uses one scratch array of
 * spec_verify_noalloc_max_bytes() bytes (8 MiB) that is part of this library's
 * device code: every GPU that loads the library holds it until the process
 * exits.  Calls whose spec_verify_workspace_size(B, k, V, dtype) exceeds that
 * return SPEC_ENOSPACE and launch nothing (B=256, k=8, V=151936, fp32 needs
 * about 1.8 MiB).  The call allocates nothing: no cudaMalloc, no cudaFree.
 *
 * The first call on a device looks up the array's device address with that
 * device current (cudaGetSymbolAddress) and keeps it; make that first call
 * before any stream capture.  The address is never looked up again, so do
 * not call this after cudaDeviceReset in the same process (the reset unloads
 * the module that holds the array).  Every call clears the array's status
 * word on `stream` before launching.  All calls, on every stream, share the
 * one array, which keeps the last call's contents: calls that overlap on the
 * GPU race and give undefined outputs, so run them one after another (on one
 * stream, or with your own ordering between streams).  Inputs, outputs,
 * return codes and device-side sequence errors are as for spec_verify; a
 * kernel that stopped after a bounded wait ran out is reported by
 * spec_verify_noalloc_read_status (the outputs of that call are undefined).
 */
int32_t spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                            const int32_t *draft_tokens, const float *u_accept,
                            const float *u_resample, const float *temperature,
                            int32_t *out_tokens, int32_t *out_num_accepted,
                            int32_t B, int32_t k, int32_t V, int32_t dtype, void *stream);

/* Size in bytes of the scratch array spec_verify_noalloc uses. */
size_t spec_verify_noalloc_max_bytes(void);

/*
 * The device status word of spec_verify_noalloc's scratch array on the
 * current device, copied to *status (host) after synchronising `stream`:
 * SPEC_DEV_OK after a complete call, SPEC_DEV_WAIT_TIMEOUT if a kernel of the
 * last call stopped after a bounded wait ran out.  The next spec_verify_noalloc
 * call clears it.  Returns SPEC_EINVAL for a null `status`, SPEC_ECUDA if the
 * address cannot be looked up or the copy fails.
 */
int32_t spec_verify_noalloc_read_status(int32_t *status, void *stream);

/*
 * Copy the workspace's device status word to *status (host) and synchronise
 * `stream`.  SPEC_DEV_OK (0) after a complete call.
 */
int32_t spec_verify_read_status(const void *workspace, int32_t *status, void *stream);

/*
 * Bytes of caller-owned device arena spec_verify_host needs: device copies of
 * all inputs and outputs plus the workspace, each 256-byte aligned.
 */
size_t spec_verify_host_arena_size(int32_t B, int32_t k, int32_t V, int32_t dtype);

/*
 * End-to-end variant on HOST buffers: copies the inputs host->device into the
 * caller's device arena (one cudaMemcpyAsync per buffer; the draft rows only
 * of sequences whose host temperature is not 0, one copy per run of such
 * sequences, since the greedy rule never reads draft rows), runs
 * spec_verify, and copies out_tokens / out_num_accepted back to the host
 * buffers, all on `stream`; synchronises the stream before returning so the
 * host outputs are ready.  Pinned host memory makes the copies asynchronous DMA.  The arena
 * must be >= spec_verify_host_arena_size(...) bytes and 256-byte aligned; the
 * status word of its workspace part is zeroed by this call.  Host pointers follow the device
 * entry point's shapes.
 */
int32_t spec_verify_host(const void *target_logits, const void *draft_logits,
                         const int32_t *draft_tokens, const float *u_accept,
                         const float *u_resample, const float *temperature,
                         int32_t *out_tokens, int32_t *out_num_accepted,
                         int32_t B, int32_t k, int32_t V, int32_t dtype,
                         void *device_arena, size_t arena_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
