/*
 * spec_tree.h -- C ABI of tree verification in libspecverify.so: several
 * candidate continuations per sequence, verified together ("Speculative
 * Decoding and the Art of Fast LLM Inference", "Where the Draft Comes From",
 * EAGLE-2/3; techaiinterview, "Drafts and limits", tree verification).
 *
 * The pages name the idea but give no rule for accepting among siblings.  The
 * rule implemented is the one that keeps the first page's exactness argument
 * ("Why It Stays Exact") at every node:
 *   - node 0 is the root (the last committed position); node n >= 1 holds a
 *     draft token below parent[n] < n.  Target row n holds the target's
 *     logits after the path to node n; draft row n the draft's logits there,
 *     from which node n's children were drawn independently (with
 *     replacement) -- that drafting is what makes the output law the target's.
 *   - p = softmax(t / T), q = softmax(d / T), T per sequence as in
 *     spec_verify.h.  At node c the children are tested in node-index order:
 *     child i is accepted when u_accept[b, child] is strictly below
 *     p_i(x)/q(x) (always when it is >= 1), with p_1 = p_c and, after each
 *     rejection, p_{i+1} = norm(max(0, p_i - q_c)).  An accepted child becomes
 *     the current node; when every child is rejected, or c is a leaf, one
 *     token is drawn from the current p_{m+1} (the bonus draw from p_c at a
 *     leaf) by inverse CDF with u_resample[b] (smallest x whose running mass
 *     exceeds u * R), and the walk ends.
 *   - T == 0: the lowest-index child whose token is the target's argmax
 *     (lowest index on ties) is accepted; if none, the argmax is emitted.
 *   - a tree with at most one child per node is exactly spec_verify's chain.
 *   - rows are read only as the walk visits them: the target row of every
 *     visited node, the draft row of a visited node with children (T > 0).
 * Everything is computed in fp32 (one pass over a visited node's rows for the
 * softmax statistics, one more per rejected sibling for the residual mass,
 * and a search of the crossing segment for the draw); no draw is recomputed
 * exactly, so a draw whose u * R lies within ~1e-6 of R of a cell edge may
 * pick the neighbouring token, and an accept test whose uniform lies within
 * ~1e-6 of its threshold may flip.
 *
 * Sequence errors (out_num_accepted = -1, out_tokens and out_nodes all -1): T
 * NaN, negative, infinite or positive below FLT_MIN; n_nodes outside [1, N];
 * for 1 <= n < n_nodes, parent[n] outside [0, n) or tokens[n] outside
 * [0, V); a visited row holding NaN or +inf, or entirely -inf; a tested
 * child whose draft logit is -inf (q = 0).  A NaN in a row the walk never
 * reaches is not an error.
 */
#ifndef SPEC_TREE_H
#define SPEC_TREE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define SPEC_TREE_MAX_NODES 1024

/*
 * Tree verification of B sequences with up to N nodes each.
 *   target_logits    device, [B, N, V] of dtype (spec_verify.h's spec_dtype_t)
 *   draft_logits     device, [B, N, V] of dtype; row n is read only when node n is
 *                    visited, has children and T > 0
 *   parent           device int32 [B, N]; entry 0 is ignored
 *   tokens           device int32 [B, N]; entry 0 is ignored
 *   n_nodes          device int32 [B]: nodes 0 .. n_nodes-1 of the sequence are used
 *   u_accept         device float32 [B, N] in [0, 1): entry n drives node n's test
 *   u_resample       device float32 [B] in [0, 1): the one draw
 *   temperature      device float32 [B] >= 0; 0 selects greedy mode
 *   out_tokens       device int32 [B, N]: the accepted path's tokens, the drawn (or
 *                    argmax) token, then -1
 *   out_nodes        device int32 [B, N]: the accepted path's node indices, then -1
 *   out_num_accepted device int32 [B]: accepted path length; -1 = sequence error.  The
 *                    sequence emits out_num_accepted[b] + 1 tokens.
 *   B >= 0 (0 is a no-op), 1 <= N <= SPEC_TREE_MAX_NODES, 2 <= V <= SPEC_MAX_V.
 *   Logit base addresses 16-byte aligned, the int32 and float32 arrays 4-byte
 *   aligned.
 * One kernel on `stream` (cudaStream_t as void*), one CTA per sequence; no
 * workspace and no allocation.  Returns SPEC_OK once it is launched,
 * SPEC_EINVAL for a size, pointer or alignment error, SPEC_ECUDA if the launch
 * failed.
 */
int32_t spec_verify_tree(const void *target_logits, const void *draft_logits,
                         const int32_t *parent, const int32_t *tokens, const int32_t *n_nodes,
                         const float *u_accept, const float *u_resample,
                         const float *temperature, int32_t *out_tokens, int32_t *out_nodes,
                         int32_t *out_num_accepted, int32_t B, int32_t N, int32_t V,
                         int32_t dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_TREE_H */
