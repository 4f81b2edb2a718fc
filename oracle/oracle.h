/*
 * oracle.h -- plain, slow, single-threaded fp64 CPU oracle for paged
 * decode/verify attention, KV append and speculative acceptance.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link
 * or call this code: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no source, header, table or helper with
 * the CUDA library; the two meet only through the seeded input arrays.
 *
 * Layouts (row-major, element counts):
 *   q, out          [batch, q_len, num_q_heads, head_dim]   (q in `dtype`)
 *   lse             [batch, q_len, num_q_heads]              natural log
 *   k_cache,v_cache [num_blocks, num_kv_heads, block_size, head_dim]
 *   block_table     [batch, max_blocks_per_seq]  int32
 *   seq_lens        [batch] int32, logical length INCLUDING the q_len new rows
 * dtype: 0 = IEEE fp32, 1 = bfloat16 given as raw 16-bit patterns.
 */
#ifndef SVP_ORACLE_H
#define SVP_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Exact attention by full materialisation over the logically gathered cache.
 * rows (optional): flat query-row ids (b*q_len + i)*num_q_heads + h to
 * compute; NULL computes every row in order.  out gets n_rows*head_dim
 * doubles, lse n_rows doubles.  Returns 0, or -1 for bad sizes, -2 if a
 * visible key maps to a block id outside [0, num_blocks), -3 if
 * seq_len < q_len. */
int oracle_paged_attention(int batch, int num_q_heads, int num_kv_heads,
                           int head_dim, int block_size, int max_blocks_per_seq,
                           int num_blocks, int dtype, const void *q,
                           const void *k_cache, const void *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           int q_len, int n_sink, int window, float scale,
                           const int64_t *rows, int64_t n_rows, double *out,
                           double *lse);

/* The same definition with a draft-tree mask instead of the causal verify
 * mask: the q_len new rows of a sequence are the tree's nodes (node k at
 * position seq_len - q_len + k) and query node i sees every earlier key plus
 * the node keys k <= i whose bit k is set in tree_mask[b*q_len + i]
 * (uint32, its ancestors and itself).  No sinks or window.  q_len <= 32.
 * Same returns as oracle_paged_attention. */
int oracle_paged_tree_attention(int batch, int num_q_heads, int num_kv_heads,
                                int head_dim, int block_size,
                                int max_blocks_per_seq, int num_blocks,
                                int dtype, const void *q, const void *k_cache,
                                const void *v_cache,
                                const int32_t *block_table,
                                const int32_t *seq_lens, int q_len,
                                const uint32_t *tree_mask, float scale,
                                const int64_t *rows, int64_t n_rows,
                                double *out, double *lse);

/* The same definition over an FP8 cache: q in bf16, k_cache / v_cache E4M3
 * codes (1 byte per element, same layout), value = code's value * k_scale
 * (or v_scale).  Same returns as oracle_paged_attention. */
int oracle_paged_attention_fp8(int batch, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size,
                               int max_blocks_per_seq, int num_blocks,
                               const void *q, const void *k_cache,
                               const void *v_cache, double k_scale,
                               double v_scale, const int32_t *block_table,
                               const int32_t *seq_lens, int q_len, int n_sink,
                               int window, float scale, const int64_t *rows,
                               int64_t n_rows, double *out, double *lse);

/* FP8 E4M3 codes: decode (values, NaN for the NaN codes); encode
 * x / scale (fp32 division) to the nearest code, ties to even, saturating
 * at +-448.  Return 0 (-1 for scale <= 0). */
int oracle_e4m3_decode(const uint8_t *codes, long n, double *out);
int oracle_e4m3_encode(const float *x, long n, float scale, uint8_t *out);

/* KV append into FP8 caches: k_new / v_new bf16 [batch, n_new, Hkv, D];
 * each value stored as the E4M3 code of value / scale.  Returns as
 * oracle_kv_append. */
int oracle_kv_append_fp8(int batch, int num_kv_heads, int head_dim,
                         int block_size, int max_blocks_per_seq,
                         int num_blocks, const uint16_t *k_new,
                         const uint16_t *v_new, uint8_t *k_cache,
                         uint8_t *v_cache, float k_scale, float v_scale,
                         const int32_t *block_table, const int32_t *seq_lens,
                         int n_new);

/* The same quantity computed the tiled way: the visible keys of each row are
 * cut into n_splits contiguous parts, each part is folded in `tile`-key
 * blocks with a running (max, sum, accumulator), and the parts are merged by
 * their log-sum-exp.  Self-check of the online-softmax algebra only. */
int oracle_paged_attention_tiled(int batch, int num_q_heads, int num_kv_heads,
                                 int head_dim, int block_size,
                                 int max_blocks_per_seq, int num_blocks,
                                 int dtype, const void *q, const void *k_cache,
                                 const void *v_cache,
                                 const int32_t *block_table,
                                 const int32_t *seq_lens, int q_len, int n_sink,
                                 int window, float scale, int tile,
                                 int n_splits, double *out, double *lse);

/* Writes the n_new new K/V rows of every sequence at logical positions
 * seq_lens[b]-n_new .. seq_lens[b]-1 into the paged caches (byte copy).
 * k_new, v_new: [batch, n_new, num_kv_heads, head_dim] of elem_bytes each.
 * Returns 0, -1 for bad sizes, -2 for a block id out of range. */
int oracle_kv_append(int batch, int num_kv_heads, int head_dim, int block_size,
                     int max_blocks_per_seq, int num_blocks, int elem_bytes,
                     const void *k_new, const void *v_new, void *k_cache,
                     void *v_cache, const int32_t *block_table,
                     const int32_t *seq_lens, int n_new);

/* Speculative acceptance, literal rejection-sampling loop.
 *   target_logits [batch, K+1, vocab] fp32, draft_logits [batch, K, vocab]
 *   draft_tokens [batch, K], uniforms [batch, K+1] in [0,1)
 *   out_tokens [batch, K+1] (-1 padded), n_accepted [batch]
 *   near_boundary [batch] (may be NULL): 1 if a decision of that sequence
 *     fell within eps of its boundary (accept test: |r - p/q| < eps;
 *     sampling: |u*W - C(x)| < eps*W at the chosen or preceding x).
 *   residual_fallback [batch] (may be NULL): 1 if a rejection met a residual
 *     of zero mass and p itself was sampled instead.
 * Returns 0, -1 for bad sizes, -4 for a draft token outside [0, vocab). */
int oracle_spec_accept(int batch, int num_draft, int vocab,
                       const float *target_logits, const float *draft_logits,
                       const int32_t *draft_tokens, const float *uniforms,
                       int32_t *out_tokens, int32_t *n_accepted,
                       int32_t *near_boundary, int32_t *residual_fallback,
                       double eps);

/* spec_accept with the verify epilogue: both distributions at temperature
 * T (softmax(logits / T)); allowed (may be NULL) [batch, K+1, (vocab+31)/32]
 * uint32 bit masks of the tokens position i may emit (row i applies to
 * target row i and draft row i; an excluded draft token is rejected); with
 * greedy != 0 a draft is accepted iff it is the most likely allowed target
 * token (smallest index on ties), the replacement or bonus is that token,
 * and temperature and uniforms are not used.  Returns as oracle_spec_accept
 * (-1 also for temperature <= 0 without greedy). */
int oracle_spec_accept_ex(int batch, int num_draft, int vocab,
                          const float *target_logits,
                          const float *draft_logits,
                          const int32_t *draft_tokens, const float *uniforms,
                          double temperature, const uint32_t *allowed,
                          int greedy, int32_t *out_tokens,
                          int32_t *n_accepted, int32_t *near_boundary,
                          double eps);

/* Tree acceptance (draft tree of num_nodes nodes; node 0 is the root, the
 * last token already accepted; parents[c] < c for c >= 1, parents[0] = -1).
 *   target_logits [batch, N, vocab]: row i = target distribution after node i
 *   draft_logits  [batch, N, vocab]: row i = draft distribution node i's
 *                 children were drawn from
 *   node_tokens   [batch, N] (entry 0 unused), uniforms [batch, N]: entry
 *                 c >= 1 decides node c, entry 0 drives the final draw
 *   out_tokens    [batch, N]: accepted path tokens, then the drawn token,
 *                 -1 padded; out_nodes [batch, N]: node of each accepted
 *                 path token, -1 padded; n_accepted [batch]: path length
 * At each node the children are tried in index order: child c is accepted
 * iff u_c <= r(x_c)/q(x_c), r being the target distribution after the node,
 * replaced by the normalised residual max(0, r - q) after each rejected
 * child; when no child is accepted one token is drawn from r with u_0.
 * near_boundary / residual_fallback as for oracle_spec_accept.
 * Returns 0, -1 for bad sizes or a malformed tree, -4 for a node token
 * outside [0, vocab). */
int oracle_spec_accept_tree(int batch, int num_nodes, int vocab,
                            const float *target_logits,
                            const float *draft_logits, const int32_t *parents,
                            const int32_t *node_tokens, const float *uniforms,
                            int32_t *out_tokens, int32_t *out_nodes,
                            int32_t *n_accepted, int32_t *near_boundary,
                            int32_t *residual_fallback, double eps);

/* The outcomes the acceptance rule can reach when every comparison that
 * lies within eps of its boundary may go either way (accept test:
 * |u_i - p(x)/q(x)| < eps; draw: running sums within eps*W of u*W), every
 * other comparison going as in exact arithmetic.  With eps = 0 this is the
 * single outcome of the rule.
 *
 * Linear rule (temperature and allowed as for oracle_spec_accept_ex, no
 * greedy): path_valid [batch, K+1]: entry j < K is 1 iff "drafts 0..j-1
 * accepted, draft j rejected" is reachable, entry K iff "all accepted" is;
 * cand [batch, K+1, max_cand] (-1 padded) and n_cand [batch, K+1]: the
 * tokens the draw on that path may return (n_cand may exceed max_cand).
 * Returns as oracle_spec_accept_ex. */
int oracle_spec_accept_valid(int batch, int num_draft, int vocab,
                             const float *target_logits,
                             const float *draft_logits,
                             const int32_t *draft_tokens,
                             const float *uniforms, double temperature,
                             const uint32_t *allowed, int32_t *path_valid,
                             int32_t *cand, int32_t *n_cand, int max_cand,
                             double eps);

/* Tree walk (arguments as oracle_spec_accept_tree; num_nodes <= 64):
 * outcomes [batch, max_out, N + 2 + max_cand]: each reachable outcome as
 * [accepted nodes in order, -1 padded (N)] [n_accepted] [n_cand]
 * [candidate tokens of the final draw, -1 padded (max_cand)];
 * n_outcomes [batch] (may exceed max_out: only the first max_out rows are
 * written).  Returns as oracle_spec_accept_tree. */
int oracle_spec_accept_tree_valid(int batch, int num_nodes, int vocab,
                                  const float *target_logits,
                                  const float *draft_logits,
                                  const int32_t *parents,
                                  const int32_t *node_tokens,
                                  const float *uniforms, int32_t *outcomes,
                                  int32_t *n_outcomes, int max_out,
                                  int max_cand, double eps);

#ifdef __cplusplus
}
#endif
#endif
