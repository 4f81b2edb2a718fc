/*
 * svp.h -- C ABI of libsvp.so: paged decode/verify attention, KV append and
 * speculative acceptance on one GB300 GPU (sm_103a).
 *
 * The three calls are the step of a speculative decoding loop that runs on
 * the GPU's memory: store the new tokens' K/V in the paged cache
 * (kv_append), let the new query rows attend to their sequence's cached
 * rows (paged_decode_attention), and accept or resample the draft tokens
 * (spec_accept).
 *
 * Conventions shared by every entry point
 *  - Every tensor argument is a caller-owned DEVICE pointer, row-major and
 *    densely packed.  The library never frees or keeps a pointer beyond
 *    the call.
 *  - Every call is asynchronous on `stream` (0 = legacy default stream),
 *    does not synchronise the host, and allocates nothing when the caller
 *    passes the workspace it asks for (paged_decode_attention with
 *    dims->workspace == NULL falls back to a library-owned buffer, see
 *    below).
 *  - Return value: SVP_OK or a negative svp_status.  Arguments are checked
 *    on the host BEFORE anything is launched; a failed check launches
 *    nothing and writes nothing.  SVP_ERR_CUDA reports a launch error.
 *  - Data that can only be checked on the device (block ids, sequence
 *    lengths, token ids) never faults or traps: the kernel skips the bad
 *    item, records a flag in a device status word and carries on;
 *    svp_read_device_status() returns and clears the flags.
 *  - bf16 tensors hold IEEE bfloat16 bit patterns (uint16).
 */
#ifndef SVP_H
#define SVP_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SVP_OK = 0,
  SVP_ERR_INVALID_ARG = -1, /* null pointer, bad size or bad combination */
  SVP_ERR_UNSUPPORTED = -2, /* valid request outside what is built      */
  SVP_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed      */
  SVP_ERR_WORKSPACE = -4    /* caller workspace smaller than required    */
} svp_status;

/* SVP_FP8_E4M3: the K/V caches hold FP8 E4M3 codes (OCP: 1 sign bit, 4
 * exponent bits, bias 7, 3 mantissa bits; 1 byte per element), a value
 * being code * dims->k_scale (K) or code * dims->v_scale (V); q, out and the
 * new rows of kv_append are bf16 ("KV cache & Flash Attention", section
 * "Practical use": an fp8 KV cache halves the bytes attention reads). */
typedef enum { SVP_F32 = 0, SVP_BF16 = 1, SVP_FP8_E4M3 = 2 } svp_dtype;

/* Flags returned by svp_read_device_status(). */
enum {
  SVP_DEV_BAD_BLOCK_ID = 1,  /* a visible page maps outside [0,num_blocks) */
  SVP_DEV_BAD_SEQ_LEN = 2,   /* seq_len < q_len or > max_blocks_per_seq*16 */
  SVP_DEV_BAD_TOKEN = 4,     /* a draft token outside [0, vocab)           */
  SVP_DEV_TIMEOUT = 8        /* a bounded device-side wait gave up         */
};

/* Shapes shared by kv_append and paged_decode_attention.
 *   q, out           [batch, q_len, num_q_heads, head_dim]        dtype
 *                    (bf16 when dtype is SVP_FP8_E4M3)
 *   k_cache, v_cache [num_blocks, num_kv_heads, block_size, head_dim] dtype
 *                    (one head's page is one contiguous run)
 *   block_table      [batch, max_blocks_per_seq] int32; entry lb of row b
 *                    is the physical page of logical block lb of sequence b
 *                    (positions lb*16 .. lb*16+15).  Entries of pages that
 *                    the call does not need may hold anything (e.g. -1).
 *   seq_lens         [batch] int32, logical length of each sequence
 *                    INCLUDING its q_len new rows.
 * num_q_heads must be a multiple of num_kv_heads; query head h reads kv
 * head h / (num_q_heads / num_kv_heads).  head_dim is 64 or 128; block_size
 * is 16 (the page size of the lesson "KV cache & Flash Attention", section
 * "PagedAttention"). */
typedef struct {
  int batch;
  int num_q_heads;
  int num_kv_heads;
  int head_dim;
  int block_size;
  int max_blocks_per_seq;
  int num_blocks;
  int dtype;              /* svp_dtype of q, out and both caches           */
  void *workspace;        /* device scratch for split partials, or NULL    */
  size_t workspace_bytes; /* size of `workspace`                           */
  int split_pages;        /* fewest pages per CTA slice; 0 = automatic (8) */
  int kernel_path;        /* svp_kernel_path; SVP_PATH_AUTO by default     */
  float k_scale;          /* SVP_FP8_E4M3 caches: value = code * scale    */
  float v_scale;          /* (finite, > 0); ignored for other dtypes      */
} svp_dims;

/* Which attention kernel variant runs.  AUTO picks tensor cores (bf16 only)
 * when a kv head serves at least 3 query rows (GQA group x q_len): TCGEN05
 * for head_dim 128, TENSOR_CORES for head_dim 64; CUDA cores otherwise.
 * All compute the same quantity; forcing a path exists for testing and
 * tuning.
 *   CUDA_CORES    fp32 FMA dot products, any dtype.
 *   TENSOR_CORES  warp-level mma.sync (bf16 in, fp32 accumulate).
 *   TCGEN05       fifth-generation tensor cores: tcgen05.mma with fp32
 *                 accumulators in tensor memory, keys as the 128-row M
 *                 dimension (bf16, head_dim 128, 512 sequences per
 *                 kernel launch).
 * A forced tensor path on data it cannot take (fp32; head_dim 64 for
 * TCGEN05) is SVP_ERR_UNSUPPORTED. */
typedef enum {
  SVP_PATH_AUTO = 0,
  SVP_PATH_CUDA_CORES = 1,
  SVP_PATH_TENSOR_CORES = 2,
  SVP_PATH_TCGEN05 = 3
} svp_kernel_path;

/* Paged decode / speculative-verify attention.
 *
 * Defines (pages: "KV cache & Flash Attention", sections "FlashAttention --
 * the tiling trick" and "PagedAttention"; "How speculative decoding doubles
 * LLM speed", step 2 (verification); "How StreamingLLM stabilizes
 * million-token streams via attention sinks", section "The StreamingLLM
 * solution"):
 *   query row i in [0, q_len) of sequence b sits at absolute position
 *   t_i = seq_lens[b] - q_len + i.  Key j is visible to it iff j <= t_i
 *   and (window == 0 or j < n_sink or j > t_i - window).
 *   out[b,i,h]  = sum_j softmax_j(scale * <q[b,i,h], K_j>) V_j over the
 *                 visible keys of kv head h / (Hq/Hkv), written in dtype;
 *   lse[b,i,h]  = natural log of sum_j exp(scale * <q, K_j>), fp32.
 *   window == 0 disables the window (n_sink is then ignored); n_sink
 *   counts from position 0; window counts the query's own key.  Only pages
 *   holding visible keys are read; other block_table entries are not read.
 * q_len: 1 (decode) .. 16 (verify of q_len-1 drafts + bonus position).
 * Work: every CTA of one persistent launch takes an equal slice of all
 * visible pages of all (sequence, kv head) groups (at least
 * dims->split_pages pages each; each group also counts a few pages' worth
 * for its fixed cost, and the TCGEN05 path slices in 8-page tiles); a
 * group that spans several slices is finished by a second kernel, launched
 * as a programmatic dependent of the first, which merges the slices'
 * partial results by log-sum-exp.
 * Workspace: paged_decode_workspace_size() bytes, passed in dims; it needs
 * no initialisation: each CTA rewrites the split record it owns in every
 * launch, and the merge kernel reads partials only where a record of the
 * same launch points.  Two kernel launches (attention, merge) per 4096
 * sequences (512 on the TCGEN05 path).  With
 * dims->workspace == NULL the library uses a buffer of its own per device,
 * (re)allocated inside the call when it is too small -- that first call is
 * then not capturable in a CUDA graph.  Calls that share a workspace must
 * not overlap on the GPU.
 * q, k_cache, v_cache and out must be 16-byte aligned.
 * Errors: SVP_ERR_INVALID_ARG for null or misaligned pointers, sizes < 0,
 * num_q_heads not a multiple of num_kv_heads, q_len < 1, n_sink < 0,
 * window < 0, a non-finite scale or an unknown kernel_path;
 * SVP_ERR_UNSUPPORTED for head_dim not in {64,128}, block_size != 16,
 * q_len > 16, batch > 65535, or a forced tensor-core path on data it cannot
 * take;
 * SVP_ERR_WORKSPACE for a caller workspace that is too small.  batch == 0
 * returns SVP_OK at once. */
int paged_decode_attention(const svp_dims *dims, const void *q,
                           const void *k_cache, const void *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           int q_len, int n_sink, int window, float scale,
                           void *out, float *lse, cudaStream_t stream);

/* Draft-tree verify attention (pages: "How speculative decoding doubles LLM
 * speed", section "Modern architecture variants" -- SpecInfer verifies a
 * tree of draft branches in one pass with a two-dimensional attention mask;
 * "Speculative decoding: how AI models get faster without getting bigger",
 * on tree speculation).
 * The q_len new rows of sequence b are the nodes of its draft tree, node k
 * at position seq_lens[b] - q_len + k (node 0 the root: the last accepted
 * token).  tree_mask [batch, q_len] uint32 (DEVICE, 4-byte aligned): bit k
 * of entry (b, i) is set iff node k is an ancestor of node i or i itself
 * (so only bits k <= i matter; higher bits are ignored).  Query node i
 * attends to every cached key before the tree and to the node keys its
 * bits select; otherwise exactly paged_decode_attention with n_sink = 0 and
 * window = 0 (same layouts, workspace, alignment and errors).  A chain
 * (bits 0..i for node i) reproduces the causal verify block.  q_len
 * <= 16.  Errors: those of paged_decode_attention, plus SVP_ERR_INVALID_ARG
 * for a null or misaligned tree_mask. */
int paged_tree_attention(const svp_dims *dims, const void *q,
                         const void *k_cache, const void *v_cache,
                         const int32_t *block_table, const int32_t *seq_lens,
                         int q_len, const uint32_t *tree_mask, float scale,
                         void *out, float *lse, cudaStream_t stream);

/* Size of the fixed device scratch used by paged_decode_attention_noalloc. */
#define SVP_STATIC_SCRATCH_BYTES ((size_t)32 << 20) /* 32 MiB */

/* paged_decode_attention for callers that cannot allocate device memory.
 *
 * No counterpart in the source pages: this entry point exists for callers
 * that must not call cudaMalloc when they run attention -- code executing
 * while a CUDA graph is being captured (allocation is not capturable),
 * plug-ins whose host framework owns every device allocation through its
 * own pool, and latency-critical loops where cudaMalloc/cudaFree would
 * synchronise the device.
 *
 * Same arguments, layouts and results as paged_decode_attention, except
 * that dims->workspace and dims->workspace_bytes are ignored: the split-K
 * scratch is a fixed SVP_STATIC_SCRATCH_BYTES array inside the library's
 * device memory, which every GPU that loads the library holds until the
 * process exits.  Nothing is allocated by this call.  The caller still
 * passes q, the caches, block_table, seq_lens, out and lse.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, once per device, with that device current);
 *     make that first call before any stream capture.  The address is
 *     cached for the life of the CUDA context: after cudaDeviceReset the
 *     cached address is stale, so do not use this entry point across a
 *     device reset.
 *   - Every call shares the one array and leaves its contents behind;
 *     nothing in it needs to start at zero (every launch rewrites the
 *     split records it reads), so calls in sequence on one stream are
 *     independent.  Calls that overlap on the GPU (other streams, other
 *     host threads) race on the array.
 *   - With dims->split_pages == 0 the automatic slice size is enlarged (64,
 *     then 128 pages per CTA: fewer partial slots) when the default plan
 *     would not fit the array.
 * Errors: those of paged_decode_attention, plus SVP_ERR_WORKSPACE when the
 * scratch this request needs exceeds SVP_STATIC_SCRATCH_BYTES (use fewer
 * sequences per call or longer splits). */
int paged_decode_attention_noalloc(const svp_dims *dims, const void *q,
                                   const void *k_cache, const void *v_cache,
                                   const int32_t *block_table,
                                   const int32_t *seq_lens, int q_len,
                                   int n_sink, int window, float scale,
                                   void *out, float *lse, cudaStream_t stream);

/* Bytes of workspace paged_decode_attention needs for these dims and this
 * (q_len, n_sink, window).  Returns 0 for invalid dims. */
size_t paged_decode_workspace_size(const svp_dims *dims, int q_len,
                                   int n_sink, int window);

/* KV append: writes the n_new new K/V rows of every sequence, k_new/v_new
 * [batch, n_new, num_kv_heads, head_dim] (dtype of dims; bf16 for an
 * SVP_FP8_E4M3 cache), at logical positions seq_lens[b]-n_new ..
 * seq_lens[b]-1 of the paged caches, i.e. page block_table[b][pos/16], row
 * pos%16 (pages: "KV cache & Flash Attention", sections "KV cache" and
 * "PagedAttention").  seq_lens are the lengths AFTER the append.  A byte
 * copy; into an FP8 cache each value x is stored as the E4M3 code of the
 * fp32 quotient x / k_scale (resp. v_scale), nearest with ties to even,
 * saturating at +-448.  Uses no workspace.
 * Errors as for paged_decode_attention; n_new in [0, 64]; k_new, v_new,
 * k_cache and v_cache must be 16-byte aligned (else SVP_ERR_INVALID_ARG,
 * before any launch). */
int kv_append(const svp_dims *dims, const void *k_new, const void *v_new,
              void *k_cache, void *v_cache, const int32_t *block_table,
              const int32_t *seq_lens, int n_new, cudaStream_t stream);

/* Speculative acceptance (pages: "How speculative decoding doubles LLM
 * speed", step 3 (sampling) and section "Absolute mathematical exactness";
 * "Speculative decoding: how AI models get faster without getting bigger").
 *   target_logits [batch, num_draft+1, vocab] fp32 (rows p_0 .. p_K)
 *   draft_logits  [batch, num_draft, vocab]   fp32 (rows q_0 .. q_{K-1})
 *   draft_tokens  [batch, num_draft] int32
 *   uniforms      [batch, num_draft+1] fp32 in [0,1): entry i < K decides
 *                 draft i, entry K drives the one resample or bonus draw
 *   out_tokens    [batch, num_draft+1] int32, written: accepted drafts,
 *                 then the resampled or bonus token, then -1 padding
 *   n_accepted    [batch] int32: number of accepted drafts (0..K)
 * With p = softmax(target row), q = softmax(draft row): draft i is accepted
 * iff u_i * q_i(x_i) <= p_i(x_i), i.e. u_i <= min(1, p/q); at the first
 * rejection j the replacement is drawn from max(0, p_j - q_j) normalised;
 * if all K are accepted the bonus token is drawn from p_K.  A draw takes
 * the smallest token index whose running sum (token order) exceeds
 * u_K * total.  A residual of zero mass (impossible in exact arithmetic)
 * falls back to p_j.  A sequence with a draft token outside [0, vocab) gets
 * n_accepted = -1 and all-(-1) tokens and sets SVP_DEV_BAD_TOKEN.
 * Softmax normalisers are sums of fp32 exponentials relative to integer
 * power-of-two references, accumulated in compensated fp32 pairs and
 * combined by exact power-of-two scaling; the accept ratio and the draw's
 * prefix sums use error-free fp32 transformations (no fp64).  One
 * thread-block cluster per sequence: 16 CTAs when the whole batch fits one
 * wave of such clusters, else 8.  Uses no workspace.
 * Errors: SVP_ERR_INVALID_ARG for null pointers, batch < 0, num_draft < 1,
 * vocab < 2; SVP_ERR_UNSUPPORTED for num_draft > 15 or batch > 65535. */
int spec_accept(int batch, int num_draft, int vocab,
                const float *target_logits, const float *draft_logits,
                const int32_t *draft_tokens, const float *uniforms,
                int32_t *out_tokens, int32_t *n_accepted, cudaStream_t stream);

/* The verify epilogue for spec_accept (pages: "How speculative decoding
 * doubles LLM speed", section "Deployment limits" -- sampling temperature;
 * "How Moondream cut VLM inference latency by 35% via pipelined decoding",
 * section "Mechanism two: forward first, then sample" -- constrained
 * decoding sets the logits of disallowed tokens to -inf before sampling).
 *   temperature  > 0: p = softmax(target / T), q = softmax(draft / T)
 *                (1 = the logits as given); ignored with greedy
 *   allowed      NULL, or DEVICE [batch, num_draft+1, (vocab+31)/32] uint32,
 *                4-byte aligned: bit x%32 of word x/32 of row (b, i) set iff
 *                position i may emit token x; row i restricts target row i
 *                and draft row i (disallowed logits read as -inf).  A draft
 *                token the row excludes is rejected.  Every row must allow
 *                at least one token.
 *   greedy       0: rejection sampling; 1: argmax verification -- draft i
 *                is accepted iff it is the most likely allowed token of
 *                target row i (smallest index on ties), and the first
 *                mismatch (or the bonus position) emits that token;
 *                uniforms are not read. */
typedef struct {
  float temperature;
  const uint32_t *allowed;
  int greedy;
} svp_accept_opts;

/* spec_accept with the verify epilogue above applied inside the kernel
 * (opts == NULL: temperature 1, no mask, sampling -- exactly spec_accept).
 * Same layouts, outputs and errors as spec_accept, plus
 * SVP_ERR_INVALID_ARG for temperature <= 0 or non-finite without greedy,
 * or a misaligned mask. */
int spec_accept_ex(int batch, int num_draft, int vocab,
                   const float *target_logits, const float *draft_logits,
                   const int32_t *draft_tokens, const float *uniforms,
                   const svp_accept_opts *opts, int32_t *out_tokens,
                   int32_t *n_accepted, cudaStream_t stream);

/* Tree acceptance (pages: "How speculative decoding doubles LLM speed",
 * sections "Modern architecture variants" -- SpecInfer's draft tree -- and
 * step 3 (sampling); "Speculative decoding: how AI models get faster without
 * getting bigger": the verifier keeps the longest accepted path).
 * A draft tree of num_nodes = N nodes per sequence; node 0 is the root (the
 * last accepted token), every other node c has parents[b][c] < c.
 *   target_logits [batch, N, vocab] fp32: row i = target logits after node i
 *   draft_logits  [batch, N, vocab] fp32: row i = draft logits the children
 *                 of node i were drawn from (rows of leaves are not read)
 *   parents       [batch, N] int32 (parents[b][0] = -1)
 *   node_tokens   [batch, N] int32 (entry 0 unused)
 *   uniforms      [batch, N] fp32 in [0,1): entry c >= 1 decides node c,
 *                 entry 0 drives the one final draw
 *   out_tokens    [batch, N] int32, written: the accepted path's tokens,
 *                 then the drawn token, then -1 padding
 *   out_nodes     [batch, N] int32: the node of each accepted path token
 *                 (for compacting the KV cache), then -1
 *   n_accepted    [batch] int32: length of the accepted path
 * The walk starts at the root; a node's children are tried in index order,
 * child c being accepted iff u_c <= r(x_c) / q(x_c), where q is the draft
 * distribution of the node and r starts as its target distribution p and,
 * after each rejected child, becomes the normalised residual max(0, r - q).
 * An accepted child becomes the current node; when no child is accepted
 * (or the node is a leaf) one token is drawn from r with u_0 (inverse CDF
 * in token order, as in spec_accept).  On a chain this is spec_accept with
 * uniforms (u_1 .. u_K, u_0).  With the children of a node drawn
 * independently from its q, the emitted tokens follow the target model.
 * A malformed tree or a token outside [0, vocab) gives n_accepted = -1 and
 * all -1 outputs and sets SVP_DEV_BAD_TOKEN.  Numerics as spec_accept; one
 * rejected child costs one more pass over the node's two rows.  Uses no
 * workspace.
 * Errors: SVP_ERR_INVALID_ARG for null pointers, batch < 0, num_nodes < 1,
 * vocab < 2; SVP_ERR_UNSUPPORTED for num_nodes > 16 or batch > 65535. */
int spec_accept_tree(int batch, int num_nodes, int vocab,
                     const float *target_logits, const float *draft_logits,
                     const int32_t *parents, const int32_t *node_tokens,
                     const float *uniforms, int32_t *out_tokens,
                     int32_t *out_nodes, int32_t *n_accepted,
                     cudaStream_t stream);

/* ---- the graph-captured decode step ----------------------------------
 * (page: "How Moondream cut VLM inference latency by 35% via pipelined
 * decoding", sections "The problem: the GPU bubble" and "Mechanism one:
 * ping-pong slots").  A runner owns two slots; each has pinned host buffers
 * for the step's inputs and outputs and device copies of them, and one CUDA
 * graph, captured at creation, that runs kv_append (the q_len new rows),
 * paged_decode_attention and, with num_draft > 0, spec_accept
 * (spec_accept_ex with epilogue options) -- or, for a draft tree
 * (tree_nodes > 0), paged_tree_attention and spec_accept_tree -- on the
 * slot's device buffers.  svp_step_launch copies the slot's inputs to the
 * device on an upload stream (once the slot's previous step has finished
 * with them, so the upload overlaps the other slot's step), replays the
 * slot's graph on the runner's compute stream after that copy, and queues
 * the copy of its outputs back to the slot on a separate copy stream,
 * ordered after an event recorded when that step's outputs are written --
 * so the next step (the other slot) can run while the copy is in flight.
 * The host fills one slot while the GPU works on the other.
 * Protocol: write a slot's inputs only before its first launch or after
 * svp_step_wait on it returned; read its outputs after svp_step_wait.
 * Launching a slot again waits (on the device) for its previous result
 * copy.  The caches are the caller's and are updated by every step, in
 * launch order.  All memory is allocated at creation; launches allocate
 * nothing. */
typedef struct {
  svp_dims dims;      /* shapes of the cache and the batch (workspace and
                         split/path fields: as for paged_decode_attention;
                         the runner allocates its own workspace) */
  int q_len;          /* new rows per sequence: appended, then attending */
  int n_sink, window; /* as for paged_decode_attention */
  float scale;
  void *k_cache;      /* DEVICE caches, caller-owned */
  void *v_cache;
  int num_draft;      /* 0: no acceptance step or a tree; else q_len - 1 */
  int vocab;          /* vocabulary of the acceptance step */
  /* the verify epilogue of a draft chain (num_draft > 0), as
     svp_accept_opts: temperature (0 is read as 1), greedy, and with
     use_mask != 0 the token mask from the slot's SVP_STEP_ALLOWED field */
  float temperature;
  int greedy;
  int use_mask;
  /* a draft tree instead of a chain: tree_nodes = q_len (<= 16) nodes,
     num_draft 0, no sinks or window, no epilogue options; the slot then
     takes SVP_STEP_TREE_MASK, SVP_STEP_PARENTS, SVP_STEP_NODE_TOKENS and
     N-row logits and uniforms, and returns SVP_STEP_OUT_NODES */
  int tree_nodes;
} svp_step_desc;

/* Fields of a slot (pinned host memory; layouts as in the single calls;
 * N = tree_nodes for a tree, where K+1 and K rows read N). */
typedef enum {
  SVP_STEP_Q = 0,          /* in:  [batch, q_len, Hq, D] dtype          */
  SVP_STEP_K_NEW,          /* in:  [batch, q_len, Hkv, D] dtype         */
  SVP_STEP_V_NEW,          /* in:  [batch, q_len, Hkv, D] dtype         */
  SVP_STEP_BLOCK_TABLE,    /* in:  [batch, max_blocks_per_seq] int32    */
  SVP_STEP_SEQ_LENS,       /* in:  [batch] int32 (after the append)     */
  SVP_STEP_TARGET_LOGITS,  /* in:  [batch, K+1, vocab] fp32             */
  SVP_STEP_DRAFT_LOGITS,   /* in:  [batch, K, vocab] fp32               */
  SVP_STEP_DRAFT_TOKENS,   /* in:  [batch, K] int32 (chain)             */
  SVP_STEP_UNIFORMS,       /* in:  [batch, K+1] fp32                    */
  SVP_STEP_OUT,            /* out: [batch, q_len, Hq, D] dtype          */
  SVP_STEP_LSE,            /* out: [batch, q_len, Hq] fp32              */
  SVP_STEP_OUT_TOKENS,     /* out: [batch, K+1] int32                   */
  SVP_STEP_N_ACCEPTED,     /* out: [batch] int32                        */
  SVP_STEP_ALLOWED,        /* in:  [batch, K+1, ceil(vocab/32)] uint32
                                   (chain with use_mask)                 */
  SVP_STEP_TREE_MASK,      /* in:  [batch, N] uint32 (tree)             */
  SVP_STEP_PARENTS,        /* in:  [batch, N] int32 (tree)              */
  SVP_STEP_NODE_TOKENS,    /* in:  [batch, N] int32 (tree)              */
  SVP_STEP_OUT_NODES,      /* out: [batch, N] int32 (tree)              */
  SVP_STEP_NUM_FIELDS
} svp_step_field;

typedef struct svp_step svp_step;

/* Allocates the runner (streams, workspace, both slots) and captures the
 * two slot graphs.  Errors: SVP_ERR_INVALID_ARG for null pointers, sizes
 * < 1, num_draft not in {0, q_len - 1}, epilogue options without drafts,
 * or a tree with tree_nodes != q_len, drafts, sinks, a window or epilogue
 * options; SVP_ERR_UNSUPPORTED for more than 16 tree nodes; the errors of
 * the single calls for their arguments; SVP_ERR_CUDA if an allocation or
 * the capture fails. */
int svp_step_create(const svp_step_desc *desc, svp_step **runner);
/* Pinned host memory of one field of slot 0 or 1 and its size in bytes
 * (*bytes may be NULL); NULL for a bad slot/field or an empty field. */
void *svp_step_host_buffer(svp_step *runner, int slot, int field,
                           size_t *bytes);
/* Queues one step on the slot (asynchronous). */
int svp_step_launch(svp_step *runner, int slot);
/* Waits until the slot's last step has finished and its outputs are in the
 * slot's host buffers. */
int svp_step_wait(svp_step *runner, int slot);
/* The runner's compute stream (for ordering other work after its steps). */
cudaStream_t svp_step_stream(svp_step *runner);
/* Waits for outstanding work and frees everything. */
int svp_step_destroy(svp_step *runner);

/* Synchronises `stream`, returns SVP_OK and stores in *flags the OR of the
 * SVP_DEV_* flags raised by kernels since the last read, then clears them.
 * flags may be NULL. */
int svp_read_device_status(cudaStream_t stream, int *flags);

/* Human-readable name of an svp_status value (static string). */
const char *svp_status_string(int status);

/* Number of kernels the last successful call of each entry point launched
 * on the calling thread (for launch accounting). */
int svp_last_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* SVP_H */
