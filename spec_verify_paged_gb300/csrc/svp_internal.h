// svp_internal.h -- parameter blocks and launchers shared between the C-ABI
// host layer (api.cu) and the kernel translation units.  Not installed.
#pragma once
#include <cuda_runtime_api.h>
#include <cstddef>
#include <cstdint>

namespace svp {

struct SplitDesc;

constexpr int kBlockSize = 16;     // tokens per KV page
constexpr int kMaxQLen = 16;
constexpr int kMaxBatch = 65535;
constexpr int kMaxDraft = 15;
constexpr int kMaxNodes = 16;    // draft-tree nodes (= the verify rows)

// One paged_decode_attention launch.
struct AttnParams {
  const void *q;
  const void *k_cache;
  const void *v_cache;
  const int32_t *block_table;
  const int32_t *seq_lens;
  void *out;
  float *lse;
  // workspace pieces
  struct SplitDesc *desc;  // [grid] split group whose first page a CTA owns
  float *part_o;       // [2 * grid][RB][D] normalised partials: each CTA's
                       // first- and last-segment slot
  float *part_lse;     // [2 * grid][RB] log2-domain LSE of the partials
  int batch, num_q_heads, num_kv_heads, head_dim, group;
  int q_len, n_sink, window;
  int max_blocks, num_blocks;
  int rows;            // group * q_len query rows per (sequence, kv head)
  int rb;              // rows per work unit (row-group size)
  int n_rg;            // ceil(rows / rb)
  int min_pages;       // fewest items a CTA's slice may hold
  int seg_items;       // items that stand for a segment's fixed cost
  int ppi;             // pages per item: 1, or the tcgen05 kernel's tile
                       // (slices then split groups at tile boundaries)
  float qscale;        // scale * log2(e)
  const uint32_t *tree_mask;  // [batch, q_len] ancestor bits, or null
  float v_scale;       // FP8 caches: V value = code * v_scale (else 1)
  // 1: the previous kernel on the stream appended the q_len newest
  // positions of these sequences and wrote nothing else this call reads,
  // and every other input was written before it started.  The kernel then
  // reads everything but the pages holding those positions before its
  // grid-dependency wait, and waits before the first such page and before
  // its first write.  0: it waits before touching global memory.
  int early;
};

struct AttnPlan {
  int rb, n_rg, min_pages, seg_items, grid, ctas_per_sm;
  bool mma;            // warp-level mma.sync path
  bool tc;             // tcgen05 path (tensor-memory accumulators)
  int batch_cap;       // sequences per launch
  size_t ws_head, ws_desc, ws_part_o, ws_part_lse, ws_total;
};

// paged_decode_attention (tree_mask null) or paged_tree_attention launched
// right after kv_append of the q_len newest positions on the same stream
// (the fused step): the prefix pages are read while the append runs.
int attention_after_append(const svp_dims *dims, const void *q,
                           const void *k_cache, const void *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           int q_len, int n_sink, int window,
                           const uint32_t *tree_mask, float scale, void *out,
                           float *lse, cudaStream_t stream);

// Fills the plan (no CUDA launches).  dtype 0 = f32, 1 = bf16.  Returns 0 or
// a negative svp_status.
int plan_attention(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                   int dtype, int max_blocks, int q_len, int n_sink,
                   int window, int split_pages, int kernel_path, int num_sms,
                   long long num_blocks, AttnPlan *plan);

// The tcgen05 kernel's stream-K items are 8-page tiles; a segment's fixed
// cost (the masked last tile, epilogue, next Q) takes about two tiles'
// time: the split counts it.
constexpr int kTilePagesTc = 8;
constexpr int kSegItemsTc = 2;
// The CUDA-core kernel's items are pages; a segment's epilogue (the four
// warps' states merged through shared memory, the rows written out) is
// counted as this many pages.
constexpr int kSegItemsCc = 12;

// Query rows per kv head (GQA group x q_len) from which the automatic path
// choice uses tensor cores (bf16 only): tcgen05 for head_dim 128, warp-level
// mma.sync for head_dim 64.
constexpr int kMmaMinRows = 3;

// Occupancy-derived CTAs per SM for the attention kernel of this shape
// (queried once per device and shape, cached).
int attention_ctas_per_sm(int dtype, int head_dim, int rb, bool mma,
                          int batch);

cudaError_t launch_attention(const AttnParams &p, int dtype, bool mma,
                             int grid, cudaStream_t stream);

// The merge of split groups after either attention kernel (same grid).
cudaError_t launch_merge(const AttnParams &p, int dtype, int grid,
                         cudaStream_t stream);

// True when the driver provides cuTensorMapEncodeTiled.
bool tensor_maps_available();

// The tcgen05 kernel (attention_tc.cu): bf16, head_dim 128, 16 or 32 rows
// per group, at most tc_batch_cap() sequences per launch.
int tc_batch_cap();
int attention_tc_ctas_per_sm(int rb, int batch);
cudaError_t launch_attention_tc(const AttnParams &p, int grid,
                                cudaStream_t stream);

struct AppendParams {
  const void *k_new;
  const void *v_new;
  void *k_cache;
  void *v_cache;
  const int32_t *block_table;
  const int32_t *seq_lens;
  int batch, num_kv_heads, head_dim, n_new, max_blocks, num_blocks;
  int elem_bytes;
  int fp8;                   // bf16 rows quantised into E4M3 caches
  float k_scale, v_scale;
};
cudaError_t launch_kv_append(const AppendParams &p, cudaStream_t stream);

struct AcceptParams {
  const float *target_logits;
  const float *draft_logits;
  const int32_t *draft_tokens;
  const float *uniforms;
  int32_t *out_tokens;
  int32_t *n_accepted;
  int batch, num_draft, vocab;
  float sc;                  // log2(e) / temperature
  const uint32_t *allowed;   // [batch, K+1, words] token masks, or null
  int words;                 // (vocab + 31) / 32
  int greedy;                // argmax verification
  cudaStream_t stream;       // set by the launcher
};
cudaError_t launch_spec_accept(const AcceptParams &p, cudaStream_t stream);

struct AcceptTreeParams {
  const float *target_logits;  // [batch, N, vocab]
  const float *draft_logits;   // [batch, N, vocab]
  const int32_t *parents;      // [batch, N]
  const int32_t *node_tokens;  // [batch, N]
  const float *uniforms;       // [batch, N]
  int32_t *out_tokens;         // [batch, N]
  int32_t *out_nodes;          // [batch, N]
  int32_t *n_accepted;         // [batch]
  int batch, num_nodes, vocab;
};
cudaError_t launch_spec_accept_tree(const AcceptTreeParams &p,
                                    cudaStream_t stream);

// Device status words (one per translation unit): read-and-clear.
cudaError_t read_status_attention(cudaStream_t s, unsigned *flags);
cudaError_t read_status_attention_tc(cudaStream_t s, unsigned *flags);
cudaError_t read_status_append(cudaStream_t s, unsigned *flags);
cudaError_t read_status_accept(cudaStream_t s, unsigned *flags);

#ifdef __CUDACC__
// A launch that may start while the previous kernel on the stream is still
// running (programmatic dependent launch); the kernel itself waits for that
// kernel's results (pdl_wait) before it reads anything it could have
// written.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), unsigned grid, unsigned block,
                       size_t smem, cudaStream_t stream, Args &&...args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}
#endif

}  // namespace svp
