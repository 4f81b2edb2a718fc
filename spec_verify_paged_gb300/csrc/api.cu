// api.cu -- the C ABI of libsvp.so: argument checks, split planning,
// workspace handling and kernel launches.  Declarations and the full
// contract of every entry point are in include/svp.h.
#include <cmath>
#include <cstdint>
#include <algorithm>
#include <cstring>
#include <mutex>
#include <vector>

#include "svp.h"
#include "svp_internal.h"

namespace svp {

static thread_local int t_last_launches = 0;

// ---- per-device facts, queried once ----
struct DeviceInfo {
  int sms = 0;
};
static std::mutex g_mu;
static std::vector<DeviceInfo> g_dev;

static int device_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_dev.size() <= dev) g_dev.resize(dev + 1);
  if (g_dev[dev].sms == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
        cudaSuccess)
      return -1;
    g_dev[dev].sms = n;
  }
  return g_dev[dev].sms;
}

// ---- library-owned workspace (only when the caller passes none) ----
struct OwnedWs {
  void *ptr = nullptr;
  size_t bytes = 0;
};
static std::vector<OwnedWs> g_ws;

static int owned_workspace(size_t need, cudaStream_t stream, void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SVP_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_mu);
  if ((int)g_ws.size() <= dev) g_ws.resize(dev + 1);
  OwnedWs &w = g_ws[dev];
  if (w.bytes < need) {
    if (w.ptr) {
      if (cudaDeviceSynchronize() != cudaSuccess) return SVP_ERR_CUDA;
      cudaFree(w.ptr);
      w.ptr = nullptr;
      w.bytes = 0;
    }
    if (cudaMalloc(&w.ptr, need) != cudaSuccess) return SVP_ERR_CUDA;
    if (cudaMemsetAsync(w.ptr, 0, need, stream) != cudaSuccess)
      return SVP_ERR_CUDA;
    w.bytes = need;
  }
  *out = w.ptr;
  return SVP_OK;
}

static size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

static int check_dims(const svp_dims *d) {
  if (!d) return SVP_ERR_INVALID_ARG;
  if (d->batch < 0 || d->num_q_heads < 1 || d->num_kv_heads < 1 ||
      d->head_dim < 1 || d->block_size < 1 || d->max_blocks_per_seq < 0 ||
      d->num_blocks < 0 || d->split_pages < 0 || d->kernel_path < 0 ||
      d->kernel_path > SVP_PATH_TCGEN05)
    return SVP_ERR_INVALID_ARG;
  if (d->num_q_heads % d->num_kv_heads != 0) return SVP_ERR_INVALID_ARG;
  if (d->dtype != SVP_F32 && d->dtype != SVP_BF16 && d->dtype != SVP_FP8_E4M3)
    return SVP_ERR_INVALID_ARG;
  if (d->dtype == SVP_FP8_E4M3 &&
      !(std::isfinite(d->k_scale) && d->k_scale > 0.f &&
        std::isfinite(d->v_scale) && d->v_scale > 0.f))
    return SVP_ERR_INVALID_ARG;
  if (d->head_dim != 64 && d->head_dim != 128) return SVP_ERR_UNSUPPORTED;
  if (d->block_size != kBlockSize) return SVP_ERR_UNSUPPORTED;
  if (d->batch > kMaxBatch) return SVP_ERR_UNSUPPORTED;
  return SVP_OK;
}

// Upper bound of the pages one sequence's visible set can span.
static int max_visible_pages(int max_blocks, int q_len, int n_sink,
                             int window) {
  if (window == 0) return max_blocks;
  const long long sink_pages = (n_sink + kBlockSize - 1) / kBlockSize;
  const long long win_pages =
      ((long long)window + q_len - 1 + kBlockSize - 1) / kBlockSize + 1;
  const long long b = sink_pages + win_pages;
  return (int)(b < max_blocks ? b : max_blocks);
}

constexpr int kBatchPerLaunch = 4096;

// The kernel variant for this shape (a svp_kernel_path other than AUTO), or
// SVP_ERR_UNSUPPORTED for a forced path the shape cannot take.
static int select_path(int dtype, int head_dim, int rows, int kernel_path,
                       long long num_blocks, int num_kv_heads) {
  // the tensor paths address the cache as a 2-D tensor with int32 rows
  const bool tma_ok = tensor_maps_available() &&
                      num_blocks * num_kv_heads * kBlockSize < (1LL << 31);
  switch (kernel_path) {
    case SVP_PATH_CUDA_CORES:
      return SVP_PATH_CUDA_CORES;
    case SVP_PATH_TENSOR_CORES:
      if (dtype != SVP_BF16 || !tma_ok) return SVP_ERR_UNSUPPORTED;
      return SVP_PATH_TENSOR_CORES;
    case SVP_PATH_TCGEN05:
      if (dtype != SVP_BF16 || head_dim != 128 || !tma_ok)
        return SVP_ERR_UNSUPPORTED;
      return SVP_PATH_TCGEN05;
    default:
      if (dtype != SVP_BF16 || rows < kMmaMinRows || !tma_ok)
        return SVP_PATH_CUDA_CORES;
      return head_dim == 128 ? SVP_PATH_TCGEN05 : SVP_PATH_TENSOR_CORES;
  }
}

int plan_attention(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                   int dtype, int max_blocks, int q_len, int n_sink,
                   int window, int split_pages, int kernel_path, int num_sms,
                   long long num_blocks, AttnPlan *plan) {
  const int group = num_q_heads / num_kv_heads;
  const int rows = group * q_len;
  int path = select_path(dtype, head_dim, rows, kernel_path, num_blocks,
                         num_kv_heads);
  if (path < 0) return path;
  const bool mma = path == SVP_PATH_TENSOR_CORES;
  const bool tc = path == SVP_PATH_TCGEN05;
  // mma.sync: one m16 tile per warp, two warps share a page beyond 16 rows;
  // tcgen05: the rows are the MMA's N (16 or 32), or two 32-row groups
  // sharing each K/V tile beyond 32 rows
  int rb = tc    ? (rows <= 16 ? 16 : rows <= 32 ? 32 : 64)
           : mma ? (rows <= 16 ? 16 : 32)
                 : rows <= 1 ? 1 : rows <= 2 ? 2 : rows <= 4 ? 4 : 8;
  const int n_rg = (rows + rb - 1) / rb;
  const int ctas = tc ? attention_tc_ctas_per_sm(rb, batch)
                      : attention_ctas_per_sm(dtype, head_dim, rb, mma, batch);
  const long long groups = (long long)batch * num_kv_heads * n_rg;
  // Every CTA of the persistent grid takes an equal slice of all pages;
  // a slice holds at least min_pages pages (fewer CTAs for small calls).
  int min_pages = split_pages > 0 ? split_pages : 8;
  long long grid = (long long)num_sms * ctas;
  const long long page_bound =
      groups * (long long)max_visible_pages(max_blocks, q_len, n_sink, window);
  if (grid > page_bound / min_pages) grid = page_bound / min_pages;
  if (grid < 1) grid = 1;
  plan->rb = rb;
  plan->n_rg = n_rg;
  plan->mma = mma;
  plan->tc = tc;
  plan->batch_cap = tc ? tc_batch_cap() : kBatchPerLaunch;
  plan->min_pages = min_pages;
  plan->seg_items = tc ? kSegItemsTc : kSegItemsCc;
  plan->grid = (int)grid;
  plan->ctas_per_sm = ctas;
  plan->ws_head = 256;
  plan->ws_desc = align256((size_t)grid * 32);  // one SplitDesc per CTA
  plan->ws_part_o = align256((size_t)2 * grid * rb * head_dim * 4);
  plan->ws_part_lse = align256((size_t)2 * grid * rb * 4);
  plan->ws_total =
      plan->ws_head + plan->ws_desc + plan->ws_part_o + plan->ws_part_lse;
  return SVP_OK;
}

// Sequences per launch: at most the path's cap (the in-kernel prefix lives
// in shared memory) and few enough that the flattened page count fits in
// 32 bits.
static int batch_per_launch(const svp_dims *d, int q_len, int n_sink,
                            int window, int cap, int seg_items) {
  const long long rows = (long long)(d->num_q_heads / d->num_kv_heads) * q_len;
  const long long per_seq =
      (long long)d->num_kv_heads * rows *
      (max_visible_pages(d->max_blocks_per_seq, q_len, n_sink, window) +
       seg_items);
  long long bl = per_seq > 0 ? ((1LL << 31) - 1) / per_seq : cap;
  if (bl > cap) bl = cap;
  if (bl > d->batch) bl = d->batch;
  return bl < 1 ? 1 : (int)bl;
}

// The plan of one launch of a call: its path fixes the sequences per
// launch, which fix the grid and workspace.  plan->batch_cap is then the
// call's sequences per launch.
static int plan_call(const svp_dims *d, int q_len, int n_sink, int window,
                     int sms, AttnPlan *plan) {
  const int rows = (d->num_q_heads / d->num_kv_heads) * q_len;
  const int path = select_path(d->dtype, d->head_dim, rows, d->kernel_path,
                               d->num_blocks, d->num_kv_heads);
  if (path < 0) return path;
  const int cap = path == SVP_PATH_TCGEN05 ? tc_batch_cap() : kBatchPerLaunch;
  const int bl = batch_per_launch(d, q_len, n_sink, window, cap,
                                  path == SVP_PATH_TCGEN05 ? kSegItemsTc : kSegItemsCc);
  const int st = plan_attention(bl, d->num_q_heads, d->num_kv_heads,
                                d->head_dim, d->dtype, d->max_blocks_per_seq,
                                q_len, n_sink, window, d->split_pages, path,
                                sms, d->num_blocks, plan);
  plan->batch_cap = bl;
  return st;
}

}  // namespace svp

using namespace svp;

extern "C" {

const char *svp_status_string(int s) {
  switch (s) {
    case SVP_OK: return "SVP_OK";
    case SVP_ERR_INVALID_ARG: return "SVP_ERR_INVALID_ARG";
    case SVP_ERR_UNSUPPORTED: return "SVP_ERR_UNSUPPORTED";
    case SVP_ERR_CUDA: return "SVP_ERR_CUDA";
    case SVP_ERR_WORKSPACE: return "SVP_ERR_WORKSPACE";
    default: return "SVP_UNKNOWN_STATUS";
  }
}

int svp_last_launch_count(void) { return t_last_launches; }

static int check_attention_args(const svp_dims *dims, int q_len, int n_sink,
                                int window, float scale) {
  int st = check_dims(dims);
  if (st != SVP_OK) return st;
  if (q_len < 1 || n_sink < 0 || window < 0 || !std::isfinite(scale))
    return SVP_ERR_INVALID_ARG;
  if (q_len > kMaxQLen) return SVP_ERR_UNSUPPORTED;
  return SVP_OK;
}

size_t paged_decode_workspace_size(const svp_dims *dims, int q_len, int n_sink,
                                   int window) {
  if (check_attention_args(dims, q_len, n_sink, window, 1.0f) != SVP_OK)
    return 0;
  const int sms = device_sms();
  AttnPlan plan;
  if (plan_call(dims, q_len, n_sink, window, sms > 0 ? sms : 1, &plan) !=
      SVP_OK)
    return 0;
  return plan.ws_total;
}

// The attention call behind both entry points; tree_mask (device, [batch,
// q_len] uint32 ancestor bits) replaces the causal block when not null.
static int attention_call(const svp_dims *dims, const void *q,
                          const void *k_cache, const void *v_cache,
                          const int32_t *block_table, const int32_t *seq_lens,
                          int q_len, int n_sink, int window,
                          const uint32_t *tree_mask, float scale, void *out,
                          float *lse, cudaStream_t stream, int early = 0) {
  t_last_launches = 0;
  int st = check_attention_args(dims, q_len, n_sink, window, scale);
  if (st != SVP_OK) return st;
  if (dims->batch == 0) return SVP_OK;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !out || !lse)
    return SVP_ERR_INVALID_ARG;
  if (dims->num_blocks == 0 || dims->max_blocks_per_seq == 0)
    return SVP_ERR_INVALID_ARG;
  // pages, q and out move with 16-byte bulk copies
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache) | reinterpret_cast<uintptr_t>(out)) %
          16 != 0)
    return SVP_ERR_INVALID_ARG;
  const int sms = device_sms();
  if (sms <= 0) return SVP_ERR_CUDA;

  AttnPlan plan;
  st = plan_call(dims, q_len, n_sink, window, sms, &plan);
  if (st != SVP_OK) return st;
  const int bl = plan.batch_cap;
  void *ws = dims->workspace;
  if (ws) {
    if (dims->workspace_bytes < plan.ws_total) return SVP_ERR_WORKSPACE;
  } else {
    st = owned_workspace(plan.ws_total, stream, &ws);
    if (st != SVP_OK) return st;
  }
  // every CTA rewrites its split descriptor, so the workspace needs no
  // clearing between calls
  char *wp = static_cast<char *>(ws);
  const size_t eb = dims->dtype == SVP_F32 ? 4 : 2;  // q / out (bf16 for FP8)
  const size_t row_elems = (size_t)dims->num_q_heads * dims->head_dim;
  const bool fp8 = dims->dtype == SVP_FP8_E4M3;
  int launches = 0;
  for (int b0 = 0; b0 < dims->batch; b0 += bl) {
    const int nb = dims->batch - b0 < bl ? dims->batch - b0 : bl;
    AttnParams p;
    p.q = static_cast<const char *>(q) + (size_t)b0 * q_len * row_elems * eb;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.block_table = block_table + (size_t)b0 * dims->max_blocks_per_seq;
    p.seq_lens = seq_lens + b0;
    p.out = static_cast<char *>(out) + (size_t)b0 * q_len * row_elems * eb;
    p.lse = lse + (size_t)b0 * q_len * dims->num_q_heads;
    p.desc = reinterpret_cast<SplitDesc *>(wp + plan.ws_head);
    p.part_o = reinterpret_cast<float *>(wp + plan.ws_head + plan.ws_desc);
    p.part_lse = reinterpret_cast<float *>(wp + plan.ws_head + plan.ws_desc +
                                           plan.ws_part_o);
    p.batch = nb;
    p.num_q_heads = dims->num_q_heads;
    p.num_kv_heads = dims->num_kv_heads;
    p.head_dim = dims->head_dim;
    p.group = dims->num_q_heads / dims->num_kv_heads;
    p.q_len = q_len;
    p.n_sink = n_sink;
    p.window = window;
    p.max_blocks = dims->max_blocks_per_seq;
    p.num_blocks = dims->num_blocks;
    p.rows = p.group * q_len;
    p.rb = plan.rb;
    p.n_rg = plan.n_rg;
    // tcgen05: items are 8-page tiles (a slice's minimum in tiles)
    p.ppi = plan.tc ? kTilePagesTc : 1;
    p.min_pages = plan.tc ? std::max(1, plan.min_pages / kTilePagesTc)
                          : plan.min_pages;
    p.seg_items = plan.seg_items;
    // an FP8 cache's K scale folds into the query scale, its V scale
    // multiplies the outputs
    p.qscale = scale * 1.4426950408889634f * (fp8 ? dims->k_scale : 1.0f);
    p.v_scale = fp8 ? dims->v_scale : 1.0f;
    p.tree_mask = tree_mask ? tree_mask + (size_t)b0 * q_len : nullptr;
    // only the first launch follows the append: a later one follows the
    // previous launch's merge, which reads the workspace it would reset
    p.early = early && b0 == 0;
    AttnPlan sub = plan;
    if (nb != bl) {
      plan_attention(nb, dims->num_q_heads, dims->num_kv_heads,
                     dims->head_dim, dims->dtype, dims->max_blocks_per_seq,
                     q_len, n_sink, window, plan.min_pages,
                     plan.tc    ? SVP_PATH_TCGEN05
                     : plan.mma ? SVP_PATH_TENSOR_CORES
                                : SVP_PATH_CUDA_CORES,
                     sms, dims->num_blocks, &sub);
    }
    cudaError_t e =
        plan.tc ? launch_attention_tc(p, sub.grid, stream)
                : launch_attention(p, dims->dtype, plan.mma, sub.grid, stream);
    if (e != cudaSuccess) return SVP_ERR_CUDA;
    // groups split over several CTAs are finished by the merge kernel
    if (launch_merge(p, dims->dtype, sub.grid, stream) != cudaSuccess)
      return SVP_ERR_CUDA;
    launches += 2;
  }
  t_last_launches = launches;
  return SVP_OK;
}

int paged_decode_attention(const svp_dims *dims, const void *q,
                           const void *k_cache, const void *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           int q_len, int n_sink, int window, float scale,
                           void *out, float *lse, cudaStream_t stream) {
  return attention_call(dims, q, k_cache, v_cache, block_table, seq_lens,
                        q_len, n_sink, window, nullptr, scale, out, lse,
                        stream);
}

static int tree_call(const svp_dims *dims, const void *q, const void *k_cache,
                     const void *v_cache, const int32_t *block_table,
                     const int32_t *seq_lens, int q_len,
                     const uint32_t *tree_mask, float scale, void *out,
                     float *lse, cudaStream_t stream, int early) {
  t_last_launches = 0;
  const int st = check_attention_args(dims, q_len, 0, 0, scale);
  if (st != SVP_OK) return st;
  if (dims->batch == 0) return SVP_OK;
  if (!tree_mask || reinterpret_cast<uintptr_t>(tree_mask) % 4 != 0)
    return SVP_ERR_INVALID_ARG;
  return attention_call(dims, q, k_cache, v_cache, block_table, seq_lens,
                        q_len, 0, 0, tree_mask, scale, out, lse, stream, early);
}

int paged_tree_attention(const svp_dims *dims, const void *q,
                         const void *k_cache, const void *v_cache,
                         const int32_t *block_table, const int32_t *seq_lens,
                         int q_len, const uint32_t *tree_mask, float scale,
                         void *out, float *lse, cudaStream_t stream) {
  return tree_call(dims, q, k_cache, v_cache, block_table, seq_lens, q_len,
                   tree_mask, scale, out, lse, stream, 0);
}

int kv_append(const svp_dims *dims, const void *k_new, const void *v_new,
              void *k_cache, void *v_cache, const int32_t *block_table,
              const int32_t *seq_lens, int n_new, cudaStream_t stream) {
  t_last_launches = 0;
  int st = check_dims(dims);
  if (st != SVP_OK) return st;
  if (n_new < 0) return SVP_ERR_INVALID_ARG;
  if (n_new > 64) return SVP_ERR_UNSUPPORTED;
  if (dims->batch == 0 || n_new == 0) return SVP_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !block_table || !seq_lens)
    return SVP_ERR_INVALID_ARG;
  if (dims->num_blocks == 0 || dims->max_blocks_per_seq == 0)
    return SVP_ERR_INVALID_ARG;
  // rows move as 16-byte (8-byte for FP8 codes) vectors: reject unaligned
  // pointers here rather than fault on the device
  if ((reinterpret_cast<uintptr_t>(k_new) | reinterpret_cast<uintptr_t>(v_new) |
       reinterpret_cast<uintptr_t>(k_cache) |
       reinterpret_cast<uintptr_t>(v_cache)) % 16 != 0)
    return SVP_ERR_INVALID_ARG;
  AppendParams p;
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.batch = dims->batch;
  p.num_kv_heads = dims->num_kv_heads;
  p.head_dim = dims->head_dim;
  p.n_new = n_new;
  p.max_blocks = dims->max_blocks_per_seq;
  p.num_blocks = dims->num_blocks;
  p.elem_bytes = dims->dtype == SVP_F32 ? 4 : 2;
  p.fp8 = dims->dtype == SVP_FP8_E4M3;
  p.k_scale = p.fp8 ? dims->k_scale : 1.0f;
  p.v_scale = p.fp8 ? dims->v_scale : 1.0f;
  if (launch_kv_append(p, stream) != cudaSuccess) return SVP_ERR_CUDA;
  t_last_launches = 1;
  return SVP_OK;
}

int spec_accept_ex(int batch, int num_draft, int vocab,
                   const float *target_logits, const float *draft_logits,
                   const int32_t *draft_tokens, const float *uniforms,
                   const svp_accept_opts *opts, int32_t *out_tokens,
                   int32_t *n_accepted, cudaStream_t stream) {
  t_last_launches = 0;
  if (batch < 0 || num_draft < 1 || vocab < 2) return SVP_ERR_INVALID_ARG;
  if (num_draft > kMaxDraft || batch > kMaxBatch) return SVP_ERR_UNSUPPORTED;
  if ((long long)vocab > 8LL * 40000) return SVP_ERR_UNSUPPORTED;
  const float temperature = opts ? opts->temperature : 1.0f;
  const bool greedy = opts && opts->greedy;
  if (!greedy && !(std::isfinite(temperature) && temperature > 0.f))
    return SVP_ERR_INVALID_ARG;
  const uint32_t *allowed = opts ? opts->allowed : nullptr;
  if (allowed && reinterpret_cast<uintptr_t>(allowed) % 4 != 0)
    return SVP_ERR_INVALID_ARG;
  if (batch == 0) return SVP_OK;
  if (!target_logits || !draft_logits || !draft_tokens || !uniforms ||
      !out_tokens || !n_accepted)
    return SVP_ERR_INVALID_ARG;
  AcceptParams p;
  p.target_logits = target_logits;
  p.draft_logits = draft_logits;
  p.draft_tokens = draft_tokens;
  p.uniforms = uniforms;
  p.out_tokens = out_tokens;
  p.n_accepted = n_accepted;
  p.batch = batch;
  p.num_draft = num_draft;
  p.vocab = vocab;
  p.sc = 1.4426950408889634f / (greedy ? 1.0f : temperature);
  p.allowed = allowed;
  p.words = (vocab + 31) / 32;
  p.greedy = greedy ? 1 : 0;
  p.stream = stream;
  if (launch_spec_accept(p, stream) != cudaSuccess) return SVP_ERR_CUDA;
  t_last_launches = 1;
  return SVP_OK;
}

int spec_accept(int batch, int num_draft, int vocab,
                const float *target_logits, const float *draft_logits,
                const int32_t *draft_tokens, const float *uniforms,
                int32_t *out_tokens, int32_t *n_accepted,
                cudaStream_t stream) {
  return spec_accept_ex(batch, num_draft, vocab, target_logits, draft_logits,
                        draft_tokens, uniforms, nullptr, out_tokens,
                        n_accepted, stream);
}

int spec_accept_tree(int batch, int num_nodes, int vocab,
                     const float *target_logits, const float *draft_logits,
                     const int32_t *parents, const int32_t *node_tokens,
                     const float *uniforms, int32_t *out_tokens,
                     int32_t *out_nodes, int32_t *n_accepted,
                     cudaStream_t stream) {
  t_last_launches = 0;
  if (batch < 0 || num_nodes < 1 || vocab < 2) return SVP_ERR_INVALID_ARG;
  if (num_nodes > kMaxNodes || batch > kMaxBatch) return SVP_ERR_UNSUPPORTED;
  if ((long long)vocab > 8LL * 40000) return SVP_ERR_UNSUPPORTED;
  if (batch == 0) return SVP_OK;
  if (!target_logits || !draft_logits || !parents || !node_tokens ||
      !uniforms || !out_tokens || !out_nodes || !n_accepted)
    return SVP_ERR_INVALID_ARG;
  AcceptTreeParams p;
  p.target_logits = target_logits;
  p.draft_logits = draft_logits;
  p.parents = parents;
  p.node_tokens = node_tokens;
  p.uniforms = uniforms;
  p.out_tokens = out_tokens;
  p.out_nodes = out_nodes;
  p.n_accepted = n_accepted;
  p.batch = batch;
  p.num_nodes = num_nodes;
  p.vocab = vocab;
  if (launch_spec_accept_tree(p, stream) != cudaSuccess) return SVP_ERR_CUDA;
  t_last_launches = 1;
  return SVP_OK;
}

int svp_read_device_status(cudaStream_t stream, int *flags) {
  unsigned f = 0;
  if (read_status_attention(stream, &f) != cudaSuccess) return SVP_ERR_CUDA;
  if (read_status_attention_tc(stream, &f) != cudaSuccess) return SVP_ERR_CUDA;
  if (read_status_append(stream, &f) != cudaSuccess) return SVP_ERR_CUDA;
  if (read_status_accept(stream, &f) != cudaSuccess) return SVP_ERR_CUDA;
  if (flags) *flags = (int)f;
  return SVP_OK;
}

}  // extern "C"

namespace svp {

int attention_after_append(const svp_dims *dims, const void *q,
                           const void *k_cache, const void *v_cache,
                           const int32_t *block_table, const int32_t *seq_lens,
                           int q_len, int n_sink, int window,
                           const uint32_t *tree_mask, float scale, void *out,
                           float *lse, cudaStream_t stream) {
  if (tree_mask)
    return tree_call(dims, q, k_cache, v_cache, block_table, seq_lens, q_len,
                     tree_mask, scale, out, lse, stream, 1);
  return attention_call(dims, q, k_cache, v_cache, block_table, seq_lens,
                        q_len, n_sink, window, nullptr, scale, out, lse, stream,
                        1);
}

}  // namespace svp
