// step.cu -- the graph-captured decode step: kv_append, attention and the
// acceptance step replayed as one CUDA graph per ping-pong slot, with the
// result copy on its own stream.
//
// Page: "How Moondream cut VLM inference latency by 35% via pipelined
// decoding", sections "The problem: the GPU bubble" and "Mechanism one:
// ping-pong slots": a decode step's working buffers live in pinned host
// slots; fixed buffer addresses let the step be captured once as a CUDA
// graph and replayed; two slots alternate so the host prepares one step
// while the GPU runs the other; the device-to-host copy of a step's result
// runs on a separate copy stream, ordered after an event recorded when that
// step's outputs are written (not after work queued behind it); a slot is
// reused only once its result copy has completed.  The slot's input copy
// runs on an upload stream of its own, ordered only after the slot's
// previous step has finished with its inputs, so the next step's upload
// overlaps the current step's kernels.
//
// Host code only: the kernels are the library's own entry points, called
// while the slot's graph is captured.
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "svp.h"
#include "svp_internal.h"

struct svp_step {
  svp_step_desc desc;
  cudaStream_t compute = nullptr, copy = nullptr, upload = nullptr;
  void *workspace = nullptr;
  size_t ws_bytes = 0;
  size_t off[SVP_STEP_NUM_FIELDS] = {};    // offsets in the input / output blocks
  size_t bytes[SVP_STEP_NUM_FIELDS] = {};
  size_t in_bytes = 0, out_bytes = 0;
  struct Slot {
    unsigned char *host_in = nullptr, *host_out = nullptr;  // pinned
    unsigned char *dev_in = nullptr, *dev_out = nullptr;
    cudaGraphExec_t exec = nullptr;
    cudaEvent_t done = nullptr;  // the step's outputs are written
    cudaEvent_t out = nullptr;   // its result copy has completed
    cudaEvent_t in = nullptr;    // its input copy has completed
    bool launched = false;
  } slot[2];
};

namespace {

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool is_input(int f) {
  return f < SVP_STEP_OUT ||
         (f >= SVP_STEP_ALLOWED && f <= SVP_STEP_NODE_TOKENS);
}

void release(svp_step *s) {
  for (auto &sl : s->slot) {
    if (sl.exec) cudaGraphExecDestroy(sl.exec);
    if (sl.done) cudaEventDestroy(sl.done);
    if (sl.out) cudaEventDestroy(sl.out);
    if (sl.in) cudaEventDestroy(sl.in);
    if (sl.host_in) cudaFreeHost(sl.host_in);
    if (sl.host_out) cudaFreeHost(sl.host_out);
    if (sl.dev_in) cudaFree(sl.dev_in);
    if (sl.dev_out) cudaFree(sl.dev_out);
  }
  if (s->workspace) cudaFree(s->workspace);
  if (s->compute) cudaStreamDestroy(s->compute);
  if (s->copy) cudaStreamDestroy(s->copy);
  if (s->upload) cudaStreamDestroy(s->upload);
  delete s;
}

// Captures slot i's step on the compute stream: kv_append, attention and
// (with drafts or a tree) the acceptance step on the slot's device buffers
// (the input copy from the pinned slot is issued at launch).
int capture_slot(svp_step *s, int i) {
  svp_step::Slot &sl = s->slot[i];
  const svp_step_desc &d = s->desc;
  auto in = [&](int f) { return (void *)(sl.dev_in + s->off[f]); };
  auto out = [&](int f) { return (void *)(sl.dev_out + s->off[f]); };
  svp_dims dims = d.dims;
  dims.workspace = s->workspace;
  dims.workspace_bytes = s->ws_bytes;
  cudaGraph_t graph = nullptr;
  if (cudaStreamBeginCapture(s->compute, cudaStreamCaptureModeRelaxed) !=
      cudaSuccess)
    return SVP_ERR_CUDA;
  int st = kv_append(&dims, in(SVP_STEP_K_NEW), in(SVP_STEP_V_NEW), d.k_cache,
                   d.v_cache, (const int32_t *)in(SVP_STEP_BLOCK_TABLE),
                   (const int32_t *)in(SVP_STEP_SEQ_LENS), d.q_len, s->compute);
  const bool tree = d.tree_nodes > 0;
  // attention right behind the append of its q_len newest positions: it
  // reads the prefix pages while the append runs
  if (st == SVP_OK)
    st = svp::attention_after_append(
        &dims, in(SVP_STEP_Q), d.k_cache, d.v_cache,
        (const int32_t *)in(SVP_STEP_BLOCK_TABLE),
        (const int32_t *)in(SVP_STEP_SEQ_LENS), d.q_len, tree ? 0 : d.n_sink,
        tree ? 0 : d.window,
        tree ? (const uint32_t *)in(SVP_STEP_TREE_MASK) : nullptr, d.scale,
        out(SVP_STEP_OUT), (float *)out(SVP_STEP_LSE), s->compute);
  if (st == SVP_OK && tree) {
    st = spec_accept_tree(d.dims.batch, d.tree_nodes, d.vocab,
                          (const float *)in(SVP_STEP_TARGET_LOGITS),
                          (const float *)in(SVP_STEP_DRAFT_LOGITS),
                          (const int32_t *)in(SVP_STEP_PARENTS),
                          (const int32_t *)in(SVP_STEP_NODE_TOKENS),
                          (const float *)in(SVP_STEP_UNIFORMS),
                          (int32_t *)out(SVP_STEP_OUT_TOKENS),
                          (int32_t *)out(SVP_STEP_OUT_NODES),
                          (int32_t *)out(SVP_STEP_N_ACCEPTED), s->compute);
  } else if (st == SVP_OK && d.num_draft > 0) {
    svp_accept_opts o;
    o.temperature = d.temperature > 0.f ? d.temperature : 1.f;
    o.allowed = d.use_mask ? (const uint32_t *)in(SVP_STEP_ALLOWED) : nullptr;
    o.greedy = d.greedy;
    st = spec_accept_ex(d.dims.batch, d.num_draft, d.vocab,
                        (const float *)in(SVP_STEP_TARGET_LOGITS),
                        (const float *)in(SVP_STEP_DRAFT_LOGITS),
                        (const int32_t *)in(SVP_STEP_DRAFT_TOKENS),
                        (const float *)in(SVP_STEP_UNIFORMS), &o,
                        (int32_t *)out(SVP_STEP_OUT_TOKENS),
                        (int32_t *)out(SVP_STEP_N_ACCEPTED), s->compute);
  }
  const cudaError_t e = cudaStreamEndCapture(s->compute, &graph);
  if (st != SVP_OK) {
    if (graph) cudaGraphDestroy(graph);
    return st;
  }
  if (e != cudaSuccess || !graph) return SVP_ERR_CUDA;
  const cudaError_t ei = cudaGraphInstantiate(&sl.exec, graph, 0);
  cudaGraphDestroy(graph);
  return ei == cudaSuccess ? SVP_OK : SVP_ERR_CUDA;
}

}  // namespace

extern "C" {

int svp_step_create(const svp_step_desc *desc, svp_step **out) {
  if (!desc || !out) return SVP_ERR_INVALID_ARG;
  *out = nullptr;
  const svp_dims &dm = desc->dims;
  if (dm.batch < 1 || dm.num_q_heads < 1 || dm.num_kv_heads < 1 ||
      dm.head_dim < 1 || dm.max_blocks_per_seq < 1 || dm.num_blocks < 1 ||
      desc->q_len < 1 || desc->num_draft < 0 || !desc->k_cache ||
      !desc->v_cache)
    return SVP_ERR_INVALID_ARG;
  if (desc->num_draft > 0 && (desc->num_draft != desc->q_len - 1 ||
                              desc->vocab < 2))
    return SVP_ERR_INVALID_ARG;
  const bool opts = desc->greedy || desc->use_mask ||
                    (desc->temperature > 0.f && desc->temperature != 1.f);
  if (desc->temperature < 0.f || (opts && desc->num_draft == 0))
    return SVP_ERR_INVALID_ARG;
  if (desc->tree_nodes < 0 ||
      (desc->tree_nodes > 0 &&
       (desc->tree_nodes != desc->q_len || desc->num_draft != 0 || opts ||
        desc->n_sink != 0 || desc->window != 0 || desc->vocab < 2)))
    return SVP_ERR_INVALID_ARG;
  if (desc->tree_nodes > svp::kMaxNodes) return SVP_ERR_UNSUPPORTED;
  const size_t ws = paged_decode_workspace_size(&dm, desc->q_len,
                                                desc->n_sink, desc->window);
  if (ws == 0) return SVP_ERR_INVALID_ARG;

  svp_step *s = new (std::nothrow) svp_step;
  if (!s) return SVP_ERR_INVALID_ARG;
  s->desc = *desc;
  s->ws_bytes = ws;
  const size_t B = (size_t)dm.batch, Q = (size_t)desc->q_len;
  const size_t eb = dm.dtype == SVP_F32 ? 4 : 2;
  const size_t K = (size_t)desc->num_draft, V = (size_t)desc->vocab;
  const size_t N = (size_t)desc->tree_nodes;
  const size_t rows_t = N ? N : (K ? K + 1 : 0);  // target rows, uniforms
  const size_t rows_d = N ? N : K;                // draft rows
  s->bytes[SVP_STEP_Q] = B * Q * dm.num_q_heads * dm.head_dim * eb;
  s->bytes[SVP_STEP_K_NEW] = B * Q * dm.num_kv_heads * dm.head_dim * eb;
  s->bytes[SVP_STEP_V_NEW] = s->bytes[SVP_STEP_K_NEW];
  s->bytes[SVP_STEP_BLOCK_TABLE] = B * dm.max_blocks_per_seq * 4;
  s->bytes[SVP_STEP_SEQ_LENS] = B * 4;
  s->bytes[SVP_STEP_TARGET_LOGITS] = B * rows_t * V * 4;
  s->bytes[SVP_STEP_DRAFT_LOGITS] = B * rows_d * V * 4;
  s->bytes[SVP_STEP_DRAFT_TOKENS] = B * K * 4;
  s->bytes[SVP_STEP_UNIFORMS] = B * rows_t * 4;
  s->bytes[SVP_STEP_OUT] = s->bytes[SVP_STEP_Q];
  s->bytes[SVP_STEP_LSE] = B * Q * dm.num_q_heads * 4;
  s->bytes[SVP_STEP_OUT_TOKENS] = B * rows_t * 4;
  s->bytes[SVP_STEP_N_ACCEPTED] = rows_t ? B * 4 : 0;
  s->bytes[SVP_STEP_ALLOWED] =
      desc->use_mask ? B * (K + 1) * ((V + 31) / 32) * 4 : 0;
  s->bytes[SVP_STEP_TREE_MASK] = B * N * 4;
  s->bytes[SVP_STEP_PARENTS] = B * N * 4;
  s->bytes[SVP_STEP_NODE_TOKENS] = B * N * 4;
  s->bytes[SVP_STEP_OUT_NODES] = B * N * 4;
  for (int f = 0; f < SVP_STEP_NUM_FIELDS; ++f) {
    size_t &total = is_input(f) ? s->in_bytes : s->out_bytes;
    s->off[f] = total;
    total += align256(s->bytes[f]);
  }
  int st = SVP_OK;
  if (cudaStreamCreateWithFlags(&s->compute, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&s->copy, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&s->upload, cudaStreamNonBlocking) != cudaSuccess ||
      cudaMalloc(&s->workspace, ws) != cudaSuccess)
    st = SVP_ERR_CUDA;
  for (int i = 0; i < 2 && st == SVP_OK; ++i) {
    svp_step::Slot &sl = s->slot[i];
    if (cudaHostAlloc((void **)&sl.host_in, s->in_bytes, cudaHostAllocDefault) != cudaSuccess ||
        cudaHostAlloc((void **)&sl.host_out, s->out_bytes, cudaHostAllocDefault) != cudaSuccess ||
        cudaMalloc((void **)&sl.dev_in, s->in_bytes) != cudaSuccess ||
        cudaMalloc((void **)&sl.dev_out, s->out_bytes) != cudaSuccess ||
        cudaEventCreateWithFlags(&sl.done, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sl.out, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sl.in, cudaEventDisableTiming) != cudaSuccess) {
      st = SVP_ERR_CUDA;
      break;
    }
    memset(sl.host_in, 0, s->in_bytes);
    memset(sl.host_out, 0, s->out_bytes);
  }
  for (int i = 0; i < 2 && st == SVP_OK; ++i) st = capture_slot(s, i);
  if (st != SVP_OK) {
    release(s);
    return st;
  }
  *out = s;
  return SVP_OK;
}

void *svp_step_host_buffer(svp_step *s, int slot, int field, size_t *bytes) {
  if (!s || slot < 0 || slot > 1 || field < 0 || field >= SVP_STEP_NUM_FIELDS)
    return nullptr;
  if (bytes) *bytes = s->bytes[field];
  if (s->bytes[field] == 0) return nullptr;
  svp_step::Slot &sl = s->slot[slot];
  return (is_input(field) ? sl.host_in : sl.host_out) + s->off[field];
}

int svp_step_launch(svp_step *s, int slot) {
  if (!s || slot < 0 || slot > 1) return SVP_ERR_INVALID_ARG;
  svp_step::Slot &sl = s->slot[slot];
  // the input copy: once the slot's previous step has finished with its
  // inputs, on the upload stream, so it overlaps the other slot's kernels
  if (sl.launched && cudaStreamWaitEvent(s->upload, sl.done, 0) != cudaSuccess)
    return SVP_ERR_CUDA;
  if (cudaMemcpyAsync(sl.dev_in, sl.host_in, s->in_bytes,
                      cudaMemcpyHostToDevice, s->upload) != cudaSuccess ||
      cudaEventRecord(sl.in, s->upload) != cudaSuccess)
    return SVP_ERR_CUDA;
  // the slot's previous result must have left its device buffers
  if (sl.launched && cudaStreamWaitEvent(s->compute, sl.out, 0) != cudaSuccess)
    return SVP_ERR_CUDA;
  if (cudaStreamWaitEvent(s->compute, sl.in, 0) != cudaSuccess ||
      cudaGraphLaunch(sl.exec, s->compute) != cudaSuccess ||
      cudaEventRecord(sl.done, s->compute) != cudaSuccess ||
      cudaStreamWaitEvent(s->copy, sl.done, 0) != cudaSuccess ||
      cudaMemcpyAsync(sl.host_out, sl.dev_out, s->out_bytes,
                      cudaMemcpyDeviceToHost, s->copy) != cudaSuccess ||
      cudaEventRecord(sl.out, s->copy) != cudaSuccess)
    return SVP_ERR_CUDA;
  sl.launched = true;
  return SVP_OK;
}

int svp_step_wait(svp_step *s, int slot) {
  if (!s || slot < 0 || slot > 1) return SVP_ERR_INVALID_ARG;
  svp_step::Slot &sl = s->slot[slot];
  if (!sl.launched) return SVP_OK;
  return cudaEventSynchronize(sl.out) == cudaSuccess ? SVP_OK : SVP_ERR_CUDA;
}

cudaStream_t svp_step_stream(svp_step *s) { return s ? s->compute : nullptr; }

int svp_step_destroy(svp_step *s) {
  if (!s) return SVP_OK;
  const bool ok = cudaStreamSynchronize(s->upload) == cudaSuccess &&
                  cudaStreamSynchronize(s->compute) == cudaSuccess &&
                  cudaStreamSynchronize(s->copy) == cudaSuccess;
  release(s);
  return ok ? SVP_OK : SVP_ERR_CUDA;
}

}  // extern "C"
