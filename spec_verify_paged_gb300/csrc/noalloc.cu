// noalloc.cu -- paged_decode_attention for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc at the point where they need
// attention: code running while a CUDA graph is being captured (allocation
// is not a capturable operation), plug-ins whose host framework owns every
// device allocation through its own pool, and latency-critical loops where
// cudaMalloc/cudaFree would synchronise the device.  For them this file
// provides the split-K scratch of the attention kernel as a fixed array in
// the library's own device memory.
//
// The array lives in every GPU that loads the library, from module load
// until process exit.  Every call shares it, and it keeps the last call's
// contents.  Nothing in it must start at zero: every attention launch
// rewrites the split descriptor of each of its CTAs before the merge kernel
// reads any of them, and it writes them only after its grid-dependency
// wait, i.e. after the previous kernel on the stream (the previous call's
// merge) has finished, so the next call on the same stream cannot
// overwrite descriptors or partials the previous merge still reads.
// Calls that overlap on the GPU (other streams, other host threads) race
// on it.  The device address of the array is looked up once per device and
// cached for the life of the process's CUDA context.
#include <mutex>

#include "svp.h"
#include "svp_internal.h"

namespace svp {

constexpr size_t kStaticScratchBytes = SVP_STATIC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
static std::mutex g_scratch_mu;
static void *g_scratch_ptr[kMaxDevices];

// Device address of the scratch array on the current device, looked up once
// per device.  In host code the array's name is only a host-side stand-in,
// so the address must come from the runtime.
static int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return SVP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return SVP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess ||
        p == nullptr)
      return SVP_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return SVP_OK;
}

}  // namespace svp

extern "C" int paged_decode_attention_noalloc(
    const svp_dims *dims, const void *q, const void *k_cache,
    const void *v_cache, const int32_t *block_table, const int32_t *seq_lens,
    int q_len, int n_sink, int window, float scale, void *out, float *lse,
    cudaStream_t stream) {
  if (dims == nullptr) return SVP_ERR_INVALID_ARG;
  svp_dims d = *dims;
  d.workspace = nullptr;
  d.workspace_bytes = 0;
  size_t need = paged_decode_workspace_size(&d, q_len, n_sink, window);
  // automatic split size: fall back to longer splits (fewer partials) when
  // the default plan does not fit the fixed scratch
  for (int pps = 64; need > svp::kStaticScratchBytes && d.split_pages == 0 &&
                     pps <= 128;
       pps *= 2) {
    svp_dims t = d;
    t.split_pages = pps;
    const size_t n2 = paged_decode_workspace_size(&t, q_len, n_sink, window);
    if (n2 != 0 && n2 <= svp::kStaticScratchBytes) {
      d.split_pages = pps;
      need = n2;
    }
  }
  if (need > svp::kStaticScratchBytes) return SVP_ERR_WORKSPACE;
  void *scratch = nullptr;
  const int st = svp::scratch_address(&scratch);
  if (st != SVP_OK) return st;
  d.workspace = scratch;
  // need == 0 marks an invalid request: a zero size lets the checks of the
  // entry point below report the exact status before anything is launched
  d.workspace_bytes = need == 0 ? 0 : svp::kStaticScratchBytes;
  return paged_decode_attention(&d, q, k_cache, v_cache, block_table,
                                seq_lens, q_len, n_sink, window, scale, out,
                                lse, stream);
}
