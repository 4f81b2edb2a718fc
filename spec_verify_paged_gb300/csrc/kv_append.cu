// kv_append.cu -- scatter the new tokens' K/V rows into the paged cache.
//
// Page: "KV cache & Flash Attention", sections "KV cache" (store K and V of
// every token once) and "PagedAttention" (logical position -> physical
// block via the page table).  Row (b, k, g) of k_new/v_new goes to logical
// position pos = seq_lens[b] - n_new + k, i.e. page block_table[b][pos/16],
// row pos % 16, kv head g.  A byte copy: one warp moves one K row and one V
// row with 16-byte vector accesses.  Into an FP8 E4M3 cache each bf16 value
// x becomes the code of x / scale (round to nearest even, saturating).
#include <cuda_fp8.h>

#include <cstdint>

#include "ptx.cuh"
#include "svp.h"
#include "svp_internal.h"

namespace svp {

static __device__ unsigned int g_status_append;

constexpr int kAppendWarps = 8;

__global__ void __launch_bounds__(32 * kAppendWarps)
    kv_append_kernel(const AppendParams p) {
  // the attention kernel that usually follows may set itself up meanwhile;
  // it reads the caches only after this grid has completed
  pdl_launch_dependents();
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * kAppendWarps + (threadIdx.x >> 5);
  const long long n_rows = (long long)p.batch * p.n_new * p.num_kv_heads;
  if (row >= n_rows) return;
  const int g = (int)(row % p.num_kv_heads);
  const int k = (int)((row / p.num_kv_heads) % p.n_new);
  const int b = (int)(row / ((long long)p.num_kv_heads * p.n_new));
  const int L = p.seq_lens[b];
  if (L < p.n_new || L > p.max_blocks * kBlockSize) {
    if (lane == 0) atomicOr(&g_status_append, (unsigned)SVP_DEV_BAD_SEQ_LEN);
    return;
  }
  const int pos = L - p.n_new + k;
  const int phys = p.block_table[(size_t)b * p.max_blocks + pos / kBlockSize];
  if (phys < 0 || phys >= p.num_blocks) {
    if (lane == 0) atomicOr(&g_status_append, (unsigned)SVP_DEV_BAD_BLOCK_ID);
    return;
  }
  if (p.fp8) {
    // 8 bf16 values (16 bytes) in, 8 codes (8 bytes) out per lane step
    const size_t dst = ((((size_t)phys * p.num_kv_heads + g) * kBlockSize) +
                        pos % kBlockSize) * (size_t)p.head_dim;
    const size_t src = (size_t)row * p.head_dim * 2;
    for (int c = lane; c < p.head_dim / 8; c += 32) {
      const uint4 kv = reinterpret_cast<const uint4 *>(
          static_cast<const char *>(p.k_new) + src)[c];
      const uint4 vv = reinterpret_cast<const uint4 *>(
          static_cast<const char *>(p.v_new) + src)[c];
      auto quant = [](uint4 w, float s) {
        const uint32_t in[4] = {w.x, w.y, w.z, w.w};
        uint32_t out[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          uint32_t packed = 0;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const uint32_t u = in[2 * h + t];
            const float2 f = make_float2(__uint_as_float(u << 16) / s,
                                         __uint_as_float(u & 0xffff0000u) / s);
            packed |= (uint32_t)__nv_cvt_float2_to_fp8x2(f, __NV_SATFINITE,
                                                         __NV_E4M3)
                      << (16 * t);
          }
          out[h] = packed;
        }
        return make_uint2(out[0], out[1]);
      };
      reinterpret_cast<uint2 *>(static_cast<char *>(p.k_cache) + dst)[c] =
          quant(kv, p.k_scale);
      reinterpret_cast<uint2 *>(static_cast<char *>(p.v_cache) + dst)[c] =
          quant(vv, p.v_scale);
    }
    return;
  }
  const size_t row_bytes = (size_t)p.head_dim * p.elem_bytes;
  const size_t dst = ((((size_t)phys * p.num_kv_heads + g) * kBlockSize) +
                      pos % kBlockSize) * row_bytes;
  const size_t src = (size_t)row * row_bytes;
  const int chunks = (int)(row_bytes / 16);
  for (int c = lane; c < chunks; c += 32) {
    const uint4 kv = reinterpret_cast<const uint4 *>(
        static_cast<const char *>(p.k_new) + src)[c];
    const uint4 vv = reinterpret_cast<const uint4 *>(
        static_cast<const char *>(p.v_new) + src)[c];
    reinterpret_cast<uint4 *>(static_cast<char *>(p.k_cache) + dst)[c] = kv;
    reinterpret_cast<uint4 *>(static_cast<char *>(p.v_cache) + dst)[c] = vv;
  }
}

cudaError_t launch_kv_append(const AppendParams &p, cudaStream_t stream) {
  const long long n_rows = (long long)p.batch * p.n_new * p.num_kv_heads;
  if (n_rows == 0) return cudaSuccess;
  const long long grid = (n_rows + kAppendWarps - 1) / kAppendWarps;
  kv_append_kernel<<<(unsigned)grid, 32 * kAppendWarps, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t read_status_append(cudaStream_t s, unsigned *flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status_append, sizeof v, 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbolAsync(g_status_append, &zero, sizeof zero, 0,
                              cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  *flags |= v;
  return e;
}

}  // namespace svp
