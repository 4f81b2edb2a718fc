// attn_common.cuh -- pieces shared by the two paged-attention kernels
// (attention.cu: CUDA-core and warp-level mma.sync consumers;
// attention_tc.cu: tcgen05 consumers with tensor-memory accumulators).
//
// Scheduling (both kernels): the work of a call is the flattened list of
// (sequence b, kv head g, row group rg, visible page) items, sequence-major.
// CTA c of the n_ctas working CTAs takes the slice [c*P/n, (c+1)*P/n) of the
// P items ("stream-K"): every CTA reads the same number of pages whatever the
// length mix.  A slice cut into one or more segments, each a run of pages of
// a single group.  A group whose pages lie in several slices is finished by
// the CTA whose ticket arrives last: each contributor writes a normalised
// partial (o, log2-LSE) to its first- or last-segment slot, and the last one
// merges them by log-sum-exp in slice order ("KV cache & Flash Attention",
// section "FlashAttention -- the tiling trick": partial softmax states
// combine exactly by rescaling with exp(m_i - m)).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>
#include <mutex>

#include "ptx.cuh"
#include "svp.h"
#include "svp_internal.h"

namespace svp {

constexpr int kUnitRing = 4;
constexpr int kTableChunk = 128;     // block-table entries loaded per round
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kBoxElems = 64;        // 128-byte swizzle box: 64 bf16 columns
constexpr int kBoxBytes = kBlockSize * 128;

// One segment of a CTA's slice: pages [page0, page0 + n_pages) of group
// (b, g, rg).  CTAs f..l own the group's pages; `slot` says whether this is
// the CTA's first (0) or last (1) segment, which is where its partial goes.
struct UnitInfo {
  int b, g, rg, slot;
  int f, l, gstart, page0;
  int n_pages, seq_len, n_a, b_start;
  int valid, pad0, pad1, pad2;
};

struct TensorMaps {
  CUtensorMap k;
  CUtensorMap v;
};

// Visible logical blocks of a sequence: [0, n_a) followed by
// [b_start, b_start + n_pages - n_a).  (window == 0: all blocks.)
__device__ __forceinline__ void visible_pages(int L, int q_len, int n_sink,
                                              int window, int &n_a,
                                              int &b_start, int &n_pages) {
  const int nblk = (L + kBlockSize - 1) / kBlockSize;
  n_a = 0;
  b_start = 0;
  n_pages = nblk;
  if (window == 0) return;
  const int t0 = L - q_len;                     // first query position
  const int lo = max(0, t0 - window + 1);       // first window key (union)
  const int sink_end = min(n_sink, L);
  const int na = (sink_end + kBlockSize - 1) / kBlockSize;
  const int bs = lo / kBlockSize;
  if (bs <= na) return;                         // ranges touch: all blocks
  n_a = na;
  b_start = bs;
  n_pages = na + (nblk - bs);
}

// Logical block of the pidx-th visible page.
__device__ __forceinline__ int logical_block(const UnitInfo &ui, int pidx) {
  return pidx < ui.n_a ? pidx : ui.b_start + (pidx - ui.n_a);
}

__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(uint16_t *p, float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  *p = *reinterpret_cast<uint16_t *>(&h);
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map,
                                            int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::"
      "complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y),
      "r"(smem_u32(bar))
      : "memory");
}

// Barrier of the consumer warps on an mbarrier initialised with their
// count: bounded, unlike bar.sync.
__device__ __forceinline__ bool consumer_sync(uint64_t *bar, uint32_t &phase,
                                              int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(bar);
  bool ok = mbar_wait(bar, phase);
  phase ^= 1u;
  __syncwarp();
  return ok;
}

// Warp 0: prefix[b + 1] = items of sequences 0..b (visible pages x groups
// per sequence); returns the total on lane 0.  A sequence whose length is
// out of range contributes nothing and raises SVP_DEV_BAD_SEQ_LEN.
__device__ __forceinline__ int build_prefix(const AttnParams &p, int *prefix,
                                            int groups_per_seq, int lane,
                                            unsigned *status) {
  int run = 0;
  if (lane == 0) prefix[0] = 0;
  for (int b0 = 0; b0 < p.batch; b0 += 32) {
    const int b = b0 + lane;
    int n = 0;
    if (b < p.batch) {
      const int L = p.seq_lens[b];
      if (L < p.q_len || L > p.max_blocks * kBlockSize) {
        if (blockIdx.x == 0) atomicOr(status, (unsigned)SVP_DEV_BAD_SEQ_LEN);
      } else {
        int na, bs, np;
        visible_pages(L, p.q_len, p.n_sink, p.window, na, bs, np);
        n = np * groups_per_seq;
      }
    }
    int incl = n;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int y = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += y;
    }
    if (b < p.batch) prefix[b + 1] = run + incl;
    run += __shfl_sync(kFull, incl, 31);
  }
  return run;
}

// CTAs that share the items: each slice holds at least min_pages items.
__device__ __forceinline__ int working_ctas(int total, int min_pages) {
  long long ce = total / (min_pages > 0 ? min_pages : 1);
  if (ce > (long long)gridDim.x) ce = gridDim.x;
  if (ce < 1) ce = 1;
  return (int)ce;
}

__device__ __forceinline__ int slice_begin(int cta, int total, int n_ctas) {
  return cta < n_ctas ? (int)((long long)cta * total / n_ctas) : total;
}

// The segment that starts at flat item `pos` of this CTA's slice.
__device__ __forceinline__ UnitInfo decode_segment(const AttnParams &p,
                                                   const int *prefix,
                                                   int groups_per_seq, int pos,
                                                   int range_begin,
                                                   int range_end, int total,
                                                   int n_ctas) {
  int lo = 0, hi = p.batch;  // b with prefix[b] <= pos < prefix[b + 1]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (prefix[mid] <= pos) lo = mid; else hi = mid;
  }
  UnitInfo ui;
  const int b = lo;
  const int np = (prefix[b + 1] - prefix[b]) / groups_per_seq;
  const int qoff = pos - prefix[b];
  const int gi = qoff / np;              // group within the sequence
  ui.page0 = qoff - gi * np;             // first page of this segment
  ui.b = b;
  ui.g = gi / p.n_rg;
  ui.rg = gi - ui.g * p.n_rg;
  ui.n_pages = min(range_end - pos, np - ui.page0);
  ui.gstart = pos - ui.page0;            // the group's first flat item
  // CTAs that own the group's first and last pages
  ui.f = (int)(((long long)(ui.gstart + 1) * n_ctas - 1) / total);
  ui.l = (int)(((long long)(ui.gstart + np) * n_ctas - 1) / total);
  ui.slot = (pos == range_begin) ? 0 : 1;
  ui.seq_len = __ldg(p.seq_lens + b);
  int np_seq;
  visible_pages(ui.seq_len, p.q_len, p.n_sink, p.window, ui.n_a, ui.b_start,
                np_seq);
  ui.pad0 = ui.pad1 = ui.pad2 = 0;
  ui.valid = 1;
  return ui;
}

// One arrival on the group's ticket; true for the last contributor.  The
// ticket's high word holds the epoch of the launch that last wrote it; a
// ticket of another launch (or never written) counts as zero arrivals.
__device__ __forceinline__ bool take_ticket(const AttnParams &p, int grp,
                                            int n_contrib) {
  unsigned long long *tk = p.tickets + grp;
  unsigned long long seen = __ldcg(tk), want;
  unsigned int before;
  while (true) {
    before = (unsigned int)(seen >> 32) == p.epoch ? (unsigned int)seen : 0u;
    want = ((unsigned long long)p.epoch << 32) | (before + 1u);
    const unsigned long long got = atomicCAS(tk, seen, want);
    if (got == seen) break;
    seen = got;
  }
  return before + 1u == (unsigned int)n_contrib;
}

// The last contributor's merge of a group's partials, by NT consumer
// threads (ctid 0..NT-1, NT/32 warps).  wts: shared scratch of wcap floats;
// row_m / row_w: RB floats each.  Returns false if a barrier timed out.
template <typename T, int D, int RB, int NT>
__device__ __forceinline__ bool merge_partials(
    const AttnParams &p, const UnitInfo &ui, int total, int n_ctas, float *wts,
    int wcap, float *row_m, float *row_w, uint64_t *bar, uint32_t &phase,
    int ctid) {
  constexpr int NW = NT / 32;
  const int lane = ctid & 31, warp = ctid >> 5;
  const int rg = ui.rg, g = ui.g, b = ui.b;
  // contributors are CTAs f..l in order; CTA f's partial sits in its
  // last-segment slot when its slice began before this group
  const int ns = ui.l - ui.f + 1;
  const int f_begin = (int)((long long)ui.f * total / n_ctas);
  const int f_tail = f_begin < ui.gstart ? 1 : 0;
  auto prow_of = [&](int sidx) -> size_t {
    return (size_t)(2 * (ui.f + sidx) + (sidx == 0 ? f_tail : 0));
  };
  const int vrows = min(RB, p.rows - rg * RB);
  // per-row max and weight sum over the splits (warp w: rows w, w+NW, ...)
  for (int r = warp; r < vrows; r += NW) {
    float M = -INFINITY;
    for (int s = lane; s < ns; s += 32)
      M = fmaxf(M, __ldcg(p.part_lse + prow_of(s) * RB + r));
#pragma unroll
    for (int off = 16; off; off >>= 1)
      M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    float W = 0.f;
    if (M != -INFINITY)
      for (int s = lane; s < ns; s += 32)
        W += ex2(__ldcg(p.part_lse + prow_of(s) * RB + r) - M);
#pragma unroll
    for (int off = 16; off; off >>= 1)
      W += __shfl_xor_sync(kFull, W, off);
    if (lane == 0) { row_m[r] = M; row_w[r] = W; }
  }
  if (!consumer_sync(bar, phase, lane)) return false;
  // normalised split weights go to shared memory, CH splits at a time; each
  // thread then sums float4 slices of the partial outputs with independent
  // loads (an empty split has lse2 = -inf and weight 0)
  const int CH = wcap / RB;
  constexpr int NE4 = RB * D / 4;
  constexpr int EPT = (NE4 + NT - 1) / NT;
  const float4 *po4 = reinterpret_cast<const float4 *>(p.part_o);
  float4 acc[EPT];
#pragma unroll
  for (int k = 0; k < EPT; ++k) acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < ns; s0 += CH) {
    const int cn = min(CH, ns - s0);
#pragma unroll 4
    for (int idx = ctid; idx < cn * RB; idx += NT) {
      const int s = s0 + idx / RB, r = idx % RB;
      const float ls = __ldcg(p.part_lse + prow_of(s) * RB + r);
      const float w = r < vrows ? ex2(ls - row_m[r]) / row_w[r] : 0.f;
      wts[idx] = w;
    }
    if (!consumer_sync(bar, phase, lane)) return false;
#pragma unroll
    for (int k = 0; k < EPT; ++k) {
      const int e4 = ctid + k * NT;
      if (e4 >= vrows * (D / 4)) continue;
      const int r = e4 / (D / 4), d4 = e4 % (D / 4);
      float4 a = acc[k];
#pragma unroll 8
      for (int s = 0; s < cn; ++s) {
        const float w = wts[s * RB + r];
        const float4 v = __ldcg(po4 + (prow_of(s0 + s) * RB + r) * (D / 4) + d4);
        a.x = fmaf(w, v.x, a.x);
        a.y = fmaf(w, v.y, a.y);
        a.z = fmaf(w, v.z, a.z);
        a.w = fmaf(w, v.w, a.w);
      }
      acc[k] = a;
    }
    if (!consumer_sync(bar, phase, lane)) return false;
  }
#pragma unroll
  for (int k = 0; k < EPT; ++k) {
    const int e4 = ctid + k * NT;
    if (e4 >= vrows * (D / 4)) continue;
    const int r = e4 / (D / 4), d = (e4 % (D / 4)) * 4;
    const int gr = rg * RB + r;
    const int i = gr / p.group;
    const int h = g * p.group + gr % p.group;
    const size_t row = ((size_t)b * p.q_len + i) * p.num_q_heads + h;
    T *dst = static_cast<T *>(p.out) + row * D + d;
    store_out(dst + 0, acc[k].x);
    store_out(dst + 1, acc[k].y);
    store_out(dst + 2, acc[k].z);
    store_out(dst + 3, acc[k].w);
    if (d == 0) p.lse[row] = (row_m[r] + log2f(row_w[r])) * kLn2;
  }
  return true;
}

// ---- host side ----

// cuTensorMapEncodeTiled, fetched once through the runtime (no -lcuda).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t,
                                  void *, const cuuint64_t *, const cuuint64_t *,
                                  const cuuint32_t *, const cuuint32_t *,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// The cache as a 2-D bf16 tensor [num_blocks*Hkv*16 rows, D], 128-byte
// swizzled boxes of 16 rows x 64 columns.
inline bool make_kv_map(CUtensorMap *map, const void *base, int num_blocks,
                        int hkv, int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {(cuuint64_t)d,
                              (cuuint64_t)num_blocks * hkv * kBlockSize};
  const cuuint64_t strides[1] = {(cuuint64_t)d * 2};
  const cuuint32_t box[2] = {(cuuint32_t)kBoxElems, (cuuint32_t)kBlockSize};
  const cuuint32_t estr[2] = {1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace svp
