// accept.cu -- speculative acceptance (rejection sampling) for sm_103a:
// the linear draft (spec_accept) and the draft tree (spec_accept_tree).
//
// Pages: "How speculative decoding doubles LLM speed", step 3 (sampling),
// sections "Absolute mathematical exactness" and "Modern architecture
// variants" (SpecInfer's draft tree); "Speculative decoding: how AI models
// get faster without getting bigger", sections "What speculative decoding
// does" and on real-world adoption (the verifier keeps the longest accepted
// path of the tree).  For one sequence: p = softmax(target row), q =
// softmax(draft row); a draft token x is accepted iff u <= p(x)/q(x); at a
// rejection the replacement is drawn from max(0, p - q) normalised, and if
// every draft passes the bonus is drawn from the last target row.  On a
// tree, a node's children are tried in index order and each rejected child
// replaces p by that normalised residual before the next is tried.
//
// GB300 design: one thread-block cluster of NC CTAs per sequence (16 when
// the whole batch fits one wave of 16-CTA clusters, else 8); CTA c owns
// vocab slice c of every logit row.
//  * At kernel start each CTA issues 1-D bulk copies of its slice of the
//    rows it needs into shared memory (about 72 KB for K = 4 and vocab
//    32,000 with 16-CTA clusters, three CTAs per SM); more rows cycle
//    through a ring of slots.  The loops stay rolled: the kernel's code has
//    to fit the instruction cache, since every warp runs it once.
//  * Pass 1: one warp per staged piece; a sweep for the piece's maximum
//    fixes an integer reference exponent E >= max(x * log2 e), a second
//    sweep sums exp2(x * log2 e - E) as a compensated fp32 pair.  Warps,
//    CTAs and the cluster merge partial sums by exact power-of-two scaling,
//    so no rounding enters the merges (GB300's fp64 rate is low: no fp64 on
//    this path).
//  * The CTAs exchange slice statistics through distributed shared memory;
//    every CTA then takes the accept decisions itself (they are scalar).
//  * Draws and residual masses weigh only the rows they need, from shared
//    memory when those stayed resident.  Thread t owns a contiguous run of
//    its CTA's slice, so (CTA, thread, element) is token order; the CTA
//    holding the crossing of u * W finds the run by a block scan and that
//    thread walks its run once more to find the token.
#include <cooperative_groups.h>

#include <algorithm>
#include <atomic>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "ptx.cuh"
#include "svp.h"
#include "svp_internal.h"

namespace cg = cooperative_groups;

namespace svp {

static __device__ unsigned int g_status_accept;

namespace {

constexpr int kAThreads = 256;
constexpr int kAWarps = kAThreads / 32;
constexpr int kMaxRows = 2 * kMaxDraft + 1;  // also 2 * kMaxNodes - 1
constexpr int kStageBytes = 72000;  // staged logits per CTA (3 CTAs per SM)
constexpr int kMaxSlots = 32;
#ifndef SVP_ACCEPT_PIECES
#define SVP_ACCEPT_PIECES 1
#endif
constexpr int kAcceptPieces = SVP_ACCEPT_PIECES;
constexpr float kL2E = 1.4426950408889634f;
constexpr int kNoExp = INT_MIN / 4;  // reference exponent of an empty sum
static_assert(2 * kMaxNodes - 1 <= kMaxRows, "tree rows exceed the row arrays");
static_assert(kMaxRows <= 127, "staged row indices are kept in bytes");

// A sum of exp2 terms relative to 2^e, as a compensated fp32 pair.
struct ESum {
  int e;
  float hi, lo;
};

// A slice's ESum as other cluster CTAs read it: one 16-byte record, one
// vector load per CTA.
struct alignas(16) ESum4 {
  int e;
  float hi, lo, pad;
};

// Reads of another cluster CTA's shared memory: `mapa` gives the address
// of this CTA's shared word `a` in CTA `rank`; the loads are issued back to
// back and only their uses wait, and each reads a whole record (vector
// loads: the request count, not the bytes, sets their cost).
__device__ __forceinline__ uint32_t cluster_map(uint32_t a, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;"
               : "=r"(r)
               : "r"(a), "r"(rank));
  return r;
}
__device__ __forceinline__ uint4 ld_cluster_v4(uint32_t a) {  // 16-B aligned
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(a)
               : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_cluster_v2f(uint32_t a) {  // 8-B aligned
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0,%1}, [%2];"
               : "=f"(v.x), "=f"(v.y)
               : "r"(a)
               : "memory");
  return v;
}

__device__ __forceinline__ float pow2i(int k) {  // exact 2^k (0 below range)
  return k < -126 ? 0.f : __int_as_float((127 + min(k, 127)) << 23);
}

// (hi, lo) += (bh, bl) for compensated pairs
__device__ __forceinline__ void pair_add(float &hi, float &lo, float bh,
                                         float bl) {
  const float s = hi + bh;
  const float v = s - hi;
  float err = (hi - (s - v)) + (bh - v);
  err += lo + bl;
  hi = s + err;
  lo = err - (hi - s);
}

// (hi, lo) += x, compensated (Kahan): hi + lo tracks the exact sum
__device__ __forceinline__ void kahan_add(float &hi, float &lo, float x) {
  const float y = x + lo;
  const float t = hi + y;
  lo = y - (t - hi);
  hi = t;
}

// a < b for compensated pairs
__device__ __forceinline__ bool pair_less(float ah, float al, float bh,
                                          float bl) {
  return (ah - bh) + (al - bl) < 0.f;
}

// Split cluster barrier: arrive (release: this CTA's earlier accesses to
// other CTAs' shared memory are complete) ... wait (acquire).
__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ ESum esum_merge(ESum a, ESum b) {
  if (a.e == kNoExp) return b;
  if (b.e == kNoExp) return a;
  const int e = max(a.e, b.e);
  const float fa = pow2i(a.e - e), fb = pow2i(b.e - e);  // exact
  ESum r{e, a.hi * fa, a.lo * fa};
  pair_add(r.hi, r.lo, b.hi * fb, b.lo * fb);
  return r;
}

// p(x) / q(x) for logits a (target) and c (draft) and row normalisers
// 2^ep * Sp, 2^eq * Sq: 2^d * Sq / Sp with d = (a - c) sc - (ep - eq),
// sc = log2(e) / temperature (the same fp32 scale as the sums' terms),
// split as 2^k * 2^frac with a - c and its product with sc carried as
// unevaluated pairs (error-free transformations).  q(x) = 0 gives +inf.
__device__ __forceinline__ float accept_ratio(float a, float c, int ep,
                                              float Sp, int eq, float Sq,
                                              float sc) {
  const float s = a - c;
  const float bv = s - a;
  const float err = (a - (s - bv)) + (-c - bv);
  const float xh = s * sc;
  const float xl = fmaf(s, sc, -xh) + err * sc;
  const float kf = floorf(xh);
  const float m = exp2f((xh - kf) + xl) * (Sq / Sp);
  const float k = kf - ((float)ep - (float)eq);
  return ldexpf(m, (int)fmaxf(fminf(k, 400.f), -400.f));
}

// Per-element filters applied to staged logits (4 tokens from `tok`, a
// multiple of 4, of staged row r): none, or the constrained-decoding mask
// (disallowed tokens become -inf).
struct NoFilter {
  static constexpr bool kActive = false;
  __device__ void operator()(int, int, float4 &) const {}
  __device__ bool allows(int, int) const { return true; }
};
struct TokenMask {
  static constexpr bool kActive = true;
  const uint32_t *base;  // [batch, K+1, words] for this call
  int words, K, b;
  // mask row of staged row r: target row r <= K, draft row r - K - 1
  __device__ const uint32_t *row(int r) const {
    const int pos = r <= K ? r : r - K - 1;
    return base + ((size_t)b * (K + 1) + pos) * words;
  }
  __device__ void operator()(int r, int tok, float4 &v) const {
    const uint32_t bits = __ldg(row(r) + (tok >> 5)) >> (tok & 31);
    if (!(bits & 1u)) v.x = -INFINITY;
    if (!(bits & 2u)) v.y = -INFINITY;
    if (!(bits & 4u)) v.z = -INFINITY;
    if (!(bits & 8u)) v.w = -INFINITY;
  }
  __device__ bool allows(int r, int tok) const {
    return (__ldg(row(r) + (tok >> 5)) >> (tok & 31)) & 1u;
  }
};

// Slice statistics of every staged row (read cluster-wide).
struct StageShared {
  ESum warp_s[kAWarps][kMaxRows];  // pass 1: per-warp partials
  ESum4 slice_s[kMaxRows];         // this CTA's slice
  int row_e[kMaxRows];             // row normaliser 2^row_e * row_s
  float row_s[kMaxRows];
  uint64_t full[kMaxSlots];        // staging slots' arrival barriers
};
// 16-byte records that fit in warp_s once pass 1 is over (gather scratch)
constexpr int kGatherCap = (int)(sizeof(ESum) * kAWarps * kMaxRows / 16);

// Exchange state of cluster-wide sums and draws (read cluster-wide).
struct alignas(16) DrawShared {
  float mass_hi, mass_lo;  // draw: this slice's total weight
  int last;                // draw: its last token of positive weight
  float pad0;              // (the four words above: one 16-byte record)
  float zs[2][2];          // cluster sums (hi, lo), by parity of the sum
  float red_hi[kAWarps], red_lo[kAWarps];
  int red_i[kAWarps];
  int sel_t;
};
static_assert(offsetof(DrawShared, mass_hi) == 0 &&
                  offsetof(DrawShared, mass_lo) == 4 &&
                  offsetof(DrawShared, last) == 8 &&
                  offsetof(DrawShared, zs) % 8 == 0,
              "the records other CTAs read with vector loads");

// Staging of this CTA's slice [s0, s0 + n) of rows 0 .. R-1: item
// it = (row it / np, piece it % np), psz floats per piece, goes to slot
// it % slots of the dynamic shared memory xs.  With bulk (16-byte aligned
// rows) thread 0 moves items with 1-D bulk copies, a wave of `slots` at a
// time; otherwise all threads copy with plain loads.  When every item has a
// slot, the rows stay resident after pass 1; with whole-row items the last
// `slots` rows do (the ones a caller stages last).
template <class RowPtr, class Filter = NoFilter, bool ARGMAX = false>
struct SliceStage {
  RowPtr row_ptr;
  int R, s0, n, psz, np, slots, bulk;
  float *xs;
  StageShared *st;
  Filter filter;
  float sc;  // log2(e) / temperature

  __device__ int items() const { return R * np; }
  __device__ int piece_len(int pc) const { return min(psz, n - pc * psz); }
  // every item has its own slot: row r's pieces are consecutive slots
  __device__ bool resident() const { return slots >= items(); }
  // row r of the slice: shared memory while a slot still holds it (every
  // row when all are resident; with whole-row items, a row no later row
  // has replaced), else global memory
  __device__ const float *row(int r) const {
    if (resident()) return xs + (size_t)r * np * psz;
    if (np == 1 && r + slots >= R) return xs + (size_t)(r % slots) * psz;
    return row_ptr(r) + s0;
  }

  __device__ void issue(int it) const {  // thread 0, bulk mode
    const int r = it / np, pc = it - r * np;
    const int len = piece_len(pc);
    const int s = it % slots;
    if (len <= 0) {  // nothing to copy: the slot's phase still completes
      mbar_arrive(&st->full[s]);
      return;
    }
    mbar_arrive_expect_tx(&st->full[s], (uint32_t)len * 4u);
    bulk_g2s(xs + (size_t)s * psz, row_ptr(r) + s0 + pc * psz,
             (uint32_t)len * 4u, &st->full[s]);
  }

  // Thread 0 initialises the slot barriers; the caller synchronises the
  // block before pass1, where each warp issues the copies of the first
  // wave's pieces it will sum (one thread issuing them all was measured
  // slower: the copies start one after another).
  __device__ void begin(int tid) const {
    if (tid == 0 && bulk) {
      for (int s = 0; s < slots; ++s) mbar_init(&st->full[s], 1);
      fence_mbar_init();
    }
  }

  // Pass 1: one warp per staged piece, in waves of `slots` pieces: a sweep
  // for the piece's maximum fixes E = ceil(max * sc), a second sweep sums
  // exp2(x * sc - E); the warp's partial sums per row (warp_s) are merged by
  // exact power-of-two scaling.  A filter rewrites the staged values on the
  // first sweep.  In ARGMAX mode the warp keeps the piece's largest value
  // and its smallest token index instead (as ESum{index, value, 0}).
  // Returns false if a wait timed out.  finish() then forms slice_s.
  __device__ static ESum empty() {
    return ARGMAX ? ESum{INT_MAX, -INFINITY, 0.f} : ESum{kNoExp, 0.f, 0.f};
  }
  __device__ static ESum merge(ESum a, ESum b) {
    if (!ARGMAX) return esum_merge(a, b);
    return (b.hi > a.hi || (b.hi == a.hi && b.e < a.e)) ? b : a;
  }
  // Max and exp-sum of float4 groups [g_lo, g_hi) of staged item `it`
  // (slot pointer x4), merged into this warp's partial of its row.
  __device__ void sum_groups(int it, float4 *x4, int g_lo, int g_hi,
                             int lane, int warp) const {
    const int r = it / np, pc = it - r * np;
    const int tok0 = s0 + pc * psz;  // token of the piece's first element
    if (ARGMAX) {
      float bv = -INFINITY;
      int bi = INT_MAX;
#pragma unroll 4
      for (int g = g_lo + lane; g < g_hi; g += 32) {
        float4 v = x4[g];
        if (Filter::kActive) filter(r, tok0 + 4 * g, v);
        const int t = tok0 + 4 * g;  // first of 4: ties keep the lowest
        if (v.x > bv) { bv = v.x; bi = t; }
        if (v.y > bv) { bv = v.y; bi = t + 1; }
        if (v.z > bv) { bv = v.z; bi = t + 2; }
        if (v.w > bv) { bv = v.w; bi = t + 3; }
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
      }
      if (lane == 0)
        st->warp_s[warp][r] = merge(st->warp_s[warp][r], ESum{bi, bv, 0.f});
      return;
    }
    float m = -INFINITY;
#pragma unroll 4
    for (int g = g_lo + lane; g < g_hi; g += 32) {
      float4 v = x4[g];
      if (Filter::kActive) {
        filter(r, tok0 + 4 * g, v);
        x4[g] = v;  // the filtered row is what later reads see
      }
      m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
    }
#pragma unroll
    for (int off = 16; off; off >>= 1)
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    if (!(m > -INFINITY)) return;  // nothing but -inf (warp-uniform)
    const int e = (int)ceilf(fminf(m * sc, 1.0e9f));
    const float eb = (float)e;
    float hi = 0.f, lo = 0.f;
#pragma unroll 4
    for (int g = g_lo + lane; g < g_hi; g += 32) {
      const float4 v = x4[g];
      const float t =
          (ex2(fmaf(v.x, sc, -eb)) + ex2(fmaf(v.y, sc, -eb))) +
          (ex2(fmaf(v.z, sc, -eb)) + ex2(fmaf(v.w, sc, -eb)));
      kahan_add(hi, lo, t);
    }
#pragma unroll
    for (int off = 16; off; off >>= 1) {
      const float oh = __shfl_xor_sync(0xffffffffu, hi, off);
      const float ol = __shfl_xor_sync(0xffffffffu, lo, off);
      pair_add(hi, lo, oh, ol);
    }
    if (lane == 0)
      st->warp_s[warp][r] = merge(st->warp_s[warp][r], ESum{e, hi, lo});
  }

  __device__ bool pass1(int tid, int lane, int warp) const {
    bool ok = true;
    if (bulk && lane == 0)  // this warp's pieces of the first wave
      for (int it = warp; it < min(slots, items()); it += kAWarps) issue(it);
    if (lane == 0)
      for (int r = 0; r < R; ++r) st->warp_s[warp][r] = empty();
    for (int w0 = 0; w0 < items(); w0 += slots) {
      const int w1 = min(items(), w0 + slots);
      if (!bulk) {  // plain loads into the wave's slots
        for (int it = w0; it < w1; ++it) {
          const int r = it / np, pc = it - r * np;
          const int len = piece_len(pc);
          float *x = xs + (size_t)(it - w0) * psz;
          const float *src = row_ptr(r) + s0 + pc * psz;
          for (int e = tid; e < ((len + 3) & ~3); e += kAThreads)
            x[e] = e < len ? __ldg(src + e) : -INFINITY;
        }
        __syncthreads();
      }
      for (int it = w0 + warp; it < w1; it += kAWarps) {
        const int len = piece_len(it % np);
        if (bulk) ok = mbar_wait(&st->full[it - w0], (it / slots) & 1) && ok;
        if (len > 0)
          sum_groups(it, reinterpret_cast<float4 *>(xs + (size_t)(it - w0) * psz),
                     0, (len + 3) >> 2, lane, warp);
        // bulk ring: only this warp read the slot in this wave, so the
        // slot's piece of the next wave may be copied now (values a filter
        // wrote back are ordered before the copy that overwrites them)
        if (bulk && it + slots < items()) {
          if (Filter::kActive) fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) issue(it + slots);
        }
      }
      // plain loads: every thread refills the slots of the next wave
      if (!bulk && w1 < items()) __syncthreads();
    }
    return ok;
  }

  __device__ void finish(int tid) const {
    __syncthreads();
    if (tid < R) {
      ESum s = empty();
      for (int w = 0; w < kAWarps; ++w) s = merge(s, st->warp_s[w][tid]);
      st->slice_s[tid] = ESum4{s.e, s.hi, s.lo, 0.f};
    }
  }
};

// The whole block, after the cluster barrier that follows finish(): every
// row's normaliser 2^e * S from the NC CTAs' slice statistics, kept in
// row_e / row_s.  The remote records are gathered into `gath` by many
// threads at once (one vector load each, a batch of rows at a time), then
// warp 0, lane r, combines row r from shared memory: one lane issuing all
// NC loads of its row was measured slower.  Ends with a block barrier.
template <int NC>
__device__ void row_normalisers(StageShared &st, uint4 *gath, int gath_cap,
                                int R, int tid, int lane, int warp) {
  const int rows_per = max(1, gath_cap / NC);
  for (int r0 = 0; r0 < R; r0 += rows_per) {
    const int nr = min(rows_per, R - r0);
    for (int i = tid; i < NC * nr; i += kAThreads) {
      const int c = i / nr, r = r0 + (i - c * nr);
      gath[i] = ld_cluster_v4(cluster_map(smem_u32(&st.slice_s[r]), c));
    }
    __syncthreads();
    if (warp == 0 && lane < nr) {
      const int r = r0 + lane;
      int e = kNoExp;
      ESum o[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const uint4 v = gath[c * nr + lane];
        o[c] = ESum{(int)v.x, __uint_as_float(v.y), __uint_as_float(v.z)};
        e = max(e, o[c].e);
      }
      float hi = 0.f, lo = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (o[c].e != kNoExp) {
          const float f = pow2i(o[c].e - e);  // exact
          pair_add(hi, lo, o[c].hi * f, o[c].lo * f);
        }
      st.row_e[r] = e;
      st.row_s[r] = hi + lo;
    }
    __syncthreads();
  }
}

// Sum of weight(e) over every CTA's slice (thread runs [e0, e1)), the same
// compensated pair in every CTA.  One cluster barrier; `parity` alternates
// between consecutive sums so a slot is rewritten only after a barrier.
template <int NC, class Weight>
__device__ void cluster_sum(cg::cluster_group &cluster, DrawShared &ds,
                            uint4 *scratch, const Weight &weight, int e0,
                            int e1, int tid, int lane, int warp, int parity,
                            float &h, float &l) {
  float hi = 0.f, lo = 0.f;
#pragma unroll 4
  for (int e = e0; e < e1; ++e) kahan_add(hi, lo, weight(e));
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    const float oh = __shfl_xor_sync(0xffffffffu, hi, off);
    const float ol = __shfl_xor_sync(0xffffffffu, lo, off);
    pair_add(hi, lo, oh, ol);
  }
  if (lane == 0) {
    ds.red_hi[warp] = hi;
    ds.red_lo[warp] = lo;
  }
  __syncthreads();
  if (tid == 0) {
    float h2 = 0.f, l2 = 0.f;
    for (int w = 0; w < kAWarps; ++w) pair_add(h2, l2, ds.red_hi[w], ds.red_lo[w]);
    ds.zs[parity][0] = h2;
    ds.zs[parity][1] = l2;
  }
  cluster.sync();
  h = 0.f;
  l = 0.f;
  // warp 0 reads the NC pairs (one remote load per lane) for the block
  if (warp == 0 && lane < NC) {
    const float2 z = ld_cluster_v2f(cluster_map(smem_u32(&ds.zs[parity][0]), lane));
    scratch[lane] = make_uint4(__float_as_uint(z.x), __float_as_uint(z.y), 0u, 0u);
  }
  __syncthreads();
#pragma unroll
  for (int c = 0; c < NC; ++c)
    pair_add(h, l, __uint_as_float(scratch[c].x), __uint_as_float(scratch[c].y));
}

// Inverse-CDF draw over weight(e) of every CTA's slice: the smallest token
// whose running sum (token order) exceeds u * total.  Returns false, after a
// cluster barrier, if the total is zero (nothing written); otherwise one
// thread of one CTA writes the token to *dst and this CTA has arrived at
// the exit barrier (no further reads of other CTAs' shared memory).
template <int NC, class Weight>
__device__ bool draw_token(cg::cluster_group &cluster, DrawShared &ds,
                           uint4 *scratch, const Weight &weight, int e0,
                           int e1, float u, int s0, int crank, int tid,
                           int lane, int warp, int32_t *dst) {
  // visit(e, w) sees this thread's run in token order; false stops it
  auto for_run = [&](auto visit) {
#pragma unroll 4
    for (int e = e0; e < e1; ++e)
      if (!visit(e, weight(e))) return;
  };
  float hi = 0.f, lo = 0.f;  // my run's mass
  int my_last = -1;          // my last slice index with w > 0
  for_run([&](int e, float w) {
    if (w > 0.f) my_last = e;
    kahan_add(hi, lo, w);
    return true;
  });
  // this slice's mass and last positive token; the inclusive warp scan of
  // the run masses is kept for the draw
  float ih = hi, il = lo;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float oh = __shfl_up_sync(0xffffffffu, ih, off);
    const float ol = __shfl_up_sync(0xffffffffu, il, off);
    if (lane >= off) pair_add(ih, il, oh, ol);
  }
  int lst = my_last;
#pragma unroll
  for (int off = 16; off; off >>= 1)
    lst = max(lst, __shfl_xor_sync(0xffffffffu, lst, off));
  if (lane == 31) {
    ds.red_hi[warp] = ih;
    ds.red_lo[warp] = il;
  }
  if (lane == 0) ds.red_i[warp] = lst;
  __syncthreads();
  if (tid == 0) {
    float h2 = 0.f, l2 = 0.f;
    int l = -1;
    for (int w = 0; w < kAWarps; ++w) {
      pair_add(h2, l2, ds.red_hi[w], ds.red_lo[w]);
      l = max(l, ds.red_i[w]);
    }
    ds.mass_hi = h2;
    ds.mass_lo = l2;
    ds.last = l < 0 ? -1 : s0 + l;
  }
  cluster.sync();  // slice masses visible cluster-wide
  // cumulative masses in CTA order: the same operations in every CTA
  float Ph = 0.f, Pl = 0.f, loh = 0.f, lol = 0.f, hih = 0.f, hil = 0.f;
  int last_tok = -1;
  // warp 0 reads the NC records (mass_hi, mass_lo, last: one remote load
  // per lane) for the block
  if (warp == 0 && lane < NC)
    scratch[lane] = ld_cluster_v4(cluster_map(smem_u32(&ds), lane));
  __syncthreads();
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    const uint4 v = scratch[c];
    const float mh = __uint_as_float(v.x), ml = __uint_as_float(v.y);
    const int lt = (int)v.z;
    if (c == crank) { loh = Ph; lol = Pl; }
    pair_add(Ph, Pl, mh, ml);
    if (c == crank) { hih = Ph; hil = Pl; }
    if (lt >= 0) last_tok = lt;
  }
  if (!(Ph > 0.f)) {  // cluster-uniform
    cluster.sync();   // nobody rewrites ds while it may still be read
    return false;
  }
  cluster_arrive();
  float Th = u * Ph;  // T = u * W
  float Tl = fmaf(u, Ph, -Th) + u * Pl;
  const bool mine_cta = ds.mass_hi > 0.f && !pair_less(Th, Tl, loh, lol) &&
                        pair_less(Th, Tl, hih, hil);  // CTA-uniform
  if (mine_cta) {
    pair_add(Th, Tl, -loh, -lol);  // T within this slice
    // exclusive prefix of my run: the warp scan, shifted, plus the earlier
    // warps' totals
    float xh = __shfl_up_sync(0xffffffffu, ih, 1);
    float xl = __shfl_up_sync(0xffffffffu, il, 1);
    if (lane == 0) xh = xl = 0.f;
    for (int w = 0; w < warp; ++w) pair_add(xh, xl, ds.red_hi[w], ds.red_lo[w]);
    float nh = xh, nl = xl;  // ... and its inclusive end
    pair_add(nh, nl, hi, lo);
    if (tid == 0) ds.sel_t = -1;
    __syncthreads();
    if (hi > 0.f && !pair_less(Th, Tl, xh, xl) && pair_less(Th, Tl, nh, nl))
      ds.sel_t = tid;
    __syncthreads();
    if (ds.sel_t < 0) {
      // rounding left T outside every run: this slice's last token
      if (tid == 0) *dst = ds.last;
    } else if (tid == ds.sel_t) {
      // the run once more, to the first token whose prefix passes T
      pair_add(Th, Tl, -xh, -xl);  // T within this run
      float h2 = 0.f, l2 = 0.f;
      int found = -1, lastpos = -1;
      for_run([&](int e, float w) {
        if (w > 0.f) lastpos = e;
        kahan_add(h2, l2, w);
        if (w > 0.f && pair_less(Th, Tl, h2, l2)) {
          found = e;
          return false;
        }
        return true;
      });
      if (found < 0) found = lastpos;  // rounding: stay inside this run
      *dst = s0 + found;
    }
  }
  if (!pair_less(Th, Tl, Ph, Pl) && !mine_cta && crank == NC - 1 && tid == 0)
    *dst = last_tok;  // rounded past the end
  return true;
}

struct AcceptShared {
  StageShared st;
  DrawShared ds;
  float logit_x[2 * kMaxDraft];  // target / draft logits at the drafts
  float u[kMaxDraft + 1];        // the sequence's uniforms
  int tok[kMaxDraft];
  int accept_upto;
  int bad;
};

struct TreeShared {
  StageShared st;
  DrawShared ds;
  int tok[kMaxNodes];
  // node and row indices fit a byte (the static shared memory stays small
  // enough for three CTAs per SM)
  int8_t par[kMaxNodes];
  int8_t trow[kMaxNodes];    // staged target row of a node
  int8_t drow[kMaxNodes];    // staged draft row of an inner node, else -1
  int8_t lastc[kMaxNodes];   // a node's last child, else -1
  int8_t rowsrc[kMaxRows];   // node whose target (r < N) or draft row r is
  int8_t path[kMaxNodes];    // accepted nodes
  float lx_t[kMaxNodes];   // target / draft logits of node c's token in the
  float lx_d[kMaxNodes];   // rows of its parent
  float zinv[kMaxNodes];   // 1 / residual mass after each rejected child
  float u[kMaxNodes];      // the sequence's uniforms
  int R;
  int bad;
};

}  // namespace

// ---- linear draft: spec_accept (Filter: NoFilter or TokenMask) ----
template <int NC, class Filter>
__global__ void __launch_bounds__(kAThreads, 3)
    spec_accept_kernel(const AcceptParams p, int chunk, int psz, int np,
                       int slots, int bulk) {
  // launched early (programmatic dependent launch): no global memory is
  // touched before the previous kernel on the stream has completed
  pdl_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int b = blockIdx.x / NC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.num_draft, V = p.vocab, R2 = 2 * K + 1;
  __shared__ AcceptShared sh;
  extern __shared__ __align__(16) float xs[];

  const int s0 = min(V, crank * chunk);
  const int n = min(V, s0 + chunk) - s0;  // slice length (may be 0)

  // logit row r of this sequence: r <= K target row r, else draft row r-K-1
  auto row_ptr = [=](int r) -> const float * {
    return r <= K ? p.target_logits + ((size_t)b * (K + 1) + r) * V
                  : p.draft_logits + ((size_t)b * K + (r - K - 1)) * V;
  };
  Filter filter;
  if constexpr (Filter::kActive) filter = Filter{p.allowed, p.words, K, b};
  const float sc = p.sc;
  const SliceStage<decltype(row_ptr), Filter> stage{
      row_ptr, R2, s0, n, psz, np, slots, bulk, xs, &sh.st, filter, sc};
  stage.begin(tid);
  // the draft tokens and the uniforms, read by the last warp (it has the
  // fewest pieces); they land while pass 1 runs
  const bool tok_lane = warp == kAWarps - 1 && lane < K;
  const int xtok = tok_lane ? p.draft_tokens[(size_t)b * K + lane] : 0;
  const bool u_lane = warp == kAWarps - 1 && lane <= K;
  const float uval = u_lane ? p.uniforms[(size_t)b * (K + 1) + lane] : 0.f;
  __syncthreads();  // barriers initialised

  const bool ok = stage.pass1(tid, lane, warp);
  if (u_lane) sh.u[lane] = uval;
  if (tok_lane) {  // the logits at the drafts (from L2, while others sum)
    const bool good = xtok >= 0 && xtok < V;
    sh.tok[lane] = xtok;
    sh.logit_x[lane] = good ? __ldg(row_ptr(lane) + xtok) : 0.f;
    sh.logit_x[K + lane] = good ? __ldg(row_ptr(K + 1 + lane) + xtok) : 0.f;
  }
  stage.finish(tid);
  cluster.sync();  // #1: slice statistics visible cluster-wide

  // ---- normalisers, then the accept decisions in warp 0 ----
  row_normalisers<NC>(sh.st, reinterpret_cast<uint4 *>(&sh.st.warp_s[0][0]),
                      kGatherCap, R2, tid, lane, warp);
  if (warp == 0) {
    const int e = lane < R2 ? sh.st.row_e[lane] : kNoExp;
    const float S = lane < R2 ? sh.st.row_s[lane] : 0.f;
    const int eq = __shfl_sync(0xffffffffu, e, min(lane + K + 1, 31));
    const float Sq = __shfl_sync(0xffffffffu, S, min(lane + K + 1, 31));
    bool bad_i = false, acc_i = true;
    if (lane < K) {
      const int x = sh.tok[lane];
      bad_i = x < 0 || x >= V;
      const float ratio = accept_ratio(sh.logit_x[lane], sh.logit_x[K + lane],
                                       e, S, eq, Sq, sc);
      acc_i = sh.u[lane] <= ratio;
      // a token the mask excludes has p(x) = 0: rejected
      if (Filter::kActive && !bad_i && !filter.allows(lane, x)) acc_i = false;
    }
    const unsigned bad_mask = __ballot_sync(0xffffffffu, bad_i);
    const unsigned rej_mask = __ballot_sync(0xffffffffu, !acc_i) & ((1u << K) - 1u);
    if (lane == 0) {
      sh.bad = bad_mask != 0;
      sh.accept_upto = rej_mask ? __ffs(rej_mask) - 1 : K;  // first rejection
    }
  }
  __syncthreads();
  const bool bad = sh.bad != 0;
  const int j = bad ? K : sh.accept_upto;
  const float uK = sh.u[K];

  // ---- the draw: residual max(0, p_j - q_j), or the bonus from p_K ----
  // thread t owns slice elements [t*per, t*per + per); per odd, so the
  // threads' walks through shared memory fall in different banks
  // scratch for the records other cluster CTAs expose: the pass-1 partials,
  // consumed by finish()
  uint4 *scratch = reinterpret_cast<uint4 *>(&sh.st.warp_s[0][0]);
  static_assert(sizeof(sh.st.warp_s) >= 16 * sizeof(uint4), "scratch");
  const int per = ((n + kAThreads - 1) / kAThreads) | 1;
  const int e0 = min(n, tid * per), e1 = min(n, e0 + per);
  bool arrived = false;  // this CTA has arrived at the exit barrier
  for (int attempt = 0; attempt < 2 && !bad && !arrived; ++attempt) {
    const bool residual = (j < K) && attempt == 0;
    const int rt = j;          // target row j (j == K: the bonus row)
    const int rd = K + 1 + j;  // draft row j (residual only)
    const float *xt = stage.row(rt);
    const float *xd = stage.row(residual ? rd : rt);
    const float et = (float)sh.st.row_e[rt];
    const float it_ = 1.f / sh.st.row_s[rt];
    const float ed = residual ? (float)sh.st.row_e[rd] : 0.f;
    const float id_ = residual ? 1.f / sh.st.row_s[rd] : 0.f;
    auto weight = [&](int e) {
      float w = ex2(fmaf(xt[e], sc, -et)) * it_;
      if (residual) w = fmaxf(w - ex2(fmaf(xd[e], sc, -ed)) * id_, 0.f);
      if (Filter::kActive && !filter.allows(rt, s0 + e)) w = 0.f;
      return w;
    };
    // a zero residual (impossible in exact arithmetic) falls back to p_j
    arrived = draw_token<NC>(cluster, sh.ds, scratch, weight, e0, e1, uK, s0, crank,
                             tid, lane, warp,
                             p.out_tokens + (size_t)b * (K + 1) + j);
  }

  // ---- accepted drafts, padding and the count (rank 0) ----
  if (crank == 0 && tid == 0) {
    int32_t *out = p.out_tokens + (size_t)b * (K + 1);
    if (bad) {
      for (int k = 0; k <= K; ++k) out[k] = -1;
      p.n_accepted[b] = -1;
      atomicOr(&g_status_accept, (unsigned)SVP_DEV_BAD_TOKEN);
    } else {
      for (int k = 0; k < j; ++k) out[k] = sh.tok[k];
      for (int k = j + 1; k <= K; ++k) out[k] = -1;
      p.n_accepted[b] = j;
    }
  }
  if (!ok && tid == 0) atomicOr(&g_status_accept, (unsigned)SVP_DEV_TIMEOUT);
  // no CTA leaves while its shared memory may be read
  if (!arrived) cluster_arrive();
  cluster_wait();
}

// ---- linear draft, greedy verification (Filter: NoFilter or TokenMask) --
// A draft is accepted iff it is the target row's most likely allowed token
// (smallest index on ties); the first mismatch, or the bonus position,
// emits that token.  Only the K+1 target rows are read.
template <int NC, class Filter>
__global__ void __launch_bounds__(kAThreads, 3)
    spec_accept_greedy_kernel(const AcceptParams p, int chunk, int psz,
                              int np, int slots, int bulk) {
  // launched early (programmatic dependent launch): no global memory is
  // touched before the previous kernel on the stream has completed
  pdl_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int b = blockIdx.x / NC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.num_draft, V = p.vocab, R = K + 1;
  __shared__ AcceptShared sh;
  extern __shared__ __align__(16) float xs[];

  const int s0 = min(V, crank * chunk);
  const int n = min(V, s0 + chunk) - s0;
  auto row_ptr = [=](int r) -> const float * {
    return p.target_logits + ((size_t)b * (K + 1) + r) * V;
  };
  Filter filter;
  if constexpr (Filter::kActive) filter = Filter{p.allowed, p.words, K, b};
  const SliceStage<decltype(row_ptr), Filter, true> stage{
      row_ptr, R, s0, n, psz, np, slots, bulk, xs, &sh.st, filter, kL2E};
  stage.begin(tid);
  const bool tok_lane = warp == kAWarps - 1 && lane < K;
  const int xtok = tok_lane ? p.draft_tokens[(size_t)b * K + lane] : 0;
  __syncthreads();  // barriers initialised
  const bool ok = stage.pass1(tid, lane, warp);
  if (tok_lane) sh.tok[lane] = xtok;
  stage.finish(tid);
  cluster.sync();  // slice maxima visible cluster-wide

  if (warp == 0 && crank == 0) {
    // lane r <= K: the row's best (value, token) over the NC slices
    int best = -1;
    if (lane < R) {
      ESum m{INT_MAX, -INFINITY, 0.f};
      int oe[NC];
      float oh[NC];
      const uint32_t a0 = smem_u32(&sh.st.slice_s[lane]);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        const uint4 v = ld_cluster_v4(cluster_map(a0, c));
        oe[c] = (int)v.x;
        oh[c] = __uint_as_float(v.y);
      }
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (oh[c] > m.hi || (oh[c] == m.hi && oe[c] < m.e)) m = ESum{oe[c], oh[c], 0.f};
      best = m.e == INT_MAX ? -1 : m.e;  // no allowed token: -1
    }
    bool bad_i = false, acc_i = true;
    if (lane < K) {
      const int x = sh.tok[lane];
      bad_i = x < 0 || x >= V;
      acc_i = x == best;
    }
    const unsigned bad_mask = __ballot_sync(0xffffffffu, bad_i);
    const unsigned rej_mask = __ballot_sync(0xffffffffu, !acc_i) & ((1u << K) - 1u);
    const int j = rej_mask ? __ffs(rej_mask) - 1 : K;
    const int best_j = __shfl_sync(0xffffffffu, best, j);
    int32_t *out = p.out_tokens + (size_t)b * (K + 1);
    if (bad_mask) {
      if (lane <= K) out[lane] = -1;
      if (lane == 0) {
        p.n_accepted[b] = -1;
        atomicOr(&g_status_accept, (unsigned)SVP_DEV_BAD_TOKEN);
      }
    } else {
      if (lane < j) out[lane] = sh.tok[lane];
      if (lane == j) out[lane] = best_j;
      if (lane > j && lane <= K) out[lane] = -1;
      if (lane == 0) p.n_accepted[b] = j;
    }
  }
  if (!ok && tid == 0) atomicOr(&g_status_accept, (unsigned)SVP_DEV_TIMEOUT);
  cluster.sync();  // no CTA leaves while its shared memory may be read
}

// ---- draft tree: spec_accept_tree ----
template <int NC>
__global__ void __launch_bounds__(kAThreads, 3)
    spec_accept_tree_kernel(const AcceptTreeParams p, int chunk, int psz,
                            int np, int slots, int bulk) {
  // launched early (programmatic dependent launch): no global memory is
  // touched before the previous kernel on the stream has completed
  pdl_wait();
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int b = blockIdx.x / NC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = p.num_nodes, V = p.vocab;
  __shared__ TreeShared sh;
  extern __shared__ __align__(16) float xs[];

  const int s0 = min(V, crank * chunk);
  const int n = min(V, s0 + chunk) - s0;  // slice length (may be 0)
  const float *tl = p.target_logits + (size_t)b * N * V;
  const float *dl = p.draft_logits + (size_t)b * N * V;

  // the tree: warp 0 reads parents and tokens, checks them, and lists the
  // rows to stage -- the target rows of all nodes, then the draft rows of
  // the inner nodes (the rows their children came from).  Leaves' target
  // rows go first and inner nodes' rows in decreasing node order, so the
  // rows that stay in shared memory after pass 1 (the last ones staged)
  // are those the walk from the root reads first
  if (warp == 0) {
    int pa = -1, tk = -1;
    float uv = 0.f;
    if (lane < N) {
      pa = p.parents[(size_t)b * N + lane];
      tk = p.node_tokens[(size_t)b * N + lane];
      uv = p.uniforms[(size_t)b * N + lane];
    }
    const bool bad_l =
        lane < N && (lane == 0 ? pa != -1
                               : (pa < 0 || pa >= lane || tk < 0 || tk >= V));
    const unsigned bad_mask = __ballot_sync(0xffffffffu, bad_l);
    unsigned inner = 0;  // nodes with a child
    int lastc = -1;      // this lane's node's last child
    for (int c = 1; c < N; ++c) {
      const int pc = __shfl_sync(0xffffffffu, pa, c);
      if (pc >= 0 && pc < c) inner |= 1u << pc;
      if (pc == lane) lastc = c;
    }
    if (lane < N) {
      sh.par[lane] = pa;
      sh.tok[lane] = tk;
      sh.u[lane] = uv;
      sh.lastc[lane] = lastc;
      const bool in = (inner >> lane) & 1u;
      const unsigned below = (1u << lane) - 1u;      // nodes before this one
      const unsigned above = ~((2u << lane) - 1u);   // nodes after it
      const unsigned leaves = ((1u << N) - 1u) & ~inner;
      const int tr = in ? __popc(leaves) + __popc(inner & above)
                        : __popc(leaves & below);
      sh.trow[lane] = tr;
      sh.rowsrc[tr] = lane;
      const int r = N + __popc(inner & above);
      sh.drow[lane] = in ? r : -1;
      if (in) sh.rowsrc[r] = lane;
    }
    if (lane == 0) {
      sh.bad = bad_mask != 0;
      sh.R = N + __popc(inner);
    }
  }
  __syncthreads();
  const int R = sh.R;
  const bool bad = sh.bad != 0;
  const int8_t *rowsrc = sh.rowsrc;
  auto row_ptr = [=](int r) -> const float * {
    return (r < N ? tl : dl) + (size_t)rowsrc[r] * V;
  };
  const SliceStage<decltype(row_ptr)> stage{
      row_ptr, R, s0, n, psz, np, slots, bulk, xs, &sh.st, NoFilter{}, kL2E};
  stage.begin(tid);
  __syncthreads();  // barriers initialised

  const bool ok = stage.pass1(tid, lane, warp);
  // the logits of each node's token in its parent's rows (last warp)
  if (warp == kAWarps - 1 && lane >= 1 && lane < N && !bad) {
    const int pa = sh.par[lane], x = sh.tok[lane];
    sh.lx_t[lane] = __ldg(tl + (size_t)pa * V + x);
    sh.lx_d[lane] = __ldg(dl + (size_t)pa * V + x);
  }
  stage.finish(tid);
  cluster.sync();  // slice statistics visible cluster-wide
  row_normalisers<NC>(sh.st, reinterpret_cast<uint4 *>(&sh.st.warp_s[0][0]),
                      kGatherCap, R, tid, lane, warp);

  // scratch for the records other cluster CTAs expose: the pass-1 partials,
  // consumed by finish()
  uint4 *scratch = reinterpret_cast<uint4 *>(&sh.st.warp_s[0][0]);
  static_assert(sizeof(sh.st.warp_s) >= 16 * sizeof(uint4), "scratch");
  const int per = ((n + kAThreads - 1) / kAThreads) | 1;
  const int e0 = min(n, tid * per), e1 = min(n, e0 + per);
  bool arrived = false;
  int n_acc = 0;
  if (!bad) {
    int cur = 0, k = 0, parity = 0;
    const float *xt = nullptr, *xd = nullptr;
    float et = 0.f, it_ = 0.f, ed = 0.f, id_ = 0.f;
    // r_k of the current node, its q in `q` (meaningful at an inner node):
    // r_0 = p, r_j = max(0, r_{j-1} - q) / Z_j
    auto rk = [&](int e, float &q) {
      float r = ex2(fmaf(xt[e], kL2E, -et)) * it_;
      q = ex2(fmaf(xd[e], kL2E, -ed)) * id_;
      for (int jj = 0; jj < k; ++jj) r = fmaxf(r - q, 0.f) * sh.zinv[jj];
      return r;
    };
    // a node's last child rejected: the draw weighs max(0, r_k - q)
    // unnormalised (the draw takes its own total), so its mass Z, a
    // cluster-wide sum, is not formed
    bool lazy = false;
    for (;;) {
      const int rt = sh.trow[cur], rd = sh.drow[cur];
      xt = stage.row(rt);
      xd = stage.row(rd >= 0 ? rd : rt);
      et = (float)sh.st.row_e[rt];
      it_ = 1.f / sh.st.row_s[rt];
      ed = rd >= 0 ? (float)sh.st.row_e[rd] : 0.f;
      id_ = rd >= 0 ? 1.f / sh.st.row_s[rd] : 0.f;
      k = 0;
      int next = -1;
      for (int c = cur + 1; c < N && rd >= 0; ++c) {  // CTA-uniform
        if (sh.par[c] != cur) continue;
        // r_k(x) / q(x) = max(0, r_{k-1}(x)/q(x) - 1) / Z_k, from p/q
        float ratio = accept_ratio(sh.lx_t[c], sh.lx_d[c], sh.st.row_e[rt],
                                   sh.st.row_s[rt], sh.st.row_e[rd],
                                   sh.st.row_s[rd], kL2E);
        for (int jj = 0; jj < k; ++jj)
          ratio = fmaxf(ratio - 1.f, 0.f) * sh.zinv[jj];
        if (sh.u[c] <= ratio) {
          next = c;
          break;
        }
        // rejected: the residual's mass Z = sum max(0, r_k - q)
        float zh = 1.f, zl = 0.f;
        lazy = c == sh.lastc[cur];
        if (!lazy) {
          cluster_sum<NC>(
              cluster, sh.ds, scratch,
              [&](int e) {
                float q;
                const float r = rk(e, q);
                return fmaxf(r - q, 0.f);
              },
              e0, e1, tid, lane, warp, parity, zh, zl);
          parity ^= 1;
        }
        if (zh > 0.f) {  // else (impossible in exact arithmetic) keep r_k
          __syncthreads();  // zinv[k] is not being read
          if (tid == 0) sh.zinv[k] = 1.f / (zh + zl);
          __syncthreads();
          ++k;
        }
      }
      if (next < 0) break;
      if (tid == 0) sh.path[n_acc] = next;
      ++n_acc;
      cur = next;
    }
    // one token from r_k of the last node (p itself at a leaf); a zero
    // mass by rounding falls back to r_{k-1} (when r_k's mass was not
    // formed: where a zero Z would have left it), then to p
    int32_t *dst = p.out_tokens + (size_t)b * N + n_acc;
    const float u0 = sh.u[0];
    const int tries[3] = {k, lazy ? k - 1 : -1, 0};
    for (int t = 0; t < 3 && !arrived; ++t) {
      if (tries[t] < 0 || (t == 2 && tries[1] == 0)) continue;
      k = tries[t];
      arrived = draw_token<NC>(
          cluster, sh.ds, scratch,
          [&](int e) {
            float q;
            return rk(e, q);
          },
          e0, e1, u0, s0, crank, tid, lane, warp, dst);
    }
  }

  // ---- accepted path, padding and the count (rank 0) ----
  if (crank == 0 && tid == 0) {
    int32_t *out = p.out_tokens + (size_t)b * N;
    int32_t *nodes = p.out_nodes + (size_t)b * N;
    if (bad) {
      for (int k = 0; k < N; ++k) out[k] = nodes[k] = -1;
      p.n_accepted[b] = -1;
      atomicOr(&g_status_accept, (unsigned)SVP_DEV_BAD_TOKEN);
    } else {
      for (int k = 0; k < n_acc; ++k) {
        out[k] = sh.tok[sh.path[k]];
        nodes[k] = sh.path[k];
      }
      for (int k = n_acc; k < N; ++k) nodes[k] = -1;
      for (int k = n_acc + 1; k < N; ++k) out[k] = -1;
      p.n_accepted[b] = n_acc;
    }
  }
  if (!ok && tid == 0) atomicOr(&g_status_accept, (unsigned)SVP_DEV_TIMEOUT);
  if (!arrived) cluster_arrive();
  cluster_wait();
}

namespace {

struct AcceptPlan {
  int chunk, psz, np, slots, bulk;
  size_t smem;
};

template <int NC>
AcceptPlan accept_plan(int vocab, int rows, const float *a, const float *b) {
  AcceptPlan pl;
  pl.chunk = (vocab + NC - 1) / NC;
  pl.chunk = (pl.chunk + 3) & ~3;  // whole 16-byte groups per slice
  // SVP_ACCEPT_PIECES pieces per row slice when they fit the staging
  // budget and the slot count, else whole rows (or the budget).  Whole
  // rows (1) measured fastest: each bulk copy has a fixed cost, and the
  // waits and merges grow with the pieces
  const int want = (((pl.chunk + kAcceptPieces - 1) / kAcceptPieces) + 3) & ~3;
  pl.psz = std::min(rows * kAcceptPieces <= kMaxSlots ? want : pl.chunk,
                    kStageBytes / 4);
  pl.np = (pl.chunk + pl.psz - 1) / pl.psz;
  const int items = rows * pl.np;
  pl.slots = std::min(std::min(items, kMaxSlots), kStageBytes / (pl.psz * 4));
  const bool aligned = (reinterpret_cast<uintptr_t>(a) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(b) % 16 == 0);
  pl.bulk = aligned && (vocab % 4 == 0);
  pl.smem = (size_t)pl.slots * pl.psz * sizeof(float);
  return pl;
}

template <int NC>
cudaLaunchConfig_t accept_config(int batch, size_t smem, cudaStream_t stream,
                                 cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(batch * NC), 1, 1);
  cfg.blockDim = dim3(kAThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cfg;
}

template <class Kern>
cudaError_t prepare_kernel(Kern kern, int nc, std::atomic<bool> &done) {
  if (done.load(std::memory_order_acquire)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kStageBytes);
  if (e == cudaSuccess && nc > 8)
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done.store(true, std::memory_order_release);
  return e;
}

// How many 16-CTA clusters of `kern` with `smem` bytes of staging are
// resident at once on the current device (0 if none); cached.
template <class Kern>
int max_clusters16(Kern kern, std::atomic<bool> &prepared, size_t smem) {
  struct Entry { const void *kern; int dev; size_t smem; int n; };
  static std::mutex mu;
  static Entry cache[32];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].kern == (const void *)kern && cache[i].dev == dev &&
        cache[i].smem == smem)
      return cache[i].n;
  int n = 0;
  if (prepare_kernel(kern, 16, prepared) == cudaSuccess) {
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = accept_config<16>(1, smem, nullptr, attr);
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) n = 0;
  }
  (void)cudaGetLastError();  // a refused query leaves 8-CTA clusters
  if (used < 32) cache[used++] = Entry{(const void *)kern, dev, smem, n};
  return n;
}

std::atomic<bool> g_prep_lin8{false}, g_prep_lin16{false};
std::atomic<bool> g_prep_tree8{false}, g_prep_tree16{false};

template <int NC, class Kern, class Params>
cudaError_t launch_accept(Kern kern, std::atomic<bool> &prepared,
                          const Params &p, int batch, const AcceptPlan &pl,
                          cudaStream_t stream) {
  cudaError_t e = prepare_kernel(kern, NC, prepared);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = accept_config<NC>(batch, pl.smem, stream, attr);
  e = cudaLaunchKernelEx(&cfg, kern, p, pl.chunk, pl.psz, pl.np, pl.slots,
                         pl.bulk);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

// 16-CTA clusters when the whole batch is resident at once (twice the SMs
// per sequence, half the slice each); otherwise 8-CTA clusters.
template <class K16, class K8>
cudaError_t launch_linear(K16 k16, std::atomic<bool> &prep16, K8 k8,
                          std::atomic<bool> &prep8, const AcceptParams &p,
                          int rows) {
  const AcceptPlan a16 =
      accept_plan<16>(p.vocab, rows, p.target_logits, p.draft_logits);
  if (p.batch <= max_clusters16(k16, prep16, a16.smem))
    return launch_accept<16>(k16, prep16, p, p.batch, a16, p.stream);
  return launch_accept<8>(
      k8, prep8, p, p.batch,
      accept_plan<8>(p.vocab, rows, p.target_logits, p.draft_logits), p.stream);
}

std::atomic<bool> g_prep_var[6][2];  // masked / greedy variants, by NC

cudaError_t launch_spec_accept(const AcceptParams &p, cudaStream_t stream) {
  if (p.batch == 0) return cudaSuccess;
  AcceptParams q = p;
  q.stream = stream;
  const int rows = 2 * p.num_draft + 1;
  if (p.greedy) {
    if (p.allowed)
      return launch_linear(spec_accept_greedy_kernel<16, TokenMask>,
                           g_prep_var[0][1],
                           spec_accept_greedy_kernel<8, TokenMask>,
                           g_prep_var[0][0], q, p.num_draft + 1);
    return launch_linear(spec_accept_greedy_kernel<16, NoFilter>,
                         g_prep_var[1][1],
                         spec_accept_greedy_kernel<8, NoFilter>,
                         g_prep_var[1][0], q, p.num_draft + 1);
  }
  if (p.allowed)
    return launch_linear(spec_accept_kernel<16, TokenMask>, g_prep_var[2][1],
                         spec_accept_kernel<8, TokenMask>, g_prep_var[2][0], q,
                         rows);
  return launch_linear(spec_accept_kernel<16, NoFilter>, g_prep_lin16,
                       spec_accept_kernel<8, NoFilter>, g_prep_lin8, q, rows);
}

cudaError_t launch_spec_accept_tree(const AcceptTreeParams &p,
                                    cudaStream_t stream) {
  if (p.batch == 0) return cudaSuccess;
  const int rows = 2 * p.num_nodes - 1;  // the most a tree can need
  const AcceptPlan a16 =
      accept_plan<16>(p.vocab, rows, p.target_logits, p.draft_logits);
  if (p.batch <= max_clusters16(spec_accept_tree_kernel<16>, g_prep_tree16,
                                a16.smem))
    return launch_accept<16>(spec_accept_tree_kernel<16>, g_prep_tree16, p,
                             p.batch, a16, stream);
  return launch_accept<8>(
      spec_accept_tree_kernel<8>, g_prep_tree8, p, p.batch,
      accept_plan<8>(p.vocab, rows, p.target_logits, p.draft_logits), stream);
}

cudaError_t read_status_accept(cudaStream_t s, unsigned *flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status_accept, sizeof v, 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbolAsync(g_status_accept, &zero, sizeof zero, 0,
                              cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  *flags |= v;
  return e;
}

}  // namespace svp
