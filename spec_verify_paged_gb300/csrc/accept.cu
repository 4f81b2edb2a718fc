// accept.cu -- speculative acceptance (rejection sampling) for sm_103a.
//
// Pages: "How speculative decoding doubles LLM speed", step 3 (sampling)
// and section "Absolute mathematical exactness"; "Speculative decoding: how
// AI models get faster without getting bigger", section "What speculative
// decoding does".  For one sequence: p_i = softmax(target row i), q_i =
// softmax(draft row i); draft i is accepted iff u_i <= p_i(x_i)/q_i(x_i);
// at the first rejection j a replacement is drawn from max(0, p_j - q_j)
// normalised, and if all K drafts pass the bonus is drawn from p_K.
//
// GB300 design: one thread-block cluster of NC = 8 CTAs per sequence; CTA c
// owns vocab slice c of every logit row.
//  * Pass 1 streams the slice of all 2K+1 rows through a 4-slot shared
//    memory ring filled by 1-D bulk copies (16 KB sub-chunks), so a CTA
//    needs ~90 KB of shared memory and every sequence of a batch runs in
//    the same wave.  A thread keeps, per row, an integer reference exponent
//    E >= max(x * log2 e) and the sum of exp2(x * log2 e - E) as a
//    compensated fp32 pair; partial sums with different E combine by exact
//    power-of-two scaling, so no rounding enters when warps, CTAs and the
//    cluster merge their sums (GB300's fp64 rate is low: fp64 is used only
//    for O(1) scalar steps).
//  * The CTAs exchange slice statistics through distributed shared memory;
//    every CTA then takes the accept decisions itself (they are scalar).
//  * Pass 2 streams only the one or two rows the draw needs.  Thread t owns
//    a contiguous run of each sub-chunk, so (CTA, sub-chunk, thread, element)
//    is token order; run sums are compensated fp32.  The CTA holding the
//    crossing of u * W finds the run by a block scan and one thread walks
//    it again from L2.
#include <cooperative_groups.h>

#include <climits>
#include <cmath>
#include <cstdint>

#include "ptx.cuh"
#include "svp.h"
#include "svp_internal.h"

namespace cg = cooperative_groups;

namespace svp {

static __device__ unsigned int g_status_accept;

namespace {

constexpr int kNC = 8;            // CTAs per cluster (one cluster per sequence)
constexpr int kAThreads = 256;
constexpr int kAWarps = kAThreads / 32;
constexpr int kMaxRows = 2 * kMaxDraft + 1;
constexpr int kSub = 4096;        // floats per staged sub-chunk (16 KB)
constexpr int kRingA = 4;         // sub-chunks in flight
constexpr int kMaxSub = 10;       // sub-chunks of a slice (vocab <= 8 x 40960)
constexpr int kPer = kSub / kAThreads;  // elements per thread per sub-chunk
constexpr float kL2E = 1.4426950408889634f;
constexpr int kNoExp = INT_MIN / 4;  // reference exponent of an empty sum

// A sum of exp2 terms relative to 2^e, as a compensated fp32 pair.
struct ESum {
  int e;
  float hi, lo;
};

__device__ __forceinline__ float pow2i(int k) {  // exact 2^k (0 below range)
  return k < -126 ? 0.f : __int_as_float((127 + min(k, 127)) << 23);
}

// a + b for compensated pairs (both relative to the same exponent)
__device__ __forceinline__ void pair_add(float &hi, float &lo, float bh,
                                         float bl) {
  const float s = hi + bh;
  const float v = s - hi;
  float err = (hi - (s - v)) + (bh - v);
  err += lo + bl;
  hi = s + err;
  lo = err - (hi - s);
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

__device__ __forceinline__ ESum warp_esum(ESum v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) {
    ESum o;
    o.e = __shfl_xor_sync(0xffffffffu, v.e, off);
    o.hi = __shfl_xor_sync(0xffffffffu, v.hi, off);
    o.lo = __shfl_xor_sync(0xffffffffu, v.lo, off);
    v = esum_merge(v, o);
  }
  return v;
}

struct AcceptShared {
  alignas(128) float ring[kRingA][kSub];
  float part_hi[kMaxSub][kAThreads];  // pass 2: run sums per sub-chunk
  float part_lo[kMaxSub][kAThreads];
  ESum warp_s[kAWarps][kMaxRows];     // pass 1: per-warp partials
  ESum slice_s[kMaxRows];             // this CTA's slice (read cluster-wide)
  int row_e[kMaxRows];                // row normaliser 2^row_e * row_s
  double row_s[kMaxRows];
  double mass;                        // pass 2: this slice's mass (cluster-wide)
  int last;                           // pass 2: its last token with w > 0
  float red_hi[kAWarps], red_lo[kAWarps];
  int red_i[kAWarps];
  int acc[kMaxDraft];
  int tok[kMaxDraft];
  int accept_upto;
  int bad;
  int sel_ks, sel_t;
  double sel_excl;
  uint64_t full[kRingA];
};

}  // namespace

__global__ void __launch_bounds__(kAThreads)
    spec_accept_kernel(const AcceptParams p, int chunk, int staged) {
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int b = blockIdx.x / kNC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.num_draft, V = p.vocab, R2 = 2 * K + 1;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  AcceptShared &sh = *reinterpret_cast<AcceptShared *>(smem_raw);

  const int s0 = min(V, crank * chunk);
  const int n = min(V, s0 + chunk) - s0;  // slice length (may be 0)
  const int nsub = (n + kSub - 1) / kSub;

  // logit row r of this sequence: r <= K target row r, else draft row r-K-1
  auto row_ptr = [&](int r) -> const float * {
    return r <= K ? p.target_logits + ((size_t)b * (K + 1) + r) * V
                  : p.draft_logits + ((size_t)b * K + (r - K - 1)) * V;
  };
  auto sub_len = [&](int ks) { return min(kSub, n - ks * kSub); };

  if (tid == 0) {
    for (int s = 0; s < kRingA; ++s) mbar_init(&sh.full[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool ok = true;
  // Streams items it = 0 .. count-1 (item -> (row, sub-chunk) by item_of)
  // through the ring; body(it, src, len) reads the sub-chunk at src.
  // Unstaged (unaligned rows): src points into global memory.
  uint32_t ring_phase_base = 0;  // items streamed before this pass
  auto stream_items = [&](int count, auto item_of, auto body) {
    if (staged && tid == 0) {
      for (int it = 0; it < min(count, kRingA); ++it) {
        int r, ks;
        item_of(it, r, ks);
        const int slot = (int)((ring_phase_base + it) % kRingA);
        const uint32_t bytes = (uint32_t)sub_len(ks) * 4u;
        mbar_arrive_expect_tx(&sh.full[slot], bytes);
        bulk_g2s(sh.ring[slot], row_ptr(r) + s0 + ks * kSub, bytes,
                 &sh.full[slot]);
      }
    }
    for (int it = 0; it < count; ++it) {
      int r, ks;
      item_of(it, r, ks);
      const uint32_t g = ring_phase_base + it;
      const int slot = (int)(g % kRingA);
      const float *src;
      if (staged) {
        ok = mbar_wait(&sh.full[slot], (g / kRingA) & 1) && ok;
        src = sh.ring[slot];
      } else {
        src = row_ptr(r) + s0 + ks * kSub;
      }
      body(it, r, ks, src, sub_len(ks));
      __syncthreads();  // everyone is done with the slot
      if (staged && tid == 0 && it + kRingA < count) {
        int r2, k2;
        item_of(it + kRingA, r2, k2);
        const uint32_t bytes = (uint32_t)sub_len(k2) * 4u;
        mbar_arrive_expect_tx(&sh.full[slot], bytes);
        bulk_g2s(sh.ring[slot], row_ptr(r2) + s0 + k2 * kSub, bytes,
                 &sh.full[slot]);
      }
    }
    ring_phase_base += (uint32_t)count;
  };

  // ---- pass 1: every row's slice sum of exp2(x log2e - E) ----
  {
    ESum cur{kNoExp, 0.f, 0.f};
    stream_items(
        R2 * nsub,
        [&](int it, int &r, int &ks) { r = it / nsub; ks = it - r * nsub; },
        [&](int, int r, int ks, const float *src, int len) {
          float x[kPer];
          float lmax = -INFINITY;
#pragma unroll
          for (int k = 0; k < kPer; ++k) {
            const int e = tid + k * kAThreads;
            x[k] = e < len ? src[e] : -INFINITY;
            lmax = fmaxf(lmax, x[k]);
          }
          if (lmax != -INFINITY) {
            const int e_new = max(cur.e, (int)ceilf(lmax * kL2E));
            if (cur.e != kNoExp && e_new != cur.e) {
              const float f = pow2i(cur.e - e_new);
              cur.hi *= f;
              cur.lo *= f;
            }
            cur.e = e_new;
            const float eb = (float)e_new;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {  // Kahan
              const float y = ex2(fmaf(x[k], kL2E, -eb)) - cur.lo;
              const float t = cur.hi + y;
              cur.lo = (t - cur.hi) - y;
              cur.hi = t;
            }
          }
          if (ks == nsub - 1) {  // the row's slice is complete
            const ESum w = warp_esum(cur);
            if (lane == 0) sh.warp_s[warp][r] = w;
            cur = ESum{kNoExp, 0.f, 0.f};
          }
        });
  }
  if (tid < R2) {
    ESum s{kNoExp, 0.f, 0.f};
    if (nsub > 0)
      for (int w = 0; w < kAWarps; ++w) s = esum_merge(s, sh.warp_s[w][tid]);
    sh.slice_s[tid] = s;
  }
  if (tid < K) sh.tok[tid] = p.draft_tokens[(size_t)b * K + tid];
  cluster.sync();  // #1: slice statistics visible cluster-wide

  // ---- the rows' normalisers (identical in every CTA) ----
  if (tid < R2) {
    ESum o[kNC];
    int e = kNoExp;
    for (int c = 0; c < kNC; ++c) {
      o[c] = cluster.map_shared_rank(&sh, c)->slice_s[tid];
      e = max(e, o[c].e);
    }
    double z = 0.0;
    for (int c = 0; c < kNC; ++c)
      if (o[c].e != kNoExp)
        z += ldexp((double)o[c].hi + (double)o[c].lo, o[c].e - e);
    sh.row_e[tid] = e;
    sh.row_s[tid] = z;
  }
  if (tid == 0) {
    int bad = 0;
    for (int i = 0; i < K; ++i) bad |= (sh.tok[i] < 0 || sh.tok[i] >= V);
    sh.bad = bad;
  }
  __syncthreads();
  const bool bad = sh.bad != 0;

  // ---- accept decisions: u_i <= p_i(x)/q_i(x) ----
  // p_i(x) = 2^(a log2e - E_p) / S_p, q_i(x) = 2^(c log2e - E_q) / S_q, with
  // the same fp32 log2 e as the sums' terms
  if (!bad && tid < K) {
    const int x = sh.tok[tid];
    const double a = (double)__ldg(row_ptr(tid) + x);
    const double c = (double)__ldg(row_ptr(K + 1 + tid) + x);
    const int ep = sh.row_e[tid], eq = sh.row_e[K + 1 + tid];
    const double ratio = exp2((a - c) * (double)kL2E - (double)(ep - eq)) *
                         (sh.row_s[K + 1 + tid] / sh.row_s[tid]);
    const double u = (double)p.uniforms[(size_t)b * (K + 1) + tid];
    sh.acc[tid] = (u <= ratio);  // q(x) = 0 gives ratio +inf: accepted
  }
  __syncthreads();
  if (tid == 0) {
    int j = K;
    if (!bad)
      for (int i = 0; i < K; ++i)
        if (!sh.acc[i]) { j = i; break; }
    sh.accept_upto = j;
  }
  __syncthreads();
  const int j = sh.accept_upto;
  const double uK = (double)p.uniforms[(size_t)b * (K + 1) + K];

  // ---- pass 2: residual (or bonus) weights, their scan and the draw ----
  // thread t owns elements [t*per, t*per + per) of a sub-chunk; `per` odd
  // so the threads' walks through shared memory do not collide on banks
  for (int attempt = 0; attempt < 2 && !bad; ++attempt) {
    const bool residual = (j < K) && attempt == 0;
    const int rt = j;              // target row j (j == K: the bonus row)
    const int rd = K + 1 + j;      // draft row j (residual only)
    const int nrow = residual ? 2 : 1;
    const float et = (float)sh.row_e[rt];
    const float it_ = (float)(1.0 / sh.row_s[rt]);
    const float ed = residual ? (float)sh.row_e[rd] : 0.f;
    const float id_ = residual ? (float)(1.0 / sh.row_s[rd]) : 0.f;
    auto weight = [&](float xt, float xd) -> float {
      const float pt = ex2(fmaf(xt, kL2E, -et)) * it_;
      if (!residual) return pt;
      const float qd = ex2(fmaf(xd, kL2E, -ed)) * id_;
      return fmaxf(pt - qd, 0.f);
    };
    int my_last = -1;       // my last token index with w > 0 (slice-relative)
    float xt_run[kPer + 1];  // the target row's run while its draft arrives
    stream_items(
        nrow * nsub,
        [&](int it, int &r, int &ks) {
          ks = it / nrow;
          r = (nrow == 2 && (it % 2) == 1) ? rd : rt;
        },
        [&](int it, int r, int ks, const float *src, int len) {
          int per = (len + kAThreads - 1) / kAThreads;
          per |= 1;
          const int e0 = min(len, tid * per), e1 = min(len, e0 + per);
          if (nrow == 2 && r == rt) {  // keep the target run, wait for draft
            for (int e = e0; e < e1; ++e) xt_run[e - e0] = src[e];
            return;
          }
          float hi = 0.f, lo = 0.f;
          for (int e = e0; e < e1; ++e) {
            const float w = nrow == 2 ? weight(xt_run[e - e0], src[e])
                                      : weight(src[e], 0.f);
            if (w > 0.f) my_last = ks * kSub + e;
            const float y = w - lo;
            const float t = hi + y;
            lo = (t - hi) - y;
            hi = t;
          }
          sh.part_hi[ks][tid] = hi;
          sh.part_lo[ks][tid] = lo;
          (void)it;
        });
    // this slice's mass and last positive token
    {
      float hi = 0.f, lo = 0.f;
      for (int ks = 0; ks < nsub; ++ks)
        pair_add(hi, lo, sh.part_hi[ks][tid], sh.part_lo[ks][tid]);
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, hi, off);
        const float ol = __shfl_xor_sync(0xffffffffu, lo, off);
        pair_add(hi, lo, oh, ol);
      }
      int lst = my_last;
#pragma unroll
      for (int off = 16; off; off >>= 1)
        lst = max(lst, __shfl_xor_sync(0xffffffffu, lst, off));
      if (lane == 0) {
        sh.red_hi[warp] = hi;
        sh.red_lo[warp] = lo;
        sh.red_i[warp] = lst;
      }
      __syncthreads();
      if (tid == 0) {
        float h2 = 0.f, l2 = 0.f;
        int l = -1;
        for (int w = 0; w < kAWarps; ++w) {
          pair_add(h2, l2, sh.red_hi[w], sh.red_lo[w]);
          l = max(l, sh.red_i[w]);
        }
        sh.mass = (double)h2 + (double)l2;
        sh.last = l < 0 ? -1 : s0 + l;
      }
    }
    cluster.sync();  // slice masses visible cluster-wide
    double P = 0.0, Pmine = 0.0;
    int last_tok = -1;
    for (int c = 0; c < kNC; ++c) {
      const AcceptShared *o = cluster.map_shared_rank(&sh, c);
      if (c == crank) Pmine = P;
      P += o->mass;
      if (o->last >= 0) last_tok = o->last;
    }
    const double W = P;  // identical in every CTA of the cluster
    if (W > 0.0) {
      const double T = uK * W;  // draw: smallest x with C(x) > T
      const double Tl = T - Pmine;
      if (sh.mass > 0.0 && Tl >= 0.0 && Tl < sh.mass) {
        // the run holding the crossing: scan the (sub-chunk, thread) sums
        // in token order, compensated pairs
        if (tid == 0) sh.sel_ks = -1;
        __syncthreads();
        float bh = 0.f, bl = 0.f;  // mass of the earlier sub-chunks
        for (int ks = 0; ks < nsub; ++ks) {
          const float mh = sh.part_hi[ks][tid], ml = sh.part_lo[ks][tid];
          float ih = mh, il = ml;  // inclusive warp scan
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const float oh = __shfl_up_sync(0xffffffffu, ih, off);
            const float ol = __shfl_up_sync(0xffffffffu, il, off);
            if (lane >= off) pair_add(ih, il, oh, ol);
          }
          if (lane == 31) { sh.red_hi[warp] = ih; sh.red_lo[warp] = il; }
          __syncthreads();
          float xh = bh, xl = bl;  // my run's exclusive prefix
          float th = bh, tl = bl;  // the next sub-chunk's base
          for (int w = 0; w < kAWarps; ++w) {
            if (w < warp) pair_add(xh, xl, sh.red_hi[w], sh.red_lo[w]);
            pair_add(th, tl, sh.red_hi[w], sh.red_lo[w]);
          }
          pair_add(xh, xl, ih, il);
          pair_add(xh, xl, -mh, -ml);
          const double excl = (double)xh + (double)xl;
          const double mine = (double)mh + (double)ml;
          if (mine > 0.0 && excl <= Tl && Tl < excl + mine) {
            sh.sel_ks = ks;
            sh.sel_t = tid;
            sh.sel_excl = excl;
          }
          bh = th;
          bl = tl;
          __syncthreads();  // red_* are rewritten next; sel_* visible
        }
        if (sh.sel_ks < 0) {
          // rounding left Tl outside every run: this slice's last token
          if (tid == 0) p.out_tokens[(size_t)b * (K + 1) + j] = sh.last;
        } else if (tid == sh.sel_t) {
          // walk the run again (from L2) to the first token past Tl
          const int ks = sh.sel_ks;
          const int len = sub_len(ks);
          int per = (len + kAThreads - 1) / kAThreads;
          per |= 1;
          const int e0 = min(len, tid * per), e1 = min(len, e0 + per);
          const double excl = sh.sel_excl;
          const float *pt = row_ptr(rt) + s0 + ks * kSub;
          const float *pd = residual ? row_ptr(rd) + s0 + ks * kSub : pt;
          float h2 = 0.f, l2 = 0.f;
          int found = -1, lastpos = -1;
          for (int e = e0; e < e1; ++e) {
            const float w = residual ? weight(__ldg(pt + e), __ldg(pd + e))
                                     : weight(__ldg(pt + e), 0.f);
            if (w > 0.f) lastpos = e;
            const float y = w - l2;
            const float t = h2 + y;
            l2 = (t - h2) - y;
            h2 = t;
            if (w > 0.f && excl + ((double)h2 - (double)l2) > Tl) {
              found = e;
              break;
            }
          }
          if (found < 0) found = lastpos;  // rounding: stay inside this run
          p.out_tokens[(size_t)b * (K + 1) + j] = s0 + ks * kSub + found;
        }
      }
      if (T >= W && crank == kNC - 1 && tid == 0)  // rounded past the end
        p.out_tokens[(size_t)b * (K + 1) + j] = last_tok;
      break;
    }
    // zero residual mass (impossible in exact arithmetic): draw from p_j
    cluster.sync();
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
  cluster.sync();  // no CTA leaves while its shared memory may be read
}

static int accept_chunk(int vocab) {
  int chunk = (vocab + kNC - 1) / kNC;
  return (chunk + 3) & ~3;  // 16-byte multiple
}

cudaError_t launch_spec_accept(const AcceptParams &p, cudaStream_t stream) {
  if (p.batch == 0) return cudaSuccess;
  const int chunk = accept_chunk(p.vocab);
  if (chunk > kMaxSub * kSub) return cudaErrorInvalidValue;
  const bool aligned = (reinterpret_cast<uintptr_t>(p.target_logits) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(p.draft_logits) % 16 == 0);
  const int staged = aligned && (p.vocab % 4 == 0);
  const size_t smem = sizeof(AcceptShared);
  cudaError_t e = cudaFuncSetAttribute(
      spec_accept_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
      (int)smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.batch * kNC), 1, 1);
  cfg.blockDim = dim3(kAThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kNC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, spec_accept_kernel, p, chunk, staged);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
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
