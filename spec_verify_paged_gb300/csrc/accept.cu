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
// GB300 design: one thread-block cluster of NC CTAs per sequence (16 when
// the whole batch fits one wave of 16-CTA clusters, else 8); CTA c owns
// vocab slice c of every logit row.
//  * At kernel start each CTA issues 1-D bulk copies of its slice of all
//    2K+1 rows into shared memory (about 72 KB for K = 4 and vocab 32,000
//    with 16-CTA clusters, three CTAs per SM); larger K x vocab cycle through
//    a ring of slots.  The loops stay rolled: the kernel's code has to fit
//    the instruction cache, since every warp runs it once.
//  * Pass 1: per row, a thread keeps an integer reference exponent
//    E >= max(x * log2 e) and the sum of exp2(x * log2 e - E) as a
//    compensated fp32 pair, in one pass: when E grows the sum is rescaled by
//    an exact power of two.  Warps, CTAs and the cluster merge partial sums
//    the same way, so no rounding enters the merges (GB300's fp64 rate is
//    low: fp64 appears only in a few scalar steps).
//  * The CTAs exchange slice statistics through distributed shared memory;
//    every CTA then takes the accept decisions itself (they are scalar).
//  * Pass 2 weighs only the one or two rows the draw needs, from shared
//    memory when they stayed resident.  Thread t owns a contiguous run of
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
constexpr int kMaxRows = 2 * kMaxDraft + 1;
constexpr int kStageBytes = 72000;  // staged logits per CTA (3 CTAs per SM)
constexpr int kMaxSlots = 32;
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

struct AcceptShared {
  ESum warp_s[kAWarps][kMaxRows];  // pass 1: per-warp partials
  ESum slice_s[kMaxRows];          // this CTA's slice (read cluster-wide)
  int row_e[kMaxRows];             // row normaliser 2^row_e * row_s
  float row_s[kMaxRows];
  float mass_hi, mass_lo;          // pass 2: this slice's mass (cluster-wide)
  int last;                        // pass 2: its last token with w > 0
  float red_hi[kAWarps], red_lo[kAWarps];
  int red_i[kAWarps];
  float logit_x[2 * kMaxDraft];    // target / draft logits at the drafts
  int acc[kMaxDraft];
  int tok[kMaxDraft];
  int accept_upto;
  int bad;
  int sel_t;
  uint64_t full[kMaxSlots];        // staging slots' arrival barriers
};

}  // namespace

// Staging: item it = (row it / np, piece it % np) of this CTA's slice, psz
// floats per piece, goes to slot it % slots of the dynamic shared memory.
// With bulk != 0 (16-byte aligned rows) thread 0 moves items with 1-D bulk
// copies, the first `slots` at once; otherwise all threads copy with plain
// loads.  When every row is one piece and every row has a slot, the rows
// stay resident for pass 2.
template <int NC>
__global__ void __launch_bounds__(kAThreads, 3)
    spec_accept_kernel(const AcceptParams p, int chunk, int psz, int np,
                       int slots, int bulk) {
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int b = blockIdx.x / NC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.num_draft, V = p.vocab, R2 = 2 * K + 1;
  __shared__ AcceptShared sh;
  extern __shared__ __align__(16) float xs[];

  const int s0 = min(V, crank * chunk);
  const int n = min(V, s0 + chunk) - s0;  // slice length (may be 0)
  const int items = R2 * np;

  // logit row r of this sequence: r <= K target row r, else draft row r-K-1
  auto row_ptr = [&](int r) -> const float * {
    return r <= K ? p.target_logits + ((size_t)b * (K + 1) + r) * V
                  : p.draft_logits + ((size_t)b * K + (r - K - 1)) * V;
  };
  auto piece_len = [&](int pc) { return min(psz, n - pc * psz); };
  auto issue = [&](int it) {  // thread 0, bulk mode
    const int r = it / np, pc = it - r * np;
    const int len = piece_len(pc);
    const int s = it % slots;
    if (len <= 0) {  // nothing to copy: the slot's phase still completes
      mbar_arrive(&sh.full[s]);
      return;
    }
    mbar_arrive_expect_tx(&sh.full[s], (uint32_t)len * 4u);
    bulk_g2s(xs + (size_t)s * psz, row_ptr(r) + s0 + pc * psz,
             (uint32_t)len * 4u, &sh.full[s]);
  };

  if (tid == 0 && bulk) {
    for (int s = 0; s < slots; ++s) mbar_init(&sh.full[s], 1);
    fence_mbar_init();
    for (int it = 0; it < min(slots, items); ++it) issue(it);
  }
  // the draft tokens, read by the last warp (it has the fewest pieces)
  const bool tok_lane = warp == kAWarps - 1 && lane < K;
  const int xtok = tok_lane ? p.draft_tokens[(size_t)b * K + lane] : 0;
  __syncthreads();  // barriers initialised

  // ---- pass 1: every row's slice sum of exp2(x log2e - E) ----
  // One warp per staged piece, in waves of `slots` pieces: a sweep for the
  // piece's maximum fixes E = ceil(max * log2 e), a second sweep sums
  // exp2(x * log2 e - E); the warp's partial sums per row (warp_s) are
  // merged by exact power-of-two scaling.
  bool ok = true;
  if (lane == 0)
    for (int r = 0; r < R2; ++r) sh.warp_s[warp][r] = ESum{kNoExp, 0.f, 0.f};
  for (int w0 = 0; w0 < items; w0 += slots) {
    const int w1 = min(items, w0 + slots);
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
      const int r = it / np, pc = it - r * np;
      const int len = piece_len(pc);
      if (bulk) ok = mbar_wait(&sh.full[it - w0], (it / slots) & 1) && ok;
      if (len <= 0) continue;
      const float4 *x4 = reinterpret_cast<const float4 *>(xs + (size_t)(it - w0) * psz);
      const int ng = (len + 3) >> 2;
      float m = -INFINITY;
#pragma unroll 4
      for (int g = lane; g < ng; g += 32) {
        const float4 v = x4[g];
        m = fmaxf(m, fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)));
      }
#pragma unroll
      for (int off = 16; off; off >>= 1)
        m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      if (!(m > -INFINITY)) continue;  // nothing but -inf (warp-uniform)
      const int e = (int)ceilf(fminf(m * kL2E, 1.0e9f));
      const float eb = (float)e;
      float hi = 0.f, lo = 0.f;
#pragma unroll 4
      for (int g = lane; g < ng; g += 32) {
        const float4 v = x4[g];
        const float t = (ex2(fmaf(v.x, kL2E, -eb)) + ex2(fmaf(v.y, kL2E, -eb))) +
                        (ex2(fmaf(v.z, kL2E, -eb)) + ex2(fmaf(v.w, kL2E, -eb)));
        kahan_add(hi, lo, t);
      }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float oh = __shfl_xor_sync(0xffffffffu, hi, off);
        const float ol = __shfl_xor_sync(0xffffffffu, lo, off);
        pair_add(hi, lo, oh, ol);
      }
      if (lane == 0)
        sh.warp_s[warp][r] = esum_merge(sh.warp_s[warp][r], ESum{e, hi, lo});
    }
    if (w1 < items) {  // ring: the next wave into the same slots
      __syncthreads();
      if (tid == 0 && bulk)
        for (int it = w1; it < min(items, w1 + slots); ++it) issue(it);
    }
  }
  if (tok_lane) {  // the logits at the drafts (from L2, while others sum)
    const bool good = xtok >= 0 && xtok < V;
    sh.tok[lane] = xtok;
    sh.logit_x[lane] = good ? __ldg(row_ptr(lane) + xtok) : 0.f;
    sh.logit_x[K + lane] = good ? __ldg(row_ptr(K + 1 + lane) + xtok) : 0.f;
  }
  __syncthreads();
  if (tid < R2) {
    ESum s{kNoExp, 0.f, 0.f};
    for (int w = 0; w < kAWarps; ++w) s = esum_merge(s, sh.warp_s[w][tid]);
    sh.slice_s[tid] = s;
  }
  cluster.sync();  // #1: slice statistics visible cluster-wide

  // ---- normalisers and accept decisions, in warp 0 ----
  // lane r < R2 holds row r's normaliser 2^e * S; decision i (lane i < K):
  // u_i <= p_i(x)/q_i(x) = 2^d * S_q / S_p with
  // d = (a - c) log2e - (E_p - E_q) (the same fp32 log2 e as the sums'
  // terms), split as 2^k * 2^frac with a - c and its product with log2 e
  // carried as unevaluated pairs (error-free transformations)
  if (warp == 0) {
    int e = kNoExp;
    float S = 0.f;
    if (lane < R2) {
      ESum o[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        o[c] = cluster.map_shared_rank(&sh, c)->slice_s[lane];
        e = max(e, o[c].e);
      }
      float hi = 0.f, lo = 0.f;
#pragma unroll
      for (int c = 0; c < NC; ++c)
        if (o[c].e != kNoExp) {
          const float f = pow2i(o[c].e - e);  // exact
          pair_add(hi, lo, o[c].hi * f, o[c].lo * f);
        }
      S = hi + lo;
      sh.row_e[lane] = e;
      sh.row_s[lane] = S;
    }
    const int eq = __shfl_sync(0xffffffffu, e, min(lane + K + 1, 31));
    const float Sq = __shfl_sync(0xffffffffu, S, min(lane + K + 1, 31));
    bool bad_i = false, acc_i = true;
    if (lane < K) {
      const int x = sh.tok[lane];
      bad_i = x < 0 || x >= V;
      const float a = sh.logit_x[lane], c = sh.logit_x[K + lane];
      const float s = a - c;
      const float bv = s - a;
      const float err = (a - (s - bv)) + (-c - bv);
      const float xh = s * kL2E;
      const float xl = fmaf(s, kL2E, -xh) + err * kL2E;
      const float kf = floorf(xh);
      const float m = exp2f((xh - kf) + xl) * (Sq / S);
      const float k = kf - ((float)e - (float)eq);
      const float ratio = ldexpf(m, (int)fmaxf(fminf(k, 400.f), -400.f));
      acc_i = p.uniforms[(size_t)b * (K + 1) + lane] <= ratio;  // q(x) = 0: +inf
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
  const float uK = p.uniforms[(size_t)b * (K + 1) + K];

  // ---- pass 2: residual (or bonus) weights, their scan and the draw ----
  // thread t owns slice elements [t*per, t*per + per); per odd, so the
  // threads' walks through shared memory fall in different banks.  Masses
  // and prefix sums are compensated fp32 pairs throughout.
  const int per = ((n + kAThreads - 1) / kAThreads) | 1;
  const int e0 = min(n, tid * per), e1 = min(n, e0 + per);
  const bool resident = np == 1 && slots >= R2;
  bool arrived = false;  // this thread has arrived at the exit barrier
  for (int attempt = 0; attempt < 2 && !bad; ++attempt) {
    const bool residual = (j < K) && attempt == 0;
    const int rt = j;          // target row j (j == K: the bonus row)
    const int rd = K + 1 + j;  // draft row j (residual only)
    const float *xt = resident ? xs + (size_t)rt * psz : row_ptr(rt) + s0;
    const float *xd = resident ? xs + (size_t)rd * psz : row_ptr(rd) + s0;
    const float et = (float)sh.row_e[rt];
    const float it_ = 1.f / sh.row_s[rt];
    const float ed = residual ? (float)sh.row_e[rd] : 0.f;
    const float id_ = residual ? 1.f / sh.row_s[rd] : 0.f;
    // visit(e, w) sees this thread's run in token order; false stops it
    auto for_run = [&](auto visit) {
#pragma unroll 4
      for (int e = e0; e < e1; ++e) {
        float w = ex2(fmaf(xt[e], kL2E, -et)) * it_;
        if (residual) w = fmaxf(w - ex2(fmaf(xd[e], kL2E, -ed)) * id_, 0.f);
        if (!visit(e, w)) return;
      }
    };
    float hi = 0.f, lo = 0.f;  // my run's mass
    int my_last = -1;          // my last slice index with w > 0
    for_run([&](int e, float w) {
      if (w > 0.f) my_last = e;
      kahan_add(hi, lo, w);
      return true;
    });
    // this slice's mass and last positive token; the inclusive warp scan
    // of the run masses is kept for the draw
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
      sh.red_hi[warp] = ih;
      sh.red_lo[warp] = il;
    }
    if (lane == 0) sh.red_i[warp] = lst;
    __syncthreads();
    if (tid == 0) {
      float h2 = 0.f, l2 = 0.f;
      int l = -1;
      for (int w = 0; w < kAWarps; ++w) {
        pair_add(h2, l2, sh.red_hi[w], sh.red_lo[w]);
        l = max(l, sh.red_i[w]);
      }
      sh.mass_hi = h2;
      sh.mass_lo = l2;
      sh.last = l < 0 ? -1 : s0 + l;
    }
    cluster.sync();  // slice masses visible cluster-wide
    // cumulative masses in CTA order: the same operations in every CTA
    float Ph = 0.f, Pl = 0.f, loh = 0.f, lol = 0.f, hih = 0.f, hil = 0.f;
    int last_tok = -1;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
      const AcceptShared *o = cluster.map_shared_rank(&sh, c);
      const float mh = o->mass_hi, ml = o->mass_lo;
      const int lt = o->last;
      if (c == crank) { loh = Ph; lol = Pl; }
      pair_add(Ph, Pl, mh, ml);
      if (c == crank) { hih = Ph; hil = Pl; }
      if (lt >= 0) last_tok = lt;
    }
    if (Ph > 0.f) {
      cluster_arrive();  // no further reads of other CTAs' shared memory
      arrived = true;
      // draw: the smallest x with C(x) > T, T = u_K * W
      float Th = uK * Ph;
      float Tl = fmaf(uK, Ph, -Th) + uK * Pl;
      const bool mine_cta = sh.mass_hi > 0.f && !pair_less(Th, Tl, loh, lol) &&
                            pair_less(Th, Tl, hih, hil);  // CTA-uniform
      if (mine_cta) {
        pair_add(Th, Tl, -loh, -lol);  // T within this slice
        // exclusive prefix of my run: the warp scan, shifted, plus the
        // earlier warps' totals
        float xh = __shfl_up_sync(0xffffffffu, ih, 1);
        float xl = __shfl_up_sync(0xffffffffu, il, 1);
        if (lane == 0) xh = xl = 0.f;
        for (int w = 0; w < warp; ++w) pair_add(xh, xl, sh.red_hi[w], sh.red_lo[w]);
        float nh = xh, nl = xl;  // ... and its inclusive end
        pair_add(nh, nl, hi, lo);
        if (tid == 0) sh.sel_t = -1;
        __syncthreads();
        if (hi > 0.f && !pair_less(Th, Tl, xh, xl) && pair_less(Th, Tl, nh, nl))
          sh.sel_t = tid;
        __syncthreads();
        if (sh.sel_t < 0) {
          // rounding left T outside every run: this slice's last token
          if (tid == 0) p.out_tokens[(size_t)b * (K + 1) + j] = sh.last;
        } else if (tid == sh.sel_t) {
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
          p.out_tokens[(size_t)b * (K + 1) + j] = s0 + found;
        }
      }
      if (!pair_less(Th, Tl, Ph, Pl) && !mine_cta && crank == NC - 1 && tid == 0)
        p.out_tokens[(size_t)b * (K + 1) + j] = last_tok;  // rounded past the end
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
  // no CTA leaves while its shared memory may be read
  if (!arrived) cluster_arrive();
  cluster_wait();
}

namespace {

struct AcceptPlan {
  int chunk, psz, np, slots, bulk;
  size_t smem;
};

template <int NC>
AcceptPlan accept_plan(const AcceptParams &p) {
  AcceptPlan a;
  a.chunk = (p.vocab + NC - 1) / NC;
  a.chunk = (a.chunk + 3) & ~3;  // whole 16-byte groups per slice
  a.psz = std::min(a.chunk, kStageBytes / 4);
  a.np = (a.chunk + a.psz - 1) / a.psz;
  const int items = (2 * p.num_draft + 1) * a.np;
  a.slots = std::min(std::min(items, kMaxSlots), kStageBytes / (a.psz * 4));
  const bool aligned = (reinterpret_cast<uintptr_t>(p.target_logits) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(p.draft_logits) % 16 == 0);
  a.bulk = aligned && (p.vocab % 4 == 0);
  a.smem = (size_t)a.slots * a.psz * sizeof(float);
  return a;
}

template <int NC>
cudaLaunchConfig_t accept_config(const AcceptParams &p, size_t smem,
                                 cudaStream_t stream,
                                 cudaLaunchAttribute *attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(p.batch * NC), 1, 1);
  cfg.blockDim = dim3(kAThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = NC;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

template <int NC>
cudaError_t prepare_kernel() {  // idempotent
  static std::atomic<bool> done{false};
  if (done.load(std::memory_order_acquire)) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(
      spec_accept_kernel<NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
      kStageBytes);
  if (e == cudaSuccess && NC > 8)
    e = cudaFuncSetAttribute(spec_accept_kernel<NC>,
                             cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e == cudaSuccess) done.store(true, std::memory_order_release);
  return e;
}

template <int NC>
cudaError_t launch_nc(const AcceptParams &p, const AcceptPlan &a,
                      cudaStream_t stream) {
  cudaError_t e = prepare_kernel<NC>();
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[1];
  cudaLaunchConfig_t cfg = accept_config<NC>(p, a.smem, stream, attr);
  e = cudaLaunchKernelEx(&cfg, spec_accept_kernel<NC>, p, a.chunk, a.psz, a.np,
                         a.slots, a.bulk);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// How many 16-CTA clusters of the kernel with `smem` bytes of staging are
// resident at once on the current device (0 if none); cached.
int max_clusters16(size_t smem) {
  struct Entry { int dev; size_t smem; int n; };
  static std::mutex mu;
  static Entry cache[16];
  static int used = 0;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < used; ++i)
    if (cache[i].dev == dev && cache[i].smem == smem) return cache[i].n;
  int n = 0;
  if (prepare_kernel<16>() == cudaSuccess) {
    AcceptParams dummy = {};
    dummy.batch = 1;
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = accept_config<16>(dummy, smem, nullptr, attr);
    if (cudaOccupancyMaxActiveClusters(&n, spec_accept_kernel<16>, &cfg) !=
        cudaSuccess)
      n = 0;
  }
  (void)cudaGetLastError();  // a refused query leaves 8-CTA clusters
  if (used < 16) cache[used++] = Entry{dev, smem, n};
  return n;
}

}  // namespace

cudaError_t launch_spec_accept(const AcceptParams &p, cudaStream_t stream) {
  if (p.batch == 0) return cudaSuccess;
  // 16-CTA clusters when the whole batch is resident at once (twice the
  // SMs per sequence, half the slice each); otherwise 8-CTA clusters
  const AcceptPlan a16 = accept_plan<16>(p);
  if (p.batch <= max_clusters16(a16.smem)) return launch_nc<16>(p, a16, stream);
  return launch_nc<8>(p, accept_plan<8>(p), stream);
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
