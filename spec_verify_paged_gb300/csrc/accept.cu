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
// GB300 design: one thread-block cluster of NC = 8 CTAs per sequence.  CTA c
// owns vocab slice c of every one of the 2K+1 logit rows and stages all of
// them into its shared memory with 1-D bulk copies (one mbarrier, every
// byte in flight at once).  Softmax normalisers: per-slice max, then the sum
// of exp2 terms with compensated (Kahan) fp32 accumulation per thread,
// combined in fp64.  The CTAs exchange slice statistics and CDF slice sums
// through distributed shared memory (no global workspace, one launch).  The
// accept decisions are taken redundantly by every CTA (they are scalar);
// the CTA whose slice holds the inverse-CDF crossing resolves the token.
#include <cooperative_groups.h>

#include <cmath>
#include <cstdint>

#include "ptx.cuh"
#include "svp.h"
#include "svp_internal.h"

namespace cg = cooperative_groups;

namespace svp {

static __device__ unsigned int g_status_accept;

constexpr int kNC = 8;            // CTAs per cluster (one cluster per sequence)
constexpr int kAThreads = 256;
constexpr int kAWarps = kAThreads / 32;
constexpr int kMaxRows = 2 * kMaxDraft + 1;
constexpr size_t kMaxCacheBytes = 200 * 1024;
constexpr float kL2E = 1.4426950408889634f;

struct AcceptShared {
  float slice_m[kMaxRows];        // per-row max of this slice
  double slice_z[kMaxRows];       // per-row sum exp(x - slice_m) of this slice
  float row_m[kMaxRows];          // per-row global max
  double row_z[kMaxRows];         // per-row global normaliser
  double w_sum;                   // this slice's residual mass
  int w_last;                     // last index of this slice with w > 0
  double red_d[kAWarps][kMaxRows];
  float red_f[kAWarps][kMaxRows];
  double scan[kAWarps];
  int red_i[kAWarps];
  int sel[kAWarps];
  int acc[kMaxDraft];
  int tok[kMaxDraft];
  int accept_upto;                // first rejected position, or K
  int bad;
  uint64_t bar;
};

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  return v;
}
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int off = 16; off; off >>= 1)
    v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

__global__ void __launch_bounds__(kAThreads)
    spec_accept_kernel(const AcceptParams p, int chunk, int cached) {
  cg::cluster_group cluster = cg::this_cluster();
  const int crank = (int)cluster.block_rank();
  const int b = blockIdx.x / kNC;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = p.num_draft, V = p.vocab, R2 = 2 * K + 1;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  AcceptShared &sh = *reinterpret_cast<AcceptShared *>(smem_raw);
  float *cache = reinterpret_cast<float *>(smem_raw + ((sizeof(AcceptShared) + 127) / 128) * 128);
  float *wbuf = cached ? nullptr : cache;  // uncached: cache region holds w

  const int s0 = min(V, crank * chunk);
  const int n = min(V, s0 + chunk) - s0;   // slice length (may be 0)

  // logit row r of this sequence: r <= K target row r, else draft row r-K-1
  auto row_ptr = [&](int r) -> const float * {
    return r <= K ? p.target_logits + ((size_t)b * (K + 1) + r) * V
                  : p.draft_logits + ((size_t)b * K + (r - K - 1)) * V;
  };

  // ---- stage the slices (bulk copies, all in flight together) ----
  if (tid == 0) {
    mbar_init(&sh.bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  bool staged = true;
  if (cached) {
    if (tid == 0) {
      const uint32_t bytes = (uint32_t)n * 4u;
      mbar_arrive_expect_tx(&sh.bar, bytes * (uint32_t)R2);
      if (bytes)
        for (int r = 0; r < R2; ++r)
          bulk_g2s(cache + (size_t)r * chunk, row_ptr(r) + s0, bytes, &sh.bar);
    }
    staged = mbar_wait(&sh.bar, 0);
    if (!staged && tid == 0) atomicOr(&g_status_accept, (unsigned)SVP_DEV_TIMEOUT);
  }
  auto val = [&](int r, int e) -> float {
    return cached ? cache[(size_t)r * chunk + e] : __ldg(row_ptr(r) + s0 + e);
  };

  // ---- phase 1: slice max and sum of exponentials for every row ----
  for (int r = 0; r < R2; ++r) {
    float mx = -INFINITY;
    for (int e = tid; e < n; e += kAThreads) mx = fmaxf(mx, val(r, e));
    mx = warp_max_f(mx);
    if (lane == 0) sh.red_f[warp][r] = mx;
  }
  __syncthreads();
  if (tid < R2) {
    float mx = -INFINITY;
    for (int w = 0; w < kAWarps; ++w) mx = fmaxf(mx, sh.red_f[w][tid]);
    sh.slice_m[tid] = mx;
  }
  __syncthreads();
  for (int r = 0; r < R2; ++r) {
    const float mb = sh.slice_m[r] * kL2E;
    float hi = 0.f, lo = 0.f;  // Kahan
    for (int e = tid; e < n; e += kAThreads) {
      const float y = ex2(fmaf(val(r, e), kL2E, -mb)) - lo;
      const float t = hi + y;
      lo = (t - hi) - y;
      hi = t;
    }
    const double d = warp_sum_d((double)hi - (double)lo);
    if (lane == 0) sh.red_d[warp][r] = d;
  }
  __syncthreads();
  if (tid < R2) {
    double z = 0.0;
    for (int w = 0; w < kAWarps; ++w) z += sh.red_d[w][tid];
    sh.slice_z[tid] = z;
  }
  // draft tokens (validated by every CTA alike)
  if (tid < K) {
    const int x = p.draft_tokens[(size_t)b * K + tid];
    sh.tok[tid] = x;
  }
  cluster.sync();  // #1: slice statistics visible cluster-wide

  // ---- combine the slices: row max and normaliser ----
  if (tid < R2) {
    float M = -INFINITY;
    for (int c = 0; c < kNC; ++c) {
      const AcceptShared *o = cluster.map_shared_rank(&sh, c);
      M = fmaxf(M, o->slice_m[tid]);
    }
    double Z = 0.0;
    for (int c = 0; c < kNC; ++c) {
      const AcceptShared *o = cluster.map_shared_rank(&sh, c);
      const float mc = o->slice_m[tid];
      if (mc != -INFINITY) Z += o->slice_z[tid] * (double)ex2((mc - M) * kL2E);
    }
    sh.row_m[tid] = M;
    sh.row_z[tid] = Z;
  }
  if (tid == 0) {
    int bad = 0;
    for (int i = 0; i < K; ++i) bad |= (sh.tok[i] < 0 || sh.tok[i] >= V);
    sh.bad = bad;
  }
  __syncthreads();
  const bool bad = sh.bad != 0;

  // ---- accept decisions: u_i <= p_i(x)/q_i(x) ----
  if (!bad && tid < K) {
    const int x = sh.tok[tid];
    const double a = (double)__ldg(row_ptr(tid) + x) - (double)sh.row_m[tid];
    const double c = (double)__ldg(row_ptr(K + 1 + tid) + x) -
                     (double)sh.row_m[K + 1 + tid];
    const double ratio = (double)expf((float)(a - c)) *
                         (sh.row_z[K + 1 + tid] / sh.row_z[tid]);
    const double u = (double)p.uniforms[(size_t)b * (K + 1) + tid];
    sh.acc[tid] = (u <= ratio);
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

  // ---- residual (or bonus) weights of this slice and their scan ----
  // One thread owns a contiguous run of `per` entries (odd stride: no bank
  // conflicts when the threads walk their runs in shared memory).
  int per = (n + kAThreads - 1) / kAThreads;
  per |= 1;
  for (int attempt = 0; attempt < 2 && !bad; ++attempt) {
    const bool residual = (j < K) && attempt == 0;
    const int rt = j;              // target row j (j == K: the bonus row)
    const int rd = K + 1 + j;      // draft row j (residual only)
    const float mt = sh.row_m[rt] * kL2E;
    const float izt = (float)(1.0 / sh.row_z[rt]);
    const float md = residual ? sh.row_m[rd] * kL2E : 0.f;
    const float izd = residual ? (float)(1.0 / sh.row_z[rd]) : 0.f;
    // w overwrites the draft row's staged slice (the target row stays intact
    // for a fallback attempt); the bonus overwrites its own target row.
    float *w = cached ? cache + (size_t)((j < K) ? rd : rt) * chunk : wbuf;
    __syncthreads();
    for (int e = tid; e < n; e += kAThreads) {
      const float pt = ex2(fmaf(val(rt, e), kL2E, -mt)) * izt;
      float we = pt;
      if (residual) {
        const float qd = ex2(fmaf(val(rd, e), kL2E, -md)) * izd;
        we = fmaxf(pt - qd, 0.f);
      }
      w[e] = we;
    }
    __syncthreads();
    const int e0 = min(n, tid * per), e1 = min(n, e0 + per);
    float hi = 0.f, lo = 0.f;
    int last = -1;
    for (int e = e0; e < e1; ++e) {
      const float we = w[e];
      if (we > 0.f) last = e;
      const float y = we - lo;
      const float t = hi + y;
      lo = (t - hi) - y;
      hi = t;
    }
    const double mine = (double)hi - (double)lo;
    // block exclusive scan of `mine` in fp64
    double incl = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const double y = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += y;
    }
    int lmax = last;
#pragma unroll
    for (int off = 16; off; off >>= 1)
      lmax = max(lmax, __shfl_xor_sync(0xffffffffu, lmax, off));
    if (lane == 31) sh.scan[warp] = incl;
    if (lane == 0) sh.red_i[warp] = lmax;
    __syncthreads();
    double wbase = 0.0;
    for (int w2 = 0; w2 < warp; ++w2) wbase += sh.scan[w2];
    const double excl = wbase + incl - mine;
    if (tid == 0) {
      double tot = 0.0;
      int lst = -1;
      for (int w2 = 0; w2 < kAWarps; ++w2) {
        tot += sh.scan[w2];
        lst = max(lst, sh.red_i[w2]);
      }
      sh.w_sum = tot;
      sh.w_last = lst;
    }
    cluster.sync();  // slice masses visible cluster-wide
    double P = 0.0, Pmine = 0.0;
    int c_last = -1, last_idx = -1;
    for (int c = 0; c < kNC; ++c) {
      const AcceptShared *o = cluster.map_shared_rank(&sh, c);
      if (c == crank) Pmine = P;
      P += o->w_sum;
      if (o->w_last >= 0) { c_last = c; last_idx = o->w_last + c * chunk; }
    }
    const double W = P;            // identical in every CTA of the cluster
    if (W > 0.0) {
      const double T = uK * W;     // draw: smallest x with C(x) > T
      const double Tl = T - Pmine;
      const bool mine_has = sh.w_sum > 0.0 && Tl >= 0.0 && Tl < sh.w_sum;
      // the last thread whose run starts at or below Tl walks its run
      int cand = (mine_has && mine > 0.0 && excl <= Tl) ? tid : -1;
#pragma unroll
      for (int off = 16; off; off >>= 1)
        cand = max(cand, __shfl_xor_sync(0xffffffffu, cand, off));
      if (lane == 0) sh.sel[warp] = cand;
      __syncthreads();
      int sel = -1;
      for (int w2 = 0; w2 < kAWarps; ++w2) sel = max(sel, sh.sel[w2]);
      if (tid == sel) {
        float h2 = 0.f, l2 = 0.f;
        int found = -1;
        for (int e = e0; e < e1; ++e) {
          const float y = w[e] - l2;
          const float t = h2 + y;
          l2 = (t - h2) - y;
          h2 = t;
          if (w[e] > 0.f && excl + ((double)h2 - (double)l2) > Tl) {
            found = e;
            break;
          }
        }
        if (found < 0) found = last;  // rounding: stay inside this run
        p.out_tokens[(size_t)b * (K + 1) + j] = s0 + found;
      }
      if (T >= W && crank == c_last && tid == 0)  // rounded past the end
        p.out_tokens[(size_t)b * (K + 1) + j] = last_idx;
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
  cluster.sync();  // no CTA leaves while its shared memory may be read
  (void)staged;
  (void)wbuf;
}

int accept_chunk(int vocab) {
  int chunk = (vocab + kNC - 1) / kNC;
  return (chunk + 3) & ~3;  // 16-byte multiple
}

cudaError_t launch_spec_accept(const AcceptParams &p, cudaStream_t stream) {
  if (p.batch == 0) return cudaSuccess;
  const int K = p.num_draft, R2 = 2 * K + 1;
  const int chunk = accept_chunk(p.vocab);
  const size_t head = ((sizeof(AcceptShared) + 127) / 128) * 128;
  const size_t cache_bytes = (size_t)R2 * chunk * 4;
  const bool aligned = (reinterpret_cast<uintptr_t>(p.target_logits) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(p.draft_logits) % 16 == 0);
  int cached = aligned && (p.vocab % 4 == 0) && cache_bytes <= kMaxCacheBytes;
  const size_t smem = head + (cached ? cache_bytes : (size_t)chunk * 4);
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
  e = cudaLaunchKernelEx(&cfg, spec_accept_kernel, p, chunk, cached);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

size_t accept_max_smem(int vocab, int num_draft) {
  const int chunk = accept_chunk(vocab);
  const size_t head = ((sizeof(AcceptShared) + 127) / 128) * 128;
  return head + (size_t)chunk * 4;
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
