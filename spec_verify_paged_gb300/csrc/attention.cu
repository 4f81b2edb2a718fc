// attention.cu -- paged decode / speculative-verify attention for sm_103a.
//
// What it computes (pages: "KV cache & Flash Attention", sections
// "FlashAttention -- the tiling trick" and "PagedAttention"; "How
// speculative decoding doubles LLM speed", step 2; "How StreamingLLM
// stabilizes million-token streams via attention sinks", section "The
// StreamingLLM solution"): for every query row (b, i, h) the softmax of the
// scaled scores over the keys visible to it, times V, plus the log-sum-exp.
//
// How (GB300 design):
//  * Work unit = (sequence b, kv head g, row group rg, split s).  The rows of
//    a unit are up to RB query rows (i, h) that share kv head g (GQA group x
//    q_len), so each K/V page fetched serves all of them.  Only pages that
//    hold visible keys are enumerated (sink pages, then window pages), so
//    masked-out pages are never read.
//  * Persistent CTAs pull units from a global work queue (atomic counter).
//    One producer warp streams the unit's pages: it reads the block table
//    once per unit (one coalesced load per 32 pages) and issues one 1-D bulk
//    copy (TMA engine, cp.async.bulk) per 16-row K page and V page into an
//    NSTAGES-deep shared-memory ring guarded by mbarriers.  The producer runs
//    ahead across unit boundaries.
//  * Four consumer warps take pages round-robin.  Lane l owns D/32
//    contiguous dims; a page's 16 partial dot products are reduced with a
//    transposing butterfly (16 shuffles per row) so that lane l ends with the
//    score of key l/2.  Scores are in the log2 domain (q prescaled by
//    scale*log2 e) and folded into a running (max, sum, acc) per row with
//    exp2; the four warps' states are merged by log-sum-exp at unit end.
//  * Split-K: a unit covers split_pages pages.  If a sequence needs more
//    than one split, each writes its normalised partial (o, lse2) to the
//    workspace and takes an atomic ticket; the CTA that takes the last
//    ticket merges all partials in split order (deterministic) and resets
//    the ticket.  No CTA ever waits for another.
//  * Every wait is bounded (mbar_wait); a timeout raises SVP_DEV_TIMEOUT and
//    the CTA drains its outstanding copies and exits.
#include <cuda_bf16.h>

#include <cmath>
#include <cstdint>

#include "ptx.cuh"
#include "svp.h"
#include "svp_internal.h"

namespace svp {

static __device__ unsigned int g_status_attn;

constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
constexpr int kUnitRing = 4;
constexpr int kMaxSplitPages = 128;  // 4 block-table entries per producer lane
constexpr float kLn2 = 0.6931471805599453f;
constexpr unsigned kFull = 0xffffffffu;

struct UnitInfo {
  int b, g, rg, split;
  int n_splits, page0, n_pages, seq_len;
  int n_a, b_start, valid, pad;
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

template <typename T, int D>
struct Vec;
// lane owns VEC = D/32 consecutive elements; load them as fp32
template <>
struct Vec<float, 64> {
  static constexpr int N = 2;
  __device__ static void load(const float *p, float (&f)[2]) {
    float2 v = *reinterpret_cast<const float2 *>(p);
    f[0] = v.x; f[1] = v.y;
  }
};
template <>
struct Vec<float, 128> {
  static constexpr int N = 4;
  __device__ static void load(const float *p, float (&f)[4]) {
    float4 v = *reinterpret_cast<const float4 *>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};
template <>
struct Vec<uint16_t, 64> {
  static constexpr int N = 2;
  __device__ static void load(const uint16_t *p, float (&f)[2]) {
    uint32_t v = *reinterpret_cast<const uint32_t *>(p);
    f[0] = __uint_as_float(v << 16);
    f[1] = __uint_as_float(v & 0xffff0000u);
  }
};
template <>
struct Vec<uint16_t, 128> {
  static constexpr int N = 4;
  __device__ static void load(const uint16_t *p, float (&f)[4]) {
    uint2 v = *reinterpret_cast<const uint2 *>(p);
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
  }
};

__device__ __forceinline__ void store_out(float *p, float v) { *p = v; }
__device__ __forceinline__ void store_out(uint16_t *p, float v) {
  __nv_bfloat16 h = __float2bfloat16_rn(v);
  *p = *reinterpret_cast<uint16_t *>(&h);
}

template <typename T, int D, int RB>
struct Cfg {
  static constexpr int VEC = D / 32;
  static constexpr int PAGE_ELEMS = kBlockSize * D;
  static constexpr int PAGE_BYTES = PAGE_ELEMS * (int)sizeof(T);
  static constexpr int STAGES = (65536 / (2 * PAGE_BYTES)) < 4
                                    ? 4
                                    : (65536 / (2 * PAGE_BYTES)) > 16
                                          ? 16
                                          : (65536 / (2 * PAGE_BYTES));
};

template <typename T, int D, int RB>
struct __align__(128) Smem {
  using C = Cfg<T, D, RB>;
  T kv[C::STAGES][2][C::PAGE_ELEMS];               // K page, V page
  float red_o[kConsumerWarps][RB][D];
  float red_m[kConsumerWarps][RB];
  float red_l[kConsumerWarps][RB];
  float pbuf[kConsumerWarps][RB][kBlockSize];
  float row_m[RB], row_w[RB];
  UnitInfo unit[kUnitRing];
  int stage_ok[C::STAGES];
  uint64_t full[C::STAGES], empty[C::STAGES];
  uint64_t ufull[kUnitRing], uempty[kUnitRing];
  uint64_t epi;                                    // consumer-only barrier
  int abort_flag;
  int is_last;
  int total_units;
  int prefix[1];                                   // [batch + 1], dynamic
};

template <typename T, int D, int RB>
constexpr size_t smem_bytes(int batch) {
  return sizeof(Smem<T, D, RB>) + sizeof(int) * (size_t)batch + 16;
}

__device__ __forceinline__ void raise_flag(unsigned f) {
  atomicOr(&g_status_attn, f);
}

// Consumer-only barrier (4 warps) on an mbarrier: bounded.
template <typename S>
__device__ __forceinline__ bool epi_sync(S &sm, uint32_t &phase, int lane) {
  __syncwarp();
  if (lane == 0) mbar_arrive(&sm.epi);
  bool ok = mbar_wait(&sm.epi, phase);
  phase ^= 1u;
  __syncwarp();
  return ok;
}

// --------------------------------------------------------------------------
// per-page consumer work
// --------------------------------------------------------------------------
template <typename T, int D, int RB>
__device__ __forceinline__ void process_page(
    const T *__restrict__ kp, const T *__restrict__ vp,
    const float (&q)[RB][D / 32], float (&o)[RB][D / 32], float (&m)[RB],
    float (&l)[RB], float *pbuf /* [RB][16] of this warp */, int lane, int j0,
    bool all_visible, const int (&t)[RB], int n_sink, int window) {
  constexpr int VEC = D / 32;
  float kf[kBlockSize][VEC];
#pragma unroll
  for (int jj = 0; jj < kBlockSize; ++jj)
    Vec<T, D>::load(kp + jj * D + lane * VEC, kf[jj]);

  const int jkey = j0 + (lane >> 1);  // key held by this lane after reduce
  float p_row[RB];
#pragma unroll
  for (int r = 0; r < RB; ++r) {
    float v[kBlockSize];
#pragma unroll
    for (int jj = 0; jj < kBlockSize; ++jj) {
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < VEC; ++e) acc = fmaf(q[r][e], kf[jj][e], acc);
      v[jj] = acc;
    }
    // transposing butterfly: 16 values over 32 lanes -> lane holds key l/2
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const bool up = lane & 16;
      float send = up ? v[i] : v[i + 8];
      float keep = up ? v[i + 8] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, 16);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const bool up = lane & 8;
      float send = up ? v[i] : v[i + 4];
      float keep = up ? v[i + 4] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, 8);
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      const bool up = lane & 4;
      float send = up ? v[i] : v[i + 2];
      float keep = up ? v[i + 2] : v[i];
      v[i] = keep + __shfl_xor_sync(kFull, send, 4);
    }
    {
      const bool up = lane & 2;
      float send = up ? v[0] : v[1];
      float keep = up ? v[1] : v[0];
      v[0] = keep + __shfl_xor_sync(kFull, send, 2);
    }
    float s = v[0] + __shfl_xor_sync(kFull, v[0], 1);

    if (!all_visible) {
      const int tr = t[r];
      const bool vis = (jkey <= tr) &&
                       (window == 0 || jkey < n_sink || jkey > tr - window);
      s = vis ? s : -INFINITY;
    }
    float pm = s;
    pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 2));
    pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 4));
    pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 8));
    pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 16));
    const float m_new = fmaxf(m[r], pm);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float p = ex2(s - m_use);
    float ps = p;
    ps += __shfl_xor_sync(kFull, ps, 2);
    ps += __shfl_xor_sync(kFull, ps, 4);
    ps += __shfl_xor_sync(kFull, ps, 8);
    ps += __shfl_xor_sync(kFull, ps, 16);
    if (m_new != m[r]) {  // warp-uniform
      const float alpha = ex2(m[r] - m_use);
      l[r] *= alpha;
#pragma unroll
      for (int e = 0; e < VEC; ++e) o[r][e] *= alpha;
      m[r] = m_new;
    }
    l[r] += ps;
    p_row[r] = p;
  }
  // publish p (one lane per key) for the PV broadcast reads
  if ((lane & 1) == 0) {
#pragma unroll
    for (int r = 0; r < RB; ++r) pbuf[r * kBlockSize + (lane >> 1)] = p_row[r];
  }
  __syncwarp();
#pragma unroll
  for (int jq = 0; jq < kBlockSize; jq += 4) {
    float vf[4][VEC];
#pragma unroll
    for (int u = 0; u < 4; ++u)
      Vec<T, D>::load(vp + (jq + u) * D + lane * VEC, vf[u]);
#pragma unroll
    for (int r = 0; r < RB; ++r) {
      const float4 pv = *reinterpret_cast<const float4 *>(pbuf + r * kBlockSize + jq);
#pragma unroll
      for (int e = 0; e < VEC; ++e) {
        o[r][e] = fmaf(pv.x, vf[0][e], o[r][e]);
        o[r][e] = fmaf(pv.y, vf[1][e], o[r][e]);
        o[r][e] = fmaf(pv.z, vf[2][e], o[r][e]);
        o[r][e] = fmaf(pv.w, vf[3][e], o[r][e]);
      }
    }
  }
  __syncwarp();
}

// Zero the V rows of a page that lie outside the union of the visible sets
// (positions >= seq_len or evicted stream positions): their storage may hold
// anything, and p = 0 times a NaN is still NaN.
template <typename T, int D>
__device__ __forceinline__ void zero_invalid_rows(T *vp, int lane, int j0,
                                                  int L, int t0, int n_sink,
                                                  int window) {
  constexpr int CHUNKS = D * (int)sizeof(T) / 16;  // 16-B chunks per row
  for (int idx = lane; idx < kBlockSize * CHUNKS; idx += 32) {
    const int r = idx / CHUNKS, c = idx % CHUNKS;
    const int j = j0 + r;
    const bool valid = (j < L) &&
                       (window == 0 || j < n_sink || j > t0 - window);
    if (!valid)
      reinterpret_cast<uint4 *>(vp + r * D)[c] = make_uint4(0, 0, 0, 0);
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// --------------------------------------------------------------------------
// the kernel
// --------------------------------------------------------------------------
template <typename T, int D, int RB>
__global__ void __launch_bounds__(kThreads, 2)
    paged_attention_kernel(const AttnParams p) {
  using C = Cfg<T, D, RB>;
  constexpr int VEC = C::VEC;
  constexpr int STAGES = C::STAGES;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Smem<T, D, RB> &sm = *reinterpret_cast<Smem<T, D, RB> *>(smem_raw);

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int B = p.batch;
  const int units_per_split = p.num_kv_heads * p.n_rg;

  // ---- set-up: barriers and the per-sequence unit prefix ----
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int u = 0; u < kUnitRing; ++u) {
      mbar_init(&sm.ufull[u], 1);
      mbar_init(&sm.uempty[u], 1);
    }
    mbar_init(&sm.epi, kConsumerWarps);
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    int run = 0;
    if (lane == 0) sm.prefix[0] = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < B) {
        const int L = p.seq_lens[b];
        if (L < p.q_len || L > p.max_blocks * kBlockSize) {
          if (blockIdx.x == 0) raise_flag(SVP_DEV_BAD_SEQ_LEN);
        } else {
          int na, bs, np;
          visible_pages(L, p.q_len, p.n_sink, p.window, na, bs, np);
          n = (np + p.split_pages - 1) / p.split_pages * units_per_split;
        }
      }
      int incl = n;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        int y = __shfl_up_sync(kFull, incl, off);
        if (lane >= off) incl += y;
      }
      if (b < B) sm.prefix[b + 1] = run + incl;
      run += __shfl_sync(kFull, incl, 31);
    }
    if (lane == 0) sm.total_units = run;
  }
  __syncthreads();
  const int total_units = sm.total_units;

  if (warp == kConsumerWarps) {
    // ======================= producer warp =======================
    int c = 0;   // pages issued so far
    int us = 0;  // units taken so far
    bool ok = true;
    while (true) {
      int u = 0;
      if (lane == 0) u = atomicAdd(&p.counters[0], 1);
      u = __shfl_sync(kFull, u, 0);
      const int slot = us % kUnitRing;
      if (lane == 0)
        ok = mbar_wait(&sm.uempty[slot], ((us / kUnitRing) & 1) ^ 1);
      ok = __shfl_sync(kFull, ok, 0) && !sm.abort_flag;
      if (!ok) break;
      if (u >= total_units) {
        if (lane == 0) {
          sm.unit[slot].valid = 0;
          mbar_arrive(&sm.ufull[slot]);
        }
        break;
      }
      // decode unit u -> (b, g, split, rg): binary search in the prefix
      int lo = 0, hi = B;  // find b with prefix[b] <= u < prefix[b+1]
      while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (sm.prefix[mid] <= u) lo = mid; else hi = mid;
      }
      const int b = lo;
      const int ub = u - sm.prefix[b];
      const int n_units_b = sm.prefix[b + 1] - sm.prefix[b];
      const int n_splits = n_units_b / units_per_split;
      const int rg = ub % p.n_rg;
      const int t2 = ub / p.n_rg;
      const int split = t2 % n_splits;
      const int g = t2 / n_splits;
      const int L = p.seq_lens[b];
      int na, bs, np;
      visible_pages(L, p.q_len, p.n_sink, p.window, na, bs, np);
      const int page0 = split * p.split_pages;
      const int n_pages = min(p.split_pages, np - page0);
      if (lane == 0) {
        UnitInfo &ui = sm.unit[slot];
        ui.b = b; ui.g = g; ui.rg = rg; ui.split = split;
        ui.n_splits = n_splits; ui.page0 = page0; ui.n_pages = n_pages;
        ui.seq_len = L; ui.n_a = na; ui.b_start = bs; ui.valid = 1;
        mbar_arrive(&sm.ufull[slot]);
      }
      // block-table entries of this unit's pages, one coalesced load each
      int phys[kMaxSplitPages / 32];
#pragma unroll
      for (int k4 = 0; k4 < kMaxSplitPages / 32; ++k4) {
        const int k = k4 * 32 + lane;
        phys[k4] = -1;
        if (k < n_pages) {
          const int pidx = page0 + k;
          const int lb = (pidx < na) ? pidx : bs + (pidx - na);
          phys[k4] = __ldg(p.block_table + (size_t)b * p.max_blocks + lb);
        }
      }
      const size_t head_off = (size_t)g * C::PAGE_ELEMS;
#pragma unroll
      for (int k4 = 0; k4 < kMaxSplitPages / 32; ++k4) {
        for (int kk = 0; kk < 32; ++kk) {
          const int k = k4 * 32 + kk;
          if (k >= n_pages) break;
          const int ph = __shfl_sync(kFull, phys[k4], kk);
          if (lane == 0) {
            const int s = c % STAGES;
            if (!mbar_wait(&sm.empty[s], ((c / STAGES) & 1) ^ 1)) {
              ok = false;
            } else if (ph < 0 || ph >= p.num_blocks) {
              raise_flag(SVP_DEV_BAD_BLOCK_ID);
              sm.stage_ok[s] = 0;
              mbar_arrive(&sm.full[s]);
            } else {
              sm.stage_ok[s] = 1;
              const size_t off = (size_t)ph * p.num_kv_heads * C::PAGE_ELEMS + head_off;
              mbar_arrive_expect_tx(&sm.full[s], 2 * C::PAGE_BYTES);
              bulk_g2s(sm.kv[s][0], static_cast<const T *>(p.k_cache) + off,
                       C::PAGE_BYTES, &sm.full[s]);
              bulk_g2s(sm.kv[s][1], static_cast<const T *>(p.v_cache) + off,
                       C::PAGE_BYTES, &sm.full[s]);
            }
          }
          ok = __shfl_sync(kFull, ok, 0);
          if (!ok) break;
          ++c;
        }
        if (!ok) break;
      }
      if (!ok) break;
      ++us;
    }
    if (!ok) {
      // give up: flag it, then wait (bounded) for copies still in flight
      if (lane == 0) {
        raise_flag(SVP_DEV_TIMEOUT);
        sm.abort_flag = 1;
        for (int k = max(0, c - STAGES); k < c; ++k)
          (void)mbar_wait(&sm.full[k % STAGES], (k / STAGES) & 1);
      }
    }
  } else {
    // ======================= consumer warps =======================
    const int ctid = tid;  // 0..127
    int c = 0, us = 0;
    uint32_t epi_phase = 0;
    float *pbuf = &sm.pbuf[warp][0][0];
    while (true) {
      const int slot = us % kUnitRing;
      // every lane waits itself: each thread acquires the producer's writes
      const bool ok =
          __all_sync(kFull, mbar_wait(&sm.ufull[slot], (us / kUnitRing) & 1));
      if (!ok) {
        if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
        break;
      }
      const UnitInfo ui = sm.unit[slot];
      if (!ui.valid || sm.abort_flag) break;

      const int b = ui.b, g = ui.g, rg = ui.rg, L = ui.seq_len;
      const int t0 = L - p.q_len;
      // this unit's query rows
      float q[RB][VEC], o[RB][VEC], m[RB], l[RB];
      int t[RB];
      int t_min = 0x7fffffff, t_max = -1;
#pragma unroll
      for (int r = 0; r < RB; ++r) {
        const int gr = rg * RB + r;
        m[r] = -INFINITY;
        l[r] = 0.f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) { o[r][e] = 0.f; q[r][e] = 0.f; }
        t[r] = -1;
        if (gr < p.rows) {
          const int i = gr / p.group;
          const int h = g * p.group + gr % p.group;
          const T *qp = static_cast<const T *>(p.q) +
                        (((size_t)b * p.q_len + i) * p.num_q_heads + h) * D +
                        lane * VEC;
          Vec<T, D>::load(qp, q[r]);
#pragma unroll
          for (int e = 0; e < VEC; ++e) q[r][e] *= p.qscale;
          t[r] = t0 + i;
          t_min = min(t_min, t[r]);
          t_max = max(t_max, t[r]);
        }
      }
      // pages of this unit owned by this warp: global page index == warp mod 4
      const int first = ((warp - c) % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
      bool aborted = false;
      for (int k = first; k < ui.n_pages; k += kConsumerWarps) {
        const int cc = c + k;
        const int s = cc % STAGES;
        const bool got =
            __all_sync(kFull, mbar_wait(&sm.full[s], (cc / STAGES) & 1));
        if (!got) {
          if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
          aborted = true;
          break;
        }
        if (sm.stage_ok[s]) {
          const int pidx = ui.page0 + k;
          const int lb = (pidx < ui.n_a) ? pidx : ui.b_start + (pidx - ui.n_a);
          const int j0 = lb * kBlockSize;
          const int j1 = j0 + kBlockSize - 1;
          // rows of this page outside the union of visible sets?
          const bool union_full =
              (j1 < L) && (p.window == 0 || j1 < p.n_sink ||
                           j0 > t0 - p.window);
          if (!union_full)
            zero_invalid_rows<T, D>(sm.kv[s][1], lane, j0, L, t0, p.n_sink,
                                    p.window);
          const bool all_vis =
              (j1 <= t_min) && (p.window == 0 || j1 < p.n_sink ||
                                j0 > t_max - p.window);
          process_page<T, D, RB>(sm.kv[s][0], sm.kv[s][1], q, o, m, l, pbuf,
                                 lane, j0, all_vis, t, p.n_sink, p.window);
        }
        if (lane == 0) mbar_arrive(&sm.empty[s]);
      }
      c += ui.n_pages;

      // ---- epilogue: merge the 4 warps' states ----
      if (lane == 0) {
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          sm.red_m[warp][r] = m[r];
          sm.red_l[warp][r] = l[r];
        }
      }
#pragma unroll
      for (int r = 0; r < RB; ++r)
#pragma unroll
        for (int e = 0; e < VEC; ++e) sm.red_o[warp][r][lane * VEC + e] = o[r][e];
      if (!epi_sync(sm, epi_phase, lane) || aborted) {
        if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
        break;
      }
      const int grp = (b * p.num_kv_heads + g) * p.n_rg + rg;
      const bool single = ui.n_splits == 1;
      for (int e = ctid; e < RB * D; e += kConsumerWarps * 32) {
        const int r = e / D, d = e % D;
        const int gr = rg * RB + r;
        if (gr >= p.rows) continue;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm.red_m[w][r]);
        float Lsum = 0.f, O = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w) {
            const float f = ex2(sm.red_m[w][r] - M);
            Lsum = fmaf(f, sm.red_l[w][r], Lsum);
            O = fmaf(f, sm.red_o[w][r][d], O);
          }
        }
        const float on = Lsum > 0.f ? O / Lsum : 0.f;
        const float lse2 = Lsum > 0.f ? M + log2f(Lsum) : -INFINITY;
        if (single) {
          const int i = gr / p.group;
          const int h = g * p.group + gr % p.group;
          const size_t row = ((size_t)b * p.q_len + i) * p.num_q_heads + h;
          store_out(static_cast<T *>(p.out) + row * D + d, on);
          if (d == 0) p.lse[row] = lse2 * kLn2;
        } else {
          const size_t prow = ((size_t)grp * p.max_splits + ui.split) * RB + r;
          p.part_o[prow * D + d] = on;
          if (d == 0) p.part_lse[prow] = lse2;
        }
      }
      if (!single) {
        __threadfence();
        if (!epi_sync(sm, epi_phase, lane)) {
          if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
          break;
        }
        if (ctid == 0) {
          const int ticket = atomicAdd(&p.tickets[grp], 1);
          sm.is_last = (ticket == ui.n_splits - 1);
        }
        if (!epi_sync(sm, epi_phase, lane)) {
          if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
          break;
        }
        if (sm.is_last) {
          __threadfence();
          const int ns = ui.n_splits;
          const size_t base = (size_t)grp * p.max_splits;
          // per-row max and weight sum over the splits (warp w: rows w, w+4..)
          for (int r = warp; r < RB; r += kConsumerWarps) {
            float M = -INFINITY;
            for (int s = lane; s < ns; s += 32)
              M = fmaxf(M, __ldcg(p.part_lse + (base + s) * RB + r));
#pragma unroll
            for (int off = 16; off; off >>= 1)
              M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
            float W = 0.f;
            if (M != -INFINITY)
              for (int s = lane; s < ns; s += 32)
                W += ex2(__ldcg(p.part_lse + (base + s) * RB + r) - M);
#pragma unroll
            for (int off = 16; off; off >>= 1)
              W += __shfl_xor_sync(kFull, W, off);
            if (lane == 0) { sm.row_m[r] = M; sm.row_w[r] = W; }
          }
          if (!epi_sync(sm, epi_phase, lane)) {
            if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
            break;
          }
          for (int e = ctid; e < RB * D; e += kConsumerWarps * 32) {
            const int r = e / D, d = e % D;
            const int gr = rg * RB + r;
            if (gr >= p.rows) continue;
            const float M = sm.row_m[r], W = sm.row_w[r];
            float acc = 0.f;
            for (int s = 0; s < ns; ++s) {
              const float ls = __ldcg(p.part_lse + (base + s) * RB + r);
              if (ls == -INFINITY) continue;
              acc = fmaf(ex2(ls - M),
                         __ldcg(p.part_o + ((base + s) * RB + r) * D + d), acc);
            }
            const int i = gr / p.group;
            const int h = g * p.group + gr % p.group;
            const size_t row = ((size_t)b * p.q_len + i) * p.num_q_heads + h;
            store_out(static_cast<T *>(p.out) + row * D + d, W > 0.f ? acc / W : 0.f);
            if (d == 0) p.lse[row] = (M + log2f(W)) * kLn2;
          }
          if (ctid == 0) p.tickets[grp] = 0;
        }
      }
      // all consumers are done with this unit's info and scratch
      if (!epi_sync(sm, epi_phase, lane)) {
        if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
        break;
      }
      if (ctid == 0) mbar_arrive(&sm.uempty[slot]);
      ++us;
    }
  }

  // ---- tear-down: the last CTA out resets the work queue ----
  __syncthreads();
  if (tid == 0) {
    __threadfence();
    const int done = atomicAdd(&p.counters[1], 1);
    if (done == (int)gridDim.x - 1) {
      p.counters[0] = 0;
      p.counters[1] = 0;
      __threadfence();
    }
  }
}

// --------------------------------------------------------------------------
// host side
// --------------------------------------------------------------------------
template <typename T, int D, int RB>
static cudaError_t launch_t(const AttnParams &p, int grid, cudaStream_t st) {
  const size_t smem = smem_bytes<T, D, RB>(p.batch);
  auto kern = paged_attention_kernel<T, D, RB>;
  cudaError_t e = cudaFuncSetAttribute(
      kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(p);
  return cudaGetLastError();
}

template <typename T, int D, int RB>
static int occupancy_t(int batch) {
  const size_t smem = smem_bytes<T, D, RB>(batch);
  auto kern = paged_attention_kernel<T, D, RB>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return 1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) !=
      cudaSuccess)
    return 1;
  return n > 0 ? n : 1;
}

#define SVP_DISPATCH_RB(T, D, RB, CALL) \
  switch (RB) {                         \
    case 1: CALL(T, D, 1); break;       \
    case 2: CALL(T, D, 2); break;       \
    case 4: CALL(T, D, 4); break;       \
    default: CALL(T, D, 8); break;      \
  }

cudaError_t launch_attention(const AttnParams &p, int dtype, int grid,
                             cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
#define SVP_CALL(T, D, RB) e = launch_t<T, D, RB>(p, grid, stream)
  if (dtype == 0) {
    if (p.head_dim == 64) { SVP_DISPATCH_RB(float, 64, p.rb, SVP_CALL) }
    else { SVP_DISPATCH_RB(float, 128, p.rb, SVP_CALL) }
  } else {
    if (p.head_dim == 64) { SVP_DISPATCH_RB(uint16_t, 64, p.rb, SVP_CALL) }
    else { SVP_DISPATCH_RB(uint16_t, 128, p.rb, SVP_CALL) }
  }
#undef SVP_CALL
  return e;
}

int attention_ctas_per_sm(int dtype, int head_dim, int rb, int batch) {
  int n = 1;
#define SVP_CALL(T, D, RB) n = occupancy_t<T, D, RB>(batch)
  if (dtype == 0) {
    if (head_dim == 64) { SVP_DISPATCH_RB(float, 64, rb, SVP_CALL) }
    else { SVP_DISPATCH_RB(float, 128, rb, SVP_CALL) }
  } else {
    if (head_dim == 64) { SVP_DISPATCH_RB(uint16_t, 64, rb, SVP_CALL) }
    else { SVP_DISPATCH_RB(uint16_t, 128, rb, SVP_CALL) }
  }
#undef SVP_CALL
  return n;
}

cudaError_t read_status_attention(cudaStream_t s, unsigned *flags) {
  unsigned v = 0;
  cudaError_t e = cudaMemcpyFromSymbolAsync(&v, g_status_attn, sizeof v, 0,
                                            cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return e;
  const unsigned zero = 0;
  e = cudaMemcpyToSymbolAsync(g_status_attn, &zero, sizeof zero, 0,
                              cudaMemcpyHostToDevice, s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  *flags |= v;
  return e;
}

}  // namespace svp
