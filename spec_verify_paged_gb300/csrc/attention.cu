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
//  * A group = (sequence b, kv head g, row group rg): up to RB query rows
//    (i, h) that share kv head g (GQA group x q_len), so each K/V page
//    fetched serves all of them.  Only pages that hold visible keys are
//    enumerated (sink pages, then window pages), so masked-out pages are
//    never read.
//  * Persistent CTAs take equal slices of the flattened (group, page) list
//    (stream-K, attn_common.cuh).  One producer warp walks the slice's
//    segments: it reads the block table once per 128 pages (coalesced) and
//    fills an NSTAGES-deep shared-memory ring guarded by mbarriers, running
//    ahead across segment boundaries.
//  * CUDA-core path (few rows per kv head): one 1-D bulk copy (TMA engine,
//    cp.async.bulk) per 16-row K page and V page.  Four consumer warps take
//    pages round-robin; lane l owns D/32 dims; a page's 16 partial dot
//    products are reduced with a transposing butterfly so lane l ends with
//    the score of key l/2; online softmax in the log2 domain with exp2.
//  * Tensor-core path (bf16, many rows: GQA groups x verify positions): each
//    page arrives as 2-D tensor copies (cp.async.bulk.tensor, 128-byte
//    swizzle, 64-element boxes) so ldmatrix reads are bank-conflict free.
//    A consumer warp owns whole pages for a 16-row group: S = Q K^T with
//    mma.sync m16n8k16 (keys as N), the S accumulators are re-used in
//    registers as the A operand of P V (no shared-memory round trip), V is
//    read with ldmatrix.trans.  The running row sums stay per lane and are
//    reduced once per unit.
//  * The warps' states are merged by log-sum-exp at segment end.  A group
//    split over several slices leaves one partial per slice; the merge
//    kernel (attn_common.cuh) combines them in slice order
//    (deterministic).  No CTA ever waits for another.
//  * Rows of a page that hold no valid data (positions >= seq_len, evicted
//    stream rows) are zeroed in shared memory before P V, because p = 0
//    times a NaN left in unused cache memory is still NaN.
//  * Every wait is bounded (mbar_wait); a timeout raises SVP_DEV_TIMEOUT and
//    the CTA drains its outstanding copies and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <type_traits>

#include "attn_common.cuh"

namespace svp {

static __device__ unsigned int g_status_attn;

constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (kConsumerWarps + 1);
template <typename T, int D>
struct Vec;
// lane owns VEC = D/32 consecutive elements; load them as fp32
template <>
struct Vec<float, 64> {
  __device__ static void load(const float *p, float (&f)[2]) {
    float2 v = *reinterpret_cast<const float2 *>(p);
    f[0] = v.x; f[1] = v.y;
  }
};
template <>
struct Vec<float, 128> {
  __device__ static void load(const float *p, float (&f)[4]) {
    float4 v = *reinterpret_cast<const float4 *>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
};
template <>
struct Vec<uint16_t, 64> {
  __device__ static void load(const uint16_t *p, float (&f)[2]) {
    uint32_t v = *reinterpret_cast<const uint32_t *>(p);
    f[0] = __uint_as_float(v << 16);
    f[1] = __uint_as_float(v & 0xffff0000u);
  }
};
template <>
struct Vec<uint16_t, 128> {
  __device__ static void load(const uint16_t *p, float (&f)[4]) {
    uint2 v = *reinterpret_cast<const uint2 *>(p);
    f[0] = __uint_as_float(v.x << 16);
    f[1] = __uint_as_float(v.x & 0xffff0000u);
    f[2] = __uint_as_float(v.y << 16);
    f[3] = __uint_as_float(v.y & 0xffff0000u);
  }
};

// FP8 E4M3 pages: lane owns VEC codes, converted exactly (through half)
template <>
struct Vec<uint8_t, 64> {
  __device__ static void load(const uint8_t *p, float (&f)[2]) {
    const __nv_fp8x2_storage_t v = *reinterpret_cast<const uint16_t *>(p);
    const float2 a = __half22float2(__half2(__nv_cvt_fp8x2_to_halfraw2(v, __NV_E4M3)));
    f[0] = a.x; f[1] = a.y;
  }
};
template <>
struct Vec<uint8_t, 128> {
  __device__ static void load(const uint8_t *p, float (&f)[4]) {
    const uint32_t v = *reinterpret_cast<const uint32_t *>(p);
    const float2 a = __half22float2(
        __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v & 0xffffu), __NV_E4M3)));
    const float2 c = __half22float2(
        __half2(__nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(v >> 16), __NV_E4M3)));
    f[0] = a.x; f[1] = a.y; f[2] = c.x; f[3] = c.y;
  }
};

// element type of q and out: the cache's, bf16 bits for an FP8 cache
template <typename T> struct QT { using type = T; };
template <> struct QT<uint8_t> { using type = uint16_t; };

template <typename T, int D>
struct Cfg {
  static constexpr int PAGE_ELEMS = kBlockSize * D;
  static constexpr int PAGE_BYTES = PAGE_ELEMS * (int)sizeof(T);
  static constexpr int STAGES = (65536 / (2 * PAGE_BYTES)) < 4
                                    ? 4
                                    : (65536 / (2 * PAGE_BYTES)) > 16
                                          ? 16
                                          : (65536 / (2 * PAGE_BYTES));
};

// RW = rows one consumer warp accumulates: RB on the CUDA-core path, one
// m16 tile (16) on the tensor-core path, where a unit of 32 rows is shared
// by warp pairs.
template <typename T, int D, int RB, int RW>
struct Smem {
  using C = Cfg<T, D>;
  alignas(1024) unsigned char kv[C::STAGES][2][C::PAGE_BYTES];  // K, V page
  float red_o[kConsumerWarps][RW][D];
  float red_m[kConsumerWarps][RW];
  float red_l[kConsumerWarps][RW];
  float pbuf[kConsumerWarps][RW][kBlockSize];
  float wf[kConsumerWarps][RB];                    // per-warp row weights
  UnitInfo unit[kUnitRing];
  int stage_ok[C::STAGES];
  uint64_t full[C::STAGES], empty[C::STAGES];
  uint64_t ufull[kUnitRing], uempty[kUnitRing];
  uint64_t epi;                                    // consumer-only barrier
#ifdef SVP_TEST_STALL_AFTER
  uint64_t stall;  // test builds: a barrier nothing arrives on
#endif
  int abort_flag;
  int prefix[1];  // [batch + 1] item prefix, then [batch] lengths: dynamic
};

template <typename T, int D, int RB, bool MMA>
constexpr size_t smem_bytes(int batch) {
  // + 1024 so the ring can be aligned to 1024 bytes (the swizzle atom)
  return sizeof(Smem<T, D, RB, MMA ? 16 : RB>) +
         sizeof(int) * (2 * (size_t)batch + 1) + 1024;
}

__device__ __forceinline__ void raise_flag(unsigned f) {
  atomicOr(&g_status_attn, f);
}

// Consumer-only barrier (4 warps) on an mbarrier: bounded, warp-uniform.
template <typename S>
__device__ __forceinline__ bool epi_sync(S &sm, uint32_t &phase, int lane) {
  return consumer_sync(&sm.epi, phase, lane);
}

// --------------------------------------------------------------------------
// tensor-core helpers (warp-level MMA, bf16 in, fp32 accumulate)
// --------------------------------------------------------------------------
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0,
                                        uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0,
                                          uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile(
      "ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
      : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
      : "r"(addr));
}
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4],
                                         uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// two fp32 -> bf16x2 (round to nearest even); `lo` goes to the low half
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// Byte offset of 16-byte chunk `chunk` of row `key` in a page stored as
// D/64 boxes of [16 rows][128 B] with the TMA 128-byte swizzle (the chunk
// index within a 128-byte row is XOR-ed with the row index mod 8).
__device__ __forceinline__ uint32_t swz(int key, int chunk) {
  return (uint32_t)((chunk >> 3) * kBoxBytes + key * 128 +
                    (((chunk & 7) ^ (key & 7)) << 4));
}

// --------------------------------------------------------------------------
// CUDA-core consumer work on one page
// --------------------------------------------------------------------------
template <typename T, int D, int RB>
__device__ __forceinline__ void process_page_fma(
    const T *__restrict__ kp, const T *__restrict__ vp,
    const float (&q)[RB][D / 32], float (&o)[RB][D / 32], float (&m)[RB],
    float (&l)[RB], float *pbuf /* [RB][16] of this warp */, int lane, int j0,
    bool all_visible, const int (&t)[RB], const uint32_t (&tm)[RB], int base,
    int n_sink, int window) {
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

    if (!all_visible)
      s = key_visible(jkey, t[r], tm[r], base, n_sink, window) ? s : -INFINITY;
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

// --------------------------------------------------------------------------
// FP8 pages with one query row per kv head (head_dim 128): key per lane
// --------------------------------------------------------------------------
// d = a * b + c with a, b fp16 and c, d fp32: the product of two fp16 values
// is exact in fp32, so this equals widening both and one fmaf.
__device__ __forceinline__ float fma_h(float c, unsigned short a,
                                       unsigned short b) {
  float d;
  asm("fma.rn.f32.f16 %0, %1, %2, %3;" : "=f"(d) : "h"(a), "h"(b), "f"(c));
  return d;
}
// two E4M3 codes (low 16 bits) -> fp16x2, exact
__device__ __forceinline__ uint32_t e4m3x2_h2(uint32_t w) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
      (__nv_fp8x2_storage_t)(w & 0xffffu), __NV_E4M3);
  return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Lane l takes key l/2 of the page and half l%2 of its 128 dims: 64
// fp16 x E4M3 products summed in fp32 with mixed-precision FMAs, then one
// shuffle joins the halves -- no transposing reduction of 16 partial dot
// products.  The four 16-code chunks of a half are visited in an order
// rotated by the key (qr holds q's chunks in the same order), so the eight
// lanes of a 16-byte load phase hit eight different bank groups.  P V: the
// lane owns dims 4l..4l+3, p goes through shared memory as fp16.  q is the
// row's bf16 values as fp16 (exact in fp16's normal range), unscaled; the
// score is scaled once (qscale).
__device__ __forceinline__ void process_page_fp8_k1(
    const uint8_t *__restrict__ kp, const uint8_t *__restrict__ vp,
    const uint32_t (&qr)[4][8], float (&o)[4], float &m, float &l,
    uint16_t *pb16 /* [16] of this warp */, int lane, int j0,
    bool all_visible, int t, uint32_t tm, int base, int n_sink, int window,
    float qscale) {
  const int key = lane >> 1, half = lane & 1;
  const uint8_t *krow = kp + key * 128 + half * 64;
  float acc = 0.f, acc2 = 0.f;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 w = *reinterpret_cast<const uint4 *>(krow + ((c + key) & 3) * 16);
    const uint32_t wv[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const uint32_t k01 = e4m3x2_h2(wv[i]), k23 = e4m3x2_h2(wv[i] >> 16);
      const uint32_t q01 = qr[c][2 * i], q23 = qr[c][2 * i + 1];
      acc = fma_h(acc, (unsigned short)(k01 & 0xffffu), (unsigned short)(q01 & 0xffffu));
      acc2 = fma_h(acc2, (unsigned short)(k01 >> 16), (unsigned short)(q01 >> 16));
      acc = fma_h(acc, (unsigned short)(k23 & 0xffffu), (unsigned short)(q23 & 0xffffu));
      acc2 = fma_h(acc2, (unsigned short)(k23 >> 16), (unsigned short)(q23 >> 16));
    }
  }
  acc += acc2;
  float sc = (acc + __shfl_xor_sync(kFull, acc, 1)) * qscale;
  const int jkey = j0 + key;
  if (!all_visible)
    sc = key_visible(jkey, t, tm, base, n_sink, window) ? sc : -INFINITY;
  float pm = sc;
  pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 2));
  pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 4));
  pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 8));
  pm = fmaxf(pm, __shfl_xor_sync(kFull, pm, 16));
  const float m_new = fmaxf(m, pm);
  const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
  const float pv = ex2(sc - m_use);
  float ps = half ? 0.f : pv;  // each key once
  ps += __shfl_xor_sync(kFull, ps, 2);
  ps += __shfl_xor_sync(kFull, ps, 4);
  ps += __shfl_xor_sync(kFull, ps, 8);
  ps += __shfl_xor_sync(kFull, ps, 16);
  if (m_new != m) {  // warp-uniform
    const float alpha = ex2(m - m_use);
    l *= alpha;
#pragma unroll
    for (int e = 0; e < 4; ++e) o[e] *= alpha;
    m = m_new;
  }
  l += ps;
  if (!half) pb16[key] = __half_as_ushort(__float2half_rn(pv));
  __syncwarp();
#pragma unroll
  for (int jq = 0; jq < kBlockSize; jq += 4) {
    const uint2 p4 = *reinterpret_cast<const uint2 *>(pb16 + jq);
    const unsigned short pj[4] = {(unsigned short)(p4.x & 0xffffu),
                                  (unsigned short)(p4.x >> 16),
                                  (unsigned short)(p4.y & 0xffffu),
                                  (unsigned short)(p4.y >> 16)};
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const uint32_t w = *reinterpret_cast<const uint32_t *>(vp + (jq + u) * 128 + lane * 4);
      const uint32_t v01 = e4m3x2_h2(w), v23 = e4m3x2_h2(w >> 16);
      o[0] = fma_h(o[0], (unsigned short)(v01 & 0xffffu), pj[u]);
      o[1] = fma_h(o[1], (unsigned short)(v01 >> 16), pj[u]);
      o[2] = fma_h(o[2], (unsigned short)(v23 & 0xffffu), pj[u]);
      o[3] = fma_h(o[3], (unsigned short)(v23 >> 16), pj[u]);
    }
  }
  __syncwarp();
}

// --------------------------------------------------------------------------
// tensor-core consumer work on one page (16 query rows x 16 keys)
// Lane layout of m16n8k16: g = lane/4 (rows g, g+8), t = lane%4.
// --------------------------------------------------------------------------
// All MMA operand fragments of one page: K as the B operand of S = Q K^T
// (ldmatrix) and V as the B operand of P V (ldmatrix.trans), so the ring
// stage can be released before any arithmetic.
template <int D>
__device__ __forceinline__ void load_page_frags(uint32_t kbase, uint32_t vbase,
                                                uint32_t (&kb)[D / 16][4],
                                                uint32_t (&vb)[D / 16][4],
                                                int lane) {
  const int mi = lane >> 3, mrow = lane & 7;
  const int kkey = (mi >> 1) * 8 + mrow;
  const int vkey = (mi & 1) * 8 + mrow;
#pragma unroll
  for (int ks = 0; ks < D / 16; ++ks)
    ldsm_x4(kbase + swz(kkey, 2 * ks + (mi & 1)), kb[ks][0], kb[ks][1],
            kb[ks][2], kb[ks][3]);
#pragma unroll
  for (int d2 = 0; d2 < D / 16; ++d2)
    ldsm_x4_t(vbase + swz(vkey, 2 * d2 + (mi >> 1)), vb[d2][0], vb[d2][1],
              vb[d2][2], vb[d2][3]);
}

template <int D>
__device__ __forceinline__ void process_page_mma(
    const uint32_t (&kb)[D / 16][4], const uint32_t (&vb)[D / 16][4],
    const uint32_t (&qa)[D / 16][4], float (&o)[D / 8][4], float (&m)[2],
    float (&lp)[2], int lane, int j0, bool all_visible, const int (&t)[2],
    const uint32_t (&tm)[2], int base, int n_sink, int window, float qscale) {
  const int tq = lane & 3;
  // S = Q K^T : two n8 tiles (keys 0-7, 8-15), k over D, accumulated in two
  // independent chains (even / odd k steps) to halve the dependent depth
  float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
  {
    float s2[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
    for (int ks = 0; ks < D / 16; ks += 2) {
      mma16816(s[0], qa[ks], kb[ks][0], kb[ks][1]);
      mma16816(s[1], qa[ks], kb[ks][2], kb[ks][3]);
      mma16816(s2[0], qa[ks + 1], kb[ks + 1][0], kb[ks + 1][1]);
      mma16816(s2[1], qa[ks + 1], kb[ks + 1][2], kb[ks + 1][3]);
    }
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) s[nt][e] += s2[nt][e];
  }
  // scale into the log2 domain, mask, running max per row (rows g, g+8)
  float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float v = s[nt][e] * qscale;
      if (!all_visible) {
        const int j = j0 + nt * 8 + 2 * tq + (e & 1);
        v = key_visible(j, t[e >> 1], tm[e >> 1], base, n_sink, window)
                ? v : -INFINITY;
      }
      s[nt][e] = v;
      mx[e >> 1] = fmaxf(mx[e >> 1], v);
    }
  float alpha[2], mu[2];
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 1));
    mx[r] = fmaxf(mx[r], __shfl_xor_sync(kFull, mx[r], 2));
    const float m_new = fmaxf(m[r], mx[r]);
    mu[r] = (m_new == -INFINITY) ? 0.f : m_new;
    alpha[r] = ex2(m[r] - mu[r]);
    m[r] = m_new;
  }
  float ps[2] = {0.f, 0.f};
#pragma unroll
  for (int nt = 0; nt < 2; ++nt)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float pv = ex2(s[nt][e] - mu[e >> 1]);
      s[nt][e] = pv;
      ps[e >> 1] += pv;
    }
  lp[0] = lp[0] * alpha[0] + ps[0];
  lp[1] = lp[1] * alpha[1] + ps[1];
  if (__any_sync(kFull, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
    for (int dn = 0; dn < D / 8; ++dn) {
      o[dn][0] *= alpha[0];
      o[dn][1] *= alpha[0];
      o[dn][2] *= alpha[1];
      o[dn][3] *= alpha[1];
    }
  }
  // P as the A operand (the S accumulator layout is the A fragment layout)
  const uint32_t pa[4] = {pack_bf16(s[0][0], s[0][1]), pack_bf16(s[0][2], s[0][3]),
                          pack_bf16(s[1][0], s[1][1]), pack_bf16(s[1][2], s[1][3])};
#pragma unroll
  for (int d2 = 0; d2 < D / 16; ++d2) {
    mma16816(o[2 * d2], pa, vb[d2][0], vb[d2][1]);
    mma16816(o[2 * d2 + 1], pa, vb[d2][2], vb[d2][3]);
  }
}

// Zero the V rows of a page that lie outside the union of the visible sets.
template <typename T, int D, bool MMA>
__device__ __forceinline__ void zero_invalid_rows(unsigned char *vp, int lane,
                                                  int j0, int L, int t0,
                                                  int n_sink, int window) {
  constexpr int ROWB = D * (int)sizeof(T);
  constexpr int CHUNKS = ROWB / 16;  // 16-B chunks per row
  for (int idx = lane; idx < kBlockSize * CHUNKS; idx += 32) {
    const int r = idx / CHUNKS, c = idx % CHUNKS;
    const int j = j0 + r;
    const bool valid = (j < L) &&
                       (window == 0 || j < n_sink || j > t0 - window);
    if (!valid) {
      // every chunk of the row is cleared, so the swizzle does not matter
      const int off = MMA ? (c >> 3) * kBoxBytes + r * 128 + (c & 7) * 16
                          : r * ROWB + c * 16;
      *reinterpret_cast<uint4 *>(vp + off) = make_uint4(0, 0, 0, 0);
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
}

// --------------------------------------------------------------------------
// the kernel
// --------------------------------------------------------------------------
// CTAs per SM the registers must allow: three for the single-row paths
// (their shared-memory rings allow three), two otherwise
template <typename T, int D, int RB, bool MMA>
constexpr int min_ctas() {
  return (!MMA && RB == 1) ? 3 : 2;
}

template <typename T, int D, int RB, bool MMA>
__global__ void __launch_bounds__(kThreads, (min_ctas<T, D, RB, MMA>()))
    paged_attention_kernel(const AttnParams p,
                           const __grid_constant__ TensorMaps tm) {
  using C = Cfg<T, D>;
  constexpr int VEC = D / 32;
  constexpr int STAGES = C::STAGES;
  extern __shared__ unsigned char smem_raw[];
  // tensor path: MT m16 tiles per unit, one per warp of a warp group that
  // shares each page; NSTREAM groups take pages round-robin
  constexpr int MT = MMA ? RB / 16 : 1;
  constexpr int RW = MMA ? 16 : RB;
  constexpr int NSTREAM = kConsumerWarps / MT;
  // A stage's previous page (c - STAGES) must belong to the same stream as
  // page c: that stream has then waited for it, so its wait for page c is
  // at most one phase ahead of the stage's full barrier.  Otherwise the
  // parity wait can pass two phases early, on a copy still in flight.
  static_assert(STAGES % NSTREAM == 0, "ring depth: a multiple of the streams");
  Smem<T, D, RB, RW> &sm = *reinterpret_cast<Smem<T, D, RB, RW> *>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));

  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const int groups_per_seq = p.num_kv_heads * p.n_rg;

  // ---- set-up: barriers and the per-sequence unit prefix ----
  if constexpr (MMA) {
    if (tid == 32) {
      prefetch_tensormap(&tm.k);
      prefetch_tensormap(&tm.v);
    }
  }
  if (tid == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], MT);  // every warp of the owning group
    }
    for (int u = 0; u < kUnitRing; ++u) {
      mbar_init(&sm.ufull[u], 1);
      mbar_init(&sm.uempty[u], 1);
    }
    mbar_init(&sm.epi, kConsumerWarps);
#ifdef SVP_TEST_STALL_AFTER
    mbar_init(&sm.stall, 1);
#endif
    sm.abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();  // barriers initialised
  // launched early (programmatic dependent launch): nothing in global
  // memory is touched before the previous kernel on the stream is done --
  // or, right behind the append of the newest positions (p.early), nothing
  // but the pages holding them (the producer waits before the first batch
  // with such a page, the consumers before their first output)
  if (!p.early) pdl_wait();
  if (tid == 0) {
    p.desc[blockIdx.x].valid = 0;  // until a split group starts
    pdl_launch_dependents();       // the merge may be scheduled
  }

  if (warp == kConsumerWarps) {
    // ======================= producer warp =======================
    // pages of every sequence, times its groups (kv heads x row groups):
    // only this warp walks the slices, so it builds the prefix itself
    int *const seqlen = sm.prefix + p.batch + 1;
    const int total_pages = build_prefix(p, sm.prefix, seqlen, groups_per_seq,
                                         lane, &g_status_attn);
    const int n_ctas = working_ctas(total_pages, p.min_pages);
    // this CTA's slice of the flattened (sequence, group, page) space
    const int range_begin = slice_begin(blockIdx.x, total_pages, n_ctas);
    const int range_end = blockIdx.x < n_ctas
                              ? slice_begin(blockIdx.x + 1, total_pages, n_ctas)
                              : total_pages;
    int c = 0;   // pages issued so far
    int us = 0;  // segments published so far
    bool waited = !p.early;  // the grid-dependency wait is behind us
    bool ok = true;
    int pos = range_begin;
    while (true) {
      const int slot = us % kUnitRing;
      if (lane == 0)
        ok = mbar_wait(&sm.uempty[slot], ((us / kUnitRing) & 1) ^ 1);
      ok = __shfl_sync(kFull, ok, 0) && !sm.abort_flag;
      if (!ok) break;
      const UnitInfo seg =
          pos < range_end
              ? decode_segment(p, sm.prefix, seqlen, groups_per_seq, pos,
                               us == 0, range_end, total_pages, n_ctas)
              : UnitInfo{};
      if (!seg.valid) {
        if (lane == 0) {
          sm.unit[slot].valid = 0;
          mbar_arrive(&sm.ufull[slot]);
        }
        break;
      }
      const int b = seg.b, g = seg.g, n_pages = seg.n_pages;
      const int page0 = seg.page0, na = seg.n_a, bs = seg.b_start;
      if (lane == 0) {
        sm.unit[slot] = seg;
        mbar_arrive(&sm.ufull[slot]);
      }
      const size_t head_off = (size_t)g * C::PAGE_ELEMS;
      for (int k0 = 0; k0 < n_pages && ok; k0 += kTableChunk) {
        // block-table entries of the next chunk, one coalesced load each
        int phys[kTableChunk / 32];
#pragma unroll
        for (int k4 = 0; k4 < kTableChunk / 32; ++k4) {
          const int k = k0 + k4 * 32 + lane;
          phys[k4] = -1;
          if (k < n_pages) {
            const int pidx = page0 + k;
            const int lb = (pidx < na) ? pidx : bs + (pidx - na);
            phys[k4] = __ldg(p.block_table + (size_t)b * p.max_blocks + lb);
          }
        }
        // Pages go out in batches, every step spread over the lanes: lane
        // 0 waits for the next stage, lane i tests whether stage c + i is
        // free too, the run of free stages from c is the batch; lane i arms
        // stage c + i, and the batch's K and V copies are issued one per
        // lane.  One thread doing all of it page by page cannot keep 2 KB
        // FP8 pages coming: each barrier operation and copy it issues
        // waits for the one before.
        constexpr int CPP = MMA ? 2 * (D / kBoxElems) : 2;  // copies per page
        constexpr int MAXB = (32 / CPP) < STAGES ? (32 / CPP) : STAGES;
        const int part = lane % CPP;
#pragma unroll
        for (int k4 = 0; k4 < kTableChunk / 32; ++k4) {
          for (int kk = 0; kk < 32;) {
            const int k = k0 + k4 * 32 + kk;
            if (k >= n_pages) break;
#ifdef SVP_TEST_STALL_AFTER
            // test builds only: the producer stops after a few pages and
            // waits on a barrier nothing arrives on, so every role's wait
            // runs out and takes its timeout path
            if (c >= SVP_TEST_STALL_AFTER) {
              if (lane == 0) ok = mbar_wait(&sm.stall, 0);
              ok = __shfl_sync(kFull, ok, 0);
              if (!ok) break;
            }
#endif
            const int left = min(min(32 - kk, n_pages - k), MAXB);
            if (!waited) {
              const int pl = page0 + k + left - 1;  // the batch's last page
              const int lb = pl < na ? pl : bs + (pl - na);
              if ((lb + 1) * kBlockSize > seg.seq_len - p.q_len) {
                pdl_wait();  // it may hold some of the appended positions
                waited = true;
              }
            }
            // lane i: page c + i's block (arming), and the page of this
            // lane's copy
            const int ph_i = __shfl_sync(kFull, phys[k4], min(kk + lane, 31));
            const int pg = lane / CPP;
            const int ph_c = __shfl_sync(kFull, phys[k4], min(kk + pg, 31));
            bool ready = false;
            if (lane == 0)
              ready = mbar_wait(&sm.empty[c % STAGES], ((c / STAGES) & 1) ^ 1);
            ok = __shfl_sync(kFull, ready, 0);
            if (!ok) break;
            if (lane > 0 && lane < left)
              ready = mbar_ready(&sm.empty[(c + lane) % STAGES],
                                 (((c + lane) / STAGES) & 1) ^ 1);
            const unsigned run = __ballot_sync(kFull, lane < left && ready);
            const int n = __ffs(~run) - 1;  // stages c .. c + n - 1 are free
            if (lane < n) {
              const int s = (c + lane) % STAGES;
              if (ph_i >= 0 && ph_i < p.num_blocks) {
                sm.stage_ok[s] = 1;
                mbar_arrive_expect_tx(&sm.full[s], 2 * C::PAGE_BYTES);
              } else {
                raise_flag(SVP_DEV_BAD_BLOCK_ID);
                sm.stage_ok[s] = 0;
                mbar_arrive(&sm.full[s]);
              }
            }
            __syncwarp();
            if (pg < n && ph_c >= 0 && ph_c < p.num_blocks) {
              const int s = (c + pg) % STAGES;
              if constexpr (MMA) {
                const int y = (ph_c * p.num_kv_heads + g) * kBlockSize;
                const int bx = part >> 1;
                if (part & 1)
                  tma_load_2d(sm.kv[s][1] + bx * kBoxBytes, &tm.v,
                              bx * kBoxElems, y, &sm.full[s]);
                else
                  tma_load_2d(sm.kv[s][0] + bx * kBoxBytes, &tm.k,
                              bx * kBoxElems, y, &sm.full[s]);
              } else {
                const size_t off = (size_t)ph_c * p.num_kv_heads * C::PAGE_ELEMS +
                                   head_off;
                bulk_g2s(sm.kv[s][part],
                         static_cast<const T *>(part ? p.v_cache : p.k_cache) + off,
                         C::PAGE_BYTES, &sm.full[s]);
              }
            }
            c += n;
            kk += n;
          }
          if (!ok) break;
        }
      }
      if (!ok) break;
      pos = seg.item0 + (seg.n_pages + p.ppi - 1) / p.ppi;
      ++us;
    }
    if (!ok) {
      // give up: flag it, then wait (bounded) for copies still in flight
      if (lane == 0) {
        raise_flag(SVP_DEV_TIMEOUT);
        sm.abort_flag = 1;
        for (int k = max(0, c - STAGES); k < c; ++k)
          (void)mbar_wait_drain(&sm.full[k % STAGES], (k / STAGES) & 1);
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
      const int stream = warp / MT, mt = warp % MT;
      const int first = ((stream - c) % NSTREAM + NSTREAM) % NSTREAM;
      bool aborted = false;
      int t_min = 0x7fffffff, t_max = -1;  // positions of the unit's rows
      for (int r = 0; r < RB; ++r) {
        const int gr = rg * RB + r;
        if (gr < p.rows) {
          const int tt = t0 + gr / p.group;
          t_min = min(t_min, tt);
          t_max = max(t_max, tt);
        }
      }
      // a page is visible to every row without checks if it ends by the
      // first row's position (with a tree: before the tree's nodes)
      if (p.tree_mask) t_min = min(t_min, t0 - 1);

      if constexpr (MMA) {
        // ---- tensor-core path: 16 rows, lane rows g and g+8 ----
        const int gq = lane >> 2, tq = lane & 3;
        uint32_t qa[D / 16][4];
        float o[D / 8][4];
        float m[2] = {-INFINITY, -INFINITY}, lp[2] = {0.f, 0.f};
        int t[2] = {-1, -1};
        uint32_t tm[2] = {0u, 0u};
        // Q fragments straight from global memory: rows past the unit's
        // last row read row 0 of the group and are masked to zero, so all
        // loads are unconditional and issue back to back.
        const uint32_t *qrow[2];
        uint32_t qmask[2];
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          const int gr = rg * RB + mt * 16 + gq + 8 * r;
          const bool valid = gr < p.rows;
          const int grc = valid ? gr : 0;
          const int i = grc / p.group;
          const int h = g * p.group + grc % p.group;
          qrow[r] = reinterpret_cast<const uint32_t *>(
              static_cast<const uint16_t *>(p.q) +
              (((size_t)b * p.q_len + i) * p.num_q_heads + h) * D);
          qmask[r] = valid ? 0xffffffffu : 0u;
          t[r] = valid ? t0 + i : -1;
          tm[r] = row_tree_bits(p, b, i);
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int w0 = ks * 8 + tq;  // 32-bit word of columns 16ks+2tq, +1
          qa[ks][0] = __ldg(qrow[0] + w0);
          qa[ks][1] = __ldg(qrow[1] + w0);
          qa[ks][2] = __ldg(qrow[0] + w0 + 4);
          qa[ks][3] = __ldg(qrow[1] + w0 + 4);
        }
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          qa[ks][0] &= qmask[0];
          qa[ks][1] &= qmask[1];
          qa[ks][2] &= qmask[0];
          qa[ks][3] &= qmask[1];
        }
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn)
          o[dn][0] = o[dn][1] = o[dn][2] = o[dn][3] = 0.f;

        for (int k = first; k < ui.n_pages; k += NSTREAM) {
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
            const bool union_full = (j1 < L) && (p.window == 0 || j1 < p.n_sink ||
                                                 j0 > t0 - p.window);
            if (!union_full)
              zero_invalid_rows<T, D, true>(sm.kv[s][1], lane, j0, L, t0,
                                            p.n_sink, p.window);
            const bool all_vis = (j1 <= t_min) &&
                                 (p.window == 0 || j1 < p.n_sink ||
                                  j0 > t_max - p.window);
            uint32_t kb[D / 16][4], vb[D / 16][4];
            load_page_frags<D>(smem_u32(sm.kv[s][0]), smem_u32(sm.kv[s][1]),
                               kb, vb, lane);
            // the page is in registers: hand the stage back to the producer
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
            process_page_mma<D>(kb, vb, qa, o, m, lp, lane, j0, all_vis, t,
                                tm, t0, p.n_sink, p.window, p.qscale);
          } else {
            __syncwarp();
            if (lane == 0) mbar_arrive(&sm.empty[s]);
          }
        }
        // per-lane partial row sums -> the quad (same g) total
#pragma unroll
        for (int r = 0; r < 2; ++r) {
          lp[r] += __shfl_xor_sync(kFull, lp[r], 1);
          lp[r] += __shfl_xor_sync(kFull, lp[r], 2);
        }
        if (tq == 0) {
          sm.red_m[warp][gq] = m[0];
          sm.red_m[warp][gq + 8] = m[1];
          sm.red_l[warp][gq] = lp[0];
          sm.red_l[warp][gq + 8] = lp[1];
        }
#pragma unroll
        for (int dn = 0; dn < D / 8; ++dn) {
          const int d = dn * 8 + 2 * tq;
          *reinterpret_cast<float2 *>(&sm.red_o[warp][gq][d]) =
              make_float2(o[dn][0], o[dn][1]);
          *reinterpret_cast<float2 *>(&sm.red_o[warp][gq + 8][d]) =
              make_float2(o[dn][2], o[dn][3]);
        }
      } else {
        // ---- CUDA-core path ----
        // FP8 pages, one row, head_dim 128: key per lane (see
        // process_page_fp8_k1); q kept as fp16 of this lane's half
        constexpr bool kKeyLane = std::is_same<T, uint8_t>::value && RB == 1 &&
                                  D == 128;
        uint32_t qr[4][8];
        float q[RB][VEC], o[RB][VEC], m[RB], l[RB];
        int t[RB];
        uint32_t tm[RB];
#pragma unroll
        for (int r = 0; r < RB; ++r) {
          const int gr = rg * RB + r;
          tm[r] = 0u;
          m[r] = -INFINITY;
          l[r] = 0.f;
#pragma unroll
          for (int e = 0; e < VEC; ++e) { o[r][e] = 0.f; q[r][e] = 0.f; }
          t[r] = -1;
          if (gr < p.rows) {
            const int i = gr / p.group;
            const int h = g * p.group + gr % p.group;
            using TQ = typename QT<T>::type;
            const TQ *qp = static_cast<const TQ *>(p.q) +
                           (((size_t)b * p.q_len + i) * p.num_q_heads + h) * D +
                           lane * VEC;
            if constexpr (kKeyLane) {
              // dims half*64 + ((c + key) & 3)*16 .. +16 of the row, bf16
              // -> fp16 pairs, in this lane's chunk order
              const int key = lane >> 1, half = lane & 1;
              const uint16_t *qrow = static_cast<const uint16_t *>(p.q) +
                                     (((size_t)b * p.q_len + i) * p.num_q_heads + h) * D +
                                     half * 64;
#pragma unroll
              for (int c = 0; c < 4; ++c) {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    qrow + ((c + key) & 3) * 16);
                const uint4 a = __ldg(src), b2 = __ldg(src + 1);
                const uint32_t w[8] = {a.x, a.y, a.z, a.w, b2.x, b2.y, b2.z, b2.w};
#pragma unroll
                for (int k2 = 0; k2 < 8; ++k2) {
                  const float lo = __uint_as_float(w[k2] << 16);
                  const float hi = __uint_as_float(w[k2] & 0xffff0000u);
                  const __half2 hh = __floats2half2_rn(lo, hi);
                  qr[c][k2] = *reinterpret_cast<const uint32_t *>(&hh);
                }
              }
            } else {
              Vec<TQ, D>::load(qp, q[r]);
#pragma unroll
              for (int e = 0; e < VEC; ++e) q[r][e] *= p.qscale;
            }
            t[r] = t0 + i;
            tm[r] = row_tree_bits(p, b, i);
          }
        }
        for (int k = first; k < ui.n_pages; k += NSTREAM) {
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
            const bool union_full = (j1 < L) && (p.window == 0 || j1 < p.n_sink ||
                                                 j0 > t0 - p.window);
            if (!union_full)
              zero_invalid_rows<T, D, false>(sm.kv[s][1], lane, j0, L, t0,
                                             p.n_sink, p.window);
            const bool all_vis = (j1 <= t_min) &&
                                 (p.window == 0 || j1 < p.n_sink ||
                                  j0 > t_max - p.window);
            if constexpr (kKeyLane)
              process_page_fp8_k1(
                  reinterpret_cast<const uint8_t *>(sm.kv[s][0]),
                  reinterpret_cast<const uint8_t *>(sm.kv[s][1]), qr,
                  reinterpret_cast<float (&)[4]>(o[0]), m[0], l[0],
                  reinterpret_cast<uint16_t *>(pbuf), lane, j0, all_vis,
                  t[0], tm[0], t0, p.n_sink, p.window, p.qscale);
            else
              process_page_fma<T, D, RB>(
                  reinterpret_cast<const T *>(sm.kv[s][0]),
                  reinterpret_cast<const T *>(sm.kv[s][1]), q, o, m, l, pbuf,
                  lane, j0, all_vis, t, tm, t0, p.n_sink, p.window);
          }
          if (lane == 0) mbar_arrive(&sm.empty[s]);
        }
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
      }
      c += ui.n_pages;

      // ---- epilogue: merge the 4 warps' states ----
      if (p.early) pdl_wait();  // outputs are written from here on
      if (!epi_sync(sm, epi_phase, lane) || aborted) {
        if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
        break;
      }
      // a group owned by one CTA is finished here; else a partial goes to
      // this CTA's first- or last-segment slot
      const bool single = ui.f == ui.l;
      const size_t pslot = (size_t)(2 * blockIdx.x + ui.slot);
      const int vrows = min(RB, p.rows - rg * RB);  // valid rows of the unit
      // per-row statistics, once per row: row r lives in local row lr of
      // the warps w with w % MT == r / RW; their states are weighted by
      // exp2(m_w - M) / L so that the elements below only multiply-add
      if (ctid < vrows) {
        const int r = ctid, w0 = r / RW, lr = r % RW;
        float M = -INFINITY;
#pragma unroll
        for (int w = w0; w < kConsumerWarps; w += MT)
          M = fmaxf(M, sm.red_m[w][lr]);
        float Lsum = 0.f;
        float f[kConsumerWarps];
#pragma unroll
        for (int w = w0, k = 0; w < kConsumerWarps; w += MT, ++k) {
          const float mw = sm.red_m[w][lr];
          f[k] = (mw == -INFINITY) ? 0.f : ex2(mw - M);
          Lsum = fmaf(f[k], sm.red_l[w][lr], Lsum);
        }
        const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
        for (int w = w0, k = 0; w < kConsumerWarps; w += MT, ++k)
          sm.wf[w][r] = f[k] * inv;
        const float lse2 = Lsum > 0.f ? M + log2f(Lsum) : -INFINITY;
        const int gr = rg * RB + r;
        if (single) {
          const int i = gr / p.group;
          const int h = g * p.group + gr % p.group;
          p.lse[((size_t)b * p.q_len + i) * p.num_q_heads + h] = lse2 * kLn2;
        } else {
          p.part_lse[pslot * RB + r] = lse2;
        }
      }
      if (!epi_sync(sm, epi_phase, lane)) {
        if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
        break;
      }
      for (int e4 = ctid; e4 < vrows * (D / 4); e4 += kConsumerWarps * 32) {
        const int r = e4 / (D / 4), d = (e4 % (D / 4)) * 4;
        const int w0 = r / RW, lr = r % RW;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = w0; w < kConsumerWarps; w += MT) {
          const float f = sm.wf[w][r];
          const float4 v = *reinterpret_cast<const float4 *>(&sm.red_o[w][lr][d]);
          a.x = fmaf(f, v.x, a.x);
          a.y = fmaf(f, v.y, a.y);
          a.z = fmaf(f, v.z, a.z);
          a.w = fmaf(f, v.w, a.w);
        }
        // an FP8 cache's V scale (1 otherwise) applies to every output
        a.x *= p.v_scale;
        a.y *= p.v_scale;
        a.z *= p.v_scale;
        a.w *= p.v_scale;
        const int gr = rg * RB + r;
        if (single) {
          const int i = gr / p.group;
          const int h = g * p.group + gr % p.group;
          using TQ = typename QT<T>::type;
          TQ *dst = static_cast<TQ *>(p.out) +
                    (((size_t)b * p.q_len + i) * p.num_q_heads + h) * D + d;
          store_out(dst + 0, a.x);
          store_out(dst + 1, a.y);
          store_out(dst + 2, a.z);
          store_out(dst + 3, a.w);
        } else {
          const size_t prow = pslot * RB + r;
          *reinterpret_cast<float4 *>(p.part_o + prow * D + d) = a;
        }
      }
      if (!single && ctid == 0) record_split(p, ui, blockIdx.x);
      // all consumers are done with this unit's info and scratch
      if (!epi_sync(sm, epi_phase, lane)) {
        if (lane == 0) { raise_flag(SVP_DEV_TIMEOUT); sm.abort_flag = 1; }
        break;
      }
      if (ctid == 0) mbar_arrive(&sm.uempty[slot]);
      ++us;
    }
  }

  __syncthreads();  // no warp leaves while the others may use the barriers
}

// --------------------------------------------------------------------------
// host side
// --------------------------------------------------------------------------

// per (device, instantiation, shared-memory size): attribute set + occupancy
static std::mutex g_occ_mu;
static std::map<std::tuple<int, const void *, size_t>, int> g_occ;

static size_t batch_bucket(int batch) { return (size_t)(batch + 255) / 256 * 256; }

template <typename T, int D, int RB, bool MMA>
static int prepare_t(int batch) {
  const size_t smem = smem_bytes<T, D, RB, MMA>((int)batch_bucket(batch));
  auto kern = paged_attention_kernel<T, D, RB, MMA>;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  const auto key = std::make_tuple(dev, (const void *)kern, smem);
  {
    std::lock_guard<std::mutex> lk(g_occ_mu);
    auto it = g_occ.find(key);
    if (it != g_occ.end()) return it->second;
  }
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem) != cudaSuccess)
    return -1;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem) !=
      cudaSuccess)
    return -1;
  n = n > 0 ? n : 1;
  std::lock_guard<std::mutex> lk(g_occ_mu);
  g_occ[key] = n;
  return n;
}

template <typename T, int D, int RB, bool MMA>
static cudaError_t launch_t(const AttnParams &p, int grid, cudaStream_t st) {
  if (prepare_t<T, D, RB, MMA>(p.batch) < 0) return cudaErrorInvalidValue;
  const size_t smem = smem_bytes<T, D, RB, MMA>((int)batch_bucket(p.batch));
  TensorMaps tm;
  memset(&tm, 0, sizeof tm);
  if constexpr (MMA) {
    if (!cached_map(&tm.k, 0, p.k_cache, p.num_blocks, p.num_kv_heads, D) ||
        !cached_map(&tm.v, 0, p.v_cache, p.num_blocks, p.num_kv_heads, D))
      return cudaErrorInvalidValue;
  }
  return launch_pdl(paged_attention_kernel<T, D, RB, MMA>, (unsigned)grid,
                    (unsigned)kThreads, smem, st, p, tm);
}

#define SVP_DISPATCH(DTYPE, HD, RB, MMA, CALL)                        \
  do {                                                                \
    if (MMA) {                                                        \
      if (HD == 64) {                                                 \
        if (RB == 16) CALL(uint16_t, 64, 16, true);                   \
        else CALL(uint16_t, 64, 32, true);                            \
      } else {                                                        \
        if (RB == 16) CALL(uint16_t, 128, 16, true);                  \
        else CALL(uint16_t, 128, 32, true);                           \
      }                                                               \
    } else if (DTYPE == 2) {                                          \
      if (HD == 64) {                                                 \
        switch (RB) { case 1: CALL(uint8_t, 64, 1, false); break;     \
                      case 2: CALL(uint8_t, 64, 2, false); break;     \
                      case 4: CALL(uint8_t, 64, 4, false); break;     \
                      default: CALL(uint8_t, 64, 8, false); }         \
      } else {                                                        \
        switch (RB) { case 1: CALL(uint8_t, 128, 1, false); break;    \
                      case 2: CALL(uint8_t, 128, 2, false); break;    \
                      case 4: CALL(uint8_t, 128, 4, false); break;    \
                      default: CALL(uint8_t, 128, 8, false); }        \
      }                                                               \
    } else if (DTYPE == 0) {                                          \
      if (HD == 64) {                                                 \
        switch (RB) { case 1: CALL(float, 64, 1, false); break;       \
                      case 2: CALL(float, 64, 2, false); break;       \
                      case 4: CALL(float, 64, 4, false); break;       \
                      default: CALL(float, 64, 8, false); }           \
      } else {                                                        \
        switch (RB) { case 1: CALL(float, 128, 1, false); break;      \
                      case 2: CALL(float, 128, 2, false); break;      \
                      case 4: CALL(float, 128, 4, false); break;      \
                      default: CALL(float, 128, 8, false); }          \
      }                                                               \
    } else {                                                          \
      if (HD == 64) {                                                 \
        switch (RB) { case 1: CALL(uint16_t, 64, 1, false); break;    \
                      case 2: CALL(uint16_t, 64, 2, false); break;    \
                      case 4: CALL(uint16_t, 64, 4, false); break;    \
                      default: CALL(uint16_t, 64, 8, false); }        \
      } else {                                                        \
        switch (RB) { case 1: CALL(uint16_t, 128, 1, false); break;   \
                      case 2: CALL(uint16_t, 128, 2, false); break;   \
                      case 4: CALL(uint16_t, 128, 4, false); break;   \
                      default: CALL(uint16_t, 128, 8, false); }       \
      }                                                               \
    }                                                                 \
  } while (0)

cudaError_t launch_attention(const AttnParams &p, int dtype, bool mma,
                             int grid, cudaStream_t stream) {
  cudaError_t e = cudaSuccess;
#define SVP_CALL(T, D, RB, M) e = launch_t<T, D, RB, M>(p, grid, stream)
  SVP_DISPATCH(dtype, p.head_dim, p.rb, mma, SVP_CALL);
#undef SVP_CALL
  return e;
}

int attention_ctas_per_sm(int dtype, int head_dim, int rb, bool mma,
                          int batch) {
  int n = 1;
#define SVP_CALL(T, D, RB, M) n = prepare_t<T, D, RB, M>(batch)
  SVP_DISPATCH(dtype, head_dim, rb, mma, SVP_CALL);
#undef SVP_CALL
  return n > 0 ? n : 1;
}

bool tensor_maps_available() { return encode_fn() != nullptr; }

cudaError_t launch_merge(const AttnParams &p, int dtype, int grid,
                         cudaStream_t stream) {
#define SVP_MERGE(T, D, RB)                                            \
  e = launch_pdl(merge_splits_kernel<T, D, RB, (RB >= 32 ? RB / 16 : 1)>, \
                 (unsigned)grid * (RB >= 32 ? RB / 16u : 1u),           \
                 (unsigned)kMergeThreads, 0, stream, p)
  const bool f32 = dtype == 0;
  const int D = p.head_dim;
  cudaError_t e = cudaSuccess;
  switch (p.rb) {
#define SVP_MERGE_RB(RB)                                             \
  case RB:                                                           \
    if (f32) { if (D == 64) SVP_MERGE(float, 64, RB); else SVP_MERGE(float, 128, RB); } \
    else { if (D == 64) SVP_MERGE(uint16_t, 64, RB); else SVP_MERGE(uint16_t, 128, RB); } \
    break;
    SVP_MERGE_RB(1)
    SVP_MERGE_RB(2)
    SVP_MERGE_RB(4)
    SVP_MERGE_RB(8)
    SVP_MERGE_RB(16)
    SVP_MERGE_RB(32)
    SVP_MERGE_RB(64)
#undef SVP_MERGE_RB
    default:
      return cudaErrorInvalidValue;
  }
#undef SVP_MERGE
  return e;
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
